// Tensor-core kernels for bf16 packed-tree KDA on sm_103a (dk = dv = 128, chunk 64).
//
// One CTA (256 threads) per (sequence, head) of a round, chunks in order; the fp32
// state lives in tensor memory (TMEM) for the whole sequence as S^T (lane = value
// channel, column = key channel).  Every product of the chunkwise form runs on
// tcgen05.mma (bf16 operands in shared memory, fp32 accumulation in TMEM), all as
// M = 128 tiles whose 128 rows are a channel dimension or the stacked [Kp; Qp] rows:
//   AP   = [Kp; Qp] Km^T            (A = strict_lower rows 0-63, P = incl_lower rows 64-127)
//   WkT  = (beta Kd)^T T^T          UT = (beta V)^T T^T - S^T Wk^T      (= U^T)
//   OT   = S^T Qd^T + U^T P^T       (= O^T)
//   ST  <- ST diag(e^{Gamma_L}) + U^T Kt                                 (= S^T update)
// with Kp = K e^{Gamma-m}, Km = K e^{m-Gamma}, Qp = Q e^{Gamma-m}, Kd = K e^{Gamma},
// Qd = Q e^{Gamma}, Kt = K e^{Gamma_L-Gamma} (m: Gamma at a reference row, so no factor
// exceeds exp(|Gamma_L|/2)), and T = (I + diag(beta) A)^-1 by blocked forward
// substitution in fp32 on the CUDA cores.  Bounded replay (page "HARTS ... 精读",
// section 4.2): the first chunk of a side branch starts with its replay rows, which
// update the state but write no output.
#include "kda_common.cuh"
#include "tc_primitives.cuh"

namespace harts {
namespace {

constexpr int D = 128, BC = 64, NT = 256;

// Shared-memory layout (bytes from a 1024-aligned base).  Regions are reused once the
// MMA that reads them has completed.
namespace fwd_sm {
constexpr uint32_t KQp = 0;                 // [128 rows][128 K]  Kp rows 0-63, Qp 64-127
constexpr uint32_t Mf = KQp;                //   -> fp32 [64][64] M = diag(beta) A
constexpr uint32_t Tf = KQp + 16384;        //   -> fp32 [64][64] T
constexpr uint32_t Os = KQp;                //   -> bf16 [64 t][128 dv] output staging
constexpr uint32_t Km = KQp + 32768;        // [64][128]
constexpr uint32_t Tm = Km;                 //   -> [64 t][64 s] T (bf16)
constexpr uint32_t Pm = Km + 8192;          //   -> [64 t][64 s] P (bf16)
constexpr uint32_t BKdT = Km + 16384;       // [128 dk][64 t]  (beta Kd)^T
constexpr uint32_t nWk = BKdT;              //   -> [64 t][128 dk]  -Wk
constexpr uint32_t BVT = BKdT + 16384;      // [128 dv][64 t]  (beta V)^T
constexpr uint32_t UTs = BVT;               //   -> [128 dv][64 t]  U^T
constexpr uint32_t Qd = BVT + 16384;        // [64 t][128 dk]
constexpr uint32_t KtT = Qd + 16384;        // [128 dk][64 t]
constexpr uint32_t STs = KtT + 16384;       // [128 dv][128 dk]  bf16 copy of S^T
constexpr uint32_t Stage = STs + 32768;     // raw next-chunk inputs, row-major [64][128] bf16
constexpr uint32_t SQ = Stage, SK = Stage + 16384, SV = Stage + 32768, SG = Stage + 49152;
constexpr uint32_t SBeta = Stage + 65536;   // [64] 32-bit words holding the bf16 beta
constexpr uint32_t SBpar = SBeta + 256;     // [64] int: which half of the word
constexpr uint32_t Vec = SBpar + 256;       // fp32 vectors
constexpr uint32_t vBeta = Vec, vEl = vBeta + 64 * 4, vT0 = vEl + 128 * 4, vT1 = vT0 + 128 * 4,
                   vM = vT1 + 128 * 4, vEnd = vM + 128 * 4;
constexpr uint32_t bytes = vEnd + 1024;     // + alignment slack
}  // namespace fwd_sm

// fp32 64x64 scratch index with a per-row XOR so that column-wise access is conflict-free.
__device__ __forceinline__ int fidx(int t, int s) { return t * 64 + (s ^ (t & 31)); }

__device__ __forceinline__ void st_bf16(uint8_t *tile, int rows, int row, int col, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(tile + tc::sw128_offset(rows, row, col)) =
        __float2bfloat16_rn(x);
}

// Blocked inversion of the unit lower-triangular (I + Mf) into Tf (fp32, lower part;
// entries above the diagonal inside the diagonal blocks are written as zero).
// Diagonal 16x16 blocks: one column per thread held in registers.  Off-diagonal blocks
// by increasing distance: T_ij = -T_ii * sum_{k=j}^{i-1} M_ik T_kj, the inner sums kept
// in the unused upper triangle of Mf at the transposed block.
__device__ void invert_unit_lower(float *Mf, float *Tf) {
    const int tid = threadIdx.x;
    if (tid < 64) {
        const int b = tid >> 4, s = tid & 15;
        float col[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < t; ++j) acc += Mf[fidx(16 * b + t, 16 * b + j)] * col[j];
            col[t] = t < s ? 0.f : (t == s ? 1.f : -acc);
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) Tf[fidx(16 * b + t, 16 * b + s)] = col[t];
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
        const int nblk = 4 - d;
        for (int e = threadIdx.x; e < nblk * 256; e += NT) {
            const int j = e >> 8, i = j + d, t = (e >> 4) & 15, s = e & 15;
            float acc = 0.f;
            for (int kb = j; kb < i; ++kb) {
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    acc += Mf[fidx(16 * i + t, 16 * kb + u)] * Tf[fidx(16 * kb + u, 16 * j + s)];
            }
            Mf[fidx(16 * j + s, 16 * i + t)] = acc;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < nblk * 256; e += NT) {
            const int j = e >> 8, i = j + d, t = (e >> 4) & 15, s = e & 15;
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u)
                acc += Tf[fidx(16 * i + t, 16 * i + u)] * Mf[fidx(16 * j + s, 16 * i + u)];
            Tf[fidx(16 * i + t, 16 * j + s)] = -acc;
        }
        __syncthreads();
    }
}

// Wait for an MMA batch on every thread; a shared flag records a timeout.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t phase, int *s_fail) {
    if (!tc::mbar_wait(bar, phase)) atomicOr(s_fail, 1);
    __syncthreads();
    tc::fence_after_sync();
    return *s_fail == 0;
}

// Make shared-memory writes and TMEM reads of all threads ordered before the next MMA.
__device__ __forceinline__ void sync_for_mma() {
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

// Issue asynchronous copies of one chunk's raw q, k, v, g rows (256 B each) and beta
// into the staging buffer; rows past the sequence end are zero-filled.
__device__ void prefetch_chunk(const FwdParams &p, const PlanDev &pd, int32_t seq, int32_t h,
                               int32_t rho, int32_t L, int32_t c0, uint8_t *sm) {
    using namespace fwd_sm;
    const int H = p.H;
    const uint8_t *base[4] = {static_cast<const uint8_t *>(p.q), static_cast<const uint8_t *>(p.k),
                              static_cast<const uint8_t *>(p.v), static_cast<const uint8_t *>(p.g)};
    for (int e = threadIdx.x; e < 64 * 16 * 4; e += NT) {
        const int ten = e >> 10, t = (e >> 4) & 63, piece = e & 15;
        const int64_t row = local_row(pd, seq, rho, L, c0 + t);
        const uint8_t *src = row >= 0 ? base[ten] + ((row * H + h) * D * 2 + piece * 16) : base[ten];
        tc::cp_async16(sm + Stage + ten * 16384 + t * 256 + piece * 16, src, row >= 0 ? 16u : 0u);
    }
    for (int t = threadIdx.x; t < 64; t += NT) {
        const int64_t row = local_row(pd, seq, rho, L, c0 + t);
        const int64_t idx = row >= 0 ? row * H + h : 0;
        const uint8_t *src = static_cast<const uint8_t *>(p.beta) + (idx & ~int64_t(1)) * 2;
        tc::cp_async4(sm + SBeta + t * 4, src, row >= 0 ? 4u : 0u);
        reinterpret_cast<int *>(sm + SBpar)[t] = static_cast<int>(idx & 1);
    }
    tc::cp_async_commit();
}

__device__ __forceinline__ float stage_val(const uint8_t *sm, uint32_t off, int t, int c) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + off + t * 256 + c * 2));
}

__global__ void __launch_bounds__(NT, 1) kda_fwd_tc(FwdParams p, PlanDev pd, int32_t round_base) {
    using namespace fwd_sm;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    __shared__ uint64_t bars[4];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    float *vbeta = reinterpret_cast<float *>(sm + vBeta), *vel = reinterpret_cast<float *>(sm + vEl),
          *vt0 = reinterpret_cast<float *>(sm + vT0), *vt1 = reinterpret_cast<float *>(sm + vT1),
          *vm = reinterpret_cast<float *>(sm + vM);
    float *Mfp = reinterpret_cast<float *>(sm + Mf), *Tfp = reinterpret_cast<float *>(sm + Tf);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lg = warp & 3, ch = warp >> 2;
    const int H = p.H;
    const int32_t h = blockIdx.x % H;
    const int32_t seq = pd.round_order[round_base + blockIdx.x / H];
    const int32_t rho = pd.seq_rho[seq], L = rho + pd.seq_nown[seq];
    const int32_t nch = (L + BC - 1) / BC;
    const int32_t src = pd.seq_src[seq];
    const int32_t row0 = pd.seq_row0[seq], cbase = pd.seq_cbase[seq];
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
    uint8_t *cst = static_cast<uint8_t *>(p.chunk_states);

    prefetch_chunk(p, pd, seq, h, rho, L, 0, sm);
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) tc::mbar_init(&bars[i], 1);
        s_fail = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
    const uint32_t tST = tm, tAP = tm + 128, tWk = tm + 192, tUT = tm + 256, tOT = tm + 320;
    const int jv = lg * 32 + lane;                       // this thread's TMEM lane

    // Copy the bf16 S^T tile (SW128) to a saved chunk state, [dv][dk] row-major, 16 B per thread.
    auto save_chunk_state = [&](int32_t chunk_index) {
        if (!cst) return;
        uint8_t *dst = cst + (static_cast<int64_t>(chunk_index) * H + h) * D * D * 2;
        for (int e = tid; e < 128 * 16; e += NT) {
            const int r = e >> 4, piece = e & 15;
            *reinterpret_cast<uint4 *>(dst + r * 256 + piece * 16) =
                *reinterpret_cast<const uint4 *>(sm + STs + tc::sw128_offset(128, r, piece * 8));
        }
    };

    // ---- initial state into TMEM (S^T) and its bf16 copy ----------------------------------
    {
        const float *S0 = src >= 0 ? p.states + (static_cast<int64_t>(src) * H + h) * D * D
                        : (p.h0 ? p.h0 + (static_cast<int64_t>(-1 - src) * H + h) * D * D : nullptr);
        for (int hf = 0; hf < 2; ++hf) {
            float r[32];
            const int cb = ch * 64 + hf * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = S0 ? S0[(cb + j) * D + jv] : 0.f;
            tc::tmem_st32(tST + lane_off + cb, r);
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + STs, 128, jv, cb + j, r + j);
        }
        __syncthreads();
        save_chunk_state(cbase);
    }
    sync_for_mma();

    int32_t sp = pd.seq_sptr[seq];
    const int32_t sp_end = pd.seq_sptr[seq + 1];
    const int c = tid & 127, half = tid >> 7;
    for (int32_t ci = 0; ci < nch; ++ci) {
        const uint32_t ph = ci & 1;
        const int32_t c0 = ci * BC;
        const int nv = min(BC, L - c0);
        const int mid = (nv - 1) / 2;
        tc::cp_async_wait_all();
        __syncthreads();
        // ---- prep: cumulative decay, scaled operands (from the staged raw tiles) ----------
        {
            float s = 0.f, mref = 0.f;
#pragma unroll 8
            for (int t = half * 32; t < half * 32 + 32; ++t) {
                s += stage_val(sm, SG, t, c);
                if (t == mid) mref = s;
            }
            if (half == 0) { vt0[c] = s; vm[c] = mref; } else vt1[c] = s;
            if (tid < 64) {
                const uint32_t w = reinterpret_cast<const uint32_t *>(sm + SBeta)[tid];
                const int par = reinterpret_cast<const int *>(sm + SBpar)[tid];
                const uint16_t hb = par ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w & 0xFFFF);
                vbeta[tid] = __bfloat162float(__ushort_as_bfloat16(hb));
            }
            __syncthreads();
            const float m = vm[c], gl = vt0[c] + vt1[c];
            float gam = half ? vt0[c] : 0.f;
            if (-m > kMaxExpArg || m - gl > kMaxExpArg) dev_error(pd, kDevErrDecayRange, seq, c0);
            const float em = __expf(m), ekt = __expf(gl - m);
            if (half == 0) vel[c] = __expf(gl);
            for (int t0 = half * 32; t0 < half * 32 + 32; t0 += 8) {
                float bkd[8], bv[8], kt[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = t0 + u;
                    const float kk = stage_val(sm, SK, t, c), qq = stage_val(sm, SQ, t, c) * p.scale,
                                vv = stage_val(sm, SV, t, c), bb = vbeta[t];
                    gam += stage_val(sm, SG, t, c);
                    const float e1 = __expf(gam - m), e2 = __expf(m - gam);
                    st_bf16(sm + KQp, 128, t, c, kk * e1);
                    st_bf16(sm + KQp, 128, 64 + t, c, qq * e1);
                    st_bf16(sm + Km, 64, t, c, kk * e2);
                    st_bf16(sm + Qd, 64, t, c, qq * e1 * em);
                    bkd[u] = bb * kk * e1 * em;
                    bv[u] = bb * vv;
                    kt[u] = kk * e2 * ekt;
                }
                tc::st_sw128_8(sm + BKdT, 128, c, t0, bkd);
                tc::st_sw128_8(sm + BVT, 128, c, t0, bv);
                tc::st_sw128_8(sm + KtT, 128, c, t0, kt);
            }
        }
        sync_for_mma();
        // the staging buffer is free: fetch the next chunk while this one computes
        if (ci + 1 < nch) prefetch_chunk(p, pd, seq, h, rho, L, c0 + BC, sm);
        if (tid == 0) {
            tc::mma_tile(tAP, tc::smem_addr(sm + KQp), 128 * 128, tc::smem_addr(sm + Km), 64 * 128,
                         128, tc::idesc_bf16(128, 64), false);
            tc::mma_tile(tOT, tc::smem_addr(sm + STs), 128 * 128, tc::smem_addr(sm + Qd), 64 * 128,
                         128, tc::idesc_bf16(128, 64), false);
            tc::mma_commit(&bars[0]);
        }
        // ---- scale the TMEM state by e^{Gamma_L} per key channel (used by MMA7) -----------
        for (int hf = 0; hf < 2; ++hf) {
            float r[32];
            const int cb = ch * 64 + hf * 32;
            tc::tmem_ld32(tST + lane_off + cb, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] *= vel[cb + j];
            tc::tmem_st32(tST + lane_off + cb, r);
        }
        if (!wait_all(&bars[0], ph, &s_fail)) break;
        // ---- A -> Mf (scaled by beta, strict lower), P -> Pm (incl lower) -----------------
        {
            float r[32];
            tc::tmem_ld32(tAP + lane_off + ch * 32, r);
            if (lg < 2) {
                const int t = jv;
                const float bt = vbeta[t];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int s = ch * 32 + j;
                    Mfp[fidx(t, s)] = s < t ? bt * r[j] : 0.f;
                }
            } else {
                const int t = jv - 64;
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = (ch * 32 + j <= t) ? r[j] : 0.f;
#pragma unroll
                for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + Pm, 64, t, ch * 32 + j, r + j);
            }
        }
        __syncthreads();
        invert_unit_lower(Mfp, Tfp);
        {
            const int t = tid >> 2, s0 = (tid & 3) * 16;
            float r[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = (s0 + j <= t) ? Tfp[fidx(t, s0 + j)] : 0.f;
            tc::st_sw128_8(sm + Tm, 64, t, s0, r);
            tc::st_sw128_8(sm + Tm, 64, t, s0 + 8, r + 8);
        }
        sync_for_mma();
        if (tid == 0) {
            tc::mma_tile(tWk, tc::smem_addr(sm + BKdT), 128 * 128, tc::smem_addr(sm + Tm), 64 * 128,
                         64, tc::idesc_bf16(128, 64), false);
            tc::mma_tile(tUT, tc::smem_addr(sm + BVT), 128 * 128, tc::smem_addr(sm + Tm), 64 * 128,
                         64, tc::idesc_bf16(128, 64), false);
            tc::mma_commit(&bars[1]);
        }
        if (!wait_all(&bars[1], ph, &s_fail)) break;
        // ---- Wk^T -> -Wk as the B operand [t][dk] ------------------------------------------
        {
            float r[32];
            tc::tmem_ld32(tWk + lane_off + ch * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) st_bf16(sm + nWk, 64, ch * 32 + j, jv, -r[j]);
        }
        sync_for_mma();
        if (tid == 0) {
            tc::mma_tile(tUT, tc::smem_addr(sm + STs), 128 * 128, tc::smem_addr(sm + nWk), 64 * 128,
                         128, tc::idesc_bf16(128, 64), true);
            tc::mma_commit(&bars[2]);
        }
        if (!wait_all(&bars[2], ph, &s_fail)) break;
        // ---- U^T -> UTs [dv][t] -----------------------------------------------------------
        {
            float r[32];
            tc::tmem_ld32(tUT + lane_off + ch * 32, r);
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + UTs, 128, jv, ch * 32 + j, r + j);
        }
        sync_for_mma();
        if (tid == 0) {
            tc::mma_tile(tOT, tc::smem_addr(sm + UTs), 128 * 128, tc::smem_addr(sm + Pm), 64 * 128,
                         64, tc::idesc_bf16(128, 64), true);
            tc::mma_tile(tST, tc::smem_addr(sm + UTs), 128 * 128, tc::smem_addr(sm + KtT), 128 * 128,
                         64, tc::idesc_bf16(128, 128), true);
            tc::mma_commit(&bars[3]);
        }
        if (!wait_all(&bars[3], ph, &s_fail)) break;
        // ---- outputs: O rows (staged), next state copy, saved states -----------------------
        {
            float r[32];
            tc::tmem_ld32(tOT + lane_off + ch * 32, r);
            __nv_bfloat16 *os = reinterpret_cast<__nv_bfloat16 *>(sm + Os);
#pragma unroll
            for (int j = 0; j < 32; ++j) os[(ch * 32 + j) * D + jv] = __float2bfloat16_rn(r[j]);
        }
        const int32_t pend = c0 + BC;
        const bool slot = sp < sp_end && pd.state_lpos[sp] == pend;
        const bool last = ci == nch - 1;
        for (int hf = 0; hf < 2; ++hf) {
            float r[32];
            const int cb = ch * 64 + hf * 32;
            tc::tmem_ld32(tST + lane_off + cb, r);
            if (!last) {
#pragma unroll
                for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + STs, 128, jv, cb + j, r + j);
            }
            if (slot) {
                float *dst = p.states + (static_cast<int64_t>(sp) * H + h) * D * D;
#pragma unroll
                for (int j = 0; j < 32; ++j) dst[(cb + j) * D + jv] = r[j];
            }
            if (last && p.final_state) {
                float *dst = p.final_state + (static_cast<int64_t>(seq) * H + h) * D * D;
#pragma unroll
                for (int j = 0; j < 32; ++j) dst[(cb + j) * D + jv] = r[j];
            }
        }
        if (slot) ++sp;
        __syncthreads();
        for (int e = tid; e < 64 * 16; e += NT) {
            const int t = e >> 4, piece = e & 15;
            const int32_t lr = c0 + t;
            if (lr < rho || lr >= L) continue;
            const int64_t row = static_cast<int64_t>(row0) + (lr - rho);
            *reinterpret_cast<uint4 *>(o + (row * H + h) * D + piece * 8) =
                *reinterpret_cast<const uint4 *>(sm + Os + t * 256 + piece * 16);
        }
        if (!last) save_chunk_state(cbase + ci + 1);
        sync_for_mma();
    }
    tc::cp_async_wait_all();
    if (s_fail) {
        dev_error(pd, kDevErrTimeout, seq, h);
        // let any MMA still in flight drain before the columns are released
        for (int i = 0; i < 4; ++i) tc::mbar_wait(&bars[i], 0, 100000000LL);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tm, 512);
}

}  // namespace

bool tc_supported(bool backward, int dtype, int Dd, int BCc) {
    if (backward) return false;
    return dtype == HARTS_BF16 && Dd == D && BCc == BC;
}

cudaError_t tc_fwd_round(const FwdParams &p, const PlanDev &pd, int32_t base, int32_t n_items,
                         int32_t, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kda_fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(fwd_sm::bytes));
    if (e != cudaSuccess) return e;
    kda_fwd_tc<<<n_items, NT, fwd_sm::bytes, st>>>(p, pd, base);
    return cudaGetLastError();
}

cudaError_t tc_bwd_round(const BwdParams &, const PlanDev &, int32_t, int32_t, int32_t, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace harts
