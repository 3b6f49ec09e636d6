// Forward of bf16 packed-tree KDA for no-replay plans (dk = dv = 128, chunk 64): the
// ablation plans whose side branches start from the producer's exact state at the fork,
// a state inside a chunk (page "HARTS ... 精读", section 5.3: the replay ablation hands the
// parent's end state over directly), so slots are emitted inside chunks.  The minimum-call
// and node-wise plans run the two-CTA kernels of kda_seq.cu instead.
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
// Qd = Q e^{Gamma}, Kt = K e^{Gamma_L-Gamma} (m = Gamma_L / 2, half the chunk's total
// log-decay, so no factor exceeds exp(|Gamma_L|/2)), and T = (I + diag(beta) A)^-1 by blocked forward
// substitution in fp32 on the CUDA cores.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "tc_primitives.cuh"
#include "tensor_map.h"

namespace harts {
namespace {

constexpr int D = 128, BC = 64, NT = 256;
// Saved per (chunk, head): S^T [dv][dk] then T [t][s], bf16.
constexpr int64_t kRecBytes = (D * D + BC * BC) * 2;

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
constexpr uint32_t vBeta = Vec, vEl = vBeta + 64 * 4, vGp = vEl + 128 * 4, vM = vGp + 256 * 4,
                   vPart = vM + 128 * 4, vEnd = vPart + 4 * 128 * 4;
constexpr uint32_t bytes = vEnd + 1024;     // + alignment slack
}  // namespace fwd_sm

// fp32 64x64 scratch index with a per-row XOR so that column-wise access is conflict-free.
__device__ __forceinline__ int fidx(int t, int s) { return t * 64 + (s ^ (t & 31)); }

// Element (r, c) of a [rows][*] 128-byte-swizzled bf16 tile.
__device__ __forceinline__ float sw_val(const uint8_t *tile, int rows, int r, int c) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + tc::sw128_offset(rows, r, c)));
}

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
            const float *mrow = Mf + (16 * b + t) * 64;
            const int x = (16 * b + t) & 31;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int j = 0; j < t; j += 2) {
                a0 += mrow[(16 * b + j) ^ x] * col[j];
                if (j + 1 < t) a1 += mrow[(16 * b + j + 1) ^ x] * col[j + 1];
            }
            col[t] = t < s ? 0.f : (t == s ? 1.f : -(a0 + a1));
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) Tf[fidx(16 * b + t, 16 * b + s)] = col[t];
    }
    __syncthreads();
    // off-diagonal blocks: each thread forms four adjacent columns of one row
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
        const int nstrip = (4 - d) * 64;
        if (tid < nstrip) {
            const int j = tid >> 6, i = j + d, t = (tid >> 2) & 15, s0 = (tid & 3) * 4;
            const int rowM = 16 * i + t, xm = rowM & 31;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            for (int kb = j; kb < i; ++kb) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float mv = Mf[rowM * 64 + ((16 * kb + u) ^ xm)];
                    const int rT = 16 * kb + u, xt = rT & 31;
                    const float *tr = Tf + rT * 64;
                    a0 += mv * tr[(16 * j + s0) ^ xt];
                    a1 += mv * tr[(16 * j + s0 + 1) ^ xt];
                    a2 += mv * tr[(16 * j + s0 + 2) ^ xt];
                    a3 += mv * tr[(16 * j + s0 + 3) ^ xt];
                }
            }
            // X_ij kept transposed in the unused upper triangle of Mf
            Mf[fidx(16 * j + s0, rowM)] = a0;
            Mf[fidx(16 * j + s0 + 1, rowM)] = a1;
            Mf[fidx(16 * j + s0 + 2, rowM)] = a2;
            Mf[fidx(16 * j + s0 + 3, rowM)] = a3;
        }
        __syncthreads();
        if (tid < nstrip) {
            const int j = tid >> 6, i = j + d, t = (tid >> 2) & 15, s0 = (tid & 3) * 4;
            const int rowT = 16 * i + t, xt = rowT & 31;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float tv = Tf[rowT * 64 + ((16 * i + u) ^ xt)];
                const int col = 16 * i + u;
                a0 += tv * Mf[fidx(16 * j + s0, col)];
                a1 += tv * Mf[fidx(16 * j + s0 + 1, col)];
                a2 += tv * Mf[fidx(16 * j + s0 + 2, col)];
                a3 += tv * Mf[fidx(16 * j + s0 + 3, col)];
            }
            Tf[fidx(rowT, 16 * j + s0)] = -a0;
            Tf[fidx(rowT, 16 * j + s0 + 1)] = -a1;
            Tf[fidx(rowT, 16 * j + s0 + 2)] = -a2;
            Tf[fidx(rowT, 16 * j + s0 + 3)] = -a3;
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

// Final bounded wait for a copy or product still in flight before the block releases
// its shared memory and TMEM; a wait that runs out is recorded in the plan's error word
// (the host then reports HARTS_EDEVICE), it is never silently dropped.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t phase, long long max_cycles,
                                           const PlanDev &pd, int32_t a, int32_t b) {
    if (!tc::mbar_wait(bar, phase, max_cycles)) dev_error(pd, kDevErrTimeout, a, b);
}

// Make shared-memory writes and TMEM reads of all threads ordered before the next MMA.
__device__ __forceinline__ void sync_for_mma() {
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

// Issue asynchronous copies of one chunk's raw q, k, v, g rows (256 B each) and beta
// into the staging buffer; rows past the sequence end are zero-filled.  `tab` receives
// the chunk's compact rows (-1 past the end); all threads call this.
__device__ void prefetch_chunk(const FwdParams &p, const PlanDev &pd, int32_t seq, int32_t h,
                               int32_t rho, int32_t L, int32_t c0, uint8_t *sm, int *tab) {
    using namespace fwd_sm;
    const int H = p.H;
    if (threadIdx.x < 64) tab[threadIdx.x] = static_cast<int>(local_row(pd, seq, rho, L, c0 + threadIdx.x));
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * 16 * 4; e += NT) {
        const int ten = e >> 10, t = (e >> 4) & 63, piece = e & 15;
        const uint8_t *base = static_cast<const uint8_t *>(ten == 0 ? p.q : ten == 1 ? p.k : ten == 2 ? p.v : p.g);
        const int row = tab[t];
        const uint8_t *src = row >= 0 ? base + ((static_cast<int64_t>(row) * H + h) * D * 2 + piece * 16) : base;
        tc::cp_async16(sm + Stage + ten * 16384 + t * 256 + piece * 16, src, row >= 0 ? 16u : 0u);
    }
    for (int t = threadIdx.x; t < 64; t += NT) {
        const int row = tab[t];
        const int64_t idx = row >= 0 ? static_cast<int64_t>(row) * H + h : 0;
        const uint8_t *src = static_cast<const uint8_t *>(p.beta) + (idx & ~int64_t(1)) * 2;
        tc::cp_async4(sm + SBeta + t * 4, src, row >= 0 ? 4u : 0u);
        reinterpret_cast<int *>(sm + SBpar)[t] = static_cast<int>(idx & 1);
    }
    tc::cp_async_commit();
}

// q, k, v, g as {128 channels, H, C} with boxes of one head's 64 rows, unswizzled: a box
// lands as the staging buffer's row-major [64][128] tile.
struct FwdMaps {
    CUtensorMap t[4];
};

// A chunk of own rows only, and full: staged by four TMA boxes instead of row gathers.
__device__ __forceinline__ bool tma_chunk(int32_t rho, int32_t L, int32_t c0) { return c0 >= rho && c0 + BC <= L; }

__device__ void prefetch_chunk_tma(const FwdParams &p, const FwdMaps &maps, int32_t h, int32_t row0, int32_t rho,
                                   int32_t c0, uint8_t *sm, uint64_t *bar) {
    using namespace fwd_sm;
    const int H = p.H;
    const int32_t r = row0 + (c0 - rho);
    if (threadIdx.x == 0) {
        tc::mbar_expect_tx(bar, 4 * 16384);
#pragma unroll
        for (int ten = 0; ten < 4; ++ten) tc::tma_load_3d(sm + Stage + ten * 16384, &maps.t[ten], 0, h, r, bar);
    }
    if (threadIdx.x < 64) {
        const int64_t idx = (static_cast<int64_t>(r) + threadIdx.x) * H + h;
        const uint8_t *src = static_cast<const uint8_t *>(p.beta) + (idx & ~int64_t(1)) * 2;
        tc::cp_async4(sm + SBeta + threadIdx.x * 4, src, 4u);
        reinterpret_cast<int *>(sm + SBpar)[threadIdx.x] = static_cast<int>(idx & 1);
    }
    tc::cp_async_commit();
}

__device__ __forceinline__ float2 stage2(const uint8_t *sm, uint32_t off, int t, int c) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm + off + t * 256 + c * 2));
}

// Two adjacent columns (col even) of one row of a SW128 tile, packed into one 4-byte store.
__device__ __forceinline__ void st_bf16x2(uint8_t *tile, int rows, int row, int col, float a, float b) {
    *reinterpret_cast<uint32_t *>(tile + tc::sw128_offset(rows, row, col)) = tc::pack_bf16(a, b);
}

// kInner: the plan may put slots inside a chunk (no-replay plans); the minimum-call and
// node-wise plans never do, and their instance carries none of that code.
template <bool kInner>
__global__ void __launch_bounds__(NT, 1) kda_fwd_tc(FwdParams p, PlanDev pd, int32_t round_base,
                                                    const __grid_constant__ FwdMaps maps) {
    using namespace fwd_sm;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    __shared__ uint64_t bars[5];                  // four MMA groups, staged chunk (TMA)
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ int s_rows[64];
    float *vbeta = reinterpret_cast<float *>(sm + vBeta), *vel = reinterpret_cast<float *>(sm + vEl),
          *vpart = reinterpret_cast<float *>(sm + vPart),
          *vgp = reinterpret_cast<float *>(sm + vGp);
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

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) tc::mbar_init(&bars[i], 1);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    __syncthreads();
    uint32_t n_tma = 0;                                  // chunks staged by TMA so far (uniform)
    bool tma_pending = tma_chunk(rho, L, 0);
    if (tma_pending) prefetch_chunk_tma(p, maps, h, row0, rho, 0, sm, &bars[4]);
    else prefetch_chunk(p, pd, seq, h, rho, L, 0, sm, s_rows);
    tc::fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
    const uint32_t tST = tm, tAP = tm + 128, tWk = tm + 192, tUT = tm + 256, tOT = tm + 320;
    const int jv = lg * 32 + lane;                       // this thread's TMEM lane

    // Copy the bf16 S^T tile (SW128) to a saved chunk state, [dv][dk] row-major, 16 B per thread.
    auto save_chunk_state = [&](int32_t chunk_index) {
        if (!cst) return;
        uint8_t *dst = cst + (static_cast<int64_t>(chunk_index) * H + h) * kRecBytes;
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
    for (int32_t ci = 0; ci < nch; ++ci) {
        const uint32_t ph = ci & 1;
        const int32_t c0 = ci * BC;
        const int nv = min(BC, L - c0);
        tc::cp_async_wait_all();
        if (tma_pending) {
            if (!tc::mbar_wait(&bars[4], n_tma & 1)) atomicOr(&s_fail, 1);
            ++n_tma;
            tma_pending = false;
        }
        __syncthreads();
        if (s_fail) break;
        // ---- prep: cumulative decay, scaled operands (from the staged raw tiles) ----------
        // thread: key channels c2, c2 + 1; rows 16 qr .. 16 qr + 15
        {
            const int cp = tid & 63, qr = tid >> 6, c2 = 2 * cp;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float2 gg = stage2(sm, SG, qr * 16 + u, c2);
                s0 += gg.x; s1 += gg.y;
            }
            vpart[qr * 128 + c2] = s0; vpart[qr * 128 + c2 + 1] = s1;
            if (tid < 64) {
                const uint32_t w = reinterpret_cast<const uint32_t *>(sm + SBeta)[tid];
                const int par = reinterpret_cast<const int *>(sm + SBpar)[tid];
                const uint16_t hb = par ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w & 0xFFFF);
                vbeta[tid] = __bfloat162float(__ushort_as_bfloat16(hb));
            }
            __syncthreads();
            float gam0 = 0.f, gam1 = 0.f, gl0 = 0.f, gl1 = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float p0 = vpart[q * 128 + c2], p1 = vpart[q * 128 + c2 + 1];
                if (q < qr) { gam0 += p0; gam1 += p1; }
                gl0 += p0; gl1 += p1;
            }
            const float m0 = 0.5f * gl0, m1 = 0.5f * gl1;        // the reference: Gamma_L / 2
            if (-m0 > kMaxExpArg || -m1 > kMaxExpArg) dev_error(pd, kDevErrDecayRange, seq, c0);
            const float em0 = __expf(m0), ekt0 = __expf(gl0 - m0), em1 = __expf(m1), ekt1 = __expf(gl1 - m1);
            if (qr == 0) { vel[c2] = __expf(gl0); vel[c2 + 1] = __expf(gl1); }
            const bool lo = lane < 16;    // half-warps store even / odd rows of the transposed tiles
#pragma unroll
            for (int grp = 0; grp < 2; ++grp) {
                const int t0 = qr * 16 + grp * 8;
                float bkd0[8], bkd1[8], bv0[8], bv1[8], kt0[8], kt1[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = t0 + u;
                    const float2 kk = stage2(sm, SK, t, c2), qv = stage2(sm, SQ, t, c2),
                                 vv = stage2(sm, SV, t, c2), gg = stage2(sm, SG, t, c2);
                    const float bb = vbeta[t], q0 = qv.x * p.scale, q1 = qv.y * p.scale;
                    gam0 += gg.x; gam1 += gg.y;
                    const float e10 = __expf(gam0 - m0), e20 = __expf(m0 - gam0);
                    const float e11 = __expf(gam1 - m1), e21 = __expf(m1 - gam1);
                    st_bf16x2(sm + KQp, 128, t, c2, kk.x * e10, kk.y * e11);
                    st_bf16x2(sm + KQp, 128, 64 + t, c2, q0 * e10, q1 * e11);
                    st_bf16x2(sm + Km, 64, t, c2, kk.x * e20, kk.y * e21);
                    st_bf16x2(sm + Qd, 64, t, c2, q0 * e10 * em0, q1 * e11 * em1);
                    bkd0[u] = bb * kk.x * e10 * em0; bkd1[u] = bb * kk.y * e11 * em1;
                    bv0[u] = bb * vv.x; bv1[u] = bb * vv.y;
                    kt0[u] = kk.x * e20 * ekt0; kt1[u] = kk.y * e21 * ekt1;
                }
                float a[8], b[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) { a[u] = lo ? bkd0[u] : bkd1[u]; b[u] = lo ? bkd1[u] : bkd0[u]; }
                tc::st_sw128_8(sm + BKdT, 128, c2 + (lo ? 0 : 1), t0, a);
                tc::st_sw128_8(sm + BKdT, 128, c2 + (lo ? 1 : 0), t0, b);
#pragma unroll
                for (int u = 0; u < 8; ++u) { a[u] = lo ? bv0[u] : bv1[u]; b[u] = lo ? bv1[u] : bv0[u]; }
                tc::st_sw128_8(sm + BVT, 128, c2 + (lo ? 0 : 1), t0, a);
                tc::st_sw128_8(sm + BVT, 128, c2 + (lo ? 1 : 0), t0, b);
#pragma unroll
                for (int u = 0; u < 8; ++u) { a[u] = lo ? kt0[u] : kt1[u]; b[u] = lo ? kt1[u] : kt0[u]; }
                tc::st_sw128_8(sm + KtT, 128, c2 + (lo ? 0 : 1), t0, a);
                tc::st_sw128_8(sm + KtT, 128, c2 + (lo ? 1 : 0), t0, b);
            }
        }
        sync_for_mma();
        if (tid == 0) {
            tc::mma_tile(tAP, tc::smem_addr(sm + KQp), 128 * 128, tc::smem_addr(sm + Km), 64 * 128,
                         128, tc::idesc_bf16(128, 64), false);
            tc::mma_tile(tOT, tc::smem_addr(sm + STs), 128 * 128, tc::smem_addr(sm + Qd), 64 * 128,
                         128, tc::idesc_bf16(128, 64), false);
            tc::mma_commit(&bars[0]);
        }
        // the staging buffer is free: fetch the next chunk while this one computes
        if (ci + 1 < nch) {
            tma_pending = tma_chunk(rho, L, c0 + BC);
            if (tma_pending) prefetch_chunk_tma(p, maps, h, row0, rho, c0 + BC, sm, &bars[4]);
            else prefetch_chunk(p, pd, seq, h, rho, L, c0 + BC, sm, s_rows);
        }
        // ---- scale the TMEM state by e^{Gamma_L} per key channel (used by MMA7) -----------
        {
            float r0[32], r1[32];
            const int cb = ch * 64;
            tc::tmem_ld32x2(tST + lane_off + cb, r0, tST + lane_off + cb + 32, r1);
#pragma unroll
            for (int j = 0; j < 32; ++j) { r0[j] *= vel[cb + j]; r1[j] *= vel[cb + 32 + j]; }
            tc::tmem_st32x2(tST + lane_off + cb, r0, tST + lane_off + cb + 32, r1);
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
            if (cst) {
                uint8_t *dst = cst + (static_cast<int64_t>(cbase + ci) * H + h) * kRecBytes + D * D * 2;
                uint4 w0, w1;
                w0.x = tc::pack_bf16(r[0], r[1]); w0.y = tc::pack_bf16(r[2], r[3]);
                w0.z = tc::pack_bf16(r[4], r[5]); w0.w = tc::pack_bf16(r[6], r[7]);
                w1.x = tc::pack_bf16(r[8], r[9]); w1.y = tc::pack_bf16(r[10], r[11]);
                w1.z = tc::pack_bf16(r[12], r[13]); w1.w = tc::pack_bf16(r[14], r[15]);
                *reinterpret_cast<uint4 *>(dst + t * 128 + s0 * 2) = w0;
                *reinterpret_cast<uint4 *>(dst + t * 128 + s0 * 2 + 16) = w1;
            }
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
        // ---- slots inside this chunk (no-replay plans) ------------------------------------
        // The state after the chunk's first r rows is diag(e^{Gamma_{r-1}}) S +
        // (K e^{Gamma_{r-1} - Gamma})_{<r}^T U_{<r}.  TMEM holds S^T diag(e^{Gamma_L}) until
        // the update MMA below, and KtT = (K e^{Gamma_L - Gamma})^T, so its transpose is
        // (S^T diag(e^{Gamma_L}) + U_{<r}^T Kt_{<r}) diag(e^{Gamma_{r-1} - Gamma_L}), the last
        // factor from the raw g rows r .. nv-1 (read through the plan: the row table
        // already holds the next chunk).  Thread (dv = jv, 64 key channels per half).
        while (kInner && sp < sp_end && pd.state_lpos[sp] < min(c0 + BC, L)) {
            const int r = pd.state_lpos[sp] - c0;       // 1 <= r < nv
            if (tid < 128) {
                float sum = 0.f;
                for (int t = r; t < nv; ++t) {
                    const int64_t row = local_row(pd, seq, rho, L, c0 + t);
                    sum += __bfloat162float(static_cast<const __nv_bfloat16 *>(p.g)[(row * H + h) * D + tid]);
                }
                vgp[tid] = __expf(-sum);
            }
            __syncthreads();
            float *dst = p.states + (static_cast<int64_t>(sp) * H + h) * D * D;
            for (int hf = 0; hf < 2; ++hf) {
                float rr[32];
                const int cb = ch * 64 + hf * 32;
                tc::tmem_ld32(tST + lane_off + cb, rr);
                for (int t = 0; t < r; ++t) {
                    const float u = sw_val(sm + UTs, 128, jv, t);
#pragma unroll
                    for (int j = 0; j < 32; ++j) rr[j] += u * sw_val(sm + KtT, 128, cb + j, t);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) dst[(cb + j) * D + jv] = rr[j] * vgp[cb + j];
            }
            ++sp;
            sync_for_mma();     // TMEM reads and vgp done before the next slot or the update MMA
        }
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
        const int32_t pend = min(c0 + BC, L);     // a slot may sit at the sequence end
        const bool slot = sp < sp_end && pd.state_lpos[sp] == pend;
        const bool last = ci == nch - 1;
        float rr2[2][32];
        tc::tmem_ld32x2(tST + lane_off + ch * 64, rr2[0], tST + lane_off + ch * 64 + 32, rr2[1]);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float (&r)[32] = rr2[hf];
            const int cb = ch * 64 + hf * 32;
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
    if (tma_pending) drain_wait(&bars[4], n_tma & 1, 1000000000LL, pd, seq, h);   // a staged chunk in flight
    if (s_fail) {
        dev_error(pd, kDevErrTimeout, seq, h);
        // let any MMA still in flight drain before the columns are released
        for (int i = 0; i < 4; ++i) drain_wait(&bars[i], 0, 100000000LL, pd, seq, h);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tm, 512);
}

}  // namespace

bool tc_supported(bool, int dtype, int Dd, int BCc) {
    return dtype == HARTS_BF16 && Dd == D && BCc == BC;
}

cudaError_t tc_fwd_round(const FwdParams &p, const PlanDev &pd, int32_t base, int32_t n_items,
                         int32_t, cudaStream_t st) {
    const bool inner = (pd.flags & HARTS_PLAN_NOREPLAY) != 0;
    cudaError_t e = cudaFuncSetAttribute(inner ? kda_fwd_tc<true> : kda_fwd_tc<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(fwd_sm::bytes));
    if (e != cudaSuccess) return e;
    FwdMaps maps;
    {
        const int H = p.H;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(pd.C)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
        const cuuint32_t box[3] = {D, 1, BC};
        const void *src[4] = {p.q, p.k, p.v, p.g};
        for (int i = 0; i < 4; ++i)
            if (!encode_bf16(&maps.t[i], src[i], 3, dims, strides, box, false)) return cudaErrorInvalidValue;
    }
    if (inner)
        kda_fwd_tc<true><<<n_items, NT, fwd_sm::bytes, st>>>(p, pd, base, maps);
    else
        kda_fwd_tc<false><<<n_items, NT, fwd_sm::bytes, st>>>(p, pd, base, maps);
    return cudaGetLastError();
}

}  // namespace harts
