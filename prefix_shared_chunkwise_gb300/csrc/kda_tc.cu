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
          *vm = reinterpret_cast<float *>(sm + vM), *vpart = reinterpret_cast<float *>(sm + vPart),
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
        const int mid = (nv - 1) / 2;
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
            const int cp = tid & 63, qr = tid >> 6, c2 = 2 * cp, qmid = mid >> 4;
            float s0 = 0.f, s1 = 0.f, ml0 = 0.f, ml1 = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = qr * 16 + u;
                const float2 gg = stage2(sm, SG, t, c2);
                s0 += gg.x; s1 += gg.y;
                if (t == mid) { ml0 = s0; ml1 = s1; }
            }
            vpart[qr * 128 + c2] = s0; vpart[qr * 128 + c2 + 1] = s1;
            if (qr == qmid) { vm[c2] = ml0; vm[c2 + 1] = ml1; }
            if (tid < 64) {
                const uint32_t w = reinterpret_cast<const uint32_t *>(sm + SBeta)[tid];
                const int par = reinterpret_cast<const int *>(sm + SBpar)[tid];
                const uint16_t hb = par ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w & 0xFFFF);
                vbeta[tid] = __bfloat162float(__ushort_as_bfloat16(hb));
            }
            __syncthreads();
            float gam0 = 0.f, gam1 = 0.f, m0 = vm[c2], m1 = vm[c2 + 1], gl0 = 0.f, gl1 = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float p0 = vpart[q * 128 + c2], p1 = vpart[q * 128 + c2 + 1];
                if (q < qr) { gam0 += p0; gam1 += p1; }
                if (q < qmid) { m0 += p0; m1 += p1; }
                gl0 += p0; gl1 += p1;
            }
            if (-m0 > kMaxExpArg || m0 - gl0 > kMaxExpArg || -m1 > kMaxExpArg || m1 - gl1 > kMaxExpArg)
                dev_error(pd, kDevErrDecayRange, seq, c0);
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

// ======================================================================================
// Backward, tensor-core path.  Two kernels:
//  kda_bwd_state_tc : per (sequence, head), chunks in reverse; carries dS (as dS^T in
//                     TMEM) and saves the carry at every chunk end.  Per chunk:
//                       dU^T = dO^T P + (dS'^T e^{Gamma_L-m}) Km^T     (= (P^T dO + Kt dS')^T)
//                       Z^T  = dU^T T                                   (Z = T^T dU)
//                       dS^T <- dS'^T diag(e^{Gamma_L}) + dO^T Qd - (beta Z)^T Kd
//  kda_bwd_grad_tc  : per (chunk, head), all chunks independent; recomputes the chunk
//                     from its saved S and dS' and forms every input gradient.
// T comes from the forward pass's saved chunk record.
// ======================================================================================

// 16-byte piece p of row t of a [64 rows][128 cols] SW128 tile.
__device__ __forceinline__ uint32_t piece64(int t, int p) {
    return static_cast<uint32_t>((p >> 3) * 8192 + t * 128 + (((p & 7) ^ (t & 7)) << 4));
}
// 16-byte piece p of row r of a [128 rows][128 cols] SW128 tile.
__device__ __forceinline__ uint32_t piece128(int r, int p) {
    return static_cast<uint32_t>((p >> 3) * 16384 + r * 128 + (((p & 7) ^ (r & 7)) << 4));
}

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// Stage rows through a per-chunk table of compact rows (-1: past the sequence end);
// rows t < zero_below read as zero.
__device__ void stage_tab(uint8_t *tile, const void *src_, const int *tab, int32_t h, int H,
                          int zero_below) {
    const uint8_t *src = static_cast<const uint8_t *>(src_);
    for (int e = threadIdx.x; e < 64 * 16; e += NT) {
        const int t = e >> 4, pc = e & 15;
        const int row = t < zero_below ? -1 : tab[t];
        const uint8_t *sp = row >= 0 ? src + ((static_cast<int64_t>(row) * H + h) * D * 2 + pc * 16) : src;
        tc::cp_async16(tile + piece64(t, pc), sp, row >= 0 ? 16u : 0u);
    }
}

__device__ void stage_beta_tab(uint8_t *words, int *par, const void *beta, const int *tab,
                               int32_t h, int H) {
    for (int t = threadIdx.x; t < 64; t += NT) {
        const int row = tab[t];
        const int64_t idx = row >= 0 ? static_cast<int64_t>(row) * H + h : 0;
        const uint8_t *sp = static_cast<const uint8_t *>(beta) + (idx & ~int64_t(1)) * 2;
        tc::cp_async4(words + t * 4, sp, row >= 0 ? 4u : 0u);
        par[t] = static_cast<int>(idx & 1);
    }
}

__device__ __forceinline__ float beta_of(const uint8_t *words, const int *par, int t) {
    const uint32_t w = reinterpret_cast<const uint32_t *>(words)[t];
    const uint16_t hb = par[t] ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w & 0xFFFF);
    return __bfloat162float(__ushort_as_bfloat16(hb));
}

__device__ __forceinline__ float2 sw_val2(const uint8_t *tile, int rows, int r, int c) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(tile + tc::sw128_offset(rows, r, c)));
}

// Two-channel cumulative decay over row quarters, thread (cp, qr): channels 2cp, 2cp+1,
// rows 16 qr .. 16 qr + 15.  Pass 1 publishes quarter sums and the local prefix at the
// reference row; after a barrier, gamma2_setup gives the starting offsets, the reference
// value m and Gamma_L of both channels.
struct Gam2 { float gam0, gam1, m0, m1, gl0, gl1; };

__device__ __forceinline__ void gamma2_pass1(const uint8_t *G, int cp, int qr, int mid, float *vpart,
                                             float *vm) {
    const int c2 = 2 * cp;
    float s0 = 0.f, s1 = 0.f, ml0 = 0.f, ml1 = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const int t = qr * 16 + u;
        const float2 gg = sw_val2(G, 64, t, c2);
        s0 += gg.x; s1 += gg.y;
        if (t == mid) { ml0 = s0; ml1 = s1; }
    }
    vpart[qr * 128 + c2] = s0; vpart[qr * 128 + c2 + 1] = s1;
    if (qr == (mid >> 4)) { vm[c2] = ml0; vm[c2 + 1] = ml1; }
}

__device__ __forceinline__ Gam2 gamma2_setup(int cp, int qr, int mid, const float *vpart, const float *vm) {
    const int c2 = 2 * cp, qmid = mid >> 4;
    Gam2 r{0.f, 0.f, vm[c2], vm[c2 + 1], 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float p0 = vpart[q * 128 + c2], p1 = vpart[q * 128 + c2 + 1];
        if (q < qr) { r.gam0 += p0; r.gam1 += p1; }
        if (q < qmid) { r.m0 += p0; r.m1 += p1; }
        r.gl0 += p0; r.gl1 += p1;
    }
    return r;
}

// Cumulative decay pass 1 for thread (c, half): partial sums and the reference row.
__device__ __forceinline__ void gamma_pass1(const uint8_t *G, int c, int half, int mid, float *vt0,
                                            float *vt1, float *vm) {
    float s = 0.f, mref = 0.f;
#pragma unroll 8
    for (int t = half * 32; t < half * 32 + 32; ++t) {
        s += sw_val(G, 64, t, c);
        if (t == mid) mref = s;
    }
    if (half == 0) { vt0[c] = s; vm[c] = mref; } else vt1[c] = s;
}

namespace bws_sm {
constexpr uint32_t RawQ = 0, RawK = 16384, RawG = 32768, dOm = 49152;
constexpr uint32_t Qpm = 65536, Km = 81920, Kdm = 98304, Qdm = 114688;
constexpr uint32_t Pm = 131072, Tm = 139264, dSTs = 147456, dUTs = 180224;
constexpr uint32_t dOm2 = 196608, Tm2 = 212992;          // second buffers (prefetch)
constexpr uint32_t SBeta = 221184, SBpar = SBeta + 256, Vec = SBpar + 256;
constexpr uint32_t vBeta = Vec, vEl = vBeta + 256, vEkt = vEl + 512, vM = vEkt + 512,
                   vPart = vM + 512, vEnd = vPart + 2048;
constexpr uint32_t bytes = vEnd + 1024;
}  // namespace bws_sm

// q, k, g, dO as {128 channels, H, C} with boxes of 64 channels x 64 rows (128-byte
// swizzle, the staging tiles' layout); the saved records as [rows][64] bf16 with 64 x 64
// boxes (a chunk's T).
struct StateMaps {
    CUtensorMap q, k, g, dout, rec_t;
};

__global__ void __launch_bounds__(NT, 1) kda_bwd_state_tc(BwdParams p, PlanDev pd, int32_t round_base,
                                                          const __grid_constant__ StateMaps maps) {
    using namespace bws_sm;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    __shared__ uint64_t bars[5];                  // four MMA groups, staged chunk (TMA)
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ int s_rows[64];
    float *vbeta = reinterpret_cast<float *>(sm + vBeta), *vel = reinterpret_cast<float *>(sm + vEl),
          *vekt = reinterpret_cast<float *>(sm + vEkt), *vm = reinterpret_cast<float *>(sm + vM),
          *vpart = reinterpret_cast<float *>(sm + vPart);
    int *spar = reinterpret_cast<int *>(sm + SBpar);
    const FwdParams &f = p.f;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lg = warp & 3, ch = warp >> 2;
    const int H = f.H;
    const int32_t h = blockIdx.x % H;
    const int32_t seq = pd.round_order[round_base + blockIdx.x / H];
    const int32_t rho = pd.seq_rho[seq], L = rho + pd.seq_nown[seq];
    const int32_t nch = (L + BC - 1) / BC;
    const int32_t src = pd.seq_src[seq], cbase = pd.seq_cbase[seq];
    const uint8_t *rec0 = static_cast<const uint8_t *>(f.chunk_states);
    uint8_t *dch = static_cast<uint8_t *>(p.dchunk);

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) tc::mbar_init(&bars[i], 1);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
    const uint32_t tST = tm, tP = tm + 128, tUT = tm + 192, tZT = tm + 256;
    const int jv = lg * 32 + lane;

    // carry <- d_final (S layout [dk][dv] in memory; TMEM holds dS^T)
    for (int hf = 0; hf < 2; ++hf) {
        float r[32];
        const int cb = ch * 64 + hf * 32;
        const float *df = p.d_final ? p.d_final + (static_cast<int64_t>(seq) * H + h) * D * D : nullptr;
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = df ? df[(cb + j) * D + jv] : 0.f;
        tc::tmem_st32(tST + lane_off + cb, r);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    const int32_t sp_begin = pd.seq_sptr[seq];
    int32_t sp = pd.seq_sptr[seq + 1] - 1;
    // Stage chunk cj's raw q, k, g, beta and (into buffer `b`) dO and the forward's T.
    uint32_t n_tma = 0;                                  // chunks staged by TMA so far (uniform)
    bool tma_pending = false;
    auto stage_chunk = [&](int32_t cj, int b) {
        const int32_t cc0 = cj * BC;
        if (cc0 >= rho && cc0 + BC <= L) {
            // own rows only, full: q, k, g, dO (two 64-channel halves each) and T by TMA
            const int32_t r = pd.seq_row0[seq] + (cc0 - rho);
            tma_pending = true;
            if (tid == 0) {
                uint64_t *bar = &bars[4];
                tc::mbar_expect_tx(bar, 8 * 8192 + 8192);
                const CUtensorMap *mp[4] = {&maps.q, &maps.k, &maps.g, &maps.dout};
                uint8_t *dst[4] = {sm + RawQ, sm + RawK, sm + RawG, sm + (b ? dOm2 : dOm)};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    tc::tma_load_3d(dst[q], mp[q], 0, h, r, bar);
                    tc::tma_load_3d(dst[q] + 8192, mp[q], 64, h, r, bar);
                }
                tc::tma_load_2d(sm + (b ? Tm2 : Tm), &maps.rec_t, 0,
                                static_cast<int>((static_cast<int64_t>(cbase + cj) * H + h) * (kRecBytes / 128) + 2 * D),
                                bar);
            }
            if (tid < 64) s_rows[tid] = r + tid;
            stage_beta_tab(sm + SBeta, spar, f.beta, s_rows, h, H);   // each thread reads only its own entry
            tc::cp_async_commit();
            return;
        }
        if (tid < 64) s_rows[tid] = static_cast<int>(local_row(pd, seq, rho, L, cc0 + tid));
        __syncthreads();
        stage_tab(sm + RawQ, f.q, s_rows, h, H, 0);
        stage_tab(sm + RawK, f.k, s_rows, h, H, 0);
        stage_tab(sm + RawG, f.g, s_rows, h, H, 0);
        stage_tab(sm + (b ? dOm2 : dOm), p.d_o, s_rows, h, H, max(0, rho - cc0));
        stage_beta_tab(sm + SBeta, spar, f.beta, s_rows, h, H);
        const uint8_t *rt = rec0 + (static_cast<int64_t>(cbase + cj) * H + h) * kRecBytes + D * D * 2;
        for (int e = tid; e < 64 * 8; e += NT) {
            const int t = e >> 3, pc = e & 7;
            tc::cp_async16(sm + (b ? Tm2 : Tm) + t * 128 + ((pc ^ (t & 7)) << 4), rt + t * 128 + pc * 16, 16u);
        }
        tc::cp_async_commit();
    };
    stage_chunk(nch - 1, 0);
    for (int32_t ci = nch - 1; ci >= 0; --ci) {
        const uint32_t ph = (nch - 1 - ci) & 1;
        const int32_t c0 = ci * BC, pend = min(c0 + BC, L), g = cbase + ci;
        const int nv = min(BC, L - c0);
        const int mid = (nv - 1) / 2;
        const int buf = (nch - 1 - ci) & 1;
        const uint32_t dOc = buf ? dOm2 : dOm, Tc = buf ? Tm2 : Tm;
        // ---- consumers of the boundary state at this chunk's end add their gradients ----
        if (sp >= sp_begin && pd.state_lpos[sp] == pend) {
            const int32_t cb_ = pd.state_cptr[sp], ce_ = pd.state_cptr[sp + 1];
            for (int hf = 0; hf < 2; ++hf) {
                float r[32];
                const int cb = ch * 64 + hf * 32;
                tc::tmem_ld32(tST + lane_off + cb, r);
                for (int32_t cc = cb_; cc < ce_; ++cc) {
                    const float *di = p.ds_init + (static_cast<int64_t>(pd.state_cons[cc]) * H + h) * D * D;
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] += di[(cb + j) * D + jv];
                }
                tc::tmem_st32(tST + lane_off + cb, r);
            }
            --sp;
        }
        // ---- save the carry dS' (bf16 dS^T) for the gradient kernel ----------------------
        {
            float r0[32], r1[32];
            const int cb = ch * 64;
            tc::tmem_ld32x2(tST + lane_off + cb, r0, tST + lane_off + cb + 32, r1);
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                tc::st_sw128_8(sm + dSTs, 128, jv, cb + j, r0 + j);
                tc::st_sw128_8(sm + dSTs, 128, jv, cb + 32 + j, r1 + j);
            }
        }
        tc::cp_async_wait_all();
        if (tma_pending) {
            if (!tc::mbar_wait(&bars[4], n_tma & 1)) atomicOr(&s_fail, 1);
            ++n_tma;
            tma_pending = false;
        }
        __syncthreads();
        if (s_fail) break;
        {
            uint8_t *dst = dch + (static_cast<int64_t>(g) * H + h) * D * D * 2;
            for (int e = tid; e < 128 * 16; e += NT) {
                const int r = e >> 4, pc = e & 15;
                *reinterpret_cast<uint4 *>(dst + r * 256 + pc * 16) =
                    *reinterpret_cast<const uint4 *>(sm + dSTs + piece128(r, pc));
            }
        }
        // ---- prep: two key channels per thread over a quarter of the rows ---------------
        {
            const int cp = tid & 63, qr = tid >> 6, c2 = 2 * cp;
            gamma2_pass1(sm + RawG, cp, qr, mid, vpart, vm);
            if (tid < 64) vbeta[tid] = beta_of(sm + SBeta, spar, tid);
            __syncthreads();
            Gam2 gs = gamma2_setup(cp, qr, mid, vpart, vm);
            if (-gs.m0 > kMaxExpArg || gs.m0 - gs.gl0 > kMaxExpArg || -gs.m1 > kMaxExpArg ||
                gs.m1 - gs.gl1 > kMaxExpArg)
                dev_error(pd, kDevErrDecayRange, seq, c0);
            const float em0 = __expf(gs.m0), em1 = __expf(gs.m1);
            if (qr == 0) {
                vel[c2] = __expf(gs.gl0); vel[c2 + 1] = __expf(gs.gl1);
                vekt[c2] = __expf(gs.gl0 - gs.m0); vekt[c2 + 1] = __expf(gs.gl1 - gs.m1);
            }
#pragma unroll 4
            for (int u = 0; u < 16; ++u) {
                const int t = qr * 16 + u;
                const float2 kk = sw_val2(sm + RawK, 64, t, c2), qv = sw_val2(sm + RawQ, 64, t, c2),
                             gg = sw_val2(sm + RawG, 64, t, c2);
                const float q0 = qv.x * f.scale, q1 = qv.y * f.scale;
                gs.gam0 += gg.x; gs.gam1 += gg.y;
                const float e10 = __expf(gs.gam0 - gs.m0), e20 = __expf(gs.m0 - gs.gam0);
                const float e11 = __expf(gs.gam1 - gs.m1), e21 = __expf(gs.m1 - gs.gam1);
                st_bf16x2(sm + Qpm, 64, t, c2, q0 * e10, q1 * e11);
                st_bf16x2(sm + Km, 64, t, c2, kk.x * e20, kk.y * e21);
                st_bf16x2(sm + Kdm, 64, t, c2, kk.x * e10 * em0, kk.y * e11 * em1);
                st_bf16x2(sm + Qdm, 64, t, c2, q0 * e10 * em0, q1 * e11 * em1);
            }
        }
        sync_for_mma();
        // raw q, k, g, beta are consumed: prefetch the previous chunk while this one runs
        if (ci > 0) stage_chunk(ci - 1, buf ^ 1);
        if (tid == 0) {
            tc::mma_tile(tP, tc::smem_addr(sm + Qpm), 8192, tc::smem_addr(sm + Km), 8192, 128,
                         tc::idesc_bf16(64, 64), false);
            tc::mma_commit(&bars[0]);
        }
        // carry: bf16 copy scaled by e^{Gamma_L - m} per key channel; TMEM scaled by e^{Gamma_L}
        {
            float r2[2][32];
            tc::tmem_ld32x2(tST + lane_off + ch * 64, r2[0], tST + lane_off + ch * 64 + 32, r2[1]);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int cb = ch * 64 + hf * 32;
                float w[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) { w[j] = r2[hf][j] * vekt[cb + j]; r2[hf][j] *= vel[cb + j]; }
#pragma unroll
                for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + dSTs, 128, jv, cb + j, w + j);
            }
            tc::tmem_st32x2(tST + lane_off + ch * 64, r2[0], tST + lane_off + ch * 64 + 32, r2[1]);
        }
        if (!wait_all(&bars[0], ph, &s_fail)) break;
        // ---- P (M = 64 layout: warp lg holds rows 16 lg .. 16 lg + 15 in lanes 0-15) ------
        {
            float r[32];
            tc::tmem_ld32(tP + lane_off + ch * 32, r);
            if (lane < 16) {
                const int t = lg * 16 + lane;
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = (ch * 32 + j <= t) ? r[j] : 0.f;
#pragma unroll
                for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + Pm, 64, t, ch * 32 + j, r + j);
            }
        }
        sync_for_mma();
        if (tid == 0) {
            tc::mma_op(tUT, tc::Opnd{tc::smem_addr(sm + dOc), 8192, true},
                       tc::Opnd{tc::smem_addr(sm + Pm), 8192, true}, 128, 64, 64, false);
            tc::mma_op(tUT, tc::Opnd{tc::smem_addr(sm + dSTs), 16384, false},
                       tc::Opnd{tc::smem_addr(sm + Km), 8192, false}, 128, 64, 128, true);
            tc::mma_commit(&bars[1]);
        }
        if (!wait_all(&bars[1], ph, &s_fail)) break;
        {
            float r[32];
            tc::tmem_ld32(tUT + lane_off + ch * 32, r);
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + dUTs, 128, jv, ch * 32 + j, r + j);
        }
        sync_for_mma();
        if (tid == 0) {
            tc::mma_op(tZT, tc::Opnd{tc::smem_addr(sm + dUTs), 16384, false},
                       tc::Opnd{tc::smem_addr(sm + Tc), 8192, true}, 128, 64, 64, false);
            tc::mma_commit(&bars[2]);
        }
        if (!wait_all(&bars[2], ph, &s_fail)) break;
        {
            float r[32];
            tc::tmem_ld32(tZT + lane_off + ch * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] *= -vbeta[ch * 32 + j];
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + dUTs, 128, jv, ch * 32 + j, r + j);
        }
        sync_for_mma();
        if (tid == 0) {
            tc::mma_op(tST, tc::Opnd{tc::smem_addr(sm + dOc), 8192, true},
                       tc::Opnd{tc::smem_addr(sm + Qdm), 8192, true}, 128, 128, 64, true);
            tc::mma_op(tST, tc::Opnd{tc::smem_addr(sm + dUTs), 16384, false},
                       tc::Opnd{tc::smem_addr(sm + Kdm), 8192, true}, 128, 128, 64, true);
            tc::mma_commit(&bars[3]);
        }
        if (!wait_all(&bars[3], ph, &s_fail)) break;
    }
    tc::cp_async_wait_all();
    if (tma_pending) drain_wait(&bars[4], n_tma & 1, 1000000000LL, pd, seq, h);   // a staged chunk in flight
    if (!s_fail && (src >= 0 || p.dh0)) {
        float *dst = p.ds_init + (static_cast<int64_t>(seq) * H + h) * D * D;
        for (int hf = 0; hf < 2; ++hf) {
            float r[32];
            const int cb = ch * 64 + hf * 32;
            tc::tmem_ld32(tST + lane_off + cb, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[(cb + j) * D + jv] = r[j];
        }
    }
    if (s_fail) {
        dev_error(pd, kDevErrTimeout, seq, h);
        for (int i = 0; i < 4; ++i) drain_wait(&bars[i], 0, 100000000LL, pd, seq, h);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tm, 512);
}

// Tensor maps of the gradient kernel.  Row tensors (q, k, g, v, dO, in that order) are
// 3-D {D, H, C}, one map per box height 8 << j rows (j = 0..3) of 64 channels; the
// chunk records are 2-D: S^T as 256-byte rows (box 128 x 64), T as 128-byte rows (box
// 64 x 64), dS'^T as 256-byte rows (box 128 x 64).  All use the 128-byte swizzle of the
// MMA operand tiles.
struct GradMaps {
    CUtensorMap rows[5][4];
    CUtensorMap rec_s, rec_t, dch;
};

// Box b (largest first, heights 8 << j rows) of the cover of the 8-row groups [glo, ghi):
// its first group and its height index j.  At most four boxes.
__device__ __forceinline__ void cover_box(int glo, int ghi, int b, int &gi, int &j) {
    gi = glo;
    j = 0;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        j = 3;
        while ((1 << j) > ghi - gi) --j;
        if (x == b) break;
        gi += 1 << j;
    }
}

__device__ __forceinline__ int cover_count(int glo, int ghi) {
    int n = 0;
    for (int gi = glo; gi < ghi; ++n) {
        int j = 3;
        while ((1 << j) > ghi - gi) --j;
        gi += 1 << j;
    }
    return n;
}

namespace bwg_sm {
constexpr uint32_t SemT = 0, dSekT = 32768, dOm = 65536, KQp = 81920, Km = 114688, Tm = 131072;
constexpr uint32_t RV = 139264, RQ = 155648, RK = 172032, RG = 188416, PmS = 204800, TBm = 212992;
constexpr uint32_t SBeta = 221184, SBpar = SBeta + 256, Vec = SBpar + 256;
// fp32 vectors
constexpr uint32_t vBeta = Vec, vM = vBeta + 256, vEm = vM + 512, vEkt = vEm + 512, vEl = vEkt + 512,
                   vT0 = vEl + 512, vT1 = vT0 + 512, vDel = vT1 + 512, vDgl = vDel + 2048,
                   vTot = vDgl + 1024, rZY = vTot + 512, rMA = rZY + 256, vEnd = rMA + 512;
constexpr uint32_t bytes = vEnd + 1024;
}  // namespace bwg_sm

// A work item of the gradient kernel is one (chunk, head); a block takes items in steps
// of the grid size.
struct GradItem {
    int32_t h, g, seq, rho, L, c0, nv, row0, rptr;
};

__device__ __forceinline__ GradItem grad_item(const PlanDev &pd, int32_t chunk_begin, int H, int32_t item) {
    GradItem it;
    it.h = item % H;
    it.g = chunk_begin + item / H;
    it.seq = pd.chunk_seq[it.g];
    it.rho = pd.seq_rho[it.seq];
    it.L = it.rho + pd.seq_nown[it.seq];
    it.c0 = (it.g - pd.seq_cbase[it.seq]) * BC;
    it.nv = min(BC, it.L - it.c0);
    it.row0 = pd.seq_row0[it.seq];
    it.rptr = pd.seq_rptr[it.seq];
    return it;
}

// Staging of the gradient kernel's inputs in three groups, waited for in the order they
// are used: A = q, k, g, beta (the prep); C = v, dO and the forward's T; B = S^T and
// dS'^T.  Row tiles: every 8-row group made only of own rows of the sequence comes by TMA
// (the lanes of warp 0 issue one box each, counted on the group's barrier); the other rows
// (replayed rows, a group cut by the sequence's start or end, zero rows) by cp.async
// through the row table `tab`.
__device__ __forceinline__ void grad_stage_ac(const GradMaps *maps, const void *q, const void *k, const void *g,
                                              const void *v, const void *d_o, const void *beta, GradItem it,
                                              const int *tab, int H, uint8_t *sm, uint64_t *tbar) {
    using namespace bwg_sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int glo = (max(0, it.rho - it.c0) + 7) >> 3, ghi = max(glo, it.nv >> 3);
    const int t_zero = max(0, it.rho - it.c0);        // dO rows below this are zero
    if (warp == 0) {
        const int nb = cover_count(glo, ghi);
        const int z0 = it.row0 + it.c0 - it.rho;       // compact row of local row 0
        if (lane == 0) {
            tc::mbar_expect_tx(&tbar[0], static_cast<uint32_t>(3 * (ghi - glo) * 2048));
            tc::mbar_expect_tx(&tbar[1], static_cast<uint32_t>(2 * (ghi - glo) * 2048 + 8192));
        }
        __syncwarp();
        // jobs: tensor x (q, k, g, v, dO) x box x half; one per lane
        for (int jb = lane; jb < 5 * nb * 2; jb += 32) {
            const int x = jb / (nb * 2), r = jb - x * nb * 2, a = r & 1;
            int gi, j;
            cover_box(glo, ghi, r >> 1, gi, j);
            const uint32_t tile = x == 0 ? RQ : x == 1 ? RK : x == 2 ? RG : x == 3 ? RV : dOm;
            tc::tma_load_3d(sm + tile + a * 8192 + gi * 1024, &maps->rows[x][j], 64 * a, it.h, z0 + 8 * gi,
                            &tbar[x < 3 ? 0 : 1]);
        }
        if (lane == 31) {
            const int64_t rid = static_cast<int64_t>(it.g) * H + it.h;
            tc::tma_load_2d(sm + Tm, &maps->rec_t, 0, static_cast<int>(rid * 320 + 256), &tbar[1]);
        }
    }
    // rows outside the TMA groups, A then C
    for (int x = 0; x < 5; ++x) {
        if (x == 3) {
            stage_beta_tab(sm + SBeta, reinterpret_cast<int *>(sm + SBpar), beta, tab, it.h, H);
            tc::cp_async_commit();
        }
        const uint8_t *src = static_cast<const uint8_t *>(x == 0 ? q : x == 1 ? k : x == 2 ? g : x == 3 ? v : d_o);
        uint8_t *tile = sm + (x == 0 ? RQ : x == 1 ? RK : x == 2 ? RG : x == 3 ? RV : dOm);
        const int zero_below = x == 4 ? t_zero : 0;
        for (int e = tid; e < 64 * 16; e += NT) {
            const int t = e >> 4, pc = e & 15;
            if ((t >> 3) >= glo && (t >> 3) < ghi) continue;
            const int row = t < zero_below ? -1 : tab[t];
            const uint8_t *sp = row >= 0 ? src + ((static_cast<int64_t>(row) * H + it.h) * D * 2 + pc * 16) : src;
            tc::cp_async16(tile + piece64(t, pc), sp, row >= 0 ? 16u : 0u);
        }
    }
    tc::cp_async_commit();
}

__device__ __forceinline__ void grad_stage_b(const GradMaps *maps, GradItem it, int H, uint8_t *sm, uint64_t *bar) {
    using namespace bwg_sm;
    const int lane = threadIdx.x & 31;
    if ((threadIdx.x >> 5) != 0) return;
    const int64_t rid = static_cast<int64_t>(it.g) * H + it.h;
    if (lane == 0) tc::mbar_expect_tx(bar, 4 * 16384);
    __syncwarp();
    if (lane < 4) {
        const int a = lane & 1;
        if (lane < 2)
            tc::tma_load_2d(sm + SemT + a * 16384, &maps->rec_s, 64 * a, static_cast<int>(rid * 160), bar);
        else
            tc::tma_load_2d(sm + dSekT + a * 16384, &maps->dch, 64 * a, static_cast<int>(rid * 128), bar);
    }
}

__global__ void __launch_bounds__(NT, 1) kda_bwd_grad_tc(BwdParams p, PlanDev pd, int32_t chunk_begin,
                                                         int32_t n_items,
                                                         const __grid_constant__ GradMaps maps) {
    using namespace bwg_sm;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    __shared__ uint64_t bars[6];
    __shared__ uint64_t tbar[3];      // staging groups A, C, B (see below)
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ int s_rows[2][64];
    float *vbeta = reinterpret_cast<float *>(sm + vBeta), *vm = reinterpret_cast<float *>(sm + vM),
          *vem = reinterpret_cast<float *>(sm + vEm), *vekt = reinterpret_cast<float *>(sm + vEkt),
          *vel = reinterpret_cast<float *>(sm + vEl), *vt0 = reinterpret_cast<float *>(sm + vT0),
          *vt1 = reinterpret_cast<float *>(sm + vT1), *vdel = reinterpret_cast<float *>(sm + vDel),
          *vdgl = reinterpret_cast<float *>(sm + vDgl), *vtot = reinterpret_cast<float *>(sm + vTot),
          *rzy = reinterpret_cast<float *>(sm + rZY), *rma = reinterpret_cast<float *>(sm + rMA);
    int *spar = reinterpret_cast<int *>(sm + SBpar);
    const FwdParams &f = p.f;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lg = warp & 3, ch = warp >> 2;
    const int H = f.H;
    const int W = 3 * D + 1;
    const int jv = lg * 32 + lane;
    const int c = tid & 127, half = tid >> 7;
    const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;

    auto decode = [&](int32_t item) { return grad_item(pd, chunk_begin, H, item); };
    auto rows_of = [&](const GradItem &it, int *tab) {
        if (tid < 64) tab[tid] = static_cast<int>(local_row(pd, it.seq, it.rho, it.L, it.c0 + tid));
    };
    auto stage_ac = [&](const GradItem &it, const int *tab) {
        grad_stage_ac(&maps, f.q, f.k, f.g, f.v, p.d_o, f.beta, it, tab, H, sm, tbar);
    };
    auto stage_b = [&](const GradItem &it) { grad_stage_b(&maps, it, H, sm, &tbar[2]); };

    if (tid == 0) {
        for (int i = 0; i < 6; ++i) tc::mbar_init(&bars[i], 1);
        for (int i = 0; i < 3; ++i) tc::mbar_init(&tbar[i], 1);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    int32_t item = blockIdx.x;
    GradItem nx{};
    if (item < n_items) {
        nx = decode(item);
        rows_of(nx, s_rows[0]);
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tAP = tm, tGam = tm + 64, tXm = tm + 128, tXq = tm + 192, tP1 = tm + 256,
                   tP2 = tm + 320, tS1 = tm + 384, tS2 = tm + 448;
    if (item < n_items) {
        stage_ac(nx, s_rows[0]);
        stage_b(nx);
    }
    uint32_t ph = 0;
    int32_t cur_seq = 0, cur_h = 0, n_done = 0, n_armed = item < n_items ? 1 : 0;
    for (; item < n_items; item += gridDim.x, ++n_done) {
    ph = n_done & 1;
    const GradItem I = nx;
    const int32_t h = I.h, seq = I.seq, rho = I.rho, c0 = I.c0, row0 = I.row0, rptr = I.rptr;
    cur_seq = seq; cur_h = h;
    const int mid = (I.nv - 1) / 2;
    // local rows [t_own, t_end) of this chunk are own rows of the sequence
    const int t_own = max(0, rho - c0), t_end = I.nv;
    const int32_t nxt = item + gridDim.x;
    int *nrows = s_rows[(n_done + 1) & 1];

    // ---- prep: Gamma (kept in TMEM, lane = key channel), Kp, Qp, Km --------------------
    cp_async_wait_group<1>();
    tc::fence_before_sync();
    if (!wait_all(&tbar[0], ph, &s_fail)) goto done;
    gamma_pass1(sm + RG, c, half, mid, vt0, vt1, vm);
    if (tid < 64) vbeta[tid] = beta_of(sm + SBeta, spar, tid);
    __syncthreads();
    {
        const float m = vm[c], gl = vt0[c] + vt1[c];
        float gam = half ? vt0[c] : 0.f;
        if (-m > kMaxExpArg || m - gl > kMaxExpArg) dev_error(pd, kDevErrDecayRange, seq, c0);
        if (half == 0) { vem[c] = __expf(m); vekt[c] = __expf(gl - m); vel[c] = __expf(gl); }
        float gv[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int t = half * 32 + u;
            const float kk = sw_val(sm + RK, 64, t, c), qq = sw_val(sm + RQ, 64, t, c) * f.scale;
            gam += sw_val(sm + RG, 64, t, c);
            gv[u] = gam;
            const float e1 = __expf(gam - m), e2 = __expf(m - gam);
            st_bf16(sm + KQp, 128, t, c, kk * e1);
            st_bf16(sm + KQp, 128, 64 + t, c, qq * e1);
            st_bf16(sm + Km, 64, t, c, kk * e2);
        }
        tc::tmem_st32(tGam + lane_off + half * 32, gv);   // thread (c, half) sits in lane c
    }
    // ---- d_el = sum_dv S . dS' per key channel (before scaling), two channels per thread --
    cp_async_wait_group<0>();
    if (!tc::mbar_wait(&tbar[1], ph) || !tc::mbar_wait(&tbar[2], ph)) atomicOr(&s_fail, 1);
    __syncthreads();
    if (s_fail) goto done;
    {
        const int pr = tid & 63, qr = tid >> 6;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
        for (int r = qr * 32; r < qr * 32 + 32; ++r) {
            const uint32_t off = tc::sw128_offset(128, r, 2 * pr);
            const float2 sv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm + SemT + off));
            const float2 dv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm + dSekT + off));
            a0 += sv.x * dv.x;
            a1 += sv.y * dv.y;
        }
        vdel[qr * 128 + 2 * pr] = a0;
        vdel[qr * 128 + 2 * pr + 1] = a1;
    }
    __syncthreads();
    // S^T columns * e^{m}, dS'^T columns * e^{Gamma_L - m}, T columns * beta
    for (int e = tid; e < 128 * 16; e += NT) {
        const int r = e >> 4, pc = e & 15;
        for (int which = 0; which < 2; ++which) {
            uint8_t *a = sm + (which ? dSekT : SemT) + piece128(r, pc);
            const float *sc = which ? vekt : vem;
            uint4 w = *reinterpret_cast<uint4 *>(a);
            __nv_bfloat162 *b2 = reinterpret_cast<__nv_bfloat162 *>(&w);
            float v[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 fv = __bfloat1622float2(b2[i]);
                v[2 * i] = fv.x * sc[pc * 8 + 2 * i];
                v[2 * i + 1] = fv.y * sc[pc * 8 + 2 * i + 1];
            }
            w.x = tc::pack_bf16(v[0], v[1]); w.y = tc::pack_bf16(v[2], v[3]);
            w.z = tc::pack_bf16(v[4], v[5]); w.w = tc::pack_bf16(v[6], v[7]);
            *reinterpret_cast<uint4 *>(a) = w;
        }
    }
    for (int e = tid; e < 64 * 8; e += NT) {
        const int t = e >> 3, pc = e & 7;
        const uint32_t off = t * 128 + ((pc ^ (t & 7)) << 4);
        uint4 w = *reinterpret_cast<const uint4 *>(sm + Tm + off);
        __nv_bfloat162 *b2 = reinterpret_cast<__nv_bfloat162 *>(&w);
        float v[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 fv = __bfloat1622float2(b2[i]);
            v[2 * i] = fv.x * vbeta[pc * 8 + 2 * i];
            v[2 * i + 1] = fv.y * vbeta[pc * 8 + 2 * i + 1];
        }
        w.x = tc::pack_bf16(v[0], v[1]); w.y = tc::pack_bf16(v[2], v[3]);
        w.z = tc::pack_bf16(v[4], v[5]); w.w = tc::pack_bf16(v[6], v[7]);
        *reinterpret_cast<uint4 *>(sm + TBm + off) = w;
    }
    sync_for_mma();
    if (tid == 0) {
        tc::mma_tile(tAP, tc::smem_addr(sm + KQp), 16384, tc::smem_addr(sm + Km), 8192, 128,
                     tc::idesc_bf16(128, 64), false);
        // X^T = (S^T e^m) Kp^T = S^T Kd^T
        tc::mma_tile(tS1, tc::smem_addr(sm + SemT), 16384, tc::smem_addr(sm + KQp), 16384, 128,
                     tc::idesc_bf16(128, 64), false);
        tc::mma_commit(&bars[0]);
    }
    if (nxt < n_items) {           // the plan-table loads overlap the MMAs
        nx = decode(nxt);
        rows_of(nx, nrows);
    }
    if (!wait_all(&bars[0], ph, &s_fail)) goto done;
    // epilogues walk this thread's 32 columns in two rolled halves of 16 (code size)
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        const int cb = ch * 32 + hh * 16;
        float r[16];
        // P (lanes 64-127) -> Pm, incl lower
        tc::tmem_ld16(tAP + lane_off + cb, r);
        if (lg >= 2) {
            const int t = jv - 64;
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = (cb + j <= t) ? r[j] : 0.f;
            tc::st_sw128_8(sm + PmS, 64, t, cb, r);
            tc::st_sw128_8(sm + PmS, 64, t, cb + 8, r + 8);
        }
        // Y^T = V^T - X^T -> YT [dv][t] (in RQ; raw q was last read in the prep)
        tc::tmem_ld16(tS1 + lane_off + cb, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = sw_val(sm + RV, 64, cb + j, jv) - r[j];
        tc::st_sw128_8(sm + RQ, 128, jv, cb, r);
        tc::st_sw128_8(sm + RQ, 128, jv, cb + 8, r + 8);
    }
    sync_for_mma();
    if (tid == 0) {
        // U^T = Y^T (T diag(beta))^T
        tc::mma_op(tS1, tc::Opnd{tc::smem_addr(sm + RQ), 16384, false},
                   tc::Opnd{tc::smem_addr(sm + TBm), 8192, false}, 128, 64, 64, false);
        // dU^T = dO^T P + (dS'^T e^{Gamma_L-m}) Km^T
        tc::mma_op(tS2, tc::Opnd{tc::smem_addr(sm + dOm), 8192, true},
                   tc::Opnd{tc::smem_addr(sm + PmS), 8192, true}, 128, 64, 64, false);
        tc::mma_op(tS2, tc::Opnd{tc::smem_addr(sm + dSekT), 16384, false},
                   tc::Opnd{tc::smem_addr(sm + Km), 8192, false}, 128, 64, 128, true);
        tc::mma_commit(&bars[1]);
    }
    if (!wait_all(&bars[1], ph, &s_fail)) goto done;
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        const int cb = ch * 32 + hh * 16;
        float r[16];
        tc::tmem_ld16(tS1 + lane_off + cb, r);
        tc::st_sw128_8(sm + RV, 128, jv, cb, r);            // UTs
        tc::st_sw128_8(sm + RV, 128, jv, cb + 8, r + 8);
        tc::tmem_ld16(tS2 + lane_off + cb, r);
        tc::st_sw128_8(sm + RK, 128, jv, cb, r);            // dUTs
        tc::st_sw128_8(sm + RK, 128, jv, cb + 8, r + 8);
    }
    sync_for_mma();
    if (tid == 0) {
        // Z^T = dU^T T
        tc::mma_op(tS1, tc::Opnd{tc::smem_addr(sm + RK), 16384, false},
                   tc::Opnd{tc::smem_addr(sm + Tm), 8192, true}, 128, 64, 64, false);
        // dP = dO U^T (rows 64-127 of the A operand are padding)
        tc::mma_op(tS2, tc::Opnd{tc::smem_addr(sm + dOm), 8192, false},
                   tc::Opnd{tc::smem_addr(sm + RV), 16384, true}, 128, 64, 128, false);
        // Xm <- dK~ e^{Gamma_L-m} = U (dS' e^{Gamma_L-m})^T, transposed: [dk][s]
        tc::mma_op(tXm, tc::Opnd{tc::smem_addr(sm + dSekT), 16384, true},
                   tc::Opnd{tc::smem_addr(sm + RV), 16384, true}, 128, 64, 128, false);
        // dT' = dU Y^T (padding rows)
        tc::mma_op(tP1, tc::Opnd{tc::smem_addr(sm + RK), 16384, true},
                   tc::Opnd{tc::smem_addr(sm + RQ), 16384, true}, 128, 64, 128, false);
        tc::mma_commit(&bars[2]);
    }
    if (!wait_all(&bars[2], ph, &s_fail)) goto done;
    {
        float acc = 0.f;
        __nv_bfloat16 *dvs = reinterpret_cast<__nv_bfloat16 *>(sm + RV);
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            const int cb = ch * 32 + hh * 16;
            float r[16];
            // Z^T: dv = beta Z staged [t][dv] in RV (U^T is consumed); replay rows go to the
            // replay-gradient buffer; unscaled Z^T tile in RG
            tc::tmem_ld16(tS1 + lane_off + cb, r);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int t = cb + j;
                const float x = vbeta[t] * r[j];
                dvs[t * D + jv] = __float2bfloat16_rn(x);
                if (t < t_own && t < t_end)
                    p.rep_grad[(static_cast<int64_t>(rptr + c0 + t) * H + h) * W + D + jv] = x;
            }
            tc::st_sw128_8(sm + RG, 128, jv, cb, r);
            tc::st_sw128_8(sm + RG, 128, jv, cb + 8, r + 8);
            // dP -> PmS (incl lower)
            tc::tmem_ld16(tS2 + lane_off + cb, r);
            if (lg < 2) {
                const int t = jv;
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = (cb + j <= t) ? r[j] : 0.f;
                tc::st_sw128_8(sm + PmS, 64, t, cb, r);
                tc::st_sw128_8(sm + PmS, 64, t, cb + 8, r + 8);
            }
            // dT = dT' diag(beta), strict lower -> RK (dTm)
            tc::tmem_ld16(tP1 + lane_off + cb, r);
            if (lg < 2) {
                const int t = jv;
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = (cb + j < t) ? r[j] * vbeta[cb + j] : 0.f;
                tc::st_sw128_8(sm + RK, 64, t, cb, r);
                tc::st_sw128_8(sm + RK, 64, t, cb + 8, r + 8);
            }
            // sum_s (dK~ e^{Gamma_L-m})[dk][s] Km[s][dk] for dGamma_L
            tc::tmem_ld16(tXm + lane_off + cb, r);
#pragma unroll
            for (int j = 0; j < 16; ++j) acc += r[j] * sw_val(sm + Km, 64, cb + j, jv);
        }
        vdgl[ch * 128 + jv] = acc;
    }
    sync_for_mma();
    if (tid == 0) {
        // W = dT T^T (padding rows)
        tc::mma_op(tS1, tc::Opnd{tc::smem_addr(sm + RK), 8192, false},
                   tc::Opnd{tc::smem_addr(sm + Tm), 8192, false}, 128, 64, 64, false);
        // diag(Z Y^T) = sum_dv Z (V - Kd S) per row, for dbeta (padding rows)
        tc::mma_op(tS2, tc::Opnd{tc::smem_addr(sm + RG), 16384, true},
                   tc::Opnd{tc::smem_addr(sm + RQ), 16384, true}, 128, 64, 128, false);
        tc::mma_commit(&bars[3]);
    }
    // own rows of dv, coalesced, while the MMAs run
    for (int e = tid; e < 64 * 16; e += NT) {
        const int t = e >> 4, pc = e & 15;
        if (t < t_own || t >= t_end) continue;
        const int64_t row = static_cast<int64_t>(row0) + (c0 + t - rho);
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dv) + (row * H + h) * D + pc * 8) =
            *reinterpret_cast<const uint4 *>(sm + RV + t * 256 + pc * 16);
    }
    if (!wait_all(&bars[3], ph, &s_fail)) goto done;
    {
        float r[32];
        tc::tmem_ld32(tS1 + lane_off + ch * 32, r);
        if (lg < 2) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + RQ, 64, jv, ch * 32 + j, r + j);  // Wm
        }
        tc::tmem_ld32(tS2 + lane_off + ch * 32, r);
        if (lg < 2 && (jv >> 5) == ch) {
            float d = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) d = (j == (jv & 31)) ? r[j] : d;
            rzy[jv] = d;
        }
    }
    sync_for_mma();
    if (tid == 0) {
        // T^T W (padding rows); dM = -T^T W
        tc::mma_op(tS2, tc::Opnd{tc::smem_addr(sm + Tm), 8192, true},
                   tc::Opnd{tc::smem_addr(sm + RQ), 8192, true}, 128, 64, 64, false);
        tc::mma_commit(&bars[4]);
    }
    if (!wait_all(&bars[4], ph, &s_fail)) goto done;
    {
        float r[32], a[32];
        tc::tmem_ld32(tS2 + lane_off + ch * 32, r);
        tc::tmem_ld32(tAP + lane_off + ch * 32, a);
        if (lg < 2) {
            const int t = jv;
            const float bt = vbeta[t];
            float dba = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const bool low = ch * 32 + j < t;
                const float dm = low ? -r[j] : 0.f;
                dba += dm * a[j];
                r[j] = bt * dm;
            }
            rma[ch * 64 + t] = dba;
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + TBm, 64, t, ch * 32 + j, r + j);  // dAm
        }
    }
    sync_for_mma();
    if (tid == 0) {
        // Xq^T = (S e^m) dO^T + Km^T dP^T
        tc::mma_op(tXq, tc::Opnd{tc::smem_addr(sm + SemT), 16384, true},
                   tc::Opnd{tc::smem_addr(sm + dOm), 8192, false}, 128, 64, 128, false);
        tc::mma_op(tXq, tc::Opnd{tc::smem_addr(sm + Km), 8192, true},
                   tc::Opnd{tc::smem_addr(sm + PmS), 8192, false}, 128, 64, 64, true);
        // P1^T = Km^T dA^T
        tc::mma_op(tP1, tc::Opnd{tc::smem_addr(sm + Km), 8192, true},
                   tc::Opnd{tc::smem_addr(sm + TBm), 8192, false}, 128, 64, 64, false);
        // P2^T = (S e^m) Z^T
        tc::mma_op(tP2, tc::Opnd{tc::smem_addr(sm + SemT), 16384, true},
                   tc::Opnd{tc::smem_addr(sm + RG), 16384, true}, 128, 64, 128, false);
        // Xm^T += Kp^T dA + Qp^T dP
        tc::mma_op(tXm, tc::Opnd{tc::smem_addr(sm + KQp), 16384, true},
                   tc::Opnd{tc::smem_addr(sm + TBm), 8192, true}, 128, 64, 64, true);
        tc::mma_op(tXm, tc::Opnd{tc::smem_addr(sm + KQp) + 8192, 16384, true},
                   tc::Opnd{tc::smem_addr(sm + PmS), 8192, true}, 128, 64, 64, true);
        tc::mma_commit(&bars[5]);
    }
    if (!wait_all(&bars[5], ph, &s_fail)) goto done;
    if (nxt < n_items) {
        stage_ac(nx, nrows);
        ++n_armed;
    }
    {
        // thread: key channel dk = jv, rows t = 32 ch .. 32 ch + 31.  dq, dk, dg are staged
        // [t][dk] (dq, dk over S^T, dg over dS'^T: both consumed) for coalesced stores.
        __nv_bfloat16 *dqs = reinterpret_cast<__nv_bfloat16 *>(sm + SemT);
        __nv_bfloat16 *dks = reinterpret_cast<__nv_bfloat16 *>(sm + SemT + 16384);
        __nv_bfloat16 *dgs = reinterpret_cast<__nv_bfloat16 *>(sm + dSekT);
        const int dk = jv;
        const float m = vm[dk];
#pragma unroll 1
        for (int hc = 0; hc < 2; ++hc) {
            const int tb = ch * 32 + hc * 16;
            float xq[16], p1[16], p2[16], xm[16], gm[16];
            tc::tmem_ld16(tXq + lane_off + tb, xq);
            tc::tmem_ld16(tP1 + lane_off + tb, p1);
            tc::tmem_ld16(tP2 + lane_off + tb, p2);
            tc::tmem_ld16(tXm + lane_off + tb, xm);
            tc::tmem_ld16(tGam + lane_off + tb, gm);
            float dgm[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = tb + u;
                const float ep = __expf(gm[u] - m), en = __expf(m - gm[u]);
                // dGamma pairs row and column terms of A and P (and Kt with Gamma_L); they
                // cancel in the suffix sums only if both use the operands the MMAs used,
                // so take Kp, Qp, Km as the rounded tile values.
                const float kp = sw_val(sm + KQp, 128, t, dk), qp = sw_val(sm + KQp, 128, 64 + t, dk),
                            km = sw_val(sm + Km, 64, t, dk);
                const float bt = vbeta[t];
                const float xp = p1[u] - bt * p2[u];
                const float dqv = xq[u] * ep * f.scale;
                const float dkv = xp * ep + xm[u] * en;
                dgm[u] = xq[u] * qp + xp * kp - xm[u] * km;
                dqs[t * D + dk] = __float2bfloat16_rn(dqv);
                dks[t * D + dk] = __float2bfloat16_rn(dkv);
                if (t < t_own && t < t_end)
                    p.rep_grad[(static_cast<int64_t>(rptr + c0 + t) * H + h) * W + dk] = dkv;
            }
            // keep dGamma through TMEM (reuse the Gamma columns)
            {
                uint32_t *uu = reinterpret_cast<uint32_t *>(dgm);
                asm volatile(
                    "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                    "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                    :: "r"(tGam + lane_off + tb), "r"(uu[0]), "r"(uu[1]), "r"(uu[2]), "r"(uu[3]),
                       "r"(uu[4]), "r"(uu[5]), "r"(uu[6]), "r"(uu[7]), "r"(uu[8]), "r"(uu[9]),
                       "r"(uu[10]), "r"(uu[11]), "r"(uu[12]), "r"(uu[13]), "r"(uu[14]), "r"(uu[15])
                    : "memory");
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
        }
        // reverse cumulative sum of dGamma over t, plus dGamma_L
        float dg[32];
        tc::tmem_ld32(tGam + lane_off + ch * 32, dg);
        float run = 0.f;
#pragma unroll
        for (int j = 31; j >= 0; --j) { run += dg[j]; dg[j] = run; }
        if (ch == 1) vtot[dk] = run;
        __syncthreads();
        const float dgl = vdgl[dk] + vdgl[128 + dk] +
                          (vdel[dk] + vdel[128 + dk] + vdel[256 + dk] + vdel[384 + dk]) * vel[dk];
        const float off = (ch == 0 ? vtot[dk] : 0.f) + dgl;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int t = ch * 32 + j;
            const float x = dg[j] + off;
            dgs[t * D + dk] = __float2bfloat16_rn(x);
            if (t < t_own && t < t_end)
                p.rep_grad[(static_cast<int64_t>(rptr + c0 + t) * H + h) * W + 2 * D + dk] = x;
        }
    }
    __syncthreads();
    for (int e = tid; e < 3 * 64 * 16; e += NT) {
        const int which = e >> 10, t = (e >> 4) & 63, pc = e & 15;
        if (t < t_own || t >= t_end) continue;
        const int64_t row = static_cast<int64_t>(row0) + (c0 + t - rho);
        void *dst = which == 0 ? p.dq : (which == 1 ? p.dk : p.dg);
        const uint8_t *srcp = which == 2 ? sm + dSekT : sm + SemT + which * 16384;
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(dst) + (row * H + h) * D + pc * 8) =
            *reinterpret_cast<const uint4 *>(srcp + t * 256 + pc * 16);
    }
    if (tid < 64) {
        const int t = tid;
        // dbeta = sum_dv Z (V - Kd S) + sum_s dM A   (the first sum holds both the beta V
        // and the beta Kd paths of W = T diag(beta) [Kd | V])
        const float db = rzy[t] + rma[t] + rma[64 + t];
        if (t < t_end) {
            if (t >= t_own)
                static_cast<__nv_bfloat16 *>(p.dbeta)[(static_cast<int64_t>(row0) + (c0 + t - rho)) * H + h] =
                    __float2bfloat16_rn(db);
            else
                p.rep_grad[(static_cast<int64_t>(rptr + c0 + t) * H + h) * W + 3 * D] = db;
        }
    }
    tc::fence_smem_to_async();     // SemT / dSekT were read and written by threads
    __syncthreads();
    if (nxt < n_items) stage_b(nx);
    }
done:
    tc::cp_async_wait_all();
    if (s_fail) {
        dev_error(pd, kDevErrTimeout, cur_seq, cur_h);
        for (int i = 0; i < 6; ++i) drain_wait(&bars[i], ph, 100000000LL, pd, cur_seq, cur_h);
        // staging copies still in flight land before the block's shared memory is released
        if (tid == 0)
            for (int j = n_done; j < n_armed; ++j)
                for (int k = 0; k < 3; ++k) drain_wait(&tbar[k], j & 1, 100000000LL, pd, cur_seq, cur_h);
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

cudaError_t tc_bwd_state_round(const BwdParams &p, const PlanDev &pd, int32_t base,
                               int32_t n_items, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_state_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bws_sm::bytes));
    if (e != cudaSuccess) return e;
    StateMaps maps;
    {
        const int H = p.f.H;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(pd.C)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
        const cuuint32_t box[3] = {64, 1, BC};
        const void *src[4] = {p.f.q, p.f.k, p.f.g, p.d_o};
        CUtensorMap *dst[4] = {&maps.q, &maps.k, &maps.g, &maps.dout};
        for (int i = 0; i < 4; ++i)
            if (!encode_bf16(dst[i], src[i], 3, dims, strides, box)) return cudaErrorInvalidValue;
        const int64_t n_rec = pd.n_chunks * H;
        const cuuint64_t rdims[2] = {64, static_cast<cuuint64_t>(n_rec * (kRecBytes / 128))};
        const cuuint64_t rstrides[1] = {128};
        const cuuint32_t rbox[2] = {64, 64};
        if (!encode_bf16(&maps.rec_t, p.f.chunk_states, 2, rdims, rstrides, rbox)) return cudaErrorInvalidValue;
    }
    kda_bwd_state_tc<<<n_items, NT, bws_sm::bytes, st>>>(p, pd, base, maps);
    return cudaGetLastError();
}

namespace {

bool encode(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
            const cuuint32_t *box) {
    return encode_bf16(m, base, rank, dims, strides, box);
}

// [C rows][H heads][D] bf16, boxes of (8 << j) rows of 64 channels, j = 0..3.
bool rows_maps(CUtensorMap *m, const void *base, int H, int64_t C) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(C)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
    for (int j = 0; j < 4; ++j) {
        const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(8 << j)};
        if (!encode(m + j, base, 3, dims, strides, box)) return false;
    }
    return true;
}

// A buffer seen as [n_rows][cols] bf16, boxes of box_rows x 64.
bool flat_map(CUtensorMap *m, const void *base, int64_t n_rows, int cols, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(n_rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    return encode(m, base, 2, dims, strides, box);
}

}  // namespace

cudaError_t tc_bwd_grad(const BwdParams &p, const PlanDev &pd, int32_t chunk_begin,
                        int32_t n_items, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_grad_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bwg_sm::bytes));
    if (e != cudaSuccess) return e;
    if (n_items <= 0) return cudaSuccess;
    const int H = p.f.H;
    const int64_t n_rec = pd.n_chunks * H;
    if (n_rec * (kRecBytes / 128) > INT32_MAX) return cudaErrorInvalidValue;   // TMA coordinates are int32
    GradMaps maps;
    if (!rows_maps(maps.rows[0], p.f.q, H, pd.C) || !rows_maps(maps.rows[1], p.f.k, H, pd.C) ||
        !rows_maps(maps.rows[2], p.f.g, H, pd.C) || !rows_maps(maps.rows[3], p.f.v, H, pd.C) ||
        !rows_maps(maps.rows[4], p.d_o, H, pd.C) ||
        !flat_map(&maps.rec_s, p.f.chunk_states, n_rec * (kRecBytes / 256), 128, 128) ||
        !flat_map(&maps.rec_t, p.f.chunk_states, n_rec * (kRecBytes / 128), 64, 64) ||
        !flat_map(&maps.dch, p.dchunk, n_rec * D, 128, 128))
        return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // persistent: one block per SM, items in steps of the grid size
    kda_bwd_grad_tc<<<min(n_items, nsm), NT, bwg_sm::bytes, st>>>(p, pd, chunk_begin, n_items, maps);
    return cudaGetLastError();
}

}  // namespace harts
