// The two sequential passes of bf16 packed-tree KDA on sm_103a (dk = dv = 128, chunk 64),
// forward and backward state pass, each with two CTAs per SM.
//
// One CTA (256 threads) per sequence of a round and group of 1, 2 or 4 of its heads, the
// heads in turn and each head's chunks in order (page "HARTS ... 精读", section 4.3, KDA
// paragraph: one packed call per round, each sequence resuming from its boundary state;
// section 4.2: a side branch first replays its ancestor rows back to the chunk boundary,
// which update the state but write no output).  Each CTA holds about 104 KB of shared
// memory and 256 TMEM columns, so two CTAs share an SM and one's elementwise phases run
// while the other waits on its products or loads.  The next head's first chunk is fetched
// while the current head's last runs, so a CTA sets up once for several short sequences.
//
// Chunk math (local rows t, s; gamma = cumulative log-decay from the chunk start, m = half
// the chunk's total log-decay Gamma_L, per key channel):
//   Kp = K e^{gamma-m}, Qp = scale Q e^{gamma-m}, Km = K e^{m-gamma}
//   [A; P] = [Kp; Qp] Km^T          A strictly lower, P lower with the diagonal
//   T = (I + diag(beta) A)^-1,  Tb = T diag(beta)
//   R = S^T diag(e^m)               (the state as the products use it; S^T: lane = value channel)
//   U^T = V^T Tb^T - R (Kp^T Tb^T)  (= (W_v - W_k S)^T)
//   O^T = R Qp^T + U^T P^T          (= (Q e^gamma S + P U)^T)
//   S'^T = (R + U^T Km) diag(e^{Gamma_L - m})
// so no operand needs e^{-gamma} alone except Km (bounded by e^{|m - gamma|}) and the state
// is never rescaled in place: the next chunk's R is S'^T diag(e^{m'}), formed once per chunk
// as the fp32 state leaves TMEM and goes back in.
//
// Each chunk's record for the gradient pass holds the bf16 R the products used (not S^T)
// and T, so the gradient pass needs neither m-scaling of the state nor an inversion; R
// (forward) and Q' (state pass) leave shared memory by tiled TMA stores.
//
// TMEM (256 columns): S = R in fp32 (128), R as bf16 pairs, the A operand of two products
// (64), one work tile W (64) that holds in turn [A; P], Kp^T Tb^T, U^T and O^T.
// Shared memory: KQ [Kp; Qp] (raw k and q land there), Km, V (then U^T, then the output
// staging), a 16 KB scratch (diag(beta) A in fp32 for the inversion, then Tb and P), and
// the next chunk's raw g.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "tc_primitives.cuh"
#include "tensor_map.h"
#include "kda_stage.cuh"

namespace harts {
namespace {

constexpr int D = 128, BC = 64, NT = 256;
// Record per (chunk, head) read by the backward: S^T at the chunk start [dv][dk], then
// T [t][s], bf16.
constexpr int64_t kRecBytes = (D * D + BC * BC) * 2;

namespace f2 {
constexpr uint32_t KQ = 0;          // [128 rows][128] SW128, atoms of 16 KB: rows 0-63 Kp, 64-127 Qp
constexpr uint32_t KM = 32768;      // [64][128] SW128, atoms of 8 KB: Km
constexpr uint32_t VV = 49152;      // raw v [64][128] (atoms 8 KB) -> U^T [128][64] -> O staging [64][128]
constexpr uint32_t SC = 65536;      // fp32 [64][64] diag(beta) A -> T; then Tb [64][64] bf16 and P at +8 KB
constexpr uint32_t GP = 81920;      // next chunk's raw g [64][128], atoms of 8 KB
constexpr uint32_t VQS = 98304;     // fp32 [16][128] sums of g over 4-row groups, then exclusive prefixes
constexpr uint32_t VM = VQS + 8704;         // fp32 [2][128] m log2(e) (by chunk parity)
constexpr uint32_t VEM = VM + 1024;       // fp32 [2][128] e^m
constexpr uint32_t VEG = VEM + 1024;      // fp32 [2][128] e^{Gamma_L - m}
constexpr uint32_t VBETA = VEG + 1024;    // fp32 [64] beta of the current chunk
constexpr uint32_t END = VBETA + 256;
constexpr uint32_t bytes = END + 1024;    // + alignment slack
}  // namespace f2

// fp32 [64][64] scratch index: row t's aligned groups of 4 columns are XOR-permuted by
// t % 8, so float4 accesses stay contiguous while the fragment loads of the 16 x 8 tiles
// below fall into distinct banks.
__device__ __forceinline__ int fx(int t, int s) { return t * 64 + (s ^ ((t & 7) << 2)); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void unpack8(const uint4 &w, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u[i]));
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(tc::pack_bf16(f[0], f[1]), tc::pack_bf16(f[2], f[3]), tc::pack_bf16(f[4], f[5]),
                      tc::pack_bf16(f[6], f[7]));
}
// 16-byte chunk j (8 channels) of row t of a [rows][64]-column SW128 atom.
__device__ __forceinline__ uint32_t chunk_off(int t, int j) {
    return static_cast<uint32_t>(t * 128 + ((j ^ (t & 7)) << 4));
}

__device__ __forceinline__ uint32_t tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// Warp-level D += A B on a 16 x 8 x 8 tile, TF32 operands and fp32 accumulation; fragment
// (gid = lane / 4, tig = lane % 4): a = A[gid][tig], A[gid+8][tig], A[gid][tig+4],
// A[gid+8][tig+4]; b = B[tig][gid], B[tig+4][gid]; d = D[gid][2tig], D[gid][2tig+1],
// D[gid+8][2tig], D[gid+8][2tig+1].
__device__ __forceinline__ void mma16x8x8(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}


struct Maps2 {
    RowMaps q, k, v, g;
    CUtensorMap rec_s;           // chunk records as [rows of 256 B], boxes of 64 columns x 128 rows
};

// Pass A of a chunk whose raw g sits in the SW128 tile `g` ([64][128], atoms of 8 KB): sums
// of g over 4-row groups, turned into exclusive prefixes (vqs, natural log units), the
// reference m = Gamma_L / 2 (half the chunk's total log-decay, so that every row's exponent
// gamma - m lies within |Gamma_L| / 2 of zero), m log2(e), e^m, e^{Gamma_L - m} (into slot b
// of vm / vem / veg), and beta (raw bf16 bits from this thread if tid < 64).  Records the
// decay-range error when an exponent would leave the representable range.
// Thread: 8 channels (group cg = tid % 16) x 4 rows (group rg = tid / 16).
__device__ __forceinline__ void chunk_pass_a(uint8_t *sm, const uint8_t *g, float *vqs, float *vbeta,
                                             uint8_t *vm, uint8_t *vem, uint8_t *veg, int b, uint16_t braw,
                                             const PlanDev &pd, int32_t seq, int32_t c0) {
    const int tid = threadIdx.x;
    const int cg = tid & 15, rg = tid >> 4;
    float sacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = 4 * rg + u;
        float gv[8];
        unpack8(*reinterpret_cast<const uint4 *>(g + (cg >> 3) * 8192 + chunk_off(t, cg & 7)), gv);
#pragma unroll
        for (int i = 0; i < 8; ++i) sacc[i] += gv[i];
    }
    float4 *q4 = reinterpret_cast<float4 *>(vqs + rg * 128 + 8 * cg);
    q4[0] = make_float4(sacc[0], sacc[1], sacc[2], sacc[3]);
    q4[1] = make_float4(sacc[4], sacc[5], sacc[6], sacc[7]);
    if (tid < 64) vbeta[tid] = __bfloat162float(__ushort_as_bfloat16(braw));
    __syncthreads();
    if (tid < 128) {
        float run = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float x = vqs[r * 128 + tid];
            vqs[r * 128 + tid] = run;
            run += x;
        }
        // reference m = Gamma_L / 2: every row's exponent gamma - m stays within |Gamma_L| / 2
        const float m = 0.5f * run;
        if (-m > kMaxExpArg) dev_error(pd, kDevErrDecayRange, seq, c0);
        reinterpret_cast<float *>(vm)[b * 128 + tid] = m * kLog2e;
        reinterpret_cast<float *>(vem)[b * 128 + tid] = ex2(m * kLog2e);
        reinterpret_cast<float *>(veg)[b * 128 + tid] = ex2((run - m) * kLog2e);
    }
}

// Pass B: Kp = K e^{Gamma-m} and Qp = scale Q e^{Gamma-m} in place over the raw k and q
// rows of the [Kp; Qp] tile, Km = K e^{m-Gamma} into `km` (which may be the g tile itself:
// each element is read before the same thread overwrites it).  Thread as in pass A.
__device__ __forceinline__ void chunk_pass_b(uint8_t *kq, const uint8_t *g, uint8_t *km, const float *vqs,
                                             const float *vm2, float sc) {
    const int tid = threadIdx.x;
    const int cg = tid & 15, rg = tid >> 4, j = cg & 7;
    const float4 *p4 = reinterpret_cast<const float4 *>(vqs + rg * 128 + 8 * cg);
    const float4 *m4 = reinterpret_cast<const float4 *>(vm2 + 8 * cg);
    const float4 pa = p4[0], pb = p4[1], ma = m4[0], mb = m4[1];
    float gam[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
    const float m2[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
    uint8_t *kqa = kq + (cg >> 3) * 16384;
    const uint8_t *ga = g + (cg >> 3) * 8192;
    uint8_t *kma = km + (cg >> 3) * 8192;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = 4 * rg + u;
        const uint32_t o64 = chunk_off(t, j), oq = chunk_off(64 + t, j);
        float gv[8], kv[8], qv[8], kp[8], qp[8], kmv[8];
        unpack8(*reinterpret_cast<const uint4 *>(ga + o64), gv);
        unpack8(*reinterpret_cast<const uint4 *>(kqa + o64), kv);
        unpack8(*reinterpret_cast<const uint4 *>(kqa + oq), qv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            gam[i] += gv[i];
            const float x = fmaf(gam[i], kLog2e, -m2[i]);
            const float e1 = ex2(x), e2 = ex2(-x);
            kp[i] = kv[i] * e1;
            qp[i] = sc * qv[i] * e1;
            kmv[i] = kv[i] * e2;
        }
        *reinterpret_cast<uint4 *>(kqa + o64) = pack8(kp);
        *reinterpret_cast<uint4 *>(kqa + oq) = pack8(qp);
        *reinterpret_cast<uint4 *>(kma + o64) = pack8(kmv);
    }
}

__device__ __forceinline__ bool wait_all2(uint64_t *bar, uint32_t phase, int *s_fail) {
    if (threadIdx.x == 0 && !tc::mbar_wait(bar, phase)) *s_fail = 1;
    __syncthreads();
    tc::fence_after_sync();
    return *reinterpret_cast<volatile int *>(s_fail) == 0;
}

__device__ __forceinline__ bool wait_data(uint64_t *bar, uint32_t phase, int *s_fail) {
    if (threadIdx.x == 0 && !tc::mbar_wait(bar, phase)) *s_fail = 1;
    __syncthreads();
    return *reinterpret_cast<volatile int *>(s_fail) == 0;
}

__device__ __forceinline__ void sync_mma() {
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

// Thread 0 waits for a barrier phase (bounded) without a block barrier of its own; the next
// sync_check / sync_mma_check publishes the outcome, so several waits share one barrier.
__device__ __forceinline__ void poll0(uint64_t *bar, uint32_t phase, int *s_fail) {
    if (threadIdx.x == 0 && *reinterpret_cast<volatile int *>(s_fail) == 0 && !tc::mbar_wait(bar, phase)) *s_fail = 1;
}
__device__ __forceinline__ bool sync_check(int *s_fail) {
    __syncthreads();
    return *reinterpret_cast<volatile int *>(s_fail) == 0;
}
__device__ __forceinline__ bool sync_mma_check(int *s_fail) {
    sync_mma();
    return *reinterpret_cast<volatile int *>(s_fail) == 0;
}

// In-place inversion of the unit lower-triangular I + M held (M strictly lower) in the fp32
// scratch F.  The four diagonal 16 x 16 blocks by forward substitution (one column per
// thread, fp32); then the blocks below them by T_ij = -T_ii (M_ij T_jj): first the 16-row
// blocks (1, 0) and (3, 2), then the 32-row block (rows 32-63, columns 0-31), each product
// on warp-level TF32 tiles, the inner product parked in the unused upper triangle.
__device__ __forceinline__ void invert64(float *F) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
    float col[16];
    if (tid < 64) {
        const int b = tid >> 4, s = tid & 15;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * b + i;
            float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < i; ++j) a[j & 3] += F[fx(r, 16 * b + j)] * col[j];
            col[i] = i < s ? 0.f : (i == s ? 1.f : -((a[0] + a[1]) + (a[2] + a[3])));
        }
        // a block's 16 columns are one half-warp's: the warp's reads finish before its writes
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 16; ++i) F[fx(16 * b + i, 16 * b + s)] = col[i];
    }
    __syncthreads();
    // blocks (1, 0) and (3, 2): warps 0-3, warp -> (pair, 8-column tile)
    const int bi = 2 * (warp >> 1) + 1, bj = bi - 1, nt = warp & 1;
    if (warp < 4) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        const int c = 8 * nt + gid;                       // column of T_jj this lane's b reads
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
            if (kt < nt) continue;                        // T_jj is zero above its diagonal
            const int k0 = 8 * kt;
            const uint32_t a[4] = {tf32(F[fx(16 * bi + gid, 16 * bj + k0 + tig)]),
                                   tf32(F[fx(16 * bi + gid + 8, 16 * bj + k0 + tig)]),
                                   tf32(F[fx(16 * bi + gid, 16 * bj + k0 + tig + 4)]),
                                   tf32(F[fx(16 * bi + gid + 8, 16 * bj + k0 + tig + 4)])};
            const uint32_t b[2] = {k0 + tig >= c ? tf32(F[fx(16 * bj + k0 + tig, 16 * bj + c)]) : 0u,
                                   k0 + tig + 4 >= c ? tf32(F[fx(16 * bj + k0 + tig + 4, 16 * bj + c)]) : 0u};
            mma16x8x8(d, a, b);
        }
        const int cc = 16 * bi + 8 * nt + 2 * tig;       // X into the upper block (bj, bi)
        F[fx(16 * bj + gid, cc)] = d[0];
        F[fx(16 * bj + gid, cc + 1)] = d[1];
        F[fx(16 * bj + gid + 8, cc)] = d[2];
        F[fx(16 * bj + gid + 8, cc + 1)] = d[3];
        // -T_ii X reads only the X columns this warp wrote, but its result overwrites columns
        // of M_ij that the pair's other warp reads above: the pair meets first
        if (warp < 2) asm volatile("bar.sync 2, 64;" ::: "memory");
        else asm volatile("bar.sync 3, 64;" ::: "memory");
    }
    if (warp < 4) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
            const int k0 = 8 * kt;
            const uint32_t a[4] = {k0 + tig <= gid ? tf32(F[fx(16 * bi + gid, 16 * bi + k0 + tig)]) : 0u,
                                   k0 + tig <= gid + 8 ? tf32(F[fx(16 * bi + gid + 8, 16 * bi + k0 + tig)]) : 0u,
                                   k0 + tig + 4 <= gid ? tf32(F[fx(16 * bi + gid, 16 * bi + k0 + tig + 4)]) : 0u,
                                   k0 + tig + 4 <= gid + 8 ? tf32(F[fx(16 * bi + gid + 8, 16 * bi + k0 + tig + 4)]) : 0u};
            const uint32_t b[2] = {tf32(F[fx(16 * bj + k0 + tig, 16 * bi + 8 * nt + gid)]),
                                   tf32(F[fx(16 * bj + k0 + tig + 4, 16 * bi + 8 * nt + gid)])};
            mma16x8x8(d, a, b);
        }
        const int cc = 16 * bj + 8 * nt + 2 * tig;
        F[fx(16 * bi + gid, cc)] = -d[0];
        F[fx(16 * bi + gid, cc + 1)] = -d[1];
        F[fx(16 * bi + gid + 8, cc)] = -d[2];
        F[fx(16 * bi + gid + 8, cc + 1)] = -d[3];
    }
    __syncthreads();
    // block (rows 32-63, columns 0-31): warp -> (16-row tile mt, 8-column tile n8)
    const int mt = warp >> 2, n8 = warp & 3;
    {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        const int c = 8 * n8 + gid;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
            if (kt < n8) continue;
            const int k0 = 8 * kt;
            const int r0 = 32 + 16 * mt + gid;
            const uint32_t a[4] = {tf32(F[fx(r0, k0 + tig)]), tf32(F[fx(r0 + 8, k0 + tig)]),
                                   tf32(F[fx(r0, k0 + tig + 4)]), tf32(F[fx(r0 + 8, k0 + tig + 4)])};
            const uint32_t b[2] = {k0 + tig >= c ? tf32(F[fx(k0 + tig, c)]) : 0u,
                                   k0 + tig + 4 >= c ? tf32(F[fx(k0 + tig + 4, c)]) : 0u};
            mma16x8x8(d, a, b);
        }
        const int cc = 32 + 8 * n8 + 2 * tig;            // X into rows 0-31, columns 32-63
        F[fx(16 * mt + gid, cc)] = d[0];
        F[fx(16 * mt + gid, cc + 1)] = d[1];
        F[fx(16 * mt + gid + 8, cc)] = d[2];
        F[fx(16 * mt + gid + 8, cc + 1)] = d[3];
    }
    // -T_II X reads X from the warps of both row tiles, and its result overwrites columns of
    // M_IJ that the row tile's other warps read above: every warp meets
    __syncthreads();
    {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        const int r0 = 16 * mt + gid;                     // row of T_II (local)
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
            if (kt > 2 * mt + 1) continue;                // T_II is zero right of its diagonal
            const int k0 = 8 * kt;
            const uint32_t a[4] = {k0 + tig <= r0 ? tf32(F[fx(32 + r0, 32 + k0 + tig)]) : 0u,
                                   k0 + tig <= r0 + 8 ? tf32(F[fx(32 + r0 + 8, 32 + k0 + tig)]) : 0u,
                                   k0 + tig + 4 <= r0 ? tf32(F[fx(32 + r0, 32 + k0 + tig + 4)]) : 0u,
                                   k0 + tig + 4 <= r0 + 8 ? tf32(F[fx(32 + r0 + 8, 32 + k0 + tig + 4)]) : 0u};
            const uint32_t b[2] = {tf32(F[fx(k0 + tig, 32 + 8 * n8 + gid)]), tf32(F[fx(k0 + tig + 4, 32 + 8 * n8 + gid)])};
            mma16x8x8(d, a, b);
        }
        const int cc = 8 * n8 + 2 * tig;
        F[fx(32 + r0, cc)] = -d[0];
        F[fx(32 + r0, cc + 1)] = -d[1];
        F[fx(32 + r0 + 8, cc)] = -d[2];
        F[fx(32 + r0 + 8, cc + 1)] = -d[3];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(NT, 2) kda_fwd_tc2(FwdParams p, PlanDev pd, int32_t round_base,
                                                     int32_t hpb, const __grid_constant__ Maps2 maps) {
    using namespace f2;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    // mbarriers: 0-3 the four product batches of a chunk, 4 g, 5 k, 6 q, 7 v (one phase per chunk)
    __shared__ uint64_t bars[8];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ int s_rows[64];                      // compact rows of the chunk being staged (gathers)
    float *vqs = reinterpret_cast<float *>(sm + VQS);
    float *vbeta = reinterpret_cast<float *>(sm + VBETA);
    float *F = reinterpret_cast<float *>(sm + SC);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lq = warp & 3, ch = warp >> 2;
    const int H = p.H;
    // one block: heads [hfirst, hfirst + hpb) of one sequence, one after the other; the next
    // head's first chunk is staged, its reference formed and its initial state loaded while
    // the current head's last chunk runs
    const int32_t ngrp = H / hpb;
    const int32_t seq = pd.round_order[round_base + blockIdx.x / ngrp];
    const int32_t hfirst = (blockIdx.x % ngrp) * hpb, hlast = hfirst + hpb - 1;
    int32_t h = hfirst;
    const int32_t rho = pd.seq_rho[seq], L = rho + pd.seq_nown[seq];
    const int32_t nch = (L + BC - 1) / BC;
    const int32_t src = pd.seq_src[seq];
    const int32_t row0 = pd.seq_row0[seq], cbase = pd.seq_cbase[seq];
    uint8_t *rec = static_cast<uint8_t *>(p.chunk_states);
    const uint16_t *beta = static_cast<const uint16_t *>(p.beta);

    if (tid == 0) {
        for (int i = 0; i < 8; ++i) tc::mbar_init(&bars[i], 1);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 256);
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t lane_off = static_cast<uint32_t>(lq * 32) << 16;
    const uint32_t tS = tm, tR = tm + 128, tW = tm + 192;
    const int jv = lq * 32 + lane;                   // this thread's TMEM lane

    auto nv_of = [&](int32_t c) { return min(BC, L - c * BC); };
    // Row table of chunk c (threads 0-63; read by the gathers after a barrier) and this
    // thread's beta of row t = tid (raw bf16 bits, 0 past the end).
    auto rows_of = [&](int32_t c, int32_t hh) -> uint16_t {
        if (tid >= 64) return 0;
        const int64_t row = local_row(pd, seq, rho, L, c * BC + tid);
        s_rows[tid] = static_cast<int>(row);
        return row >= 0 ? beta[row * H + hh] : static_cast<uint16_t>(0);
    };
    int armed[8] = {0, 0, 0, 0, 0, 0, 0, 0};     // phases armed per barrier (uniform over threads)
    auto stage = [&](int which, int32_t c, int32_t hh) {
        ++armed[4 + which];
        const int32_t c0 = c * BC;
        const int t_own = max(0, rho - c0), t_end = nv_of(c);
        const int32_t own0 = row0 + c0 - rho;
        switch (which) {
        case 0: stage_chunk_rows<NT>(p.g, maps.g, s_rows, hh, H, t_own, t_end, own0, 0, sm + GP, sm + GP + 8192, &bars[4]); break;
        case 1: stage_chunk_rows<NT>(p.k, maps.k, s_rows, hh, H, t_own, t_end, own0, 0, sm + KQ, sm + KQ + 16384, &bars[5]); break;
        case 2: stage_chunk_rows<NT>(p.q, maps.q, s_rows, hh, H, t_own, t_end, own0, 0, sm + KQ + 8192, sm + KQ + 24576, &bars[6]); break;
        default: stage_chunk_rows<NT>(p.v, maps.v, s_rows, hh, H, t_own, t_end, own0, 0, sm + VV, sm + VV + 8192, &bars[7]); break;
        }
    };
    auto pass_a = [&](int32_t c, uint32_t slot, uint16_t braw) {
        chunk_pass_a(sm, sm + GP, vqs, vbeta, sm + VM, sm + VEM, sm + VEG, slot, braw, pd, seq, c * BC);
    };
    // the initial state of head hh (null: zero)
    auto state0 = [&](int32_t hh) -> const float * {
        return src >= 0 ? p.states + (static_cast<int64_t>(src) * H + hh) * D * D
                        : (p.h0 ? p.h0 + (static_cast<int64_t>(-1 - src) * H + hh) * D * D : nullptr);
    };

    // ---- sequence start: chunk 0's rows, the initial state (loaded while they arrive), pass A
    uint16_t braw = rows_of(0, h);
    __syncthreads();
    stage(0, 0, h);
    stage(1, 0, h);
    stage(2, 0, h);
    stage(3, 0, h);
    const int32_t sp_end = pd.seq_sptr[seq + 1];
    {
        // S0^T (lane = value channel) into TMEM unscaled
        const float *S0 = state0(h);
        float r0[32], r1[32];
        const int cb = ch * 64;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            r0[j] = S0 ? S0[(cb + j) * D + jv] : 0.f;
            r1[j] = S0 ? S0[(cb + 32 + j) * D + jv] : 0.f;
        }
        tc::tmem_st32x2(tS + lane_off + cb, r0, tS + lane_off + cb + 32, r1);
    }
    bool ok = wait_data(&bars[4], 0, &s_fail);
    if (ok) {
        pass_a(0, 0, braw);
        __syncthreads();
        // R = S0^T diag(e^{m_0}): fp32 back into TMEM, bf16 pairs into the R columns and
        // into the chunk-0 record
        const float *em = reinterpret_cast<const float *>(sm + VEM);
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            const int cb = ch * 64 + hf * 32;
            float r[32];
            uint32_t pk[16];
            tc::tmem_ld32(tS + lane_off + cb, r);
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 a = *reinterpret_cast<const float4 *>(em + cb + j);
                r[j] *= a.x; r[j + 1] *= a.y; r[j + 2] *= a.z; r[j + 3] *= a.w;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = tc::pack_bf16(r[2 * j], r[2 * j + 1]);
            if (rec) {
                uint4 *dst = reinterpret_cast<uint4 *>(rec + (static_cast<int64_t>(cbase) * H + h) * kRecBytes +
                                                       jv * 256 + cb * 2);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
            tc::tmem_st32_issue(tS + lane_off + cb, r);
            asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                         "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                         :: "r"(tR + lane_off + cb / 2), "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]),
                            "r"(pk[5]), "r"(pk[6]), "r"(pk[7]), "r"(pk[8]), "r"(pk[9]), "r"(pk[10]), "r"(pk[11]),
                            "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15]) : "memory");
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        tc::fence_before_sync();
    }

    uint32_t it = 0;                                  // chunks this block has processed
    for (; ok; ++h) {
    int32_t sp = pd.seq_sptr[seq];
    for (int32_t ci = 0; ci < nch; ++ci, ++it) {
        const uint32_t ph = it & 1, b = it & 1;       // barrier phases and vector slots
        const int32_t c0 = ci * BC;
        const int nv = nv_of(ci);
        // the next chunk: this head's, or the next head's first after this head's last
        const bool last = ci + 1 == nch, hnext = last && h < hlast, more = !last || hnext;
        const int32_t cn = last ? 0 : ci + 1, hn = last ? h + 1 : h;
        // ---- pass B: scaled operands Kp, Qp (in place over raw k, q), Km ------------------
        if (tid == 0) tc::bulk_wait_read();             // the last record store has read KM and SC
        poll0(&bars[5], ph, &s_fail);
        poll0(&bars[6], ph, &s_fail);
        if (!sync_check(&s_fail)) break;
        chunk_pass_b(sm + KQ, sm + GP, sm + KM, vqs, reinterpret_cast<const float *>(sm + VM) + b * 128, p.scale);
        if (more) braw = rows_of(cn, hn);
        sync_mma();
        if (tid == 0) {
            tc::mma_tile(tW, tc::smem_addr(sm + KQ), 16384, tc::smem_addr(sm + KM), 8192, 128,
                         tc::idesc_bf16(128, 64), false);
            tc::mma_commit(&bars[0]);
        }
        ++armed[0];
        // raw g is consumed, the V tile is free: fetch the next chunk's g and this chunk's v
        // ... v(ci) was requested at the previous chunk's end or the sequence start
        if (more) stage(0, cn, hn);
        if (!wait_all2(&bars[0], ph, &s_fail)) break;
        // ---- [A; P] out of TMEM: diag(beta) A (strict lower, fp32) into the scratch ----------
        if (lq < 2) {
            float r[32];
            tc::tmem_ld32(tW + lane_off + ch * 32, r);
            const int t = jv;
            const float bt = vbeta[t];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const int s = ch * 32 + j;
                *reinterpret_cast<float4 *>(F + fx(t, s)) =
                    make_float4(s < t ? bt * r[j] : 0.f, s + 1 < t ? bt * r[j + 1] : 0.f,
                                s + 2 < t ? bt * r[j + 2] : 0.f, s + 3 < t ? bt * r[j + 3] : 0.f);
            }
        }
        __syncthreads();
        invert64(F);
        // ---- T out: Tb = T diag(beta) and P as bf16 tiles, T into the record ----------------
        {
            const int t = tid >> 2, s0 = (tid & 3) * 16;
            float tv[16];
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(F + fx(t, s0 + j));
                tv[j] = s0 + j <= t ? x.x : 0.f;
                tv[j + 1] = s0 + j + 1 <= t ? x.y : 0.f;
                tv[j + 2] = s0 + j + 2 <= t ? x.z : 0.f;
                tv[j + 3] = s0 + j + 3 <= t ? x.w : 0.f;
            }
            float pv[32];
            if (lq >= 2) {
                tc::tmem_ld32(tW + lane_off + ch * 32, pv);
                const int tp = jv - 64;
#pragma unroll
                for (int j = 0; j < 32; ++j) pv[j] = (ch * 32 + j <= tp) ? pv[j] : 0.f;
            }
            __syncthreads();
            float tb[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) tb[j] = tv[j] * vbeta[s0 + j];
            tc::st_sw128_8(sm + SC, 64, t, s0, tb);
            tc::st_sw128_8(sm + SC, 64, t, s0 + 8, tb + 8);
            if (rec) {
                uint8_t *dst = rec + (static_cast<int64_t>(cbase + ci) * H + h) * kRecBytes + D * D * 2 + t * 128 + s0 * 2;
                reinterpret_cast<uint4 *>(dst)[0] =
                    make_uint4(tc::pack_bf16(tv[0], tv[1]), tc::pack_bf16(tv[2], tv[3]), tc::pack_bf16(tv[4], tv[5]),
                               tc::pack_bf16(tv[6], tv[7]));
                reinterpret_cast<uint4 *>(dst)[1] =
                    make_uint4(tc::pack_bf16(tv[8], tv[9]), tc::pack_bf16(tv[10], tv[11]), tc::pack_bf16(tv[12], tv[13]),
                               tc::pack_bf16(tv[14], tv[15]));
            }
            if (lq >= 2) {
                const int tp = jv - 64;
#pragma unroll
                for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + SC + 8192, 64, tp, ch * 32 + j, pv + j);
            }
        }
        sync_mma();
        if (tid == 0) {
            // Kp^T Tb^T (Kp read MN-major)
            tc::mma_op(tW, tc::Opnd{tc::smem_addr(sm + KQ), 16384, true}, tc::Opnd{tc::smem_addr(sm + SC), 8192, false},
                       128, 64, 64, false);
            tc::mma_commit(&bars[1]);
        }
        ++armed[1];
        // ---- pass A of the next chunk while the product runs --------------------------------
        if (more) {
            if (!wait_data(&bars[4], ph ^ 1, &s_fail)) break;
            pass_a(cn, b ^ 1, braw);
        }
        if (!wait_all2(&bars[1], ph, &s_fail)) break;
        // ---- -(Kp^T Tb^T) as the MN-major B tile [dk][t] over the Kp half of KQ -----------------
        {
            float r[32];
            tc::tmem_ld32(tW + lane_off + ch * 32, r);
            const int dk = jv;
            uint8_t *row = sm + KQ + (dk >> 6) * 16384 + (dk & 63) * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int chunk16 = ch * 4 + q;
                *reinterpret_cast<uint4 *>(row + ((chunk16 ^ (dk & 7)) << 4)) =
                    make_uint4(tc::pack_bf16(-r[8 * q], -r[8 * q + 1]), tc::pack_bf16(-r[8 * q + 2], -r[8 * q + 3]),
                               tc::pack_bf16(-r[8 * q + 4], -r[8 * q + 5]), tc::pack_bf16(-r[8 * q + 6], -r[8 * q + 7]));
            }
        }
        poll0(&bars[7], ph, &s_fail);                      // this chunk's v
        if (!sync_mma_check(&s_fail)) break;
        if (tid == 0) {
            // U^T = V^T Tb^T - R (Kp^T Tb^T)
            tc::mma_op(tW, tc::Opnd{tc::smem_addr(sm + VV), 8192, true}, tc::Opnd{tc::smem_addr(sm + SC), 8192, false},
                       128, 64, 64, false);
            const uint32_t id = tc::idesc_bf16(128, 64, false, true);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16_ta(tW, tR + kk * 8, tc::desc_sw128_mn(tc::smem_addr(sm + KQ) + (kk >> 2) * 16384 + (kk & 3) * 2048, 8192),
                       id, 1u);
            tc::mma_commit(&bars[2]);
        }
        ++armed[2];
        if (!wait_all2(&bars[2], ph, &s_fail)) break;
        if (more) stage(1, cn, hn);                         // the Kp half is free: next k
        // ---- U^T -> bf16 tile [dv][t] (K-major A) over V --------------------------------------
        {
            float r[32];
            tc::tmem_ld32(tW + lane_off + ch * 32, r);
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + VV, 128, jv, ch * 32 + j, r + j);
        }
        sync_mma();
        if (tid == 0) {
            // O^T = R Qp^T + U^T P^T;  S += U^T Km
            const uint32_t id = tc::idesc_bf16(128, 64, false, false);
            const tc::Opnd qp{tc::smem_addr(sm + KQ) + 8192, 16384, false};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16_ta(tW, tR + kk * 8, tc::opnd_desc(qp, kk), id, kk > 0 ? 1u : 0u);
            tc::mma_op(tW, tc::Opnd{tc::smem_addr(sm + VV), 16384, false},
                       tc::Opnd{tc::smem_addr(sm + SC) + 8192, 8192, false}, 128, 64, 64, true);
            tc::mma_op(tS, tc::Opnd{tc::smem_addr(sm + VV), 16384, false}, tc::Opnd{tc::smem_addr(sm + KM), 8192, true},
                       128, 128, 64, true);
            tc::mma_commit(&bars[3]);
        }
        ++armed[3];
        if (!wait_all2(&bars[3], ph, &s_fail)) break;
        if (more) stage(2, cn, hn);                         // the Qp half is free: next q
        // ---- outputs: O rows (staged [t][dv] over U^T), the state leaves and re-enters TMEM ----
        {
            float r[32];
            tc::tmem_ld32(tW + lane_off + ch * 32, r);
            __nv_bfloat16 *os = reinterpret_cast<__nv_bfloat16 *>(sm + VV);
#pragma unroll
            for (int j = 0; j < 32; ++j) os[(ch * 32 + j) * D + jv] = __float2bfloat16_rn(r[j]);
        }
        {
            const int32_t pend = min(c0 + BC, L);
            const bool slot = sp < sp_end && pd.state_lpos[sp] == pend;
            const float *eg = reinterpret_cast<const float *>(sm + VEG) + b * 128;
            const float *emn = reinterpret_cast<const float *>(sm + VEM) + (b ^ 1) * 128;
            float *sdst = slot ? p.states + (static_cast<int64_t>(sp) * H + h) * D * D
                        : (last && p.final_state ? p.final_state + (static_cast<int64_t>(seq) * H + h) * D * D : nullptr);
            const bool rdst = more && rec;
            const float *S0n = hnext ? state0(hn) : nullptr;
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                const int cb = ch * 64 + hf * 32;
                float r[32];
                tc::tmem_ld32(tS + lane_off + cb, r);
#pragma unroll
                for (int j = 0; j < 32; j += 4) {                             // S'^T
                    const float4 a = *reinterpret_cast<const float4 *>(eg + cb + j);
                    r[j] *= a.x; r[j + 1] *= a.y; r[j + 2] *= a.z; r[j + 3] *= a.w;
                }
                if (sdst) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) sdst[(cb + j) * D + jv] = r[j];
                }
                if (last && slot && p.final_state) {
                    float *fd = p.final_state + (static_cast<int64_t>(seq) * H + h) * D * D;
#pragma unroll
                    for (int j = 0; j < 32; ++j) fd[(cb + j) * D + jv] = r[j];
                }
                if (more) {
                    uint32_t pk[16];
                    if (hnext) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = S0n ? S0n[(cb + j) * D + jv] : 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {                         // next chunk's R
                        const float4 a = *reinterpret_cast<const float4 *>(emn + cb + j);
                        r[j] *= a.x; r[j + 1] *= a.y; r[j + 2] *= a.z; r[j + 3] *= a.w;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) pk[j] = tc::pack_bf16(r[2 * j], r[2 * j + 1]);
                    if (rdst) {
                        // the next chunk's record (its bf16 R), staged [dv][64] per column half
                        // in the record map's box layout (128-byte swizzle) for its TMA stores
                        uint8_t *stg = sm + (ch ? SC : KM) + jv * 128;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4 *>(stg + (((hf * 4 + q) ^ (jv & 7)) << 4)) =
                                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                    }
                    tc::tmem_st32_issue(tS + lane_off + cb, r);
                    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                                 :: "r"(tR + lane_off + cb / 2), "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]),
                                    "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7]), "r"(pk[8]), "r"(pk[9]), "r"(pk[10]),
                                    "r"(pk[11]), "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15]) : "memory");
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
            }
            if (slot) ++sp;
        }
        tc::fence_smem_to_async();                       // the staged record, for its TMA store
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0 && more && rec) {
            // the next chunk's R record: columns 0-63 staged in KM, 64-127 in SC
            const int y = static_cast<int>((static_cast<int64_t>(cbase + cn) * H + hn) * (kRecBytes / 256));
            tc::tma_store_2d(&maps.rec_s, 0, y, sm + KM);
            tc::tma_store_2d(&maps.rec_s, 64, y, sm + SC);
            tc::bulk_commit();
        }
        {
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
            const int t_lo = max(0, rho - c0);
            for (int e = tid; e < 64 * 16; e += NT) {
                const int t = e >> 4, piece = e & 15;
                if (t < t_lo || t >= nv) continue;
                const int64_t row = static_cast<int64_t>(row0) + (c0 + t - rho);
                *reinterpret_cast<uint4 *>(o + (row * H + h) * D + piece * 8) =
                    *reinterpret_cast<const uint4 *>(sm + VV + t * 256 + piece * 16);
            }
        }
        __syncthreads();
        tc::fence_after_sync();
        if (more) stage(3, cn, hn);                         // the output staging is read: next v
    }
    // every stop inside the chunk loop follows a failed wait, which all threads see in s_fail
    if (*reinterpret_cast<volatile int *>(&s_fail) != 0 || h == hlast) break;
    }
    if (tid == 0) tc::bulk_wait_all();               // the record stores have landed
    // ---- drain: copies and products still in flight land before shared memory is released --
    tc::cp_async_wait_all();
    __syncthreads();
    if (s_fail) {
        dev_error(pd, kDevErrTimeout, seq, h);
        // the last phase armed on each barrier completes before the block exits (phases
        // complete in order, so the earlier ones have too)
        if (tid == 0)
            for (int i = 0; i < 8; ++i)
                if (armed[i] > 0 && !tc::mbar_wait(&bars[i], (armed[i] - 1) & 1, 200000000LL))
                    dev_error(pd, kDevErrTimeout, seq, h);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tm, 256);
}


// ======================================================================================
// Backward state pass, two CTAs per SM: per (sequence, head), chunks in reverse, the
// carried state gradient in TMEM (page "HARTS ... 精读", section 4.3, KDA paragraph: the
// initial-state gradient of a resumed sequence flows back into the call that produced its
// boundary; here each chunk end where a later round resumed adds those consumers'
// initial-state gradients to the carry).  With dS' the gradient at the chunk end and
// Q' = dS'^T diag(e^{Gamma_L - m}) (lane = value channel):
//   dU^T = dO^T P + Q' Km^T,   dY^T = dU^T Tb,   dS^T = (Q' + dO^T Qp - dY^T Kp) diag(e^m)
// where Tb = T diag(beta) with T from the forward's chunk record.  The bf16 Q' (the operand
// the products use) is saved per chunk for the gradient pass.  TMEM: the carry C (fp32, 128 columns), Q' as bf16 pairs
// (the A operand of Q' Km^T, 64), one work tile W (64) for P, dU^T and dY^T in turn.
// ======================================================================================
namespace s2 {
constexpr uint32_t KQ = 0;          // [128][128] SW128 (atoms 16 KB): raw k -> Kp (rows 0-63), raw q -> Qp (64-127)
constexpr uint32_t KM = 32768;      // [64][128] (atoms 8 KB): raw g -> Km in place
constexpr uint32_t DO = 49152;      // [64][128] (atoms 8 KB): dO (zero on replay rows)
constexpr uint32_t TB = 65536;      // [64][64]: T from the record -> Tb = T diag(beta) in place
constexpr uint32_t PP = 73728;      // [64][64]: P (lower with the diagonal)
constexpr uint32_t DU = 81920;      // [128][64]: dU^T, then -dY^T
constexpr uint32_t VQS = 98304;     // fp32 [16][128]
constexpr uint32_t VM = VQS + 8704;         // fp32 [2][128] m log2(e) (by processing parity)
constexpr uint32_t VEM = VM + 1024;       // fp32 [2][128] e^m
constexpr uint32_t VEG = VEM + 1024;      // fp32 [2][128] e^{Gamma_L - m}
constexpr uint32_t VBETA = VEG + 1024;    // fp32 [64]
constexpr uint32_t END = VBETA + 256;
constexpr uint32_t bytes = END + 1024;
}  // namespace s2

struct StateMaps2 {
    RowMaps q, k, g, dout;
    CUtensorMap rec_t;           // chunk records as [rows of 128 B], boxes of 64 x 64 (a chunk's T)
    CUtensorMap dch;             // the saved Q' as [rows of 256 B], boxes of 64 columns x 128 rows
};

__global__ void __launch_bounds__(NT, 2) kda_bwd_state_tc2(BwdParams p, PlanDev pd, int32_t round_base,
                                                           int32_t hpb, const __grid_constant__ StateMaps2 maps) {
    using namespace s2;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    // mbarriers: 0-3 product batches, 4 g, 5 k, 6 q, 7 dO, 8 T (one phase per chunk)
    __shared__ uint64_t bars[9];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ int s_rows[64];
    float *vqs = reinterpret_cast<float *>(sm + VQS);
    float *vbeta = reinterpret_cast<float *>(sm + VBETA);
    const FwdParams &f = p.f;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lq = warp & 3, ch = warp >> 2;
    const int H = f.H;
    // one block: heads [hfirst, hfirst + hpb) of one sequence in turn; the next head's last
    // chunk is staged while the current head's first chunk runs
    const int32_t ngrp = H / hpb;
    const int32_t seq = pd.round_order[round_base + blockIdx.x / ngrp];
    const int32_t hfirst = (blockIdx.x % ngrp) * hpb, hlast = hfirst + hpb - 1;
    int32_t h = hfirst;
    const int32_t rho = pd.seq_rho[seq], L = rho + pd.seq_nown[seq];
    const int32_t nch = (L + BC - 1) / BC;
    const int32_t src = pd.seq_src[seq], cbase = pd.seq_cbase[seq], row0 = pd.seq_row0[seq];
    const uint16_t *beta = static_cast<const uint16_t *>(f.beta);

    if (tid == 0) {
        for (int i = 0; i < 9; ++i) tc::mbar_init(&bars[i], 1);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 256);
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t lane_off = static_cast<uint32_t>(lq * 32) << 16;
    const uint32_t tC = tm, tQ = tm + 128, tW = tm + 192;
    const int jv = lq * 32 + lane;

    int armed[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    auto nv_of = [&](int32_t c) { return min(BC, L - c * BC); };
    auto rows_of = [&](int32_t c, int32_t hh) -> uint16_t {
        if (tid >= 64) return 0;
        const int64_t row = local_row(pd, seq, rho, L, c * BC + tid);
        s_rows[tid] = static_cast<int>(row);
        return row >= 0 ? beta[row * H + hh] : static_cast<uint16_t>(0);
    };
    auto stage = [&](int which, int32_t c, int32_t hh) {
        ++armed[4 + which];
        const int32_t c0 = c * BC;
        const int t_own = max(0, rho - c0), t_end = nv_of(c);
        const int32_t own0 = row0 + c0 - rho;
        switch (which) {
        case 0: stage_chunk_rows<NT>(f.g, maps.g, s_rows, hh, H, t_own, t_end, own0, 0, sm + KM, sm + KM + 8192, &bars[4]); break;
        case 1: stage_chunk_rows<NT>(f.k, maps.k, s_rows, hh, H, t_own, t_end, own0, 0, sm + KQ, sm + KQ + 16384, &bars[5]); break;
        case 2: stage_chunk_rows<NT>(f.q, maps.q, s_rows, hh, H, t_own, t_end, own0, 0, sm + KQ + 8192, sm + KQ + 24576, &bars[6]); break;
        case 3: stage_chunk_rows<NT>(p.d_o, maps.dout, s_rows, hh, H, t_own, t_end, own0, t_own, sm + DO, sm + DO + 8192,
                                     &bars[7]); break;
        default:
            if (tid == 0) {
                tc::mbar_expect_tx(&bars[8], 8192);
                tc::tma_load_2d(sm + TB, &maps.rec_t, 0,
                                static_cast<int>((static_cast<int64_t>(cbase + c) * H + hh) * (kRecBytes / 128) + 2 * D),
                                &bars[8]);
            }
            break;
        }
    };

    // carry <- d_final^T of head hh (the loop scales it by e^{m} of the chunk after; 1 for the last)
    auto carry_init = [&](int32_t hh) {
        const float *df = p.d_final ? p.d_final + (static_cast<int64_t>(seq) * H + hh) * D * D : nullptr;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            const int cb = ch * 64 + hf * 32;
            float r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = df ? df[(cb + j) * D + jv] : 0.f;
            tc::tmem_st32(tC + lane_off + cb, r);
        }
    };
    carry_init(h);
    uint16_t braw = rows_of(nch - 1, h);
    __syncthreads();
    for (int w = 0; w < 5; ++w) stage(w, nch - 1, h);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    const int32_t sp_begin = pd.seq_sptr[seq];
    bool ok = true;
    uint32_t it = 0;                               // chunks this block has processed
    for (;; ++h) {
    int32_t sp = pd.seq_sptr[seq + 1] - 1;
    for (int32_t ci = nch - 1; ci >= 0; --ci, ++it) {
        const int32_t n = nch - 1 - ci;            // processing index within the head
        const uint32_t ph = it & 1, b = it & 1;    // barrier phases and vector slots
        const int32_t c0 = ci * BC, pend = min(c0 + BC, L);
        const int nv = nv_of(ci);
        // the next chunk to process: this head's previous one, or the next head's last
        const bool hnext = ci == 0 && h < hlast, more = ci > 0 || hnext;
        const int32_t cn = ci > 0 ? ci - 1 : nch - 1, hn = ci > 0 ? h : h + 1;
        // ---- pass A (needs g) ---------------------------------------------------------------
        if (!(ok = wait_data(&bars[4], ph, &s_fail))) break;
        chunk_pass_a(sm, sm + KM, vqs, vbeta, sm + VM, sm + VEM, sm + VEG, b, braw, pd, seq, c0);
        __syncthreads();

        // ---- carry: dS' = C e^{m_next} (+ consumers' initial-state gradients at a slot);
        //      Q' = dS'^T diag(e^{Gamma_L - m}), its bf16 copy saved for the gradient pass ------
        {
            const bool slot = sp >= sp_begin && pd.state_lpos[sp] == pend;
            const int32_t cb_ = slot ? pd.state_cptr[sp] : 0, ce_ = slot ? pd.state_cptr[sp + 1] : 0;
            const float *emn = reinterpret_cast<const float *>(sm + VEM) + (b ^ 1) * 128;
            const float *eg = reinterpret_cast<const float *>(sm + VEG) + b * 128;
            const int rec_row = static_cast<int>((static_cast<int64_t>(cbase + ci) * H + h) * D);
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                const int cb = hf * 64 + ch * 32;           // columns [64 hf, 64 hf + 64): this warp's 32
                float r[32];
                tc::tmem_ld32(tC + lane_off + cb, r);
                if (n > 0) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 a = *reinterpret_cast<const float4 *>(emn + cb + j);
                        r[j] *= a.x; r[j + 1] *= a.y; r[j + 2] *= a.z; r[j + 3] *= a.w;
                    }
                }
                for (int32_t cc = cb_; cc < ce_; ++cc) {
                    const float *di = p.ds_init + (static_cast<int64_t>(pd.state_cons[cc]) * H + h) * D * D;
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] += di[(cb + j) * D + jv];
                }
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 a = *reinterpret_cast<const float4 *>(eg + cb + j);
                    r[j] *= a.x; r[j + 1] *= a.y; r[j + 2] *= a.z; r[j + 3] *= a.w;
                }
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) pk[j] = tc::pack_bf16(r[2 * j], r[2 * j + 1]);
                // the bf16 Q' of this half's 64 columns into DU as the record map's box ([dv][64],
                // 128-byte swizzle), then out by one TMA store
                uint8_t *stg = sm + DU + jv * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4 *>(stg + (((ch * 4 + q) ^ (jv & 7)) << 4)) =
                        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                tc::tmem_st32_issue(tC + lane_off + cb, r);
                asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                             "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                             :: "r"(tQ + lane_off + cb / 2), "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]),
                                "r"(pk[5]), "r"(pk[6]), "r"(pk[7]), "r"(pk[8]), "r"(pk[9]), "r"(pk[10]), "r"(pk[11]),
                                "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15]) : "memory");
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc::fence_smem_to_async();
                __syncthreads();
                if (tid == 0) {
                    tc::tma_store_2d(&maps.dch, hf * 64, rec_row, sm + DU);
                    tc::bulk_commit();
                    if (hf == 0) tc::bulk_wait_read();      // DU takes the second half next
                }
                if (hf == 0) __syncthreads();
            }
            if (slot) --sp;
        }
        // ---- pass B: Kp, Qp in place, Km over g; Tb = T diag(beta) in place -------------------
        poll0(&bars[5], ph, &s_fail);
        poll0(&bars[6], ph, &s_fail);
        poll0(&bars[8], ph, &s_fail);
        if (!(ok = sync_check(&s_fail))) break;
        chunk_pass_b(sm + KQ, sm + KM, sm + KM, vqs, reinterpret_cast<const float *>(sm + VM) + b * 128, f.scale);
        {
            const int t = tid >> 2, q = tid & 3;             // row t, 16-column quarter q of T
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int jj = 2 * q + hh;                  // 16-byte chunk (8 columns)
                uint4 *pw = reinterpret_cast<uint4 *>(sm + TB + chunk_off(t, jj));
                float v[8];
                unpack8(*pw, v);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] *= vbeta[8 * jj + i];
                *pw = pack8(v);
            }
        }
        tc::fence_before_sync();
        sync_mma();
        if (tid == 0) {
            tc::mma_tile(tW, tc::smem_addr(sm + KQ), 16384, tc::smem_addr(sm + KM), 8192, 128,
                         tc::idesc_bf16(128, 64), false);
            tc::mma_commit(&bars[0]);
        }
        ++armed[0];
        if (!(ok = wait_all2(&bars[0], ph, &s_fail))) break;
        // ---- P (rows 64-127 of W) -> bf16 tile [t][s] --------------------------------------------
        if (lq >= 2) {
            float pv[32];
            tc::tmem_ld32(tW + lane_off + ch * 32, pv);
            const int tp = jv - 64;
#pragma unroll
            for (int j = 0; j < 32; ++j) pv[j] = (ch * 32 + j <= tp) ? pv[j] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + PP, 64, tp, ch * 32 + j, pv + j);
        }
        poll0(&bars[7], ph, &s_fail);                      // dO
        if (!(ok = sync_mma_check(&s_fail))) break;
        if (tid == 0) {
            // dU^T = dO^T P + Q' Km^T
            tc::mma_op(tW, tc::Opnd{tc::smem_addr(sm + DO), 8192, true}, tc::Opnd{tc::smem_addr(sm + PP), 8192, true},
                       128, 64, 64, false);
            const uint32_t id = tc::idesc_bf16(128, 64, false, false);
            const tc::Opnd kmo{tc::smem_addr(sm + KM), 8192, false};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16_ta(tW, tQ + kk * 8, tc::opnd_desc(kmo, kk), id, 1u);
            tc::mma_commit(&bars[1]);
            tc::bulk_wait_read();                           // the Q' store has read DU (written below)
        }
        ++armed[1];
        if (more) braw = rows_of(cn, hn);                   // the next chunk's rows, read after the wait
        if (!(ok = wait_all2(&bars[1], ph, &s_fail))) break;
        if (more) stage(0, cn, hn);                          // Km is consumed: next g
        {
            float r[32];
            tc::tmem_ld32(tW + lane_off + ch * 32, r);
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + DU, 128, jv, ch * 32 + j, r + j);
        }
        sync_mma();
        if (tid == 0) {
            // dY^T = dU^T Tb (Tb read MN-major)
            tc::mma_op(tW, tc::Opnd{tc::smem_addr(sm + DU), 16384, false}, tc::Opnd{tc::smem_addr(sm + TB), 8192, true},
                       128, 64, 64, false);
            tc::mma_commit(&bars[2]);
        }
        ++armed[2];
        if (!(ok = wait_all2(&bars[2], ph, &s_fail))) break;
        if (more) stage(4, cn, hn);                          // T consumed: next chunk's T
        {
            float r[32];
            tc::tmem_ld32(tW + lane_off + ch * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = -r[j];
#pragma unroll
            for (int j = 0; j < 32; j += 8) tc::st_sw128_8(sm + DU, 128, jv, ch * 32 + j, r + j);
        }
        sync_mma();
        if (tid == 0) {
            // C += dO^T Qp - dY^T Kp  (Qp, Kp read MN-major)
            tc::mma_op(tC, tc::Opnd{tc::smem_addr(sm + DO), 8192, true},
                       tc::Opnd{tc::smem_addr(sm + KQ) + 8192, 16384, true}, 128, 128, 64, true);
            tc::mma_op(tC, tc::Opnd{tc::smem_addr(sm + DU), 16384, false}, tc::Opnd{tc::smem_addr(sm + KQ), 16384, true},
                       128, 128, 64, true);
            tc::mma_commit(&bars[3]);
        }
        ++armed[3];
        if (!(ok = wait_all2(&bars[3], ph, &s_fail))) break;
        if (more) { stage(1, cn, hn); stage(2, cn, hn); stage(3, cn, hn); }
    }
    // every stop inside the chunk loop follows a failed wait, which all threads see in s_fail
    if (!ok || *reinterpret_cast<volatile int *>(&s_fail) != 0) break;
    // ---- the head's initial-state gradient: dS_0 = C diag(e^{m_0}) (chunk 0 was the last
    //      processed, slot (it - 1) & 1) ----------------------------------------------------------
    if (src >= 0 || p.dh0) {
        const float *em = reinterpret_cast<const float *>(sm + VEM) + ((it - 1) & 1) * 128;
        float *dst = p.ds_init + (static_cast<int64_t>(seq) * H + h) * D * D;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            const int cb = ch * 64 + hf * 32;
            float r[32];
            tc::tmem_ld32(tC + lane_off + cb, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[(cb + j) * D + jv] = r[j] * em[cb + j];
        }
    }
    if (h == hlast) break;
    // the next head's carry (each warp rewrites the TMEM lanes and columns it just read)
    carry_init(h + 1);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    }
    if (tid == 0) tc::bulk_wait_all();               // the record stores have landed
    tc::cp_async_wait_all();
    __syncthreads();
    if (s_fail) {
        dev_error(pd, kDevErrTimeout, seq, h);
        if (tid == 0)
            for (int i = 0; i < 9; ++i)
                if (armed[i] > 0 && !tc::mbar_wait(&bars[i], (armed[i] - 1) & 1, 200000000LL))
                    dev_error(pd, kDevErrTimeout, seq, h);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tm, 256);
}

}  // namespace

cudaError_t tc2_fwd_round(const FwdParams &p, const PlanDev &pd, int32_t base, int32_t n_items, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kda_fwd_tc2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(f2::bytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_fwd_tc2, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) return e;
    Maps2 maps{};
    {
        const int H = p.H;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(pd.C)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
        (void)dims; (void)strides;
        const void *src[4] = {p.q, p.k, p.v, p.g};
        RowMaps *dst[4] = {&maps.q, &maps.k, &maps.v, &maps.g};
        for (int i = 0; i < 4; ++i)
            if (!encode_row_maps(dst[i], src[i], H, pd.C)) return cudaErrorInvalidValue;
        if (p.chunk_states) {
            const int64_t rows = pd.n_chunks * H * (kRecBytes / 256);
            if (rows > INT32_MAX) return cudaErrorInvalidValue;      // TMA coordinates are int32
            const cuuint64_t rdims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
            const cuuint64_t rstrides[1] = {static_cast<cuuint64_t>(D) * 2};
            const cuuint32_t rbox[2] = {64, 128};
            if (!encode_bf16(&maps.rec_s, p.chunk_states, 2, rdims, rstrides, rbox)) return cudaErrorInvalidValue;
        }
    }
    // heads per block: 4 or 2 when the round still gives every SM's two block slots eight
    // blocks or more (a block then pays its start-up once for several heads and overlaps
    // each next head's first loads with the current head's last chunk), else 1
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int hpb = 1;
    for (int c : {4, 2})
        if (p.H % c == 0 && n_items / c >= 16 * nsm) { hpb = c; break; }
    kda_fwd_tc2<<<n_items / hpb, NT, f2::bytes, st>>>(p, pd, base, hpb, maps);
    return cudaGetLastError();
}

cudaError_t tc2_bwd_state_round(const BwdParams &p, const PlanDev &pd, int32_t base, int32_t n_items,
                                cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_state_tc2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(s2::bytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_bwd_state_tc2, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) return e;
    StateMaps2 maps{};
    {
        const int H = p.f.H;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(pd.C)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
        (void)dims; (void)strides;
        const void *src[4] = {p.f.q, p.f.k, p.f.g, p.d_o};
        RowMaps *dst[4] = {&maps.q, &maps.k, &maps.g, &maps.dout};
        for (int i = 0; i < 4; ++i)
            if (!encode_row_maps(dst[i], src[i], H, pd.C)) return cudaErrorInvalidValue;
        const int64_t n_rec = pd.n_chunks * H;
        if (n_rec * (kRecBytes / 128) > INT32_MAX) return cudaErrorInvalidValue;   // TMA coordinates are int32
        const cuuint64_t rdims[2] = {64, static_cast<cuuint64_t>(n_rec * (kRecBytes / 128))};
        const cuuint64_t rstrides[1] = {128};
        const cuuint32_t rbox[2] = {64, 64};
        if (!encode_bf16(&maps.rec_t, p.f.chunk_states, 2, rdims, rstrides, rbox)) return cudaErrorInvalidValue;
        const cuuint64_t qdims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(n_rec * D)};
        const cuuint64_t qstrides[1] = {static_cast<cuuint64_t>(D) * 2};
        const cuuint32_t qbox[2] = {64, 128};
        if (!encode_bf16(&maps.dch, p.dchunk, 2, qdims, qstrides, qbox)) return cudaErrorInvalidValue;
    }
    // heads per block: as the forward's
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int hpb = 1;
    for (int c : {4, 2})
        if (p.f.H % c == 0 && n_items / c >= 16 * nsm) { hpb = c; break; }
    kda_bwd_state_tc2<<<n_items / hpb, NT, s2::bytes, st>>>(p, pd, base, hpb, maps);
    return cudaGetLastError();
}

}  // namespace harts
