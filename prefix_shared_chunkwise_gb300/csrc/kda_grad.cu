// Gradient pass of bf16 packed-tree KDA on sm_103a (dk = dv = 128, chunk 64).
//
// Every (chunk, head) of every round is one independent item: with the chunk's R (the
// forward's record), Q' (the state pass's record) and T = (I + diag(beta) A)^-1 (the
// forward's record), all input gradients of the chunk follow without any sequential
// dependence.  One CTA per SM walks the items in steps of the grid size: 16 compute warps
// run the products and epilogues of one item while four load warps stage the next item's
// tiles, each as soon as the product batch that last reads its buffer is done (one lane of
// load warp 1 issues the product batches).
// Notation (gamma the cumulative log-decay from the chunk start, m = Gamma_L / 2 half the
// chunk's total log-decay, per key channel; t, s local rows):
//   Kp = K e^{gamma-m}, Qp = scale Q e^{gamma-m}, Km = K e^{m-gamma}
//   [A; P] = [Kp; Qp] Km^T, Tb = T diag(beta), R = S^T diag(e^m), Q' = dS'^T diag(e^{Gamma_L-m})
//   Y^T = V^T - R Kp^T, U^T = Y^T Tb^T                              (the forward's U)
//   dU^T = dO^T P + Q' Km^T,  Z = T^T dU,  dY = diag(beta) Z,  dv = dY
//   dP = lower(dO U^T),  dM = -strict(Z U^T),  dA = diag(beta) dM
//   dbeta = diag(Z Y^T) + rowsum(dM .* A)
//   dQp^T = R^T dO^T + Km^T dP^T,  dKp^T = -R^T dY^T + Km^T dA^T,
//   dKm^T = Q'^T U^T + Kp^T dA + Qp^T dP
//   dq = scale dQp e^{gamma-m},  dk = dKp e^{gamma-m} + dKm e^{m-gamma}
//   dgamma = dKp Kp + dQp Qp - dKm Km (the rounded operands the products used),
//   dGamma_L = colsum(Q' .* R) + colsum(Km .* (Q'^T U^T)^T), dg = suffix sums of dgamma + dGamma_L.
// Z collapses the inverse's gradient: with U = Tb Y, dT = dU Y^T diag(beta) and
// T^T dT T^T = (T^T dU)(T diag(beta) Y)^T = Z U^T, so dM needs one product instead of two,
// and colsum(dTb .* T) (dTb = dU Y^T) is the diagonal of Z Y^T.
// (Page "HARTS ... 精读", section 4.3, KDA paragraph: gradients of replayed rows add into the
// ancestor rows they copy; they go to the replay-gradient buffer, folded later in a fixed
// order.)
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "tc_primitives.cuh"
#include "tensor_map.h"
#include "kda_stage.cuh"

namespace harts {
namespace {

constexpr int D = 128, BC = 64, NC = 512, NT = NC + 128;    // 16 compute warps + 4 load warps
constexpr int64_t kRecBytes = (D * D + BC * BC) * 2;

namespace g2 {
constexpr uint32_t RR = 0;          // [128 dv][128 dk] R record (atoms 16 KB)
constexpr uint32_t QQ = 32768;      // [128 dv][128 dk] Q' record -> Z^T [128 dv][64 t] in its first atom
constexpr uint32_t KQ = 65536;      // [128][128]: raw k -> Kp (rows 0-63), raw q -> Qp (64-127)
constexpr uint32_t KM = 98304;      // [64][128] (atoms 8 KB): Km
constexpr uint32_t VV = 114688;     // raw v [64][128] (atoms 8 KB) -> U^T [128][64]
// DO: two atoms of [128 rows][64 columns] (16 KB apart): rows 0-63 hold dO [t][dv], rows 64-127
// (DX) hold dU [t][dv] (the MN-major B operand of T^T dU), then -dY [t][dv].
constexpr uint32_t DO = 131072;
constexpr uint32_t DX = DO + 8192;  // the dU / -dY rows
constexpr uint32_t TT = 163840;     // T [64][64]
constexpr uint32_t TB = 172032;     // Tb [64][64]    } TB..PT: raw g of the next item
constexpr uint32_t PT = 180224;     // P [64][64]     }
constexpr uint32_t YT = 188416;     // Y^T [128][64]
constexpr uint32_t DP = 204800;     // dP [64][64]   } one [128][64] operand [dP; dA]
constexpr uint32_t WA = 212992;     // dA [64][64]   }
constexpr uint32_t VQS = 221184;    // fp32 [4][128] partial sums (several uses)
constexpr uint32_t VM2 = VQS + 2560;      // m log2(e)
constexpr uint32_t VBETA = VM2 + 512;     // fp32 [64]
constexpr uint32_t VDB = VBETA + 256;     // fp32 [64] dbeta
constexpr uint32_t VDGL = VDB + 256;      // fp32 [128] dGamma_L
constexpr uint32_t END = VDGL + 512;
constexpr uint32_t bytes = END + 1024;
}  // namespace g2

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// TMEM loads issued back to back and waited for once.  The wait names the loaded registers
// ("+r"), so no use of them can be scheduled above it.
__device__ __forceinline__ void tld16(uint32_t taddr, float (&r)[16]) {
    uint32_t *u = reinterpret_cast<uint32_t *>(r);
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
                   "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
                 : "r"(taddr));
}
__device__ __forceinline__ void tld8(uint32_t taddr, uint32_t (&u)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7])
                 : "r"(taddr));
}
#define HARTS_R16(a) "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), \
    "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15])
__device__ __forceinline__ void twait1(float (&a)[16]) {
    uint32_t *x = reinterpret_cast<uint32_t *>(a);
    asm volatile("tcgen05.wait::ld.sync.aligned;" : HARTS_R16(x) :: "memory");
}
__device__ __forceinline__ void twait(float (&a)[16], float (&b)[16]) {
    uint32_t *x = reinterpret_cast<uint32_t *>(a), *y = reinterpret_cast<uint32_t *>(b);
    asm volatile("tcgen05.wait::ld.sync.aligned;" : HARTS_R16(x), HARTS_R16(y) :: "memory");
}
__device__ __forceinline__ void twait(float (&a)[16], float (&b)[16], float (&c)[16]) {
    uint32_t *x = reinterpret_cast<uint32_t *>(a), *y = reinterpret_cast<uint32_t *>(b),
             *z = reinterpret_cast<uint32_t *>(c);
    asm volatile("tcgen05.wait::ld.sync.aligned;" : HARTS_R16(x), HARTS_R16(y), HARTS_R16(z) :: "memory");
}
__device__ __forceinline__ void tmem_st8f(uint32_t taddr, const float (&r)[8]) {
    const uint32_t *u = reinterpret_cast<const uint32_t *>(r);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]),
                    "r"(u[7]) : "memory");
}
__device__ __forceinline__ void tmem_st4u(uint32_t taddr, const uint32_t (&u)[4]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};"
                 :: "r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]) : "memory");
}
__device__ __forceinline__ void tld8f(uint32_t taddr, float (&r)[8]) { tld8(taddr, reinterpret_cast<uint32_t (&)[8]>(r)); }
__device__ __forceinline__ void tld4(uint32_t taddr, uint32_t (&u)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]) : "r"(taddr));
}
#define HARTS_R8(a) "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7])
#define HARTS_R4(a) "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3])
// One wait for four 8-column and two 4-column loads (the wait names all their registers).
__device__ __forceinline__ void twait8(float (&a)[8], float (&b)[8], float (&c)[8], float (&d)[8], uint32_t (&e)[4],
                                       uint32_t (&g)[4]) {
    uint32_t *x = reinterpret_cast<uint32_t *>(a), *y = reinterpret_cast<uint32_t *>(b),
             *z = reinterpret_cast<uint32_t *>(c), *w = reinterpret_cast<uint32_t *>(d);
    asm volatile("tcgen05.wait::ld.sync.aligned;" : HARTS_R8(x), HARTS_R8(y), HARTS_R8(z), HARTS_R8(w), HARTS_R4(e), HARTS_R4(g)
                 :: "memory");
}
#undef HARTS_R8
#undef HARTS_R4
#undef HARTS_R16

__device__ __forceinline__ float bf(const uint8_t *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}
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

struct GradMaps2 {
    RowMaps q, k, g, v, dout;
    CUtensorMap rec_s;              // records as [rows of 256 B], boxes of 64 x 128 (a chunk's R)
    CUtensorMap rec_t;              // records as [rows of 128 B], boxes of 64 x 64 (a chunk's T)
    CUtensorMap dch;                // Q' records as [rows of 256 B], boxes of 64 x 128
};

struct Item {
    int32_t h, g, seq, rho, L, c0, nv, row0, rptr;
};

__device__ __forceinline__ Item item_of(const PlanDev &pd, int32_t chunk_begin, int H, int32_t item) {
    Item it;
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

constexpr long long kWaitCycles = 4000000000LL;

// The compute warps meet at named barrier 1 (the load warps never join it).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" :: "n"(NC) : "memory"); }

// The same meeting, returning the OR of `v` over the compute warps (a decision all of them take).
__device__ __forceinline__ bool csync_or(bool v) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 1, %2, q;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r) : "r"(static_cast<uint32_t>(v)), "n"(NC) : "memory");
    return r != 0;
}

__device__ __forceinline__ void csync_mma() {
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    csync();
    tc::fence_after_sync();
}

// Bounded poll of one barrier phase; gives up (and records the failure) when it runs out or
// when the other side has already failed.
__device__ __forceinline__ bool poll_bar(uint64_t *bar, uint32_t phase, int *s_fail) {
    if (tc::mbar_try(bar, phase)) return true;
    const long long t0 = clock64();
    while (!tc::mbar_try(bar, phase)) {
        if (*reinterpret_cast<volatile int *>(s_fail) || clock64() - t0 > kWaitCycles) {
            *reinterpret_cast<volatile int *>(s_fail) = 1;
            return false;
        }
    }
    return true;
}

// Offset of element (row, col) in a [rows][64]-column SW128 atom (bf16).
__device__ __forceinline__ uint32_t sw64(int row, int col) {
    return static_cast<uint32_t>(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}

__global__ void __launch_bounds__(NT, 1) kda_bwd_grad_tc2(BwdParams p, PlanDev pd, int32_t chunk_begin,
                                                          int32_t n_items, const __grid_constant__ GradMaps2 maps) {
    using namespace g2;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    // mbarriers: product batches 0 B1, 1 B2, 2 B3a, 5 B3b, 3 B4a, 14 B4b, 4 B6 (each of the
    // compute warps' phases waits only for the batch whose results it reads, and writes no tile
    // a batch still in flight reads); copies 6 q, 7 k,
    // 8 g, 9 v, 10 dO, 11 T, 12 R, 13 Q'; rdy: the compute warps' operands for B1, B2, B3, B4, B6
    __shared__ uint64_t bars[15];
    __shared__ uint64_t rdy[5];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ int s_rows[4][64];                   // each load warp's row table
    __shared__ uint16_t s_braw[2][64];              // raw beta of an item's rows, by item parity
    // an item's indices, by item number mod 4: the load warp fills item n + 1's slot while the
    // compute warps still read item n - 1's
    __shared__ Item s_items[4];
    const FwdParams &f = p.f;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lq = warp & 3, cg = (warp >> 2) & 3;
    const int H = f.H;
    const int W3 = rep_width(D);
    const int jv = lq * 32 + lane;                  // TMEM lane of this thread
    const uint32_t lane_off = static_cast<uint32_t>(lq * 32) << 16;
    float *vqs = reinterpret_cast<float *>(sm + VQS);
    float *vm2 = reinterpret_cast<float *>(sm + VM2), *vbeta = reinterpret_cast<float *>(sm + VBETA);
    float *vdb = reinterpret_cast<float *>(sm + VDB), *vdgl = reinterpret_cast<float *>(sm + VDGL);

    if (tid == 0) {
        for (int i = 0; i < 15; ++i) tc::mbar_init(&bars[i], 1);
        for (int i = 0; i < 5; ++i) tc::mbar_init(&rdy[i], 1);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tAP = tm, tX = tm + 64, tDU = tm + 128, tDY = tm + 192, tDT = tm + 256, tKM = tm + 320,
                   tGM = tm + 384, tPK = tm + 448;
    int armed[15] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
    int32_t cur_seq = 0, cur_h = 0;

    if (warp >= NC / 32) {
        // ================= load warps: every copy of the next item, issued as its buffer frees ====
        // Load warp 0: g, T and the two records (and the item's indices and beta for the compute
        // warps); 2: q and v; 3: k and dO.  Each walks the items on its own, so that one warp's
        // row gathers (replay rows, a sequence's last partial chunk) never hold up another's copies.
        // Load warp 1 issues the product batches instead (lane 0), as the compute warps signal
        // that their operands are written, so that no compute warp stalls while the tensor
        // pipe's queue drains.
        const int lw = warp - NC / 32;
        int *rows = s_rows[lw];
        const uint16_t *beta = static_cast<const uint16_t *>(f.beta);
        // row table of item number `n` (`it`); load warp 0 also publishes its indices and beta
        auto rows_of = [&](const Item &it, uint32_t n) {
            if (lw == 0 && lane == 0) s_items[n & 3] = it;
            for (int t = lane; t < 64; t += 32) {
                const int64_t row = local_row(pd, it.seq, it.rho, it.L, it.c0 + t);
                rows[t] = static_cast<int>(row);
                if (lw == 0) s_braw[n & 1][t] = row >= 0 ? beta[row * H + it.h] : static_cast<uint16_t>(0);
            }
            __syncwarp();
        };
        // which: 0 q, 1 k, 2 g, 3 v, 4 dO, 5 T, 6 R record, 7 Q' record
        auto stage = [&](int which, const Item &it) {
            ++armed[6 + which];
            uint64_t *bar = &bars[6 + which];
            const int t_own = max(0, it.rho - it.c0), t_end = it.nv;
            const int32_t own0 = it.row0 + it.c0 - it.rho;
            const int64_t rid = static_cast<int64_t>(it.g) * H + it.h;
            switch (which) {
            case 0: stage_chunk_rows_warp(f.q, maps.q, rows, it.h, H, t_own, t_end, own0, 0, sm + KQ + 8192, sm + KQ + 24576, bar); break;
            case 1: stage_chunk_rows_warp(f.k, maps.k, rows, it.h, H, t_own, t_end, own0, 0, sm + KQ, sm + KQ + 16384, bar); break;
            case 2: stage_chunk_rows_warp(f.g, maps.g, rows, it.h, H, t_own, t_end, own0, 0, sm + TB, sm + TB + 8192, bar); break;
            case 3: stage_chunk_rows_warp(f.v, maps.v, rows, it.h, H, t_own, t_end, own0, 0, sm + VV, sm + VV + 8192, bar); break;
            case 4: stage_chunk_rows_warp(p.d_o, maps.dout, rows, it.h, H, t_own, t_end, own0, t_own, sm + DO,
                                          sm + DO + 16384, bar); break;
            case 5:
                if (lane == 0) {
                    tc::mbar_expect_tx(bar, 8192);
                    tc::tma_load_2d(sm + TT, &maps.rec_t, 0, static_cast<int>(rid * (kRecBytes / 128) + 2 * D), bar);
                }
                break;
            case 6:
                if (lane == 0) {
                    tc::mbar_expect_tx(bar, 32768);
                    tc::tma_load_2d(sm + RR, &maps.rec_s, 0, static_cast<int>(rid * (kRecBytes / 256)), bar);
                    tc::tma_load_2d(sm + RR + 16384, &maps.rec_s, 64, static_cast<int>(rid * (kRecBytes / 256)), bar);
                }
                break;
            default:
                if (lane == 0) {
                    tc::mbar_expect_tx(bar, 32768);
                    tc::tma_load_2d(sm + QQ, &maps.dch, 0, static_cast<int>(rid * D), bar);
                    tc::tma_load_2d(sm + QQ + 16384, &maps.dch, 64, static_cast<int>(rid * D), bar);
                }
                break;
            }
        };
        // the product batches of every item, in order, each once the compute warps signal that
        // its operands are in place (lane 0 of load warp 1)
        auto issue_products = [&]() {
            const uint32_t a = tc::smem_addr(sm);
            for (uint32_t n = 0; static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(n) * gridDim.x < n_items; ++n) {
                const uint32_t ph = n & 1;
                // B1: [A; P] = [Kp; Qp] Km^T;  X = R Kp^T;  dU = Km Q'^T (M = 64, rows t)
                if (!poll_bar(&rdy[0], ph, &s_fail)) return;
                tc::fence_after_sync();
                {
                    const uint32_t id = tc::idesc_bf16(128, 64);
                    tc::mma_tile(tAP, a + KQ, 16384, a + KM, 8192, 128, id, false);
                    tc::mma_tile(tX, a + RR, 16384, a + KQ, 16384, 128, id, false);
                    tc::mma_op(tDU, tc::Opnd{a + KM, 8192, false}, tc::Opnd{a + QQ, 16384, false}, 64, 128, 128, false);
                    tc::mma_commit(&bars[0]);
                    ++armed[0];
                }
                // B2: U^T = Y^T Tb^T;  dU += P^T dO (P and dO read MN-major)
                if (!poll_bar(&rdy[1], ph, &s_fail)) return;
                tc::fence_after_sync();
                tc::mma_op(tX, tc::Opnd{a + YT, 16384, false}, tc::Opnd{a + TB, 8192, false}, 128, 64, 64, false);
                tc::mma_op(tDU, tc::Opnd{a + PT, 8192, true}, tc::Opnd{a + DO, 16384, true}, 64, 128, 64, true);
                tc::mma_commit(&bars[1]);
                ++armed[1];
                // B3a: Z = T^T dU (M = 64; T and dU read MN-major; 128 columns from tX);  dP = dO U^T
                // (M = 64);  Km' = Q'^T U^T (the last read of Q': Z overwrites it once B3a is done);
                // B3b: dQp^T = R^T dO^T
                if (!poll_bar(&rdy[2], ph, &s_fail)) return;
                tc::fence_after_sync();
                tc::mma_op(tX, tc::Opnd{a + TT, 8192, true}, tc::Opnd{a + DX, 16384, true}, 64, 128, 64, false);
                tc::mma_op(tDT, tc::Opnd{a + DO, 16384, false}, tc::Opnd{a + VV, 16384, true}, 64, 64, 128, false);
                tc::mma_op(tKM, tc::Opnd{a + QQ, 16384, true}, tc::Opnd{a + VV, 16384, true}, 128, 64, 128, false);
                tc::mma_commit(&bars[2]);
                ++armed[2];
                tc::mma_op(tDY, tc::Opnd{a + RR, 16384, true}, tc::Opnd{a + DO, 16384, false}, 128, 64, 128, false);
                tc::mma_commit(&bars[5]);
                ++armed[5];
                // B4a: [W D] = Z [U^T Y^T] (M = 128: rows 64-127 of the Z operand are padding, so row t
                // lands in lane t, next to A; N = 128: U^T and Y^T are the two 64-column blocks of one
                // MN-major operand);  B4b: dKp^T = -R^T dY^T
                if (!poll_bar(&rdy[3], ph, &s_fail)) return;
                tc::fence_after_sync();
                tc::mma_op(tX, tc::Opnd{a + QQ, 16384, false}, tc::Opnd{a + VV, YT - VV, true}, 128, 128, 128, false);
                tc::mma_commit(&bars[3]);
                ++armed[3];
                tc::mma_op(tDT, tc::Opnd{a + RR, 16384, true}, tc::Opnd{a + DX, 16384, false}, 128, 64, 128, false);
                tc::mma_commit(&bars[14]);
                ++armed[14];
                // B6: [dQp^T dKp^T] += Km^T [dP; dA]^T (N = 128);  Km' += Kp^T dA + Qp^T dP with Kp^T
                // and Qp^T from their bf16 copies in TMEM (lane = channel, column = row pair), so the
                // [Kp; Qp] tile is free once B1 is done
                if (!poll_bar(&rdy[4], ph, &s_fail)) return;
                tc::fence_after_sync();
                tc::mma_op(tDY, tc::Opnd{a + KM, 8192, true}, tc::Opnd{a + DP, 16384, false}, 128, 128, 64, true);
                {
                    const uint32_t id = tc::idesc_bf16(128, 64, false, true);
                    const tc::Opnd da{a + WA, 8192, true}, dp{a + DP, 8192, true};
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) tc::mma_bf16_ta(tKM, tPK + kk * 8, tc::opnd_desc(da, kk), id, 1u);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) tc::mma_bf16_ta(tKM, tPK + 32 + kk * 8, tc::opnd_desc(dp, kk), id, 1u);
                }
                tc::mma_commit(&bars[4]);
                ++armed[4];
            }
        };
        // lane 0 waits for a product batch of the compute warps (its operands are then free)
        auto wait_free = [&](int b, uint32_t ph) -> bool {
            int ok = 1;
            if (lane == 0) ok = poll_bar(&bars[b], ph, &s_fail) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            return ok != 0;
        };
        int32_t item = blockIdx.x;
        if (item < n_items) {
            const Item it = item_of(pd, chunk_begin, H, item);
            rows_of(it, 0u);
            if (lw == 0) { stage(2, it); stage(5, it); stage(6, it); stage(7, it); }
            else if (lw == 2) { stage(0, it); stage(3, it); }
            else if (lw == 3) { stage(1, it); stage(4, it); }
        }
        if (lw == 1) {
            if (lane == 0) issue_products();
        } else {
            for (uint32_t n = 0; item < n_items; item += gridDim.x, ++n) {
                const int32_t nxt = item + gridDim.x;
                if (nxt >= n_items) break;
                const uint32_t ph = n & 1;
                const Item nx = item_of(pd, chunk_begin, H, nxt);
                rows_of(nx, n + 1);
                if (lw == 0) {
                    if (!wait_free(1, ph)) break;            // B2 done: Tb and P (TB..PT) are free
                    stage(2, nx);
                    if (!wait_free(2, ph)) break;            // B3a done: T is free
                    stage(5, nx);
                    if (!wait_free(14, ph)) break;           // B4b done: R and Q' (then Z) are free
                    stage(6, nx);
                    stage(7, nx);
                } else {
                    if (!wait_free(0, ph)) break;            // B1 done: the [Kp; Qp] tile is free
                    stage(lw == 2 ? 0 : 1, nx);
                    if (!wait_free(lw == 2 ? 3 : 5, ph)) break;   // B4a: U^T (over v) / B3b: dO rows
                    stage(lw == 2 ? 3 : 4, nx);
                }
            }
        }
        // every copy issued lands before shared memory is released
        tc::cp_async_wait_all();
        __syncwarp();
        // (the issuer: every product batch it issued completes before TMEM is released)
        if (lane == 0 && *reinterpret_cast<volatile int *>(&s_fail))
            for (int i = 0; i < 15; ++i)
                if (armed[i] > 0 && !tc::mbar_wait(&bars[i], (armed[i] - 1) & 1, 200000000LL))
                    dev_error(pd, kDevErrTimeout, -1, i);
    } else {
        // ================= compute warps ===================================================
        int32_t item = blockIdx.x;
        uint32_t ph = 0;
        bool tfail = false;                             // thread 0: a wait of its own ran out
        auto poll = [&](int b) {
            if (tid == 0 && !tfail) tfail = !poll_bar(&bars[b], ph, &s_fail);
        };
        // the compute warps meet; all of them stop when thread 0's waits failed or the load
        // warp recorded a failure
        auto meet = [&]() -> bool {
            const bool stop = csync_or(tid == 0 && (tfail || *reinterpret_cast<volatile int *>(&s_fail) != 0));
            tc::fence_after_sync();
            if (stop && tid == 0) *reinterpret_cast<volatile int *>(&s_fail) = 1;
            return !stop;
        };
        for (uint32_t n_done = 0; item < n_items; item += gridDim.x, ++n_done) {
            ph = n_done & 1;
            // ---- pass A: sums of g over row quarters (g of this item sits in TB..PT) -----------
            poll(8);
            if (!meet()) break;
            const Item &I = s_items[n_done & 3];            // written by the load warp before g
            cur_seq = I.seq; cur_h = I.h;
            const int t_own = max(0, I.rho - I.c0), t_end = I.nv;
            {
                const int c = jv, q4 = cg;
                float s_ = 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) s_ += bf(sm + TB + (c >> 6) * 8192 + sw64(q4 * 16 + u, c & 63));
                vqs[q4 * 128 + c] = s_;
                if (tid < 64) vbeta[tid] = __bfloat162float(__ushort_as_bfloat16(s_braw[ph][tid]));
            }
            csync();
            if (tid < 128) {
                const int c = tid;
                float gl = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) gl += vqs[q * 128 + c];
                const float m = 0.5f * gl;                  // the reference: Gamma_L / 2
                if (-m > kMaxExpArg) dev_error(pd, kDevErrDecayRange, I.seq, I.c0);
                vm2[c] = m * kLog2e;
            }
            poll(6);
            poll(7);
            if (!meet()) break;
            // ---- pass B: Kp, Qp in place, Km; gamma and the bf16 Kp, Qp (pairs) into TMEM ------
            {
                const int c = jv, q4 = cg;
                float gam = 0.f;
#pragma unroll
                for (int q = 0; q < 3; ++q) gam += q < q4 ? vqs[q * 128 + c] : 0.f;
                const float m2 = vm2[c], sc = f.scale;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float g2v[8];
                    uint32_t kpk[4], qpk[4];
#pragma unroll
                    for (int u = 0; u < 8; u += 2) {
                        float kp2[2], qp2[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int t = q4 * 16 + hh * 8 + u + e;
                            const uint32_t o = (c >> 6) * 16384 + sw64(t, c & 63), oq = (c >> 6) * 16384 + sw64(64 + t, c & 63);
                            gam += bf(sm + TB + (c >> 6) * 8192 + sw64(t, c & 63));
                            const float kk = bf(sm + KQ + o), qq = bf(sm + KQ + oq);
                            const float x = fmaf(gam, kLog2e, -m2);
                            const float e1 = ex2(x), e2 = ex2(-x);
                            const __nv_bfloat16 kpb = __float2bfloat16_rn(kk * e1), qpb = __float2bfloat16_rn(sc * qq * e1);
                            *reinterpret_cast<__nv_bfloat16 *>(sm + KQ + o) = kpb;
                            *reinterpret_cast<__nv_bfloat16 *>(sm + KQ + oq) = qpb;
                            *reinterpret_cast<__nv_bfloat16 *>(sm + KM + (c >> 6) * 8192 + sw64(t, c & 63)) =
                                __float2bfloat16_rn(kk * e2);
                            g2v[u + e] = gam * kLog2e;
                            kp2[e] = __bfloat162float(kpb);
                            qp2[e] = __bfloat162float(qpb);
                        }
                        kpk[u / 2] = tc::pack_bf16(kp2[0], kp2[1]);
                        qpk[u / 2] = tc::pack_bf16(qp2[0], qp2[1]);
                    }
                    tmem_st8f(tGM + lane_off + q4 * 16 + hh * 8, g2v);
                    tmem_st4u(tPK + lane_off + q4 * 8 + hh * 4, kpk);
                    tmem_st4u(tPK + lane_off + 32 + q4 * 8 + hh * 4, qpk);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            // ---- B1 once the records are in (pass B's tiles and TMEM copies are written) ------------
            poll(12);
            poll(13);
            tc::fence_smem_to_async();
            tc::fence_before_sync();
            if (!meet()) break;
            // ---- B1: [A; P] = [Kp; Qp] Km^T;  X = R Kp^T;  dU = Km Q'^T (M = 64, rows t) ---------------
            if (tid == 0) mbar_arrive_one(&rdy[0]);         // operands written: the issuer goes
            // ---- while B1 runs: colsum(Q' .* R) (dGamma_L's first term); Tb = T diag(beta) -------
            {
                // warp w: logical 8-column chunk w (atom w / 8) of every row; lane: rows lane + 32 i
                const int jl = warp & 7, atom = warp >> 3, col0 = atom * 64 + jl * 8;
                float dot[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane + 32 * i;
                    const uint32_t off = atom * 16384 + r * 128 + ((jl ^ (r & 7)) << 4);
                    float vr[8], vq[8];
                    unpack8(*reinterpret_cast<const uint4 *>(sm + RR + off), vr);
                    unpack8(*reinterpret_cast<const uint4 *>(sm + QQ + off), vq);
#pragma unroll
                    for (int k = 0; k < 8; ++k) dot[k] += vr[k] * vq[k];
                }
                // sum the 8 columns over the 32 lanes: three halving exchanges (each lane keeps the
                // half of its columns selected by one lane bit), then two plain ones
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const bool hi = lane & 16;
                    const float send = hi ? dot[k] : dot[k + 4];
                    const float keep = hi ? dot[k + 4] : dot[k];
                    dot[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const bool hi = lane & 8;
                    const float send = hi ? dot[k] : dot[k + 2];
                    const float keep = hi ? dot[k + 2] : dot[k];
                    dot[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                {
                    const bool hi = lane & 4;
                    const float send = hi ? dot[0] : dot[1];
                    const float keep = hi ? dot[1] : dot[0];
                    dot[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                }
                dot[0] += __shfl_xor_sync(0xffffffffu, dot[0], 2);
                dot[0] += __shfl_xor_sync(0xffffffffu, dot[0], 1);
                // lane bits 4, 3, 2 pick the column: 4 * b4 + 2 * b3 + b2
                if ((lane & 3) == 0)
                    vdgl[col0 + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1)] = dot[0];
            }
            poll(11);
            if (!meet()) break;
            {
                const int t = tid >> 3, j = tid & 7;              // Tb: row t, 16-byte chunk j
                const uint4 w = *reinterpret_cast<const uint4 *>(sm + TT + t * 128 + (j << 4));
                const int col0 = (j ^ (t & 7)) << 3;
                float v[8];
                unpack8(w, v);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] *= vbeta[col0 + i];
                *reinterpret_cast<uint4 *>(sm + TB + t * 128 + (j << 4)) = pack8(v);
            }
            poll(9);                                            // v, read below
            poll(0);
            if (!meet()) break;
            // ---- E1: P -> PT (lower with the diagonal); Y^T = V^T - X -> YT ------------------------
            {
                float r[16], pv[16];
                tld16(tAP + lane_off + cg * 16, pv);
                tld16(tX + lane_off + cg * 16, r);
                twait(pv, r);
                if (lq >= 2) {
                    const int t = jv - 64;
#pragma unroll
                    for (int j = 0; j < 16; ++j) pv[j] = (cg * 16 + j <= t) ? pv[j] : 0.f;
                    tc::st_sw128_8(sm + PT, 64, t, cg * 16, pv);
                    tc::st_sw128_8(sm + PT, 64, t, cg * 16 + 8, pv + 8);
                }
                const int dv = jv;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = cg * 16 + j;
                    r[j] = bf(sm + VV + (dv >> 6) * 8192 + sw64(t, dv & 63)) - r[j];
                }
                tc::st_sw128_8(sm + YT, 128, dv, cg * 16, r);
                tc::st_sw128_8(sm + YT, 128, dv, cg * 16 + 8, r + 8);
            }
            poll(10);                                           // dO
            tc::fence_smem_to_async();
            tc::fence_before_sync();
            if (!meet()) break;
            // ---- B2: U^T = Y^T Tb^T;  dU += P^T dO (P and dO read MN-major) ----------------------------
            if (tid == 0) mbar_arrive_one(&rdy[1]);         // operands written: the issuer goes
            poll(1);
            if (!meet()) break;
            // ---- E2: U^T -> VV (raw v is consumed), dU rows -> DX ----------------------------------------
            {
                float r[16], ua[16], ub[16];
                tld16(tX + lane_off + cg * 16, r);
                tld16(tDU + lane_off + cg * 32, ua);            // dU, M = 64: row 16 lq + lane in lanes 0-15
                tld16(tDU + lane_off + cg * 32 + 16, ub);
                twait(r, ua, ub);
                tc::st_sw128_8(sm + VV, 128, jv, cg * 16, r);
                tc::st_sw128_8(sm + VV, 128, jv, cg * 16 + 8, r + 8);
                if (lane < 16) {
                    const int t = 16 * lq + lane, dv0 = cg * 32;
                    tc::st_sw128_8(sm + DX, 128, t, dv0, ua);
                    tc::st_sw128_8(sm + DX, 128, t, dv0 + 8, ua + 8);
                    tc::st_sw128_8(sm + DX, 128, t, dv0 + 16, ub);
                    tc::st_sw128_8(sm + DX, 128, t, dv0 + 24, ub + 8);
                }
            }
            csync_mma();
            // ---- B3: Z = T^T dU (M = 64, rows t; T and dU read MN-major; 128 columns from tX);
            //      dP = dO U^T (M = 64);  Km' = Q'^T U^T;  dQp^T = R^T dO^T (dO is then free) ----------------
            if (tid == 0) mbar_arrive_one(&rdy[2]);         // operands written: the issuer goes
            poll(2);
            if (!meet()) break;
            // ---- E3: Z rows -> QQ (over Q'); dY = diag(beta) Z: -dY rows -> DX; dP -> DP;
            //      sum_t Km Km' for dGamma_L ---------------------------------------------------------------
            {
                float za[16], zb[16], a[16];
                tld16(tX + lane_off + cg * 32, za);             // Z, M = 64: row 16 lq + lane in lanes 0-15
                tld16(tX + lane_off + cg * 32 + 16, zb);
                tld16(tDT + lane_off + cg * 16, a);             // dP, M = 64
                twait(za, zb, a);
                if (lane < 16) {
                    const int t = 16 * lq + lane, dv0 = cg * 32;
                    // Z rows: rows 0-63 of the K-major [128][64]-atom operand in QQ (rows 64-127: padding)
                    tc::st_sw128_8(sm + QQ, 128, t, dv0, za);
                    tc::st_sw128_8(sm + QQ, 128, t, dv0 + 8, za + 8);
                    tc::st_sw128_8(sm + QQ, 128, t, dv0 + 16, zb);
                    tc::st_sw128_8(sm + QQ, 128, t, dv0 + 24, zb + 8);
                    const float bt = vbeta[t];
#pragma unroll
                    for (int j = 0; j < 16; ++j) { za[j] *= bt; zb[j] *= bt; }
                    if (t < t_own && t < t_end) {
                        // a replayed row's dv goes to the replay-gradient buffer in fp32; own rows
                        // leave from DX below
                        float4 *dst = reinterpret_cast<float4 *>(
                            p.rep_grad + (static_cast<int64_t>(I.rptr + I.c0 + t) * H + I.h) * W3 + D + dv0);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            dst[q] = make_float4(za[4 * q], za[4 * q + 1], za[4 * q + 2], za[4 * q + 3]);
                            dst[4 + q] = make_float4(zb[4 * q], zb[4 * q + 1], zb[4 * q + 2], zb[4 * q + 3]);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) { za[j] = -za[j]; zb[j] = -zb[j]; }
                    tc::st_sw128_8(sm + DX, 128, t, dv0, za);
                    tc::st_sw128_8(sm + DX, 128, t, dv0 + 8, za + 8);
                    tc::st_sw128_8(sm + DX, 128, t, dv0 + 16, zb);
                    tc::st_sw128_8(sm + DX, 128, t, dv0 + 24, zb + 8);
#pragma unroll
                    for (int j = 0; j < 16; ++j) a[j] = (cg * 16 + j <= t) ? a[j] : 0.f;
                    tc::st_sw128_8(sm + DP, 64, t, cg * 16, a);
                    tc::st_sw128_8(sm + DP, 64, t, cg * 16 + 8, a + 8);
                }
            }
            {
                // sum_t Km[t][c] Km'[c][t]
                float km2[16];
                tld16(tKM + lane_off + cg * 16, km2);
                twait1(km2);
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) acc += km2[j] * bf(sm + KM + (jv >> 6) * 8192 + sw64(cg * 16 + j, jv & 63));
                vqs[cg * 128 + jv] = acc;
            }
            csync_mma();
            // ---- B4: [W D] = Z [U^T Y^T] (M = 128: rows 64-127 of the Z operand are padding, so row t
            //      lands in lane t, next to A; N = 128: U^T and Y^T are the two 64-column blocks of one
            //      MN-major operand);  dKp^T = -R^T dY^T ------------------------------------------------------
            if (tid == 0) mbar_arrive_one(&rdy[3]);         // operands written: the issuer goes
            if (tid < 128) vdgl[tid] += vqs[tid] + vqs[128 + tid] + vqs[256 + tid] + vqs[384 + tid];
            // the own rows' dv = -(the bf16 -dY rows in DX), 16 bytes per store, while B4 runs
            for (int e = tid; e < 64 * 16; e += NC) {
                const int t = e >> 4, pc = e & 15;
                if (t < t_own || t >= t_end) continue;
                const uint4 w = *reinterpret_cast<const uint4 *>(sm + DX + (pc >> 3) * 16384 + t * 128 +
                                                                 (((pc & 7) ^ (t & 7)) << 4));
                *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dv) +
                                           ((static_cast<int64_t>(I.row0) + I.c0 + t - I.rho) * H + I.h) * D + pc * 8) =
                    make_uint4(w.x ^ 0x80008000u, w.y ^ 0x80008000u, w.z ^ 0x80008000u, w.w ^ 0x80008000u);
            }
            poll(3);
            if (!meet()) break;
            // ---- E4: dM = -strict(W); dA = diag(beta) dM -> WA; dbeta = D[t][t] + rowsum(dM .* A) ----------
            {
                if (lq < 2) {
                    float w[16], d2[16], a[16];
                    tld16(tX + lane_off + cg * 16, w);
                    tld16(tDU + lane_off + cg * 16, d2);
                    tld16(tAP + lane_off + cg * 16, a);
                    twait(w, d2, a);
                    const int t = jv;
                    const float bt = vbeta[t];
                    float db = 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s = cg * 16 + j;
                        const float dm = s < t ? -w[j] : 0.f;
                        if (s < t) db += dm * a[j];         // A above the diagonal may be inf
                        if (s == t) db += d2[j];
                        w[j] = bt * dm;
                    }
                    tc::st_sw128_8(sm + WA, 64, t, cg * 16, w);
                    tc::st_sw128_8(sm + WA, 64, t, cg * 16 + 8, w + 8);
                    vqs[cg * 64 + t] = db;
                }
                csync();
                if (tid < 64) vdb[tid] = vqs[tid] + vqs[64 + tid] + vqs[128 + tid] + vqs[192 + tid];
            }
            csync_mma();
            // ---- B6: [dQp^T dKp^T] += Km^T [dP; dA]^T (N = 128);  Km' += Kp^T dA + Qp^T dP ----------------
            if (tid == 0) mbar_arrive_one(&rdy[4]);         // operands written: the issuer goes
            poll(4);
            if (!meet()) break;
            // ---- E6: dq, dk, dgamma per (channel, row); dg = suffix sums + dGamma_L -----------------------
            //      (two halves of 8 rows, the later half first, so the suffix sums run in one pass).  The
            //      rows go out through shared memory, 16 bytes per store: dq over Y^T, dk over [dP; dA],
            //      then dg over Y^T.
            {
                const int c = jv;
                const float m2 = vm2[c], sc = f.scale;
                const int64_t r0 = (static_cast<int64_t>(I.rptr + I.c0) * H + I.h) * W3 + c;   // replay rows
                const int gs = H * W3;
                __nv_bfloat16 *dqs = reinterpret_cast<__nv_bfloat16 *>(sm + YT);
                __nv_bfloat16 *dks = reinterpret_cast<__nv_bfloat16 *>(sm + DP);
                auto rows_out = [&](uint32_t from, void *to) {
                    for (int e = tid; e < 64 * 16; e += NC) {
                        const int t = e >> 4, pc = e & 15;
                        if (t < t_own || t >= t_end) continue;
                        const int64_t row = static_cast<int64_t>(I.row0) + (I.c0 + t - I.rho);
                        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(to) + (row * H + I.h) * D + pc * 8) =
                            *reinterpret_cast<const uint4 *>(sm + from + t * 256 + pc * 16);
                    }
                };
                float dgm[16];
                float run = 0.f;
#pragma unroll
                for (int hh = 1; hh >= 0; --hh) {
                    const int cb = cg * 16 + hh * 8;
                    float xq[8], xp[8], xm[8], g2v[8];
                    uint32_t kpk[4], qpk[4];
                    tld8f(tDY + lane_off + cb, xq);
                    tld8f(tDT + lane_off + cb, xp);
                    tld8f(tKM + lane_off + cb, xm);
                    tld8f(tGM + lane_off + cb, g2v);
                    tld4(tPK + lane_off + cg * 8 + hh * 4, kpk);
                    tld4(tPK + lane_off + 32 + cg * 8 + hh * 4, qpk);
                    twait8(xq, xp, xm, g2v, kpk, qpk);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int t = cb + j;
                        const float2 kp2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kpk[j >> 1]));
                        const float2 qp2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qpk[j >> 1]));
                        const float kp = (j & 1) ? kp2.y : kp2.x, qp = (j & 1) ? qp2.y : qp2.x;
                        const float km = bf(sm + KM + (c >> 6) * 8192 + sw64(t, c & 63));
                        const float x = g2v[j] - m2;
                        const float e1 = ex2(x), e2 = ex2(-x);
                        const float dqv = sc * xq[j] * e1;
                        const float dkv = xp[j] * e1 + xm[j] * e2;
                        dgm[hh * 8 + j] = xq[j] * qp + xp[j] * kp - xm[j] * km;
                        dqs[t * D + c] = __float2bfloat16_rn(dqv);
                        dks[t * D + c] = __float2bfloat16_rn(dkv);
                        if (t < t_own && t < t_end) p.rep_grad[r0 + t * gs] = dkv;
                    }
                    // suffix sums over t within this thread's rows, continuing the later half's
#pragma unroll
                    for (int j = 7; j >= 0; --j) { run += dgm[hh * 8 + j]; dgm[hh * 8 + j] = run; }
                }
                // then the later quarters' totals
                vqs[cg * 128 + c] = run;
                csync();
                rows_out(YT, p.dq);
                rows_out(DP, p.dk);
                float off = vdgl[c];
#pragma unroll
                for (int q = 1; q < 4; ++q) off += q > cg ? vqs[q * 128 + c] : 0.f;
                csync();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = cg * 16 + j;
                    const float x = dgm[j] + off;
                    dqs[t * D + c] = __float2bfloat16_rn(x);
                    if (t < t_own && t < t_end) p.rep_grad[r0 + t * gs + 2 * D] = x;
                }
                csync();
                rows_out(YT, p.dg);
            }
            if (tid < 64) {
                const int t = tid;
                const float db = vdb[t];
                if (t < t_end) {
                    if (t >= t_own)
                        static_cast<__nv_bfloat16 *>(p.dbeta)[(static_cast<int64_t>(I.row0) + (I.c0 + t - I.rho)) * H + I.h] =
                            __float2bfloat16_rn(db);
                    else
                        p.rep_grad[(static_cast<int64_t>(I.rptr + I.c0 + t) * H + I.h) * W3 + 3 * D] = db;
                }
            }
            tc::fence_before_sync();
            csync();
            tc::fence_after_sync();
        }
        if (tid == 0 && *reinterpret_cast<volatile int *>(&s_fail)) dev_error(pd, kDevErrTimeout, cur_seq, cur_h);
    }
    // ---- drain --------------------------------------------------------------------------------------
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tm, 512);
}

bool flat_map2(CUtensorMap *m, const void *base, int64_t n_rows, int cols, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(n_rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    return encode_bf16(m, base, 2, dims, strides, box);
}

}  // namespace

cudaError_t tc2_bwd_grad(const BwdParams &p, const PlanDev &pd, int32_t chunk_begin, int32_t n_items,
                         cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_grad_tc2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(g2::bytes));
    if (e != cudaSuccess) return e;
    if (n_items <= 0) return cudaSuccess;
    const int H = p.f.H;
    const int64_t n_rec = pd.n_chunks * H;
    if (n_rec * (kRecBytes / 128) > INT32_MAX) return cudaErrorInvalidValue;   // TMA coordinates are int32
    GradMaps2 maps;
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(pd.C)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
        (void)dims; (void)strides;
        const void *src[5] = {p.f.q, p.f.k, p.f.g, p.f.v, p.d_o};
        RowMaps *dst[5] = {&maps.q, &maps.k, &maps.g, &maps.v, &maps.dout};
        for (int i = 0; i < 5; ++i)
            if (!encode_row_maps(dst[i], src[i], H, pd.C)) return cudaErrorInvalidValue;
        if (!flat_map2(&maps.rec_s, p.f.chunk_states, n_rec * (kRecBytes / 256), 128, 128) ||
            !flat_map2(&maps.rec_t, p.f.chunk_states, n_rec * (kRecBytes / 128), 64, 64) ||
            !flat_map2(&maps.dch, p.dchunk, n_rec * D, 128, 128))
            return cudaErrorInvalidValue;
    }
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    kda_bwd_grad_tc2<<<min(n_items, nsm), NT, g2::bytes, st>>>(p, pd, chunk_begin, n_items, maps);
    return cudaGetLastError();
}

}  // namespace harts
