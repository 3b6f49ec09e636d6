// Branch attention over the compact layout, forward and backward, tensor cores (bf16,
// d = 128).
//
// HARTS (page "HARTS ... 精读", section 4.3, MLA paragraph; summary page, section 4 "MLA
// execution"; figures page, Figure C.1(c)): a branch's queries (its own l tokens) attend
// to the keys and values of its ancestors and itself (h + l) with bottom-right causal
// alignment: own query t sees view entries j <= h + t.  The ancestor view is a temporary
// gather inside the kernel; outputs go back to the unique compact rows.  The core is plain
// softmax attention on projected inputs: o = softmax(scale q k^T) v per head.
//
// Forward: one block per (sequence, 128-query tile, head); the planner orders the tiles
// tree by tree (longest first within a tree) with the heads innermost, so the key / value
// rows a tree's blocks share stay in L2.  The block's warps have fixed roles and meet only
// at mbarriers (every wait bounded):
//   loaders (2 threads) Q and the K_j of each 128-row key tile into a three-slot ring, and
//                       the V_j into a two-slot ring, by tiled TMA over the padded view; a
//                       slot is refilled once the product that reads it has completed
//   S issuer (1 thread) S_j = Q K_j^T into TMEM buffer j mod 2 once the softmax has read
//                       S_{j-2}
//   O issuer (1 thread) O += P_j V_j (P from TMEM buffer j mod 2, V read MN-major)
//   softmax (8 warps)   one query row and 64 columns per thread; scores in base-2 units
//                       (scale * log2 e folded into one FMA); the two warps holding a row
//                       exchange its max through shared memory; the running max moves,
//                       and O is rescaled in TMEM, only when a row max grows by more than
//                       2^8 -- any common offset gives the same softmax, the threshold
//                       only bounds P by 256; P goes to TMEM as bf16 pairs
// Masking runs only on tiles that reach past the first query's causal limit.  A timeout
// records code 3 in the plan's error word, stops issuing products and drains the ones
// in flight.
#include <algorithm>
#include <cstring>

#include "kda_common.cuh"
#include "tc_primitives.cuh"
#include "tensor_map.h"

namespace harts {
namespace {

constexpr int AD = 128, AT = kAttnTile;
constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;               // running max moves when a row max grows by more

namespace at_sm {
constexpr uint32_t Q = 0, K0 = 32768, V0 = 131072;    // K ring: 3 slots of 32 KB; V ring: 2 slots
constexpr uint32_t Max = 196608;                  // [2 tiles][2 halves][128] fp32 row maxima
constexpr uint32_t Sum = Max + 2048;              // [2 halves][128] fp32 row sums
constexpr uint32_t bytes = Sum + 1024 + 1024;     // + alignment slack
}  // namespace at_sm

constexpr int kKSlots = 3;

// Roles of the forward's 11 warps.
constexpr int kFwdSoftmaxWarps = 8, kFwdMmaWarp = 8, kFwdPvWarp = 11, kFwdLoadWarp0 = 9, kFwdLoadWarps = 2;
constexpr int kFwdThreads = 12 * 32;
constexpr int kSoftThreads = kFwdSoftmaxWarps * 32;

struct AttnParams {
    const __nv_bfloat16 *q, *k, *v;
    __nv_bfloat16 *o;
    float *lse;
    int32_t H;
    float scale;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(tc::smem_addr(bar)) : "memory");
}

// Waits unless the block has already failed; a timeout records 1 + 2 * which + phase.
__device__ __forceinline__ void wait_or_fail(uint64_t *bar, uint32_t phase, int which, int *s_fail) {
    if (*reinterpret_cast<volatile int *>(s_fail)) return;
    if (!tc::mbar_wait(bar, phase)) atomicCAS(s_fail, 0, 1 + 2 * which + static_cast<int>(phase));
}

__device__ __forceinline__ bool failed(int *s_fail) { return *reinterpret_cast<volatile int *>(s_fail) != 0; }

// Tensor maps of [C][H][128] bf16 tensors: boxes of 64 channels x 128 rows (q, dO) and of
// 64 channels x (8 << j) rows, j = 0..4 (k, v: any 8-aligned run of a view tile).
struct AttnMaps {
    CUtensorMap q, dout, k[5], v[5];
};

// Issue the TMA boxes of padded-view key tile `kt` of sequence `sq` into a [128][128] SW128
// tile (two 64-channel halves 16 KB apart), 32 KB in all; `ri` walks the sequence's runs
// across calls.  Runs start at multiples of 8 and pad up to one; positions past the view
// read rows beyond the tensor (zeros).
__device__ __forceinline__ void tma_view_tile(const CUtensorMap *maps, uint8_t *tile, const PlanDev &pd, int32_t sq,
                                              int32_t kt, int h, int &ri, uint64_t *bar) {
    const int32_t r_end = pd.attn_rptr[sq + 1];
    int x = 0;
    while (x < AT) {
        const int32_t pos = kt * AT + x;
        int32_t ps = 0, pend = 0, row = 0;
        while (ri < r_end) {
            ps = pd.attn_runs[3 * ri];
            row = pd.attn_runs[3 * ri + 1];
            pend = ps + ((pd.attn_runs[3 * ri + 2] + 7) & ~7);
            if (pend > pos) break;
            ++ri;
        }
        int n, src;
        if (ri < r_end && ps <= pos) {
            n = min(AT - x, pend - pos);
            src = row + (pos - ps);
        } else {
            n = AT - x;
            src = static_cast<int32_t>(pd.C);             // past the last row: zero fill
        }
        while (n > 0) {
            const int j = n >= 128 ? 4 : n >= 64 ? 3 : n >= 32 ? 2 : n >= 16 ? 1 : 0;
            const int R = 8 << j;
            tc::tma_load_3d(tile + x * 128, &maps[j], 0, h, src, bar);
            tc::tma_load_3d(tile + 16384 + x * 128, &maps[j], 64, h, src, bar);
            x += R;
            src += R;
            n -= R;
        }
    }
}

// Validity of padded-view positions base .. base + 31 (base a multiple of 32): real
// ancestor positions (planner bitmask) and own positions (hp .. hp + own - 1).
__device__ __forceinline__ uint32_t view_bits(const PlanDev &pd, int32_t sq, int32_t hp, int32_t own, int32_t base) {
    uint32_t m = 0;
    if (base < hp) m = static_cast<uint32_t>(pd.attn_mask[pd.attn_mptr[sq] + base / 32]);
    const int32_t lo = max(base, hp), hi = min(base + 32, hp + own);
    if (lo < hi) {
        const int a = lo - base, n = hi - lo;
        m |= (n == 32 ? 0xffffffffu : ((1u << n) - 1u)) << a;
    }
    return m;
}

// Barriers of the forward (index into bars[]).
// Per S buffer: S full, S released; per P buffer: P written, the O that read it done (which
// also says every earlier O is done: one thread issues them all, in order).  Every barrier
// that several warps arrive on, or that a wait may lag by one use, is per buffer: a warp can
// then never arrive for use j + 2 of a barrier before use j completed, so arrivals of
// different steps never mix in one phase and no parity check sees a barrier two phases
// ahead.
enum FwdBar { bQ = 0, bKF = 1, bKE = 4, bVF = 7, bVE = 9, bSF = 11, bSE = 13, bPF = 15, bPD = 17, bN = 19 };

// O (+)= P V with P (bf16, packed in pairs) read from TMEM: one row per lane, 8 columns per
// 16 keys.
// Two TMEM loads of one warp, issued back to back and waited for once; the wait names the
// destination registers so that no use of them can move above it.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&u)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld16x2(uint32_t (&a)[16], uint32_t (&b)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                   "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]),
                   "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
                   "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15])
                 :: "memory");
}

__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, float (&ra)[16], uint32_t tb, float (&rb)[16]) {
    uint32_t(&ua)[16] = reinterpret_cast<uint32_t(&)[16]>(ra);
    uint32_t(&ub)[16] = reinterpret_cast<uint32_t(&)[16]>(rb);
    tmem_ld16_issue(ta, ua);
    tmem_ld16_issue(tb, ub);
    tmem_wait_ld16x2(ua, ub);
}

// Two 16-column TMEM stores of one warp, then one wait.
__device__ __forceinline__ void tmem_st16x2(uint32_t ta, const uint32_t (&a)[16], uint32_t tb, const uint32_t (&b)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(ta), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]),
           "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15])
        : "memory");
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(tb), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(b[4]), "r"(b[5]), "r"(b[6]), "r"(b[7]),
           "r"(b[8]), "r"(b[9]), "r"(b[10]), "r"(b[11]), "r"(b[12]), "r"(b[13]), "r"(b[14]), "r"(b[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 columns of one TMEM lane per thread (warp-collective), then wait for the stores.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&u)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]),
           "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]), "r"(u[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mma_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_saddr, bool accumulate) {
    const uint32_t id = tc::idesc_bf16(AT, AD, false, true);
    for (int kk = 0; kk < AT / 16; ++kk) {
        const uint64_t bd = tc::desc_sw128_mn(v_saddr + kk * 2048, 16384);
        const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                     :: "r"(d_tmem), "r"(p_tmem + kk * 8), "l"(bd), "r"(id), "r"(acc) : "memory");
    }
}

__global__ void __launch_bounds__(kFwdThreads, 1) attn_fwd_tc(AttnParams p, PlanDev pd,
                                                                const __grid_constant__ AttnMaps maps) {
    using namespace at_sm;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    __shared__ uint64_t bars[bN];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int32_t h = blockIdx.x % H, qi = blockIdx.x / H;
    const int32_t sq = pd.attn_qt[2 * qi], qt = pd.attn_qt[2 * qi + 1];
    const int32_t hh = pd.attn_hp[sq];                  // padded ancestor length
    const int32_t row0 = pd.seq_row0[sq], own = pd.seq_nown[sq];
    const int32_t q0 = qt * AT, nq = min(AT, own - q0);
    const int32_t n_kt = (hh + q0 + nq - 1) / AT + 1;   // key tiles covering every visible entry

    if (tid == 0) {
        tc::mbar_init(&bars[bQ], 1);
        for (int i = 0; i < kKSlots; ++i) {
            tc::mbar_init(&bars[bKF + i], 1);
            tc::mbar_init(&bars[bKE + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&bars[bVF + i], 1);
            tc::mbar_init(&bars[bVE + i], 1);
            tc::mbar_init(&bars[bSF + i], 1);
            tc::mbar_init(&bars[bSE + i], kSoftThreads);
            tc::mbar_init(&bars[bPD + i], 1);
        }
        for (int i = 0; i < 2; ++i) tc::mbar_init(&bars[bPF + i], kSoftThreads);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == kFwdMmaWarp) {
        tc::tmem_alloc(&s_tmem, 512);
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem, tO = tm + 256, tPb = tm + 384;

    if (warp >= kFwdLoadWarp0 && warp < kFwdLoadWarp0 + kFwdLoadWarps) {
        // ---- loaders: one thread for Q and the K ring, one for the V ring, tiled TMA
        if (lane == 0) {
            const int is_v = warp - kFwdLoadWarp0;
            int ri = pd.attn_rptr[sq];
            if (!is_v) {
                tc::mbar_expect_tx(&bars[bQ], 32768);
                tc::tma_load_3d(sm + Q, &maps.q, 0, h, row0 + q0, &bars[bQ]);
                tc::tma_load_3d(sm + Q + 16384, &maps.q, 64, h, row0 + q0, &bars[bQ]);
            }
            const int nslot = is_v ? 2 : kKSlots;
            for (int32_t kt = 0; kt < n_kt; ++kt) {
                const int b = kt % nslot, use = kt / nslot;
                if (use > 0) wait_or_fail(&bars[(is_v ? bVE : bKE) + b], (use - 1) & 1, 2, &s_fail);
                uint64_t *full = &bars[(is_v ? bVF : bKF) + b];
                tc::mbar_expect_tx(full, 32768);
                tma_view_tile(is_v ? maps.v : maps.k, sm + (is_v ? V0 : K0) + b * 32768, pd, sq, kt, h, ri, full);
            }
        }
    } else if (warp == kFwdMmaWarp) {
        // ---- S issuer: S_j = Q K_j^T into S buffer j % 2 once the softmax has read S_{j-2}
        if (lane == 0) {
            const tc::Opnd aQ{tc::smem_addr(sm + Q), 16384, false};
            uint32_t nc_s0 = 0, nc_s1 = 0;
            wait_or_fail(&bars[bQ], 0, 0, &s_fail);
            for (int32_t kt = 0; kt < n_kt && !failed(&s_fail); ++kt) {
                const int b = kt & 1, ks = kt % kKSlots;
                wait_or_fail(&bars[bKF + ks], (kt / kKSlots) & 1, 0, &s_fail);
                if (kt >= 2) wait_or_fail(&bars[bSE + b], ((kt - 2) >> 1) & 1, 1, &s_fail);
                tc::fence_after_sync();
                if (failed(&s_fail)) break;
                tc::mma_op(tm + b * 128, aQ, tc::Opnd{tc::smem_addr(sm + K0 + ks * 32768), 16384, false},
                           AT, AT, AD, false);
                tc::mma_commit(&bars[bSF + b]);
                tc::mma_commit(&bars[bKE + ks]);
                if (b) ++nc_s1; else ++nc_s0;
            }
            if (failed(&s_fail)) {                      // drain the products still in flight
                dev_error(pd, kDevErrTimeout, sq, h);
                if (nc_s0) tc::mbar_wait(&bars[bSF], (nc_s0 - 1) & 1, 1000000000LL);
                if (nc_s1) tc::mbar_wait(&bars[bSF + 1], (nc_s1 - 1) & 1, 1000000000LL);
            }
        }
    } else if (warp == kFwdPvWarp) {
        // ---- O issuer: O += P_j V_j once P_j is written (P from TMEM buffer j % 2)
        if (lane == 0) {
            uint32_t nc_o0 = 0, nc_o1 = 0;
            for (int32_t kt = 0; kt < n_kt && !failed(&s_fail); ++kt) {
                const int b = kt & 1;
                wait_or_fail(&bars[bPF + b], (kt >> 1) & 1, 1, &s_fail);
                wait_or_fail(&bars[bVF + b], (kt >> 1) & 1, 0, &s_fail);
                tc::fence_after_sync();
                if (failed(&s_fail)) break;
                mma_pv(tO, tPb + b * 64, tc::smem_addr(sm + V0 + b * 32768), kt > 0);
                tc::mma_commit(&bars[bPD + b]);
                tc::mma_commit(&bars[bVE + b]);
                if (b) ++nc_o1; else ++nc_o0;
            }
            if (failed(&s_fail)) {                      // drain the products still in flight
                if (nc_o0) tc::mbar_wait(&bars[bPD], (nc_o0 - 1) & 1, 1000000000LL);
                if (nc_o1) tc::mbar_wait(&bars[bPD + 1], (nc_o1 - 1) & 1, 1000000000LL);
            }
        }
    } else {
        // ---- softmax: one query row and 64 columns per thread
        float *smax = reinterpret_cast<float *>(sm + Max), *ssum = reinterpret_cast<float *>(sm + Sum);
        const int lg = warp & 3, half = warp >> 2;
        const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
        const int qrow = lg * 32 + lane;
        const int32_t vis = hh + q0 + qrow;
        const float c = p.scale * kLog2e;
        float m_run = -INFINITY, l_half = 0.f;
        // validity of this thread's 64 columns, one tile ahead
        uint32_t nb0 = view_bits(pd, sq, hh, own, half * 64), nb1 = view_bits(pd, sq, hh, own, half * 64 + 32);
        for (int32_t kt = 0; kt < n_kt; ++kt) {
            const int b = kt & 1;
            const uint32_t vb0 = nb0, vb1 = nb1;
            if (kt + 1 < n_kt) {
                nb0 = view_bits(pd, sq, hh, own, (kt + 1) * AT + half * 64);
                nb1 = view_bits(pd, sq, hh, own, (kt + 1) * AT + half * 64 + 32);
            }
            wait_or_fail(&bars[bSF + b], (kt >> 1) & 1, 1, &s_fail);
            tc::fence_after_sync();
            float s[64];
            tc::tmem_ld32x2(tm + b * 128 + lane_off + half * 64, *reinterpret_cast<float(*)[32]>(s),
                        tm + b * 128 + lane_off + half * 64 + 32, *reinterpret_cast<float(*)[32]>(s + 32));
            tc::fence_before_sync();
            mbar_arrive(&bars[bSE + b]);
            const int32_t lim = vis - (kt * AT + half * 64);
            if (__any_sync(0xffffffffu, (vb0 & vb1) != 0xffffffffu || lim < 63)) {
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const bool ok = ((i < 32 ? vb0 >> i : vb1 >> (i - 32)) & 1u) && i <= lim;
                    s[i] = ok ? s[i] : -INFINITY;
                }
            }
            float mp[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mp[i] = fmaxf(fmaxf(fmaxf(s[i], s[i + 8]), fmaxf(s[i + 16], s[i + 24])),
                              fmaxf(fmaxf(s[i + 32], s[i + 40]), fmaxf(s[i + 48], s[i + 56])));
#pragma unroll
            for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                for (int i = 0; i < w; ++i) mp[i] = fmaxf(mp[i], mp[i + w]);
            smax[(b * 2 + half) * AT + qrow] = mp[0];
            tc::fence_before_sync();                     // both halves' reads of S precede P's writes
            asm volatile("bar.sync %0, 64;" :: "r"(1 + lg) : "memory");   // the row's two warps
            tc::fence_after_sync();
            const float m_tile = c * fmaxf(smax[(b * 2) * AT + qrow], smax[(b * 2 + 1) * AT + qrow]);
            const bool move = __any_sync(0xffffffffu, m_tile > m_run + kRescaleLog2);
            float alpha = 1.f;
            if (move) {
                const float m_new = fmaxf(m_run, m_tile);
                alpha = ex2(m_run - m_new);
                m_run = m_new;
            }
            float sp[8];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                s[i] = ex2(fmaf(s[i], c, -m_run));
                sp[i & 7] = (i < 8) ? s[i] : sp[i & 7] + s[i];
            }
#pragma unroll
            for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                for (int i = 0; i < w; ++i) sp[i] += sp[i + w];
            l_half = l_half * alpha + sp[0];
            if (kt >= 2) wait_or_fail(&bars[bPD + b], ((kt - 2) >> 1) & 1, 1, &s_fail);
            tc::fence_after_sync();
            {
                float w[32];
                uint32_t *u = reinterpret_cast<uint32_t *>(w);
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] = tc::pack_bf16(s[2 * i], s[2 * i + 1]);
                tc::tmem_st32(tPb + b * 64 + lane_off + half * 32, w);
            }
            if (move && kt > 0) {
                wait_or_fail(&bars[bPD + ((kt - 1) & 1)], ((kt - 1) >> 1) & 1, 1, &s_fail);  // O_{kt-1} done
                tc::fence_after_sync();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float r[32];
                    tc::tmem_ld32(tO + lane_off + half * 64 + hf * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] *= alpha;
                    tc::tmem_st32(tO + lane_off + half * 64 + hf * 32, r);
                }
            }
            tc::fence_before_sync();
            mbar_arrive(&bars[bPF + b]);
        }
        wait_or_fail(&bars[bPD + ((n_kt - 1) & 1)], ((n_kt - 1) >> 1) & 1, 1, &s_fail);   // every O done
        tc::fence_after_sync();
        ssum[half * AT + qrow] = l_half;
        asm volatile("bar.sync %0, 64;" :: "r"(1 + lg) : "memory");
        if (!failed(&s_fail)) {
            const float l = ssum[qrow] + ssum[AT + qrow], inv = 1.f / l;
            const int64_t row = static_cast<int64_t>(row0) + q0 + qrow;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float r[32];
                tc::tmem_ld32(tO + lane_off + half * 64 + hf * 32, r);
                if (qrow < nq) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.o + (row * H + h) * AD + half * 64 + hf * 32);
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 w;
                        w.x = tc::pack_bf16(r[i] * inv, r[i + 1] * inv);
                        w.y = tc::pack_bf16(r[i + 2] * inv, r[i + 3] * inv);
                        w.z = tc::pack_bf16(r[i + 4] * inv, r[i + 5] * inv);
                        w.w = tc::pack_bf16(r[i + 6] * inv, r[i + 7] * inv);
                        dst[i / 8] = w;
                    }
                }
            }
            if (p.lse && half == 0 && qrow < nq) p.lse[row * H + h] = m_run * kLn2 + logf(l);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kFwdMmaWarp) tc::tmem_dealloc(tm, 512);
}

// ======================================================================================
// Backward.  With D_t = sum_d dO_t o_t (per query row and head), P = softmax(scale S):
//   dV_j = sum_t P_tj dO_t,  dS_tj = scale P_tj (dP_tj - D_t) with dP = dO V^T,
//   dQ_t = sum_j dS_tj K_j,  dK_j = sum_t dS_tj Q_t,
// every query row once (its own compact row), over its view.  P is recomputed from the
// forward's log-sum-exp.  The kernels form dS / scale = P (dP - D) (bf16 into the
// products) and apply the scale once, to dQ and dK as they are stored.  dQ: one block per
// (query tile, head) over the view's key tiles, as the forward.  dK, dV: one block per
// (key tile of a sequence's own rows, head) over the query tiles that see it (planner
// lists: the sequence's own tiles, causal, and the tiles of every sequence whose prefix
// runs through it, a prefix of the key tile visible).  Fixed summation orders, no
// atomics.
// ======================================================================================

__global__ void attn_bwd_prep(const __nv_bfloat16 *o, const __nv_bfloat16 *dout, float *D, int64_t rows) {
    // one warp per (row, head): 128 channels, 4 per lane
    const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    for (int64_t r = w; r < rows; r += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        const uint2 a = *reinterpret_cast<const uint2 *>(o + r * AD + lane * 4);
        const uint2 g = *reinterpret_cast<const uint2 *>(dout + r * AD + lane * 4);
        const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a);
        const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&g);
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float2 x = __bfloat1622float2(a2[i]), y = __bfloat1622float2(g2[i]);
            acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (lane == 0) D[r] = acc;
    }
}

struct AttnBwdParams {
    const __nv_bfloat16 *q, *k, *v, *dout;
    const float *lse, *D;
    __nv_bfloat16 *dq, *dk, *dv;
    int32_t H;
    float scale;
};

// dQ kernel roles: 16 warps form dS (lg = warp & 3: 32 query rows; cq = warp >> 2: 32 key
// columns), one thread issues S and dP, another dQ (an issuing thread blocks while the
// tensor pipe is full), one loads Q, dO and the K ring, one the V ring (the two rings free
// their slots at different products, so neither waits for the other).
constexpr int kDqWorkWarps = 16, kDqMmaWarp = 16, kDqLoadWarp = 17, kDqVLoadWarp = 18, kDqQWarp = 19;
constexpr int kDqThreads = 20 * 32;
constexpr int kDqWork = kDqWorkWarps * 32;
constexpr int kDqKSlots = 3;

namespace bq_sm {
constexpr uint32_t Q = 0, dO = 32768, K0 = 65536;      // K ring: 3 slots of 32 KB (K_j is read by S_j and dQ_j)
constexpr uint32_t V0 = K0 + kDqKSlots * 32768;         // V ring: 2 slots (V_j is read by dP_j only)
constexpr uint32_t bytes = V0 + 2 * 32768 + 1024;       // + alignment slack
}  // namespace bq_sm

// Barriers of the dQ kernel (index into bars[]): Q and dO landed; K slot full / free; V slot
// full / free; per S buffer: S_j and dP_j done; dP_j read by every dS thread; per S buffer:
// dS_j written; per S buffer: dQ_j done (also every earlier dQ product: one thread issues
// them all).
// As in the forward, a barrier that many threads arrive on is either per buffer or gates
// the product that the next phase's arrivals depend on, so phases never mix.
enum DqBar { qQ = 0, qKF = 1, qKE = 4, qVF = 7, qVE = 9, qSP = 11, qPE = 13, qDS = 14, qQD = 16, qN = 18 };

__device__ __forceinline__ void store_tile_bf16(__nv_bfloat16 *dst_row, const float (&r)[32], float mul) {
    uint4 *dst = reinterpret_cast<uint4 *>(dst_row);
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        uint4 w;
        w.x = tc::pack_bf16(r[i] * mul, r[i + 1] * mul);
        w.y = tc::pack_bf16(r[i + 2] * mul, r[i + 3] * mul);
        w.z = tc::pack_bf16(r[i + 4] * mul, r[i + 5] * mul);
        w.w = tc::pack_bf16(r[i + 6] * mul, r[i + 7] * mul);
        dst[i / 8] = w;
    }
}

__global__ void __launch_bounds__(kDqThreads, 1) attn_bwd_dq_tc(AttnBwdParams p, PlanDev pd,
                                                                const __grid_constant__ AttnMaps maps) {
    // S_j (one of two TMEM buffers) and dP_j (one buffer) feed the dS warps; dS_j (bf16
    // pairs) overwrites S_j and dQ += dS_j K_j reads it there.  The products thread runs a
    // tile ahead of the dQ thread: S_{j+1} once dQ_{j-1} has released its buffer, dP_{j+1}
    // once every dS thread has read dP_j, so the tensor pipe works through dQ_{j-1}, S_{j+1}
    // and dP_{j+1} while the dS warps work on tile j.
    using namespace bq_sm;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    __shared__ uint64_t bars[qN];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lg = warp & 3, cq = (warp >> 2) & 3;
    const int H = p.H;
    const int32_t h = blockIdx.x % H, qi = blockIdx.x / H;
    const int32_t sq = pd.attn_qt[2 * qi], qt = pd.attn_qt[2 * qi + 1];
    const int32_t hh = pd.attn_hp[sq];
    const int32_t row0 = pd.seq_row0[sq], own = pd.seq_nown[sq];
    const int32_t q0 = qt * AT, nq = min(AT, own - q0);
    const int32_t n_kt = (hh + q0 + nq - 1) / AT + 1;

    if (tid == 0) {
        tc::mbar_init(&bars[qQ], 1);
        for (int i = 0; i < kDqKSlots; ++i) {
            tc::mbar_init(&bars[qKF + i], 1);
            tc::mbar_init(&bars[qKE + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&bars[qVF + i], 1);
            tc::mbar_init(&bars[qVE + i], 1);
            tc::mbar_init(&bars[qSP + i], 1);
            tc::mbar_init(&bars[qDS + i], kDqWork);
            tc::mbar_init(&bars[qQD + i], 1);
        }
        tc::mbar_init(&bars[qPE], kDqWork);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == kDqMmaWarp) {
        tc::tmem_alloc(&s_tmem, 512);
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem, tP = tm + 256, tQ = tm + 384;   // S buffers at tm and tm + 128

    if (warp == kDqLoadWarp || warp == kDqVLoadWarp) {
        // ---- loaders: Q and dO once and the K_j (one thread), the V_j (another), in view
        // order, tiled TMA
        if (lane == 0) {
            const bool is_v = warp == kDqVLoadWarp;
            const int nslot = is_v ? 2 : kDqKSlots;
            uint64_t *fullb = &bars[is_v ? qVF : qKF], *freeb = &bars[is_v ? qVE : qKE];
            uint8_t *ring = sm + (is_v ? V0 : K0);
            int ri = pd.attn_rptr[sq];
            if (!is_v) {
                tc::mbar_expect_tx(&bars[qQ], 65536);
                tc::tma_load_3d(sm + Q, &maps.q, 0, h, row0 + q0, &bars[qQ]);
                tc::tma_load_3d(sm + Q + 16384, &maps.q, 64, h, row0 + q0, &bars[qQ]);
                tc::tma_load_3d(sm + dO, &maps.dout, 0, h, row0 + q0, &bars[qQ]);
                tc::tma_load_3d(sm + dO + 16384, &maps.dout, 64, h, row0 + q0, &bars[qQ]);
            }
            int32_t n = 0;
            for (int32_t j = 0; j < n_kt && !failed(&s_fail); ++j) {
                const int sl = j % nslot, use = j / nslot;
                if (use > 0) wait_or_fail(freeb + sl, (use - 1) & 1, 2, &s_fail);
                if (failed(&s_fail)) break;
                tc::mbar_expect_tx(fullb + sl, 32768);
                tma_view_tile(is_v ? maps.v : maps.k, ring + sl * 32768, pd, sq, j, h, ri, fullb + sl);
                n = j + 1;
            }
            // every copy lands before the block exits: only a slot's last load can be in flight
            for (int i = 0; i < nslot; ++i) {
                const int32_t uses = n > i ? (n - 1 - i) / nslot + 1 : 0;
                if (uses) tc::mbar_wait(fullb + i, (uses - 1) & 1, 1000000000LL);
            }
            if (!is_v) tc::mbar_wait(&bars[qQ], 0, 1000000000LL);
        }
    } else if (warp == kDqMmaWarp) {
        // ---- products issuer: S_j once dQ_{j-2} has released its buffer, dP_j once every dS
        // thread has read dP_{j-1}
        if (lane == 0) {
            const tc::Opnd aQ{tc::smem_addr(sm + Q), 16384, false}, adO{tc::smem_addr(sm + dO), 16384, false};
            uint32_t nc_sp0 = 0, nc_sp1 = 0;
            wait_or_fail(&bars[qQ], 0, 0, &s_fail);
            for (int32_t j = 0; j < n_kt && !failed(&s_fail); ++j) {
                const int b = j & 1, ks = j % kDqKSlots;
                wait_or_fail(&bars[qKF + ks], (j / kDqKSlots) & 1, 0, &s_fail);
                if (j >= 2) wait_or_fail(&bars[qQD + b], ((j - 2) >> 1) & 1, 1, &s_fail);   // dQ_{j-2} read dS there
                tc::fence_after_sync();
                if (failed(&s_fail)) break;
                tc::mma_op(tm + b * 128, aQ, tc::Opnd{tc::smem_addr(sm + K0 + ks * 32768), 16384, false},
                           AT, AT, AD, false);
                wait_or_fail(&bars[qVF + b], (j >> 1) & 1, 0, &s_fail);
                if (j >= 1) wait_or_fail(&bars[qPE], (j - 1) & 1, 1, &s_fail);  // dP_{j-1} read by every dS thread
                tc::fence_after_sync();
                if (failed(&s_fail)) break;
                tc::mma_op(tP, adO, tc::Opnd{tc::smem_addr(sm + V0 + b * 32768), 16384, false}, AT, AT, AD, false);
                tc::mma_commit(&bars[qSP + b]);
                tc::mma_commit(&bars[qVE + b]);
                if (b) ++nc_sp1; else ++nc_sp0;
            }
            if (failed(&s_fail)) {                      // drain the products still in flight
                if (nc_sp0) tc::mbar_wait(&bars[qSP], (nc_sp0 - 1) & 1, 1000000000LL);
                if (nc_sp1) tc::mbar_wait(&bars[qSP + 1], (nc_sp1 - 1) & 1, 1000000000LL);
            }
        }
    } else if (warp == kDqQWarp) {
        // ---- dQ issuer: dQ += dS_j K_j once dS_j is written; K_j's slot is free after it (S_j
        // completed before dS_j was formed)
        if (lane == 0) {
            const uint32_t id_dq = tc::idesc_bf16(AT, AD, false, true);
            uint32_t nc_qd0 = 0, nc_qd1 = 0;
            for (int32_t j = 0; j < n_kt && !failed(&s_fail); ++j) {
                const int b = j & 1;
                wait_or_fail(&bars[qDS + b], (j >> 1) & 1, 1, &s_fail);
                tc::fence_after_sync();
                if (failed(&s_fail)) break;
                const uint32_t kaddr = tc::smem_addr(sm + K0 + (j % kDqKSlots) * 32768);
                for (int kk = 0; kk < AT / 16; ++kk) {
                    const uint64_t bk = tc::desc_sw128_mn(kaddr + kk * 2048, 16384);
                    const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                                 :: "r"(tQ), "r"(tm + b * 128 + kk * 8), "l"(bk), "r"(id_dq), "r"(acc) : "memory");
                }
                tc::mma_commit(&bars[qQD + b]);
                tc::mma_commit(&bars[qKE + j % kDqKSlots]);
                if (b) ++nc_qd1; else ++nc_qd0;
            }
            if (failed(&s_fail)) {                      // drain the products still in flight
                if (nc_qd0) tc::mbar_wait(&bars[qQD], (nc_qd0 - 1) & 1, 1000000000LL);
                if (nc_qd1) tc::mbar_wait(&bars[qQD + 1], (nc_qd1 - 1) & 1, 1000000000LL);
            }
        }
    } else {
        // ---- dS warps: one query row and 32 key columns per thread
        const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
        const int qrow = lg * 32 + lane;
        const int32_t vis = hh + q0 + qrow;
        const int64_t grow = static_cast<int64_t>(row0) + q0 + min(qrow, nq - 1);
        const float c = p.scale * kLog2e;
        const float lse2 = p.lse[grow * H + h] * kLog2e, Dq = p.D[grow * H + h];
        uint32_t nbits = view_bits(pd, sq, hh, own, cq * 32);
        for (int32_t j = 0; j < n_kt; ++j) {
            const int b = j & 1;
            const uint32_t tS = tm + b * 128;
            const uint32_t vb = nbits;
            if (j + 1 < n_kt) nbits = view_bits(pd, sq, hh, own, (j + 1) * AT + cq * 32);
            wait_or_fail(&bars[qSP + b], (j >> 1) & 1, 0, &s_fail);
            tc::fence_after_sync();
            float sv[32], pv[32];
            tc::tmem_ld32x2(tS + lane_off + cq * 32, sv, tP + lane_off + cq * 32, pv);
            tc::fence_before_sync();
            mbar_arrive(&bars[qPE]);
            const int32_t lim = vis - (j * AT + cq * 32);
            uint32_t ud[16];
            if (__all_sync(0xffffffffu, vb == 0xffffffffu && lim >= 31)) {   // no masked column
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float ds[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        ds[u] = ex2(fmaf(sv[i + u], c, -lse2)) * (pv[i + u] - Dq);
                    ud[i / 2] = tc::pack_bf16(ds[0], ds[1]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float ds[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int ii = i + u;
                        const float pr = (((vb >> ii) & 1u) && ii <= lim) ? ex2(fmaf(sv[ii], c, -lse2)) : 0.f;
                        ds[u] = pr * (pv[ii] - Dq);
                    }
                    ud[i / 2] = tc::pack_bf16(ds[0], ds[1]);
                }
            }
            // the row's four warps have read S_j before dS_j overwrites it
            tc::fence_before_sync();
            asm volatile("bar.sync %0, 128;" :: "r"(1 + lg) : "memory");
            tc::fence_after_sync();
            tmem_st16(tS + lane_off + cq * 16, ud);
            tc::fence_before_sync();
            mbar_arrive(&bars[qDS + b]);
        }
        wait_or_fail(&bars[qQD + ((n_kt - 1) & 1)], ((n_kt - 1) >> 1) & 1, 1, &s_fail);   // every dQ product done
        tc::fence_after_sync();
    }
    __syncthreads();
    if (tid == 0 && s_fail) dev_error(pd, kDevErrTimeout, sq, h);
    if (warp < kDqWorkWarps && !s_fail) {
        const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
        const int qrow = lg * 32 + lane;
        float r[32];
        tc::tmem_ld32(tQ + lane_off + cq * 32, r);
        if (qrow < nq) store_tile_bf16(p.dq + ((static_cast<int64_t>(row0) + q0 + qrow) * H + h) * AD + cq * 32, r, p.scale);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kDqMmaWarp) tc::tmem_dealloc(tm, 512);
}

// dK / dV kernel roles: two groups of 8 warps form P^T and dS^T, group g the g-th 64-query
// half of every query tile (lg = warp & 3: 32 key rows; ch = (warp >> 2) & 1: 32 query
// columns of the half), so that two consecutive steps are formed at once; one thread
// issues the products S^T and dP^T, another the updates of dV and dK (an issuing thread
// blocks while the tensor pipe is full, so one thread for both left the pipe idle between
// them); one warp loads K, V once and then Q, dO (tiled TMA) and lse, D (plain loads into
// shared memory) per query tile.
constexpr int kKvWorkWarps = 16, kKvMmaWarp = 16, kKvLoadWarp = 17, kKvUpdWarp = 18, kKvThreads = 19 * 32;
constexpr int kKvGroup = 8 * 32;                  // threads of one work group
constexpr int kHalf = AT / 2;                     // queries per step

namespace bk_sm {
constexpr uint32_t K = 0, V = 32768, Q0 = 65536, Q1 = 98304, dO0 = 131072, dO1 = 163840;
constexpr uint32_t Vec = 196608;                  // [2 slots][128] lse * log2 e, then [2 slots][128] D
constexpr uint32_t Ent = Vec + 2048;              // [2 slots] the query tile's nq, qoff, f
constexpr uint32_t bytes = Ent + 32 + 1024;       // + alignment slack
}  // namespace bk_sm

// Barriers of the dK / dV kernel: K and V landed; per Q slot: Q, dO, lse and D of a query
// tile landed (lane 0's expect_tx, the 32 loader lanes' writes, the copy bytes), the slot
// free again; per step buffer
// (= per work group): S^T and dP^T done, P^T and dS^T written (the group's 256 threads),
// dV and dK updated (also every earlier product).
enum KvBar { vKV = 0, vQF = 1, vQE = 3, vSP = 5, vDS = 7, vDVK = 9, vN = 11 };

__global__ void __launch_bounds__(kKvThreads, 1) attn_bwd_dkdv_tc(AttnBwdParams p, PlanDev pd,
                                                                  const __grid_constant__ AttnMaps maps) {
    // One block per (key tile of a sequence's own rows, head) over the query tiles that see
    // it, each taken as two 64-query steps (the second is empty for a tile of at most 64
    // rows: no products, the barriers still advance).  Step i = 2 e + g: S^T = K Q_i^T and
    // dP^T = V dO_i^T into TMEM buffer g (64 columns each), P^T and dS^T (bf16 pairs)
    // written over them by work group g, dV += P^T dO_i and dK += dS^T Q_i read them there.
    // The issuing thread runs a step ahead: S^T, dP^T of step i + 1 once dV, dK of step
    // i - 1 have released that buffer, so the tensor pipe works through step i - 1's
    // updates and step i + 1's products while the groups form steps i and i + 1.
    using namespace bk_sm;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    __shared__ uint64_t bars[vN];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    float *slse = reinterpret_cast<float *>(sm + Vec), *sD = slse + 2 * AT;
    int32_t *sent = reinterpret_cast<int32_t *>(sm + Ent);   // per slot: nq, qoff, f (decoded by the loader)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lg = warp & 3, cq = (warp >> 2) & 3;
    const int H = p.H;
    const int32_t h = blockIdx.x % H, ki = blockIdx.x / H;
    const int32_t sk = pd.attn_kt[2 * ki], kti = pd.attn_kt[2 * ki + 1];
    const int32_t e0 = pd.attn_kptr[ki], n_e = pd.attn_kptr[ki + 1] - e0;
    const int32_t k0 = kti * AT, nk = min(AT, pd.seq_nown[sk] - k0);
    const int64_t krow0 = static_cast<int64_t>(pd.seq_row0[sk]) + k0;
    // query tile of entry e: rows, count, causal offset or visible-key limit
    auto entry = [&](int32_t e, int64_t &qrow0, int &nq, int32_t &qoff, int32_t &f) {
        const int32_t s_ = pd.attn_kq[3 * (e0 + e)], t_ = pd.attn_kq[3 * (e0 + e) + 1];
        f = pd.attn_kq[3 * (e0 + e) + 2];
        qrow0 = static_cast<int64_t>(pd.seq_row0[s_]) + t_ * AT;
        nq = min(AT, pd.seq_nown[s_] - t_ * AT);
        qoff = t_ * AT - k0;                          // query local position minus key tile start
    };

    if (tid == 0) {
        tc::mbar_init(&bars[vKV], 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&bars[vQF + i], 33);       // lane 0's expect_tx + 32 lanes' writes
            tc::mbar_init(&bars[vQE + i], 1);
            tc::mbar_init(&bars[vSP + i], 1);
            tc::mbar_init(&bars[vDS + i], kKvGroup);
            tc::mbar_init(&bars[vDVK + i], 1);
        }
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == kKvMmaWarp) {
        tc::tmem_alloc(&s_tmem, 512);
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem, tdP = tm + 128, tV = tm + 256, tK = tm + 384;   // S^T buffers at tm, tm + 64

    if (warp == kKvLoadWarp) {
        // ---- loader warp: K and V once; per query tile Q and dO by tiled TMA (lane 0), lse
        // and D by plain loads (4 rows per lane) and the tile's decoded entry; all 32 lanes
        // arrive on the slot's barrier, so the consumers never wait on the plan tables
        if (lane == 0) {
            tc::mbar_expect_tx(&bars[vKV], 65536);
            tc::tma_load_3d(sm + K, &maps.k[4], 0, h, static_cast<int>(krow0), &bars[vKV]);
            tc::tma_load_3d(sm + K + 16384, &maps.k[4], 64, h, static_cast<int>(krow0), &bars[vKV]);
            tc::tma_load_3d(sm + V, &maps.v[4], 0, h, static_cast<int>(krow0), &bars[vKV]);
            tc::tma_load_3d(sm + V + 16384, &maps.v[4], 64, h, static_cast<int>(krow0), &bars[vKV]);
        }
        int32_t issued = 0;
        for (int32_t e = 0; e < n_e; ++e) {
            const int slot = e & 1, use = e >> 1;
            if (use > 0) wait_or_fail(&bars[vQE + slot], (use - 1) & 1, 2, &s_fail);
            if (failed(&s_fail)) break;
            int64_t qr; int nq; int32_t qoff, f;
            entry(e, qr, nq, qoff, f);
            if (lane == 0) {                            // the copies first: they take longest
                uint64_t *bar = &bars[vQF + slot];
                tc::mbar_expect_tx(bar, 65536);         // lane 0's first arrival
                uint8_t *dq_ = sm + (slot ? Q1 : Q0), *dd = sm + (slot ? dO1 : dO0);
                tc::tma_load_3d(dq_, &maps.q, 0, h, static_cast<int>(qr), bar);
                tc::tma_load_3d(dq_ + 16384, &maps.q, 64, h, static_cast<int>(qr), bar);
                tc::tma_load_3d(dd, &maps.dout, 0, h, static_cast<int>(qr), bar);
                tc::tma_load_3d(dd + 16384, &maps.dout, 64, h, static_cast<int>(qr), bar);
                sent[4 * slot] = nq;
                sent[4 * slot + 1] = qoff;
                sent[4 * slot + 2] = f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = lane + 32 * u;
                const bool ok = r < nq;
                slse[slot * AT + r] = ok ? p.lse[(qr + r) * H + h] * kLog2e : 0.f;
                sD[slot * AT + r] = ok ? p.D[(qr + r) * H + h] : 0.f;
            }
            mbar_arrive(&bars[vQF + slot]);             // every lane, after its writes
            issued = e + 1;
        }
        if (lane == 0) {                                // every copy lands before the block exits
            for (int i = 0; i < 2; ++i) {
                const int32_t uses = issued > i ? (issued - 1 - i) / 2 + 1 : 0;
                if (uses) tc::mbar_wait(&bars[vQF + i], (uses - 1) & 1, 1000000000LL);
            }
            tc::mbar_wait(&bars[vKV], 0, 1000000000LL);
        }
    } else if (warp == kKvMmaWarp) {
        // ---- products issuer: S^T and dP^T of step i + 1 once dV, dK of step i - 1 have
        // released that buffer
        if (lane == 0 && n_e > 0) {
            const tc::Opnd aK{tc::smem_addr(sm + K), 16384, false}, aV{tc::smem_addr(sm + V), 16384, false};
            auto products = [&](int32_t e, int hf) {   // S^T and dP^T of (e, hf) into buffer hf
                const uint32_t qa = tc::smem_addr(sm + ((e & 1) ? Q1 : Q0)) + hf * 8192;
                const uint32_t da = tc::smem_addr(sm + ((e & 1) ? dO1 : dO0)) + hf * 8192;
                tc::mma_op(tm + hf * 64, aK, tc::Opnd{qa, 16384, false}, AT, kHalf, AD, false);
                tc::mma_op(tdP + hf * 64, aV, tc::Opnd{da, 16384, false}, AT, kHalf, AD, false);
            };
            uint32_t nc_sp0 = 0, nc_sp1 = 0;
            const int32_t n_st = 2 * n_e;
            int nq_nx = 0;
            for (int32_t i = 0; i < n_st && !failed(&s_fail); ++i) {
                const int32_t e = i >> 1;
                const int b = i & 1;
                if (b == 0) {                           // a new query tile: its slot has landed
                    if (i == 0) wait_or_fail(&bars[vKV], 0, 0, &s_fail);
                    wait_or_fail(&bars[vQF + (e & 1)], (e >> 1) & 1, 0, &s_fail);
                    nq_nx = sent[4 * (e & 1)];
                }
                if (i >= 2) wait_or_fail(&bars[vDVK + b], ((i - 2) >> 1) & 1, 1, &s_fail);
                tc::fence_after_sync();
                if (failed(&s_fail)) break;
                if (b == 0 || nq_nx > kHalf) products(e, b);   // step 0 is never empty
                tc::mma_commit(&bars[vSP + b]);
                if (b) ++nc_sp1; else ++nc_sp0;
            }
            if (failed(&s_fail)) {                      // drain the products still in flight
                if (nc_sp0) tc::mbar_wait(&bars[vSP], (nc_sp0 - 1) & 1, 1000000000LL);
                if (nc_sp1) tc::mbar_wait(&bars[vSP + 1], (nc_sp1 - 1) & 1, 1000000000LL);
            }
        }
    } else if (warp == kKvUpdWarp) {
        // ---- update issuer: dV += P^T dO_i, dK += dS^T Q_i once group i mod 2 has written
        // P^T and dS^T; the query tile's slot is free after its second step's update (its
        // products completed before that step's P^T and dS^T were formed)
        if (lane == 0 && n_e > 0) {
            const uint32_t id_up = tc::idesc_bf16(AT, AD, false, true);
            uint32_t nc_u0 = 0, nc_u1 = 0;
            const int32_t n_st = 2 * n_e;
            for (int32_t i = 0; i < n_st && !failed(&s_fail); ++i) {
                const int b = i & 1;
                const int32_t e = i >> 1;
                wait_or_fail(&bars[vDS + b], (i >> 1) & 1, 1, &s_fail);
                tc::fence_after_sync();
                if (failed(&s_fail)) break;
                const int nq = sent[4 * (e & 1)];       // written before the slot's barrier, read after this step's
                if (b == 0 || nq > kHalf) {
                    const uint32_t qa = tc::smem_addr(sm + ((e & 1) ? Q1 : Q0)) + b * 8192;
                    const uint32_t da = tc::smem_addr(sm + ((e & 1) ? dO1 : dO0)) + b * 8192;
                    for (int kk = 0; kk < kHalf / 16; ++kk) {
                        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                        const uint64_t bdo = tc::desc_sw128_mn(da + kk * 2048, 16384);
                        const uint64_t bq = tc::desc_sw128_mn(qa + kk * 2048, 16384);
                        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                                     "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                                     :: "r"(tV), "r"(tm + b * 64 + kk * 8), "l"(bdo), "r"(id_up), "r"(acc) : "memory");
                        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                                     "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                                     :: "r"(tK), "r"(tdP + b * 64 + kk * 8), "l"(bq), "r"(id_up), "r"(acc) : "memory");
                    }
                }
                tc::mma_commit(&bars[vDVK + b]);
                if (b) ++nc_u1; else ++nc_u0;
                if (b == 1) tc::mma_commit(&bars[vQE + (e & 1)]);   // the query tile's last step
            }
            if (failed(&s_fail)) {                      // drain the updates still in flight
                if (nc_u0) tc::mbar_wait(&bars[vDVK], (nc_u0 - 1) & 1, 1000000000LL);
                if (nc_u1) tc::mbar_wait(&bars[vDVK + 1], (nc_u1 - 1) & 1, 1000000000LL);
            }
        }
    } else {
        // ---- work group g = warp >> 3: one key row and 32 query columns of step 2 e + g per
        // thread, in two passes of 16
        const int g = warp >> 3, ch = (warp >> 2) & 1;
        const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
        const int krow = lg * 32 + lane;
        const float c = p.scale * kLog2e;
        const uint32_t tSb = tm + g * 64, tPb = tdP + g * 64;
        for (int32_t e = 0; e < n_e; ++e) {
            const int slot = e & 1;
            wait_or_fail(&bars[vQF + slot], (e >> 1) & 1, 0, &s_fail);
            const int nq = sent[4 * slot], qoff = sent[4 * slot + 1], f = sent[4 * slot + 2];
            wait_or_fail(&bars[vSP + g], e & 1, 0, &s_fail);
            if (g == 1 && nq <= kHalf) {                // empty second half: nothing to form
                mbar_arrive(&bars[vDS + g]);
                continue;
            }
            tc::fence_after_sync();
            uint32_t up[16], ud[16];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const int col = ch * 32 + part * 16;    // query column within the half
                float sv[16], pv[16];
                tmem_ld16x2(tSb + lane_off + col, sv, tPb + lane_off + col, pv);
                const float *lq = slse + slot * AT + g * kHalf + col;
                const float *dq_ = sD + slot * AT + g * kHalf + col;
                // every column of the warp visible (the visibility is monotone in the query
                // column): no per-element mask
                const int qc0 = g * kHalf + col;
                const bool all_vis = qc0 + 15 < nq && (f < 0 ? krow <= qoff + qc0 : k0 + krow < f);
                if (__all_sync(0xffffffffu, all_vis)) {
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        float pr[2], ds[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            pr[u] = ex2(fmaf(sv[j + u], c, -lq[j + u]));
                            ds[u] = pr[u] * (pv[j + u] - dq_[j + u]);
                        }
                        up[part * 8 + j / 2] = tc::pack_bf16(pr[0], pr[1]);
                        ud[part * 8 + j / 2] = tc::pack_bf16(ds[0], ds[1]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        float pr[2], ds[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int qc = qc0 + j + u;
                            const bool vis = qc < nq && (f < 0 ? krow <= qoff + qc : k0 + krow < f);
                            pr[u] = vis ? ex2(fmaf(sv[j + u], c, -lq[j + u])) : 0.f;
                            ds[u] = pr[u] * (pv[j + u] - dq_[j + u]);
                        }
                        up[part * 8 + j / 2] = tc::pack_bf16(pr[0], pr[1]);
                        ud[part * 8 + j / 2] = tc::pack_bf16(ds[0], ds[1]);
                    }
                }
            }
            // the row's two warps of the group have read S^T and dP^T before P^T and dS^T
            // overwrite them
            tc::fence_before_sync();
            asm volatile("bar.sync %0, 64;" :: "r"(1 + g * 4 + lg) : "memory");
            tc::fence_after_sync();
            tmem_st16x2(tSb + lane_off + ch * 16, up, tPb + lane_off + ch * 16, ud);
            tc::fence_before_sync();
            mbar_arrive(&bars[vDS + g]);
        }
        // the group of the last step waits for it: its update is the last product issued
        if (n_e > 0 && g == 1) wait_or_fail(&bars[vDVK + 1], (n_e - 1) & 1, 2, &s_fail);
        tc::fence_after_sync();
    }
    __syncthreads();
    if (tid == 0 && s_fail) dev_error(pd, kDevErrTimeout, sk, h);
    if (warp < kKvWorkWarps && !s_fail) {             // warp-collective loads, guarded stores
        const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
        const int krow = lg * 32 + lane;
        const int cc = cq * 32;                         // 32 channels per thread
        float r[32];
        tc::tmem_ld32(tV + lane_off + cc, r);
        if (n_e == 0) for (int j = 0; j < 32; ++j) r[j] = 0.f;
        if (krow < nk) store_tile_bf16(p.dv + ((krow0 + krow) * H + h) * AD + cc, r, 1.f);
        tc::tmem_ld32(tK + lane_off + cc, r);
        if (n_e == 0) for (int j = 0; j < 32; ++j) r[j] = 0.f;
        if (krow < nk) store_tile_bf16(p.dk + ((krow0 + krow) * H + h) * AD + cc, r, p.scale);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kKvMmaWarp) tc::tmem_dealloc(tm, 512);
}

}  // namespace
}  // namespace harts

using namespace harts;

static int check_attn(const harts_plan *P, const harts_attn_fwd_args *a) {
    if (!P || !a) { set_error("NULL plan or args"); return HARTS_EINVAL; }
    if (!P->attn_ok) { set_error("plan too deep for the branch-attention tables"); return HARTS_EOVERFLOW; }
    if (a->dtype != HARTS_BF16 || a->d != AD) { set_error("branch attention: bf16 and d = 128 only"); return HARTS_EUNSUPPORTED; }
    if (a->H < 1) { set_error("H must be >= 1"); return HARTS_EINVAL; }
    if (!(a->scale > 0.f) || !(a->scale < 3.0e38f)) { set_error("scale must be positive and finite"); return HARTS_EINVAL; }
    if (!a->q || !a->k || !a->v || !a->o) { set_error("NULL q, k, v or o"); return HARTS_EINVAL; }
    if ((reinterpret_cast<uintptr_t>(a->q) | reinterpret_cast<uintptr_t>(a->k) | reinterpret_cast<uintptr_t>(a->v) |
         reinterpret_cast<uintptr_t>(a->o)) & 15) {
        set_error("q, k, v and o must be 16-byte aligned"); return HARTS_EINVAL;
    }
    if (!P->dev) { set_error("plan not uploaded (harts_plan_upload)"); return HARTS_ENOPLAN; }
    if (int64_t(P->image.n_qt) * a->H > 0x7fffffff || int64_t(P->image.n_kt) * a->H > 0x7fffffff) {
        set_error("too many (tile, head) blocks"); return HARTS_EOVERFLOW;
    }
    return HARTS_OK;
}

template <typename K, typename... Args>
static cudaError_t launch_big(K kernel, unsigned blocks, int threads, uint32_t smem, cudaStream_t st,
                              const Args &...args) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kernel<<<blocks, threads, smem, st>>>(args...);
    return cudaGetLastError();
}

// [C][H][128] bf16 as a 3-D tensor {channels, heads, rows}; one box height.
static bool rows_map(CUtensorMap *m, const void *base, int H, int64_t C, int box_rows) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(AD), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(C)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(AD) * 2, static_cast<cuuint64_t>(H) * AD * 2};
    const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
    return encode_bf16(m, base, 3, dims, strides, box);
}

static bool attn_maps(AttnMaps &m, const void *q, const void *dout, const void *k, const void *v, int H, int64_t C) {
    if (!rows_map(&m.q, q, H, C, AT)) return false;
    if (dout && !rows_map(&m.dout, dout, H, C, AT)) return false;
    if (!dout) m.dout = m.q;
    for (int j = 0; j < 5; ++j)
        if (!rows_map(&m.k[j], k, H, C, 8 << j) || !rows_map(&m.v[j], v, H, C, 8 << j)) return false;
    return true;
}

extern "C" {

int harts_attn_fwd(const harts_plan *P, const harts_attn_fwd_args *a, harts_stream_t stream) {
    if (int rc = check_attn(P, a)) return rc;
    const int64_t blocks = int64_t(P->image.n_qt) * a->H;
    if (blocks == 0) { set_error(""); return HARTS_OK; }
    AttnParams p;
    p.q = static_cast<const __nv_bfloat16 *>(a->q);
    p.k = static_cast<const __nv_bfloat16 *>(a->k);
    p.v = static_cast<const __nv_bfloat16 *>(a->v);
    p.o = static_cast<__nv_bfloat16 *>(a->o);
    p.lse = a->lse;
    p.H = a->H;
    p.scale = a->scale;
    AttnMaps maps;
    if (!attn_maps(maps, a->q, nullptr, a->k, a->v, a->H, P->info.C)) {
        set_error("tensor map encoding failed"); return HARTS_ECUDA;
    }
    const cudaError_t e = launch_big(attn_fwd_tc, static_cast<unsigned>(blocks), kFwdThreads, at_sm::bytes,
                                     reinterpret_cast<cudaStream_t>(stream), p, P->view, maps);
    if (e != cudaSuccess) { set_error(std::string("attention launch: ") + cudaGetErrorString(e)); return HARTS_ECUDA; }
    set_error("");
    return HARTS_OK;
}

size_t harts_attn_bwd_workspace_bytes(const harts_plan *P, int32_t H) {
    if (!P || H < 1) return 0;
    return static_cast<size_t>((P->info.C * H * 4 + 255) / 256 * 256);
}

int harts_attn_bwd(const harts_plan *P, const harts_attn_bwd_args *a, harts_stream_t stream) {
    if (!a) { set_error("NULL args"); return HARTS_EINVAL; }
    if (int rc = check_attn(P, &a->fwd)) return rc;
    if (!a->fwd.lse || !a->d_o || !a->dq || !a->dk || !a->dv) { set_error("NULL lse, d_o, dq, dk or dv"); return HARTS_EINVAL; }
    if ((reinterpret_cast<uintptr_t>(a->d_o) | reinterpret_cast<uintptr_t>(a->dq) | reinterpret_cast<uintptr_t>(a->dk) |
         reinterpret_cast<uintptr_t>(a->dv) | reinterpret_cast<uintptr_t>(a->fwd.lse) |
         reinterpret_cast<uintptr_t>(a->workspace)) & 15) {
        set_error("d_o, dq, dk, dv, lse and workspace must be 16-byte aligned"); return HARTS_EINVAL;
    }
    const size_t need = harts_attn_bwd_workspace_bytes(P, a->fwd.H);
    if (!a->workspace || a->workspace_bytes < need) { set_error("workspace smaller than harts_attn_bwd_workspace_bytes"); return HARTS_ESMALLBUF; }
    const int64_t rows = P->info.C * a->fwd.H;
    if (rows == 0) { set_error(""); return HARTS_OK; }
    AttnBwdParams p;
    p.q = static_cast<const __nv_bfloat16 *>(a->fwd.q);
    p.k = static_cast<const __nv_bfloat16 *>(a->fwd.k);
    p.v = static_cast<const __nv_bfloat16 *>(a->fwd.v);
    p.dout = static_cast<const __nv_bfloat16 *>(a->d_o);
    p.lse = a->fwd.lse;
    float *D = static_cast<float *>(a->workspace);
    p.D = D;
    p.dq = static_cast<__nv_bfloat16 *>(a->dq);
    p.dk = static_cast<__nv_bfloat16 *>(a->dk);
    p.dv = static_cast<__nv_bfloat16 *>(a->dv);
    p.H = a->fwd.H;
    p.scale = a->fwd.scale;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t prep_blocks = std::min<int64_t>((rows * 32 + 255) / 256, 152 * 16);
    attn_bwd_prep<<<static_cast<unsigned>(prep_blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(a->fwd.o), p.dout, D, rows);
    cudaError_t e = cudaGetLastError();
    AttnMaps maps;
    if (e == cudaSuccess && !attn_maps(maps, a->fwd.q, a->d_o, a->fwd.k, a->fwd.v, p.H, P->info.C)) {
        set_error("tensor map encoding failed"); return HARTS_ECUDA;
    }
    if (e == cudaSuccess)
        e = launch_big(attn_bwd_dq_tc, static_cast<unsigned>(int64_t(P->image.n_qt) * p.H), kDqThreads, bq_sm::bytes, st, p,
                       P->view, maps);
    if (e == cudaSuccess)
        e = launch_big(attn_bwd_dkdv_tc, static_cast<unsigned>(int64_t(P->image.n_kt) * p.H), kKvThreads, bk_sm::bytes, st, p,
                       P->view, maps);
    if (e != cudaSuccess) { set_error(std::string("attention backward launch: ") + cudaGetErrorString(e)); return HARTS_ECUDA; }
    set_error("");
    return HARTS_OK;
}

}  // extern "C"
