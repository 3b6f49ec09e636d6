// Branch attention over the compact layout, forward, tensor cores (bf16, d = 128).
//
// HARTS (page "HARTS ... 精读", section 4.3, MLA paragraph; summary page, section 4 "MLA
// execution"; figures page, Figure C.1(c)): a branch's queries (its own l tokens) attend
// to the keys and values of its ancestors and itself (h + l) with bottom-right causal
// alignment: own query t sees view entries j <= h + t.  The ancestor view is a temporary
// gather inside the kernel; outputs go back to the unique compact rows.  The core is plain
// softmax attention on projected inputs: o = softmax(scale q k^T) v per head.
//
// One block per (sequence, 128-query tile, head); the planner orders the tiles tree by
// tree (longest first within a tree) with the heads innermost, so the key / value rows a
// tree's blocks share stay in L2.  Per key tile j of 128 view rows:
//   S_j = Q K_j^T           tcgen05, M = N = 128, K = d, fp32 in one of two TMEM buffers;
//                           S_{j+1} is issued as soon as S_j is ready, so the tensor core
//                           works while the warps run the softmax of tile j
//   softmax                 sixteen warps, one query row and 32 columns each; scores in
//                           base-2 units (scale * log2 e folded into one FMA); the four
//                           warps holding a row exchange its max through shared memory; the
//                           running max moves (and O is rescaled in TMEM) only when a row's
//                           max grows by more than 2^8 -- any common offset gives the same
//                           softmax, the threshold only bounds P by 256
//   O += P V_j              tcgen05, P bf16 in shared memory, V read MN-major
// Keys and values are gathered by cp.async through a four-tile ring of row tables, K two
// tiles and V one tile ahead.  Masking runs only on tiles that reach past the first
// query's causal limit.  Every wait is bounded; a timeout records code 3 in the plan's
// error word, stops issuing products and drains the ones in flight.
#include <cstring>

#include "kda_common.cuh"
#include "tc_primitives.cuh"

namespace harts {
namespace {

constexpr int AD = 128, AT = kAttnTile, ANT = 512, NQ = ANT / AT;   // NQ column quarters
constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;               // running max moves when a row max grows by more

namespace at_sm {
constexpr uint32_t Q = 0, K0 = 32768, K1 = 65536, V0 = 98304, V1 = 131072, P = 163840;
constexpr uint32_t Max = 196608;                  // [2 tiles][4 quarters][128] fp32 row maxima
constexpr uint32_t Sum = Max + 4096;              // [4 quarters][128] fp32 row sums
constexpr uint32_t Tab = Sum + 2048;              // [4][128] int32 view rows of tiles j % 4
constexpr uint32_t bytes = Tab + 2048 + 1024;     // + alignment slack
}  // namespace at_sm

struct AttnParams {
    const __nv_bfloat16 *q, *k, *v;
    __nv_bfloat16 *o;
    float *lse;
    int32_t H;
    float scale;
};

// 16-byte piece p of row r of a [128 rows][128 cols] SW128 tile.
__device__ __forceinline__ uint32_t piece(int r, int p) {
    return static_cast<uint32_t>((p >> 3) * 16384 + r * 128 + (((p & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int N>
__device__ __forceinline__ void cp_wait_group() {
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

__device__ __forceinline__ void sync_mma() {
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

// Waits unless the block has already failed; a timeout records 1 + 2 * which + phase.
__device__ __forceinline__ void wait_or_fail(uint64_t *bar, uint32_t phase, int which, int *s_fail) {
    if (*reinterpret_cast<volatile int *>(s_fail)) return;
    if (!tc::mbar_wait(bar, phase)) atomicCAS(s_fail, 0, 1 + 2 * which + static_cast<int>(phase));
}

__global__ void __launch_bounds__(ANT, 1) attn_fwd_tc(AttnParams p, PlanDev pd) {
    using namespace at_sm;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    __shared__ uint64_t bars[3];                  // S buffer 0, S buffer 1, O
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    float *smax = reinterpret_cast<float *>(sm + Max), *ssum = reinterpret_cast<float *>(sm + Sum);
    int32_t *stab = reinterpret_cast<int32_t *>(sm + Tab);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lg = warp & 3, cq = warp >> 2;
    const int H = p.H;
    const int32_t h = blockIdx.x % H, qi = blockIdx.x / H;
    const int32_t sq = pd.attn_qt[2 * qi], qt = pd.attn_qt[2 * qi + 1];
    const int32_t hb = pd.attn_hptr[sq], hh = pd.attn_hptr[sq + 1] - hb;
    const int32_t row0 = pd.seq_row0[sq], own = pd.seq_nown[sq], nview = hh + own;
    const int32_t q0 = qt * AT, nq = min(AT, own - q0);
    const int32_t n_kt = (hh + q0 + nq - 1) / AT + 1;   // key tiles covering every visible entry
    const int32_t first_masked = (hh + q0) / AT;        // tiles from here reach past a causal limit
    const float c = p.scale * kLog2e;

    // compact row of view entry j (-1 past the view)
    auto view_row = [&](int32_t j) -> int32_t {
        return j < hh ? pd.attn_hrows[hb + j] : (j < nview ? row0 + (j - hh) : -1);
    };
    // 128 rows of K or V for tile `kt` from ring slot kt % 4 into `dst`
    auto stage = [&](const __nv_bfloat16 *src, int32_t kt, uint8_t *dst) {
        const int32_t *tab = stab + (kt & 3) * AT;
#pragma unroll
        for (int i = 0; i < AT * 16 / ANT; ++i) {
            const int e = tid + i * ANT, r = e >> 4, pc = e & 15;
            const int32_t row = tab[r];
            const __nv_bfloat16 *g = src + (static_cast<int64_t>(row < 0 ? 0 : row) * H + h) * AD + pc * 8;
            tc::cp_async16(dst + piece(r, pc), g, row >= 0 ? 16u : 0u);
        }
    };

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) tc::mbar_init(&bars[i], 1);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(&s_tmem, 512);
        tc::fence_before_sync();
    }
    if (tid < AT) {
#pragma unroll
        for (int j = 0; j < 3; ++j) stab[j * AT + tid] = j * AT + tid < (n_kt * AT) ? view_row(j * AT + tid) : -1;
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem, lane_off = static_cast<uint32_t>(lg * 32) << 16;
    const uint32_t tO = tm + 256;
    const int qrow = lg * 32 + lane;                    // this thread's query row (TMEM lane)
    const int32_t vis = hh + q0 + qrow;                 // last view entry it sees

    // group 0: Q, K_0, V_0; group 1: K_1; group 2: empty (stands for "V_0" in the steady state)
#pragma unroll
    for (int i = 0; i < AT * 16 / ANT; ++i) {
        const int e = tid + i * ANT, r = e >> 4, pc = e & 15;
        const bool ok = r < nq;
        const __nv_bfloat16 *g = p.q + ((static_cast<int64_t>(row0) + q0 + (ok ? r : 0)) * H + h) * AD + pc * 8;
        tc::cp_async16(sm + Q + piece(r, pc), g, ok ? 16u : 0u);
    }
    stage(p.k, 0, sm + K0);
    stage(p.v, 0, sm + V0);
    tc::cp_async_commit();
    if (n_kt > 1) stage(p.k, 1, sm + K1);
    tc::cp_async_commit();
    tc::cp_async_commit();
    cp_wait_group<2>();
    sync_mma();
    uint32_t nc_s0 = 0, nc_s1 = 0, nc_o = 0;            // thread 0: commits per barrier
    if (tid == 0) {
        tc::mma_op(tm, tc::Opnd{tc::smem_addr(sm + Q), 16384, false}, tc::Opnd{tc::smem_addr(sm + K0), 16384, false},
                   AT, AT, AD, false);
        tc::mma_commit(&bars[0]);
        nc_s0 = 1;
    }

    float m_run = -INFINITY, l_part = 0.f;
    for (int32_t kt = 0; kt < n_kt; ++kt) {
        const int b = kt & 1;
        // A: S_kt ready; K_{kt+1} in shared memory
        cp_wait_group<1>();
        tc::fence_smem_to_async();
        wait_or_fail(&bars[b], (kt >> 1) & 1, b, &s_fail);
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        const bool failed = *reinterpret_cast<volatile int *>(&s_fail) != 0;
        // B: S_{kt+1} into the other buffer
        if (tid == 0 && kt + 1 < n_kt && !failed) {
            tc::mma_op(tm + (b ^ 1) * 128, tc::Opnd{tc::smem_addr(sm + Q), 16384, false},
                       tc::Opnd{tc::smem_addr(sm + (b ? K0 : K1)), 16384, false}, AT, AT, AD, false);
            tc::mma_commit(&bars[b ^ 1]);
            if (b) ++nc_s0; else ++nc_s1;
        }
        // C: K_{kt+2} into this tile's K buffer (S_kt has consumed it); row table of tile kt+3
        if (kt + 2 < n_kt) stage(p.k, kt + 2, sm + (b ? K1 : K0));
        tc::cp_async_commit();
        int32_t nxt = -1;
        if (tid < AT && (kt + 3) * AT + tid < n_kt * AT) nxt = view_row((kt + 3) * AT + tid);
        // D: scores, mask, row max of this half
        float s[32];
        tc::tmem_ld32(tm + b * 128 + lane_off + cq * 32, s);
        if (kt >= first_masked) {
            const int32_t lim = vis - (kt * AT + cq * 32);
#pragma unroll
            for (int i = 0; i < 32; ++i) s[i] = i <= lim ? s[i] : -INFINITY;
        }
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = fmaxf(fmaxf(s[i], s[i + 8]), fmaxf(s[i + 16], s[i + 24]));
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) mp[i] = fmaxf(mp[i], mp[i + w]);
        smax[(b * NQ + cq) * AT + qrow] = mp[0];
        // the four warps holding these rows exchange their maxima (named barrier 1 + lg)
        asm volatile("bar.sync %0, %1;" :: "r"(1 + lg), "n"(NQ * 32) : "memory");
        // F: running max (moves only past the threshold), probabilities, row sum of this quarter
        const float *mrow = smax + b * NQ * AT + qrow;
        const float m_tile = c * fmaxf(fmaxf(mrow[0], mrow[AT]), fmaxf(mrow[2 * AT], mrow[3 * AT]));
        const bool move = __any_sync(0xffffffffu, m_tile > m_run + kRescaleLog2);
        float alpha = 1.f;
        if (move) {
            const float m_new = fmaxf(m_run, m_tile);
            alpha = ex2(m_run - m_new);
            m_run = m_new;
        }
        float sp[8];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            s[i] = ex2(fmaf(s[i], c, -m_run));
            sp[i & 7] = (i < 8) ? s[i] : sp[i & 7] + s[i];
        }
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) sp[i] += sp[i + w];
        l_part = l_part * alpha + sp[0];
        // G: O_{kt-1} done (P buffer and O free); P, rescale of O, V_{kt+1}
        if (kt > 0) wait_or_fail(&bars[2], (kt - 1) & 1, 2, &s_fail);
        tc::fence_after_sync();
#pragma unroll
        for (int i = 0; i < 32; i += 8) tc::st_sw128_8(sm + P, AT, qrow, cq * 32 + i, s + i);
        if (move && kt > 0) {
            float r[32];
            tc::tmem_ld32(tO + lane_off + cq * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] *= alpha;
            tc::tmem_st32(tO + lane_off + cq * 32, r);
        }
        if (kt + 1 < n_kt) stage(p.v, kt + 1, sm + (b ? V0 : V1));
        tc::cp_async_commit();
        cp_wait_group<2>();                             // V_kt has landed
        if (tid < AT) stab[((kt + 3) & 3) * AT + tid] = nxt;
        // H: O += P V_kt
        sync_mma();
        if (tid == 0 && *reinterpret_cast<volatile int *>(&s_fail) == 0) {
            tc::mma_op(tO, tc::Opnd{tc::smem_addr(sm + P), 16384, false},
                       tc::Opnd{tc::smem_addr(sm + (b ? V1 : V0)), 16384, true}, AT, AD, AT, kt > 0);
            tc::mma_commit(&bars[2]);
            ++nc_o;
        }
    }
    wait_or_fail(&bars[2], (n_kt - 1) & 1, 2, &s_fail);
    tc::fence_after_sync();
    ssum[cq * AT + qrow] = l_part;
    __syncthreads();
    // ---- outputs ------------------------------------------------------------------------
    if (!s_fail) {
        const float l = (ssum[qrow] + ssum[AT + qrow]) + (ssum[2 * AT + qrow] + ssum[3 * AT + qrow]), inv = 1.f / l;
        const int64_t row = static_cast<int64_t>(row0) + q0 + qrow;
        float r[32];
        tc::tmem_ld32(tO + lane_off + cq * 32, r);
        if (qrow < nq) {
            uint4 *dst = reinterpret_cast<uint4 *>(p.o + (row * H + h) * AD + cq * 32);
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
        if (p.lse && cq == 0 && qrow < nq) p.lse[row * H + h] = m_run * kLn2 + logf(l);
    }
    tc::cp_async_wait_all();
    if (s_fail && tid == 0) {                           // drain the products still in flight
        dev_error(pd, kDevErrTimeout, sq, h);
        const uint32_t nc[3] = {nc_s0, nc_s1, nc_o};
#pragma unroll
        for (int i = 0; i < 3; ++i)
            if (nc[i]) tc::mbar_wait(&bars[i], (nc[i] - 1) & 1, 1000000000LL);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tm, 512);
}

}  // namespace
}  // namespace harts

using namespace harts;

extern "C" {

int harts_attn_fwd(const harts_plan *P, const harts_attn_fwd_args *a, harts_stream_t stream) {
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
    const int64_t blocks = int64_t(P->image.n_qt) * a->H;
    if (blocks > 0x7fffffff) { set_error("too many (query tile, head) blocks"); return HARTS_EOVERFLOW; }
    if (blocks == 0) { set_error(""); return HARTS_OK; }
    AttnParams p;
    p.q = static_cast<const __nv_bfloat16 *>(a->q);
    p.k = static_cast<const __nv_bfloat16 *>(a->k);
    p.v = static_cast<const __nv_bfloat16 *>(a->v);
    p.o = static_cast<__nv_bfloat16 *>(a->o);
    p.lse = a->lse;
    p.H = a->H;
    p.scale = a->scale;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(at_sm::bytes));
    if (e == cudaSuccess) {
        attn_fwd_tc<<<static_cast<unsigned>(blocks), ANT, at_sm::bytes, st>>>(p, P->view);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) { set_error(std::string("attention launch: ") + cudaGetErrorString(e)); return HARTS_ECUDA; }
    set_error("");
    return HARTS_OK;
}

}  // extern "C"
