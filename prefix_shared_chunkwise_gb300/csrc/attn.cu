// Branch attention over the compact layout, forward, tensor cores (bf16, d = 128).
//
// HARTS (page "HARTS ... 精读", section 4.3, MLA paragraph; summary page, section 4 "MLA
// execution"; figures page, Figure C.1(c)): a branch's queries (its own l tokens) attend
// to the keys and values of its ancestors and itself (h + l) with bottom-right causal
// alignment: own query t sees view entries j <= h + t.  The ancestor view is a temporary
// gather inside the kernel; outputs go back to the unique compact rows.  The core is plain
// softmax attention on projected inputs: o = softmax(scale q k^T) v per head.
//
// One block per (sequence, 128-query tile, head), tiles with the longest views first.
// Per key tile of 128 view rows: S = Q K^T (tcgen05, M = N = 128, K = d, fp32 in TMEM);
// eight warps take one query row and 64 columns each, combine the halves' row max and
// sum through shared memory, keep a running (max, sum), write P (bf16) and rescale the
// TMEM output; O += P V (tcgen05, V read MN-major).  The next key / value tile is
// gathered (cp.async through a row table) while the current one is used.  Every wait is
// bounded; a timeout records code 3 in the plan's error word.
#include <cstring>

#include "kda_common.cuh"
#include "tc_primitives.cuh"

namespace harts {
namespace {

constexpr int AD = 128, AT = kAttnTile, ANT = 256;

namespace at_sm {
constexpr uint32_t Q = 0, K0 = 32768, V0 = 65536, K1 = 98304, V1 = 131072, P = 163840;
constexpr uint32_t Vec = 196608;                  // [2][128] row max, [2][128] row sum
constexpr uint32_t bytes = Vec + 2048 + 1024;     // + alignment slack
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

// Every thread waits; a timeout anywhere sets *s_fail = 1 + 2 * (bar index) + phase.
__device__ __forceinline__ bool wait_bar(uint64_t *bars, int i, uint32_t phase, int *s_fail) {
    if (!tc::mbar_wait(&bars[i], phase)) atomicCAS(s_fail, 0, 1 + 2 * i + static_cast<int>(phase));
    __syncthreads();
    tc::fence_after_sync();
    return *s_fail == 0;
}

__device__ __forceinline__ void sync_mma() {
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

__global__ void __launch_bounds__(ANT, 1) attn_fwd_tc(AttnParams p, PlanDev pd) {
    using namespace at_sm;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smraw + ((1024 - (tc::smem_addr(smraw) & 1023)) & 1023);
    __shared__ uint64_t bars[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ int s_tab[AT];
    float *smax = reinterpret_cast<float *>(sm + Vec), *ssum = smax + 2 * AT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, lg = warp & 3, ch = warp >> 2;
    const int H = p.H;
    const int32_t h = blockIdx.x % H, qi = blockIdx.x / H;
    const int32_t sq = pd.attn_qt[2 * qi], qt = pd.attn_qt[2 * qi + 1];
    const int32_t hb = pd.attn_hptr[sq], hh = pd.attn_hptr[sq + 1] - hb;
    const int32_t row0 = pd.seq_row0[sq], own = pd.seq_nown[sq], nview = hh + own;
    const int32_t q0 = qt * AT, nq = min(AT, own - q0);
    const int32_t n_kt = (hh + q0 + nq - 1) / AT + 1;   // key tiles covering every visible entry

    if (tid == 0) {
        tc::mbar_init(&bars[0], 1);
        tc::mbar_init(&bars[1], 1);
        tc::fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(&s_tmem, 256);
        tc::fence_before_sync();
    }
    // Q rows (own q0 .. q0 + nq - 1, zero below the tile's end)
    for (int e = tid; e < AT * 16; e += ANT) {
        const int r = e >> 4, pc = e & 15;
        const bool ok = r < nq;
        const __nv_bfloat16 *src = p.q + ((static_cast<int64_t>(row0) + q0 + (ok ? r : 0)) * H + h) * AD + pc * 8;
        tc::cp_async16(sm + Q + piece(r, pc), src, ok ? 16u : 0u);
    }
    // key / value rows of view tile kt into buffer b
    auto stage_kv = [&](int32_t kt, int b) {
        if (tid < AT) {
            const int32_t j = kt * AT + tid;
            s_tab[tid] = j < hh ? pd.attn_hrows[hb + j] : (j < nview ? row0 + (j - hh) : -1);
        }
        __syncthreads();
        uint8_t *kd = sm + (b ? K1 : K0), *vd = sm + (b ? V1 : V0);
        for (int e = tid; e < 2 * AT * 16; e += ANT) {
            const int tv = e >> 11, r = (e >> 4) & (AT - 1), pc = e & 15;
            const int32_t row = s_tab[r];
            const __nv_bfloat16 *base = tv ? p.v : p.k;
            const __nv_bfloat16 *src = base + (static_cast<int64_t>(row < 0 ? 0 : row) * H + h) * AD + pc * 8;
            tc::cp_async16((tv ? vd : kd) + piece(r, pc), src, row >= 0 ? 16u : 0u);
        }
        tc::cp_async_commit();
    };
    stage_kv(0, 0);                                     // its barrier also publishes s_tmem
    tc::fence_after_sync();
    const uint32_t tm = s_tmem, lane_off = static_cast<uint32_t>(lg * 32) << 16;
    const uint32_t tS = tm, tO = tm + 128;
    const int qrow = lg * 32 + lane;                    // this thread's query row (TMEM lane)
    const int32_t vis = hh + q0 + qrow;                 // last view index it sees
    float m_run = -INFINITY, l_run = 0.f;

    for (int32_t kt = 0; kt < n_kt; ++kt) {
        const int b = kt & 1;
        const uint32_t ph = kt & 1;
        tc::cp_async_wait_all();
        sync_mma();
        if (tid == 0) {
            tc::mma_op(tS, tc::Opnd{tc::smem_addr(sm + Q), 16384, false},
                       tc::Opnd{tc::smem_addr(sm + (b ? K1 : K0)), 16384, false}, AT, AT, AD, false);
            tc::mma_commit(&bars[0]);
        }
        if (kt + 1 < n_kt) stage_kv(kt + 1, b ^ 1);     // that buffer's products are done
        if (!wait_bar(bars, 0, ph, &s_fail)) break;
        // ---- online softmax over this thread's 64 columns ---------------------------------
        float s[64];
        {
            float r[32];
            tc::tmem_ld32(tS + lane_off + ch * 64, r);
#pragma unroll
            for (int c = 0; c < 32; ++c) s[c] = r[c];
            tc::tmem_ld32(tS + lane_off + ch * 64 + 32, r);
#pragma unroll
            for (int c = 0; c < 32; ++c) s[32 + c] = r[c];
        }
        const int32_t j0 = kt * AT + ch * 64;
        float mloc = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            s[c] = (j0 + c <= vis) ? s[c] * p.scale : -INFINITY;
            mloc = fmaxf(mloc, s[c]);
        }
        smax[ch * AT + qrow] = mloc;
        __syncthreads();
        const float m_new = fmaxf(m_run, fmaxf(smax[qrow], smax[AT + qrow]));
        float sloc = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            s[c] = __expf(s[c] - m_new);
            sloc += s[c];
        }
#pragma unroll
        for (int c = 0; c < 64; c += 8) tc::st_sw128_8(sm + P, AT, qrow, ch * 64 + c, s + c);
        ssum[ch * AT + qrow] = sloc;
        const float alpha = __expf(m_run - m_new);
        __syncthreads();
        l_run = l_run * alpha + ssum[qrow] + ssum[AT + qrow];
        m_run = m_new;
        if (kt > 0) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float r[32];
                tc::tmem_ld32(tO + lane_off + ch * 64 + hf * 32, r);
#pragma unroll
                for (int c = 0; c < 32; ++c) r[c] *= alpha;
                tc::tmem_st32(tO + lane_off + ch * 64 + hf * 32, r);
            }
        }
        sync_mma();
        if (tid == 0) {
            tc::mma_op(tO, tc::Opnd{tc::smem_addr(sm + P), 16384, false},
                       tc::Opnd{tc::smem_addr(sm + (b ? V1 : V0)), 16384, true}, AT, AD, AT, kt > 0);
            tc::mma_commit(&bars[1]);
        }
        if (!wait_bar(bars, 1, ph, &s_fail)) break;
    }
    // ---- outputs ------------------------------------------------------------------------
    if (!s_fail) {
        const float inv = 1.f / l_run;
        const int64_t row = static_cast<int64_t>(row0) + q0 + qrow;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float r[32];
            tc::tmem_ld32(tO + lane_off + ch * 64 + hf * 32, r);
            if (qrow < nq) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + (row * H + h) * AD + ch * 64 + hf * 32);
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    uint4 w;
                    w.x = tc::pack_bf16(r[c] * inv, r[c + 1] * inv);
                    w.y = tc::pack_bf16(r[c + 2] * inv, r[c + 3] * inv);
                    w.z = tc::pack_bf16(r[c + 4] * inv, r[c + 5] * inv);
                    w.w = tc::pack_bf16(r[c + 6] * inv, r[c + 7] * inv);
                    dst[c / 8] = w;
                }
            }
        }
        if (p.lse && ch == 0 && qrow < nq) p.lse[row * H + h] = m_run + __logf(l_run);
    }
    tc::cp_async_wait_all();
    if (s_fail) {                                       // drain the product still in flight
        const int f = s_fail - 1;
        if (tid == 0) dev_error(pd, kDevErrTimeout, sq, h);
        tc::mbar_wait(&bars[f >> 1], static_cast<uint32_t>(f & 1), 1000000000LL);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tm, 256);
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
