// Compact-to-semantic log-probabilities (forward and backward).
//
// HARTS (page "HARTS ... 精读", section 4.4, "紧凑到语义的 log 概率"; summary page,
// "Semantic Preservation"): each compact logit row is reduced over the vocabulary once
// (its log-sum-exp); every semantic position s reads its own target logit from the row its
// token maps to, lambda_s = z[c(s), y_s] - lse[c(s)]; the backward (eq. 19) sums the
// independently formed gradients of the row's semantic positions onto it:
//   dz[c] = sum_{s -> c} g_s (onehot(y_s) - softmax(z[c])).
// Vocabulary work is O(C V) + O(S); no S x V array is formed.
//
// One block per compact row (grid-stride over rows).  Forward: one pass over the row with
// a running (max, sum-exp) per thread in 16-byte vectors, a block reduction, then the
// row's semantic positions gather their target logits.  Backward: a dense pass writes
// -G_c softmax(z[c]) (G_c = the row's g summed in list order); after a barrier the entries
// at the row's distinct targets are rewritten with -G_c p_v + (their g, summed in list
// order), formed in fp32, so the sparse terms are not rounded twice.  Deterministic.
#include <cstring>
#include <vector>

#include "kda_common.cuh"

namespace harts {
namespace {

constexpr int kThreads = 512;

struct LpParams {
    const void *logits;
    void *dlogits;
    const int32_t *row_ptr, *row_sem, *target;
    float *lse, *logp;
    const float *dlogp;
    int64_t C;
    int32_t V;
};

template <typename T> __device__ __forceinline__ float ld1(const T *p);
template <> __device__ __forceinline__ float ld1<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

__device__ __forceinline__ void ld8v(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void ld8v(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void st8v(float *p, const float (&v)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void st8v(__nv_bfloat16 *p, const float (&v)[8]) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4 *>(p) = u;
}
__device__ __forceinline__ void st1(float *p, float v) { *p = v; }
__device__ __forceinline__ void st1(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// combine running (max, sum of exp(x - max)) pairs
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
    if (m2 > m) { s = s * __expf(m - m2) + s2; m = m2; }
    else if (m2 > -INFINITY) s += s2 * __expf(m2 - m);
}

// log-sum-exp of row z (length V), every thread of the block returns it
template <typename T>
__device__ float row_lse(const T *z, int V, float *sm_m, float *sm_s) {
    const int tid = threadIdx.x, nv = V / 8;
    float m = -INFINITY, s = 0.f;
    for (int q = tid; q < nv; q += blockDim.x) {
        float v[8];
        ld8v(z + q * 8, v);
        float bm = v[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) bm = fmaxf(bm, v[e]);
        float bs = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) bs += __expf(v[e] - bm);
        lse_merge(m, s, bm, bs);
    }
    for (int q = nv * 8 + tid; q < V; q += blockDim.x) lse_merge(m, s, ld1(z + q), 1.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
        lse_merge(m, s, m2, s2);
    }
    const int warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    if (lane == 0) { sm_m[warp] = m; sm_s[warp] = s; }
    __syncthreads();
    if (warp == 0) {
        m = lane < nw ? sm_m[lane] : -INFINITY;
        s = lane < nw ? sm_s[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
            lse_merge(m, s, m2, s2);
        }
        if (lane == 0) sm_m[0] = m + __logf(s);
    }
    __syncthreads();
    const float out = sm_m[0];
    __syncthreads();            // sm_m is reused by the next row
    return out;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) logprob_fwd_kernel(LpParams p) {
    __shared__ float sm_m[32], sm_s[32];
    const T *logits = static_cast<const T *>(p.logits);
    for (int64_t c = blockIdx.x; c < p.C; c += gridDim.x) {
        const T *z = logits + c * p.V;
        const float lse = row_lse<T>(z, p.V, sm_m, sm_s);
        if (threadIdx.x == 0) p.lse[c] = lse;
        for (int32_t q = p.row_ptr[c] + threadIdx.x; q < p.row_ptr[c + 1]; q += blockDim.x) {
            const int32_t s = p.row_sem[q];
            p.logp[s] = ld1(z + p.target[s]) - lse;
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) logprob_bwd_kernel(LpParams p) {
    __shared__ float sm_g;
    const T *logits = static_cast<const T *>(p.logits);
    T *dlogits = static_cast<T *>(p.dlogits);
    for (int64_t c = blockIdx.x; c < p.C; c += gridDim.x) {
        const int32_t b = p.row_ptr[c], e = p.row_ptr[c + 1];
        if (threadIdx.x == 0) {
            float G = 0.f;
            for (int32_t q = b; q < e; ++q) G += p.dlogp[p.row_sem[q]];
            sm_g = G;
        }
        __syncthreads();
        const float G = sm_g, lse = p.lse[c];
        const T *z = logits + c * p.V;
        T *dz = dlogits + c * p.V;
        const int nv = p.V / 8;
        for (int q = threadIdx.x; q < nv; q += blockDim.x) {
            float v[8];
            ld8v(z + q * 8, v);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = -G * __expf(v[k] - lse);
            st8v(dz + q * 8, v);
        }
        for (int q = nv * 8 + threadIdx.x; q < p.V; q += blockDim.x) st1(dz + q, -G * __expf(ld1(z + q) - lse));
        __syncthreads();
        // distinct targets of the row: the first list entry of each target writes
        for (int32_t q = b + threadIdx.x; q < e; q += blockDim.x) {
            const int32_t y = p.target[p.row_sem[q]];
            bool first = true;
            for (int32_t t = b; t < q && first; ++t) first = p.target[p.row_sem[t]] != y;
            if (!first) continue;
            float gs = 0.f;
            for (int32_t t = q; t < e; ++t)
                if (p.target[p.row_sem[t]] == y) gs += p.dlogp[p.row_sem[t]];
            st1(dz + y, -G * __expf(ld1(z + y) - lse) + gs);
        }
        __syncthreads();        // sm_g is reused by the next row
    }
}

int grid_rows(int64_t C) {
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(C, int64_t(nsm) * 4)));
}

int check_args(const harts_logprob_fwd_args *a) {
    if (!a) { set_error("NULL args"); return HARTS_EINVAL; }
    if (a->dtype != HARTS_FP32 && a->dtype != HARTS_BF16) { set_error("dtype"); return HARTS_EUNSUPPORTED; }
    if (a->C < 0 || a->S < 0 || a->V < 1) { set_error("C, S >= 0 and V >= 1 required"); return HARTS_EINVAL; }
    if (a->S > 0x7fffffff) { set_error("more than 2^31-1 semantic positions"); return HARTS_EOVERFLOW; }
    if (a->C > 0 && (!a->logits || !a->row_ptr || !a->lse)) { set_error("NULL logits, row_ptr or lse"); return HARTS_EINVAL; }
    if (a->S > 0 && (!a->row_sem || !a->target)) { set_error("NULL row_sem or target"); return HARTS_EINVAL; }
    if (reinterpret_cast<uintptr_t>(a->logits) & 15) { set_error("logits must be 16-byte aligned"); return HARTS_EINVAL; }
    if (a->V % 8) { set_error("V must be a multiple of 8 (row starts 16-byte aligned)"); return HARTS_EINVAL; }
    return HARTS_OK;
}

LpParams make(const harts_logprob_fwd_args *a) {
    LpParams p;
    std::memset(&p, 0, sizeof(p));
    p.logits = a->logits; p.row_ptr = a->row_ptr; p.row_sem = a->row_sem; p.target = a->target;
    p.lse = a->lse; p.logp = a->logp; p.C = a->C; p.V = a->V;
    return p;
}

}  // namespace
}  // namespace harts

using namespace harts;

extern "C" {

int harts_plan_semantic_map(const harts_plan *P, int32_t *sem_row, int32_t *row_ptr, int32_t *row_sem) {
    if (!P || !sem_row || !row_ptr || !row_sem) { set_error("NULL argument"); return HARTS_EINVAL; }
    if (P->info.S > 0x7fffffff) { set_error("more than 2^31-1 semantic positions"); return HARTS_EOVERFLOW; }
    const int32_t n = P->info.n_seg;
    std::vector<char> has_kid(n, 0);
    for (int32_t v = 0; v < n; ++v) if (P->parent[v] >= 0) has_kid[P->parent[v]] = 1;
    std::vector<int32_t> chain;
    int64_t s = 0;
    for (int32_t leaf = 0; leaf < n; ++leaf) {
        if (has_kid[leaf]) continue;
        chain.clear();
        for (int32_t v = leaf; v >= 0; v = P->parent[v]) chain.push_back(v);
        for (auto it = chain.rbegin(); it != chain.rend(); ++it)
            for (int64_t t = 0; t < P->seg_len[*it]; ++t) sem_row[s++] = static_cast<int32_t>(P->seg_offset[*it] + t);
    }
    const int64_t C = P->info.C;
    std::memset(row_ptr, 0, sizeof(int32_t) * size_t(C + 1));
    for (int64_t q = 0; q < s; ++q) row_ptr[sem_row[q] + 1]++;
    for (int64_t c = 0; c < C; ++c) row_ptr[c + 1] += row_ptr[c];
    std::vector<int32_t> fill(row_ptr, row_ptr + C);
    for (int64_t q = 0; q < s; ++q) row_sem[fill[sem_row[q]]++] = static_cast<int32_t>(q);
    set_error("");
    return HARTS_OK;
}

int harts_logprob_fwd(const harts_logprob_fwd_args *a, harts_stream_t stream) {
    int rc = check_args(a);
    if (rc) return rc;
    if (a->S > 0 && !a->logp) { set_error("NULL logp"); return HARTS_EINVAL; }
    if (a->C == 0) { set_error(""); return HARTS_OK; }
    LpParams p = make(a);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (a->dtype == HARTS_BF16) logprob_fwd_kernel<__nv_bfloat16><<<grid_rows(a->C), kThreads, 0, st>>>(p);
    else logprob_fwd_kernel<float><<<grid_rows(a->C), kThreads, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_error(std::string("log-prob forward launch: ") + cudaGetErrorString(e)); return HARTS_ECUDA; }
    set_error("");
    return HARTS_OK;
}

int harts_logprob_bwd(const harts_logprob_bwd_args *a, harts_stream_t stream) {
    if (!a) { set_error("NULL args"); return HARTS_EINVAL; }
    int rc = check_args(&a->fwd);
    if (rc) return rc;
    if (a->fwd.C > 0 && (!a->dlogits || (reinterpret_cast<uintptr_t>(a->dlogits) & 15))) {
        set_error("dlogits must be non-NULL and 16-byte aligned"); return HARTS_EINVAL;
    }
    if (a->fwd.S > 0 && !a->dlogp) { set_error("NULL dlogp"); return HARTS_EINVAL; }
    if (a->fwd.C == 0) { set_error(""); return HARTS_OK; }
    LpParams p = make(&a->fwd);
    p.dlogits = a->dlogits;
    p.dlogp = a->dlogp;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (a->fwd.dtype == HARTS_BF16) logprob_bwd_kernel<__nv_bfloat16><<<grid_rows(a->fwd.C), kThreads, 0, st>>>(p);
    else logprob_bwd_kernel<float><<<grid_rows(a->fwd.C), kThreads, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_error(std::string("log-prob backward launch: ") + cudaGetErrorString(e)); return HARTS_ECUDA; }
    set_error("");
    return HARTS_OK;
}

}  // extern "C"
