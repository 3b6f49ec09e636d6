// Causal short convolution over the compact layout, forward and backward.
//
// HARTS (page "HARTS ... 精读", section 4.3, KDA paragraph; summary page, section 4 "KDA
// execution"): the causal convolution before KDA runs once per compact token; the window
// over the previous w - 1 tokens takes them from the token's real ancestors on its own
// trajectory and never crosses into another packed sequence.  Here: depthwise, width
// w <= 8, weight[c][w-1] on the current token and weight[c][w-1-j] on the token j
// positions earlier, optional bias, activation none or SiLU.  The plan image holds, per
// segment, the rows 1..7 positions before it (the ancestor context) and, per segment end
// and lag, the rows that follow it on every branch (for the backward, which gathers
// instead of scattering so that every sum has a fixed order).
//
// All of it is HBM-bound elementwise work in 16-byte vectors of 8 channels.  Consecutive
// threads take consecutive channel groups of one row (coalesced); a thread keeps its
// channel group for the whole launch (weights in registers) and walks runs of rows in
// order, so the predecessor rows it re-reads are rows it has just read.  The backward is
// one pass that reads x and dy and writes dx, with per-256-row partial sums of dweight and
// dbias reduced in a fixed order by a second small kernel.
#include <cstring>
#include <type_traits>

#include "kda_common.cuh"

namespace harts {
namespace {

constexpr int K = kConvMaxW - 1;
constexpr int kRowsPerPart = 256;       // rows per partial sum of dweight / dbias
constexpr int kBwdN = 4;                // channels per backward thread (8-byte bf16 vectors)

struct ConvParams {
    const void *x;
    void *y;
    const float *weight;    // [ch][w]
    const float *bias;      // [ch] or null
    const void *dy;
    void *dx;
    float *part;            // [n_part][ch][w+1] workspace
    float *dweight, *dbias;
    int64_t C;
    int32_t ch, w, act;
};

__device__ __forceinline__ void ld8(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void st8(float *p, const float (&v)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void st8(__nv_bfloat16 *p, const float (&v)[8]) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4 *>(p) = u;
}

// N = 4 channels (8 or 16 bytes).
__device__ __forceinline__ void ldn(const float *p, float (&v)[4]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void ldn(const __nv_bfloat16 *p, float (&v)[4]) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void ldn(const float *p, float (&v)[8]) { ld8(p, v); }
__device__ __forceinline__ void ldn(const __nv_bfloat16 *p, float (&v)[8]) { ld8(p, v); }
__device__ __forceinline__ void stn(float *p, const float (&v)[4]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void stn(__nv_bfloat16 *p, const float (&v)[4]) {
    uint2 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
    h[0] = __floats2bfloat162_rn(v[0], v[1]);
    h[1] = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2 *>(p) = u;
}

// Row j positions before row r (r is row i of segment seg), or -1 before the trajectory.
__device__ __forceinline__ int64_t pred_row(const PlanDev &pd, int64_t r, int32_t seg, int32_t i, int j) {
    return i >= j ? r - j : static_cast<int64_t>(pd.conv_ctx[seg * K + (j - i - 1)]);
}

// The backward's items are (block of rows, 8 channels); consecutive threads take
// consecutive channel groups (coalesced rows), and the grid stride is a multiple of the
// channel-group count, so a thread keeps one channel group -- its weights and bias stay
// in registers -- while it walks its rows (the rows it re-reads are ones it has just
// read: L1 hits).

template <int W, int N = 8>
struct Coef {
    float wt[W][N];           // wt[j][e] = weight[c0+e][W-1-j]
    float bias[N];
};

template <int W, int N>
__device__ __forceinline__ void load_coef(const ConvParams &p, int c0, Coef<W, N> &k) {
#pragma unroll
    for (int e = 0; e < N; ++e) k.bias[e] = p.bias ? __ldg(p.bias + c0 + e) : 0.f;
#pragma unroll
    for (int j = 0; j < W; ++j)
#pragma unroll
        for (int e = 0; e < N; ++e) k.wt[j][e] = __ldg(p.weight + (c0 + e) * W + (W - 1 - j));
}

// pre = bias + sum_j weight[:, w-1-j] x[row j back], N channels from c0
template <typename T, int W, int N>
__device__ __forceinline__ void conv_pre(const ConvParams &p, const PlanDev &pd, const Coef<W, N> &k, int64_t r,
                                         int32_t seg, int32_t i, int c0, float (&pre)[N]) {
    const T *x = static_cast<const T *>(p.x);
#pragma unroll
    for (int e = 0; e < N; ++e) pre[e] = k.bias[e];
#pragma unroll
    for (int j = 0; j < W; ++j) {
        const int64_t pr = pred_row(pd, r, seg, i, j);
        if (pr < 0) break;                       // so are all earlier positions
        float xv[N];
        ldn(x + pr * p.ch + c0, xv);
#pragma unroll
        for (int e = 0; e < N; ++e) pre[e] += k.wt[j][e] * xv[e];
    }
}

__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }
__device__ __forceinline__ float dsilu(float z) {
    const float s = 1.f / (1.f + __expf(-z));
    return s * (1.f + z * (1.f - s));
}

// Forward.  Item = (run of kRun consecutive rows, 8 channels); a thread keeps its channel
// group (weights in registers) and walks its runs.  A run's segment is looked up once and
// followed across segment boundaries; inside a segment, rows at least W-1 past its start
// go in batches of 4, whose W+3 input rows are loaded together (the rows shared with the
// previous batch are L1 hits); a segment's first W-1 rows take their context from the
// ancestor table.
constexpr int kRun = 32;

template <typename T>
__device__ __forceinline__ void act_store(const ConvParams &p, int64_t r, int c0, float (&v)[8]) {
    if (p.act) {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = silu(v[e]);
    }
    st8(static_cast<T *>(p.y) + r * p.ch + c0, v);
}

template <typename T, int W>
__global__ void __launch_bounds__(256) conv_fwd_kernel(ConvParams p, PlanDev pd) {
    const int G = p.ch / 8;
    const int64_t n = (p.C + kRun - 1) / kRun * G;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;   // a multiple of G
    int64_t it = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (it >= n) return;
    const int c0 = static_cast<int>(it % G) * 8;
    const T *x = static_cast<const T *>(p.x);
    Coef<W> k;
    load_coef<W, 8>(p, c0, k);
    for (; it < n; it += stride) {
        const int64_t r0 = it / G * kRun, r1 = min(p.C, r0 + kRun);
        int64_t r = r0;
        int32_t seg = pd.row_seg[r];
        int64_t srow0 = pd.seg_row0[seg], send = srow0 + pd.seg_len[seg];
        while (r < r1) {
            const int64_t rend = min(r1, send);
            // a segment's first W-1 rows: context from the ancestor table
            for (; r < rend && r - srow0 < W - 1; ++r) {
                float v[8];
                conv_pre<T, W, 8>(p, pd, k, r, seg, static_cast<int32_t>(r - srow0), c0, v);
                act_store<T>(p, r, c0, v);
            }
            // the rest in batches of 4: inputs r-W+1 .. r+3, all in this segment
            for (; r + 4 <= rend; r += 4) {
                float xin[W + 3][8];
#pragma unroll
                for (int q = 0; q < W + 3; ++q) ld8(x + (r - (W - 1) + q) * p.ch + c0, xin[q]);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = k.bias[e];
#pragma unroll
                    for (int j = 0; j < W; ++j)
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] += k.wt[j][e] * xin[u + W - 1 - j][e];
                    act_store<T>(p, r + u, c0, v);
                }
            }
            for (; r < rend; ++r) {
                float v[8];
                conv_pre<T, W, 8>(p, pd, k, r, seg, static_cast<int32_t>(r - srow0), c0, v);
                act_store<T>(p, r, c0, v);
            }
            if (r < r1) {
                seg = pd.row_seg[r];
                srow0 = r;
                send = srow0 + pd.seg_len[seg];
            }
        }
    }
}

// dL/dpre of row s (row i of segment seg): dy[s] * act'(pre[s]), pre recomputed.
template <typename T, int W, int N>
__device__ __forceinline__ void dpre_of(const ConvParams &p, const PlanDev &pd, const Coef<W, N> &k, int64_t s,
                                        int32_t seg, int32_t i, int c0, float (&g)[N]) {
    ldn(static_cast<const T *>(p.dy) + s * p.ch + c0, g);
    if (p.act) {
        float pre[N];
        conv_pre<T, W, N>(p, pd, k, s, seg, i, c0, pre);
#pragma unroll
        for (int e = 0; e < N; ++e) g[e] *= dsilu(pre[e]);
    }
}

// Fused backward.  Item = (block of kRowsPerPart rows, 8 channels); rows walked in order.
// dp[d] holds dL/dpre of row r + d (same segment) for d < W, kept as a shift register so
// that each row's value is formed once; dx[r] = sum_d weight[:, W-1-d] * (dp[d], or for
// successors beyond the segment's end the sum over the successor list of their dL/dpre,
// recomputed from dy and x); the partial sums of dweight and dbias of the block are
// written to the workspace.  Reads x and dy, writes dx: the op's own traffic.
template <typename T, int W>
__global__ void __launch_bounds__(256) conv_bwd_kernel(ConvParams p, PlanDev pd) {
    constexpr int N = kBwdN;
    const int G = p.ch / N;
    const int64_t n_part = (p.C + kRowsPerPart - 1) / kRowsPerPart;
    const int64_t n = n_part * G;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;   // a multiple of G
    const T *x = static_cast<const T *>(p.x);
    int64_t it = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (it >= n) return;
    const int c0 = static_cast<int>(it % G) * N;
    Coef<W, N> k;
    load_coef<W, N>(p, c0, k);
    for (; it < n; it += stride) {
        const int64_t pb = it / G;
        float dw[W][N], db[N], dp[W][N];
#pragma unroll
        for (int j = 0; j < W; ++j)
#pragma unroll
            for (int e = 0; e < N; ++e) { dw[j][e] = 0.f; dp[j][e] = 0.f; }
#pragma unroll
        for (int e = 0; e < N; ++e) db[e] = 0.f;
        const int64_t r0 = pb * kRowsPerPart, r1 = min(p.C, r0 + kRowsPerPart);
        // the block's segment is looked up once and followed across boundaries
        int32_t seg = pd.row_seg[r0];
        int64_t row0 = pd.seg_row0[seg];
        int32_t len = pd.seg_len[seg];
        for (int64_t r = r0; r < r1; ++r) {
            if (r == row0 + len) {
                seg = pd.row_seg[r];
                row0 = r;
                len = pd.seg_len[seg];
            }
            int32_t i = static_cast<int32_t>(r - row0);
            // interior rows (the window and the look-ahead inside the segment) run from
            // registers: the x rows r-W+1 .. r+W-1 slide, and only x, dy of row r+W-1 are
            // new, loaded one row ahead
            if (r != r0 && i >= W - 1 && i + 2 * W - 2 < len) {
                const int64_t fend = min(r1, row0 + len - (W - 1));
                float xw[2 * W - 1][N];
#pragma unroll
                for (int q = 0; q < 2 * W - 2; ++q) ldn(x + (r - (W - 1) + q) * p.ch + c0, xw[q]);
                float nx[N], nd[N];
                ldn(x + (r + W - 1) * p.ch + c0, nx);
                ldn(static_cast<const T *>(p.dy) + (r + W - 1) * p.ch + c0, nd);
                for (; r < fend; ++r) {
                    float cd[N];
#pragma unroll
                    for (int e = 0; e < N; ++e) { xw[2 * W - 2][e] = nx[e]; cd[e] = nd[e]; }
                    if (r + 1 < fend) {
                        ldn(x + (r + W) * p.ch + c0, nx);
                        ldn(static_cast<const T *>(p.dy) + (r + W) * p.ch + c0, nd);
                    }
                    if (p.act) {
                        float pre[N];
#pragma unroll
                        for (int e = 0; e < N; ++e) pre[e] = k.bias[e];
#pragma unroll
                        for (int j = 0; j < W; ++j)
#pragma unroll
                            for (int e = 0; e < N; ++e) pre[e] += k.wt[j][e] * xw[2 * W - 2 - j][e];
#pragma unroll
                        for (int e = 0; e < N; ++e) cd[e] *= dsilu(pre[e]);
                    }
#pragma unroll
                    for (int e = 0; e < N; ++e) dp[W - 1][e] = cd[e];
                    float acc[N];
#pragma unroll
                    for (int e = 0; e < N; ++e) acc[e] = 0.f;
#pragma unroll
                    for (int d = 0; d < W; ++d)
#pragma unroll
                        for (int e = 0; e < N; ++e) acc[e] += k.wt[d][e] * dp[d][e];
                    stn(static_cast<T *>(p.dx) + r * p.ch + c0, acc);
#pragma unroll
                    for (int e = 0; e < N; ++e) db[e] += dp[0][e];
#pragma unroll
                    for (int j = 0; j < W; ++j)
#pragma unroll
                        for (int e = 0; e < N; ++e) dw[j][e] += xw[W - 1 - j][e] * dp[0][e];
#pragma unroll
                    for (int d = 0; d + 1 < W; ++d)
#pragma unroll
                        for (int e = 0; e < N; ++e) dp[d][e] = dp[d + 1][e];
#pragma unroll
                    for (int q = 0; q + 1 < 2 * W - 1; ++q)
#pragma unroll
                        for (int e = 0; e < N; ++e) xw[q][e] = xw[q + 1][e];
                }
                if (r >= r1) break;
                if (r == row0 + len) {
                    seg = pd.row_seg[r];
                    row0 = r;
                    len = pd.seg_len[seg];
                }
                i = static_cast<int32_t>(r - row0);
            }
            if (r == r0 || i == 0) {
                // (re)fill dp[0 .. W-2] for this segment
#pragma unroll
                for (int d = 0; d + 1 < W; ++d)
                    if (i + d < len) dpre_of<T, W, N>(p, pd, k, r + d, seg, i + d, c0, dp[d]);
            }
            if (i + W - 1 < len) dpre_of<T, W, N>(p, pd, k, r + W - 1, seg, i + W - 1, c0, dp[W - 1]);
            // dx[r]
            float acc[N];
#pragma unroll
            for (int e = 0; e < N; ++e) acc[e] = 0.f;
#pragma unroll
            for (int d = 0; d < W; ++d) {
                if (i + d < len) {
#pragma unroll
                    for (int e = 0; e < N; ++e) acc[e] += k.wt[d][e] * dp[d][e];
                } else {
                    const int ee = i + d - len;
                    const int32_t b = pd.conv_sptr[seg * K + ee], end = pd.conv_sptr[seg * K + ee + 1];
                    for (int32_t q = b; q < end; ++q) {
                        const int64_t sr = pd.conv_succ[q];
                        const int32_t ss = pd.row_seg[sr];
                        float t[N];
                        dpre_of<T, W, N>(p, pd, k, sr, ss, static_cast<int32_t>(sr - pd.seg_row0[ss]), c0, t);
#pragma unroll
                        for (int e = 0; e < N; ++e) acc[e] += k.wt[d][e] * t[e];
                    }
                }
            }
            stn(static_cast<T *>(p.dx) + r * p.ch + c0, acc);
            // dweight / dbias partials with dL/dpre of row r
#pragma unroll
            for (int e = 0; e < N; ++e) db[e] += dp[0][e];
#pragma unroll
            for (int j = 0; j < W; ++j) {
                const int64_t pr = pred_row(pd, r, seg, i, j);
                if (pr < 0) break;
                float xv[N];
                ldn(x + pr * p.ch + c0, xv);
#pragma unroll
                for (int e = 0; e < N; ++e) dw[j][e] += xv[e] * dp[0][e];
            }
#pragma unroll
            for (int d = 0; d + 1 < W; ++d)
#pragma unroll
                for (int e = 0; e < N; ++e) dp[d][e] = dp[d + 1][e];
        }
        float *out = p.part + (pb * p.ch + c0) * (W + 1);
#pragma unroll
        for (int e = 0; e < N; ++e) {
#pragma unroll
            for (int j = 0; j < W; ++j) out[e * (W + 1) + (W - 1 - j)] = dw[j][e];
            out[e * (W + 1) + W] = db[e];
        }
    }
}

// dweight, dbias: the partial sums in block order
__global__ void __launch_bounds__(256) conv_bwd_reduce_kernel(ConvParams p) {
    const int64_t n_part = (p.C + kRowsPerPart - 1) / kRowsPerPart;
    const int W1 = p.w + 1;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < p.ch * W1; idx += gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int64_t b = 0; b < n_part; ++b) s += p.part[b * p.ch * W1 + idx];
        const int c = idx / W1, k = idx - c * W1;
        if (k < p.w) p.dweight[c * p.w + k] = s;
        else if (p.dbias) p.dbias[c] = s;
    }
}

// Blocks for `items` items of G channel groups: the grid's thread count is a multiple of
// G (so a thread keeps its channel group) and about 8 blocks per SM.
int grid_groups(int64_t items, int G) {
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    int64_t step = 1;                                   // blocks per multiple of G threads
    while ((step * 256) % G) ++step;
    const int64_t want = (items + 255) / 256;
    int64_t blocks = std::min<int64_t>(want, int64_t(nsm) * 8);
    blocks = std::max<int64_t>(step, (blocks + step - 1) / step * step);
    return static_cast<int>(blocks);
}

int grid_for(int64_t items) {
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (items + 255) / 256;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(nsm) * 16)));
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Calls f(std::integral_constant<int, w>) for w in 1..kConvMaxW (checked by the caller).
template <typename F>
void with_width(int w, F &&f) {
    switch (w) {
        case 1: f(std::integral_constant<int, 1>{}); break;
        case 2: f(std::integral_constant<int, 2>{}); break;
        case 3: f(std::integral_constant<int, 3>{}); break;
        case 4: f(std::integral_constant<int, 4>{}); break;
        case 5: f(std::integral_constant<int, 5>{}); break;
        case 6: f(std::integral_constant<int, 6>{}); break;
        case 7: f(std::integral_constant<int, 7>{}); break;
        default: f(std::integral_constant<int, 8>{}); break;
    }
}

int check_args(const harts_plan *P, const harts_conv_fwd_args *a) {
    if (!P || !a) { set_error("NULL plan or args"); return HARTS_EINVAL; }
    if (!P->dev) { set_error("plan not uploaded (harts_plan_upload)"); return HARTS_ENOPLAN; }
    if (a->dtype != HARTS_FP32 && a->dtype != HARTS_BF16) { set_error("dtype"); return HARTS_EUNSUPPORTED; }
    if (a->channels < 8 || a->channels % 8) { set_error("channels must be a positive multiple of 8"); return HARTS_EINVAL; }
    if (a->width < 1 || a->width > kConvMaxW) { set_error("width must be 1..8"); return HARTS_EUNSUPPORTED; }
    if (a->activation != 0 && a->activation != 1) { set_error("activation must be 0 (none) or 1 (silu)"); return HARTS_EINVAL; }
    if (!a->x || !a->weight) { set_error("NULL x or weight"); return HARTS_EINVAL; }
    if ((reinterpret_cast<uintptr_t>(a->x) | reinterpret_cast<uintptr_t>(a->weight)) & 15) {
        set_error("x and weight must be 16-byte aligned"); return HARTS_EINVAL;
    }
    if (P->info.C * int64_t(a->channels) > (int64_t(1) << 40)) { set_error("tensor too large"); return HARTS_EOVERFLOW; }
    return HARTS_OK;
}

ConvParams make_params(const harts_plan *P, const harts_conv_fwd_args *a) {
    ConvParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = a->x; p.y = a->y; p.weight = a->weight; p.bias = a->bias;
    p.C = P->info.C; p.ch = a->channels; p.w = a->width; p.act = a->activation;
    return p;
}

int cuda_fail(cudaError_t e, const char *what) {
    set_error(std::string(what) + ": " + cudaGetErrorString(e));
    return HARTS_ECUDA;
}

}  // namespace
}  // namespace harts

using namespace harts;

extern "C" {

int harts_conv_fwd(const harts_plan *P, const harts_conv_fwd_args *a, harts_stream_t stream) {
    int rc = check_args(P, a);
    if (rc) return rc;
    if (!a->y || (reinterpret_cast<uintptr_t>(a->y) & 15)) { set_error("y must be non-NULL and 16-byte aligned"); return HARTS_EINVAL; }
    if (P->info.C == 0) { set_error(""); return HARTS_OK; }
    ConvParams p = make_params(P, a);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int grid = grid_groups((p.C + kRun - 1) / kRun * (p.ch / 8), p.ch / 8);
    with_width(p.w, [&](auto wc) {
        constexpr int W = decltype(wc)::value;
        if (a->dtype == HARTS_BF16) conv_fwd_kernel<__nv_bfloat16, W><<<grid, 256, 0, st>>>(p, P->view);
        else conv_fwd_kernel<float, W><<<grid, 256, 0, st>>>(p, P->view);
    });
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "conv forward launch");
    set_error("");
    return HARTS_OK;
}

size_t harts_conv_bwd_workspace_bytes(const harts_plan *P, int32_t channels, int32_t width) {
    if (!P || channels < 1 || width < 1 || width > kConvMaxW) return 0;
    const int64_t n_part = (P->info.C + kRowsPerPart - 1) / kRowsPerPart;
    return align_up(sizeof(float) * size_t(n_part) * channels * (width + 1));
}

int harts_conv_bwd(const harts_plan *P, const harts_conv_bwd_args *a, harts_stream_t stream) {
    if (!a) { set_error("NULL args"); return HARTS_EINVAL; }
    int rc = check_args(P, &a->fwd);
    if (rc) return rc;
    if (!a->dy || !a->dx || !a->dweight) { set_error("NULL dy, dx or dweight"); return HARTS_EINVAL; }
    if ((reinterpret_cast<uintptr_t>(a->dy) | reinterpret_cast<uintptr_t>(a->dx) |
         reinterpret_cast<uintptr_t>(a->workspace)) & 15) {
        set_error("dy, dx and the workspace must be 16-byte aligned"); return HARTS_EINVAL;
    }
    const size_t need = harts_conv_bwd_workspace_bytes(P, a->fwd.channels, a->fwd.width);
    if (!a->workspace || a->workspace_bytes < need) { set_error("conv workspace too small"); return HARTS_ESMALLBUF; }
    ConvParams p = make_params(P, &a->fwd);
    p.dy = a->dy; p.dx = a->dx; p.dweight = a->dweight; p.dbias = a->dbias;
    p.part = static_cast<float *>(a->workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (P->info.C > 0) {
        const int64_t n_part = (p.C + kRowsPerPart - 1) / kRowsPerPart;
        const int g1 = grid_groups(n_part * (p.ch / kBwdN), p.ch / kBwdN);
        with_width(p.w, [&](auto wc) {
            constexpr int W = decltype(wc)::value;
            if (a->fwd.dtype == HARTS_BF16) conv_bwd_kernel<__nv_bfloat16, W><<<g1, 256, 0, st>>>(p, P->view);
            else conv_bwd_kernel<float, W><<<g1, 256, 0, st>>>(p, P->view);
        });
        conv_bwd_reduce_kernel<<<grid_for(int64_t(p.ch) * (p.w + 1)), 256, 0, st>>>(p);
        e = cudaGetLastError();
    } else {
        e = cudaMemsetAsync(a->dweight, 0, sizeof(float) * size_t(p.ch) * p.w, st);
        if (e == cudaSuccess && a->dbias) e = cudaMemsetAsync(a->dbias, 0, sizeof(float) * size_t(p.ch), st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "conv backward launch");
    set_error("");
    return HARTS_OK;
}

}  // extern "C"
