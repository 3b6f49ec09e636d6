// C ABI entry points that touch the device: plan upload, forward and backward dispatch.
#include <cstring>
#include <mutex>

#include "kda_common.cuh"
#include "tc_primitives.cuh"

namespace harts {

bool simt_supported(bool backward, int D, int BC);
cudaError_t simt_fwd_round(int dtype, int BC, const FwdParams &p, const PlanDev &pd,
                           int32_t base, int32_t n_items, cudaStream_t st);
cudaError_t simt_bwd_round(int dtype, int BC, const BwdParams &p, const PlanDev &pd,
                           int32_t base, int32_t n_items, cudaStream_t st);
cudaError_t bwd_finish(int dtype, const BwdParams &p, const PlanDev &pd, cudaStream_t st);

bool tc_supported(bool backward, int dtype, int D, int BC);
cudaError_t tc2_fwd_round(const FwdParams &p, const PlanDev &pd, int32_t base, int32_t n_items, cudaStream_t st);
cudaError_t tc_fwd_round(const FwdParams &p, const PlanDev &pd, int32_t base, int32_t n_items,
                         int32_t max_chunks, cudaStream_t st);
cudaError_t tc2_bwd_state_round(const BwdParams &p, const PlanDev &pd, int32_t base, int32_t n_items,
                                cudaStream_t st);

cudaError_t tc2_bwd_grad(const BwdParams &p, const PlanDev &pd, int32_t chunk_begin, int32_t n_items,
                         cudaStream_t st);


namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int cuda_fail(cudaError_t e, const char *what) {
    set_error(std::string(what) + ": " + cudaGetErrorString(e));
    return HARTS_ECUDA;
}

size_t dtype_size(int32_t dt) { return dt == HARTS_FP32 ? 4 : 2; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }   // NULL passes

int check_fwd_args(const harts_plan *P, const harts_kda_fwd_args *a) {
    if (!P || !a) { set_error("NULL plan or args"); return HARTS_EINVAL; }
    if (!P->dev) { set_error("plan not uploaded (harts_plan_upload)"); return HARTS_ENOPLAN; }
    if (a->dtype != HARTS_FP32 && a->dtype != HARTS_BF16) { set_error("dtype"); return HARTS_EUNSUPPORTED; }
    if (a->H < 1 || a->dk < 1 || a->dv < 1) { set_error("H, dk, dv must be >= 1"); return HARTS_EINVAL; }
    if (a->dk != a->dv) { set_error("dk != dv is not supported"); return HARTS_EUNSUPPORTED; }
    if (!a->q || !a->k || !a->v || !a->g || !a->beta) { set_error("NULL input"); return HARTS_EINVAL; }
    // rows are moved 16 bytes at a time (tensor maps, vector loads and stores)
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->g) || !aligned16(a->o) ||
        !aligned16(a->chunk_states)) {
        set_error("q, k, v, g, o and chunk_states must be 16-byte aligned");
        return HARTS_EINVAL;
    }
    if (P->info.n_states > 0 && !a->states) { set_error("states required (n_states > 0)"); return HARTS_EINVAL; }
    if (a->kernel < HARTS_KERNEL_AUTO || a->kernel > HARTS_KERNEL_TC) { set_error("kernel"); return HARTS_EINVAL; }
    // row * H * D offsets are formed in int64 inside the kernels; (row, head) indices of
    // beta and the launch grids are int32
    if (P->info.C * int64_t(a->H) > int64_t(0x7fffffff)) {
        set_error("C * H exceeds 2^31 - 1 (row, head) pairs");
        return HARTS_EOVERFLOW;
    }
    return HARTS_OK;
}

// Which kernel family runs: 0 = SIMT, 1 = tensor core, -1 = none.
int pick(const harts_kda_fwd_args *a, int BC, bool backward) {
    const int D = a->dk;
    const bool tc = tc_supported(backward, a->dtype, D, BC);
    const bool simt = simt_supported(backward, D, BC);
    if (a->kernel == HARTS_KERNEL_TC) return tc ? 1 : -1;
    if (a->kernel == HARTS_KERNEL_SIMT) return simt ? 0 : -1;
    if (tc) return 1;
    return simt ? 0 : -1;
}

FwdParams make_fwd(const harts_kda_fwd_args *a) {
    FwdParams p{};
    p.q = a->q; p.k = a->k; p.v = a->v; p.g = a->g; p.beta = a->beta; p.o = a->o;
    p.states = a->states; p.final_state = a->final_state; p.h0 = a->h0;
    p.chunk_states = a->chunk_states; p.H = a->H; p.D = a->dk; p.scale = a->scale;
    return p;
}

// Backward workspace: per-sequence initial-state gradients (fp32), per-replay-occurrence
// gradients (fp32), and the carried state gradient at every chunk end (bf16, tensor-core
// path only).
struct BwdWs { size_t ds_init, rep_grad, dchunk, total; };
BwdWs bwd_ws(const harts_plan *P, int32_t H, int32_t D, bool tc) {
    BwdWs w{};
    w.ds_init = 0;
    w.rep_grad = align_up(sizeof(float) * size_t(P->info.n_seq) * H * D * D);
    w.dchunk = w.rep_grad + align_up(sizeof(float) * size_t(P->info.R) * H * rep_width(D));
    w.total = w.dchunk + (tc ? align_up(size_t(2) * size_t(P->info.n_chunks) * H * D * D) : 0);
    return w;
}

}  // namespace
}  // namespace harts

using namespace harts;

namespace harts {
namespace {

// The library's bounded-wait failure path, on its own: one thread waits on an mbarrier
// that nothing completes, gives up after max_cycles and records device code 3 (timeout)
// in the plan's error word, as every kernel of the library does when a wait runs out.
__global__ void selftest_timeout_kernel(PlanDev pd, uint32_t max_cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
        if (!tc::mbar_wait(&bar, 0, static_cast<long long>(max_cycles))) dev_error(pd, kDevErrTimeout, -1, -1);
    }
}

}  // namespace
}  // namespace harts

extern "C" {

int harts_plan_upload(harts_plan *P, void *dev_buf, size_t bytes, harts_stream_t stream) {
    if (!P || !dev_buf) { set_error("NULL plan or buffer"); return HARTS_EINVAL; }
    const size_t need = harts_plan_device_bytes(P);
    if (bytes < need) { set_error("plan device buffer too small"); return HARTS_ESMALLBUF; }
    if (reinterpret_cast<uintptr_t>(dev_buf) % 256) { set_error("plan buffer must be 256-B aligned"); return HARTS_EINVAL; }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(dev_buf, P->image.words.data(), need, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "plan upload");
    // The copy reads pageable host memory; make sure it finished before the plan can change.
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "plan upload sync");
    P->dev = dev_buf;
    int32_t *w = static_cast<int32_t *>(dev_buf);
    const PlanImage &I = P->image;
    PlanDev &v = P->view;
    v.err = w + I.off_err;
    v.round_seq_ptr = w + I.off_round_seq_ptr; v.round_order = w + I.off_round_order;
    v.seq_row0 = w + I.off_seq_row0; v.seq_nown = w + I.off_seq_nown; v.seq_rho = w + I.off_seq_rho;
    v.seq_rptr = w + I.off_seq_rptr; v.seq_src = w + I.off_seq_src; v.seq_sptr = w + I.off_seq_sptr;
    v.state_lpos = w + I.off_state_lpos; v.seq_cbase = w + I.off_seq_cbase;
    v.state_cptr = w + I.off_state_cptr; v.state_cons = w + I.off_state_cons;
    v.root_cptr = w + I.off_root_cptr; v.root_cons = w + I.off_root_cons;
    v.replay_idx = w + I.off_replay_idx; v.fold_rows = w + I.off_fold_rows;
    v.fold_ptr = w + I.off_fold_ptr; v.fold_occ = w + I.off_fold_occ;
    v.chunk_seq = w + I.off_chunk_seq;
    v.row_seg = w + I.off_row_seg; v.seg_row0 = w + I.off_seg_row0; v.seg_len = w + I.off_seg_len;
    v.conv_ctx = w + I.off_conv_ctx; v.conv_sptr = w + I.off_conv_sptr; v.conv_succ = w + I.off_conv_succ;
    v.n_seg = P->info.n_seg;
    v.attn_rptr = w + I.off_attn_rptr; v.attn_runs = w + I.off_attn_runs; v.attn_mptr = w + I.off_attn_mptr;
    v.attn_mask = w + I.off_attn_mask; v.attn_hp = w + I.off_attn_hp; v.attn_qt = w + I.off_attn_qt;
    v.attn_kt = w + I.off_attn_kt; v.attn_kptr = w + I.off_attn_kptr; v.attn_kq = w + I.off_attn_kq;
    v.n_qt = I.n_qt; v.n_kt = I.n_kt;
    v.n_rounds = P->info.n_rounds; v.n_seq = P->info.n_seq; v.n_states = P->info.n_states;
    v.n_roots = P->info.n_roots; v.n_fold = P->info.n_fold_rows; v.chunk = P->info.chunk;
    v.R = P->info.R; v.n_chunks = P->info.n_chunks; v.C = P->info.C; v.flags = P->info.flags;
    set_error("");
    return HARTS_OK;
}

int harts_plan_device_error(harts_plan *P, harts_stream_t stream, int32_t *code) {
    if (!P) { set_error("NULL plan"); return HARTS_EINVAL; }
    if (!P->dev) { set_error("plan not uploaded"); return HARTS_ENOPLAN; }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t host[4] = {0, 0, 0, 0};
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "sync");
    e = cudaMemcpy(host, P->view.err, sizeof(host), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read error word");
    if (code) *code = host[0];
    if (host[0] != 0) {
        const int32_t zero[4] = {0, 0, 0, 0};
        cudaMemcpy(P->view.err, zero, sizeof(zero), cudaMemcpyHostToDevice);
        set_error("device error " + std::to_string(host[0]) + " (seq " + std::to_string(host[1]) +
                  ", pos " + std::to_string(host[2]) + ")");
        return HARTS_EDEVICE;
    }
    return HARTS_OK;
}

int harts_selftest_timeout(harts_plan *P, uint32_t max_cycles, harts_stream_t stream) {
    if (!P) { set_error("NULL plan"); return HARTS_EINVAL; }
    if (!P->dev) { set_error("plan not uploaded"); return HARTS_ENOPLAN; }
    if (max_cycles == 0 || max_cycles > 100000000u) { set_error("max_cycles must be in 1 .. 1e8"); return HARTS_EINVAL; }
    selftest_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(P->view, max_cycles);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    set_error("");
    return HARTS_OK;
}

size_t harts_kda_chunk_state_bytes(const harts_plan *P, int32_t H, int32_t dk, int32_t dv,
                                   int32_t dtype) {
    if (!P || H < 1 || dk < 1 || dv < 1) return 0;
    const size_t B = static_cast<size_t>(P->info.chunk);
    return size_t(P->info.n_chunks) * H * (size_t(dk) * dv + B * B) * dtype_size(dtype);
}

size_t harts_kda_bwd_workspace_bytes(const harts_plan *P, int32_t H, int32_t dk, int32_t dv) {
    if (!P || H < 1 || dk < 1 || dk != dv) return 0;
    return bwd_ws(P, H, dk, true).total;
}

int harts_kda_fwd(const harts_plan *P, const harts_kda_fwd_args *a, harts_stream_t stream) {
    int rc = check_fwd_args(P, a);
    if (rc) return rc;
    if (!a->o) { set_error("NULL output o"); return HARTS_EINVAL; }
    const int BC = P->info.chunk;
    const int fam = pick(a, BC, false);
    if (fam < 0) { set_error("no kernel for this dk/dv/chunk/dtype"); return HARTS_EUNSUPPORTED; }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    FwdParams p = make_fwd(a);
    for (int32_t r = 0; r < P->info.n_rounds; ++r) {
        const int32_t base = P->round_seq_ptr[r];
        const int32_t n = (P->round_seq_ptr[r + 1] - base) * a->H;
        if (n == 0) continue;
        // plans with slots inside a chunk (no-replay) keep the kernel that emits them
        const bool inner = (P->view.flags & HARTS_PLAN_NOREPLAY) != 0;
        cudaError_t e = fam == 1 ? (inner ? tc_fwd_round(p, P->view, base, n, P->info.max_seq_chunks, st)
                                          : tc2_fwd_round(p, P->view, base, n, st))
                                 : simt_fwd_round(a->dtype, BC, p, P->view, base, n, st);
        if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    }
    set_error("");
    return HARTS_OK;
}

static int kda_bwd_phases(const harts_plan *P, const harts_kda_bwd_args *a, harts_stream_t stream,
                          bool do_state, bool do_grad) {
    if (!a) { set_error("NULL args"); return HARTS_EINVAL; }
    int rc = check_fwd_args(P, &a->fwd);
    if (rc) return rc;
    if (P->info.flags & HARTS_PLAN_NOREPLAY) {
        set_error("no-replay plans are forward only");
        return HARTS_EUNSUPPORTED;
    }
    if (!a->d_o || !a->dq || !a->dk || !a->dv || !a->dg || !a->dbeta) { set_error("NULL gradient pointer"); return HARTS_EINVAL; }
    if (!aligned16(a->d_o) || !aligned16(a->dq) || !aligned16(a->dk) || !aligned16(a->dv) || !aligned16(a->dg)) {
        set_error("d_o, dq, dk, dv and dg must be 16-byte aligned");
        return HARTS_EINVAL;
    }
    if (!a->fwd.chunk_states) { set_error("chunk_states from the forward pass are required"); return HARTS_EINVAL; }
    const int D = a->fwd.dk, H = a->fwd.H, BC = P->info.chunk;
    const int fam = pick(&a->fwd, BC, true);
    if (fam < 0) { set_error("no backward kernel for this dk/dv/chunk/dtype"); return HARTS_EUNSUPPORTED; }
    const BwdWs ws = bwd_ws(P, H, D, fam == 1);
    if (!a->workspace || a->workspace_bytes < ws.total) { set_error("workspace too small"); return HARTS_ESMALLBUF; }
    if (reinterpret_cast<uintptr_t>(a->workspace) % 256) { set_error("workspace must be 256-B aligned"); return HARTS_EINVAL; }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    BwdParams p{};
    p.f = make_fwd(&a->fwd);
    p.d_o = a->d_o; p.d_final = a->d_final;
    p.dq = a->dq; p.dk = a->dk; p.dv = a->dv; p.dg = a->dg; p.dbeta = a->dbeta; p.dh0 = a->dh0;
    char *w = static_cast<char *>(a->workspace);
    p.ds_init = reinterpret_cast<float *>(w + ws.ds_init);
    p.rep_grad = reinterpret_cast<float *>(w + ws.rep_grad);
    p.dchunk = fam == 1 ? static_cast<void *>(w + ws.dchunk) : nullptr;
    if (do_state) {
        for (int32_t r = P->info.n_rounds - 1; r >= 0; --r) {
            const int32_t base = P->round_seq_ptr[r];
            const int32_t n = (P->round_seq_ptr[r + 1] - base) * H;
            if (n == 0) continue;
            cudaError_t e = fam == 1 ? tc2_bwd_state_round(p, P->view, base, n, st)
                                     : simt_bwd_round(a->fwd.dtype, BC, p, P->view, base, n, st);
            if (e != cudaSuccess) return cuda_fail(e, "backward launch");
        }
    }
    if (do_grad) {
        if (fam == 1) {
            // every chunk's gradients at once: they only depend on saved per-chunk states
            const int64_t items = P->info.n_chunks * H;
            if (items > 0x7fffffff) { set_error("too many (chunk, head) items"); return HARTS_EOVERFLOW; }
            cudaError_t e = tc2_bwd_grad(p, P->view, 0, static_cast<int32_t>(items), st);
            if (e != cudaSuccess) return cuda_fail(e, "backward gradient launch");
        }
        cudaError_t e = bwd_finish(a->fwd.dtype, p, P->view, st);
        if (e != cudaSuccess) return cuda_fail(e, "backward reductions");
    }
    set_error("");
    return HARTS_OK;
}

int harts_kda_bwd(const harts_plan *P, const harts_kda_bwd_args *a, harts_stream_t stream) {
    return kda_bwd_phases(P, a, stream, true, true);
}

int harts_kda_bwd_state(const harts_plan *P, const harts_kda_bwd_args *a, harts_stream_t stream) {
    return kda_bwd_phases(P, a, stream, true, false);
}

int harts_kda_bwd_grad(const harts_plan *P, const harts_kda_bwd_args *a, harts_stream_t stream) {
    return kda_bwd_phases(P, a, stream, false, true);
}

}  // extern "C"

// ---- backward without caller-provided device memory ------------------------------------
// Some callers cannot hand this library any device memory of its own: a plugin running
// inside a host framework that owns the whole device pool through its own allocator and
// gives third-party code no allocation hook, or a step loop that must not pay for (or
// synchronise on) an allocation.  For them the backward pass can run on scratch that the
// library carries as a file-scope device array, sized once at load time.
namespace {
constexpr size_t kStaticScratchBytes = size_t(32) << 20;   // 32 MiB per device
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
std::mutex g_static_mu;
constexpr int kMaxDevices = 64;
void *g_static_addr[kMaxDevices] = {};   // device address of the array, per device id
}  // namespace

extern "C" {

size_t harts_kda_bwd_static_max_bytes(void) { return kStaticScratchBytes; }

int harts_kda_bwd_static(const harts_plan *P, const harts_kda_bwd_args *args, harts_stream_t stream) {
    if (!args) { set_error("NULL args"); return HARTS_EINVAL; }
    int rc = check_fwd_args(P, &args->fwd);
    if (rc) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) { set_error("device id out of range"); return HARTS_EINVAL; }
    void *scratch = nullptr;
    {
        // First call on this device: look up the array's device address (the host-side
        // symbol is only a stand-in).  Done with the device current; no allocation.
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (!g_static_addr[dev]) {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_static_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
            g_static_addr[dev] = ptr;
        }
        scratch = g_static_addr[dev];
    }
    const int fam = pick(&args->fwd, P->info.chunk, true);
    if (fam < 0) { set_error("no backward kernel for this dk/dv/chunk/dtype"); return HARTS_EUNSUPPORTED; }
    const size_t need = bwd_ws(P, args->fwd.H, args->fwd.dk, fam == 1).total;
    if (need > kStaticScratchBytes) {
        set_error("backward needs " + std::to_string(need) + " bytes of scratch; the static scratch holds " +
                  std::to_string(kStaticScratchBytes) + " (use harts_kda_bwd with a workspace)");
        return HARTS_ESMALLBUF;
    }
    harts_kda_bwd_args a = *args;
    a.workspace = scratch;
    a.workspace_bytes = kStaticScratchBytes;
    return kda_bwd_phases(P, &a, stream, true, true);
}

}  // extern "C"
