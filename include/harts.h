/*
 * harts.h - C ABI of the packed-tree KDA library (GB300, sm_103a).
 *
 * The library runs chunkwise gated-delta (KDA-style) linear attention, forward and
 * backward, once over a prefix-compressed rollout tree instead of once per
 * root-to-leaf trajectory, as HARTS describes it (arXiv 2608.28158; page
 * "HARTS ... 精读", sections 4.2-4.3; page "thelatestinai ... 2608.28158", Fig. 1(c),
 * Fig. 2 and Figure C.1 captions).
 *
 * Model of one layer.  Per trajectory and head, with per-channel log-decay g_t,
 *     S_t = (I - beta_t k_t k_t^T) diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 * computed chunkwise with chunk length B (chunks anchored at trajectory position 0).
 *
 * Conventions for every call below:
 *  - Return 0 on success, or a negative HARTS_E* code; harts_last_error() then holds
 *    a message for the calling thread.  No C++ exception crosses the ABI.
 *  - "device pointer" = memory on the current CUDA device, allocated and owned by the
 *    caller.  The library never allocates device memory and never frees caller memory.
 *  - Work is enqueued on the given stream and returns without synchronising.  Faults
 *    found by the kernels (a bad plan, out-of-range decay) are recorded in the plan's
 *    device error word; harts_plan_device_error() reads it (it synchronises).
 *  - All tensors are contiguous, token-major: [rows, H, d].  Rows are compact tokens
 *    in the plan's layout (see harts_plan_arrays.seg_offset).
 *  - A plan is immutable once built; the forward and the backward pass reuse the same
 *    plan (activation recomputation re-runs the same rounds, replays and handoffs,
 *    section 4.3).  Distinct plans may be used from distinct threads.
 */
#ifndef HARTS_H
#define HARTS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HARTS_OK            0
#define HARTS_EINVAL       -1   /* malformed argument (tree, pointer, size) */
#define HARTS_EUNSUPPORTED -2   /* chunk/head dim/dtype combination without a kernel */
#define HARTS_EOVERFLOW    -3   /* a size or index does not fit the library's types */
#define HARTS_ESMALLBUF    -4   /* caller buffer smaller than required */
#define HARTS_ECUDA        -5   /* a CUDA runtime call failed */
#define HARTS_ETIMEOUT     -6   /* a bounded device wait ran out */
#define HARTS_EDEVICE      -7   /* a kernel recorded an error in the device error word */
#define HARTS_ENOPLAN      -8   /* plan not uploaded to the device */

typedef enum { HARTS_FP32 = 0, HARTS_BF16 = 1 } harts_dtype;

/* Kernel selection.  AUTO picks the tensor-core kernels where they exist
 * (bf16, dk = dv = 128, B = 64) and the exact fp32 CUDA-core kernels otherwise. */
typedef enum { HARTS_KERNEL_AUTO = 0, HARTS_KERNEL_SIMT = 1, HARTS_KERNEL_TC = 2 } harts_kernel;

typedef struct CUstream_st *harts_stream_t;   /* same type as cudaStream_t */
typedef struct harts_plan harts_plan;          /* opaque, host memory, library-owned */

/* ------------------------------------------------------------------------------ */
/* Planning (host only).                                                          */
/* ------------------------------------------------------------------------------ */

/*
 * harts_plan_calls - minimum-call plan over a segment forest (section 4.2).
 *
 * n_seg    number of segments (fork-free token paths), >= 1.
 * parent   host [n_seg]: parent[i] < i, or -1 for a root (forests allowed).
 * seg_len  host [n_seg]: tokens per segment, >= 1.
 * chunk    chunk length B >= 1 (the kernels support 16, 32, 64).
 * flags    0: the minimum-call plan below.  HARTS_PLAN_NODEWISE: the node-wise
 *          baseline the pages compare against (one call per tree level; section 5,
 *          Fig. 4 "Node-wise LA"): every segment is its own sequence, starting one
 *          round after its parent from the parent sequence's end state (a slot at
 *          that sequence's end), with its own chunk grid and no replay.
 *          HARTS_PLAN_NOREPLAY: the pages' no-replay comparison (section 5.3, Fig. 5):
 *          the continuations of the minimum-call plan, but every side branch starts
 *          one round after its producer from the producer's exact state at the fork
 *          position e_v (usually inside a chunk), with its own chunk grid and no
 *          replay; forward only (harts_kda_bwd returns HARTS_EUNSUPPORTED).
 *          Both bits, or any other bit: HARTS_EINVAL.
 * out      receives a new plan; free it with harts_plan_free.
 *
 * The plan holds: the rounds (one packed call each; their number is the minimum
 * under the packed chunkwise-call model, T_pre/T_in recurrence with a
 * max/second-max pass, linear time), the input sequences per round, the compact
 * layout, each side branch's resume anchor a(p) = B*floor(p/B) and replay rows
 * [a(p), p), and the boundary-state slots with their consumers.  Conventions that
 * make the plan unique: the continuation is the lowest-id child of maximal T_pre;
 * rounds are as early as possible; sequences are ordered by round, then by the id
 * of their first segment; slots by producer sequence, then position.
 * Errors: HARTS_EINVAL (bad parent order, zero length, chunk < 1),
 *         HARTS_EOVERFLOW (token counts beyond int32 rows).
 */
int harts_plan_calls(int32_t n_seg, const int32_t *parent, const int64_t *seg_len,
                     int32_t chunk, uint32_t flags, harts_plan **out);

#define HARTS_PLAN_NODEWISE 1u   /* harts_plan_calls flag: one sequence per segment */
#define HARTS_PLAN_NOREPLAY 2u   /* harts_plan_calls flag: exact-position handoffs, no replay */

typedef struct {
    int32_t n_seg, n_roots, n_leaves, chunk;
    int32_t n_rounds;        /* packed calls per pass */
    int32_t n_seq;           /* input sequences (= leaves) */
    int32_t n_states;        /* materialised boundary-state slots */
    int32_t n_cons;          /* sequences that start from a slot */
    int64_t C;               /* compact (non-replay) tokens */
    int64_t S;               /* expanded trajectory tokens */
    int64_t R;               /* replay tokens, sum of (|children|-1)*(e_v mod B) */
    int64_t n_chunks;        /* chunks over all sequences, replay rows included */
    int32_t max_seq_chunks;  /* longest sequence in chunks */
    int32_t n_fold_rows;     /* distinct compact rows that are replayed */
    uint32_t flags;          /* the harts_plan_calls flags the plan was built with */
} harts_plan_info;

int harts_plan_get_info(const harts_plan *plan, harts_plan_info *out);

/* Plan arrays, exported into caller-allocated host arrays sized from the info.
 * Any pointer may be NULL to skip that array. */
typedef struct {
    int64_t *seg_offset;     /* [n_seg]   compact row of the segment's first token     */
    int64_t *seg_pos;        /* [n_seg]   trajectory position s_v of that token         */
    int32_t *seg_seq;        /* [n_seg]   sequence that executes the segment            */
    int32_t *seg_ctop;       /* [n_seg]   direct-continuation child, -1 for a leaf      */
    int32_t *seg_tpre;       /* [n_seg]   T_pre(v)                                      */
    int32_t *seg_tin;        /* [n_seg]   T_in(v)                                       */
    int32_t *round_seq_ptr;  /* [n_rounds+1] sequences of round r: [ptr[r], ptr[r+1])   */
    int64_t *cu_seqlens;     /* [n_seq+1] own (non-replay) rows of sequence i           */
    int32_t *seq_round;      /* [n_seq]   1-based round                                  */
    int32_t *seq_first_seg;  /* [n_seq]                                                  */
    int64_t *seq_anchor;     /* [n_seq]   trajectory position of local position 0       */
    int32_t *seq_replay;     /* [n_seq]   replay rows rho < B before the own rows        */
    int32_t *seq_src;        /* [n_seq]   initial state: slot id >= 0, or -1-r = root r  */
    int64_t *replay_ptr;     /* [n_seq+1]                                               */
    int64_t *replay_idx;     /* [R]       compact rows replayed, in position order       */
    int32_t *seq_state_ptr;  /* [n_seq+1] slots produced by sequence i                   */
    int32_t *state_seq;      /* [n_states] producer sequence                             */
    int64_t *state_pos;      /* [n_states] local position (multiple of B) in producer    */
    int32_t *state_cons_ptr; /* [n_states+1]                                             */
    int32_t *state_cons;     /* [n_cons]   consumer sequences, ascending                 */
    int32_t *root_cons_ptr;  /* [n_roots+1]                                              */
    int32_t *root_cons;      /* [n_seq - n_cons] sequences starting from a root state    */
} harts_plan_arrays;

int harts_plan_export(const harts_plan *plan, harts_plan_arrays *dst);

/* Bytes of device memory the plan needs (int32 tables plus the device error word). */
size_t harts_plan_device_bytes(const harts_plan *plan);

/* Copy the plan tables into dev_buf (device pointer, >= harts_plan_device_bytes,
 * 256-byte aligned, caller-owned, kept alive while the plan is used) on `stream`.
 * Records dev_buf in the plan; clears the device error word. */
int harts_plan_upload(harts_plan *plan, void *dev_buf, size_t bytes, harts_stream_t stream);

/* Synchronise `stream`, read the device error word; 0 or HARTS_EDEVICE.  The word
 * is cleared after reading.  *code (nullable) receives the raw device code. */
int harts_plan_device_error(harts_plan *plan, harts_stream_t stream, int32_t *code);

void harts_plan_free(harts_plan *plan);

/* Self-test of the device failure path (for tests of error reporting): one thread waits on
 * a barrier that nothing completes, gives up after max_cycles SM cycles (1 .. 1e8) and
 * records device code 3 (timeout) in the plan's error word, the way every kernel of the
 * library reports a wait that ran out; harts_plan_device_error then returns HARTS_EDEVICE
 * and the context stays usable.  Never traps.  Errors: HARTS_EINVAL, HARTS_ENOPLAN,
 * HARTS_ECUDA. */
int harts_selftest_timeout(harts_plan *plan, uint32_t max_cycles, harts_stream_t stream);

/* ------------------------------------------------------------------------------ */
/* Forward: one packed call per round (section 4.3, "KDA").                       */
/* ------------------------------------------------------------------------------ */

typedef struct {
    int32_t H, dk, dv;
    int32_t dtype;           /* harts_dtype of q, k, v, g, beta, o, chunk_states */
    int32_t kernel;          /* harts_kernel */
    float scale;             /* o = scale * S^T q */
    const void *q;           /* device [C,H,dk], 16-byte aligned (so are k, v, g, o,
                                chunk_states and the backward's d_o, dq, dk, dv, dg) */
    const void *k;           /* device [C,H,dk] */
    const void *v;           /* device [C,H,dv] */
    const void *g;           /* device [C,H,dk] natural-log per-channel decay (<= 0) */
    const void *beta;        /* device [C,H] */
    void *o;                 /* device [C,H,dv] output */
    float *states;           /* device [n_states,H,dk,dv] fp32 boundary-state slots;
                                may be NULL only if n_states == 0 */
    float *final_state;      /* device [n_seq,H,dk,dv] fp32, nullable */
    const float *h0;         /* device [n_roots,H,dk,dv] fp32 root initial state, nullable
                                (NULL = zero state) */
    void *chunk_states;      /* device, nullable: per (chunk, head) a record of dk*dv + B*B
                                elements in `dtype`: the state at the chunk start stored
                                transposed ([dv][dk]) followed by the chunk's
                                T = (I + diag(beta) A)^-1 ([B][B]); saved for the backward
                                pass; records ordered [chunk][head], chunks by sequence.
                                The tensor-core kernels store the state column-scaled as
                                their products use it, S^T diag(e^m) with m the chunk's
                                reference log-decay (half the chunk's total per-channel
                                log-decay, Gamma_L / 2); the exact-fp32 kernels
                                store S^T.  A backward call must therefore select the same
                                kernel family as the forward call that wrote the records. */
} harts_kda_fwd_args;

/* Bytes for chunk_states (n_chunks * H * (dk*dv + B*B) * sizeof(dtype)). */
size_t harts_kda_chunk_state_bytes(const harts_plan *plan, int32_t H, int32_t dk, int32_t dv,
                                   int32_t dtype);

/*
 * harts_kda_fwd - forward pass over all rounds, enqueued on `stream`.
 * Round r launches one kernel over its (sequence, head) pairs.  A sequence starts
 * from the zero state (root; or h0), or from a slot written by an earlier round,
 * runs its replay rows and own rows chunk by chunk, writes o for its own rows only,
 * stores requested boundary states into their slots and its final state.
 * Errors: HARTS_EINVAL (NULL or misaligned pointers), HARTS_EUNSUPPORTED (dk, dv not in {32,64,128}, dk != dv,
 * B not in {16,32,64}), HARTS_ENOPLAN, HARTS_EOVERFLOW (C * H above 2^31 - 1),
 * HARTS_ECUDA.
 */
int harts_kda_fwd(const harts_plan *plan, const harts_kda_fwd_args *args, harts_stream_t stream);

/* ------------------------------------------------------------------------------ */
/* Backward: rounds in reverse, gradients through the state handoffs.             */
/* ------------------------------------------------------------------------------ */

typedef struct {
    harts_kda_fwd_args fwd;  /* the forward arguments; fwd.o is not read; fwd.states and
                                fwd.chunk_states must hold what harts_kda_fwd wrote */
    const void *d_o;         /* device [C,H,dv] gradient of the loss w.r.t. o */
    const float *d_final;    /* device [n_seq,H,dk,dv] fp32, nullable (zero) */
    void *dq, *dk, *dv, *dg; /* device [C,H,dk] / [C,H,dv] outputs in `dtype` */
    void *dbeta;             /* device [C,H] output in `dtype` */
    float *dh0;              /* device [n_roots,H,dk,dv] fp32, nullable */
    void *workspace;         /* device, >= harts_kda_bwd_workspace_bytes, 256-B aligned */
    size_t workspace_bytes;
} harts_kda_bwd_args;

size_t harts_kda_bwd_workspace_bytes(const harts_plan *plan, int32_t H, int32_t dk, int32_t dv);

/*
 * harts_kda_bwd - backward pass, enqueued on `stream`.
 * Rounds run in reverse.  Per (sequence, head) a reverse chunk loop carries dS; at a
 * slot the sequence produced, the gradients w.r.t. that slot from all its consumers
 * (sequences of later rounds) are added in ascending consumer order; the gradient
 * w.r.t. the sequence's own initial state is stored for its producer (section 4.3:
 * the initial-state gradient flows back into the call that produced the boundary).
 * Replay rows get no dq; their dk, dv, dg, dbeta are added into the ancestor rows
 * in a fixed order after all rounds.  Deterministic: no floating-point atomics.
 * Errors: as harts_kda_fwd, plus HARTS_ESMALLBUF.
 */
int harts_kda_bwd(const harts_plan *plan, const harts_kda_bwd_args *args, harts_stream_t stream);

/*
 * The backward pass in its two phases; harts_kda_bwd is harts_kda_bwd_state followed by
 * harts_kda_bwd_grad with the same arguments (same workspace, same stream order).
 *  - state: rounds in reverse, one launch per round; carries dL/dS through every
 *    sequence and its handoffs; stores each sequence's initial-state gradient and (on
 *    the tensor-core path) the carried gradient at every chunk end in the workspace.
 *    On the exact fp32 path this phase also forms all input gradients.
 *  - grad:  on the tensor-core path one launch over every (chunk, head), forming dq, dk,
 *    dv, dg, dbeta from the saved chunk states; then the deterministic fold of replay-row
 *    gradients into ancestor rows and dh0.
 * Errors: as harts_kda_bwd.
 */
int harts_kda_bwd_state(const harts_plan *plan, const harts_kda_bwd_args *args, harts_stream_t stream);
int harts_kda_bwd_grad(const harts_plan *plan, const harts_kda_bwd_args *args, harts_stream_t stream);

/*
 * harts_kda_bwd_static - harts_kda_bwd without any caller-provided device memory.
 * (This entry point has no counterpart in the paper; it is a deployment convenience.)
 *
 * For callers that cannot give the library device memory of its own: plugins inside a
 * host framework that owns the device pool and offers no allocation hook, or step loops
 * that must not allocate.  The caller still passes every input and output; the scratch
 * (initial-state gradients, replay-row gradients, saved chunk-end state gradients) lives
 * in a file-scope device array of harts_kda_bwd_static_max_bytes() = 32 MiB that every
 * GPU loading the library holds until the process exits.
 *  - args->workspace and args->workspace_bytes are ignored.
 *  - The first call on a device (with that device current) looks up the array's device
 *    address; make that first call before any stream capture.  It allocates nothing and
 *    calls no allocating routine.
 *  - Every call on a device shares the one array and leaves its last contents there.
 *    Nothing in it needs to start at zero: each call writes every scratch entry before
 *    reading it.  Calls whose work overlaps on the GPU (two streams, or two host
 *    threads) race on the array; serialise them.
 * Errors: as harts_kda_bwd, plus HARTS_ESMALLBUF when the plan, heads and head size need
 * more scratch than the array holds (harts_kda_bwd_workspace_bytes tells the need).
 */
int harts_kda_bwd_static(const harts_plan *plan, const harts_kda_bwd_args *args, harts_stream_t stream);
size_t harts_kda_bwd_static_max_bytes(void);

/* ------------------------------------------------------------------------------ */
/* Causal short convolution over the compact layout.                              */
/* ------------------------------------------------------------------------------ */

/*
 * The convolution that precedes KDA in the layer (page "HARTS ... 精读", section 4.3,
 * KDA paragraph; summary page, section 4 "KDA execution"), run once per compact row:
 * the window over the previous w - 1 tokens reads the row's real ancestors on its own
 * trajectory (a temporary prefix of the parent's rows), never the neighbouring rows of
 * another packed sequence, and is zero before the trajectory start.  Depthwise:
 *   pre[r][c] = bias[c] + sum_{j<w} weight[c][w-1-j] * x[row j positions before r][c],
 *   y = pre (activation 0) or pre * sigmoid(pre) (activation 1).
 * The plan (uploaded) carries the ancestor context and the successor lists for any
 * w <= 8; any of the three plan modes works.  Deterministic (no atomics).
 */
typedef struct {
    int32_t channels;        /* ch: values per row (e.g. H * d), a multiple of 8 */
    int32_t width;           /* w: 1..8 */
    int32_t dtype;           /* harts_dtype of x, y, dy, dx */
    int32_t activation;      /* 0 none, 1 SiLU */
    const void *x;           /* device [C][ch], compact layout, 16-byte aligned */
    const float *weight;     /* device [ch][w] fp32; weight[c][w-1] multiplies the current row */
    const float *bias;       /* device [ch] fp32, or NULL */
    void *y;                 /* device [C][ch] output (forward only), 16-byte aligned */
} harts_conv_fwd_args;

/* Forward.  Errors: HARTS_EINVAL (NULL / misaligned pointer, channels not a positive
 * multiple of 8, activation), HARTS_EUNSUPPORTED (dtype, width outside 1..8),
 * HARTS_ENOPLAN, HARTS_ECUDA. */
int harts_conv_fwd(const harts_plan *plan, const harts_conv_fwd_args *args, harts_stream_t stream);

typedef struct {
    harts_conv_fwd_args fwd; /* y is not used */
    const void *dy;          /* device [C][ch] dL/dy per compact row (already summed over the
                                trajectories that share the row) */
    void *dx;                /* device [C][ch] output */
    float *dweight;          /* device [ch][w] output (overwritten) */
    float *dbias;            /* device [ch] output (overwritten), or NULL */
    void *workspace;         /* device, harts_conv_bwd_workspace_bytes, 16-byte aligned */
    size_t workspace_bytes;
} harts_conv_bwd_args;

/* Workspace of harts_conv_bwd: the per-256-row partial sums of dweight / dbias, fp32
 * [ceil(C/256)][ch][w+1].  0 for invalid arguments. */
size_t harts_conv_bwd_workspace_bytes(const harts_plan *plan, int32_t channels, int32_t width);

/* Backward: dx[r] sums weight * dL/dpre over the rows 0..w-1 positions after r on every
 * branch below it (gathered in a fixed order); dweight and dbias are reduced over rows in
 * a fixed order.  Errors as harts_conv_fwd, plus HARTS_ESMALLBUF (workspace). */
int harts_conv_bwd(const harts_plan *plan, const harts_conv_bwd_args *args, harts_stream_t stream);

/* ------------------------------------------------------------------------------ */
/* Compact-to-semantic log-probabilities.                                         */
/* ------------------------------------------------------------------------------ */

/*
 * Page "HARTS ... 精读", section 4.4 ("紧凑到语义的 log 概率"); summary page "Semantic
 * Preservation": a compact logit row is reduced over the vocabulary once (its
 * log-sum-exp), and every semantic position s -- a token occurrence of an original
 * trajectory -- reads its own target logit from the row its token maps to:
 *   logp[s] = logits[c(s)][target[s]] - lse[c(s)].
 * The backward (eq. 19) sums the independently formed gradients of a row's semantic
 * positions onto it: dlogits[c] = sum_{s -> c} dlogp[s] (onehot(target[s]) - softmax(row c)).
 * Work is O(C V) + O(S); no S x V array is formed.  Deterministic (no atomics).
 *
 * harts_plan_semantic_map fills, on the host: sem_row[S] (compact row of each semantic
 * position; trajectories in increasing leaf id, each from its root to its leaf), and the
 * positions grouped by row: row_ptr[C+1], row_sem[S] (ascending within a row).  Callers
 * with another semantic order may build these arrays themselves.
 */
int harts_plan_semantic_map(const harts_plan *plan, int32_t *sem_row, int32_t *row_ptr, int32_t *row_sem);

typedef struct {
    int64_t C;               /* compact rows */
    int32_t V;               /* vocabulary, a multiple of 8 */
    int32_t dtype;           /* harts_dtype of logits / dlogits */
    int64_t S;               /* semantic positions, < 2^31 */
    const void *logits;      /* device [C][V], 16-byte aligned */
    const int32_t *row_ptr;  /* device [C+1]: semantic positions of row c are row_sem[row_ptr[c] ..] */
    const int32_t *row_sem;  /* device [S] */
    const int32_t *target;   /* device [S] label of each semantic position, 0 <= target < V */
    float *lse;              /* device [C]: written by the forward, read by the backward */
    float *logp;             /* device [S]: written by the forward */
} harts_logprob_fwd_args;

/* Forward.  Errors: HARTS_EINVAL (NULL / misaligned pointers, V not a multiple of 8),
 * HARTS_EUNSUPPORTED (dtype), HARTS_EOVERFLOW (S), HARTS_ECUDA. */
int harts_logprob_fwd(const harts_logprob_fwd_args *args, harts_stream_t stream);

typedef struct {
    harts_logprob_fwd_args fwd;  /* lse as written by the forward; logp unused */
    const float *dlogp;          /* device [S] dL/dlogp */
    void *dlogits;               /* device [C][V] output (overwritten), 16-byte aligned */
} harts_logprob_bwd_args;

int harts_logprob_bwd(const harts_logprob_bwd_args *args, harts_stream_t stream);

/* ------------------------------------------------------------------------------ */
/* Branch attention over the compact layout (the softmax-attention layers).       */
/* ------------------------------------------------------------------------------ */

/*
 * Page "HARTS ... 精读", section 4.3 (MLA paragraph); summary page, section 4 ("MLA
 * execution"); figures page, Figure C.1(c).  Projections run once per compact row; each
 * sequence of the plan is a branch whose queries (its own rows) attend to the keys and
 * values of its ancestors and itself with bottom-right causal alignment: own query t sees
 * view entries 0 .. h + t, where h is the number of trajectory positions before the
 * sequence.  The view is gathered inside the kernel; outputs go to the unique compact
 * rows.  Per head: o = softmax(scale q k^T) v, lse = log sum_j exp(scale q k_j).
 * Equal to plain causal attention of every trajectory through a row.
 *
 * The plan's attention tables (each sequence's ancestor rows) are built when they add up
 * to at most 2^27 rows; for deeper plans the call fails with HARTS_EOVERFLOW.
 */
typedef struct {
    int32_t H;               /* heads */
    int32_t d;               /* head dimension of q, k and v: 128 */
    int32_t dtype;           /* harts_dtype of q, k, v, o: HARTS_BF16 */
    float scale;             /* softmax scale, positive and finite (typically 1/sqrt(d)) */
    const void *q, *k, *v;   /* device [C][H][d], compact layout, 16-byte aligned */
    void *o;                 /* device [C][H][d] output, 16-byte aligned */
    float *lse;              /* device [C][H] output (natural-log sum-exp of scaled scores), or NULL */
} harts_attn_fwd_args;

/* Forward.  Errors: HARTS_EINVAL (NULL / misaligned pointers, H < 1, scale not positive), HARTS_EUNSUPPORTED
 * (dtype other than bf16, d other than 128), HARTS_ENOPLAN, HARTS_EOVERFLOW (no attention
 * tables in the plan, too many blocks), HARTS_ECUDA.  A bounded wait that runs out records
 * device code 3 (timeout) in the plan's device error word (harts_plan_device_error). */
int harts_attn_fwd(const harts_plan *plan, const harts_attn_fwd_args *args, harts_stream_t stream);

/* Backward of harts_attn_fwd for L with dL/do = d_o: each compact query row counts once,
 * over its own view; keys and values collect every query that sees them, across branches.
 * With D = rowsum(d_o * o) and P recomputed from lse:
 *   dv_j = sum_t P_tj d_o_t,  dS_tj = scale P_tj (d_o_t . v_j - D_t),
 *   dq_t = sum_j dS_tj k_j,   dk_j = sum_t dS_tj q_t.
 * Sums run in a fixed order (no atomics): per query tile over its view's key tiles, per
 * key tile (128 own rows of a sequence) over the query tiles that see it, in ascending
 * (sequence, tile) order. */
typedef struct {
    harts_attn_fwd_args fwd; /* q, k, v; o and lse as written by the forward (lse required) */
    const void *d_o;         /* device [C][H][d] bf16 dL/do per compact row */
    void *dq, *dk, *dv;      /* device [C][H][d] bf16 outputs (overwritten), 16-byte aligned */
    void *workspace;         /* device, harts_attn_bwd_workspace_bytes, 16-byte aligned */
    size_t workspace_bytes;
} harts_attn_bwd_args;

/* Workspace of harts_attn_bwd: D, fp32 [C][H] (rounded up to 256 bytes); 0 for invalid
 * arguments. */
size_t harts_attn_bwd_workspace_bytes(const harts_plan *plan, int32_t H);

/* Errors as harts_attn_fwd, plus HARTS_EINVAL (NULL / misaligned lse, d_o, dq, dk, dv,
 * workspace) and HARTS_ESMALLBUF (workspace). */
int harts_attn_bwd(const harts_plan *plan, const harts_attn_bwd_args *args, harts_stream_t stream);

/* Message for the last error on the calling thread ("" if none). */
const char *harts_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* HARTS_H */
