// Internal plan representation shared by the host planner and the kernel launchers.
#pragma once
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/harts.h"

namespace harts {

// Device view of an uploaded plan: pointers into one int32 image.
constexpr int kConvMaxW = 8;       // widest short convolution the plan tables serve
constexpr int kAttnTile = 128;     // query / key rows per branch-attention tile
constexpr int64_t kAttnMaxRows = int64_t(1) << 27;   // largest ancestor-row table built

struct PlanDev {
    int32_t *err;                // [4] device error word: code, info, info, info
    const int32_t *round_seq_ptr;  // [n_rounds+1]
    const int32_t *round_order;    // [n_seq] per round, sequences longest first
    const int32_t *seq_row0;       // [n_seq] first own compact row
    const int32_t *seq_nown;       // [n_seq] own rows
    const int32_t *seq_rho;        // [n_seq] replay rows
    const int32_t *seq_rptr;       // [n_seq] start in replay_idx
    const int32_t *seq_src;        // [n_seq] slot id, or -1-root
    const int32_t *seq_sptr;       // [n_seq+1] slots produced by the sequence
    const int32_t *state_lpos;     // [n_states] local position of the slot
    const int32_t *seq_cbase;      // [n_seq] first chunk index of the sequence
    const int32_t *state_cptr;     // [n_states+1]
    const int32_t *state_cons;     // consumers of each slot, ascending
    const int32_t *root_cptr;      // [n_roots+1]
    const int32_t *root_cons;      // sequences starting from root r, ascending
    const int32_t *replay_idx;     // [R]
    const int32_t *fold_rows;      // [n_fold] distinct replayed rows, ascending
    const int32_t *fold_ptr;       // [n_fold+1]
    const int32_t *fold_occ;       // [R] replay occurrence ids grouped by row
    const int32_t *chunk_seq;      // [n_chunks] sequence of every chunk
    // short-convolution context (widths up to kConvMaxW)
    const int32_t *row_seg;        // [C] segment of every compact row
    const int32_t *seg_row0;       // [n_seg] first compact row of every segment
    const int32_t *seg_len;        // [n_seg]
    const int32_t *conv_ctx;       // [n_seg][kConvMaxW-1] rows 1..7 positions before the segment, -1 past the root
    const int32_t *conv_sptr;      // [n_seg*(kConvMaxW-1)+1] successor lists of (segment end, lag e+1)
    const int32_t *conv_succ;      // rows e+1 positions after the segment's end, on every branch
    // branch attention: each sequence's ancestor prefix, and the query tiles
    const int32_t *attn_rptr;      // [n_seq+1] runs of sequence i: attn_runs[3 * rptr[i] ..], own run last
    const int32_t *attn_runs;      // (padded view start, first compact row, rows); starts are multiples of 8
    const int32_t *attn_mptr;      // [n_seq+1] validity words of sequence i's padded ancestor part
    const int32_t *attn_mask;      // bit t of word t / 32: padded position t holds a real row
    const int32_t *attn_hp;        // [n_seq] padded ancestor length (start of the own run)
    const int32_t *attn_qt;        // [n_qt][2] (sequence, query tile), tree by tree
    const int32_t *attn_kt;        // [n_kt][2] (sequence, key tile of its own rows), tree by tree
    const int32_t *attn_kptr;      // [n_kt+1] query tiles of key tile j: attn_kq[3 * kptr[j] ..]
    const int32_t *attn_kq;        // (sequence, query tile, f): f own rows of the key's sequence visible, -1 causal
    int32_t n_qt, n_kt;
    int32_t n_rounds, n_seq, n_states, n_roots, n_fold, chunk, n_seg;
    uint32_t flags;                // harts_plan_calls flags (HARTS_PLAN_NOREPLAY: slots inside chunks)
    int64_t R, n_chunks, C;
};

// Word offsets of each table inside the device image.
struct PlanImage {
    std::vector<int32_t> words;
    int64_t off_err, off_round_seq_ptr, off_round_order, off_seq_row0, off_seq_nown,
        off_seq_rho, off_seq_rptr, off_seq_src, off_seq_sptr, off_state_lpos, off_seq_cbase,
        off_state_cptr, off_state_cons, off_root_cptr, off_root_cons, off_replay_idx,
        off_fold_rows, off_fold_ptr, off_fold_occ, off_chunk_seq, off_row_seg, off_seg_row0,
        off_seg_len, off_conv_ctx, off_conv_sptr, off_conv_succ, off_attn_rptr, off_attn_runs,
        off_attn_mptr, off_attn_mask, off_attn_hp, off_attn_qt, off_attn_kt, off_attn_kptr, off_attn_kq;
    int32_t n_qt, n_kt;
};

void set_error(const std::string &msg);

}  // namespace harts

struct harts_plan {
    harts_plan_info info{};
    std::vector<int32_t> parent;
    std::vector<int64_t> seg_len, seg_offset, seg_pos;
    std::vector<int32_t> seg_seq, seg_ctop, seg_tpre, seg_tin;
    std::vector<int32_t> round_seq_ptr;
    std::vector<int64_t> cu_seqlens;
    std::vector<int32_t> seq_round, seq_first_seg, seq_replay, seq_src;
    std::vector<int64_t> seq_anchor, replay_ptr, replay_idx;
    std::vector<int32_t> seq_state_ptr, state_seq;
    std::vector<int64_t> state_pos;
    std::vector<int32_t> state_cons_ptr, state_cons, root_cons_ptr, root_cons;
    std::vector<int32_t> seq_nchunks;
    harts::PlanImage image;
    bool attn_ok = false;          // the image holds the branch-attention tables
    void *dev = nullptr;           // uploaded image (caller-owned)
    harts::PlanDev view{};         // valid once uploaded
};
