// Host planner: minimum number of sequential packed KDA calls over a segment forest.
//
// HARTS (page "HARTS ... 精读", section 4.2): the rollout tree is contracted into
// fork-free segments.  A boundary state produced inside a packed chunkwise call can
// only initialise another input sequence after that call returns, so at each fork at
// most one child (the direct continuation) stays in the current sequence.  A side
// branch at fork end p resumes from the chunk-boundary state at a(p) = B*floor(p/B)
// and replays the ancestor tokens [a(p), p).  T_pre(v) / T_in(v) are the fewest
// rounds for v's subtree when v's entry anchor state is ready before the call /
// when v enters the call as a direct continuation; a continuation does not wait, a
// side branch waits one round -- unless the fork lies in the chunk where the current
// sequence starts, in which case the side branch can start in the same call from the
// same anchor state (Fig. 2(c): "replay-started v2" in round 1).  Linear time: one
// bottom-up pass keeping the largest and second-largest child T_pre, one top-down
// pass assigning rounds as early as possible.
#include <algorithm>
#include <array>
#include <cstring>
#include <new>

#include "plan_internal.h"

namespace harts {

thread_local std::string g_last_error;
void set_error(const std::string &msg) { g_last_error = msg; }

namespace {

constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;

int64_t floor_to(int64_t x, int64_t B) { return (x / B) * B; }

int build(harts_plan &P, int32_t n, const int32_t *parent, const int64_t *len, int32_t B, uint32_t flags) {
    const bool nodewise = (flags & HARTS_PLAN_NODEWISE) != 0, noreplay = (flags & HARTS_PLAN_NOREPLAY) != 0;
    // ---- a1: validate, positions s_v, e_v --------------------------------------
    std::vector<int64_t> s(n), e(n);
    std::vector<int32_t> nkids(n, 0);
    int64_t C = 0;
    int32_t n_roots = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t p = parent[i];
        if (p < -1 || p >= i) { set_error("parent[i] must be -1 or < i"); return HARTS_EINVAL; }
        if (len[i] < 1) { set_error("segment length must be >= 1"); return HARTS_EINVAL; }
        if (len[i] > kMaxRows) { set_error("segment too long"); return HARTS_EOVERFLOW; }
        s[i] = p < 0 ? 0 : e[p];
        e[i] = s[i] + len[i];
        if (e[i] > (int64_t(1) << 40)) { set_error("trajectory too long"); return HARTS_EOVERFLOW; }
        C += len[i];
        if (C > kMaxRows) { set_error("more than 2^31-1 compact rows"); return HARTS_EOVERFLOW; }
        if (p >= 0) nkids[p]++; else n_roots++;
    }
    // children in ascending id order (CSR)
    std::vector<int32_t> kptr(n + 1, 0), kids(std::max(n - n_roots, 0));
    for (int32_t i = 0; i < n; ++i) kptr[i + 1] = kptr[i] + nkids[i];
    {
        std::vector<int32_t> fill(kptr.begin(), kptr.end() - 1);
        for (int32_t i = 0; i < n; ++i) if (parent[i] >= 0) kids[fill[parent[i]]++] = i;
    }

    // ---- a2: bottom-up T_pre / T_in ------------------------------------------------
    std::vector<int32_t> tpre(n), tin(n), ctop(n, -1);
    for (int32_t v = n - 1; v >= 0; --v) {
        if (nkids[v] == 0) { tpre[v] = tin[v] = 1; continue; }
        int32_t best = -1, m1 = 0, m2 = 0;
        for (int32_t j = kptr[v]; j < kptr[v + 1]; ++j) {
            int32_t c = kids[j], t = tpre[c];
            if (t > m1) { m2 = m1; m1 = t; best = c; }   // ascending ids: first max wins
            else if (t > m2) m2 = t;
        }
        ctop[v] = best;
        tin[v] = std::max(tin[best], 1 + m2);
        tpre[v] = (floor_to(s[v], B) == floor_to(e[v], B)) ? m1 : tin[v];
    }

    // Node-wise mode: no segment continues its parent's sequence; every segment is a
    // sequence of its own that starts, one round after its parent, from the parent
    // sequence's end state, with its own chunk grid and nothing replayed.
    if (nodewise) std::fill(ctop.begin(), ctop.end(), -1);

    // ---- a2: top-down ASAP recovery ------------------------------------------------
    // Sequences are first identified by their first segment.  Per segment: the first
    // segment of its sequence.  Per first segment: round, anchor, source.
    struct SeqTmp { int32_t round; int64_t anchor; int32_t src_kind; int32_t src_a; int64_t src_b; };
    // src_kind 0: root (src_a = root index); 1: slot of producer first seg src_a at src_b
    std::vector<int32_t> head(n, -1);        // first segment of v's sequence
    std::vector<SeqTmp> tmp(n);
    std::vector<int32_t> root_index(n, -1);
    // temp slots discovered in segment order; per producer the last slot for dedup
    std::vector<int32_t> last_slot(n, -1);
    std::vector<int32_t> slot_prod;          // temp slot -> producer first seg
    std::vector<int64_t> slot_lpos;          // temp slot -> local position
    std::vector<int32_t> tmp_src_slot(n, -1); // first seg -> temp slot id (src_kind 1)
    {
        int32_t r = 0;
        for (int32_t v = 0; v < n; ++v) if (parent[v] < 0) root_index[v] = r++;
    }
    for (int32_t v = 0; v < n; ++v) {
        if (parent[v] < 0) {
            head[v] = v;
            tmp[v] = SeqTmp{1, 0, 0, root_index[v], 0};
        }
        const int32_t f = head[v];
        const SeqTmp &sq = tmp[f];
        for (int32_t j = kptr[v]; j < kptr[v + 1]; ++j) {
            int32_t c = kids[j];
            if (c == ctop[v]) { head[c] = f; continue; }
            head[c] = c;
            // No-replay mode: side branches resume at the exact fork position from the
            // producer's state there, so none can start in the producer's round.
            const bool exact = nodewise || noreplay;
            const int64_t a_e = exact ? e[v] : floor_to(e[v], B);
            if (!exact && a_e == sq.anchor) {
                tmp[c] = sq;
                tmp_src_slot[c] = tmp_src_slot[f];
            } else {
                const int64_t lpos = a_e - sq.anchor;
                int32_t ls = last_slot[f];
                if (ls < 0 || slot_lpos[ls] != lpos) {
                    ls = static_cast<int32_t>(slot_prod.size());
                    slot_prod.push_back(f);
                    slot_lpos.push_back(lpos);
                    last_slot[f] = ls;
                }
                tmp[c] = SeqTmp{sq.round + 1, a_e, 1, f, lpos};
                tmp_src_slot[c] = ls;
            }
        }
    }

    // ---- a3: layout order: by round, then by first segment id (bucket pass) ----------
    int32_t n_rounds = 0, n_seq = 0;
    for (int32_t v = 0; v < n; ++v) if (head[v] == v) { n_seq++; n_rounds = std::max(n_rounds, tmp[v].round); }
    std::vector<int32_t> rptr(n_rounds + 2, 0);
    for (int32_t v = 0; v < n; ++v) if (head[v] == v) rptr[tmp[v].round + 1]++;
    for (int32_t r = 1; r <= n_rounds + 1 && r < (int32_t)rptr.size(); ++r) rptr[r] += rptr[r - 1];
    std::vector<int32_t> order(n_seq), seq_of_first(n, -1);
    {
        std::vector<int32_t> fill(rptr.begin(), rptr.end());
        for (int32_t v = 0; v < n; ++v)
            if (head[v] == v) { int32_t id = fill[tmp[v].round]++; order[id] = v; seq_of_first[v] = id; }
    }

    P.info.n_seg = n; P.info.n_roots = n_roots; P.info.chunk = B;
    P.info.n_rounds = n_rounds; P.info.n_seq = n_seq;
    int32_t n_leaves = 0;
    for (int32_t v = 0; v < n; ++v) n_leaves += nkids[v] == 0;
    P.info.n_leaves = n_leaves;
    P.round_seq_ptr.assign(n_rounds + 1, 0);
    // rptr[r] = number of sequences with round < r (rounds are 1-based)
    for (int32_t r = 0; r <= n_rounds; ++r) P.round_seq_ptr[r] = rptr[r + 1];

    // compact rows: sequence order, then continuation chain
    P.seg_offset.assign(n, 0); P.seg_pos.assign(s.begin(), s.end()); P.seg_seq.assign(n, 0);
    P.cu_seqlens.assign(n_seq + 1, 0);
    int64_t row = 0;
    for (int32_t i = 0; i < n_seq; ++i) {
        P.cu_seqlens[i] = row;
        for (int32_t v = order[i]; v >= 0; v = ctop[v]) {
            P.seg_offset[v] = row;
            P.seg_seq[v] = i;
            row += len[v];
        }
    }
    P.cu_seqlens[n_seq] = row;

    // slots numbered by producer sequence, then position (temp slots of one producer
    // were discovered in increasing position along its chain)
    const int32_t n_tmp = static_cast<int32_t>(slot_prod.size());
    std::vector<int32_t> per_seq(n_seq + 1, 0);
    for (int32_t t = 0; t < n_tmp; ++t) per_seq[seq_of_first[slot_prod[t]] + 1]++;
    for (int32_t i = 0; i < n_seq; ++i) per_seq[i + 1] += per_seq[i];
    std::vector<int32_t> slot_final(n_tmp);
    P.state_seq.assign(n_tmp, 0); P.state_pos.assign(n_tmp, 0);
    {
        std::vector<int32_t> fill(per_seq.begin(), per_seq.end() - 1);
        for (int32_t t = 0; t < n_tmp; ++t) {
            int32_t sq = seq_of_first[slot_prod[t]];
            int32_t id = fill[sq]++;
            slot_final[t] = id;
            P.state_seq[id] = sq;
            P.state_pos[id] = slot_lpos[t];
        }
    }
    P.seq_state_ptr.assign(per_seq.begin(), per_seq.end());
    P.info.n_states = n_tmp;

    // per-sequence arrays, replay gather lists
    P.seq_round.assign(n_seq, 0); P.seq_first_seg.assign(n_seq, 0); P.seq_anchor.assign(n_seq, 0);
    P.seq_replay.assign(n_seq, 0); P.seq_src.assign(n_seq, 0); P.replay_ptr.assign(n_seq + 1, 0);
    P.seq_nchunks.assign(n_seq, 0);
    P.replay_idx.clear();
    std::vector<int32_t> upath;
    int32_t n_cons = 0, max_chunks = 0;
    int64_t n_chunks = 0;
    for (int32_t i = 0; i < n_seq; ++i) {
        const int32_t f = order[i];
        const SeqTmp &sq = tmp[f];
        P.seq_round[i] = sq.round;
        P.seq_first_seg[i] = f;
        P.seq_anchor[i] = sq.anchor;
        const int64_t rho = s[f] - sq.anchor;
        if (rho < 0 || rho >= B) { set_error("internal: replay out of range"); return HARTS_EINVAL; }
        P.seq_replay[i] = static_cast<int32_t>(rho);
        if (sq.src_kind == 0) P.seq_src[i] = -1 - sq.src_a;
        else { P.seq_src[i] = slot_final[tmp_src_slot[f]]; n_cons++; }
        P.replay_ptr[i] = static_cast<int64_t>(P.replay_idx.size());
        upath.clear();
        for (int32_t w = parent[f]; w >= 0 && e[w] > sq.anchor; w = parent[w]) upath.push_back(w);
        for (auto it = upath.rbegin(); it != upath.rend(); ++it) {
            const int32_t w = *it;
            for (int64_t p = std::max(s[w], sq.anchor); p < e[w]; ++p)
                P.replay_idx.push_back(P.seg_offset[w] + (p - s[w]));
        }
        if (static_cast<int64_t>(P.replay_idx.size()) - P.replay_ptr[i] != rho) {
            set_error("internal: replay gather length mismatch"); return HARTS_EINVAL;
        }
        const int64_t L = rho + (P.cu_seqlens[i + 1] - P.cu_seqlens[i]);
        const int64_t nc = (L + B - 1) / B;
        P.seq_nchunks[i] = static_cast<int32_t>(nc);
        max_chunks = std::max<int32_t>(max_chunks, static_cast<int32_t>(nc));
        n_chunks += nc;
    }
    P.replay_ptr[n_seq] = static_cast<int64_t>(P.replay_idx.size());
    P.info.n_cons = n_cons;
    P.info.C = C;
    P.info.R = static_cast<int64_t>(P.replay_idx.size());
    P.info.n_chunks = n_chunks;
    P.info.max_seq_chunks = max_chunks;
    if (n_chunks > kMaxRows || P.info.R > kMaxRows) { set_error("too many chunks"); return HARTS_EOVERFLOW; }

    // expanded size S = sum_v len_v * leaves under v
    {
        std::vector<int64_t> lv(n, 0);
        int64_t S = 0;
        for (int32_t v = n - 1; v >= 0; --v) {
            if (nkids[v] == 0) lv[v] += 1;
            S += len[v] * lv[v];
            if (parent[v] >= 0) lv[parent[v]] += lv[v];
        }
        P.info.S = S;
    }

    // consumers of every slot and root, ascending sequence id (counting sort)
    P.state_cons_ptr.assign(n_tmp + 1, 0);
    P.root_cons_ptr.assign(n_roots + 1, 0);
    for (int32_t i = 0; i < n_seq; ++i) {
        if (P.seq_src[i] >= 0) P.state_cons_ptr[P.seq_src[i] + 1]++;
        else P.root_cons_ptr[-1 - P.seq_src[i] + 1]++;
    }
    for (int32_t j = 0; j < n_tmp; ++j) P.state_cons_ptr[j + 1] += P.state_cons_ptr[j];
    for (int32_t j = 0; j < n_roots; ++j) P.root_cons_ptr[j + 1] += P.root_cons_ptr[j];
    P.state_cons.assign(n_cons, 0);
    P.root_cons.assign(n_seq - n_cons, 0);
    {
        std::vector<int32_t> fs(P.state_cons_ptr.begin(), P.state_cons_ptr.end() - 1);
        std::vector<int32_t> fr(P.root_cons_ptr.begin(), P.root_cons_ptr.end() - 1);
        for (int32_t i = 0; i < n_seq; ++i) {
            if (P.seq_src[i] >= 0) P.state_cons[fs[P.seq_src[i]]++] = i;
            else P.root_cons[fr[-1 - P.seq_src[i]]++] = i;
        }
    }

    P.seg_ctop = ctop; P.seg_tpre = tpre; P.seg_tin = tin;
    P.parent.assign(parent, parent + n);
    P.seg_len.assign(len, len + n);
    P.info.flags = flags;
    return HARTS_OK;
}

void build_image(harts_plan &P) {
    auto &I = P.image;
    auto &w = I.words;
    w.clear();
    auto put = [&](int64_t &off, const int32_t *src, size_t cnt) {
        // 16-byte aligned tables
        while (w.size() % 4) w.push_back(0);
        off = static_cast<int64_t>(w.size());
        w.insert(w.end(), src, src + cnt);
    };
    const int32_t n_seq = P.info.n_seq, n_st = P.info.n_states, n_rounds = P.info.n_rounds;
    int32_t zero4[4] = {0, 0, 0, 0};
    put(I.off_err, zero4, 4);
    put(I.off_round_seq_ptr, P.round_seq_ptr.data(), n_rounds + 1);
    // per round: longest sequence first (ties: lower id first)
    std::vector<int32_t> ord(n_seq);
    for (int32_t i = 0; i < n_seq; ++i) ord[i] = i;
    for (int32_t r = 0; r < n_rounds; ++r)
        std::stable_sort(ord.begin() + P.round_seq_ptr[r], ord.begin() + P.round_seq_ptr[r + 1],
                         [&](int32_t a, int32_t b) { return P.seq_nchunks[a] > P.seq_nchunks[b]; });
    put(I.off_round_order, ord.data(), n_seq);
    std::vector<int32_t> t(n_seq);
    for (int32_t i = 0; i < n_seq; ++i) t[i] = static_cast<int32_t>(P.cu_seqlens[i]);
    put(I.off_seq_row0, t.data(), n_seq);
    for (int32_t i = 0; i < n_seq; ++i) t[i] = static_cast<int32_t>(P.cu_seqlens[i + 1] - P.cu_seqlens[i]);
    put(I.off_seq_nown, t.data(), n_seq);
    put(I.off_seq_rho, P.seq_replay.data(), n_seq);
    for (int32_t i = 0; i < n_seq; ++i) t[i] = static_cast<int32_t>(P.replay_ptr[i]);
    put(I.off_seq_rptr, t.data(), n_seq);
    put(I.off_seq_src, P.seq_src.data(), n_seq);
    put(I.off_seq_sptr, P.seq_state_ptr.data(), n_seq + 1);
    std::vector<int32_t> lp(n_st);
    for (int32_t j = 0; j < n_st; ++j) lp[j] = static_cast<int32_t>(P.state_pos[j]);
    put(I.off_state_lpos, lp.data(), n_st);
    int64_t cb = 0;
    for (int32_t i = 0; i < n_seq; ++i) { t[i] = static_cast<int32_t>(cb); cb += P.seq_nchunks[i]; }
    put(I.off_seq_cbase, t.data(), n_seq);
    put(I.off_state_cptr, P.state_cons_ptr.data(), n_st + 1);
    put(I.off_state_cons, P.state_cons.data(), P.state_cons.size());
    put(I.off_root_cptr, P.root_cons_ptr.data(), P.info.n_roots + 1);
    put(I.off_root_cons, P.root_cons.data(), P.root_cons.size());
    const int64_t R = P.info.R;
    std::vector<int32_t> ri(R);
    for (int64_t j = 0; j < R; ++j) ri[j] = static_cast<int32_t>(P.replay_idx[j]);
    put(I.off_replay_idx, ri.data(), R);
    // fold lists: replay occurrences grouped by compact row (stable counting sort)
    std::vector<int32_t> occ(R);
    for (int64_t j = 0; j < R; ++j) occ[j] = static_cast<int32_t>(j);
    std::stable_sort(occ.begin(), occ.end(), [&](int32_t a, int32_t b) { return ri[a] < ri[b]; });
    std::vector<int32_t> frows, fptr;
    for (int64_t j = 0; j < R; ++j) {
        if (j == 0 || ri[occ[j]] != ri[occ[j - 1]]) { frows.push_back(ri[occ[j]]); fptr.push_back(static_cast<int32_t>(j)); }
    }
    fptr.push_back(static_cast<int32_t>(R));
    P.info.n_fold_rows = static_cast<int32_t>(frows.size());
    put(I.off_fold_rows, frows.data(), frows.size());
    put(I.off_fold_ptr, fptr.data(), fptr.size());
    put(I.off_fold_occ, occ.data(), R);
    std::vector<int32_t> cseq;
    cseq.reserve(static_cast<size_t>(P.info.n_chunks));
    for (int32_t i = 0; i < n_seq; ++i)
        for (int32_t c = 0; c < P.seq_nchunks[i]; ++c) cseq.push_back(i);
    put(I.off_chunk_seq, cseq.data(), cseq.size());

    // ---- short-convolution context ----------------------------------------------------
    // A compact row's window reaches back along its own trajectory, into its ancestors'
    // last rows; a row feeds the next rows on every branch below it.
    const int32_t n = P.info.n_seg;
    constexpr int K = kConvMaxW - 1;
    std::vector<int32_t> rseg(static_cast<size_t>(P.info.C)), srow0(n), slen(n);
    for (int32_t v = 0; v < n; ++v) {
        srow0[v] = static_cast<int32_t>(P.seg_offset[v]);
        slen[v] = static_cast<int32_t>(P.seg_len[v]);
        for (int64_t r = P.seg_offset[v]; r < P.seg_offset[v] + P.seg_len[v]; ++r) rseg[r] = v;
    }
    std::vector<int32_t> ctx(static_cast<size_t>(n) * K, -1);
    for (int32_t v = 0; v < n; ++v) {
        int k = 0;
        for (int32_t u = P.parent[v]; u >= 0 && k < K; u = P.parent[u])
            for (int64_t t = P.seg_len[u] - 1; t >= 0 && k < K; --t)
                ctx[static_cast<size_t>(v) * K + k++] = static_cast<int32_t>(P.seg_offset[u] + t);
    }
    std::vector<int32_t> kptr(n + 1, 0), kids;
    for (int32_t v = 0; v < n; ++v) if (P.parent[v] >= 0) kptr[P.parent[v] + 1]++;
    for (int32_t v = 0; v < n; ++v) kptr[v + 1] += kptr[v];
    kids.assign(kptr[n], 0);
    {
        std::vector<int32_t> fill(kptr.begin(), kptr.end() - 1);
        for (int32_t v = 0; v < n; ++v) if (P.parent[v] >= 0) kids[fill[P.parent[v]]++] = v;
    }
    std::vector<int32_t> sptr(static_cast<size_t>(n) * K + 1, 0), succ;
    // rows e positions into the subtrees below v's end (children in increasing id)
    std::vector<std::pair<int32_t, int64_t>> stack;
    for (int32_t v = 0; v < n; ++v)
        for (int e = 0; e < K; ++e) {
            sptr[static_cast<size_t>(v) * K + e] = static_cast<int32_t>(succ.size());
            stack.clear();
            for (int32_t j = kptr[v + 1] - 1; j >= kptr[v]; --j) stack.push_back({kids[j], e});
            while (!stack.empty()) {
                auto [c, off] = stack.back();
                stack.pop_back();
                if (off < P.seg_len[c]) { succ.push_back(static_cast<int32_t>(P.seg_offset[c] + off)); continue; }
                for (int32_t j = kptr[c + 1] - 1; j >= kptr[c]; --j) stack.push_back({kids[j], off - P.seg_len[c]});
            }
        }
    sptr[static_cast<size_t>(n) * K] = static_cast<int32_t>(succ.size());
    put(I.off_row_seg, rseg.data(), rseg.size());
    put(I.off_seg_row0, srow0.data(), n);
    put(I.off_seg_len, slen.data(), n);
    put(I.off_conv_ctx, ctx.data(), ctx.size());
    put(I.off_conv_sptr, sptr.data(), sptr.size());
    put(I.off_conv_succ, succ.data(), succ.size());

    // ---- branch attention -------------------------------------------------------------
    // A sequence's view: the trajectory positions before its first own token (ancestor
    // segments, root first), then its own rows.  In the kernels' padded view every
    // segment's run starts at a multiple of 8 positions (up to 7 pad positions after
    // each ancestor run), so each 8-row group of a key tile is 8 consecutive compact rows
    // and moves by one tiled TMA box; a bitmask marks the real positions of the ancestor
    // part.  Runs: (padded start, first compact row, rows), the own run last at hp, the
    // padded ancestor length.  Query tiles of kAttnTile own rows, grouped by tree (so
    // the blocks that read a tree's keys and values run together and find them in L2),
    // trees in decreasing order of their longest tile, within a tree by decreasing work
    // (padded view length up to the tile's end).
    // The key-tile lists below grow with sum_i (first position of sequence i), quadratic
    // in the depth of chain-like trees: above kAttnMaxRows the plan carries no attention
    // tables.
    int64_t sum_h = 0;
    for (int32_t i = 0; i < n_seq; ++i) sum_h += P.seg_pos[P.seq_first_seg[i]];
    P.attn_ok = sum_h <= kAttnMaxRows;
    std::vector<int32_t> rptr(n_seq + 1, 0), runs, mptr(n_seq + 1, 0), vmask, hp(n_seq, 0);
    std::vector<int32_t> chain;
    for (int32_t i = 0; i < n_seq && P.attn_ok; ++i) {
        rptr[i] = static_cast<int32_t>(runs.size() / 3);
        chain.clear();
        for (int32_t u = P.parent[P.seq_first_seg[i]]; u >= 0; u = P.parent[u]) chain.push_back(u);
        int64_t ps = 0;
        std::vector<std::pair<int64_t, int64_t>> real;    // (padded start, rows)
        for (auto it = chain.rbegin(); it != chain.rend(); ++it) {
            runs.insert(runs.end(), {static_cast<int32_t>(ps), static_cast<int32_t>(P.seg_offset[*it]),
                                     static_cast<int32_t>(P.seg_len[*it])});
            real.push_back({ps, P.seg_len[*it]});
            ps += (P.seg_len[*it] + 7) / 8 * 8;
        }
        hp[i] = static_cast<int32_t>(ps);
        const int64_t own = P.cu_seqlens[i + 1] - P.cu_seqlens[i];
        runs.insert(runs.end(), {static_cast<int32_t>(ps), static_cast<int32_t>(P.seg_offset[P.seq_first_seg[i]]),
                                 static_cast<int32_t>(own)});
        mptr[i] = static_cast<int32_t>(vmask.size());
        const size_t w0 = vmask.size();
        vmask.resize(w0 + (ps + 31) / 32, 0);
        for (const auto &r : real)
            for (int64_t t = r.first; t < r.first + r.second; ++t)
                vmask[w0 + t / 32] |= static_cast<int32_t>(1u << (t % 32));
    }
    rptr[n_seq] = static_cast<int32_t>(runs.size() / 3);
    mptr[n_seq] = static_cast<int32_t>(vmask.size());
    struct QTile { int64_t work; int32_t tree, seq, tile; };
    std::vector<QTile> qts;
    std::vector<int32_t> root(P.parent.size());
    for (size_t v = 0; v < P.parent.size(); ++v) root[v] = P.parent[v] < 0 ? static_cast<int32_t>(v) : root[P.parent[v]];
    std::vector<int64_t> tree_work(P.parent.size(), 0);
    for (int32_t i = 0; i < n_seq && P.attn_ok; ++i) {
        const int64_t own = P.cu_seqlens[i + 1] - P.cu_seqlens[i], hh = hp[i];
        const int32_t r = root[P.seq_first_seg[i]];
        for (int64_t t = 0; t * kAttnTile < own; ++t) {
            const int64_t w = hh + std::min(own, (t + 1) * kAttnTile);
            qts.push_back({w, r, i, static_cast<int32_t>(t)});
            tree_work[r] = std::max(tree_work[r], w);
        }
    }
    std::stable_sort(qts.begin(), qts.end(), [&](const QTile &a, const QTile &b) {
        if (a.tree != b.tree) {
            if (tree_work[a.tree] != tree_work[b.tree]) return tree_work[a.tree] > tree_work[b.tree];
            return a.tree < b.tree;
        }
        return a.work > b.work;
    });
    std::vector<int32_t> qt(2 * qts.size());
    for (size_t j = 0; j < qts.size(); ++j) { qt[2 * j] = qts[j].seq; qt[2 * j + 1] = qts[j].tile; }
    I.n_qt = static_cast<int32_t>(qts.size());
    put(I.off_attn_rptr, rptr.data(), rptr.size());
    put(I.off_attn_runs, runs.data(), runs.size());
    put(I.off_attn_mptr, mptr.data(), mptr.size());
    put(I.off_attn_mask, vmask.data(), vmask.size());
    put(I.off_attn_hp, hp.data(), hp.size());
    put(I.off_attn_qt, qt.data(), qt.size());

    // Key tiles for the key / value gradients: kAttnTile own rows of a sequence.  The
    // query tiles that see key tile (s, i): the sequence's own tiles from i on (causal),
    // and every query tile of every sequence whose prefix runs through s, with the number
    // f of s's own rows in that prefix (keys at local position < f visible, i < ceil(f/B)).
    // Each key tile's list is in ascending (sequence, tile) order; key tiles are grouped
    // by tree like the query tiles, then by decreasing work (query rows to visit).
    std::vector<int32_t> kbase(n_seq + 1, 0);
    for (int32_t i = 0; i < n_seq; ++i) {
        const int64_t own = P.cu_seqlens[i + 1] - P.cu_seqlens[i];
        kbase[i + 1] = kbase[i] + static_cast<int32_t>((own + kAttnTile - 1) / kAttnTile);
    }
    const int32_t n_ktile = P.attn_ok ? kbase[n_seq] : 0;
    std::vector<std::vector<int32_t>> klist(n_ktile);   // (sequence, tile, f) triples
    std::vector<int64_t> kwork(n_ktile, 0);
    for (int32_t t = 0; t < n_seq && P.attn_ok; ++t) {
        const int64_t own_t = P.cu_seqlens[t + 1] - P.cu_seqlens[t];
        const int32_t nqt_t = static_cast<int32_t>((own_t + kAttnTile - 1) / kAttnTile);
        auto add = [&](int32_t kt, int32_t tile, int32_t f) {
            klist[kt].insert(klist[kt].end(), {t, tile, f});
            kwork[kt] += std::min<int64_t>(kAttnTile, own_t - int64_t(tile) * kAttnTile);
        };
        for (int32_t u = P.parent[P.seq_first_seg[t]]; u >= 0;) {
            const int32_t s_ = P.seg_seq[u];
            const int64_t f = P.seg_pos[u] + P.seg_len[u] - P.seg_pos[P.seq_first_seg[s_]];
            for (int32_t i = 0; int64_t(i) * kAttnTile < f; ++i)
                for (int32_t qt2 = 0; qt2 < nqt_t; ++qt2) add(kbase[s_] + i, qt2, static_cast<int32_t>(f));
            u = P.parent[P.seq_first_seg[s_]];
        }
        for (int32_t i = 0; i < nqt_t; ++i)
            for (int32_t qt2 = i; qt2 < nqt_t; ++qt2) add(kbase[t] + i, qt2, -1);
    }
    // lists were appended by ascending query sequence t, ancestors before its own tiles;
    // sort each into ascending (sequence, tile) so the order is a documented one
    for (auto &l : klist) {
        const size_t n = l.size() / 3;
        std::vector<std::array<int32_t, 3>> e(n);
        for (size_t j = 0; j < n; ++j) e[j] = {l[3 * j], l[3 * j + 1], l[3 * j + 2]};
        std::sort(e.begin(), e.end());
        for (size_t j = 0; j < n; ++j) { l[3 * j] = e[j][0]; l[3 * j + 1] = e[j][1]; l[3 * j + 2] = e[j][2]; }
    }
    struct KTile { int64_t work; int32_t tree, seq, tile; };
    std::vector<KTile> kts;
    std::vector<int64_t> ktree_work(P.parent.size(), 0);
    for (int32_t i = 0; i < n_seq && P.attn_ok; ++i) {
        const int32_t r = root[P.seq_first_seg[i]];
        for (int32_t j = kbase[i]; j < kbase[i + 1]; ++j) {
            kts.push_back({kwork[j], r, i, j - kbase[i]});
            ktree_work[r] = std::max(ktree_work[r], kwork[j]);
        }
    }
    std::stable_sort(kts.begin(), kts.end(), [&](const KTile &a, const KTile &b) {
        if (a.tree != b.tree) {
            if (ktree_work[a.tree] != ktree_work[b.tree]) return ktree_work[a.tree] > ktree_work[b.tree];
            return a.tree < b.tree;
        }
        return a.work > b.work;
    });
    std::vector<int32_t> akt(2 * kts.size()), akptr(kts.size() + 1, 0), kq;
    for (size_t j = 0; j < kts.size(); ++j) {
        akt[2 * j] = kts[j].seq; akt[2 * j + 1] = kts[j].tile;
        const auto &l = klist[kbase[kts[j].seq] + kts[j].tile];
        kq.insert(kq.end(), l.begin(), l.end());
        akptr[j + 1] = static_cast<int32_t>(kq.size() / 3);
    }
    I.n_kt = static_cast<int32_t>(kts.size());
    put(I.off_attn_kt, akt.data(), akt.size());
    put(I.off_attn_kptr, akptr.data(), akptr.size());
    put(I.off_attn_kq, kq.data(), kq.size());
    while (w.size() % 64) w.push_back(0);
}

}  // namespace
}  // namespace harts

using harts::set_error;

extern "C" {

const char *harts_last_error(void) { return harts::g_last_error.c_str(); }

int harts_plan_calls(int32_t n_seg, const int32_t *parent, const int64_t *seg_len, int32_t chunk,
                     uint32_t flags, harts_plan **out) {
    if (!out) { set_error("out is NULL"); return HARTS_EINVAL; }
    *out = nullptr;
    if (n_seg < 1 || !parent || !seg_len) { set_error("empty or NULL tree"); return HARTS_EINVAL; }
    if (chunk < 1 || chunk > (1 << 20)) { set_error("chunk must be >= 1"); return HARTS_EINVAL; }
    if ((flags & ~(HARTS_PLAN_NODEWISE | HARTS_PLAN_NOREPLAY)) ||
        flags == (HARTS_PLAN_NODEWISE | HARTS_PLAN_NOREPLAY)) {
        set_error("unknown or conflicting flags"); return HARTS_EINVAL;
    }
    harts_plan *P = new (std::nothrow) harts_plan();
    if (!P) { set_error("out of host memory"); return HARTS_EINVAL; }
    try {
        int rc = harts::build(*P, n_seg, parent, seg_len, chunk, flags);
        if (rc != HARTS_OK) { delete P; return rc; }
        harts::build_image(*P);
    } catch (const std::bad_alloc &) {
        delete P; set_error("out of host memory"); return HARTS_EOVERFLOW;
    }
    *out = P;
    set_error("");
    return HARTS_OK;
}

int harts_plan_get_info(const harts_plan *plan, harts_plan_info *out) {
    if (!plan || !out) { set_error("NULL argument"); return HARTS_EINVAL; }
    *out = plan->info;
    return HARTS_OK;
}

int harts_plan_export(const harts_plan *P, harts_plan_arrays *d) {
    if (!P || !d) { set_error("NULL argument"); return HARTS_EINVAL; }
    auto cp = [](auto *dst, const auto &v) {
        if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(v[0]));
    };
    cp(d->seg_offset, P->seg_offset); cp(d->seg_pos, P->seg_pos); cp(d->seg_seq, P->seg_seq);
    cp(d->seg_ctop, P->seg_ctop); cp(d->seg_tpre, P->seg_tpre); cp(d->seg_tin, P->seg_tin);
    cp(d->round_seq_ptr, P->round_seq_ptr); cp(d->cu_seqlens, P->cu_seqlens);
    cp(d->seq_round, P->seq_round); cp(d->seq_first_seg, P->seq_first_seg);
    cp(d->seq_anchor, P->seq_anchor); cp(d->seq_replay, P->seq_replay); cp(d->seq_src, P->seq_src);
    cp(d->replay_ptr, P->replay_ptr); cp(d->replay_idx, P->replay_idx);
    cp(d->seq_state_ptr, P->seq_state_ptr); cp(d->state_seq, P->state_seq);
    cp(d->state_pos, P->state_pos); cp(d->state_cons_ptr, P->state_cons_ptr);
    cp(d->state_cons, P->state_cons); cp(d->root_cons_ptr, P->root_cons_ptr);
    cp(d->root_cons, P->root_cons);
    return HARTS_OK;
}

size_t harts_plan_device_bytes(const harts_plan *P) {
    return P ? P->image.words.size() * sizeof(int32_t) : 0;
}

void harts_plan_free(harts_plan *P) { delete P; }

}  // extern "C"
