"""Planner oracle: the minimum-call recurrence in plain Python, and brute force.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg do.
It shares no code with the C++ planner in the library.

What it restates (page "HARTS ... 精读", section 4.2, and the v2 figure captions
Fig. 1(c) and Fig. 2 on page "thelatestinai ... 2608.28158"):

* A rollout tree is contracted into fork-free segments.  One packed chunkwise call
  per round; a boundary state produced inside a call can only initialise another
  input sequence after that call returns, so at each fork at most one child stays in
  the same input sequence (the direct continuation); other children start new
  sequences.
* A side branch at fork end position p resumes from the chunk-boundary state at
  a(p) = B*floor(p/B) and replays the ancestor tokens [a(p), p) (section 4.2,
  "重放的定位").  The replay is fixed by B and p; the planner only minimises the number
  of sequential calls.
* T_pre(v): fewest rounds for v's subtree when v's entry anchor state is ready
  before the current call; T_in(v): fewest rounds when v enters the current call
  as a direct continuation.  Leaves have T_pre = T_in = 1.  The equations (13)/(14)
  are not printed on the pages; the reading taken here is

      m1 = max_c T_pre(c)  (attained at c_top, lowest child id on ties)
      m2 = max_{c != c_top} T_pre(c), 0 if none
      T_in(v)  = max(T_in(c_top), 1 + m2)        side branch waits one round
      T_pre(v) = m1 if a(s_v) == a(e_v) else T_in(v)

  The first case is a fork inside the chunk where v's own sequence starts: the
  side children can start in the same call from the same anchor state, replaying
  [a(s_v), e_v) (Fig. 2(c): v2, started by replay, runs in round 1).
* Recovery is top-down and as-soon-as-possible.

Conventions (several plans are optimal; these make the plan unique):
* the continuation is the lowest-id child among those with maximal T_pre;
* sequences are ordered by round, then by the id of their first segment
  (Fig. 1(c) lists the second call as [C], then [E]);
* within a sequence, segments follow the continuation chain; compact rows follow
  that order (one compact physical layout, section 4.3);
* one state slot per distinct (producer sequence, local position); slots are
  numbered by producer sequence, then position;
* roots are numbered by increasing segment id.
"""
from __future__ import annotations

import itertools

import numpy as np


def _children(parent):
    n = len(parent)
    ch = [[] for _ in range(n)]
    for i in range(n):
        p = int(parent[i])
        if not (-1 <= p < i):
            raise ValueError(f"parent[{i}]={p} must satisfy -1 <= parent < index")
        if p >= 0:
            ch[p].append(i)
    return ch


def positions(parent, seg_len):
    """s_v (trajectory position of v's first token) and e_v = s_v + len_v."""
    n = len(parent)
    s = [0] * n
    e = [0] * n
    for i in range(n):
        if int(seg_len[i]) < 1:
            raise ValueError("segment length must be >= 1")
        s[i] = 0 if parent[i] < 0 else e[parent[i]]
        e[i] = s[i] + int(seg_len[i])
    return s, e


def min_calls(parent, seg_len, B):
    """Bottom-up T_pre / T_in and the continuation child of every internal node."""
    ch = _children(parent)
    s, e = positions(parent, seg_len)
    n = len(parent)
    Tpre = [0] * n
    Tin = [0] * n
    ctop = [-1] * n
    for v in range(n - 1, -1, -1):
        if not ch[v]:
            Tpre[v] = Tin[v] = 1
            continue
        best, m1 = -1, 0
        for c in ch[v]:              # ascending ids: strict '>' keeps the lowest id
            if Tpre[c] > m1:
                best, m1 = c, Tpre[c]
        m2 = 0
        for c in ch[v]:
            if c != best and Tpre[c] > m2:
                m2 = Tpre[c]
        ctop[v] = best
        Tin[v] = max(Tin[best], 1 + m2)
        Tpre[v] = m1 if (s[v] // B) == (e[v] // B) else Tin[v]
    roots = [i for i in range(n) if parent[i] < 0]
    calls = max(Tpre[r] for r in roots) if roots else 0
    return dict(calls=calls, Tpre=Tpre, Tin=Tin, ctop=ctop, s=s, e=e, children=ch)


def plan(parent, seg_len, B, nodewise=False, noreplay=False):
    """Full plan: rounds, sequences, replay gather lists, state slots, layout.

    nodewise=True gives the node-wise baseline of the pages' comparison (section 5,
    Fig. 4 "Node-wise LA"): no continuation anywhere, so every segment is a sequence;
    a child starts one round after its parent from the state at the parent's end
    (trajectory position e_v, not rounded to the chunk grid), replaying nothing.

    noreplay=True gives the no-replay comparison of section 5.3 / Fig. 5: the same
    continuations, but every side branch starts one round after its producer from the
    producer's exact state at e_v (a position inside a chunk in general), with its own
    chunk grid and nothing replayed."""
    parent = [int(x) for x in parent]
    seg_len = [int(x) for x in seg_len]
    n = len(parent)
    dp = min_calls(parent, seg_len, B)
    ch, ctop, s, e = dp["children"], dp["ctop"], dp["s"], dp["e"]
    if nodewise:
        ctop = [-1] * n
    roots = [i for i in range(n) if parent[i] < 0]
    root_idx = {r: j for j, r in enumerate(roots)}

    # top-down ASAP recovery; a sequence is (first segment, round, anchor, source)
    # where source = ("root", r) or ("slot", producer first segment, local position)
    seqs = []
    work = [(r, 1, 0, ("root", root_idx[r])) for r in roots]
    while work:
        first, rnd, anchor, src = work.pop()
        chain = []
        slots = []
        v = first
        while True:
            chain.append(v)
            if not ch[v]:
                break
            for c in ch[v]:
                if c == ctop[v]:
                    continue
                exact = nodewise or noreplay
                a_e = e[v] if exact else B * (e[v] // B)
                if not exact and a_e == anchor:
                    work.append((c, rnd, anchor, src))
                else:
                    pos = a_e - anchor
                    if pos not in slots:
                        slots.append(pos)
                    work.append((c, rnd + 1, a_e, ("slot", first, pos)))
            v = ctop[v]
            if v < 0:          # node-wise: no continuation
                break
        seqs.append(dict(first=first, round=rnd, anchor=anchor, src=src, chain=chain,
                         slots=sorted(slots)))
    seqs.sort(key=lambda d: (d["round"], d["first"]))
    seq_of_first = {d["first"]: i for i, d in enumerate(seqs)}
    n_seq = len(seqs)
    n_rounds = max(d["round"] for d in seqs) if seqs else 0

    # layout: compact rows follow sequence order then chain order
    seg_offset = np.zeros(n, np.int64)
    seg_seq = np.zeros(n, np.int32)
    cu = np.zeros(n_seq + 1, np.int64)
    row = 0
    for i, d in enumerate(seqs):
        cu[i] = row
        for v in d["chain"]:
            seg_offset[v] = row
            seg_seq[v] = i
            row += seg_len[v]
    cu[n_seq] = row

    # slots in (producer sequence, position) order
    state_seq, state_pos, slot_id = [], [], {}
    seq_state_ptr = np.zeros(n_seq + 1, np.int32)
    for i, d in enumerate(seqs):
        seq_state_ptr[i] = len(state_seq)
        for pos in d["slots"]:
            slot_id[(i, pos)] = len(state_seq)
            state_seq.append(i)
            state_pos.append(pos)
    seq_state_ptr[n_seq] = len(state_seq)

    seq_src = np.zeros(n_seq, np.int32)
    seq_round = np.zeros(n_seq, np.int32)
    seq_first = np.zeros(n_seq, np.int32)
    seq_anchor = np.zeros(n_seq, np.int64)
    seq_replay = np.zeros(n_seq, np.int32)
    replay_ptr = np.zeros(n_seq + 1, np.int64)
    replay_idx = []
    for i, d in enumerate(seqs):
        seq_round[i] = d["round"]
        seq_first[i] = d["first"]
        seq_anchor[i] = d["anchor"]
        if d["src"][0] == "root":
            seq_src[i] = -1 - d["src"][1]
        else:
            seq_src[i] = slot_id[(seq_of_first[d["src"][1]], d["src"][2])]
        first = d["first"]
        rho = s[first] - d["anchor"]
        assert 0 <= rho < B
        seq_replay[i] = rho
        replay_ptr[i] = len(replay_idx)
        # ancestor rows for trajectory positions [anchor, s_first), increasing position
        rows = []
        w = parent[first]
        while w >= 0 and e[w] > d["anchor"]:
            lo = max(s[w], d["anchor"])
            rows.append([seg_offset[w] + (p - s[w]) for p in range(lo, e[w])])
            w = parent[w]
        for r in reversed(rows):
            replay_idx.extend(r)
        assert len(replay_idx) - replay_ptr[i] == rho
    replay_ptr[n_seq] = len(replay_idx)

    round_seq_ptr = np.zeros(n_rounds + 1, np.int32)
    for r in range(1, n_rounds + 1):
        round_seq_ptr[r] = int(np.sum(seq_round <= r))

    n_st = len(state_seq)
    cons = [[] for _ in range(n_st)]
    rcons = [[] for _ in range(len(roots))]
    for i in range(n_seq):
        if seq_src[i] >= 0:
            cons[seq_src[i]].append(i)
        else:
            rcons[-1 - seq_src[i]].append(i)
    state_cons_ptr = np.zeros(n_st + 1, np.int32)
    state_cons = []
    for j in range(n_st):
        state_cons_ptr[j] = len(state_cons)
        state_cons.extend(cons[j])
    state_cons_ptr[n_st] = len(state_cons)
    root_cons_ptr = np.zeros(len(roots) + 1, np.int32)
    root_cons = []
    for j in range(len(roots)):
        root_cons_ptr[j] = len(root_cons)
        root_cons.extend(rcons[j])
    root_cons_ptr[len(roots)] = len(root_cons)

    leaves_under = np.zeros(n, np.int64)
    for v in range(n - 1, -1, -1):
        if not ch[v]:
            leaves_under[v] = 1
        if parent[v] >= 0:
            leaves_under[parent[v]] += leaves_under[v]

    return dict(
        n_rounds=n_rounds, n_seq=n_seq, n_states=n_st, n_roots=len(roots),
        C=int(cu[n_seq]), S=int(sum(seg_len[v] * leaves_under[v] for v in range(n))),
        R=int(replay_ptr[n_seq]),
        Tpre=np.asarray(dp["Tpre"], np.int32), Tin=np.asarray(dp["Tin"], np.int32),
        ctop=np.asarray(ctop, np.int32),
        seg_pos=np.asarray(s, np.int64), seg_offset=seg_offset, seg_seq=seg_seq,
        round_seq_ptr=round_seq_ptr, cu_seqlens=cu, seq_round=seq_round,
        seq_first_seg=seq_first, seq_anchor=seq_anchor, seq_replay=seq_replay,
        seq_src=seq_src, replay_ptr=replay_ptr,
        replay_idx=np.asarray(replay_idx, np.int64),
        seq_state_ptr=seq_state_ptr, state_seq=np.asarray(state_seq, np.int32),
        state_pos=np.asarray(state_pos, np.int64),
        state_cons_ptr=state_cons_ptr, state_cons=np.asarray(state_cons, np.int32),
        root_cons_ptr=root_cons_ptr, root_cons=np.asarray(root_cons, np.int32),
        seq_chain=[d["chain"] for d in seqs],
    )


def brute_force_calls(parent, seg_len, B, allow_none=True):
    """Fewest rounds over every choice of direct continuation at every fork
    (including, if allowed, no continuation), each side branch started as early as
    the anchor rule lets it.  Exponential: trees of a handful of segments only."""
    parent = [int(x) for x in parent]
    n = len(parent)
    ch = _children(parent)
    s, e = positions(parent, seg_len)
    internal = [v for v in range(n) if ch[v]]
    options = [ch[v] + ([None] if allow_none else []) for v in internal]
    best = None
    for choice in itertools.product(*options):
        cont = dict(zip(internal, choice))
        rounds = 0
        work = [(r, 1, 0) for r in range(n) if parent[r] < 0]
        while work:
            v, rnd, anchor = work.pop()
            while True:
                rounds = max(rounds, rnd)
                if not ch[v]:
                    break
                nxt = cont[v]
                for c in ch[v]:
                    if c == nxt:
                        continue
                    a_e = B * (e[v] // B)
                    if a_e == anchor:
                        work.append((c, rnd, anchor))
                    else:
                        work.append((c, rnd + 1, a_e))
                if nxt is None:
                    break
                v = nxt
        if best is None or rounds < best:
            best = rounds
    return best


def strahler(parent):
    """Horton-Strahler number of every node (leaf 1; internal: m1 + [m1 == m2])."""
    ch = _children(parent)
    n = len(parent)
    st = [0] * n
    for v in range(n - 1, -1, -1):
        if not ch[v]:
            st[v] = 1
            continue
        vals = sorted((st[c] for c in ch[v]), reverse=True)
        m1 = vals[0]
        m2 = vals[1] if len(vals) > 1 else 0
        st[v] = m1 + (1 if m1 == m2 else 0)
    return st
