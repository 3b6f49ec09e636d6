"""Branch attention over the compact layout (the MLA half of the hybrid layer): fp64
oracle.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module; only
``tests/`` and ``bench.py``'s reference leg do.  It shares no code with the library.

What it restates (page "HARTS ... 精读", section 4.3, MLA paragraph; summary page,
section 4 "MLA execution"; figures page, Figure C.1(c)): projections run once per compact
token; a branch's attention view packs its queries (its own l tokens) against keys and
values of its ancestors and itself (h + l), with bottom-right causal alignment, so query
i sees exactly the entries j <= h + i: the full ancestor prefix and the causal triangle
of its own tokens.  Outputs go back to the unique compact rows.

Reading taken where the pages are silent: the attention core is
plain multi-head softmax attention, o = softmax(scale q k^T) v per head, on already
projected (and position-rotated) q, k, v; head dimensions are the caller's.  Since a
row's view is its own trajectory prefix, the output of a compact row is the causal
attention of that row over its trajectory, whichever trajectory through it is used.
"""
from __future__ import annotations

import numpy as np

from oracle.conv import _paths


def attn_forest(parent, seg_len, seg_offset, q, k, v, scale):
    """q, k: [C, H, dk]; v: [C, H, dv] (compact layout).  Per trajectory: causal softmax
    attention over its rows; a shared row must come out the same from each trajectory.
    Returns dict(o [C, H, dv], lse [C, H], occ_diff)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    C, H, _ = q.shape
    o = np.full((C, H, v.shape[2]), np.nan)
    lse = np.full((C, H), np.nan)
    occ = 0.0
    for rows in _paths(parent, seg_len, seg_offset):
        L = len(rows)
        mask = np.tril(np.ones((L, L), bool))
        for h in range(H):
            s = scale * q[rows, h] @ k[rows, h].T
            s = np.where(mask, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            den = p.sum(axis=1, keepdims=True)
            oo = (p / den) @ v[rows, h]
            ll = (m + np.log(den))[:, 0]
            seen = ~np.isnan(o[rows, h, 0])
            if seen.any():
                occ = max(occ, float(np.abs(o[rows[seen], h] - oo[seen]).max()))
            o[rows, h] = oo
            lse[rows, h] = ll
    return dict(o=o, lse=lse, occ_diff=occ)


def trajectory_prefix(parent, seg_len, seg_offset, row):
    """Compact rows of the trajectory positions 0 .. p(row): the ancestors' rows, root
    first, then the row's own segment up to and including the row."""
    parent = np.asarray(parent)
    seg_offset = np.asarray(seg_offset)
    ends = seg_offset + np.asarray(seg_len)
    seg = int(np.nonzero((seg_offset <= row) & (row < ends))[0][0])
    chain = []
    v = int(parent[seg])
    while v >= 0:
        chain.append(v)
        v = int(parent[v])
    parts = [np.arange(seg_offset[u], seg_offset[u] + seg_len[u]) for u in reversed(chain)]
    parts.append(np.arange(seg_offset[seg], row + 1))
    return np.concatenate(parts).astype(np.int64)


def attn_query(q_row, k_view, v_view, scale):
    """One query over its whole view (every entry visible): q_row [H, dk], k_view
    [n, H, dk], v_view [n, H, dv] -> (o [H, dv], lse [H])."""
    q_row = np.asarray(q_row, np.float64)
    k_view = np.asarray(k_view, np.float64)
    v_view = np.asarray(v_view, np.float64)
    o = np.empty((q_row.shape[0], v_view.shape[2]))
    lse = np.empty(q_row.shape[0])
    for h in range(q_row.shape[0]):
        s = scale * k_view[:, h] @ q_row[h]
        m = s.max()
        p = np.exp(s - m)
        o[h] = (p / p.sum()) @ v_view[:, h]
        lse[h] = m + np.log(p.sum())
    return o, lse


def attn_query_bwd(q_row, k_view, v_view, do_row, scale):
    """Backward of attn_query for dL/do = do_row: (dq_row [H, dk], dk_view [n, H, dk],
    dv_view [n, H, dv])."""
    q_row = np.asarray(q_row, np.float64)
    k_view = np.asarray(k_view, np.float64)
    v_view = np.asarray(v_view, np.float64)
    do_row = np.asarray(do_row, np.float64)
    dq = np.zeros_like(q_row)
    dk, dv = np.zeros_like(k_view), np.zeros_like(v_view)
    for h in range(q_row.shape[0]):
        kv, vv = k_view[:, h], v_view[:, h]
        s = scale * kv @ q_row[h]
        p = np.exp(s - s.max())
        p /= p.sum()
        dv[:, h] = np.outer(p, do_row[h])
        dp = vv @ do_row[h]
        ds = p * (dp - p @ dp)
        dq[h] = scale * ds @ kv
        dk[:, h] = scale * np.outer(ds, q_row[h])
    return dq, dk, dv


def attn_forest_bwd(parent, seg_len, seg_offset, q, k, v, do, scale):
    """Gradients of L = sum_r <do[r], o[r]> for the compact-row outputs of attn_forest:
    each compact query row counts once, over its own trajectory prefix.  Returns dict(dq,
    dk, dv), all [C, H, d]; keys and values collect the contributions of every query that
    sees them, across branches."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for r in range(q.shape[0]):
        view = trajectory_prefix(parent, seg_len, seg_offset, r)
        g_q, g_k, g_v = attn_query_bwd(q[r], k[view], v[view], do[r], scale)
        dq[r] = g_q
        np.add.at(dk, view, g_k)
        np.add.at(dv, view, g_v)
    return dict(dq=dq, dk=dk, dv=dv)
