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

Reading taken where the pages are silent (listed in the design doc): the attention core is
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
