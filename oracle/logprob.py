"""Compact-to-semantic log-probabilities: fp64 oracle.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module; only
``tests/`` and ``bench.py``'s reference leg do.  It shares no code with the library.

What it restates (page "HARTS ... 精读", section 4.4, "紧凑到语义的 log 概率"; summary
page, "Semantic Preservation"): a compact logit row is reduced over the vocabulary once
(max and sum-exp, i.e. its log-sum-exp); every semantic position s (a token occurrence
of an original trajectory, in the original order) reads its own target logit from the
row c(s) its token maps to: lambda_s = z[c(s), y_s] - lse[c(s)].  The backward (eq. 19)
sums the independently formed gradients of all semantic positions of a row onto it:
dz[c] = sum_{s: c(s) = c} g_s (onehot(y_s) - softmax(z[c])), so distinct labels and
per-position weights (advantages, masks) all survive.
"""
from __future__ import annotations

import numpy as np


def semantic_map(parent, seg_len, seg_offset):
    """Compact row of every semantic position: trajectories in increasing leaf id, each
    from its root to its leaf."""
    parent = np.asarray(parent)
    n = len(parent)
    has_kid = np.zeros(n, bool)
    has_kid[parent[parent >= 0]] = True
    out = []
    for leaf in range(n):
        if has_kid[leaf]:
            continue
        chain = []
        v = leaf
        while v >= 0:
            chain.append(v)
            v = parent[v]
        out.extend(np.arange(seg_offset[v], seg_offset[v] + seg_len[v]) for v in reversed(chain))
    return np.concatenate(out).astype(np.int64)


def logprob_fwd(logits, sem_row, target):
    """lambda [S] and lse [C] from compact logits [C, V]."""
    z = np.asarray(logits, np.float64)
    m = z.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))[:, 0]
    lam = z[sem_row, target] - lse[sem_row]
    return lam, lse


def logprob_bwd(logits, sem_row, target, g):
    """dz [C, V] for dL/dlambda = g [S] (eq. 19: per-position gradients summed per row)."""
    z = np.asarray(logits, np.float64)
    _, lse = logprob_fwd(z, sem_row, target)
    p = np.exp(z - lse[:, None])
    G = np.zeros(z.shape[0])
    np.add.at(G, sem_row, g)
    dz = -G[:, None] * p
    np.add.at(dz, (sem_row, target), g)
    return dz
