"""fp64 chunkwise form of the gated delta rule and a plan-following tree executor.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Used on small inputs to
pin two readings the CUDA path relies on:

1. The chunkwise (UT / WY) form equals the token recurrence.  The pages say the
   high-performance kernels are chunkwise: parallel inside a chunk of fixed length B,
   recurrent state between chunks (page "HARTS ... 精读", section 1.2).  The chunk
   equations are not printed; the ones below follow from unrolling the recurrence
   over one chunk (local t = 1..L, Gamma_t = sum_{s<=t} g_s per channel):

       A    = strict_lower( (K*e^Gamma) (K*e^-Gamma)^T )
       T    = (I + diag(beta) A)^-1
       W_k  = T diag(beta) (K*e^Gamma),     W_v = T diag(beta) V
       U    = W_v - W_k S                   (U = beta * new values)
       O    = (Q*e^Gamma) S + incl_lower( (Q*e^Gamma) (K*e^-Gamma)^T ) U
       S   <- diag(e^Gamma_L) S + (K*e^(Gamma_L - Gamma))^T U

   Here the pairwise factors exp(Gamma_t - Gamma_s) are formed directly (exact in
   fp64), not through a reference row.
2. Bounded replay (section 4.2, "重放的定位"): a side branch resumes from the state at
   the chunk boundary a(p) and replays [a(p), p) inside the call, so its chunk
   partition is the trajectory's.  ``tree_exec`` runs the plan round by round and
   must reproduce per-trajectory execution.
"""
from __future__ import annotations

import numpy as np


def chunk_fwd_seq(q, k, v, g, beta, S0, B, scale=1.0, positions=()):
    """One sequence, one head. q,k,g: [L,dk]; v: [L,dv]; beta: [L]; S0: [dk,dv].
    Returns (o [L,dv], the state at every chunk end B, 2B, ... and at L, plus at each
    local position in `positions` that falls inside a chunk, as a dict keyed by local
    position, final state).  Inside a chunk, the state after its first r rows is the
    chunk update restricted to those rows: diag(e^{Gamma_r}) S + K_r~^T U_r with
    K_r~ = K e^{Gamma_r - Gamma} over rows < r."""
    L, dk = k.shape
    S = np.array(S0, dtype=np.float64)
    o = np.zeros((L, v.shape[1]))
    bstates = {}
    for c0 in range(0, L, B):
        c1 = min(c0 + B, L)
        Q, K, V, G, b = q[c0:c1] * scale, k[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1]
        n = c1 - c0
        Gam = np.cumsum(G, axis=0)
        # pairwise decay exp(Gamma_t - Gamma_s) per channel
        D = np.exp(Gam[:, None, :] - Gam[None, :, :])          # [t, s, dk]
        KK = np.einsum("tc,sc,tsc->ts", K, K, D)
        QK = np.einsum("tc,sc,tsc->ts", Q, K, D)
        A = np.tril(KK, -1)
        T = np.linalg.inv(np.eye(n) + b[:, None] * A)
        Kd = K * np.exp(Gam)
        Wk = T @ (b[:, None] * Kd)
        Wv = T @ (b[:, None] * V)
        U = Wv - Wk @ S
        o[c0:c1] = (Q * np.exp(Gam)) @ S + np.tril(QK) @ U
        for pos in positions:
            if c0 < pos < c1:
                r = pos - c0
                Kr = K[:r] * np.exp(Gam[r - 1][None, :] - Gam[:r])
                bstates[pos] = np.exp(Gam[r - 1])[:, None] * S + Kr.T @ U[:r]
        Kt = K * np.exp(Gam[-1][None, :] - Gam)
        S = np.exp(Gam[-1])[:, None] * S + Kt.T @ U
        bstates[c1] = S.copy()
    return o, bstates, S


def tree_exec(pl, q, k, v, g, beta, B, scale=1.0, h0=None):
    """Execute a plan from ``plan_twin.plan`` round by round in fp64.

    q,k,g: [C,H,dk]; v: [C,H,dv]; beta: [C,H] in the plan's compact layout.
    Returns (o [C,H,dv], final states per sequence [n_seq,H,dk,dv])."""
    C, H, dk = q.shape
    dv = v.shape[2]
    o = np.zeros((C, H, dv))
    final = np.zeros((pl["n_seq"], H, dk, dv))
    slots = np.zeros((pl["n_states"], H, dk, dv))
    for r in range(pl["n_rounds"]):
        for sq in range(pl["round_seq_ptr"][r], pl["round_seq_ptr"][r + 1]):
            src = pl["seq_src"][sq]
            rows = np.concatenate([pl["replay_idx"][pl["replay_ptr"][sq]:pl["replay_ptr"][sq + 1]],
                                   np.arange(pl["cu_seqlens"][sq], pl["cu_seqlens"][sq + 1])])
            rho = int(pl["seq_replay"][sq])
            want = {int(pl["state_pos"][j]): j
                    for j in range(pl["seq_state_ptr"][sq], pl["seq_state_ptr"][sq + 1])}
            for h in range(H):
                if src >= 0:
                    S0 = slots[src, h]
                elif h0 is not None:
                    S0 = h0[-1 - src, h]
                else:
                    S0 = np.zeros((dk, dv))
                oo, bst, Sf = chunk_fwd_seq(q[rows, h], k[rows, h], v[rows, h], g[rows, h],
                                            beta[rows, h], S0, B, scale, positions=tuple(want))
                o[rows[rho:], h] = oo[rho:]
                for pos, j in want.items():
                    slots[j, h] = bst[pos]
                final[sq, h] = Sf
    return o, final
