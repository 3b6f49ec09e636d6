"""Pins for the compact-to-semantic log-probability oracle (oracle/logprob.py): the
expanded S x V computation with scipy's log_softmax (what trajectory-wise training does),
finite differences, and the ordering of the semantic map."""
import numpy as np
import pytest

from oracle import logprob

scipy_special = pytest.importorskip("scipy.special")


def _case(seed, C=23, V=37, S=61):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((C, V)) * 3
    sem_row = rng.integers(0, C, size=S)
    target = rng.integers(0, V, size=S)
    g = rng.standard_normal(S)
    return z, sem_row, target, g


@pytest.mark.parametrize("seed", range(4))
def test_forward_equals_expanded_log_softmax(seed):
    z, sem_row, target, _ = _case(seed)
    lam, lse = logprob.logprob_fwd(z, sem_row, target)
    expanded = scipy_special.log_softmax(z[sem_row], axis=1)      # S x V, as trajectory-wise training
    np.testing.assert_allclose(lam, expanded[np.arange(len(sem_row)), target], atol=1e-12)
    np.testing.assert_allclose(lse, scipy_special.logsumexp(z, axis=1), atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_backward_equals_expanded_gradient_summed(seed):
    """Gradient of sum_s g_s lambda_s through the expanded S x V logits, each occurrence
    on its own, then summed onto the compact rows."""
    z, sem_row, target, g = _case(seed)
    dz = logprob.logprob_bwd(z, sem_row, target, g)
    soft = scipy_special.softmax(z[sem_row], axis=1)
    onehot = np.zeros_like(soft)
    onehot[np.arange(len(sem_row)), target] = 1.0
    d_exp = g[:, None] * (onehot - soft)
    ref = np.zeros_like(z)
    for s, c in enumerate(sem_row):
        ref[c] += d_exp[s]
    np.testing.assert_allclose(dz, ref, atol=1e-12)


def test_backward_finite_differences():
    z, sem_row, target, g = _case(9, C=5, V=7, S=11)
    dz = logprob.logprob_bwd(z, sem_row, target, g)
    eps = 1e-6
    num = np.zeros_like(z)
    for idx in np.ndindex(z.shape):
        z0 = z[idx]
        z[idx] = z0 + eps; lp = np.dot(g, logprob.logprob_fwd(z, sem_row, target)[0])
        z[idx] = z0 - eps; lm = np.dot(g, logprob.logprob_fwd(z, sem_row, target)[0])
        z[idx] = z0
        num[idx] = (lp - lm) / (2 * eps)
    np.testing.assert_allclose(dz, num, atol=1e-7)


def test_rows_without_semantic_positions_get_zero_gradient_and_sum_rule():
    z, sem_row, target, g = _case(3)
    used = np.zeros(z.shape[0], bool)
    used[sem_row] = True
    dz = logprob.logprob_bwd(z, sem_row, target, g)
    assert np.all(dz[~used] == 0.0)
    # each row's gradient sums to zero over the vocabulary (softmax rows sum to one)
    np.testing.assert_allclose(dz.sum(axis=1), 0.0, atol=1e-12)


def test_semantic_map_order():
    # Fig. 1(a)-like tree: A -> B -> {C, D}, A -> E (segments 0..4)
    parent = np.array([-1, 0, 1, 1, 0])
    seg_len = np.array([2, 1, 2, 1, 3])
    so = np.array([0, 2, 3, 5, 6])
    m = logprob.semantic_map(parent, seg_len, so)
    # leaves in increasing id: 2 (A B C), 3 (A B D), 4 (A E)
    np.testing.assert_array_equal(m, [0, 1, 2, 3, 4, 0, 1, 2, 5, 0, 1, 6, 7, 8])
