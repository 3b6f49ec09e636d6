"""Replay restores the chunk phase (section 4.2, "重放的定位"; section 5.3 and Fig. 5):
a side branch resumes from the chunk-boundary state at a(p) and replays [a(p), p), so
every chunk it computes holds the same rows, from the same state, as the chunk of the
per-trajectory run.  With deterministic kernels the minimum-call plan's forward output
of every compact row is therefore bit-identical to the per-trajectory run of at least
one trajectory through that row (the one whose chunks it shares: rows of a fork chunk
are computed with different chunk-mates in different trajectories).  The no-replay plan
(exact fork state, fresh chunk grid) breaks this for the rows of its side branches."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from prefix_shared_chunkwise_gb300 import _lib
from prefix_shared_chunkwise_gb300.api import Plan, kda_fwd
from prefix_shared_chunkwise_gb300.synth import expand_rows, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _fwd(pl, x, kernel):
    o = torch.empty_like(x["v"])
    st = torch.empty((max(pl.info["n_states"], 1),) + tuple(x["q"].shape[1:]) + (x["v"].shape[2],),
                     dtype=torch.float32, device="cuda")
    kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], o=o, states=st, kernel=kernel)
    torch.cuda.synchronize()
    assert pl.device_error() == 0
    return o


def _match_fraction(parent, seg_len, B, H, D, dtype, kernel, noreplay):
    """Fraction of the side-branch rows (segments outside the root sequences) whose output
    is bit-identical to some trajectory's, for the plan asked for."""
    keys = ("q", "k", "v", "g", "beta")
    pl_t = Plan(parent, seg_len, B).upload()
    so_t = pl_t.arrays()["seg_offset"]
    x = {k: t.cuda() for k, t in make_inputs(pl_t.info["C"], H, D, D, dtype, 5, device="cpu").items()}
    rows, ptr, _ = expand_rows(parent, seg_len, so_t)
    pl_e = Plan(-np.ones(len(ptr) - 1, np.int32), np.diff(ptr).astype(np.int64), B).upload()
    o_e = _fwd(pl_e, {k: x[k].index_select(0, torch.as_tensor(rows, device="cuda")) for k in keys}, kernel)
    pl = Plan(parent, seg_len, B, noreplay=noreplay).upload() if noreplay else pl_t
    so = pl.arrays()["seg_offset"]
    n, C = len(parent), pl.info["C"]
    t2p = np.empty(C, np.int64)
    for v in range(n):
        t2p[so_t[v]:so_t[v] + seg_len[v]] = so[v] + np.arange(seg_len[v])
    p2t = np.empty_like(t2p)
    p2t[t2p] = np.arange(C)
    o_p = _fwd(pl, {k: x[k].index_select(0, torch.as_tensor(p2t, device="cuda")) for k in keys}, kernel)
    o_p = o_p.index_select(0, torch.as_tensor(t2p, device="cuda"))       # back to the tree layout
    eq = (o_p.index_select(0, torch.as_tensor(rows, device="cuda")) == o_e).all(dim=2).all(dim=1).cpu().numpy()
    matched = np.zeros(C, bool)
    np.logical_or.at(matched, rows, eq)
    # rows of segments that are not in a root sequence of the minimum-call plan
    seq_of_seg = pl_t.arrays()["seg_seq"]
    root_seq = set(np.nonzero(pl_t.arrays()["seq_src"] < 0)[0].tolist())
    side = np.zeros(C, bool)
    for v in range(n):
        if seq_of_seg[v] not in root_seq:
            side[so_t[v]:so_t[v] + seg_len[v]] = True
    return matched.mean(), matched[side].mean(), side.sum()


def _forest(seed, n, B):
    rng = np.random.Generator(np.random.PCG64(seed))
    parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
    seg_len = rng.integers(1, 3 * B, size=n).astype(np.int64)
    return parent, seg_len


@pytest.mark.parametrize("kernel,dtype,D", [(_lib.HARTS_KERNEL_TC, "bf16", 128),
                                            (_lib.HARTS_KERNEL_SIMT, "fp32", 32)])
def test_replay_reproduces_a_trajectory_bit_for_bit(kernel, dtype, D):
    parent, seg_len = _forest(11, 16, 64)
    all_rows, side_rows, n_side = _match_fraction(parent, seg_len, 64, 2, D, dtype, kernel, False)
    assert n_side > 0
    assert all_rows == 1.0 and side_rows == 1.0


def test_noreplay_leaves_the_trajectory_numerics():
    parent, seg_len = _forest(11, 16, 64)
    _, side_rows, n_side = _match_fraction(parent, seg_len, 64, 2, 128, "bf16", _lib.HARTS_KERNEL_TC, True)
    assert n_side > 0
    assert side_rows < 0.5
