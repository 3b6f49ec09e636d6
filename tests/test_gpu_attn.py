"""GPU parity of the branch attention (harts_attn_fwd) against the fp64 oracle
(oracle/attn.py) on the same bf16 inputs: o within 1e-2 relative L2 (bf16 output, P
rounded to bf16 before P V), lse within 1e-5 (fp32).  Forests with ragged query tiles,
ancestor prefixes longer than a tile and not a multiple of it, single-token segments,
the node-wise plan (another sequence split of the same tree), and the full-size forest
on sampled rows."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import attn as oat
from prefix_shared_chunkwise_gb300.api import Plan, attn_fwd
from prefix_shared_chunkwise_gb300.synth import make_tree
from tests._parity import rel_l2

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL = 1e-2, 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _inputs(C, H, seed, qscale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn((C, H, 128), generator=g) * qscale).to(torch.bfloat16)
    k = torch.randn((C, H, 128), generator=g).to(torch.bfloat16)
    v = torch.randn((C, H, 128), generator=g).to(torch.bfloat16)
    return q, k, v


def _check(parent, seg_len, H, seed, nodewise=False, qscale=1.0):
    pl = Plan(parent, seg_len, 64, nodewise=nodewise)
    pl.upload()
    C = pl.info["C"]
    q, k, v = _inputs(C, H, seed, qscale)
    o, lse = attn_fwd(pl, q.cuda(), k.cuda(), v.cuda())
    assert pl.device_error() == 0
    ref = oat.attn_forest(np.asarray(parent), np.asarray(seg_len), pl.arrays()["seg_offset"],
                          q.double().numpy(), k.double().numpy(), v.double().numpy(), 128 ** -0.5)
    eo = rel_l2(o.float().cpu().numpy(), ref["o"])
    el = rel_l2(lse.cpu().numpy(), ref["lse"])
    assert eo <= O_TOL and el <= LSE_TOL, (eo, el)


def _random_forest(seed, n, len_hi):
    rng = np.random.default_rng(seed)
    parent = np.array([-1] + [int(rng.integers(-1, i)) if rng.random() < 0.1 else int(rng.integers(0, i))
                              for i in range(1, n)], np.int32)
    seg_len = rng.integers(1, len_hi, size=n).astype(np.int64)
    return parent, seg_len


@pytest.mark.parametrize("seed", range(3))
def test_random_forest_ragged_tiles(seed):
    parent, seg_len = _random_forest(seed, 14, 300)
    _check(parent, seg_len, 2, seed)


def test_deep_prefix_not_tile_multiple():
    # chain 0 -> 1 -> 2 with side branches: prefixes of 333, 333 + 200 and 533 + 70 rows
    parent = np.array([-1, 0, 1, 0, 1, 2, 2], np.int32)
    seg_len = np.array([333, 200, 70, 129, 1, 257, 128], np.int64)
    _check(parent, seg_len, 3, 11)


def test_single_token_segments_and_nodewise():
    parent, seg_len = _random_forest(7, 40, 3)           # many 1-2 token segments
    _check(parent, seg_len, 1, 12)
    parent, seg_len = _random_forest(8, 12, 200)
    _check(parent, seg_len, 2, 13, nodewise=True)


def test_sharp_scores():
    """Scores spread over tens of units: the running max moves across key tiles."""
    parent, seg_len = _random_forest(9, 6, 400)
    _check(parent, seg_len, 2, 14, qscale=6.0)


def test_fig1_tree():
    parent, seg_len = make_tree("fig1_fp32")
    _check(parent, seg_len, 2, 15)


def test_full_size_sampled_rows():
    """The 64K-token forest at H = 16: sampled rows (first, last, random) against the
    oracle evaluated on each row's own trajectory prefix."""
    parent, seg_len = make_tree("fb64k_bf16")
    pl = Plan(parent, seg_len, 64)
    pl.upload()
    C, H = pl.info["C"], 16
    g = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = (torch.randn((C, H, 128), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    o, lse = attn_fwd(pl, q, k, v)
    assert pl.device_error() == 0
    so = pl.arrays()["seg_offset"]
    rng = np.random.default_rng(6)
    rows = np.unique(np.concatenate([[0, C - 1], rng.integers(0, C, size=12)]))
    for r in rows:
        view = oat.trajectory_prefix(parent, seg_len, so, int(r))
        idx = torch.as_tensor(view, device="cuda")
        ref_o, ref_l = oat.attn_query(q[int(r)].double().cpu().numpy(), k[idx].double().cpu().numpy(),
                                      v[idx].double().cpu().numpy(), 128 ** -0.5)
        assert rel_l2(o[int(r)].float().cpu().numpy(), ref_o) <= O_TOL
        assert rel_l2(lse[int(r)].cpu().numpy(), ref_l) <= LSE_TOL


# ---- backward -------------------------------------------------------------------------

def _check_bwd(parent, seg_len, H, seed, nodewise=False, qscale=1.0):
    from prefix_shared_chunkwise_gb300.api import attn_bwd
    pl = Plan(parent, seg_len, 64, nodewise=nodewise)
    pl.upload()
    C = pl.info["C"]
    q, k, v = _inputs(C, H, seed, qscale)
    g = torch.Generator().manual_seed(seed + 100)
    do = torch.randn((C, H, 128), generator=g).to(torch.bfloat16)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn_fwd(pl, qc, kc, vc)
    dq, dk, dv = attn_bwd(pl, qc, kc, vc, o, lse, doc)
    assert pl.device_error() == 0
    ref = oat.attn_forest_bwd(np.asarray(parent), np.asarray(seg_len), pl.arrays()["seg_offset"],
                              q.double().numpy(), k.double().numpy(), v.double().numpy(),
                              do.double().numpy(), 128 ** -0.5)
    errs = {n: rel_l2(t.float().cpu().numpy(), ref[n]) for n, t in (("dq", dq), ("dk", dk), ("dv", dv))}
    assert max(errs.values()) <= O_TOL, errs


@pytest.mark.parametrize("seed", range(3))
def test_bwd_random_forest_ragged_tiles(seed):
    parent, seg_len = _random_forest(seed, 14, 300)
    _check_bwd(parent, seg_len, 2, seed)


def test_bwd_deep_prefix_and_single_tokens():
    parent = np.array([-1, 0, 1, 0, 1, 2, 2], np.int32)
    seg_len = np.array([333, 200, 70, 129, 1, 257, 128], np.int64)
    _check_bwd(parent, seg_len, 2, 21)
    parent, seg_len = _random_forest(7, 40, 3)
    _check_bwd(parent, seg_len, 1, 22)


def test_bwd_nodewise_and_sharp_scores():
    parent, seg_len = _random_forest(8, 12, 200)
    _check_bwd(parent, seg_len, 2, 23, nodewise=True)
    parent, seg_len = _random_forest(9, 6, 400)
    _check_bwd(parent, seg_len, 2, 24, qscale=6.0)


@pytest.mark.parametrize("tree,H", [("fb64k_bf16", 4), ("wide256k_bf16", 4)])
def test_bwd_full_size_one_trajectory(tree, H):
    """Backward at full size with the loss on one whole trajectory (the one through the
    most segments among those of at most 1,600 rows, so that the fp64 oracle stays
    quick): dO is the seeded normal on the trajectory's rows and zero elsewhere.  A query
    of the trajectory sees exactly the trajectory's prefix, so its dq is the oracle's
    single-query backward over that prefix, and the dk, dv of each row of the trajectory
    are those single-query gradients summed over the trajectory's queries; compared row by
    row.  Every other row must get exactly zero.  This catches a key tile listed for the wrong query tile, a
    permuted view or a missing branch in the dK / dV sums."""
    from prefix_shared_chunkwise_gb300.api import attn_bwd
    from prefix_shared_chunkwise_gb300.synth import expand_rows
    parent, seg_len = make_tree(tree)
    pl = Plan(parent, seg_len, 64)
    pl.upload()
    C = pl.info["C"]
    so = pl.arrays()["seg_offset"]
    rows_all, ptr, leaves = expand_rows(parent, seg_len, so)
    depth = np.zeros(len(parent), np.int64)
    for i in range(len(parent)):
        depth[i] = 0 if parent[i] < 0 else depth[parent[i]] + 1
    lens = np.diff(ptr)
    t = int(np.argmax(np.where(lens <= 1600, depth[leaves], -1)))
    traj = rows_all[ptr[t]:ptr[t + 1]]
    g = torch.Generator(device="cuda").manual_seed(7)
    q, k, v, w = (torch.randn((C, H, 128), generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    idx = torch.as_tensor(traj, device="cuda")
    do = torch.zeros_like(w)
    do[idx] = w[idx]
    o, lse = attn_fwd(pl, q, k, v)
    dq, dk, dv = attn_bwd(pl, q, k, v, o, lse, do)
    assert pl.device_error() == 0
    f64 = lambda x: x.index_select(0, idx).double().cpu().numpy()
    n = len(traj)
    qt, kt, vt, dot_ = f64(q), f64(k), f64(v), f64(do)
    ref = dict(dq=np.zeros_like(qt), dk=np.zeros_like(kt), dv=np.zeros_like(vt))
    for r in range(n):           # query r of the trajectory sees its rows 0 .. r
        g_q, g_k, g_v = oat.attn_query_bwd(qt[r], kt[:r + 1], vt[:r + 1], dot_[r], 128 ** -0.5)
        ref["dq"][r] = g_q
        ref["dk"][:r + 1] += g_k
        ref["dv"][:r + 1] += g_v
    got = dict(dq=f64(dq), dk=f64(dk), dv=f64(dv))
    for name in ("dq", "dk", "dv"):
        assert rel_l2(got[name], ref[name]) <= O_TOL, (tree, name, rel_l2(got[name], ref[name]))
        # row by row: each row's gradient within a few bf16 roundings of its own size
        err = np.linalg.norm((got[name] - ref[name]).reshape(n, -1), axis=1)
        mag = np.linalg.norm(ref[name].reshape(n, -1), axis=1)
        scale_ = np.linalg.norm(ref[name]) / np.sqrt(n)
        assert np.all(err <= 2e-2 * mag + 1e-2 * scale_), (tree, name, int(np.argmax(err - 2e-2 * mag)))
    off = torch.ones(C, dtype=torch.bool, device="cuda")
    off[idx] = False
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert float(x[off].abs().max()) == 0.0, (tree, name, "gradient off the trajectory")


@pytest.mark.parametrize("tree,H", [("fb64k_bf16", 16), ("wide256k_bf16", 4)])
def test_forward_backward_repeatable(tree, H):
    """Repeated launches on a large forest give bit-identical o, lse, dq, dk, dv and record
    no device error: the producer/consumer barriers of the warp-specialised kernels never
    mix arrivals of different key tiles, which would show as run-to-run differences or as a
    wait running out."""
    from prefix_shared_chunkwise_gb300.api import attn_bwd
    parent, seg_len = make_tree(tree)
    pl = Plan(parent, seg_len, 64)
    pl.upload()
    C = pl.info["C"]
    g = torch.Generator(device="cuda").manual_seed(9)
    q, k, v, do = (torch.randn((C, H, 128), generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    first = None
    for _ in range(4):
        o, lse = attn_fwd(pl, q, k, v)
        dq, dk, dv = attn_bwd(pl, q, k, v, o, lse, do)
        assert pl.device_error() == 0
        outs = (o, lse, dq, dk, dv)
        if first is None:
            first = [t.clone() for t in outs]
            continue
        for a, b in zip(first, outs):
            assert torch.equal(a, b)
