"""GPU parity of the short convolution over the compact layout (harts_conv_fwd / _bwd)
against the fp64 oracle (oracle/conv.py): y, dx, dweight, dbias by relative L2,
<= 1e-5 for fp32, <= 1e-2 for bf16 inputs (weights and gradients of the weights are
fp32 in both)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import conv as oconv
from prefix_shared_chunkwise_gb300.api import Plan, conv_bwd, conv_fwd
from prefix_shared_chunkwise_gb300.synth import make_tree, WORKLOADS, expand_rows
from tests._parity import rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _forest(seed, n, max_len, fork_bias=0.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    parent = [-1]
    for i in range(1, n):
        if rng.random() < 0.08:
            parent.append(-1)
        elif rng.random() < fork_bias:
            parent.append(int(rng.integers(0, max(1, i // 4))))      # wide forks near the top
        else:
            parent.append(int(rng.integers(0, i)))
    seg_len = rng.integers(1, max_len + 1, size=n).astype(np.int64)
    return np.array(parent, np.int32), seg_len


def _run(parent, seg_len, ch, w, dtype, act, bias, seed, nodewise=False):
    pl = Plan(parent, seg_len, 64, nodewise=nodewise).upload()
    so = pl.arrays()["seg_offset"]
    C = pl.info["C"]
    g = torch.Generator().manual_seed(seed)
    td = torch.float32 if dtype == "fp32" else torch.bfloat16
    x = torch.randn((C, ch), generator=g).to(td)
    W = torch.randn((ch, w), generator=g) * 0.5
    b = torch.randn(ch, generator=g) if bias else None
    dy = torch.randn((C, ch), generator=g).to(td)
    y = conv_fwd(pl, x.cuda(), W.cuda(), None if b is None else b.cuda(), activation=act)
    dx, dW, db = conv_bwd(pl, x.cuda(), W.cuda(), None if b is None else b.cuda(), dy.cuda(), activation=act)
    torch.cuda.synchronize()
    x64, dy64 = x.double().numpy(), dy.double().numpy()
    b64 = None if b is None else b.double().numpy()
    ref = oconv.conv_forest(parent, seg_len, so, x64, W.double().numpy(), b64, act)
    assert ref["occ_diff"] == 0.0
    g_ref = oconv.conv_forest_bwd(parent, seg_len, so, x64, W.double().numpy(), b64, act, dy64)
    errs = {"y": rel_l2(y.float().cpu().numpy(), ref["y"]),
            "dx": rel_l2(dx.float().cpu().numpy(), g_ref["dx"]),
            "dweight": rel_l2(dW.cpu().numpy(), g_ref["dweight"])}
    if bias:
        errs["dbias"] = rel_l2(db.cpu().numpy(), g_ref["dbias"])
    return errs


@pytest.mark.parametrize("w", [1, 2, 4, 8])
@pytest.mark.parametrize("act", ["none", "silu"])
def test_conv_fp32(w, act):
    # segments of 1..6 rows: windows reach through several ancestors; forks everywhere
    parent, seg_len = _forest(100 + w, 40, 6)
    errs = _run(parent, seg_len, 64, w, "fp32", act, True, w)
    assert all(v <= 1e-5 for v in errs.values()), errs


@pytest.mark.parametrize("w", [4, 8])
def test_conv_bf16_wide_forks(w):
    parent, seg_len = _forest(7 + w, 60, 40, fork_bias=0.5)
    errs = _run(parent, seg_len, 256, w, "bf16", "silu", True, w)
    assert all(v <= 1e-2 for v in errs.values()), errs


def test_conv_nodewise_layout_and_no_bias():
    parent, seg_len = _forest(3, 30, 12)
    errs = _run(parent, seg_len, 32, 4, "fp32", "none", False, 3, nodewise=True)
    assert all(v <= 1e-5 for v in errs.values()), errs


def test_conv_full_size_sampled_trajectory():
    """Bench forest, channels = H * d of its q: the rows of one trajectory against the
    oracle run on that trajectory alone; with dy only on that trajectory's rows, dx on it
    equals the single-path gradient and is exactly zero elsewhere."""
    name = "wide256k_bf16"
    wl = WORKLOADS[name]
    parent, seg_len = make_tree(name)
    pl = Plan(parent, seg_len, wl.chunk).upload()
    C, ch, w = pl.info["C"], wl.H * wl.dk, 4
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn((C, ch), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((ch, w), generator=g, device="cuda") * 0.5)
    rows, ptr, leaves = expand_rows(parent, seg_len, pl.arrays()["seg_offset"])
    t = int(np.argmax(np.diff(ptr)))                 # the longest trajectory
    tr = rows[ptr[t]:ptr[t + 1]]
    idx = torch.as_tensor(tr, device="cuda")
    dy = torch.zeros_like(x)
    dy[idx] = torch.randn((len(tr), ch), generator=g, device="cuda").to(torch.bfloat16)
    y = conv_fwd(pl, x, W, None, activation="silu")
    dx, dW, _ = conv_bwd(pl, x, W, None, dy, activation="silu")
    torch.cuda.synchronize()
    hs = slice(0, 256)                               # a slice of channels for the fp64 check
    one = (np.array([-1], np.int32), np.array([len(tr)]), np.array([0]))
    xs = x[idx][:, hs].double().cpu().numpy()
    Ws = W[hs].double().cpu().numpy()
    ref = oconv.conv_forest(*one, xs, Ws, None, "silu")
    assert rel_l2(y[idx][:, hs].float().cpu().numpy(), ref["y"]) <= 1e-2
    gr = oconv.conv_forest_bwd(*one, xs, Ws, None, "silu", dy[idx][:, hs].double().cpu().numpy())
    assert rel_l2(dx[idx][:, hs].float().cpu().numpy(), gr["dx"]) <= 1e-2
    assert rel_l2(dW[hs].cpu().numpy(), gr["dweight"]) <= 1e-2
    off = torch.ones(C, dtype=torch.bool, device="cuda")
    off[idx] = False
    assert float(dx[off].abs().max()) == 0.0
