"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same
seeded inputs.  Relative L2 per output tensor: <= 1e-5 for fp32 workloads, <= 1e-2
for bf16 workloads.  Plans are compared bit-exactly elsewhere (test_plan_abi.py)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import plan_twin
from prefix_shared_chunkwise_gb300 import _lib
from prefix_shared_chunkwise_gb300.api import Plan, kda_bwd, kda_fwd
from prefix_shared_chunkwise_gb300.synth import WORKLOADS, fig1_tree, make_inputs, make_tree
from tests._parity import oracle_run, rel_l2

pytestmark = pytest.mark.gpu
TOL = {"fp32": 1e-5, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _run(parent, seg_len, B, H, D, dtype, seed, *, backward, kernel=_lib.HARTS_KERNEL_AUTO,
         h0=False, d_final=False, decay=1.0, scale=1.0, g_rows=None):
    pl = Plan(parent, seg_len, B).upload()
    info = pl.info
    C = info["C"]
    x = make_inputs(C, H, D, D, dtype, seed, device="cpu")
    if decay != 1.0:
        x["g"] = (x["g"].float() * decay).to(x["g"].dtype)
    if g_rows is not None:
        x["g"] = g_rows(x["g"].float()).to(x["g"].dtype)
    dev = {k: v.cuda() for k, v in x.items()}
    td = dev["q"].dtype
    h0_t = None
    if h0:
        gen = torch.Generator().manual_seed(seed + 77)
        h0_t = torch.randn((info["n_roots"], H, D, D), generator=gen) * 0.3
    dF = None
    if d_final:
        gen = torch.Generator().manual_seed(seed + 78)
        dF = torch.randn((info["n_seq"], H, D, D), generator=gen)
    cs = torch.empty(pl.chunk_state_bytes(H, D, D, 0 if dtype == "fp32" else 1) // (4 if dtype == "fp32" else 2),
                     dtype=td, device="cuda")
    fin = torch.empty((info["n_seq"], H, D, D), dtype=torch.float32, device="cuda")
    o, states, fin, cs = kda_fwd(pl, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                 final_state=fin, h0=None if h0_t is None else h0_t.cuda(),
                                 chunk_states=cs, scale=scale, kernel=kernel)
    out = dict(o=o, final=fin)
    if backward:
        dh0 = torch.empty_like(h0_t).cuda() if h0 else None
        gr = kda_bwd(pl, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["W"],
                     states=states, chunk_states=cs, d_final=None if dF is None else dF.cuda(),
                     h0=None if h0_t is None else h0_t.cuda(), dh0=dh0, scale=scale,
                     kernel=kernel)
        out.update(gr)
    torch.cuda.synchronize()
    assert pl.device_error() == 0
    ref = oracle_run(parent, seg_len, B, x, backward=backward,
                     h0=None if h0_t is None else h0_t.double().numpy(),
                     d_final_seq=None if dF is None else dF.double().numpy(), scale=scale)
    errs = {"o": rel_l2(out["o"].float().cpu().numpy(), ref["o"]),
            "final": rel_l2(out["final"].cpu().numpy(), ref["final_seq"])}
    if backward:
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            errs[n] = rel_l2(out[n].float().cpu().numpy(), ref[n])
        if h0:
            errs["dh0"] = rel_l2(out["dh0"].cpu().numpy(), ref["dh0"])
    return errs


def _assert(errs, tol):
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, f"rel L2 above {tol}: {bad} (all: {errs})"


def test_fig1_fp32_fwd_bwd():
    wl = WORKLOADS["fig1_fp32"]
    parent, seg_len = fig1_tree()
    errs = _run(parent, seg_len, wl.chunk, wl.H, wl.dk, "fp32", 0, backward=True)
    _assert(errs, TOL["fp32"])


@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("seed", [1, 2])
def test_random_forest_fp32_with_h0_and_dfinal(B, seed):
    rng = np.random.Generator(np.random.PCG64(seed * 10 + B))
    n = 14
    parent = np.array([-1 if (i == 0 or rng.random() < 0.15) else int(rng.integers(0, i))
                       for i in range(n)], np.int32)
    seg_len = rng.integers(1, 3 * B, size=n).astype(np.int64)
    errs = _run(parent, seg_len, B, 2, 32, "fp32", seed, backward=True, h0=True, d_final=True,
                decay=0.1, scale=0.8)
    _assert(errs, TOL["fp32"])


def test_fp32_d64_fwd_bwd_mild_decay():
    rng = np.random.Generator(np.random.PCG64(5))
    n = 9
    parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
    seg_len = rng.integers(1, 90, size=n).astype(np.int64)
    errs = _run(parent, seg_len, 32, 2, 64, "fp32", 3, backward=True, decay=0.05)
    _assert(errs, TOL["fp32"])


@pytest.mark.parametrize("kernel", [_lib.HARTS_KERNEL_SIMT, _lib.HARTS_KERNEL_AUTO])
def test_bf16_d128_forward_small_forest(kernel):
    rng = np.random.Generator(np.random.PCG64(8))
    n = 12
    parent = np.array([-1 if (i == 0 or rng.random() < 0.1) else int(rng.integers(0, i))
                       for i in range(n)], np.int32)
    seg_len = rng.integers(1, 200, size=n).astype(np.int64)
    errs = _run(parent, seg_len, 64, 4, 128, "bf16", 4, backward=False, kernel=kernel)
    _assert(errs, TOL["bf16"])


def test_bf16_d128_forward_mild_decay():
    rng = np.random.Generator(np.random.PCG64(9))
    n = 10
    parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
    seg_len = rng.integers(1, 300, size=n).astype(np.int64)
    errs = _run(parent, seg_len, 64, 2, 128, "bf16", 6, backward=False, decay=0.02)
    _assert(errs, TOL["bf16"])


def test_fwd16k_workload_forward_tc():
    """The 8-tree, 16K-token forward workload at full size, all heads, tensor-core path."""
    wl = WORKLOADS["fwd16k_bf16"]
    parent, seg_len = make_tree("fwd16k_bf16")
    errs = _run(parent, seg_len, wl.chunk, wl.H, wl.dk, "bf16", 1, backward=False,
                kernel=_lib.HARTS_KERNEL_TC)
    _assert(errs, TOL["bf16"])


def test_tc_forward_matches_simt_forward():
    """Both kernel families on identical inputs: the tensor-core forward stays within
    bf16 rounding of the exact fp32 CUDA-core forward."""
    rng = np.random.Generator(np.random.PCG64(12))
    n = 16
    parent = np.array([-1 if (i == 0 or rng.random() < 0.1) else int(rng.integers(0, i))
                       for i in range(n)], np.int32)
    seg_len = rng.integers(1, 260, size=n).astype(np.int64)
    pl = Plan(parent, seg_len, 64).upload()
    x = make_inputs(pl.info["C"], 4, 128, 128, "bf16", 11, device="cuda")
    outs = []
    for kern in (_lib.HARTS_KERNEL_SIMT, _lib.HARTS_KERNEL_TC):
        fin = torch.empty((pl.info["n_seq"], 4, 128, 128), device="cuda")
        o, _, fin, _ = kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], final_state=fin,
                               kernel=kern)
        outs.append((o.float().cpu().numpy(), fin.cpu().numpy()))
    torch.cuda.synchronize()
    assert pl.device_error() == 0
    assert rel_l2(outs[1][0], outs[0][0]) < 5e-3
    assert rel_l2(outs[1][1], outs[0][1]) < 5e-3


@pytest.mark.parametrize("decay", [1.0, 0.03])
def test_bf16_d128_fwd_bwd_small_forest_tc(decay):
    """Tensor-core forward + backward (state-carry and per-chunk gradient kernels)."""
    rng = np.random.Generator(np.random.PCG64(31))
    n = 14
    parent = np.array([-1 if (i == 0 or rng.random() < 0.1) else int(rng.integers(0, i))
                       for i in range(n)], np.int32)
    seg_len = rng.integers(1, 220, size=n).astype(np.int64)
    errs = _run(parent, seg_len, 64, 2, 128, "bf16", 21, backward=True, kernel=_lib.HARTS_KERNEL_TC,
                d_final=True, decay=decay)
    _assert(errs, TOL["bf16"])


def test_bf16_d128_fwd_bwd_with_h0_tc():
    rng = np.random.Generator(np.random.PCG64(32))
    n = 9
    parent = np.array([-1, 0, 0, 1, -1, 4, 4, 5, 2], np.int32)
    seg_len = rng.integers(20, 200, size=n).astype(np.int64)
    errs = _run(parent, seg_len, 64, 2, 128, "bf16", 22, backward=True, kernel=_lib.HARTS_KERNEL_TC,
                h0=True, decay=0.05, scale=0.7)
    _assert(errs, TOL["bf16"])


def test_tc_fwd_bwd_repeatable_on_64k_forest():
    """Forward + backward three times on the same inputs over the 64K-token forest: every
    output, the chunk records (R and T), the state slots and the final states are identical
    bit for bit (fixed summation orders, no atomics: a race between the staged copies, the
    products and the per-chunk phases would show as run-to-run differences; the records'
    tiny T entries show a race long before a bf16 output flips) and no device error is
    recorded."""
    parent, seg_len = make_tree("fb64k_bf16")
    pl = Plan(parent, seg_len, 64).upload()
    C, H = pl.info["C"], 4
    x = make_inputs(C, H, 128, 128, "bf16", 17, device="cuda")
    cs = torch.empty(pl.chunk_state_bytes(H, 128, 128, 1) // 2, dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((pl.info["n_seq"], H, 128, 128), dtype=torch.float32, device="cuda")
    names = ("o", "final", "records", "states", "dq", "dk", "dv", "dg", "dbeta")
    runs = []
    for _ in range(3):
        o, states, fin, cs = kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], final_state=fin,
                                     chunk_states=cs, kernel=_lib.HARTS_KERNEL_TC)
        torch.cuda.synchronize()
        fwd = [o.clone(), fin.clone(), cs.clone(), states.clone()]
        gr = kda_bwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], x["W"], states=states,
                     chunk_states=cs, kernel=_lib.HARTS_KERNEL_TC)
        torch.cuda.synchronize()
        assert pl.device_error() == 0
        runs.append(fwd + [gr[n].clone() for n in ("dq", "dk", "dv", "dg", "dbeta")])
    for r in (1, 2):
        for name, a, b in zip(names, runs[0], runs[r]):
            diff = (a != b) & ~(a.isnan() & b.isnan())
            assert not bool(diff.any()), (r, name, int(diff.sum()), diff.nonzero()[:4].tolist())


def _row_depth(parent, seg_len):
    """Trajectory position (depth in the tree) of every compact row, segments in id order."""
    depth0 = np.zeros(len(parent), np.int64)
    for i, p in enumerate(parent):
        if p >= 0:
            depth0[i] = depth0[p] + seg_len[p]
    return np.concatenate([depth0[i] + np.arange(seg_len[i]) for i in range(len(parent))])


def _late_decay(parent, seg_len, B, per_token):
    """g that leaves the first half of every B-row chunk (by trajectory position) almost
    undecayed and puts a strong decay of about `per_token` on each row of the second half,
    so that a chunk's total log-decay is about B / 2 * per_token, all of it late."""
    late = torch.from_numpy((_row_depth(parent, seg_len) % B) >= B // 2)

    def f(g):
        return torch.where(late[:, None, None], per_token + 0.1 * g, 0.01 * g)
    return f


def test_bf16_d128_fwd_bwd_late_decay_tc():
    """A decay of about e^-112 per chunk, all of it in the chunk's second half: every exponent
    of the half-total reference stays within e^+-56, so the tensor-core kernels compute the
    chunk (a middle-row reference would need e^112 and refuse it)."""
    parent = np.array([-1, 0, 0, 1, 1, -1], np.int32)
    seg_len = np.array([100, 90, 70, 40, 75, 150], np.int64)
    errs = _run(parent, seg_len, 64, 2, 128, "bf16", 23, backward=True, kernel=_lib.HARTS_KERNEL_TC,
                d_final=True, g_rows=_late_decay(parent, seg_len, 64, -3.5))
    _assert(errs, TOL["bf16"])


def test_fp32_d64_fwd_bwd_late_decay_simt():
    """The same e^-112 late decay per chunk on the exact fp32 CUDA-core kernels (B = 32)."""
    parent = np.array([-1, 0, 0, 1, 1, -1], np.int32)
    seg_len = np.array([100, 90, 70, 40, 75, 150], np.int64)
    errs = _run(parent, seg_len, 32, 2, 64, "fp32", 24, backward=True, kernel=_lib.HARTS_KERNEL_SIMT,
                d_final=True, g_rows=_late_decay(parent, seg_len, 32, -7.0))
    _assert(errs, TOL["fp32"])
