"""GPU parity for node-wise plans (HARTS_PLAN_NODEWISE: one sequence per segment, one
round per tree level, every handoff at the producer sequence's exact end, which is
generally inside a chunk; the pages' "Node-wise LA" comparison point).

The same kernels run these plans.  Outputs and gradients are compared with the fp64
token recurrence, which does not depend on the plan; the end state of every sequence
(internal segments included) with the fp64 chunkwise executor of the same plan, which
the CPU tests pin to the token recurrence.  Relative L2: <= 1e-5 fp32, <= 1e-2 bf16."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import chunkwise, plan_twin
from prefix_shared_chunkwise_gb300 import _lib
from prefix_shared_chunkwise_gb300.api import Plan, kda_bwd, kda_fwd
from prefix_shared_chunkwise_gb300.synth import make_inputs
from tests._parity import leaf_order, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _forest(seed, n, B, max_len):
    rng = np.random.Generator(np.random.PCG64(seed))
    parent = np.array([-1 if (i == 0 or rng.random() < 0.1) else int(rng.integers(0, i))
                       for i in range(n)], np.int32)
    seg_len = rng.integers(1, max_len + 1, size=n).astype(np.int64)
    return parent, seg_len


def _run(parent, seg_len, B, H, D, dtype, seed, kernel):
    pl = Plan(parent, seg_len, B, nodewise=True).upload()
    tw = plan_twin.plan(parent, seg_len, B, nodewise=True)
    info = pl.info
    assert info["n_seq"] == len(parent) and info["R"] == 0
    x = make_inputs(info["C"], H, D, D, dtype, seed, device="cpu")
    dev = {k: v.cuda() for k, v in x.items()}
    leaves = leaf_order(parent)
    leaf_seq = [s for s, ch in enumerate(tw["seq_chain"]) if ch[-1] in leaves]
    gen = torch.Generator().manual_seed(seed + 78)
    dF = torch.zeros((info["n_seq"], H, D, D))
    dF[leaf_seq] = torch.randn((len(leaf_seq), H, D, D), generator=gen)
    elem = 4 if dtype == "fp32" else 2
    cs = torch.empty(pl.chunk_state_bytes(H, D, D, 0 if dtype == "fp32" else 1) // elem,
                     dtype=dev["q"].dtype, device="cuda")
    fin = torch.empty((info["n_seq"], H, D, D), dtype=torch.float32, device="cuda")
    o, states, fin, cs = kda_fwd(pl, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                 final_state=fin, chunk_states=cs, kernel=kernel)
    gr = kda_bwd(pl, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["W"], states=states,
                 chunk_states=cs, d_final=dF.cuda(), kernel=kernel)
    torch.cuda.synchronize()
    assert pl.device_error() == 0
    f64 = {k: v.double().numpy() for k, v in x.items()}
    dF_leaf = np.zeros((len(leaves), H, D, D))
    for s in leaf_seq:
        dF_leaf[leaves.index(tw["seq_chain"][s][-1])] = dF[s].double().numpy()
    ref = oracle.kda_forest(parent, seg_len, tw["seg_offset"], f64["q"], f64["k"], f64["v"], f64["g"],
                            f64["beta"], chunk=B, W=f64["W"], d_final=dF_leaf)
    _, fin_ref = chunkwise.tree_exec(tw, f64["q"], f64["k"], f64["v"], f64["g"], f64["beta"], B)
    errs = {"o": rel_l2(o.float().cpu().numpy(), ref["o"]),
            "final": rel_l2(fin.cpu().numpy(), fin_ref)}
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        errs[n] = rel_l2(gr[n].float().cpu().numpy(), ref[n])
    return errs, info


@pytest.mark.parametrize("B", [16, 64])
@pytest.mark.parametrize("seed", [1, 2])
def test_nodewise_fp32_fwd_bwd(B, seed):
    parent, seg_len = _forest(seed * 10 + B, 14, B, 3 * B)
    errs, info = _run(parent, seg_len, B, 2, 32, "fp32", seed, _lib.HARTS_KERNEL_SIMT)
    assert info["n_rounds"] >= 3
    bad = {k: v for k, v in errs.items() if not v <= 1e-5}
    assert not bad, errs


@pytest.mark.parametrize("seed", [3, 4])
def test_nodewise_bf16_d128_fwd_bwd_tc(seed):
    # segments from 1 row to several chunks: handoffs inside chunks, ragged tails
    parent, seg_len = _forest(seed, 12, 64, 200)
    errs, info = _run(parent, seg_len, 64, 2, 128, "bf16", seed, _lib.HARTS_KERNEL_TC)
    assert info["n_rounds"] >= 3
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, errs
