"""GPU parity for no-replay plans (HARTS_PLAN_NOREPLAY: the pages' no-replay comparison;
side branches resume at the exact fork position from the producer's state there, which
the forward kernels take inside a chunk; no replay; forward only).

Outputs are compared with the fp64 token recurrence, which does not depend on the plan,
and the final state of every sequence with the fp64 chunkwise executor of the same plan
(pinned to the token recurrence by the CPU tests).  The handoff states themselves are
checked through the outputs of the sequences that start from them.  The backward
entry points refuse such plans."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import chunkwise, plan_twin
from prefix_shared_chunkwise_gb300 import _lib
from prefix_shared_chunkwise_gb300.api import Plan, kda_bwd, kda_fwd
from prefix_shared_chunkwise_gb300.synth import make_inputs
from tests._parity import rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _forest(seed, n, max_len):
    rng = np.random.Generator(np.random.PCG64(seed))
    parent = np.array([-1 if (i == 0 or rng.random() < 0.1) else int(rng.integers(0, i))
                       for i in range(n)], np.int32)
    seg_len = rng.integers(1, max_len + 1, size=n).astype(np.int64)
    return parent, seg_len


def _run(parent, seg_len, B, H, D, dtype, seed, kernel):
    pl = Plan(parent, seg_len, B, noreplay=True).upload()
    tw = plan_twin.plan(parent, seg_len, B, noreplay=True)
    info = pl.info
    assert info["R"] == 0 and info["flags"] == _lib.HARTS_PLAN_NOREPLAY
    ar = pl.arrays()
    # the point of the mode: handoffs inside chunks
    assert np.any(ar["state_pos"] % B != 0)
    x = make_inputs(info["C"], H, D, D, dtype, seed, device="cpu")
    dev = {k: v.cuda() for k, v in x.items()}
    fin = torch.empty((info["n_seq"], H, D, D), dtype=torch.float32, device="cuda")
    o, states, fin, _ = kda_fwd(pl, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                final_state=fin, kernel=kernel)
    torch.cuda.synchronize()
    assert pl.device_error() == 0
    f64 = {k: v.double().numpy() for k, v in x.items()}
    ref = oracle.kda_forest(parent, seg_len, tw["seg_offset"], f64["q"], f64["k"], f64["v"], f64["g"],
                            f64["beta"], chunk=B)
    _, fin_ref = chunkwise.tree_exec(tw, f64["q"], f64["k"], f64["v"], f64["g"], f64["beta"], B)
    return pl, dev, states, {"o": rel_l2(o.float().cpu().numpy(), ref["o"]),
                             "final": rel_l2(fin.cpu().numpy(), fin_ref)}


@pytest.mark.parametrize("B", [16, 64])
@pytest.mark.parametrize("seed", [1, 2])
def test_noreplay_fp32_forward(B, seed):
    parent, seg_len = _forest(seed * 10 + B, 16, 3 * B)
    _, _, _, errs = _run(parent, seg_len, B, 2, 32, "fp32", seed, _lib.HARTS_KERNEL_SIMT)
    assert all(v <= 1e-5 for v in errs.values()), errs


@pytest.mark.parametrize("seed", [3, 4])
def test_noreplay_bf16_d128_forward_tc(seed):
    # short and long segments: several forks inside one chunk of one sequence
    parent, seg_len = _forest(seed, 14, 150)
    _, _, _, errs = _run(parent, seg_len, 64, 2, 128, "bf16", seed, _lib.HARTS_KERNEL_TC)
    assert all(v <= 1e-2 for v in errs.values()), errs


def test_noreplay_backward_is_refused():
    parent, seg_len = _forest(9, 8, 100)
    pl, dev, states, _ = _run(parent, seg_len, 64, 2, 128, "bf16", 9, _lib.HARTS_KERNEL_TC)
    cs = torch.empty(pl.chunk_state_bytes(2, 128, 128, 1) // 2, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.HartsError) as e:
        kda_bwd(pl, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["W"], states=states,
                chunk_states=cs)
    assert e.value.rc == -2
