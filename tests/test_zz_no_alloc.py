"""harts_kda_bwd_static: the backward pass for callers that cannot hand the library any
device memory (a plugin inside a framework that owns the device pool, a step loop that
must not allocate).  Its scratch is the library's own file-scope device array; the
results must match harts_kda_bwd with a caller workspace, on two calls in a row (the
array keeps the previous call's contents).

So that a scratch entry read before it is written cannot go unnoticed, the array is
first left holding another problem's values (a different forest and seed), and the
reference run's caller workspace starts as all-ones bytes (NaN in every fp32 word)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from prefix_shared_chunkwise_gb300 import _lib
from prefix_shared_chunkwise_gb300.api import Plan, kda_bwd, kda_fwd
from prefix_shared_chunkwise_gb300.synth import fig1_tree, make_inputs
from tests._parity import rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _case(parent, seg_len, B, H, D, dtype, seed):
    pl = Plan(parent, seg_len, B).upload()
    x = make_inputs(pl.info["C"], H, D, D, dtype, seed, device="cuda")
    esz = 4 if dtype == "fp32" else 2
    cs = torch.empty(pl.chunk_state_bytes(H, D, D, 0 if dtype == "fp32" else 1) // esz,
                     dtype=x["q"].dtype, device="cuda")
    o, states, _, _ = kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], chunk_states=cs)
    return pl, x, states, cs


def _bwd(pl, x, states, cs, phase, workspace=None):
    g = kda_bwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], x["W"], states=states,
                chunk_states=cs, phase=phase, workspace=workspace)
    torch.cuda.synchronize()
    return {k: v.float().cpu().numpy() for k, v in g.items()}


def _poisoned_workspace(pl, H, D):
    return torch.full((max(pl.bwd_workspace_bytes(H, D, D), 256),), 0xFF, dtype=torch.uint8,
                      device="cuda")


_CASES = {
    "fig1_fp32": lambda: (*fig1_tree(), (16, 1, 32, "fp32", 0), 1e-5),
    "forest_bf16_d128": lambda: (np.array([-1, 0, 0, 1, 1, 2, -1, 6], np.int32),
                                 np.random.Generator(np.random.PCG64(41)).integers(10, 180, size=8)
                                 .astype(np.int64), (64, 2, 128, "bf16", 5), 1e-2),
}


@pytest.mark.parametrize("which", ["fig1_fp32", "forest_bf16_d128"])
def test_static_scratch_backward_matches_workspace_backward(which):
    parent, seg_len, args, tol = _CASES[which]()
    # leave the static array holding another problem's scratch: the other case, another seed
    other = "forest_bf16_d128" if which == "fig1_fp32" else "fig1_fp32"
    o_parent, o_len, o_args, _ = _CASES[other]()
    o_args = o_args[:4] + (o_args[4] + 100,)
    _bwd(*_case(o_parent, o_len, *o_args), "static")
    pl, x, states, cs = _case(parent, seg_len, *args)
    ref = _bwd(pl, x, states, cs, "all", workspace=_poisoned_workspace(pl, args[1], args[2]))
    for n in ref:
        assert np.isfinite(ref[n]).all(), (which, n)
    for call in range(2):
        got = _bwd(pl, x, states, cs, "static")
        for n in ref:
            assert rel_l2(got[n], ref[n]) <= tol, (which, call, n)
    assert pl.device_error() == 0


def test_static_scratch_rejects_oversized_problems():
    max_bytes = _lib.lib().harts_kda_bwd_static_max_bytes()
    parent = np.array([-1], np.int32)
    seg_len = np.array([64 * 200], np.int64)      # 200 chunks x 32 heads x 32 KB > 32 MiB
    pl, x, states, cs = _case(parent, seg_len, 64, 32, 128, "bf16", 6)
    assert pl.bwd_workspace_bytes(32, 128, 128) > max_bytes
    with pytest.raises(_lib.HartsError) as e:
        _bwd(pl, x, states, cs, "static")
    assert e.value.rc == -4
