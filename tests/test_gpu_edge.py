"""Degenerate and boundary cases of every kernel family against the oracle: a one-token
tree; single chains of exactly one chunk and one chunk plus a row (no fork, no replay);
attention over a one-row forest and with all-zero queries (every visible value weighted
equally); a width-1 (pointwise) convolution; log-probabilities with no semantic position
at all."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import attn as oat
from oracle import logprob as olp
from prefix_shared_chunkwise_gb300 import _lib
from prefix_shared_chunkwise_gb300.api import Plan, attn_bwd, attn_fwd, logprob_bwd, logprob_fwd
from tests._parity import rel_l2
from tests.test_gpu_conv import _run as conv_run
from tests.test_gpu_parity import TOL, _assert
from tests.test_gpu_parity import _run as kda_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


@pytest.mark.parametrize("L", [1, 64, 65])
def test_kda_single_chain_tc(L):
    errs = kda_run(np.array([-1], np.int32), np.array([L], np.int64), 64, 2, 128, "bf16", 31 + L,
                   backward=True, kernel=_lib.HARTS_KERNEL_TC)
    _assert(errs, TOL["bf16"])


@pytest.mark.parametrize("L", [1, 16, 17])
def test_kda_single_chain_fp32(L):
    errs = kda_run(np.array([-1], np.int32), np.array([L], np.int64), 16, 1, 32, "fp32", 41 + L,
                   backward=True, kernel=_lib.HARTS_KERNEL_SIMT)
    _assert(errs, TOL["fp32"])


def _attn(parent, seg_len, H, q, k, v, do):
    pl = Plan(parent, seg_len, 64)
    pl.upload()
    o, lse = attn_fwd(pl, q.cuda(), k.cuda(), v.cuda())
    dq, dk, dv = attn_bwd(pl, q.cuda(), k.cuda(), v.cuda(), o, lse, do.cuda())
    torch.cuda.synchronize()
    assert pl.device_error() == 0
    so = pl.arrays()["seg_offset"]
    f64 = lambda t: t.double().numpy()
    ref = oat.attn_forest(parent, seg_len, so, f64(q), f64(k), f64(v), 128 ** -0.5)
    g = oat.attn_forest_bwd(parent, seg_len, so, f64(q), f64(k), f64(v), f64(do), 128 ** -0.5)
    return o, lse, dict(o=rel_l2(o.float().cpu().numpy(), ref["o"]), lse=rel_l2(lse.cpu().numpy(), ref["lse"]),
                        dq=rel_l2(dq.float().cpu().numpy(), g["dq"]), dk=rel_l2(dk.float().cpu().numpy(), g["dk"]),
                        dv=rel_l2(dv.float().cpu().numpy(), g["dv"]))


def test_attention_one_row():
    g = torch.Generator().manual_seed(3)
    q, k, v, do = (torch.randn((1, 2, 128), generator=g).to(torch.bfloat16) for _ in range(4))
    o, lse, e = _attn(np.array([-1], np.int32), np.array([1], np.int64), 2, q, k, v, do)
    # one visible key: the output is that row's value, lse its scaled score
    assert torch.equal(o.cpu(), v)
    assert e["lse"] <= 1e-5 and e["dk"] <= 1e-2 and e["dv"] <= 1e-2


def test_attention_zero_queries_average_the_view():
    parent = np.array([-1, 0, 0, 1], np.int32)
    seg_len = np.array([70, 100, 3, 200], np.int64)
    C = int(seg_len.sum())
    g = torch.Generator().manual_seed(4)
    q = torch.zeros((C, 1, 128), dtype=torch.bfloat16)
    k, v, do = (torch.randn((C, 1, 128), generator=g).to(torch.bfloat16) for _ in range(3))
    o, lse, e = _attn(parent, seg_len, 1, q, k, v, do)
    assert max(e.values()) <= 1e-2, e
    # zero scores: lse = log(number of visible keys), exactly the view length
    pl = Plan(parent, seg_len, 64)
    so = pl.arrays()["seg_offset"]
    n_vis = np.array([len(oat.trajectory_prefix(parent, seg_len, so, r)) for r in range(C)])
    np.testing.assert_allclose(lse[:, 0].cpu().numpy(), np.log(n_vis), rtol=1e-6)


def test_conv_width_one_is_pointwise():
    parent = np.array([-1, 0, 0], np.int32)
    seg_len = np.array([5, 1, 9], np.int64)
    errs = conv_run(parent, seg_len, 64, 1, "fp32", "silu", True, 5)
    assert all(v <= 1e-5 for v in errs.values()), errs


def test_logprob_without_semantic_positions():
    C, V = 7, 64
    g = torch.Generator().manual_seed(6)
    z = torch.randn((C, V), generator=g) * 3
    row_ptr = torch.zeros(C + 1, dtype=torch.int32)
    empty = torch.zeros(0, dtype=torch.int32)
    logp, lse = logprob_fwd(z.cuda(), row_ptr.cuda(), empty.cuda(), empty.cuda())
    dz = logprob_bwd(z.cuda(), row_ptr.cuda(), empty.cuda(), empty.cuda(), lse, torch.zeros(0).cuda())
    torch.cuda.synchronize()
    _, lse_ref = olp.logprob_fwd(z.double().numpy(), np.zeros(0, np.int64), np.zeros(0, np.int64))
    assert logp.numel() == 0
    assert rel_l2(lse.cpu().numpy(), lse_ref) <= 1e-6
    assert float(dz.abs().max()) == 0.0                # no position: no gradient


def test_kda_rejects_misaligned_tensors():
    """Rows move 16 bytes at a time: a q (or dq) that does not start on a 16-byte boundary is
    refused with HARTS_EINVAL before anything is launched."""
    from prefix_shared_chunkwise_gb300.api import kda_fwd, kda_bwd
    from prefix_shared_chunkwise_gb300.synth import make_inputs
    pl = Plan(np.array([-1], np.int32), np.array([70], np.int64), 64)
    pl.upload()
    x = make_inputs(pl.info["C"], 2, 128, 128, "bf16", seed=5, device="cuda")
    bad = torch.empty(x["q"].numel() + 8, dtype=x["q"].dtype, device="cuda")[1:1 + x["q"].numel()].view(x["q"].shape)
    bad.copy_(x["q"])
    with pytest.raises(_lib.HartsError) as e:
        kda_fwd(pl, bad, x["k"], x["v"], x["g"], x["beta"])
    assert e.value.rc == -1          # HARTS_EINVAL
    cs = torch.empty(pl.chunk_state_bytes(2, 128, 128, 1) // 2, dtype=torch.bfloat16, device="cuda")
    o, states, _, cs = kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], chunk_states=cs)
    grads = {n: torch.empty_like(x["q"]) for n in ("dk", "dv", "dg")}
    grads["dq"] = bad
    grads["dbeta"] = torch.empty_like(x["beta"])
    with pytest.raises(_lib.HartsError) as e:
        kda_bwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], x["W"], states=states, chunk_states=cs, grads=grads)
    assert e.value.rc == -1          # HARTS_EINVAL
