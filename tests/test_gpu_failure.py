"""Failure detection on the GPU without a fault: a device-side error is recorded in the
plan's error word and read back by the host (HARTS_EDEVICE), and the context stays usable.

* The bounded-wait path: harts_selftest_timeout waits on a barrier that nothing completes
  and gives up after ~1 ms, recording code 3 (timeout), as every kernel does when a wait
  runs out.
* A numerical precondition: a per-chunk decay span too large for the tensor-core kernels'
  reference-row factorisation records code 1 instead of producing silent overflow."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from prefix_shared_chunkwise_gb300 import _lib
from prefix_shared_chunkwise_gb300.api import Plan, attn_fwd, kda_fwd
from prefix_shared_chunkwise_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu

DEV_TIMEOUT, DEV_DECAY_RANGE = 3, 1


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _plan():
    pl = Plan(np.array([-1, 0, 0], np.int32), np.array([150, 90, 70], np.int64), 64)
    pl.upload()
    return pl


def test_wait_timeout_is_reported_and_context_survives():
    pl = _plan()
    assert pl.device_error() == 0
    rc = _lib.lib().harts_selftest_timeout(pl.handle, 2_000_000, None)
    assert rc == 0
    code = ctypes.c_int32(0)
    assert _lib.lib().harts_plan_device_error(pl.handle, None, ctypes.byref(code)) == -7   # HARTS_EDEVICE
    assert code.value == DEV_TIMEOUT
    assert pl.device_error() == 0                                  # the word was cleared
    # the context still runs kernels correctly afterwards
    C = pl.info["C"]
    q = torch.randn((C, 1, 128), device="cuda").to(torch.bfloat16)
    o, lse = attn_fwd(pl, q, q, q)
    torch.cuda.synchronize()
    assert pl.device_error() == 0 and torch.isfinite(o.float()).all()


def test_selftest_rejects_bad_arguments():
    pl = _plan()
    assert _lib.lib().harts_selftest_timeout(pl.handle, 0, None) == -1
    assert _lib.lib().harts_selftest_timeout(pl.handle, 200_000_000, None) == -1


def test_decay_span_out_of_range_is_reported():
    """g = -100 per channel and token: a 64-token chunk spans a log-decay of -6400, far
    beyond what the reference-row scaling keeps finite; the forward flags it."""
    pl = _plan()
    C = pl.info["C"]
    x = make_inputs(C, 1, 128, 128, "bf16", 0, device="cuda")
    x["g"] = torch.full_like(x["g"], -100.0)
    cs = torch.empty(pl.chunk_state_bytes(1, 128, 128, 1) // 2, dtype=torch.bfloat16, device="cuda")
    kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], chunk_states=cs, kernel=_lib.HARTS_KERNEL_TC)
    assert pl.device_error() == DEV_DECAY_RANGE
    # mild decay on the same plan runs clean again
    x = make_inputs(C, 1, 128, 128, "bf16", 1, device="cuda")
    kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], chunk_states=cs, kernel=_lib.HARTS_KERNEL_TC)
    assert pl.device_error() == 0
