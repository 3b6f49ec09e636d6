"""The mbarrier protocols of the warp-specialized branch-attention kernels, checked on a
model (tests/_barrier_model.py) under many random schedules: copies landing late, tensor
products of two issuing threads drained in any interleaving, issue blocking on a full
queue, warps at different speeds, data-dependent waits (the forward's O rescale) and
empty second halves (dK / dV).  Under every schedule there must be no deadlock, every
wait must return on the phase it waits for, no phase of a barrier that several warps
arrive on may mix steps, and every read must see the version it expects.  Earlier
designs and planted mistakes must be rejected by some schedule, so that the checker is
not vacuous."""
import pytest

from tests._barrier_model import Sim, Violation, dkdv, dq, forward

SEEDS = 300


def _violations(build, seeds=SEEDS, **kw):
    found = []
    for seed in range(seeds):
        sim = Sim(seed, qmax=1 + seed % 3)
        build(sim, 1 + seed % 7, **kw)
        try:
            sim.run()
        except Violation as e:
            found.append((seed, str(e)))
    return found


@pytest.mark.parametrize("build", [forward, dq, dkdv], ids=["forward", "dq", "dkdv"])
def test_protocol_holds_under_random_schedules(build):
    assert _violations(build) == []


def test_rejects_one_p_ready_barrier_for_both_buffers():
    """The forward's first two-issuer design: one P-ready barrier shared by both P
    buffers lets a fast softmax warp arrive for tile j + 1 inside tile j's phase."""
    found = _violations(forward, per_buffer_pf=False)
    assert found and any("mixes steps" in m for _, m in found)


def test_rejects_final_wait_on_a_single_o_done_barrier():
    """Waiting for the last O on one barrier committed per tile can return a phase early
    when two products are still outstanding."""
    found = _violations(forward, shared_o_done=True)
    assert found and any("returned with" in m for _, m in found)


def test_rejects_dp_overwritten_before_every_thread_read_it():
    found = _violations(dq, wait_dp_read=False)
    assert found and any("read dP" in m for _, m in found)


def test_rejects_buffer_reused_before_its_update_completed():
    found = _violations(dkdv, wait_release=False)
    assert found and any("read S" in m for _, m in found)
