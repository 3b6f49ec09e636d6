"""The C++ planner behind harts_plan_calls against the planner oracle: call counts,
rounds, layout, replay gather lists, slots and consumers must be bit-exact.  Also:
the library loads and exports every symbol include/harts.h declares, and host-side
argument validation rejects malformed trees."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import plan_twin
from prefix_shared_chunkwise_gb300 import _lib
from prefix_shared_chunkwise_gb300.api import Plan
from prefix_shared_chunkwise_gb300.synth import WORKLOAD_ORDER, WORKLOADS, make_tree
from tests._golden import load_calls

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def test_library_exports_every_declared_symbol():
    hdr = open(os.path.join(ROOT, "include", "harts.h")).read()
    declared = set(re.findall(r"\b(harts_[a-z_0-9]+)\s*\(", hdr))
    assert declared == set(_lib.EXPORTED)
    L = ctypes.CDLL(_lib.SO_PATH)
    for name in declared:
        assert hasattr(L, name), name


KEYS = ["seg_offset", "seg_pos", "seg_seq", "round_seq_ptr", "cu_seqlens", "seq_round",
        "seq_first_seg", "seq_anchor", "seq_replay", "seq_src", "replay_ptr", "replay_idx",
        "seq_state_ptr", "state_seq", "state_pos", "state_cons_ptr", "state_cons",
        "root_cons_ptr", "root_cons"]


def _compare(parent, seg_len, B, nodewise=False):
    tw = plan_twin.plan(parent, seg_len, B, nodewise=nodewise)
    pl = Plan(parent, seg_len, B, nodewise=nodewise)
    ar = pl.arrays()
    info = pl.info
    assert info["n_rounds"] == tw["n_rounds"]
    assert info["n_seq"] == tw["n_seq"] and info["n_states"] == tw["n_states"]
    assert info["C"] == tw["C"] and info["S"] == tw["S"] and info["R"] == tw["R"]
    for k in KEYS:
        np.testing.assert_array_equal(ar[k], tw[k], err_msg=k)
    np.testing.assert_array_equal(ar["seg_tpre"], tw["Tpre"])
    np.testing.assert_array_equal(ar["seg_tin"], tw["Tin"])
    np.testing.assert_array_equal(ar["seg_ctop"], [-1] * len(parent) if nodewise else tw["ctop"])
    return pl, tw


@pytest.mark.parametrize("fixture", ["fig1_calls.txt", "fig2_calls.txt", "figC1_calls.txt"])
def test_planner_matches_oracle_on_figures(fixture):
    gd = load_calls(fixture)
    _compare(gd["parent"], gd["seg_len"], gd["chunk"])


def test_planner_matches_oracle_random_forests():
    rng = np.random.Generator(np.random.PCG64(21))
    for _ in range(400):
        n = int(rng.integers(1, 60))
        B = int(rng.choice([1, 4, 16, 64]))
        parent = np.array([-1 if (i == 0 or rng.random() < 0.08) else int(rng.integers(0, i))
                           for i in range(n)], np.int32)
        seg_len = rng.integers(1, 3 * B + 2, size=n).astype(np.int64)
        _compare(parent, seg_len, B)


def test_nodewise_planner_matches_oracle_random_forests():
    """HARTS_PLAN_NODEWISE: one sequence per segment, rounds = tree depth + 1, no replay,
    every handoff at the producer sequence's end; bit-exact against the twin."""
    rng = np.random.Generator(np.random.PCG64(22))
    for _ in range(300):
        n = int(rng.integers(1, 60))
        B = int(rng.choice([1, 4, 16, 64]))
        parent = np.array([-1 if (i == 0 or rng.random() < 0.08) else int(rng.integers(0, i))
                           for i in range(n)], np.int32)
        seg_len = rng.integers(1, 3 * B + 2, size=n).astype(np.int64)
        pl, tw = _compare(parent, seg_len, B, nodewise=True)
        depth = np.zeros(n, np.int64)
        for i in range(n):
            depth[i] = 0 if parent[i] < 0 else depth[parent[i]] + 1
        info = pl.info
        assert info["n_seq"] == n and info["R"] == 0 and info["n_rounds"] == depth.max() + 1
        ar = pl.arrays()
        seq_len = np.diff(ar["cu_seqlens"])
        # every slot sits at its producer sequence's end
        np.testing.assert_array_equal(ar["state_pos"], seq_len[ar["state_seq"]])


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_nodewise_planner_matches_oracle_on_workloads(name):
    parent, seg_len = make_tree(name)
    pl, tw = _compare(parent, seg_len, WORKLOADS[name].chunk, nodewise=True)
    assert pl.info["n_rounds"] >= 1


@pytest.mark.parametrize("flags", [4, _lib.HARTS_PLAN_NODEWISE | _lib.HARTS_PLAN_NOREPLAY])
def test_planner_rejects_unknown_or_conflicting_flags(flags):
    import ctypes
    h = ctypes.c_void_p()
    parent = np.array([-1, 0], np.int32)
    seg_len = np.array([3, 4], np.int64)
    rc = _lib.lib().harts_plan_calls(2, parent.ctypes.data_as(_lib._pi32), seg_len.ctypes.data_as(_lib._pi64),
                                     16, flags, ctypes.byref(h))
    assert rc == -1 and not h.value


def test_noreplay_planner_matches_oracle_random_forests():
    """HARTS_PLAN_NOREPLAY: the minimum-call continuations, side branches one round after
    their producer at the exact fork position, no replay; bit-exact against the twin."""
    rng = np.random.Generator(np.random.PCG64(23))
    for _ in range(300):
        n = int(rng.integers(1, 60))
        B = int(rng.choice([1, 4, 16, 64]))
        parent = np.array([-1 if (i == 0 or rng.random() < 0.08) else int(rng.integers(0, i))
                           for i in range(n)], np.int32)
        seg_len = rng.integers(1, 3 * B + 2, size=n).astype(np.int64)
        tw = plan_twin.plan(parent, seg_len, B, noreplay=True)
        pl = Plan(parent, seg_len, B, noreplay=True)
        ar = pl.arrays()
        info = pl.info
        assert info["flags"] == _lib.HARTS_PLAN_NOREPLAY and info["R"] == 0
        assert info["n_rounds"] == tw["n_rounds"] and info["n_seq"] == tw["n_seq"]
        for k in KEYS:
            np.testing.assert_array_equal(ar[k], tw[k], err_msg=k)
        np.testing.assert_array_equal(ar["seg_ctop"], tw["ctop"])
        # a side branch's source slot sits at its fork position in the producer sequence
        for i in range(info["n_seq"]):
            if ar["seq_src"][i] >= 0:
                j = ar["seq_src"][i]
                prod = ar["state_seq"][j]
                assert ar["seq_anchor"][prod] + ar["state_pos"][j] == ar["seq_anchor"][i]


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_planner_matches_oracle_on_workloads(name):
    parent, seg_len = make_tree(name)
    pl, tw = _compare(parent, seg_len, WORKLOADS[name].chunk)
    assert pl.info["n_rounds"] >= 1


def test_planner_linear_time_on_a_million_segments():
    import time
    rng = np.random.Generator(np.random.PCG64(1))
    n = 1_000_000
    parent = np.maximum(np.arange(n) - 1 - rng.integers(0, 4, size=n), -1).astype(np.int32)
    parent[0] = -1
    seg_len = rng.integers(1, 200, size=n).astype(np.int64)
    t = time.time()
    pl = Plan(parent, seg_len, 64)
    assert time.time() - t < 10.0
    assert pl.info["n_seq"] >= 1


@pytest.mark.parametrize("parent,seg_len,chunk", [
    ([0], [5], 16),            # parent not < index
    ([-1, 1], [5, 5], 16),     # parent not < index
    ([-1, 0], [5, 0], 16),     # zero-length segment
    ([-1], [5], 0),            # chunk < 1
])
def test_planner_rejects_malformed_input(parent, seg_len, chunk):
    with pytest.raises(_lib.HartsError) as e:
        Plan(np.array(parent), np.array(seg_len), chunk)
    assert e.value.rc == -1


def _attn_call(pl, H=2, d=128, dtype=_lib.HARTS_BF16, ptr=0x10000):
    a = _lib.AttnFwdArgs()
    a.H, a.d, a.dtype, a.scale = H, d, dtype, 0.1
    a.q = a.k = a.v = a.o = ptr or None
    return _lib.lib().harts_attn_fwd(pl.handle, ctypes.byref(a), None)


def test_attention_argument_checks_on_the_host():
    """harts_attn_fwd validates before it touches the device (no pointer is read):
    dtype / head dimension, heads, NULL and misaligned pointers, then the upload."""
    pl = Plan(np.array([-1, 0, 0], np.int32), np.array([5, 3, 4], np.int64), 64)
    assert _attn_call(pl, dtype=_lib.HARTS_FP32) == -2
    assert _attn_call(pl, d=64) == -2
    assert _attn_call(pl, H=0) == -1
    assert _attn_call(pl, ptr=0) == -1
    assert _attn_call(pl, ptr=0x10008) == -1
    assert _attn_call(pl) == -8                           # not uploaded


def test_attention_tables_bounded_for_deep_combs():
    """A comb (spine of 2000 segments, a one-token side branch at each) has ancestor
    views adding up to about 2 * 10^8 rows: the plan is built without attention tables
    and harts_attn_fwd reports HARTS_EOVERFLOW; a shallower comb keeps them."""
    def comb(n, L):
        parent = np.concatenate([[-1], np.arange(n - 1), np.arange(n)]).astype(np.int32)
        seg_len = np.concatenate([np.full(n, L), np.ones(n)]).astype(np.int64)
        return Plan(parent, seg_len, 64)
    assert _attn_call(comb(2000, 100)) == -3
    assert _attn_call(comb(200, 100)) == -8


def test_attention_backward_workspace_and_checks():
    pl = Plan(np.array([-1, 0, 0], np.int32), np.array([5, 3, 4], np.int64), 64)
    assert _lib.lib().harts_attn_bwd_workspace_bytes(pl.handle, 3) == 256      # 12 rows x 3 heads x 4 B, rounded
    assert _lib.lib().harts_attn_bwd_workspace_bytes(pl.handle, 0) == 0
    b = _lib.AttnBwdArgs()
    b.fwd.H, b.fwd.d, b.fwd.dtype, b.fwd.scale = 2, 128, _lib.HARTS_BF16, 0.1
    b.fwd.q = b.fwd.k = b.fwd.v = b.fwd.o = 0x10000
    assert _lib.lib().harts_attn_bwd(pl.handle, ctypes.byref(b), None) == -8   # not uploaded
    b.fwd.d = 64
    assert _lib.lib().harts_attn_bwd(pl.handle, ctypes.byref(b), None) == -2


def test_binding_rejects_undersized_buffers_before_the_abi():
    """The C ABI sees plain pointers, so the binding checks every buffer's shape or size
    against the plan first: a short chunk_states, states or workspace, or a row tensor of
    the wrong shape, raises ValueError and nothing is passed to the library."""
    import torch
    from prefix_shared_chunkwise_gb300.api import kda_bwd, kda_fwd
    from prefix_shared_chunkwise_gb300.synth import make_inputs
    pl = Plan(np.array([-1, 0, 0], np.int32), np.array([150, 90, 70], np.int64), 64)
    H, D = 2, 128
    assert pl.info["n_states"] >= 1
    x = make_inputs(pl.info["C"], H, D, D, "bf16", 0)
    need = pl.chunk_state_bytes(H, D, D, 1)
    short = torch.empty(need // 2 - 1, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="chunk_states"):
        kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], chunk_states=short)
    with pytest.raises(ValueError, match="states"):
        kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"],
                states=torch.empty((max(pl.info["n_states"] - 1, 0), H, D, D)))
    with pytest.raises(ValueError, match="shape"):
        kda_fwd(pl, x["q"], x["k"][:-1], x["v"], x["g"], x["beta"])
    cs = torch.empty(need // 2, dtype=torch.bfloat16)
    st = torch.empty((pl.info["n_states"], H, D, D))
    with pytest.raises(ValueError, match="workspace"):
        kda_bwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], x["W"], states=st, chunk_states=cs,
                workspace=torch.empty(16, dtype=torch.uint8))
