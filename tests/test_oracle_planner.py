"""Pins of the planner oracle (oracle/plan_twin.py) against the pages' worked
examples, closed forms and brute force."""
import numpy as np
import pytest

from oracle import plan_twin
from tests._golden import calls_of, load_calls


@pytest.mark.parametrize("fixture", ["fig1_calls.txt", "fig2_calls.txt", "figC1_calls.txt"])
def test_figure_call_listings(fixture):
    gd = load_calls(fixture)
    pl = plan_twin.plan(gd["parent"], gd["seg_len"], gd["chunk"])
    got = calls_of(pl, gd["names"])
    want = {r: seqs for r, seqs in gd["calls"].items()}
    # single-child chains contract to one sequence: compare chains, not segments
    assert got == want
    for nm, rho in gd["replay"].items():
        s = int(pl["seg_seq"][gd["names"].index(nm)])
        assert pl["seq_replay"][s] == rho
    assert pl["n_rounds"] == len(want)
    assert plan_twin.brute_force_calls(gd["parent"], gd["seg_len"], gd["chunk"]) == len(want)


def test_fig1_layout_and_replay_rows():
    gd = load_calls("fig1_calls.txt")
    pl = plan_twin.plan(gd["parent"], gd["seg_len"], 16)
    assert list(pl["cu_seqlens"]) == [0, 240, 310, 350]
    assert pl["R"] == 10 and pl["n_states"] == 2 and pl["C"] == 350 and pl["S"] == 600
    # C resumes at A's boundary 96 and replays A[96,100); E resumes at 144 and
    # replays B's rows for positions [144,150)
    assert list(pl["replay_idx"]) == [96, 97, 98, 99, 144, 145, 146, 147, 148, 149]
    assert list(pl["state_pos"]) == [96, 144] and list(pl["state_seq"]) == [0, 0]


def test_figC1_sources_share_boundary_state():
    gd = load_calls("figC1_calls.txt")
    pl = plan_twin.plan(gd["parent"], gd["seg_len"], 64)
    sb = pl["seg_seq"][gd["names"].index("B")]
    sc = pl["seg_seq"][gd["names"].index("C")]
    # both side sequences read the one state after P0 (position 128)
    assert pl["seq_src"][sb] == pl["seq_src"][sc] >= 0
    assert pl["state_pos"][pl["seq_src"][sb]] == 128


def _random_tree(rng, n, max_len):
    parent = [-1] + [int(rng.integers(-1 if rng.random() < 0.1 else 0, i)) for i in range(1, n)]
    seg_len = rng.integers(1, max_len + 1, size=n)
    return np.array(parent, np.int32), seg_len.astype(np.int64)


def _replay_closed_form(parent, seg_len, B):
    # R = sum over forks of (|children| - 1) * (e_v mod B)   (section 4.2)
    s, e = plan_twin.positions(parent, seg_len)
    nk = np.bincount(np.asarray(parent)[np.asarray(parent) >= 0], minlength=len(parent))
    return int(sum((nk[v] - 1) * (e[v] % B) for v in range(len(parent)) if nk[v] > 0))


def test_dp_equals_brute_force_small_trees():
    rng = np.random.Generator(np.random.PCG64(7))
    for trial in range(1500):
        n = int(rng.integers(1, 9))
        B = int(rng.choice([4, 8, 16]))
        parent, seg_len = _random_tree(rng, n, 3 * B)
        dp = plan_twin.min_calls(parent, seg_len, B)["calls"]
        pl = plan_twin.plan(parent, seg_len, B)
        assert pl["n_rounds"] == dp
        assert plan_twin.brute_force_calls(parent, seg_len, B) == dp, (parent, seg_len, B)


def test_replay_total_is_fixed():
    rng = np.random.Generator(np.random.PCG64(11))
    for _ in range(300):
        n = int(rng.integers(1, 40))
        B = int(rng.choice([4, 16, 64]))
        parent, seg_len = _random_tree(rng, n, 4 * B)
        pl = plan_twin.plan(parent, seg_len, B)
        assert pl["R"] == _replay_closed_form(parent, seg_len, B)


def test_strahler_closed_form_when_internal_segments_span_a_chunk():
    rng = np.random.Generator(np.random.PCG64(3))
    for _ in range(300):
        n = int(rng.integers(1, 60))
        B = 8
        parent, seg_len = _random_tree(rng, n, 20)
        nk = np.bincount(parent[parent >= 0], minlength=n)
        seg_len = np.where(nk > 0, np.maximum(seg_len, B), seg_len)
        st = plan_twin.strahler(parent)
        want = max(st[r] for r in range(n) if parent[r] < 0)
        assert plan_twin.plan(parent, seg_len, B)["n_rounds"] == want


@pytest.mark.parametrize("k", [0, 1, 2, 3, 4, 5])
def test_complete_binary_tree(k):
    parent = [-1]
    frontier = [0]
    for _ in range(k):
        nxt = []
        for v in frontier:
            for _ in range(2):
                parent.append(v)
                nxt.append(len(parent) - 1)
        frontier = nxt
    seg_len = np.full(len(parent), 70)
    assert plan_twin.plan(parent, seg_len, 64)["n_rounds"] == k + 1


def test_chain_and_early_forks_take_one_call():
    assert plan_twin.plan([-1, 0, 1, 2], [500, 300, 7, 90], 64)["n_rounds"] == 1
    rng = np.random.Generator(np.random.PCG64(5))
    for _ in range(100):
        parent, seg_len = _random_tree(rng, 12, 200)
        nk = np.bincount(parent[parent >= 0], minlength=12)
        s, e = plan_twin.positions(parent, seg_len)
        B = max(e[v] for v in range(12) if nk[v] > 0) + 1 if nk.any() else 4
        B = 1 << int(np.ceil(np.log2(B)))
        assert plan_twin.plan(parent, seg_len, B)["n_rounds"] == 1
