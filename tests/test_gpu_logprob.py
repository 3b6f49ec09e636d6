"""GPU parity of the compact-to-semantic log-probabilities (harts_logprob_fwd / _bwd)
against the fp64 oracle (oracle/logprob.py) on the same (cast) inputs: logp and lse
within 1e-5 relative L2 (fp32 outputs from fp32 or bf16 logits), dlogits within 1e-5
(fp32) / 1e-2 (bf16 output)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import logprob as olp
from prefix_shared_chunkwise_gb300.api import Plan, logprob_bwd, logprob_fwd, semantic_map
from prefix_shared_chunkwise_gb300.synth import make_tree
from tests._parity import rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _csr(sem_row, C):
    row_ptr = np.zeros(C + 1, np.int32)
    np.add.at(row_ptr, sem_row + 1, 1)
    row_ptr = np.cumsum(row_ptr).astype(np.int32)
    row_sem = np.argsort(sem_row, kind="stable").astype(np.int32)
    return row_ptr, row_sem


def _run(z, sem_row, target, g, dtype):
    C, V = z.shape
    row_ptr, row_sem = _csr(sem_row, C)
    td = torch.float32 if dtype == "fp32" else torch.bfloat16
    zt = torch.as_tensor(z, dtype=torch.float32).to(td)
    dev = lambda a: torch.as_tensor(a, device="cuda")
    logp, lse = logprob_fwd(zt.cuda(), dev(row_ptr), dev(row_sem), dev(target.astype(np.int32)))
    dz = logprob_bwd(zt.cuda(), dev(row_ptr), dev(row_sem), dev(target.astype(np.int32)), lse,
                     dev(g.astype(np.float32)))
    torch.cuda.synchronize()
    z64 = zt.double().numpy()
    lam, lse_ref = olp.logprob_fwd(z64, sem_row, target)
    dz_ref = olp.logprob_bwd(z64, sem_row, target, g.astype(np.float32).astype(np.float64))
    return {"logp": rel_l2(logp.cpu().numpy(), lam), "lse": rel_l2(lse.cpu().numpy(), lse_ref),
            "dlogits": rel_l2(dz.float().cpu().numpy(), dz_ref)}


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_random_rows_with_repeated_targets(dtype):
    rng = np.random.default_rng(1)
    C, V, S = 97, 1000, 400
    z = rng.standard_normal((C, V)) * 4
    sem_row = rng.integers(0, C - 5, size=S)             # the last rows have no position
    target = rng.integers(0, 12, size=S)                 # many repeats of the same label
    g = rng.standard_normal(S)
    errs = _run(z, sem_row, target, g, dtype)
    assert errs["logp"] <= 1e-5 and errs["lse"] <= 1e-5, errs
    assert errs["dlogits"] <= (1e-5 if dtype == "fp32" else 1e-2), errs


def test_forest_semantic_map_full_vocabulary():
    """A forest's own semantic map (shared rows carry several positions with distinct
    labels) at the pages' vocabulary size."""
    parent, seg_len = make_tree("fig1_fp32")
    pl = Plan(parent, seg_len, 64)
    sem_row, row_ptr, row_sem = semantic_map(pl)
    C, S, V = pl.info["C"], len(sem_row), 157_184
    assert S == pl.info["S"] and S > C
    rng = np.random.default_rng(2)
    z = rng.standard_normal((C, V)).astype(np.float32) * 3
    target = rng.integers(0, V, size=S)
    g = rng.standard_normal(S)
    errs = _run(z, sem_row.astype(np.int64), target, g, "bf16")
    assert errs["logp"] <= 1e-5 and errs["lse"] <= 1e-5 and errs["dlogits"] <= 1e-2, errs


def test_full_size_sampled_rows():
    """The 64K-token forest at V = 157,184 (bf16 logits, 20.6 GB): sampled compact rows'
    lse and all their semantic positions' logp against the oracle; every row's gradient
    sums to zero over the vocabulary up to the rounding of its bf16 entries."""
    parent, seg_len = make_tree("fb64k_bf16")
    pl = Plan(parent, seg_len, 64)
    sem_row, row_ptr, row_sem = semantic_map(pl)
    C, S, V = pl.info["C"], len(sem_row), 157_184
    g = torch.Generator(device="cuda").manual_seed(3)
    z = (torch.randn((C, V), generator=g, device="cuda") * 3).to(torch.bfloat16)
    target = torch.randint(0, V, (S,), generator=g, device="cuda", dtype=torch.int32)
    dl = torch.randn(S, generator=g, device="cuda")
    rp, rs = torch.as_tensor(row_ptr, device="cuda"), torch.as_tensor(row_sem, device="cuda")
    logp, lse = logprob_fwd(z, rp, rs, target)
    dz = logprob_bwd(z, rp, rs, target, lse, dl)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0], rng.integers(0, C, size=20)]))
    tgt = target.cpu().numpy()
    for c in rows:
        zc = z[int(c)].double().cpu().numpy()[None, :]
        pos = row_sem[row_ptr[c]:row_ptr[c + 1]]
        lam, lse_ref = olp.logprob_fwd(zc, np.zeros(len(pos), np.int64), tgt[pos])
        assert abs(float(lse[int(c)]) - lse_ref[0]) <= 1e-5 * abs(lse_ref[0])
        if len(pos):
            assert rel_l2(logp[torch.as_tensor(pos, device="cuda")].cpu().numpy(), lam) <= 1e-5
            ref = olp.logprob_bwd(zc, np.zeros(len(pos), np.int64), tgt[pos], dl.cpu().numpy()[pos])
            assert rel_l2(dz[int(c)].float().cpu().numpy(), ref[0]) <= 1e-2
    # each row's gradient sums to zero up to the bf16 rounding of its entries
    dzf = dz.float()
    assert float((dzf.sum(dim=1).abs() / dzf.abs().sum(dim=1).clamp_min(1e-30)).max()) < 1e-2
