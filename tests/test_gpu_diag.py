"""Support diagnostics through the C ABI against the oracle: retained future
attention mass (WISE App. B, "Evaluation metrics") and the Eq 24 Jaccard
index of two supports (App. C.2). Counts are compared exactly, masses within
the rounding of a float32 result."""
import numpy as np
import pytest
import torch

import block_sparse_attention_causal_gb300 as wise
import workloads as wl
from oracle import wise_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def _masses(b, h, n, d, block, seed):
    rng = np.random.default_rng(seed)
    x = wl.bf16_round(rng.standard_normal((3, b, h, n, d)).astype(np.float32) * 2.0)
    q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
    _, _, m = wise.discover(q, k, v, block)
    return m


def _support(rows, b, h, n, d, block):
    return wise.support_from_lists(rows, b, h, n, d, block)


@pytest.mark.parametrize("shape", [(1, 2, 512, 64, 64), (2, 3, 1024, 128, 128), (1, 1, 128, 64, 128)])
def test_retained_mass_matches_oracle(shape):
    b, h, n, d, block = shape
    nb = n // block
    m = _masses(b, h, n, d, block, seed=n + h)
    rng = np.random.default_rng(7)
    rows = [r for _ in range(b * h) for r in wl.random_support(nb, 0.4, rng)]
    sup = _support(rows, b, h, n, d, block)
    got_rows, got_mean = wise.retained_mass(m, sup)
    wise.check_device()
    mh = m.cpu().numpy().reshape(b * h, nb, nb)
    ref = np.concatenate([O.retained_mass_rows(mh[i], rows[i * nb:(i + 1) * nb]) for i in range(b * h)])
    got = got_rows.cpu().numpy()
    assert np.max(np.abs(got - ref)) <= 1e-6
    ref_mean = ref.reshape(b, h * nb).mean(axis=1)
    assert np.max(np.abs(got_mean.cpu().numpy() - ref_mean)) <= 1e-6
    # the full causal support keeps the whole mass of every row
    full = _support([list(range(q + 1)) for _ in range(b * h) for q in range(nb)], b, h, n, d, block)
    fr, fm = wise.retained_mass(m, full)
    assert np.max(np.abs(fr.cpu().numpy() - 1.0)) <= 1e-5


@pytest.mark.parametrize("shape", [(1, 2, 512, 64, 64), (3, 2, 2048, 128, 128), (1, 1, 64 * 1024, 64, 64)])
def test_jaccard_matches_oracle_exactly(shape):
    b, h, n, d, block = shape
    nb = n // block
    rng = np.random.default_rng(nb + b)
    rows_a = [r for _ in range(b * h) for r in wl.random_support(nb, 0.3, rng)]
    rows_b = [r for _ in range(b * h) for r in wl.random_support(nb, 0.5, rng)]
    sa, sb = _support(rows_a, b, h, n, d, block), _support(rows_b, b, h, n, d, block)
    row_counts, counts, jac = wise.support_jaccard(sa, sb)
    wise.check_device()
    rc = row_counts.cpu().numpy()
    for i in range(len(rows_a)):
        inter, union, _ = O.jaccard([rows_a[i]], [rows_b[i]])
        assert (rc[i, 0], rc[i, 1]) == (inter, union)
    per = h * nb
    for bi in range(b):
        inter, union, j = O.jaccard(rows_a[bi * per:(bi + 1) * per], rows_b[bi * per:(bi + 1) * per])
        assert tuple(counts[bi].tolist()) == (inter, union)
        assert jac[bi].item() == j
    # a support against itself
    _, _, jself = wise.support_jaccard(sa, sa)
    assert torch.all(jself == 1.0)


def test_diagnostics_flag_malformed_rows():
    b, h, n, d, block = 1, 1, 256, 64, 64
    good = _support([[0], [0, 1], [2], [0, 3]], b, h, n, d, block)
    bad = _support([[0], [0, 3], [2], [0, 3]], b, h, n, d, block)  # block 3 is not admissible for q = 1
    m = torch.full((1, 1, 4, 4), 0.25, dtype=torch.float32, device="cuda")
    wise.retained_mass(m, bad)
    assert wise.device_status() == wise._lib.WISE_ERR_BAD_SUPPORT
    rc, counts, jac = wise.support_jaccard(good, bad)
    assert wise.device_status() == wise._lib.WISE_ERR_BAD_SUPPORT
    # the inadmissible entry is skipped: row 1 of `bad` counts as {0}
    assert tuple(counts[0].tolist()) == (5, 6)
