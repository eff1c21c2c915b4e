"""Pins for the fp64 oracle against things other than itself: a library
attention routine (torch SDPA on CPU, fp64), closed forms, invariants,
hand-derived golden fixtures and brute force over subsets.

Sources: WISE (Attention Routing Stabilizes Early: Working-Set Inference for
Recurrent Language Models) §3 Eq 2, §5.1 Eqs 5-6, §5.2 Eqs 7-8, Appendix A.1
Eqs 12-13.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import wise_oracle as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(n, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((n, d)) * scale for _ in range(3)]


def _sdpa(q, k, v, mask=None, causal=False):
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float64))[None, None]
    out = F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=None if mask is None else torch.from_numpy(mask)[None, None],
                                         is_causal=causal)
    return out[0, 0].numpy()


# ----------------------------------------------------------------- Eq 2 ----

@pytest.mark.parametrize("n,d,block,seed", [(64, 16, 16, 0), (96, 8, 32, 1), (128, 32, 64, 2)])
def test_dense_attention_matches_library_sdpa(n, d, block, seed):
    q, k, v = _rand(n, d, seed, 1.5)
    o, lse, _ = W.causal_attention(q, k, v, block)
    ref = _sdpa(q, k, v, causal=True)
    assert np.max(np.abs(o - ref)) < 1e-12


def test_scale_override_matches_library_sdpa():
    q, k, v = _rand(64, 16, 5)
    o, _, _ = W.causal_attention(q, k, v, 16, scale=0.5)
    t = lambda x: torch.from_numpy(x)[None, None]
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True, scale=0.5)[0, 0].numpy()
    assert np.max(np.abs(o - ref)) < 1e-12


def test_lse_through_library_sdpa():
    # A_ij = exp(s_ij - LSE_i); with v_j = exp(-s_{i0 j}) the output of row i0
    # is (i0 + 1) exp(-LSE_i0), so LSE_i0 = ln(i0 + 1) - ln(O_i0).
    n, d, block = 48, 8, 16
    q, k, _ = _rand(n, d, 3)
    _, lse, _ = W.causal_attention(q, k, np.zeros((n, 1)), block)
    for i0 in (0, 5, 17, 47):
        s_row = (q[i0] @ k.T) / math.sqrt(d)
        v = np.exp(-s_row)[:, None]
        out = _sdpa(q, k, v, causal=True)
        assert abs(lse[i0] - (math.log(i0 + 1) - math.log(out[i0, 0]))) < 1e-10


def test_closed_form_uniform_attention():
    # Q = 0: every admissible key gets 1/(i+1); O_i is the prefix mean of V and LSE_i = ln(i+1).
    n, d, block = 64, 4, 16
    rng = np.random.default_rng(7)
    k, v = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    o, lse, r = W.causal_attention(np.zeros((n, d)), k, v, block, want_mass=True)
    pref = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    assert np.max(np.abs(o - pref)) < 1e-12
    assert np.max(np.abs(lse - np.log(np.arange(1, n + 1)))) < 1e-12
    # Eq 5 closed form with exact rationals: r_qb = (1/B) sum_{i in q} |b ∩ [0, i]| / (i + 1)
    nb = n // block
    for qb in range(nb):
        for b in range(nb):
            exact = sum(Fraction(max(0, min(i + 1, (b + 1) * block) - b * block), i + 1)
                        for i in range(qb * block, (qb + 1) * block)) / block
            assert abs(r[qb, b] - float(exact)) < 1e-12


def test_causality():
    n, d, block = 64, 8, 16
    q, k, v = _rand(n, d, 11)
    o1, _, _ = W.causal_attention(q, k, v, block)
    k2, v2 = k.copy(), v.copy()
    k2[40:] += 5.0
    v2[40:] -= 3.0
    o2, _, _ = W.causal_attention(q, k2, v2, block)
    assert np.array_equal(o1[:40], o2[:40])
    assert not np.allclose(o1[40:], o2[40:])


# ----------------------------------------------------------------- Eq 5 ----

@pytest.mark.parametrize("block", [8, 16])
def test_block_mass_through_library_sdpa(block):
    # sum_{j in b} A_ij is the SDPA output for a value matrix of block indicators.
    n, d = 64, 8
    q, k, _ = _rand(n, d, 21, 2.0)
    r = W.block_mass(q, k, block)
    nb = n // block
    ind = np.zeros((n, nb))
    for b in range(nb):
        ind[b * block:(b + 1) * block, b] = 1.0
    per_row = _sdpa(q, k, ind, causal=True)
    ref = per_row.reshape(nb, block, nb).mean(axis=1)
    assert np.max(np.abs(r - ref)) < 1e-12


def test_block_mass_rows_sum_to_one_and_causal():
    q, k, _ = _rand(128, 16, 4, 3.0)
    r = W.block_mass(q, k, 32)
    assert np.max(np.abs(r.sum(axis=1) - 1.0)) < 1e-12
    assert np.all(np.triu(r, 1) == 0.0)


def test_one_hot_mass_concentrates():
    # q = c e and the keys of one block = c e: that block takes nearly all mass.
    n, d, block, c = 64, 8, 16, 12.0
    q = np.zeros((n, d)); q[:, 0] = c
    k = np.zeros((n, d)); k[16:32, 0] = c
    r = W.block_mass(q, k, block)
    assert r[1, 1] > 0.99 and r[2, 1] > 0.99 and r[3, 1] > 0.99


# --------------------------------------------------------------- Eq 7/8 ----

def test_sparse_attention_matches_library_sdpa_with_mask():
    n, d, block = 96, 8, 16
    q, k, v = _rand(n, d, 8)
    rng = np.random.default_rng(0)
    nb = n // block
    support = [sorted(set(rng.choice(qb + 1, size=rng.integers(1, qb + 2), replace=False).tolist()) | {qb})
               for qb in range(nb)]
    o, lse, _ = W.causal_attention(q, k, v, block, support=support)
    mask = np.zeros((n, n), bool)
    for i in range(n):
        for j in range(i + 1):
            mask[i, j] = (j // block) in support[i // block]
    ref = _sdpa(q, k, v, mask=mask)
    assert np.max(np.abs(o - ref)) < 1e-12


def test_full_support_equals_dense_exactly():
    n, d, block = 64, 8, 16
    q, k, v = _rand(n, d, 9)
    nb = n // block
    o1, l1, _ = W.causal_attention(q, k, v, block)
    o2, l2, _ = W.causal_attention(q, k, v, block, support=[list(range(qb + 1)) for qb in range(nb)])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_diagonal_only_support_is_local_attention():
    n, d, block = 64, 8, 16
    q, k, v = _rand(n, d, 10)
    nb = n // block
    o, _, _ = W.causal_attention(q, k, v, block, support=[[qb] for qb in range(nb)])
    for qb in range(nb):
        s = slice(qb * block, (qb + 1) * block)
        ref = _sdpa(q[s], k[s], v[s], causal=True)
        assert np.max(np.abs(o[s] - ref)) < 1e-12


# ----------------------------------------------------------------- Eq 6 ----

def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _load("step_support_cases.json")["cases"], ids=lambda c: c["name"])
def test_step_support_golden(case):
    assert sorted(W.step_support(case["r"], case["q"], case["eta"])) == case["expected"]


@pytest.mark.parametrize("case", _load("working_set_cases.json")["cases"], ids=lambda c: str(c["flags"]))
def test_working_set_golden(case):
    g = _load("working_set_cases.json")
    masses = [np.array(m) for m in g["masses"]]
    rows = W.working_set(masses, g["eta"], case["flags"])
    assert rows == case["expected"]
    if "row_ptr" in case:
        rp, ci = W.support_to_csr(rows)
        assert rp.tolist() == case["row_ptr"] and ci.tolist() == case["col_idx"]


def _brute_min_cardinality(fx, target):
    n = len(fx)
    for size in range(1, n + 1):
        for sub in itertools.combinations(range(n), size):
            if sum(fx[b] for b in sub) >= target:
                return size, sub
    return None, None


@pytest.mark.parametrize("seed", range(40))
def test_step_support_brute_force(seed):
    rng = np.random.default_rng(seed)
    q = int(rng.integers(0, 8))
    r = rng.dirichlet(np.full(q + 1, 0.5))
    r = np.concatenate([r, rng.random(3)])          # inadmissible junk after q
    eta = float(rng.choice([0.5, 0.8, 0.9, 0.95]))
    got = W.step_support(r, q, eta)
    fx = [int(x) for x in W.to_fixed(r[:q + 1])]
    size, _ = _brute_min_cardinality(fx, int(W.to_fixed(eta)))
    assert all(b <= q for b in got)
    if size is None:
        assert got == set(range(q + 1))
        return
    assert len(got) == size
    # without near-ties the minimum-cardinality set reaching eta is the top-`size` set
    srt = sorted(fx, reverse=True)
    gaps = [srt[i] - srt[i + 1] for i in range(len(srt) - 1)]
    if all(g > int(W.to_fixed(2e-6)) for g in gaps):
        top = sorted(range(q + 1), key=lambda b: -fx[b])[:size]
        assert got == set(top)
        assert sum(fx[b] for b in got) >= int(W.to_fixed(eta))


@pytest.mark.parametrize("seed", range(20))
def test_step_support_monotone_in_eta(seed):
    rng = np.random.default_rng(100 + seed)
    q = int(rng.integers(1, 12))
    r = rng.dirichlet(np.full(q + 1, 0.3))
    prev = set()
    for eta in (0.3, 0.5, 0.7, 0.9, 0.99, 1.0 - 1e-9):
        cur = W.step_support(r, q, eta)
        assert prev <= cur
        prev = cur
    assert prev == set(range(q + 1)) or W.to_fixed(r).sum() < W.to_fixed(1 - 1e-9)


def test_eta_near_one_takes_every_block_with_mass():
    r = np.array([0.4, 0.3, 0.2, 0.1])
    assert W.step_support(r, 3, 1.0 - 1e-12) == {0, 1, 2, 3}


@pytest.mark.parametrize("seed", range(20))
def test_identification_margin_theorem(seed):
    # Appendix A.1: any perturbation with ||eps||_inf < Delta_q keeps the support.
    rng = np.random.default_rng(300 + seed)
    q = int(rng.integers(1, 10))
    r = rng.dirichlet(np.full(q + 1, 0.4))
    eta = 0.9
    delta = W.identification_margin(r, q, eta)
    if delta <= 1e-5:
        pytest.skip("degenerate draw")
    base = W.step_support(r, q, eta)
    for _ in range(50):
        eps = rng.uniform(-1, 1, q + 1) * delta * 0.9
        assert W.step_support(r + eps, q, eta) == base


def test_margin_is_tight_for_a_two_block_example():
    # r = (0.7, 0.3), eta = 0.6: k = 1; rank gap 0.2, delta+ = 0.1 -> Delta = 0.1
    assert abs(W.identification_margin([0.7, 0.3], 1, 0.6) - 0.1) < 1e-15
    assert W.step_support([0.7, 0.3], 1, 0.6) == {0}
    # a perturbation just above the margin changes the support
    assert W.step_support([0.7 - 0.11, 0.3 + 0.11], 1, 0.6) == {0, 1}


def test_select_multihead_layout():
    rng = np.random.default_rng(3)
    wdw, bsz, nh, nb = 2, 2, 3, 5
    m = np.zeros((wdw, bsz, nh, nb, nb))
    for idx in np.ndindex(wdw, bsz, nh):
        for qb in range(nb):
            m[idx][qb, :qb + 1] = rng.dirichlet(np.ones(qb + 1))
    rp, ci = W.select(m, 0.9)
    assert rp.shape == (bsz * nh * nb + 1,)
    for b in range(bsz):
        for h in range(nh):
            rows = W.working_set([m[t, b, h] for t in range(wdw)], 0.9)
            base = (b * nh + h) * nb
            for qb in range(nb):
                assert ci[rp[base + qb]:rp[base + qb + 1]].tolist() == rows[qb]


def test_retained_mass_and_density():
    r = np.array([[1.0, 0, 0], [0.6, 0.4, 0], [0.1, 0.2, 0.7]])
    rows = [[0], [0, 1], [2]]
    assert abs(W.retained_mass(r, rows) - (1.0 + 1.0 + 0.7) / 3) < 1e-15
    assert abs(W.block_density(rows) - 4 / 6) < 1e-15


# ------------------------------------------ App. B retained mass, App. C.2 Eq 24 ----

def test_retained_mass_rows_full_support_keeps_all_mass():
    """The full causal support keeps every row's whole mass (Eq 5 rows sum to
    one); the diagonal-only support keeps exactly r_qq."""
    q, k, _ = _rand(256, 32, seed=11, scale=2.0)
    r = W.block_mass(q, k, 64)
    nb = r.shape[0]
    full = W.retained_mass_rows(r, [list(range(qb + 1)) for qb in range(nb)])
    assert np.all(np.abs(full - 1.0) < 1e-12)
    diag = W.retained_mass_rows(r, [[qb] for qb in range(nb)])
    assert np.array_equal(diag, np.diag(r))


def test_jaccard_hand_example():
    """Rows {0}|{0}, {0,1}|{1}, {0,2}|{1,2}: intersections 1+1+1, unions 1+2+3."""
    inter, union, j = W.jaccard([[0], [0, 1], [0, 2]], [[0], [1], [1, 2]])
    assert (inter, union) == (3, 6) and j == 0.5


@pytest.mark.parametrize("seed", range(4))
def test_jaccard_against_boolean_matrices(seed):
    """Eq 24 through boolean (row, key block) incidence matrices; plus the
    invariants J(A, A) = 1, symmetry and |A and B| + |A or B| = |A| + |B|."""
    rng = np.random.default_rng(seed)
    rows, nb = 40, 24
    a = rng.random((rows, nb)) < 0.3
    b = rng.random((rows, nb)) < 0.4
    la = [np.nonzero(x)[0].tolist() for x in a]
    lb = [np.nonzero(x)[0].tolist() for x in b]
    inter, union, j = W.jaccard(la, lb)
    assert inter == int(np.sum(a & b)) and union == int(np.sum(a | b))
    assert inter + union == int(a.sum() + b.sum())
    assert W.jaccard(lb, la) == (inter, union, j)
    assert W.jaccard(la, la)[2] == 1.0
    assert W.jaccard([[] for _ in range(rows)], [[] for _ in range(rows)]) == (0, 0, 1.0)


# ----------------------------------------- App. B controls, Eqs 19-22 ----

def test_mass_matched_hand_example():
    """Masses (0.5, 0.3, 0.2) for q = 2; reference {1, 2} covers 0.5, which
    the single largest block already reaches: MassMatched = {0}. Reference {2}
    covers 0.2: again {0}. Reference {0, 1} covers 0.8: {0, 1}."""
    r = [0.5, 0.3, 0.2]
    assert W.mass_matched_support(r, 2, [1, 2]) == {0}
    assert W.mass_matched_support(r, 2, [2]) == {0}
    assert W.mass_matched_support(r, 2, [0, 1]) == {0, 1}
    assert W.mass_matched_support(r, 2, []) == set()


@pytest.mark.parametrize("seed", range(5))
def test_mass_matched_is_the_smallest_set_reaching_the_reference_mass(seed):
    """Brute force over every subset of a small row: the control has the
    minimum cardinality among sets whose mass reaches the reference's, it
    never has more blocks than the reference, and it reaches that mass."""
    rng = np.random.default_rng(seed)
    q = 6
    r = rng.dirichlet(np.ones(q + 1))
    ref = sorted(rng.choice(q + 1, size=3, replace=False).tolist())
    m = sum(r[b] for b in ref)
    got = W.mass_matched_support(r, q, ref)
    best = min(len(c) for k in range(q + 2) for c in itertools.combinations(range(q + 1), k)
               if sum(r[b] for b in c) >= m - 1e-12)
    assert len(got) == best <= len(ref)
    assert sum(r[b] for b in got) >= m - 1e-12


@pytest.mark.parametrize("seed", range(5))
def test_size_matched_is_numpy_top_k(seed):
    """Eq 22 against numpy's stable sort on (-mass, index) for distinct masses."""
    rng = np.random.default_rng(seed)
    q = 20
    r = rng.random(q + 1)
    for k in (0, 1, 5, q + 1, q + 5):
        want = set(np.lexsort((np.arange(q + 1), -r))[:k].tolist())
        assert W.size_matched_support(r, q, k) == want


def test_controls_with_ties_prefer_lower_indices():
    r = [0.25, 0.25, 0.25, 0.25]
    assert W.size_matched_support(r, 3, 2) == {0, 1}
    assert W.mass_matched_support(r, 3, [2, 3]) == {0, 1}
    rows = W.control_set(np.array([r] * 4), [[0], [0, 1], [1, 2], [2, 3]], "size", flags=W.SUPPORT_DIAG)
    assert rows == [[0], [0, 1], [0, 1, 2], [0, 1, 3]]
