"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Gates: O max-abs <= 1e-2 (float32 output; bf16 output adds half a bf16 ulp
of the reference), LSE <= 1e-3, block masses <= 1e-3, support CSR bit-exact
when both sides select from the same masses. Inputs are seeded and rounded
to bf16 before either side sees them.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_causal_gb300 as wise
import workloads as wl
from oracle import wise_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

O_TOL, LSE_TOL, MASS_TOL = 1e-2, 1e-3, 1e-3


def _bf16_inputs(b, h, n, d, seed, scale=1.0, planted=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((3, b, h, n, d)).astype(np.float32) * np.float32(scale)
    if planted:
        # a shared direction in Q and in the keys of a few blocks, so masses are far from uniform
        for bi in range(b):
            for hi in range(h):
                u = rng.standard_normal(d).astype(np.float32) * 2.0
                x[0, bi, hi] += u
                for blk in rng.choice(max(1, n // 64), size=min(planted, max(1, n // 64)), replace=False):
                    x[1, bi, hi, blk * 64:(blk + 1) * 64] += u
    x = wl.bf16_round(x)
    t = torch.from_numpy(x).to(torch.bfloat16).cuda()
    return x, t[0].contiguous(), t[1].contiguous(), t[2].contiguous()


def _oracle_discover(x, block):
    return O.discover(x[0].astype(np.float64), x[1].astype(np.float64), x[2].astype(np.float64), block)


def _assert_close(name, got, ref, tol):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{name}: non-finite pattern differs"
    err = np.max(np.abs(got[fin] - ref[fin])) if fin.any() else 0.0
    assert err <= tol, f"{name}: max abs error {err:.3e} > {tol:.1e}"
    return err


SHAPES = [  # (batch, heads, n, d, block)
    (1, 2, 256, 64, 64),
    (1, 1, 64, 64, 64),      # a single block; one partial 128-row tile
    (2, 1, 192, 96, 64),     # odd number of 64-blocks: ragged last tile
    (1, 2, 384, 128, 128),   # odd number of 128-row tiles
    (1, 1, 640, 128, 128),
    (1, 1, 512, 96, 128),
    (1, 3, 128, 64, 128),    # nb = 1
    (2, 2, 320, 128, 64),
    (1, 1, 1024, 64, 128),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_discover_parity(shape):
    b, h, n, d, blk = shape
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=n + d + blk, scale=1.5, planted=2)
    o, lse, mass = wise.discover(q, k, v, blk, out_dtype=torch.float32)
    wise.check_device()
    o_ref, lse_ref, r_ref = _oracle_discover(x, blk)
    _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
    _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)
    _assert_close("mass", mass.cpu().numpy(), r_ref, MASS_TOL)
    iu = np.triu_indices(n // blk, 1)
    assert np.all(mass.cpu().numpy()[..., iu[0], iu[1]] == 0.0)


def test_discover_bf16_output_within_half_ulp():
    x, q, k, v = _bf16_inputs(1, 2, 512, 128, seed=5, scale=2.0, planted=3)
    o, _, _ = wise.discover(q, k, v, 128, want_mass=False)
    o_ref, _, _ = _oracle_discover(x, 128)
    got = o.float().cpu().numpy()
    # half a bf16 ulp of the reference value
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_ref), 1e-30))) - 8)
    assert np.all(np.abs(got - o_ref) <= O_TOL + half_ulp)


def test_discover_lse_optional_and_no_mass():
    x, q, k, v = _bf16_inputs(1, 1, 256, 64, seed=7)
    o1, lse1, _ = wise.discover(q, k, v, 64, want_mass=False, want_lse=False, out_dtype=torch.float32)
    o2, lse2, m2 = wise.discover(q, k, v, 64, out_dtype=torch.float32)
    assert lse1 is None and torch.equal(o1, o2)


def test_workload_tiny_discover():
    cfg = wl.CONFIGS["tiny"]
    x = wl.step_inputs(cfg, 0)
    q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
    o, lse, mass = wise.discover(q, k, v, cfg.block, out_dtype=torch.float32)
    o_ref, lse_ref, r_ref = _oracle_discover(x, cfg.block)
    _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
    _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)
    _assert_close("mass", mass.cpu().numpy(), r_ref, MASS_TOL)


# ------------------------------------------------------------ select (Eq 6)

def _random_masses(w, b, h, nb, seed, ties=False):
    rng = np.random.default_rng(seed)
    m = np.zeros((w, b, h, nb, nb), np.float32)
    for idx in np.ndindex(w, b, h):
        for q in range(nb):
            r = rng.dirichlet(np.full(q + 1, 0.3)).astype(np.float32)
            if ties and q >= 3:
                kind = rng.integers(0, 3)
                if kind == 0:      # exact ties among a few blocks
                    pick = rng.choice(q + 1, size=min(3, q + 1), replace=False)
                    r[pick] = r[pick].mean()
                elif kind == 1:    # near ties within the 1e-6 tolerance
                    pick = rng.choice(q + 1, size=2, replace=False)
                    r[pick[1]] = r[pick[0]] + np.float32(4e-7)
            m[idx][q, :q + 1] = r
    return m


@pytest.mark.parametrize("case", [(2, 1, 2, 4, 64, 0.9), (3, 2, 3, 32, 128, 0.9), (4, 1, 2, 64, 128, 0.95),
                                  (1, 1, 1, 1, 128, 0.5), (2, 1, 1, 300, 64, 0.8), (4, 1, 1, 1024, 64, 0.95)],
                         ids=lambda c: "W%d_B%d_H%d_nb%d_blk%d_eta%s" % c)
@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("flags", [0, 3])
def test_select_bit_exact_on_same_masses(case, ties, flags):
    w, b, h, nb, blk, eta = case
    m = _random_masses(w, b, h, nb, seed=nb * 7 + w, ties=ties)
    sup = wise.select_support(torch.from_numpy(m).cuda(), nb * blk, 64, blk, eta, flags)
    wise.check_device()
    rp_ref, ci_ref = O.select(m.astype(np.float64), eta, flags)
    rp = sup.row_ptr.cpu().numpy()
    assert np.array_equal(rp, rp_ref)
    assert np.array_equal(sup.col_idx.cpu().numpy()[:rp[-1]], ci_ref)
    assert int(sup.nnz.item()) == len(ci_ref)
    _check_tile_order(sup)


def _check_tile_order(sup):
    lib = wise._lib.load()
    desc = wise._lib.make_desc(sup.batch, sup.heads, sup.seq_len, sup.head_dim, sup.block)
    units = int(lib.wise_schedule_units(desc))
    order = sup.tile_order.cpu().numpy()[:units]
    assert sorted(order.tolist()) == list(range(units))
    # a work unit is one 128-row query tile of one (batch, head); its cost is
    # the number of blocks its query blocks list. When the ranking fits in one
    # CTA's shared memory (200 KB) every unit is ranked together: heaviest
    # first, ties by unit index.
    qpu = 128 // sup.block
    nb = sup.seq_len // sup.block
    # the ranking CTA holds one cost per unit and, per cost value, a counter
    # for each of its segments (32, or fewer when 33 counters per value take
    # more than 100 KB, down to 8) plus a total
    nc = nb * qpu + 1
    segs = 32
    while segs > 8 and nc * 4 * (segs + 1) > 100 * 1024:
        segs //= 2
    if (units + (segs + 1) * nc) * 4 <= 200 * 1024:
        counts = np.diff(sup.row_ptr.cpu().numpy().astype(np.int64)).reshape(sup.batch * sup.heads, nb)
        tiles = units // (sup.batch * sup.heads)
        pad = np.zeros((sup.batch * sup.heads, tiles * qpu), np.int64)
        pad[:, :nb] = counts
        cost = pad.reshape(sup.batch * sup.heads, tiles, qpu).sum(-1).reshape(-1)
        expect = np.argsort(-cost, kind="stable")
        assert np.array_equal(order, expect)


def _tiny_mass_rows(nb, seed, lo_exp, hi_exp):
    """One head whose rows hold mass 0.5 in block 0 and masses between
    2^lo_exp and 2^hi_exp (below 2^-29, where the 2^-52 fixed point of Eq 6's
    cumulative sum rounds) elsewhere, a few of them exactly halfway between
    two fixed-point steps, (2j + 1) * 2^-53, where rounding goes to even."""
    rng = np.random.default_rng(seed)
    m = np.zeros((1, 1, 1, nb, nb), np.float32)
    for q in range(nb):
        r = np.exp2(rng.uniform(lo_exp, hi_exp, q + 1)).astype(np.float32)
        halfway = rng.random(q + 1) < 0.2
        r[halfway] = ((2 * rng.integers(1, 1 << (hi_exp + 52), halfway.sum()) + 1) * 2.0 ** -53).astype(np.float32)
        r[0] = 0.5
        m[0, 0, 0, q, :q + 1] = r
    return m


@pytest.mark.parametrize("nb", [20, 40, 300])
@pytest.mark.parametrize("lo_exp,hi_exp,eta", [(-36, -30, 0.5 + 2.0 ** -31), (-40, -36, 0.5 + 2.0 ** -32)])
def test_select_bit_exact_where_the_fixed_point_rounds(nb, lo_exp, hi_exp, eta):
    """The cut falls among masses the 2^-52 fixed point rounds (ties to
    even): the number of blocks Eq 6 takes depends on every one of them, so
    any difference in the rounding between the kernel and the oracle changes
    the CSR. The second range needs more than 24 values to reach eta, which
    takes the kernel's search path instead of its one-value-at-a-time path."""
    m = _tiny_mass_rows(nb, seed=100 * nb - lo_exp, lo_exp=lo_exp, hi_exp=hi_exp)
    sup = wise.select_support(torch.from_numpy(m).cuda(), nb * 64, 64, 64, eta, 0)
    wise.check_device()
    rp_ref, ci_ref = O.select(m.astype(np.float64), eta, 0)
    rp = sup.row_ptr.cpu().numpy()
    assert np.array_equal(rp, rp_ref)
    assert np.array_equal(sup.col_idx.cpu().numpy()[:rp[-1]], ci_ref)


def _structured_mass_rows(nb, seed):
    """Rows whose Eq 6 cut falls in large groups of equal or near-equal
    masses, or near the smallest masses the selection kernel decides on the
    masses' float keys alone (a cut v* within the 1e-6 tie tolerance of
    2^-29): uniform rows (every admissible block equal), rows whose 40
    heaviest blocks lie within 8e-7 of each other, rows with one block at 0.5
    and the rest near 2^-20 or 2^-19, and rows with a mass above 1."""
    rng = np.random.default_rng(seed)
    m = np.zeros((2, 1, 1, nb, nb), np.float32)
    for w in range(2):
        for q in range(nb):
            kind = (q + w) % 5
            n = q + 1
            if kind == 0:
                r = np.full(n, 1.0 / n)
            elif kind == 1:
                r = rng.dirichlet(np.full(n, 0.3)) * 0.05
                top = rng.choice(n, size=min(n, 40), replace=False)
                r[top] = 0.95 / len(top) + rng.uniform(-4e-7, 4e-7, len(top))
            elif kind == 2:
                r = 2.0 ** -20 * (1 + rng.uniform(0, 2 ** -10, n))
                r[0] = 0.5
            elif kind == 3:
                r = 2.0 ** -19 * (1 + rng.uniform(0, 0.5, n))
                r[0] = 0.5
            else:
                r = rng.dirichlet(np.full(n, 0.5))
                r[rng.integers(n)] = 3.0
            m[w, 0, 0, q, :n] = r.astype(np.float32)
    return m


@pytest.mark.parametrize("nb,eta", [(64, 0.9), (300, 0.9), (300, 0.5 + 2.0 ** -12), (1024, 0.95)])
def test_select_bit_exact_on_tie_groups_and_cut_boundaries(nb, eta):
    """Cuts inside large exact- and near-tie groups (where the near group is
    only partly taken, lowest index first) and cuts at the edge of the range
    the kernel decides on float keys: the CSR must equal the oracle's."""
    m = _structured_mass_rows(nb, seed=nb)
    sup = wise.select_support(torch.from_numpy(m).cuda(), nb * 64, 64, 64, eta, 3)
    wise.check_device()
    rp_ref, ci_ref = O.select(m.astype(np.float64), eta, 3)
    rp = sup.row_ptr.cpu().numpy()
    assert np.array_equal(rp, rp_ref)
    assert np.array_equal(sup.col_idx.cpu().numpy()[:rp[-1]], ci_ref)


def test_select_on_gpu_masses_matches_oracle_select():
    cfg = wl.CONFIGS["tiny"]
    masses = []
    for t in cfg.window_steps:
        x = wl.step_inputs(cfg, t)
        q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
        masses.append(wise.discover(q, k, v, cfg.block)[2])
    m = torch.stack(masses).contiguous()
    sup = wise.select_support(m, cfg.seq_len, cfg.head_dim, cfg.block, cfg.eta)
    rp_ref, ci_ref = O.select(m.cpu().numpy().astype(np.float64), cfg.eta)
    assert np.array_equal(sup.row_ptr.cpu().numpy(), rp_ref)
    assert np.array_equal(sup.col_idx.cpu().numpy()[:len(ci_ref)], ci_ref)


# ------------------------------------------------------------ sparse (Eq 8)

@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("density", [0.15, 0.5])
def test_sparse_parity_random_support(shape, density):
    b, h, n, d, blk = shape
    nb = n // blk
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=3 * n + d, scale=1.5, planted=2)
    rng = np.random.default_rng(n + blk)
    rows = []
    for _ in range(b * h):
        rows.extend(wl.random_support(nb, density, rng, sink=bool(rng.integers(0, 2)), diag=bool(rng.integers(0, 2))))
    sup = wise.support_from_lists(rows, b, h, n, d, blk)
    o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False)
    wise.check_device()
    rp, ci = O.support_to_csr(rows)
    o_ref, lse_ref = O.sparse(x[0].astype(np.float64), x[1].astype(np.float64), x[2].astype(np.float64), blk, rp, ci)
    _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
    _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)


def test_sparse_full_support_bitwise_equals_discover():
    b, h, n, d, blk = 1, 2, 768, 128, 128
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=11, scale=1.5, planted=2)
    nb = n // blk
    rows = [list(range(qb + 1)) for _ in range(b * h) for qb in range(nb)]
    sup = wise.support_from_lists(rows, b, h, n, d, blk)
    o1, l1 = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False)
    o2, l2, _ = wise.discover(q, k, v, blk, want_mass=False, out_dtype=torch.float32)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_sparse_empty_rows_give_zero_and_neg_inf():
    b, h, n, d, blk = 1, 1, 512, 64, 128
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=2)
    rows = [[0], [], [0, 2], []]
    sup = wise.support_from_lists(rows, b, h, n, d, blk)
    o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False)
    wise.check_device()
    on, ln = o.cpu().numpy(), lse.cpu().numpy()
    assert np.all(on[0, 0, 128:256] == 0) and np.all(np.isneginf(ln[0, 0, 128:256]))
    assert np.all(on[0, 0, 384:] == 0) and np.all(np.isneginf(ln[0, 0, 384:]))
    rp, ci = O.support_to_csr(rows)
    o_ref, _ = O.sparse(x[0].astype(np.float64), x[1].astype(np.float64), x[2].astype(np.float64), blk, rp, ci)
    _assert_close("O", on, o_ref, O_TOL)


def test_sparse_malformed_support_is_flagged_not_faulted():
    b, h, n, d, blk = 1, 1, 512, 64, 128
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=4)
    rows = [[0], [1, 0], [0, 7, 2], [-3, 3]]  # descending, above the diagonal, negative
    sup = wise.support_from_lists(rows, b, h, n, d, blk)
    wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False)
    assert wise.device_status() == wise._lib.WISE_ERR_BAD_SUPPORT
    assert wise.device_status() == wise._lib.WISE_OK  # the word is cleared by the read


# ------------------------------------------------------------ trajectories

def _run_trajectory(cfg, heads=None):
    """GPU trajectory: t_d discovery steps (masses on the window), one
    selection, late steps. Returns (support, per-step GPU outputs)."""
    masses, outs = [], {}
    for t in range(cfg.t_d):
        x = wl.step_inputs(cfg, t, heads=heads)
        q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
        o, lse, m = wise.discover(q, k, v, cfg.block, want_mass=t in cfg.window_steps, out_dtype=torch.float32)
        if m is not None:
            masses.append(m)
        outs[t] = (x, o.cpu().numpy(), lse.cpu().numpy(), None if m is None else m.cpu().numpy())
    sup = wise.select_support(torch.stack(masses).contiguous(), cfg.seq_len, cfg.head_dim, cfg.block, cfg.eta)
    wise.check_device()
    return sup, outs


# End-to-end supports (GPU masses vs oracle masses) may differ only in rows
# whose Eq 13 identification margin is below this. The measured mass error
# is about 1.5e-7, so the allowance is some 70 times that error; every excused
# row is counted and printed.
FLIP_MARGIN = 1e-5


def _assert_support_matches(sup_rows, oracle_masses, cfg, head_rows, label=""):
    """CSR rows from GPU masses vs the oracle's selection from oracle masses;
    a difference is allowed only where Eq 13's margin is below FLIP_MARGIN.
    Returns the number of rows that differ."""
    ref_rows = O.working_set(oracle_masses, cfg.eta)
    flips = 0
    for qb, (got, ref) in enumerate(zip(head_rows, ref_rows)):
        if got != ref:
            margin = min(O.identification_margin(m[qb], qb, cfg.eta) for m in oracle_masses)
            assert margin < FLIP_MARGIN, \
                f"support of query block {qb} differs with margin {margin:.2e}: {got} vs {ref}"
            flips += 1
    print(f"{cfg.name} {label}: {flips} of {len(ref_rows)} support rows differ from the oracle's, "
          f"each with Eq 13 margin < {FLIP_MARGIN:.0e}")
    return flips


def test_tiny_trajectory_end_to_end():
    cfg = wl.CONFIGS["tiny"]
    sup, outs = _run_trajectory(cfg)
    rows = sup.to_lists()
    nb = cfg.n_blocks
    for bi in range(cfg.batch):
        for hi in range(cfg.heads):
            om = []
            for t in cfg.window_steps:
                x = outs[t][0]
                _, _, r = O.causal_attention(*(x[i, bi, hi].astype(np.float64) for i in range(3)), cfg.block,
                                             want_mass=True)
                om.append(r)
                _assert_close("mass", outs[t][3][bi, hi], r, MASS_TOL)
            base = (bi * cfg.heads + hi) * nb
            _assert_support_matches(rows[base:base + nb], om, cfg, rows[base:base + nb])
    # late steps over the selected support
    rp = sup.row_ptr.cpu().numpy()
    ci = sup.col_idx.cpu().numpy()
    for t in range(cfg.t_d, cfg.steps):
        x = wl.step_inputs(cfg, t)
        q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
        o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32)
        o_ref, lse_ref = O.sparse(x[0].astype(np.float64), x[1].astype(np.float64), x[2].astype(np.float64),
                                  cfg.block, rp, ci)
        _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
        _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)


# Sampled (batch, head) slices of the full-size configurations: both ends of
# a single-batch workload, and one head in every batch element of the batch-4
# workload, spread over the heads.
_FULL_SAMPLES = {"8k_b4": [(0, 0), (1, 7), (2, 19), (3, 31)]}


def _sample_heads(cfg):
    return _FULL_SAMPLES.get(cfg.name, [(0, 0), (cfg.batch - 1, cfg.heads - 1)])


def _sample_query_blocks(nb, seed):
    """Both ends, the middle and a few seeded others: the late-step work order
    ranks units by listed blocks, so these fall early, mid and late in it."""
    rng = np.random.default_rng(seed)
    picks = {0, 1, nb // 3, nb // 2, (2 * nb) // 3, nb - 2, nb - 1}
    picks |= set(int(x) for x in rng.choice(nb, size=min(nb, 4), replace=False))
    return sorted(x for x in picks if 0 <= x < nb)


def _run_trajectory_kept(cfg, keep):
    """As _run_trajectory, keeping only the (batch, head) slices in `keep`
    on the host (the full-size workloads hold GBs per step)."""
    masses, kept = [], {}
    for t in range(cfg.t_d):
        x = wl.step_inputs(cfg, t)
        q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
        o, lse, m = wise.discover(q, k, v, cfg.block, want_mass=t in cfg.window_steps, out_dtype=torch.float32)
        if m is not None:
            masses.append(m)
        kept[t] = {(bi, hi): (x[:, bi, hi].copy(), o[bi, hi].cpu().numpy(), lse[bi, hi].cpu().numpy(),
                              None if m is None else m[bi, hi].cpu().numpy()) for bi, hi in keep}
        del x, q, k, v, o, lse
    sup = wise.select_support(torch.stack(masses).contiguous(), cfg.seq_len, cfg.head_dim, cfg.block, cfg.eta)
    wise.check_device()
    return sup, kept


@pytest.mark.slow
@pytest.mark.parametrize("name", ["4k", "8k_b4", "16k_h40_d96", "4k_b32"])
def test_full_size_config_sampled(name):
    """Full-size configuration, in the launch configuration the benchmark
    times; checked on sampled (batch, head) slices and query blocks. 4k_b32 is
    the 4k workload with blocks of 32 (the pages' default granularity): 1,024
    work units, so most are claimed from the launch-wide counter. 8k_b4 is the
    batch-4 workload (8,192 work units, 16 steps, t_d = 4, eta = 0.95)."""
    cfg = wl.CONFIGS["4k"].replace(name=name, block=32) if name == "4k_b32" else wl.CONFIGS[name]
    sample = _sample_heads(cfg)
    sup, kept = _run_trajectory_kept(cfg, sample)
    rows = sup.to_lists()
    nb = cfg.n_blocks
    qbs = _sample_query_blocks(nb, seed=nb)
    for bi, hi in sample:
        om = []
        for t in cfg.window_steps:
            xs_, o_gpu, lse_gpu, m_gpu = kept[t][(bi, hi)]
            xs = [xs_[i].astype(np.float64) for i in range(3)]
            o_ref, lse_ref, r = O.causal_attention(*xs, cfg.block, want_mass=True)
            om.append(r)
            _assert_close("mass", m_gpu, r, MASS_TOL)
            _assert_close("O", o_gpu, o_ref, O_TOL)
            _assert_close("LSE", lse_gpu, lse_ref, LSE_TOL)
        base = (bi * cfg.heads + hi) * nb
        _assert_support_matches(rows[base:base + nb], om, cfg, rows[base:base + nb], label=f"(b{bi}, h{hi})")
    t = cfg.steps - 1
    x = wl.step_inputs(cfg, t)
    q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
    o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32)
    wise.check_device()
    o, lse = o.cpu().numpy(), lse.cpu().numpy()
    for bi, hi in sample:
        base = (bi * cfg.heads + hi) * nb
        supp = rows[base:base + nb]
        xs = [x[i, bi, hi].astype(np.float64) for i in range(3)]
        o_ref, lse_ref, _ = O.causal_attention(*xs, cfg.block, support=supp, query_blocks=qbs)
        for qb in qbs:
            s = slice(qb * cfg.block, (qb + 1) * cfg.block)
            _assert_close("O", o[bi, hi, s], o_ref[s], O_TOL)
            _assert_close("LSE", lse[bi, hi, s], lse_ref[s], LSE_TOL)


@pytest.mark.slow
def test_4k_every_head_and_query_block():
    """The 4k workload with nothing sampled: every (head, query block) of the
    last discovery step (O, LSE, masses) and of the last late step (O, LSE)
    against the oracle, in the launch configuration the benchmark times. A
    unit computed wrongly anywhere in the persistent work order fails here."""
    cfg = wl.CONFIGS["4k"]
    sup, outs = _run_trajectory(cfg)
    nb = cfg.n_blocks
    rows = sup.to_lists()
    x, o_gpu, lse_gpu, m_gpu = outs[cfg.t_d - 1]
    oracle_masses = {}
    for bi in range(cfg.batch):
        for hi in range(cfg.heads):
            for t in cfg.window_steps:
                xt = outs[t][0]
                xs = [xt[i, bi, hi].astype(np.float64) for i in range(3)]
                o_ref, lse_ref, r = O.causal_attention(*xs, cfg.block, want_mass=True)
                oracle_masses.setdefault((bi, hi), []).append(r)
                _assert_close("mass", outs[t][3][bi, hi], r, MASS_TOL)
                if t == cfg.t_d - 1:
                    _assert_close("O", o_gpu[bi, hi], o_ref, O_TOL)
                    _assert_close("LSE", lse_gpu[bi, hi], lse_ref, LSE_TOL)
    flips = 0
    for (bi, hi), om in oracle_masses.items():
        base = (bi * cfg.heads + hi) * nb
        flips += _assert_support_matches(rows[base:base + nb], om, cfg, rows[base:base + nb], label=f"(b{bi}, h{hi})")
    print(f"4k: {flips} support rows of {cfg.batch * cfg.heads * nb} excused in total")
    x = wl.step_inputs(cfg, cfg.steps - 1)
    q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
    o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32)
    wise.check_device()
    o, lse = o.cpu().numpy(), lse.cpu().numpy()
    for bi in range(cfg.batch):
        for hi in range(cfg.heads):
            base = (bi * cfg.heads + hi) * nb
            xs = [x[i, bi, hi].astype(np.float64) for i in range(3)]
            o_ref, lse_ref, _ = O.causal_attention(*xs, cfg.block, support=rows[base:base + nb])
            _assert_close("O", o[bi, hi], o_ref, O_TOL)
            _assert_close("LSE", lse[bi, hi], lse_ref, LSE_TOL)


def _full_causal_support(cfg, device="cuda"):
    """Every admissible block listed, with a shuffled work order (a valid
    permutation, as wise_validate_schedule checks)."""
    nb, bh = cfg.n_blocks, cfg.batch * cfg.heads
    per_row = np.concatenate([np.arange(q + 1, dtype=np.int32) for q in range(nb)])
    counts = np.tile(np.arange(1, nb + 1, dtype=np.int64), bh)
    row_ptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    col_idx = np.tile(per_row, bh)
    lib = wise._lib.load()
    desc = wise._lib.make_desc(cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block)
    units = int(lib.wise_schedule_units(desc))
    order = np.random.default_rng(units).permutation(units).astype(np.int32)
    assert lib.wise_validate_schedule(desc, order.ctypes.data) == wise._lib.WISE_OK
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return wise.Support(t(row_ptr), t(col_idx), t(order), t(np.array([len(col_idx)], np.int32)),
                        cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["4k", "8k_b4", "16k_h40_d96", "sweep_32k"])
def test_full_support_bitwise_equals_discover_at_full_size(name):
    """A property that holds at any size covers every work unit of the
    full-size launches: with every admissible block listed, Eq 8 is Eq 2, so
    the late-step kernel (units taken in a shuffled order, most of them
    claimed from the launch-wide counter) must reproduce the dense kernel bit
    for bit, O and LSE, in every row."""
    cfg = wl.CONFIGS[name]
    x = wl.step_inputs(cfg, 0)
    q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
    del x
    sup = _full_causal_support(cfg)
    o1, l1 = wise.sparse(q, k, v, sup, out_dtype=torch.float32)
    o2, l2, _ = wise.discover(q, k, v, cfg.block, want_mass=False, out_dtype=torch.float32)
    wise.check_device()
    assert torch.equal(l1, l2)
    assert torch.equal(o1, o2)


@pytest.mark.slow
def test_long_context_32k_sampled():
    """The longest context-sweep configuration (32K, 256 blocks), in the
    launch configuration the benchmark times: every launch completes without a
    device timeout, and sampled heads and query blocks match the oracle. The
    oracle evaluates only the sampled query blocks, which Eqs 2, 5, 6 and 8
    allow because each query row (and each row of masses) is independent."""
    cfg = wl.CONFIGS["sweep_32k"]
    sample = [(0, 0), (0, cfg.heads - 1)]
    nb = cfg.n_blocks
    qbs = _sample_query_blocks(nb, seed=nb)
    kept, masses = {}, []
    for t in range(cfg.t_d):
        x = wl.step_inputs(cfg, t)
        q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
        o, _, m = wise.discover(q, k, v, cfg.block, want_mass=t in cfg.window_steps, out_dtype=torch.float32)
        if m is not None:
            masses.append(m)
        kept[t] = {(bi, hi): (x[:, bi, hi].copy(), o[bi, hi].cpu().numpy(),
                              None if m is None else m[bi, hi].cpu().numpy()) for bi, hi in sample}
        del x, q, k, v, o
    sup = wise.select_support(torch.stack(masses).contiguous(), cfg.seq_len, cfg.head_dim, cfg.block, cfg.eta)
    wise.check_device()
    rows = sup.to_lists()
    for bi, hi in sample:
        step_masses = []
        for t in cfg.window_steps:
            xs, o_gpu, m_gpu = kept[t][(bi, hi)]
            o_ref, _, r = O.causal_attention(*(xs[i].astype(np.float64) for i in range(3)), cfg.block,
                                             query_blocks=qbs, want_mass=True)
            for qb in qbs:
                s = slice(qb * cfg.block, (qb + 1) * cfg.block)
                _assert_close("O", o_gpu[s], o_ref[s], O_TOL)
                _assert_close("mass", m_gpu[qb], r[qb], MASS_TOL)
            step_masses.append(r)
        base = (bi * cfg.heads + hi) * nb
        flips = 0
        for qb in qbs:
            ref = sorted(set().union(*(O.step_support(r[qb], qb, cfg.eta) for r in step_masses)) | {0, qb})
            if rows[base + qb] != ref:
                margin = min(O.identification_margin(r[qb], qb, cfg.eta) for r in step_masses)
                assert margin < FLIP_MARGIN, f"support of query block {qb} differs with margin {margin:.2e}"
                flips += 1
        print(f"sweep_32k (b{bi}, h{hi}): {flips} of {len(qbs)} sampled support rows differ from the oracle's, "
              f"each with Eq 13 margin < {FLIP_MARGIN:.0e}")
    x = wl.step_inputs(cfg, cfg.steps - 1)
    q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
    o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32)
    wise.check_device()
    o, lse = o.cpu().numpy(), lse.cpu().numpy()
    for bi, hi in sample:
        base = (bi * cfg.heads + hi) * nb
        xs = [x[i, bi, hi].astype(np.float64) for i in range(3)]
        o_ref, lse_ref, _ = O.causal_attention(*xs, cfg.block, support=rows[base:base + nb], query_blocks=qbs)
        for qb in qbs:
            s = slice(qb * cfg.block, (qb + 1) * cfg.block)
            _assert_close("O", o[bi, hi, s], o_ref[s], O_TOL)
            _assert_close("LSE", lse[bi, hi, s], lse_ref[s], LSE_TOL)


# ------------------------------------------------ grouped-query attention ----

GQA_SHAPES = [  # (batch, q heads, kv heads, n, d, block)
    (1, 4, 2, 384, 128, 128),
    (2, 4, 1, 320, 64, 64),
    (1, 6, 3, 512, 96, 128),
]


def _gqa_inputs(b, h, hk, n, d, seed):
    rng = np.random.default_rng(seed)
    q = wl.bf16_round(rng.standard_normal((b, h, n, d)).astype(np.float32) * 1.5)
    kv = wl.bf16_round(rng.standard_normal((2, b, hk, n, d)).astype(np.float32) * 1.5)
    dev = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda().contiguous()
    # the oracle sees plain multi-head attention with each key/value head
    # repeated for the query heads of its group
    full = np.stack([q, np.repeat(kv[0], h // hk, axis=1), np.repeat(kv[1], h // hk, axis=1)])
    return full, dev(q), dev(kv[0]), dev(kv[1])


@pytest.mark.parametrize("shape", GQA_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_grouped_query_discover_and_sparse(shape):
    b, h, hk, n, d, blk = shape
    x, q, k, v = _gqa_inputs(b, h, hk, n, d, seed=n + h + hk)
    o, lse, mass = wise.discover(q, k, v, blk, out_dtype=torch.float32)
    wise.check_device()
    o_ref, lse_ref, r_ref = _oracle_discover(x, blk)
    _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
    _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)
    _assert_close("mass", mass.cpu().numpy(), r_ref, MASS_TOL)
    nb = n // blk
    rng = np.random.default_rng(h * n)
    rows = [r for _ in range(b * h) for r in wl.random_support(nb, 0.4, rng)]
    sup = wise.support_from_lists(rows, b, h, n, d, blk)
    o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32)
    wise.check_device()
    rp = sup.row_ptr.cpu().numpy()
    ci = sup.col_idx.cpu().numpy()
    o_ref, lse_ref = O.sparse(x[0].astype(np.float64), x[1].astype(np.float64), x[2].astype(np.float64), blk, rp, ci)
    _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
    _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)


# --------------------------------------- App. B support controls (Eqs 19-22) ----

@pytest.mark.parametrize("case", [(1, 2, 4, 64), (2, 3, 32, 128), (1, 1, 300, 64), (1, 1, 1024, 64)],
                         ids=lambda c: "B%d_H%d_nb%d_blk%d" % c)
@pytest.mark.parametrize("mode", ["mass", "size"])
@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("flags", [0, 3])
def test_controls_bit_exact_on_same_masses(case, mode, ties, flags):
    """MassMatched / SizeMatched rows from one step's masses and a reference
    working set (the WISE selection over three other steps, with some rows
    emptied), bit for bit against the oracle."""
    b, h, nb, blk = case
    m = _random_masses(4, b, h, nb, seed=nb * 3 + b, ties=ties)
    ref = wise.select_support(torch.from_numpy(m[1:]).contiguous().cuda(), nb * blk, 64, blk, 0.9, 0)
    rows = ref.to_lists()
    rng = np.random.default_rng(nb)
    rows = [[] if rng.random() < 0.1 else r for r in rows]  # empty reference rows select nothing
    ref = wise.support_from_lists(rows, b, h, nb * blk, 64, blk)
    got = wise.select_control(torch.from_numpy(np.ascontiguousarray(m[0])).cuda(), ref, mode, flags)
    wise.check_device()
    want = []
    for bi in range(b):
        for hi in range(h):
            base = (bi * h + hi) * nb
            want += O.control_set(m[0, bi, hi].astype(np.float64), rows[base:base + nb], mode, flags)
    assert got.to_lists() == want
    _check_tile_order(got)


def test_static95_is_a_one_step_window():
    """Static-95 (Eq 19): select_support over the first step alone at eta 0.95."""
    b, h, nb, blk = 1, 2, 48, 64
    m = _random_masses(1, b, h, nb, seed=95)
    sup = wise.select_support(torch.from_numpy(m).cuda(), nb * blk, 64, blk, 0.95, 0)
    want = []
    for hi in range(h):
        want += [sorted(O.step_support(m[0, 0, hi, q].astype(np.float64), q, 0.95)) for q in range(nb)]
    assert sup.to_lists() == want


# ------------------------- blocks of 32 (the pages' default granularity) ----
# Discovery runs on contiguous 128-key spans with one Eq 5 partial sum per
# 32-key block; sparse steps gather any four 32-key blocks listed by the
# tile's four query blocks into one 128-key entry with a per-(query block,
# slot) mask.

B32_SHAPES = [  # (batch, heads, n, d)
    (1, 2, 256, 64),
    (1, 1, 32, 64),       # one block in one partial tile
    (1, 1, 96, 128),      # three query blocks in one partial tile
    (2, 1, 480, 96),      # ragged last tile: three of its four query blocks exist
    (1, 2, 1024, 128),
    (1, 1, 2048, 64),     # lists longer than 32 entries
]


@pytest.mark.parametrize("shape", B32_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_block32_discover_parity(shape):
    b, h, n, d = shape
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=n + d + 32, scale=1.5, planted=2)
    o, lse, mass = wise.discover(q, k, v, 32, out_dtype=torch.float32)
    wise.check_device()
    o_ref, lse_ref, r_ref = _oracle_discover(x, 32)
    _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
    _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)
    _assert_close("mass", mass.cpu().numpy(), r_ref, MASS_TOL)
    iu = np.triu_indices(n // 32, 1)
    assert np.all(mass.cpu().numpy()[..., iu[0], iu[1]] == 0.0)


def _sparse_vs_oracle(x, q, k, v, rows, b, h, n, d, blk=32, use_schedule=False):
    sup = wise.support_from_lists(rows, b, h, n, d, blk)
    o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=use_schedule)
    wise.check_device()
    rp, ci = O.support_to_csr(rows)
    o_ref, lse_ref = O.sparse(x[0].astype(np.float64), x[1].astype(np.float64), x[2].astype(np.float64), blk, rp, ci)
    _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
    _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)
    if blk == 32:
        # the same step over the tiles' gathered entries read from a plan:
        # the same entries in the same order, so the same bits
        wise.gather_plan(sup)
        o_p, lse_p = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=use_schedule)
        wise.check_device()
        assert torch.equal(o_p, o) and torch.equal(lse_p, lse)
        _check_plan(sup, rows)
    return o, lse


def _check_plan(sup, rows):
    """The plan's counts and entries against their definition: per 128-row
    tile, the union of its four query blocks' lists in ascending order, four
    key blocks per entry (the last repeated to fill the entry), with bit
    4j + c set when query block j lists slot c's block."""
    b, h, nb = sup.batch, sup.heads, sup.n_blocks
    tiles = (nb + 3) // 4
    raw = sup.plan.cpu().numpy()
    units = b * h * tiles
    counts = raw[:units * 4].view(np.int32)
    off = (units * 4 + 15) // 16 * 16
    words = raw[off:].view(np.uint32)
    for bh in range(b * h):
        for t in range(tiles):
            lists = [set(rows[bh * nb + qb]) for qb in range(4 * t, min(4 * t + 4, nb))]
            union = sorted(set().union(*lists))
            chunks = [union[i:i + 4] for i in range(0, len(union), 4)]
            u = bh * tiles + t
            assert counts[u] == len(chunks), (bh, t)
            base = bh * (tiles * (tiles + 1) // 2) + t * (t + 1) // 2
            for e, ch in enumerate(chunks):
                kb = ch + [ch[-1]] * (4 - len(ch))
                mask = sum(1 << (4 * j + c) for j, lst in enumerate(lists) for c in range(len(ch)) if ch[c] in lst)
                w = words[4 * (base + e):4 * (base + e) + 3]
                assert (int(w[0]), int(w[1]), int(w[2])) == (kb[0] | kb[1] << 16, kb[2] | kb[3] << 16, mask), (bh, t, e)


@pytest.mark.parametrize("shape", B32_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("density", [0.1, 0.5])
def test_block32_sparse_parity_random_support(shape, density):
    b, h, n, d = shape
    nb = n // 32
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=5 * n + d, scale=1.5, planted=2)
    rng = np.random.default_rng(n + 32)
    rows = []
    for _ in range(b * h):
        rows.extend(wl.random_support(nb, density, rng, sink=bool(rng.integers(0, 2)), diag=bool(rng.integers(0, 2))))
    _sparse_vs_oracle(x, q, k, v, rows, b, h, n, d)


def test_block32_sparse_structured_supports():
    b, h, n, d = 1, 1, 1024, 128
    nb = n // 32
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=17, scale=1.5, planted=2)
    # sink and diagonal only: each tile gathers block 0 and its four diagonal blocks
    _sparse_vs_oracle(x, q, k, v, [sorted({0, qb}) for qb in range(nb)], b, h, n, d)
    # one shared column plus the diagonal
    _sparse_vs_oracle(x, q, k, v, [sorted({min(5, qb), qb}) for qb in range(nb)], b, h, n, d)
    # the four query blocks of a tile list disjoint blocks
    rows = [[kb for kb in range(qb + 1) if kb % 4 == qb % 4] for qb in range(nb)]
    _sparse_vs_oracle(x, q, k, v, rows, b, h, n, d)
    # only the diagonal block (causal inside the block only)
    _sparse_vs_oracle(x, q, k, v, [[qb] for qb in range(nb)], b, h, n, d)


def test_block32_sparse_full_support_bitwise_equals_discover():
    b, h, n, d = 1, 2, 768, 128
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=13, scale=1.5, planted=2)
    nb = n // 32
    rows = [list(range(qb + 1)) for _ in range(b * h) for qb in range(nb)]
    sup = wise.support_from_lists(rows, b, h, n, d, 32)
    o1, l1 = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False)
    o2, l2, _ = wise.discover(q, k, v, 32, want_mass=False, out_dtype=torch.float32)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_block32_planned_long_tiles_bitwise_equals_discover():
    """Tiles with more than 32 gathered entries (the late step reads a long
    tile's plan entries 32 at a time): the full causal support at 8K (tile t
    holds t + 1 entries, up to 64) over the plan equals discovery bit for bit,
    and so does the same step without the plan."""
    b, h, n, d = 1, 1, 8192, 64
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=29, scale=1.5, planted=2)
    nb = n // 32
    rows = [list(range(qb + 1)) for qb in range(nb)]
    sup = wise.support_from_lists(rows, b, h, n, d, 32)
    wise.gather_plan(sup)
    counts = sup.plan[:4 * (nb // 4)].view(torch.int32).cpu().numpy()
    assert counts.max() == nb // 4 and np.array_equal(counts, np.arange(1, nb // 4 + 1))
    o1, l1 = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False)
    o2, l2 = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False, use_plan=False)
    o3, l3, _ = wise.discover(q, k, v, 32, want_mass=False, out_dtype=torch.float32)
    wise.check_device()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_block32_sparse_empty_rows_and_tiles():
    b, h, n, d = 1, 1, 512, 64
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=6)
    nb = n // 32
    rows = [[0] if qb % 3 == 0 else [] for qb in range(nb)]
    for qb in range(4, 8):  # a whole tile with no entries
        rows[qb] = []
    o, lse = _sparse_vs_oracle(x, q, k, v, rows, b, h, n, d)
    on, ln = o.cpu().numpy(), lse.cpu().numpy()
    assert np.all(on[0, 0, 128:256] == 0) and np.all(np.isneginf(ln[0, 0, 128:256]))
    assert np.all(on[0, 0, 32:64] == 0) and np.all(np.isneginf(ln[0, 0, 32:64]))


def test_block32_sparse_malformed_support_is_flagged_not_faulted():
    b, h, n, d = 1, 1, 256, 64
    x, q, k, v = _bf16_inputs(b, h, n, d, seed=8)
    rows = [[0], [1, 0], [0, 7, 2], [-3, 3], [0, 4], [5, 5], [2], [1 << 20]]
    sup = wise.support_from_lists(rows, b, h, n, d, 32)
    wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False)
    assert wise.device_status() == wise._lib.WISE_ERR_BAD_SUPPORT
    assert wise.device_status() == wise._lib.WISE_OK
    # the plan built from it skips and flags the same entries; the step over
    # the plan then reads only what the plan holds
    wise.gather_plan(sup)
    assert wise.device_status() == wise._lib.WISE_ERR_BAD_SUPPORT
    wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False)
    assert wise.device_status() == wise._lib.WISE_OK
    # a plan whose count exceeds a tile's room (t + 1 entries) is flagged and
    # its tile written as empty
    counts = sup.plan[:8].view(torch.int32)
    counts[1] = 9
    o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_schedule=False)
    assert wise.device_status() == wise._lib.WISE_ERR_BAD_SUPPORT
    assert torch.all(o[0, 0, 128:256] == 0) and torch.all(torch.isneginf(lse[0, 0, 128:256]))


@pytest.mark.parametrize("case", [(2, 1, 2, 40, 0.9), (3, 2, 1, 128, 0.95), (1, 1, 1, 1024, 0.8), (2, 1, 3, 7, 0.9)],
                         ids=lambda c: "W%d_B%d_H%d_nb%d_eta%s" % c)
@pytest.mark.parametrize("flags", [0, 3])
def test_block32_select_bit_exact_on_same_masses(case, flags):
    w, b, h, nb, eta = case
    m = _random_masses(w, b, h, nb, seed=nb * 11 + w, ties=True)
    sup = wise.select_support(torch.from_numpy(m).cuda(), nb * 32, 64, 32, eta, flags)
    wise.check_device()
    rp_ref, ci_ref = O.select(m.astype(np.float64), eta, flags)
    rp = sup.row_ptr.cpu().numpy()
    assert np.array_equal(rp, rp_ref)
    assert np.array_equal(sup.col_idx.cpu().numpy()[:rp[-1]], ci_ref)
    _check_tile_order(sup)


@pytest.mark.parametrize("shape", [(1, 4, 2, 384, 128), (2, 4, 1, 224, 64), (1, 6, 3, 512, 96)],
                         ids=lambda s: "x".join(map(str, s)))
def test_block32_grouped_query(shape):
    b, h, hk, n, d = shape
    x, q, k, v = _gqa_inputs(b, h, hk, n, d, seed=n + h + hk + 32)
    o, lse, mass = wise.discover(q, k, v, 32, out_dtype=torch.float32)
    wise.check_device()
    o_ref, lse_ref, r_ref = _oracle_discover(x, 32)
    _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
    _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)
    _assert_close("mass", mass.cpu().numpy(), r_ref, MASS_TOL)
    rng = np.random.default_rng(h * n + 32)
    rows = [r for _ in range(b * h) for r in wl.random_support(n // 32, 0.3, rng)]
    _sparse_vs_oracle(x, q, k, v, rows, b, h, n, d)


def test_block32_trajectory_end_to_end():
    cfg = wl.CONFIGS["tiny"].replace(name="tiny_b32", seq_len=512, block=32)
    sup, outs = _run_trajectory(cfg)
    rows = sup.to_lists()
    nb = cfg.n_blocks
    for bi in range(cfg.batch):
        for hi in range(cfg.heads):
            om = []
            for t in cfg.window_steps:
                x = outs[t][0]
                _, _, r = O.causal_attention(*(x[i, bi, hi].astype(np.float64) for i in range(3)), cfg.block,
                                             want_mass=True)
                om.append(r)
                _assert_close("mass", outs[t][3][bi, hi], r, MASS_TOL)
            base = (bi * cfg.heads + hi) * nb
            _assert_support_matches(rows[base:base + nb], om, cfg, rows[base:base + nb])
    rp = sup.row_ptr.cpu().numpy()
    ci = sup.col_idx.cpu().numpy()
    # the selection built the late steps' plan of gathered entries
    assert sup.plan is not None
    _check_plan(sup, rows)
    for t in range(cfg.t_d, cfg.steps):
        x = wl.step_inputs(cfg, t)
        q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
        o, lse = wise.sparse(q, k, v, sup, out_dtype=torch.float32)
        o_ref, lse_ref = O.sparse(x[0].astype(np.float64), x[1].astype(np.float64), x[2].astype(np.float64),
                                  cfg.block, rp, ci)
        _assert_close("O", o.cpu().numpy(), o_ref, O_TOL)
        _assert_close("LSE", lse.cpu().numpy(), lse_ref, LSE_TOL)
        o_u, lse_u = wise.sparse(q, k, v, sup, out_dtype=torch.float32, use_plan=False)
        assert torch.equal(o_u, o) and torch.equal(lse_u, lse)


# ------------------- selection fused into discovery (Eq 6 streamed over the window) ----

@pytest.mark.parametrize("case", [(1, 2, 512, 64, 64, 2), (1, 3, 1024, 128, 128, 3), (2, 1, 480, 96, 32, 2),
                                  (1, 2, 2048, 64, 128, 1), (1, 1, 8192, 64, 32, 2), (1, 2, 4096, 128, 128, 3)],
                         ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("flags", [0, 3])
def test_fused_selection_equals_separate_selection(case, flags):
    b, h, n, d, blk, window = case
    eta = 0.9
    state = wise.new_select_state((b, h, n, d), blk, window)
    masses = []
    for w in range(window):
        x, q, k, v = _bf16_inputs(b, h, n, d, seed=97 * w + n + blk, scale=1.5, planted=3)
        o1, l1, m1 = wise.discover_select(q, k, v, blk, step=w, window=window, eta=eta, select_state=state,
                                          flags=flags, out_dtype=torch.float32)
        o2, l2, m2 = wise.discover(q, k, v, blk, out_dtype=torch.float32)
        wise.check_device()
        # the same kernel and arithmetic as plain discovery with masses
        assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(m1, m2)
        masses.append(m1.clone())
    fused = wise.select_finalize(state, b, h, n, d, blk)
    sep = wise.select_support(torch.stack(masses).contiguous(), n, d, blk, eta, flags)
    wise.check_device()
    rp = fused.row_ptr.cpu().numpy()
    assert np.array_equal(rp, sep.row_ptr.cpu().numpy())
    assert np.array_equal(fused.col_idx.cpu().numpy()[:rp[-1]], sep.col_idx.cpu().numpy()[:rp[-1]])
    assert int(fused.nnz.item()) == int(sep.nnz.item()) == rp[-1]
    assert torch.equal(fused.tile_order, sep.tile_order)
    rp_ref, ci_ref = O.select(torch.stack(masses).cpu().numpy().astype(np.float64), eta, flags)
    assert np.array_equal(rp, rp_ref) and np.array_equal(fused.col_idx.cpu().numpy()[:rp[-1]], ci_ref)
    _check_tile_order(fused)


def test_fused_selection_trajectory_matches_oracle():
    cfg = wl.CONFIGS["tiny"]
    state = wise.new_select_state((cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim), cfg.block, cfg.window)
    oracle_masses = {}
    for t in range(cfg.t_d):
        x = wl.step_inputs(cfg, t)
        q, k, v = (torch.from_numpy(x[i]).to(torch.bfloat16).cuda() for i in range(3))
        if t in cfg.window_steps:
            wise.discover_select(q, k, v, cfg.block, step=t - cfg.window_steps[0], window=cfg.window, eta=cfg.eta,
                                 select_state=state)
            oracle_masses[t] = x
        else:
            wise.discover(q, k, v, cfg.block, want_mass=False)
    sup = wise.select_finalize(state, cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block)
    wise.check_device()
    rows = sup.to_lists()
    nb = cfg.n_blocks
    for bi in range(cfg.batch):
        for hi in range(cfg.heads):
            om = []
            for t in cfg.window_steps:
                x = oracle_masses[t]
                _, _, r = O.causal_attention(*(x[i, bi, hi].astype(np.float64) for i in range(3)), cfg.block,
                                             want_mass=True)
                om.append(r)
            base = (bi * cfg.heads + hi) * nb
            _assert_support_matches(rows[base:base + nb], om, cfg, rows[base:base + nb])
