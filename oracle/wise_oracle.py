"""Plain fp64 CPU oracle for the WISE hot path (discover -> select -> reuse).

TEST INFRASTRUCTURE ONLY. This module is the checker, not the product: only
the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference arm may import it. The CUDA library shares no code with it.

Everything here follows "Attention Routing Stabilizes Early: Working-Set
Inference for Recurrent Language Models" (WISE, arXiv 2609.27373):

* ``causal_attention``   -- §3 "Recurrent attention", Eq 2 (softmax of
  QK^T/sqrt(d_h) + M, then A V) with the causal mask M; with a block
  support it is §5.2 Eq 7 (working-set mask R) and Eq 8 (late-stage attention).
* ``block_mass``         -- §5.1 Eq 5, r_qb = (1/|I_q|) sum_{i in I_q} sum_{j in I_b} A_ij.
* ``step_support``       -- §5.1 Eq 6 (right): the smallest set of admissible
  key blocks whose cumulative block mass reaches eta, blocks taken in
  descending mass order (Appendix A.1, Eq 12).
* ``working_set``        -- §5.1 Eq 6 (left) / Appendix B Eq 18: union of the
  per-step supports over the last four discovery steps (clamped at the first
  step as in Appendix C.2 Eq 23).
* ``support_to_csr``     -- Appendix B "Sparse-kernel implementation": the
  support as row offsets plus active block indices.
* ``identification_margin`` -- Appendix A.1 Eq 13, the margin Delta_q.
* ``retained_mass``      -- Appendix B "Evaluation metrics": fraction of the
  unrestricted attention mass that falls inside a support.

Readings where the pages are silent (each also listed in the design notes):

* the mask M is causal: key j is admissible for query i iff j <= i, so key
  block b is admissible for query block q iff b <= q;
* |I_q| = B (the sequence length is a multiple of B), so sum_b r_qb = 1;
* cumulative sums of Eq 6 run in integers: masses are converted to int64
  fixed point with 52 fractional bits (round to nearest, ties to even);
  eta and the tie tolerance are converted the same way. If the admissible
  mass never reaches eta (rounding), every admissible block is taken;
* ties: with k the Eq 6 cardinality and r* the k-th mass in (mass desc,
  index asc) order, blocks whose mass exceeds r* + 1e-6 are kept and the
  remaining k - |kept| places go to the lowest-index blocks whose mass lies
  within 1e-6 of r*;
* the sink block (key block 0, which holds the first token) and the diagonal
  block q may be added to every support (flags), both off in the pages' own
  definition;
* the softmax scale is 1/sqrt(d_h) unless a scale is given.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Set, Tuple

import numpy as np

FIXED_POINT_BITS = 52
TIE_TOLERANCE = 1e-6
SUPPORT_SINK = 1
SUPPORT_DIAG = 2


def default_scale(head_dim: int) -> float:
    """1/sqrt(d_h) of Eq 2."""
    return 1.0 / math.sqrt(head_dim)


# ---------------------------------------------------------------------------
# Eq 2 / Eq 7 / Eq 8: causal (optionally working-set restricted) attention
# ---------------------------------------------------------------------------

def _query_block_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, row0: int,
                      block: int, scale: float, allowed_blocks: Optional[Set[int]]):
    """Attention for a contiguous run of query rows starting at ``row0``.

    Returns (O rows, LSE rows, A rows) with A over all n keys."""
    n = k.shape[0]
    m_rows = q_rows.shape[0]
    s = (q_rows @ k.T) * scale                              # Q K^T / sqrt(d_h)
    i = row0 + np.arange(m_rows)[:, None]
    j = np.arange(n)[None, :]
    keep = j <= i                                           # causal mask M
    if allowed_blocks is not None:                          # working-set mask R (Eq 7)
        in_support = np.zeros(n, dtype=bool)
        for b in allowed_blocks:
            in_support[b * block:(b + 1) * block] = True
        keep = keep & in_support[None, :]
    s = np.where(keep, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    empty = ~np.isfinite(m[:, 0])
    m = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        a = np.where(l > 0, p / np.where(l > 0, l, 1.0), 0.0)
        lse = (m + np.log(l))[:, 0]
    lse[empty] = -np.inf
    o = a @ v
    return o, lse, a


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, block: int,
                     scale: Optional[float] = None,
                     support: Optional[Sequence[Iterable[int]]] = None,
                     query_blocks: Optional[Iterable[int]] = None,
                     want_mass: bool = False):
    """Eq 2 (support=None) or Eq 8 (support = per-query-block key-block sets).

    q, k, v: [n, d] arrays of one (batch, head), widened to fp64.
    Returns (O [n, d], LSE [n] natural log, r [nb, nb] or None). Rows of
    query blocks not listed in ``query_blocks`` are left zero (O) / nan (LSE).
    ``want_mass`` also returns the Eq 5 block masses of the rows computed.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, d = q.shape
    if n % block:
        raise ValueError("sequence length must be a multiple of the block size")
    nb = n // block
    scale = default_scale(d) if scale is None else float(scale)
    qbs = range(nb) if query_blocks is None else list(query_blocks)
    o = np.zeros((n, d))
    lse = np.full(n, np.nan)
    r = np.zeros((nb, nb)) if want_mass else None
    for qb in qbs:
        rows = slice(qb * block, (qb + 1) * block)
        allowed = None if support is None else set(int(b) for b in support[qb])
        o_q, lse_q, a_q = _query_block_rows(q[rows], k, v, qb * block, block, scale, allowed)
        o[rows] = o_q
        lse[rows] = lse_q
        if want_mass:
            r[qb] = block_mass_rows(a_q, block)
    return o, lse, r


def block_mass_rows(a_rows: np.ndarray, block: int) -> np.ndarray:
    """Eq 5 for one query block: a_rows is A restricted to the rows of I_q.

    r_qb = (1/|I_q|) sum_{i in I_q} sum_{j in I_b} A_ij, for every key block b."""
    n = a_rows.shape[1]
    nb = n // block
    rows_in_q = a_rows.shape[0]
    return np.array([a_rows[:, b * block:(b + 1) * block].sum() for b in range(nb)]) / rows_in_q


def block_mass(q: np.ndarray, k: np.ndarray, block: int, scale: Optional[float] = None,
               query_blocks: Optional[Iterable[int]] = None) -> np.ndarray:
    """Eq 5 block masses [nb, nb] of the unrestricted causal attention."""
    v = np.zeros((k.shape[0], 1))
    _, _, r = causal_attention(q, k, v, block, scale, query_blocks=query_blocks, want_mass=True)
    return r


# ---------------------------------------------------------------------------
# Eq 6: per-step cumulative-mass support and its temporal union
# ---------------------------------------------------------------------------

def to_fixed(x) -> np.ndarray:
    """Masses (and eta) in int64 units of 2^-52, round to nearest even."""
    return np.rint(np.asarray(x, np.float64) * 2.0 ** FIXED_POINT_BITS).astype(np.int64)


def step_support(r_q: Sequence[float], q: int, eta: float,
                 tie_tolerance: float = TIE_TOLERANCE) -> Set[int]:
    """Eq 6 (right) for query block q at one step.

    r_q holds the block masses r_qb for b = 0..nb-1; only b <= q is admissible.
    Blocks are taken in descending mass order (lower index first on equal
    mass) until the cumulative mass reaches eta; k is that count. Near-ties at
    the cut are then resolved toward lower block indices."""
    fx = [int(x) for x in to_fixed(np.asarray(r_q, np.float64)[:q + 1])]
    admissible = list(range(q + 1))
    order = sorted(admissible, key=lambda b: (-fx[b], b))
    target = int(to_fixed(eta))
    cum = 0
    k = None
    for pos, b in enumerate(order):
        cum += fx[b]
        if cum >= target:
            k = pos + 1
            break
    if k is None:
        return set(admissible)
    r_star = fx[order[k - 1]]
    tol = int(to_fixed(tie_tolerance))
    kept = {b for b in admissible if fx[b] > r_star + tol}
    near = sorted(b for b in admissible if abs(fx[b] - r_star) <= tol)
    return kept | set(near[:k - len(kept)])


def _cut_support(fx: Sequence[int], q: int, k: int, tie_tolerance: float) -> Set[int]:
    """The k highest-mass admissible blocks (b <= q) in (mass desc, index asc)
    order, with the near-tie rule of step_support at the cut."""
    admissible = list(range(q + 1))
    if k <= 0:
        return set()
    if k >= len(admissible):
        return set(admissible)
    order = sorted(admissible, key=lambda b: (-fx[b], b))
    r_star = fx[order[k - 1]]
    tol = int(to_fixed(tie_tolerance))
    kept = {b for b in admissible if fx[b] > r_star + tol}
    near = sorted(b for b in admissible if abs(fx[b] - r_star) <= tol)
    return kept | set(near[:k - len(kept)])


def mass_matched_support(r_q: Sequence[float], q: int, reference: Iterable[int],
                         tie_tolerance: float = TIE_TOLERANCE) -> Set[int]:
    """MassMatched control (WISE App. B "Intervention controls", Eqs 20-21):
    the smallest set of highest-mass admissible blocks of this step whose
    cumulative mass reaches m_q, the mass of this step covered by the
    reference working set. m_q is summed in the same fixed point as Eq 6, so
    the cut compares exact integers."""
    fx = [int(x) for x in to_fixed(np.asarray(r_q, np.float64)[:q + 1])]
    target = sum(fx[b] for b in set(reference) if 0 <= b <= q)
    if target <= 0:
        return set()
    order = sorted(range(q + 1), key=lambda b: (-fx[b], b))
    cum = 0
    for pos, b in enumerate(order):
        cum += fx[b]
        if cum >= target:
            return _cut_support(fx, q, pos + 1, tie_tolerance)
    return set(range(q + 1))


def size_matched_support(r_q: Sequence[float], q: int, size: int,
                         tie_tolerance: float = TIE_TOLERANCE) -> Set[int]:
    """SizeMatched control (WISE App. B "Intervention controls", Eq 22): the
    `size` highest-mass admissible blocks of this step (TopK), with the near-tie
    rule of Eq 6 (reading R6) at the cut."""
    fx = [int(x) for x in to_fixed(np.asarray(r_q, np.float64)[:q + 1])]
    return _cut_support(fx, q, size, tie_tolerance)


def control_set(r: np.ndarray, reference: Sequence[Sequence[int]], mode: str,
                flags: int = 0, tie_tolerance: float = TIE_TOLERANCE) -> List[List[int]]:
    """MassMatched ("mass") or SizeMatched ("size") rows for one step's
    [nb, nb] masses against the reference working set's rows; the sink and
    diagonal blocks are added as in working_set when flags ask for them."""
    out = []
    for q in range(r.shape[0]):
        ref = [b for b in reference[q] if 0 <= b <= q]
        if mode == "mass":
            s = mass_matched_support(r[q], q, ref, tie_tolerance)
        else:
            s = size_matched_support(r[q], q, len(set(ref)), tie_tolerance)
        if flags & SUPPORT_SINK:
            s.add(0)
        if flags & SUPPORT_DIAG:
            s.add(q)
        out.append(sorted(s))
    return out


def working_set(masses: Sequence[np.ndarray], eta: float, flags: int = SUPPORT_SINK | SUPPORT_DIAG,
                tie_tolerance: float = TIE_TOLERANCE) -> List[List[int]]:
    """Eq 6 (left): B_q = union over the window steps of the step supports.

    masses: sequence of [nb, nb] arrays, one per window step (the last
    min(4, t_d) discovery steps). Returns ascending key-block lists per q."""
    nb = masses[0].shape[0]
    out = []
    for q in range(nb):
        s: Set[int] = set()
        for r in masses:
            s |= step_support(r[q], q, eta, tie_tolerance)
        if flags & SUPPORT_SINK:
            s.add(0)
        if flags & SUPPORT_DIAG:
            s.add(q)
        out.append(sorted(s))
    return out


def support_to_csr(rows: Sequence[Sequence[int]]) -> Tuple[np.ndarray, np.ndarray]:
    """Row offsets and active block indices (ascending within a row)."""
    row_ptr = np.zeros(len(rows) + 1, np.int32)
    cols: List[int] = []
    for i, r in enumerate(rows):
        cols.extend(sorted(int(b) for b in r))
        row_ptr[i + 1] = len(cols)
    return row_ptr, np.asarray(cols, np.int32)


def csr_to_support(row_ptr: np.ndarray, col_idx: np.ndarray) -> List[List[int]]:
    return [list(map(int, col_idx[row_ptr[i]:row_ptr[i + 1]])) for i in range(len(row_ptr) - 1)]


def block_density(rows: Sequence[Sequence[int]]) -> float:
    """Fraction of admissible (q, b) blocks retained (Appendix B metrics)."""
    nb = len(rows)
    return sum(len(r) for r in rows) / (nb * (nb + 1) / 2)


# ---------------------------------------------------------------------------
# Appendix A.1 Eq 13: identification margin; Appendix B: retained mass
# ---------------------------------------------------------------------------

def identification_margin(r_q: Sequence[float], q: int, eta: float) -> float:
    """Delta_q of Eq 13 for the admissible masses r_q[0..q] (in real
    arithmetic). Returns 0 for a degenerate support."""
    r = np.sort(np.asarray(r_q, np.float64)[:q + 1])[::-1]
    csum = np.cumsum(r)
    hits = np.nonzero(csum >= eta)[0]
    if len(hits) == 0:
        return 0.0
    k = int(hits[0]) + 1
    d_rank = (r[k - 1] - r[k]) / 2 if k < len(r) else math.inf
    d_minus = eta - (csum[k - 2] if k > 1 else 0.0)
    d_plus = csum[k - 1] - eta
    terms = [d_rank, d_plus / k]
    if k > 1:
        terms.append(d_minus / (k - 1))
    return max(0.0, min(terms))


def retained_mass_rows(r: np.ndarray, rows: Sequence[Sequence[int]]) -> np.ndarray:
    """Retained future attention mass per query block (WISE App. B,
    "Evaluation metrics"): sum over the support's key blocks of the
    unrestricted block masses r_qb (Eq 5) of a later step."""
    return np.array([sum(float(r[q, b]) for b in rows[q]) for q in range(len(rows))], np.float64)


def retained_mass(r: np.ndarray, rows: Sequence[Sequence[int]]) -> float:
    """Mean over query blocks of sum_{b in B_q} r_qb: the share of the
    unrestricted attention mass that lands inside the support."""
    return float(np.mean(retained_mass_rows(r, rows)))


def jaccard(rows_a: Sequence[Sequence[int]], rows_b: Sequence[Sequence[int]]) -> Tuple[int, int, float]:
    """WISE App. C.2 Eq 24 for one example: the working sets are the
    collections of active (head, query block, key block) entries; returns
    (|A intersect B|, |A union B|, their ratio), the ratio being 1 when both are empty.
    rows_a and rows_b list the key blocks of the same sequence of rows."""
    inter = union = 0
    for ra, rb in zip(rows_a, rows_b):
        sa, sb = set(ra), set(rb)
        inter += len(sa & sb)
        union += len(sa | sb)
    return inter, union, (inter / union if union else 1.0)


# ---------------------------------------------------------------------------
# Multi-head wrappers: [B, H, n, d] tensors
# ---------------------------------------------------------------------------

def discover(q: np.ndarray, k: np.ndarray, v: np.ndarray, block: int, scale: Optional[float] = None,
             heads: Optional[Iterable[Tuple[int, int]]] = None, query_blocks=None):
    """Discovery step for every (batch, head): Eq 2 output plus Eq 5 masses.

    Returns O [B,H,n,d], LSE [B,H,n], r [B,H,nb,nb] (zeros for skipped heads)."""
    bsz, nh, n, d = q.shape
    nb = n // block
    o = np.zeros((bsz, nh, n, d))
    lse = np.full((bsz, nh, n), np.nan)
    r = np.zeros((bsz, nh, nb, nb))
    pairs = heads if heads is not None else [(b, h) for b in range(bsz) for h in range(nh)]
    for b, h in pairs:
        o[b, h], lse[b, h], r[b, h] = causal_attention(q[b, h], k[b, h], v[b, h], block, scale,
                                                       query_blocks=query_blocks, want_mass=True)
    return o, lse, r


def select(masses: np.ndarray, eta: float, flags: int = SUPPORT_SINK | SUPPORT_DIAG,
           tie_tolerance: float = TIE_TOLERANCE) -> Tuple[np.ndarray, np.ndarray]:
    """Support selection for every (batch, head). masses: [W, B, H, nb, nb].

    Returns the CSR over rows ordered (batch, head, query block)."""
    w, bsz, nh, nb, _ = masses.shape
    rows: List[List[int]] = []
    for b in range(bsz):
        for h in range(nh):
            rows.extend(working_set([masses[t, b, h] for t in range(w)], eta, flags, tie_tolerance))
    return support_to_csr(rows)


def sparse(q: np.ndarray, k: np.ndarray, v: np.ndarray, block: int, row_ptr: np.ndarray,
           col_idx: np.ndarray, scale: Optional[float] = None,
           heads: Optional[Iterable[Tuple[int, int]]] = None, query_blocks=None):
    """Late step (Eq 8) for every (batch, head) over the CSR support."""
    bsz, nh, n, d = q.shape
    nb = n // block
    o = np.zeros((bsz, nh, n, d))
    lse = np.full((bsz, nh, n), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(bsz) for h in range(nh)]
    for b, h in pairs:
        base = (b * nh + h) * nb
        supp = [col_idx[row_ptr[base + qb]:row_ptr[base + qb + 1]] for qb in range(nb)]
        o[b, h], lse[b, h], _ = causal_attention(q[b, h], k[b, h], v[b, h], block, scale,
                                                 support=supp, query_blocks=query_blocks)
    return o, lse
