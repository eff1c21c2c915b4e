"""Seeded synthetic inputs for WISE block-sparse causal attention.

This module is shared by the tests, the benchmark and the oracle checks. It
holds no attention arithmetic: it only draws random tensors with the shape and
structure of a recurrent-attention workload and rounds them to bf16.

Workload recipe (one recurrent attention layer, H_q == H_kv, layout
[batch, heads, seq, head_dim], head_dim contiguous):

* per (batch, head) an independent PCG64 stream, keyed by (seed, config id,
  batch index, head index), draws the base tensors Q0, K0, V0 ~ N(0, 1) and a
  shared evidence direction u ~ N(0, I_d) (unit-variance entries);
* ``n_evidence`` distinct key blocks E are drawn uniformly without
  replacement from {0 .. n/B - 1};
* every query row gets ``Q0 += s * u``; the key rows of the evidence blocks get
  ``K0 += s * u`` (s = ``strength``), which plants blocks that attract mass;
* recurrent step t (0-indexed) sees X_t = X0 + sigma0 * gamma**t * eps_t for
  fresh independent N(0, 1) noise per tensor and per step, drawn from a second
  stream keyed by (seed, config id, batch, head, t);
* the step inputs are rounded to bf16 with round-to-nearest-even. Both the GPU
  path and the oracle consume exactly these bf16 values.

The recurrent model itself (hidden states, projections) is replaced by this
generator: the pages' method operates on whatever Q/K/V each step produces.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, Iterable, List, Optional, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    name: str
    batch: int
    heads: int
    head_dim: int
    seq_len: int
    block: int
    n_evidence: int
    strength: float
    steps: int          # T, recurrent depth
    t_d: int            # discovery depth
    eta: float          # cumulative-mass threshold
    sigma0: float
    gamma: float

    @property
    def n_blocks(self) -> int:
        return self.seq_len // self.block

    @property
    def window(self) -> int:
        """Width of the temporal union: the last min(4, t_d) discovery steps."""
        return min(4, self.t_d)

    @property
    def window_steps(self) -> List[int]:
        """0-indexed discovery steps whose supports are unioned."""
        return list(range(self.t_d - self.window, self.t_d))

    def sigma(self, t: int) -> float:
        return float(self.sigma0 * self.gamma ** t)

    def replace(self, **kw) -> "WorkloadConfig":
        return dataclasses.replace(self, **kw)


def _sweep(n: int) -> WorkloadConfig:
    return WorkloadConfig(f"sweep_{n // 1024}k", 1, 32, 128, n, 128, 8, 2.5,
                          8, 3, 0.9, 0.3, 0.7)


CONFIGS: Dict[str, WorkloadConfig] = {
    "tiny": WorkloadConfig("tiny", 1, 2, 64, 256, 64, 2, 3.0, 4, 2, 0.9, 0.5, 0.6),
    "4k": WorkloadConfig("4k", 1, 32, 128, 4096, 128, 8, 2.5, 8, 3, 0.9, 0.3, 0.7),
    "8k_b4": WorkloadConfig("8k_b4", 4, 32, 128, 8192, 128, 12, 3.0, 16, 4, 0.95, 0.3, 0.75),
    "16k_h40_d96": WorkloadConfig("16k_h40_d96", 1, 40, 96, 16384, 128, 16, 3.0, 32, 4, 0.9, 0.2, 0.8),
}
for _n in (2048, 4096, 8192, 16384, 32768):
    _c = _sweep(_n)
    CONFIGS[_c.name] = _c


def _key(cfg: WorkloadConfig) -> int:
    return zlib.crc32(cfg.name.encode())


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns float32
    arrays holding exactly representable bf16 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    rnd = ((bits >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((bits + rnd) & np.uint32(0xFFFF0000)).view(np.float32)
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


class HeadGenerator:
    """Generator for one (batch, head) slice of a workload."""

    def __init__(self, cfg: WorkloadConfig, b: int, h: int, seed: int = 0):
        self.cfg = cfg
        self.b, self.h, self.seed = b, h, seed
        rng = np.random.Generator(np.random.PCG64([seed, _key(cfg), b, h]))
        n, d = cfg.seq_len, cfg.head_dim
        base = rng.standard_normal((3, n, d), dtype=np.float32)
        u = rng.standard_normal(d, dtype=np.float32)
        ev = rng.choice(cfg.n_blocks, size=min(cfg.n_evidence, cfg.n_blocks), replace=False)
        self.evidence_blocks = np.sort(ev).astype(np.int64)
        s = np.float32(cfg.strength)
        base[0] += s * u
        for blk in self.evidence_blocks:
            base[1, blk * cfg.block:(blk + 1) * cfg.block] += s * u
        self.base = base

    def step(self, t: int) -> np.ndarray:
        """bf16-exact float32 array [3, n, d] = (Q, K, V) at recurrent step t."""
        cfg = self.cfg
        rng = np.random.Generator(np.random.PCG64([self.seed, _key(cfg), self.b, self.h, 1000 + t]))
        noise = rng.standard_normal(self.base.shape, dtype=np.float32)
        x = self.base + np.float32(cfg.sigma(t)) * noise
        return bf16_round(x)


def step_inputs(cfg: WorkloadConfig, t: int, seed: int = 0,
                heads: Optional[Iterable[Tuple[int, int]]] = None) -> np.ndarray:
    """Q, K, V for recurrent step t as a float32 array [3, B, H, n, d] of
    bf16-exact values. ``heads`` restricts generation to some (b, h) pairs
    (others are left zero)."""
    out = np.zeros((3, cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim), np.float32)
    pairs = heads if heads is not None else [(b, h) for b in range(cfg.batch) for h in range(cfg.heads)]
    for b, h in pairs:
        out[:, b, h] = HeadGenerator(cfg, b, h, seed).step(t)
    return out


def trajectory_inputs(cfg: WorkloadConfig, steps: Iterable[int], seed: int = 0,
                      heads: Optional[Iterable[Tuple[int, int]]] = None) -> Dict[int, np.ndarray]:
    """Step inputs for several steps, sharing the per-head base draw."""
    steps = list(steps)
    res = {t: np.zeros((3, cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim), np.float32) for t in steps}
    pairs = heads if heads is not None else [(b, h) for b in range(cfg.batch) for h in range(cfg.heads)]
    for b, h in pairs:
        g = HeadGenerator(cfg, b, h, seed)
        for t in steps:
            res[t][:, b, h] = g.step(t)
    return res


def _head_bits(args):
    """Worker of trajectory_inputs_bf16: one (batch, head) slice at the listed
    steps, as bf16 bit patterns [len(steps), 3, n, d]."""
    cfg, seed, steps, b, h = args
    g = HeadGenerator(cfg, b, h, seed)
    return b, h, np.stack([bf16_bits(g.step(t)) for t in steps])


def trajectory_inputs_bf16(cfg: WorkloadConfig, steps: Iterable[int], seed: int = 0,
                           processes: Optional[int] = None) -> Dict[int, np.ndarray]:
    """The values of trajectory_inputs, as bf16 bit patterns (uint16 arrays
    [3, B, H, n, d]), drawn by a pool of `processes` worker processes (default:
    the usable cores, at most 32). Each (batch, head) slice comes from its own
    generator, so the result does not depend on the number of processes. The
    pool uses the 'spawn' start method, so it is safe to call after CUDA has
    been initialised in the calling process."""
    import multiprocessing as mp
    import os
    steps = list(steps)
    shape = (3, cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim)
    res = {t: np.empty(shape, np.uint16) for t in steps}
    jobs = [(cfg, seed, steps, b, h) for b in range(cfg.batch) for h in range(cfg.heads)]
    if processes is None:
        processes = min(32, len(os.sched_getaffinity(0)))
    processes = max(1, min(processes, len(jobs)))

    def put(item):
        b, h, bits = item
        for i, t in enumerate(steps):
            res[t][:, b, h] = bits[i]

    if processes == 1:
        for j in jobs:
            put(_head_bits(j))
    else:
        with mp.get_context("spawn").Pool(processes) as pool:
            for item in pool.imap_unordered(_head_bits, jobs):
                put(item)
    return res


def random_support(n_blocks: int, density: float, rng: np.random.Generator,
                   sink: bool = True, diag: bool = True) -> List[List[int]]:
    """A random causal block support (list of ascending key blocks per query
    block) for kernel-isolation tests."""
    rows = []
    for q in range(n_blocks):
        keep = rng.random(q + 1) < density
        if sink:
            keep[0] = True
        if diag:
            keep[q] = True
        if not keep.any():
            keep[rng.integers(0, q + 1)] = True
        rows.append([int(b) for b in np.nonzero(keep)[0]])
    return rows
