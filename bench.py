"""Benchmark of the WISE hot path on GB300.

One step = one recurrent-attention trajectory of the workload: t_d discovery
steps (dense causal attention; block masses on the last min(4, t_d) steps),
one working-set selection, and T - t_d late steps of block-sparse attention
over the selected support, each step on its own seeded Q/K/V.

The headline workload is the largest single-GPU configuration, the 32K
context of the sweep (batch 1, 32 heads, head_dim 128, block 128). `value`
is its late-step sparse attention throughput in useful TFLOP/s (4 d per
admissible query-key pair inside the support), from the median of the late
steps' CUDA-event times on the launching stream inside the timed
trajectories. The line also carries ms
per trajectory, the late-step time against the library's own dense kernel on
the same inputs, the roofline of the dominant kernel, an end-to-end figure
through the public API with host buffers, the fp64 CPU oracle timed on a
bounded sample (cpu_baseline), and a per-configuration block ("configs"):
for each workload of the sweep, the median and inter-quartile range over
balanced passes of the late sparse step, the dense step, the discovery step
with masses and the selection, with speedups, throughput and density.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config sweep_32k]
                    [--sweep a,b,...|none] [--impl wise|reference]
    python bench.py --config C --profile-kernel {discover,discover_mass,sparse,select} --steps K
        (a few launches of one kernel on one configuration, for ncu captures)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "late-step sparse-attn TFLOP/s & ms/step vs dense; % of BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 2 ** 20
DEFAULT_CONFIG = "sweep_32k"
DEFAULT_SWEEP = "sweep_2k,4k,sweep_8k,8k_b4,16k_h40_d96,sweep_16k"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def support_flops(row_ptr: np.ndarray, col_idx: np.ndarray, nb: int, block: int, head_dim: int) -> float:
    """Useful FLOPs of one sparse step: 4 d per admissible pair in the listed blocks."""
    rows = len(row_ptr) - 1
    q_of_row = np.arange(rows) % nb
    counts = np.diff(row_ptr)
    q_rep = np.repeat(q_of_row, counts)
    cols = col_idx[:row_ptr[-1]]
    diag = int(np.sum(cols == q_rep))
    off = int(len(cols) - diag)
    return 4.0 * head_dim * (off * block * block + diag * block * (block + 1) / 2)


def tile_entries(row_ptr: np.ndarray, col_idx: np.ndarray, bh: int, nb: int, block: int) -> int:
    """Entries (K/V tiles) one sparse step runs: per 128-row query tile, the
    distinct key blocks its query blocks list; blocks of 32 are gathered four
    to an entry."""
    per_tile = 128 // block
    tiles = -(-nb // per_tile)
    listed = np.zeros((bh, tiles * per_tile, nb), dtype=bool)
    rows = np.repeat(np.arange(bh * nb), np.diff(row_ptr))
    cols = col_idx[:row_ptr[-1]]
    listed[rows // nb, rows % nb, cols] = True
    union = listed.reshape(bh, tiles, per_tile, nb).any(axis=2).sum(axis=2)
    if block == 32:
        union = -(-union // 4)
    return int(union.sum())


def tile_flops(entries: int, block: int, head_dim: int) -> float:
    """FLOPs the tensor core executes for `entries` tiles: S = Q K^T and
    O += P V over 128 query rows and one entry's keys (128, or 64 for blocks
    of 64)."""
    keys = 64 if block == 64 else 128
    return 4.0 * head_dim * 128 * keys * entries


def reduce_max_over_ranks(values, world, device=None):
    """Element-wise max over ranks (the slowest rank sets the time)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tflops(flops_per_rank: float, max_ms: float, world: int) -> float:
    """Aggregate throughput: every rank does the same work (weak scaling) and
    the job takes as long as its slowest rank."""
    return world * flops_per_rank / (max_ms * 1e-3) / 1e12


def median_iqr(values):
    """Median and inter-quartile range (75th minus 25th percentile)."""
    a = np.asarray(values, np.float64)
    q25, q50, q75 = np.percentile(a, [25, 50, 75])
    return float(q50), float(q75 - q25)


def setup_cost_ms(select_ms: float, mass_step_ms, dense_ms: float, window: int) -> float:
    """Cost of building the support: the selection launch plus what each of
    the window's discovery launches costs beyond the plain dense kernel (the
    mass epilogue, or the fused selection). The difference is kept signed, so
    timing noise moves the figure both ways."""
    extra = 0.0 if mass_step_ms is None else mass_step_ms - dense_ms
    return select_ms + window * extra


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources a kernel is built from (the attention kernels, or
    the selection kernels)."""
    names = (["select_kernel.cu", "select_step.cuh", "select_keys.cuh", "internal.h", "ptx.cuh"] if kernel == "select"
             else ["attn_kernel.cuh", "ptx.cuh", "select_step.cuh", "gather.cuh", "internal.h"])
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "block_sparse_attention_causal_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(f"{kernel}@{workload}")
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------- GPU arm

def workload(name, block=0):
    """The configuration's workload, with the support block size replaced
    when another one is asked for (the generator plants its evidence in
    blocks of that size)."""
    cfg = wl.CONFIGS[name]
    if block and block != cfg.block:
        cfg = cfg.replace(block=block)
    return cfg


def workload_name(name, cfg) -> str:
    base = wl.CONFIGS[name]
    return f"wise_{cfg.name}" + (f"_b{cfg.block}" if cfg.block != base.block else "")


def traffic_key(name, cfg) -> str:
    base = wl.CONFIGS[name]
    return name if cfg.block == base.block else f"{name}_b{cfg.block}"


def device_inputs(cfg, steps, seed, dev, pin=False):
    """Seeded bf16 step inputs [3, B, H, n, d] on the device (and, with pin,
    in pinned host memory too)."""
    import torch
    bits = wl.trajectory_inputs_bf16(cfg, steps, seed=seed)
    host, devs = {}, {}
    for t in steps:
        x = torch.from_numpy(bits.pop(t)).view(torch.bfloat16)
        if pin:
            host[t] = x.pin_memory()
            devs[t] = host[t].to(dev, non_blocking=False)
        else:
            devs[t] = x.to(dev)
    return devs, host


class Timer:
    """CUDA events around launches on one stream, kept per kind."""

    def __init__(self, stream):
        import torch
        self.torch = torch
        self.stream = stream
        self.ev = {}

    def __call__(self, kind, fn, record=True):
        if not record:
            return fn()
        a = self.torch.cuda.Event(enable_timing=True)
        b = self.torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        r = fn()
        b.record(self.stream)
        self.ev.setdefault(kind, []).append((a, b))
        return r

    def ms(self, kind):
        return [a.elapsed_time(b) for a, b in self.ev.get(kind, [])]

    def clear(self):
        self.ev.clear()


def measure_config(wise, name, cfg, dev, seed, passes, reps, peak_tf, inputs=None):
    """One entry of the per-configuration block: the support from the
    window's discovery steps, then `passes` balanced passes (the order of the
    dense and sparse launches alternates between passes), each timing `reps`
    late sparse steps and `reps` dense steps on rotating late-step inputs,
    plus one discovery step with masses and one selection. Each kind's time is
    the median of its per-pass medians, with the inter-quartile range over
    the passes."""
    import torch
    B, H, n, d, blk = cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block
    nb, W = cfg.n_blocks, cfg.window
    step_bytes = 3 * B * H * n * d * 2
    n_late = min(cfg.steps - cfg.t_d, max(2, math.ceil(3 * L2_BYTES / step_bytes)))
    late_steps = list(range(cfg.steps - n_late, cfg.steps))
    if inputs is None:
        inputs, _ = device_inputs(cfg, cfg.window_steps + late_steps, seed, dev)
    stream = torch.cuda.current_stream(dev)
    o = torch.empty((B, H, n, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=dev)
    masses = torch.empty((W, B, H, nb, nb), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, wise.discover_workspace_bytes((B, H, n, d), blk)), dtype=torch.uint8, device=dev)
    lib = wise._lib.load()
    desc = wise._lib.make_desc(B, H, n, d, blk)
    sel_ws = torch.empty(max(16, int(lib.wise_select_workspace(desc, W))), dtype=torch.uint8, device=dev)
    for w, t in enumerate(cfg.window_steps):
        x = inputs[t]
        wise.discover(x[0], x[1], x[2], blk, out=o, lse=lse, mass=masses[w], workspace=ws)
    support = wise.select_support(masses, n, d, blk, cfg.eta, workspace=sel_ws)
    wise.check_device()
    rp = support.row_ptr.cpu().numpy()
    ci = support.col_idx.cpu().numpy()
    sflops = support_flops(rp, ci, nb, blk, d)
    dflops = wise.dense_flops(B, H, n, d)
    entries = tile_entries(rp, ci, B * H, nb, blk)
    timer = Timer(stream)
    wx = inputs[cfg.window_steps[-1]]

    def dense(x):
        return lambda: wise.discover(x[0], x[1], x[2], blk, want_mass=False, out=o, lse=lse)

    def sparse(x):
        return lambda: wise.sparse(x[0], x[1], x[2], support, out=o, lse=lse)

    kinds = ("sparse", "dense", "discover_mass", "select")
    per_pass = {k: [] for k in kinds}
    for p in range(passes + 1):  # pass 0 warms up
        timer.clear()
        order = ("dense", "sparse") if p % 2 == 0 else ("sparse", "dense")
        for r in range(reps):
            x = inputs[late_steps[r % len(late_steps)]]
            for kind in order:
                timer(kind, dense(x) if kind == "dense" else sparse(x))
        timer("discover_mass", lambda: wise.discover(wx[0], wx[1], wx[2], blk, out=o, lse=lse, mass=masses[W - 1],
                                                     workspace=ws))
        timer("select", lambda: wise.select_support(masses, n, d, blk, cfg.eta, support=support, workspace=sel_ws))
        torch.cuda.synchronize(dev)
        if p > 0:
            for k in kinds:
                per_pass[k].append(statistics.median(timer.ms(k)))
    wise.check_device()
    stats = {k: median_iqr(v) for k, v in per_pass.items()}
    sp, dn, ms_, sel = (stats[k][0] for k in kinds)
    setup = setup_cost_ms(sel, ms_, dn, W)
    T, td = cfg.steps, cfg.t_d
    traj = (td - W) * dn + W * ms_ + sel + (T - td) * sp
    r3 = lambda v: round(v, 4)
    return {
        "workload": workload_name(name, cfg), "batch": B, "heads": H, "seq_len": n, "head_dim": d, "block": blk,
        "density": round(float(rp[-1]) / (B * H * nb * (nb + 1) / 2), 4), "nnz": int(rp[-1]),
        "late_step_ms": {"median": r3(sp), "iqr": r3(stats["sparse"][1])},
        "dense_step_ms": {"median": r3(dn), "iqr": r3(stats["dense"][1])},
        "discover_mass_ms": {"median": r3(ms_), "iqr": r3(stats["discover_mass"][1])},
        "select_ms": {"median": r3(sel), "iqr": r3(stats["select"][1])},
        "speedup_vs_dense": round(dn / sp, 3),
        "sparse_tflops": round(sflops / (sp * 1e-3) / 1e12, 2),
        "sparse_tile_tflops": round(tile_flops(entries, blk, d) / (sp * 1e-3) / 1e12, 2),
        "frac": round(sflops / (sp * 1e-3) / 1e12 / peak_tf, 4),
        "dense_tflops": round(dflops / (dn * 1e-3) / 1e12, 2),
        "dense_frac": round(dflops / (dn * 1e-3) / 1e12 / peak_tf, 4),
        "setup_ms": r3(setup),
        "setup_inclusive_speedup": round((T - td) * dn / (setup + (T - td) * sp), 3),
        "trajectory_speedup_from_parts": round(T * dn / traj, 3),
        "timing": f"median of per-pass medians over {passes} balanced passes ({reps} sparse and {reps} dense "
                  f"launches each, on {len(late_steps)} rotating late-step inputs of {step_bytes / 2**20:.0f} MiB), "
                  "iqr = 75th - 25th percentile over the passes",
    }


def h2d_bandwidth(dev, nbytes=1 << 30):
    """One host-to-device copy of `nbytes` from pinned memory (best of 5)."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = float("inf")
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize(dev)
        best = min(best, a.elapsed_time(b))
    return nbytes / (best * 1e-3) / 1e9


def run_gpu(args, rank, world):
    import torch
    import block_sparse_attention_causal_gb300 as wise

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = workload(args.config, args.block)
    B, H, n, d, blk = cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block
    nb = cfg.n_blocks
    T, td, W = cfg.steps, cfg.t_d, cfg.window
    seed = args.seed + 1000 * rank
    peaks, peak_kind = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    # seeded step inputs, bf16, in pinned host memory and resident in HBM
    dev_in, host = device_inputs(cfg, range(T), seed, dev, pin=True)

    stream = torch.cuda.current_stream(dev)
    o = torch.empty((B, H, n, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=dev)
    masses = torch.empty((W, B, H, nb, nb), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, wise.discover_workspace_bytes((B, H, n, d), blk)), dtype=torch.uint8, device=dev)
    lib = wise._lib.load()
    desc = wise._lib.make_desc(B, H, n, d, blk)
    sel_ws = torch.empty(max(16, int(lib.wise_select_workspace(desc, W))), dtype=torch.uint8, device=dev)
    support = wise.select_support(torch.zeros_like(masses), n, d, blk, cfg.eta, workspace=sel_ws)

    # selection fused into the window's discovery launches (nb <= 256), or
    # one selection pass over the window's masses
    fused = args.selection == "fused" and nb <= 256
    sel_state = wise.new_select_state((B, H, n, d), blk, W) if fused else None
    timer = Timer(stream)

    # host-to-device copies of a trajectory's step inputs run on rotating copy
    # streams, so that the copy of a later step overlaps the kernels of the
    # current one; each step's kernels wait for their own inputs only
    copy_streams = [torch.cuda.Stream(dev) for _ in range(max(1, args.copy_streams))]

    def trajectory(inputs, record=False, out_host=None, host_inputs=None):
        launches = 0
        ready = {}
        if host_inputs is not None:
            for t in range(T):
                cs = copy_streams[t % len(copy_streams)]
                cs.wait_stream(stream)  # the previous use of the buffer is done
                with torch.cuda.stream(cs):
                    inputs[t].copy_(host_inputs[t], non_blocking=True)
                ready[t] = torch.cuda.Event()
                ready[t].record(cs)
        for t in range(T):
            if host_inputs is not None:
                stream.wait_event(ready[t])
            q, k, v = inputs[t][0], inputs[t][1], inputs[t][2]
            if t < td:
                w = t - (td - W)
                if w >= 0 and fused:
                    timer("discover_select", lambda: wise.discover_select(
                        q, k, v, blk, step=w, window=W, eta=cfg.eta, select_state=sel_state, out=o, lse=lse,
                        mass=masses[w], workspace=ws), record)
                elif w >= 0:
                    timer("discover_mass", lambda: wise.discover(q, k, v, blk, out=o, lse=lse, mass=masses[w],
                                                                workspace=ws), record)
                else:
                    timer("discover", lambda: wise.discover(q, k, v, blk, want_mass=False, out=o, lse=lse), record)
                launches += 1
                if t == td - 1 and fused:
                    timer("select", lambda: wise.select_finalize(sel_state, B, H, n, d, blk, support=support), record)
                    launches += 1
                elif t == td - 1:
                    timer("select", lambda: wise.select_support(masses, n, d, blk, cfg.eta, support=support,
                                                                workspace=sel_ws), record)
                    launches += 3 if blk == 32 else 2  # Eq 6, finalize (+ the plan of gathered entries)
            else:
                timer("sparse", lambda: wise.sparse(q, k, v, support, out=o, lse=lse), record)
                launches += 1
        if out_host is not None:
            out_host.copy_(o, non_blocking=True)
        return launches

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ------------------------------------------------------------ device-resident timing
    for _ in range(args.warmup):
        trajectory(dev_in)
    wise.check_device()
    timer.clear()
    barrier()
    with ClockSampler(dev.index) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        launches = 0
        for _ in range(args.steps):
            launches += trajectory(dev_in, record=True)
        t1.record(stream)
        barrier()
    wise.check_device()
    traj_ms = t0.elapsed_time(t1) / args.steps
    per = {k_: timer.ms(k_) for k_ in ("discover_mass", "discover_select", "discover", "select", "sparse")}

    # support statistics from the selected support (identical every trajectory)
    rp = support.row_ptr.cpu().numpy()
    ci = support.col_idx.cpu().numpy()
    sparse_flops = support_flops(rp, ci, nb, blk, d)
    entries = tile_entries(rp, ci, B * H, nb, blk)
    sparse_tile_flops = tile_flops(entries, blk, d)
    dense_flops = wise.dense_flops(B, H, n, d)
    density = float(rp[-1]) / (B * H * nb * (nb + 1) / 2)

    # ------------------------------------------------------------ the same trajectory as one CUDA graph
    # (captured once, replayed: no host launch gaps between its launches)
    graph_ms = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            trajectory(dev_in)
        graph.replay()
        barrier()
        wise.check_device()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        g1.record(stream)
        barrier()
        wise.check_device()
        graph_ms = g0.elapsed_time(g1) / args.steps
        del graph
    except RuntimeError as e:  # capture refused: report it, keep the eager numbers
        graph_ms = f"capture failed: {e}"[:160]

    # ------------------------------------------------------------ the library's dense kernel, same late inputs
    dtimer = Timer(stream)
    late = list(range(td, T))
    for _ in range(2):
        for t in late:
            wise.discover(dev_in[t][0], dev_in[t][1], dev_in[t][2], blk, want_mass=False, out=o, lse=lse)
    barrier()
    for _ in range(args.steps):
        for t in late:
            dtimer("dense", lambda: wise.discover(dev_in[t][0], dev_in[t][1], dev_in[t][2], blk, want_mass=False,
                                                  out=o, lse=lse))
    barrier()
    dense_ms = statistics.median(dtimer.ms("dense"))

    # ------------------------------------------------------------ end to end, host buffers
    e2e_in = {t: torch.empty_like(dev_in[t]) for t in range(T)}
    out_host = torch.empty((B, H, n, d), dtype=torch.bfloat16).pin_memory()
    trajectory(e2e_in, host_inputs=host, out_host=out_host)
    barrier()
    e0 = time.perf_counter()
    for _ in range(args.steps):
        trajectory(e2e_in, host_inputs=host, out_host=out_host)
        torch.cuda.synchronize(dev)
    e2e_traj_ms = (time.perf_counter() - e0) * 1e3 / args.steps
    wise.check_device()
    h2d = sum(host[t].numel() * 2 for t in range(T))
    d2h = out_host.numel() * 2
    del e2e_in
    h2d_gbs = h2d_bandwidth(dev)

    # ------------------------------------------------------------ aggregate over ranks
    # the late step's time is the median of the timed launches (one host
    # stall between an event and its launch would otherwise move a mean)
    sparse_ms, sparse_iqr = median_iqr(per["sparse"])
    sparse_mean_ms = sum(per["sparse"]) / len(per["sparse"])
    traj_ms, sparse_ms, e2e_traj_ms = reduce_max_over_ranks([traj_ms, sparse_ms, e2e_traj_ms], world, dev)
    n_late = T - td
    value = whole_job_tflops(sparse_flops, sparse_ms, world)
    # e2e: the same late-step FLOPs over the whole host-to-host trajectory
    e2e_value = whole_job_tflops(n_late * sparse_flops, e2e_traj_ms, world)

    kern_stats = {}
    for k_, vals_ in per.items():
        if vals_:
            med, iqr = median_iqr(vals_)
            kern_stats[k_] = {"launches": len(vals_), "avg_ms": sum(vals_) / len(vals_), "median_ms": med,
                              "iqr_ms": iqr, "total_ms_per_step": sum(vals_) / args.steps}
    dense_tflops = dense_flops / (dense_ms * 1e-3) / 1e12
    for k_ in ("discover", "discover_mass", "discover_select"):
        if k_ in kern_stats:
            kern_stats[k_]["tflops"] = dense_flops / (kern_stats[k_]["avg_ms"] * 1e-3) / 1e12
    if "sparse" in kern_stats:
        kern_stats["sparse"]["tflops"] = sparse_flops / (kern_stats["sparse"]["avg_ms"] * 1e-3) / 1e12
        kern_stats["sparse"]["tile_tflops"] = sparse_tile_flops / (kern_stats["sparse"]["avg_ms"] * 1e-3) / 1e12
    if "select" in kern_stats:
        # read: the window's masses (separate pass) or the row bitmasks and
        # counts (fused); written: the CSR
        read = (B * H * nb * (-(-nb // 32)) * 4 + B * H * nb * 4) if fused else W * B * H * nb * nb * 4
        sel_bytes = read + (B * H * nb + 1) * 4 + rp[-1] * 4
        kern_stats["select"]["gbs"] = sel_bytes / (kern_stats["select"]["avg_ms"] * 1e-3) / 1e9
    mass_kind = "discover_select" if fused else "discover_mass"
    mass_ms = kern_stats[mass_kind]["avg_ms"] if mass_kind in kern_stats else None
    setup_ms = setup_cost_ms(kern_stats["select"]["avg_ms"], mass_ms, dense_ms, W)
    dominant = max((k_ for k_ in kern_stats if k_ != "select"), key=lambda k_: kern_stats[k_]["total_ms_per_step"])
    dom = kern_stats[dominant]
    achieved = dom["tflops"]
    kernel_name = {"sparse": "wise_attn_kernel<sparse>", "discover": "wise_attn_kernel<dense>",
                   "discover_mass": "wise_attn_kernel<dense,mass>",
                   "discover_select": "wise_attn_kernel<dense,mass,select>"}[dominant]
    tkey = traffic_key(args.config, cfg)
    roofline = {"kernel": kernel_name, "bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf,
                "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                "traffic": stored_traffic(dominant, tkey),
                "peak_source": f"bf16_tflops ({peak_kind}, burst)",
                "algorithmic": "4*d FLOPs per admissible query-key pair inside the support"}
    sparse_roof = {"achieved": round(kern_stats["sparse"]["tflops"], 2), "peak": peak_tf,
                   "frac": round(kern_stats["sparse"]["tflops"] / peak_tf, 4),
                   "traffic": stored_traffic("sparse", tkey)}

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(traj_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(args.config, cfg), "batch": B, "heads": H, "seq_len": n,
                   "head_dim": d, "block": blk, "steps_T": T, "t_d": td, "window": W, "eta": cfg.eta,
                   "selection": "fused into discovery" if fused else "separate pass",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "each trajectory reads T distinct step inputs "
                         f"({T * 3 * B * H * n * d * 2 / 1e9:.2f} GB > 129 MB L2)"},
        "late_step_ms": round(sparse_ms, 4), "late_step_iqr_ms": round(sparse_iqr, 4),
        "late_step_mean_ms": round(sparse_mean_ms, 4),
        "dense_step_ms": round(dense_ms, 4),
        "speedup_vs_dense": round(dense_ms / sparse_ms, 3),
        "dense_tflops": round(dense_tflops, 2), "frac_of_bf16_peak": round(value / world / peak_tf, 4),
        "support_density": round(density, 4), "nnz": int(rp[-1]),
        "sparse_useful_tflop_per_step": sparse_flops / 1e12, "dense_tflop_per_step": dense_flops / 1e12,
        "sparse_tile_entries": entries, "sparse_tile_tflop_per_step": sparse_tile_flops / 1e12,
        # setup = the selection launch plus what the window's discovery
        # launches cost beyond the plain dense kernel (masses, fused
        # selection), signed; the raw per-kind times are in "kernels"
        "setup_ms": round(setup_ms, 4),
        "setup_parts_ms": {"select": round(kern_stats["select"]["avg_ms"], 4),
                           "mass_step": None if mass_ms is None else round(mass_ms, 4),
                           "dense_step": round(dense_ms, 4), "window": W},
        "setup_inclusive_speedup": round((n_late * dense_ms) / (setup_ms + n_late * sparse_ms), 3),
        "trajectory_speedup": round(T * dense_ms / traj_ms, 3),
        # the same trajectory captured once as a CUDA graph and replayed
        "trajectory_graph_ms": round(graph_ms, 4) if isinstance(graph_ms, float) else graph_ms,
        "kernels": {k_: {kk: (round(vv, 5) if isinstance(vv, float) else vv) for kk, vv in s.items()}
                    for k_, s in kern_stats.items()},
        "roofline": roofline, "roofline_sparse": sparse_roof,
        "clocks": clk.summary(),
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_traj_ms, 3),
                "h2d_gbs_achieved": round(h2d / (e2e_traj_ms * 1e-3) / 1e9, 1),
                "h2d_gbs_one_copy": round(h2d_gbs, 1)},
        "gpu_launches": launches,
    }
    result["support_quality"] = support_quality(wise, cfg, dev_in, support, masses, ws, o, lse)

    # ------------------------------------------------------------ per-configuration block
    configs = {}
    sweep = [] if args.sweep == "none" else [c for c in args.sweep.split(",") if c]
    for name in sweep + [args.config]:
        if name in configs:
            continue
        ccfg = cfg if name == args.config else workload(name)
        if name == args.config:
            entry = measure_config(wise, name, ccfg, dev, seed, args.passes, args.reps, peak_tf, inputs=dev_in)
        else:
            entry = measure_config(wise, name, ccfg, dev, seed, args.passes, args.reps, peak_tf)
        configs[name] = entry
        torch.cuda.empty_cache()
    result["configs"] = configs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows_all = support.to_lists()
        by_head = [((b_, h_), rows_all[(b_ * H + h_) * nb:(b_ * H + h_ + 1) * nb])
                   for b_ in range(B) for h_ in range(H)]
        result["cpu_baseline"] = cpu_baseline(cfg, seed, by_head)
    return result


def support_quality(wise, cfg, dev_in, frozen, masses, ws, o, lse):
    """WISE's own support diagnostics on this workload, outside the timed
    region: block masses of unrestricted attention at every step, the rolling
    working sets W(t) (union of the step supports of steps max(0, t-3)..t,
    App. C.2 Eq 23), their adjacent Jaccard index (Eq 24) at the discovery
    depth, the drift J(W(t_d - 1), W(T - 1)), and the retained future
    attention mass of the frozen support at each late step (App. B)."""
    import torch
    B, H, n, d, blk = cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block
    step_mass = []
    for t in range(cfg.steps):
        m = torch.empty_like(masses[0])
        wise.discover(dev_in[t][0], dev_in[t][1], dev_in[t][2], blk, out=o, lse=lse, mass=m, workspace=ws)
        step_mass.append(m)
    rolling = [wise.select_support(torch.stack(step_mass[max(0, t - 3):t + 1]).contiguous(), n, d, blk, cfg.eta)
               for t in range(cfg.steps)]
    td = cfg.t_d
    adj = [float(wise.support_jaccard(rolling[t - 1], rolling[t])[2].mean().item()) for t in range(1, cfg.steps)]
    retained = [float(wise.retained_mass(step_mass[t], frozen)[1].mean().item()) for t in range(td, cfg.steps)]
    drift = float(wise.support_jaccard(rolling[td - 1], rolling[cfg.steps - 1])[2].mean().item())
    # the early-static controls of App. B (Eqs 19-22) against the same future steps
    static95 = wise.select_support(step_mass[0][None].contiguous(), n, d, blk, 0.95, 0)
    controls = {"static95": static95, "mass_matched": wise.select_control(step_mass[0], frozen, "mass"),
                "size_matched": wise.select_control(step_mass[0], frozen, "size")}
    causal_blocks = B * H * cfg.n_blocks * (cfg.n_blocks + 1) / 2
    ctl = {}
    for name, sup in controls.items():
        kept = [float(wise.retained_mass(step_mass[t], sup)[1].mean().item()) for t in range(td, cfg.steps)]
        ctl[name] = {"retained_future_mass": round(sum(kept) / len(kept), 5),
                     "density": round(int(sup.nnz.item()) / causal_blocks, 4)}
    wise.check_device()
    return {"retained_future_mass": {"mean": round(sum(retained) / len(retained), 5),
                                     "per_late_step": [round(x, 5) for x in retained]},
            "rolling_jaccard_adjacent": [round(x, 5) for x in adj],
            "rolling_jaccard_at_td": round(adj[td - 2], 5) if td >= 2 else None,
            "drift_jaccard_td_to_T": round(drift, 5),
            "wise_density": round(int(frozen.nnz.item()) / causal_blocks, 4),
            "controls": ctl,
            "definitions": "retained mass: App. B; rolling sets: Eq 23 (0-indexed steps); Jaccard: Eq 24"}


def profile_kernel(args):
    """A few launches of one kernel on one configuration (for ncu captures):
    the window's discovery steps and the selection run first (untimed
    set-up), then `--steps` launches of the chosen kind."""
    import torch
    import block_sparse_attention_causal_gb300 as wise
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cfg = workload(args.config, args.block)
    B, H, n, d, blk = cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block
    nb, W = cfg.n_blocks, cfg.window
    late = cfg.steps - 1
    inputs, _ = device_inputs(cfg, cfg.window_steps + [late], args.seed, dev)
    o = torch.empty((B, H, n, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=dev)
    masses = torch.empty((W, B, H, nb, nb), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, wise.discover_workspace_bytes((B, H, n, d), blk)), dtype=torch.uint8, device=dev)
    for w, t in enumerate(cfg.window_steps):
        x = inputs[t]
        wise.discover(x[0], x[1], x[2], blk, out=o, lse=lse, mass=masses[w], workspace=ws)
    support = wise.select_support(masses, n, d, blk, cfg.eta)
    x, wx = inputs[late], inputs[cfg.window_steps[-1]]
    launch = {
        "discover": lambda: wise.discover(x[0], x[1], x[2], blk, want_mass=False, out=o, lse=lse),
        "discover_mass": lambda: wise.discover(wx[0], wx[1], wx[2], blk, out=o, lse=lse, mass=masses[W - 1],
                                               workspace=ws),
        "sparse": lambda: wise.sparse(x[0], x[1], x[2], support, out=o, lse=lse),
        "select": lambda: wise.select_support(masses, n, d, blk, cfg.eta, support=support),
    }[args.profile_kernel]
    torch.cuda.synchronize(dev)
    for _ in range(args.steps):
        launch()
    torch.cuda.synchronize(dev)
    wise.check_device()
    rp = support.row_ptr.cpu().numpy()
    print(json.dumps({"profile_kernel": args.profile_kernel, "workload": workload_name(args.config, cfg),
                      "launches": args.steps, "nnz": int(rp[-1]),
                      "density": round(float(rp[-1]) / (B * H * nb * (nb + 1) / 2), 4),
                      "source_hash": kernel_source_hash("select" if args.profile_kernel == "select" else "attn")}))


# --------------------------------------------------------------------------- oracle (CPU) arm

def _rows_flops(rows, qbs, cfg):
    flops = 0.0
    for qb in qbs:
        for b in rows[qb]:
            flops += 4.0 * cfg.head_dim * (cfg.block * (cfg.block + 1) / 2 if b == qb else cfg.block ** 2)
    return flops


def _sample_query_blocks(nb, count):
    """`count` query blocks spread evenly over 0..nb-1, the last included."""
    if count >= nb:
        return list(range(nb))
    return sorted(set(int(round(x)) for x in np.linspace(0, nb - 1, count)))


def _oracle_late_rows(cfg, x, rows, qbs):
    """The fp64 oracle's late step (Eq 8) for the query blocks `qbs` of one
    (batch, head) slice x [3, n, d]; returns (useful FLOPs, seconds)."""
    from oracle import wise_oracle as O
    t0 = time.perf_counter()
    O.causal_attention(x[0], x[1], x[2], cfg.block, support=rows, query_blocks=qbs)
    return _rows_flops(rows, qbs, cfg), time.perf_counter() - t0


def _oracle_rows(cfg, seed, b, h, qbs):
    """The head's working set for the query blocks `qbs` as the oracle
    selects it (discovery masses of those rows on the window steps, then
    Eq 6); other rows are empty."""
    from oracle import wise_oracle as O
    g = wl.HeadGenerator(cfg, b, h, seed)
    masses = []
    for t in cfg.window_steps:
        x = g.step(t).astype(np.float64)
        masses.append(O.block_mass(x[0], x[1], cfg.block, query_blocks=qbs))
    rows = [[] for _ in range(cfg.n_blocks)]
    for qb in qbs:
        s = set()
        for r in masses:
            s |= O.step_support(r[qb], qb, cfg.eta)
        rows[qb] = sorted(s | {0, qb})
    return rows


def cpu_baseline(cfg, seed, rows_by_head, budget_s: float = 10.0, chunk: int = 16):
    """Oracle late steps on the machine's host cores, `chunk` query blocks at a
    time over successive heads (with the support the GPU selected for each
    head), until about `budget_s` of CPU work."""
    cores = len(os.sched_getaffinity(0))
    flops = secs = 0.0
    blocks = heads = 0
    for (b, h), rows in rows_by_head:
        x = wl.HeadGenerator(cfg, b, h, seed).step(cfg.steps - 1).astype(np.float64)
        heads += 1
        for s in range(0, cfg.n_blocks, chunk):
            qbs = list(range(s, min(s + chunk, cfg.n_blocks)))
            f, dt = _oracle_late_rows(cfg, x, rows, qbs)
            flops += f
            secs += dt
            blocks += len(qbs)
            if secs >= budget_s:
                break
        if secs >= budget_s:
            break
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"late step (Eq 8) of {blocks} query blocks ({heads} of {cfg.batch * cfg.heads} (batch, head) "
                      f"slices) of {cfg.name}, fp64 NumPy oracle over each head's GPU-selected support; "
                      f"{secs:.1f} s of CPU work"}


def run_reference(args, rank, world):
    """The oracle arm: per step, the late step of one (batch, head) slice over
    a fixed sample of query blocks, through the fp64 oracle, over the support
    the oracle itself selects for head 0 at those query blocks (selection and
    input generation untimed)."""
    cfg = workload(args.config, args.block)
    qbs = _sample_query_blocks(cfg.n_blocks, 8)
    rows = _oracle_rows(cfg, args.seed, 0, 0, qbs)

    def step(j):
        b, h = divmod(j % (cfg.batch * cfg.heads), cfg.heads)
        x = wl.HeadGenerator(cfg, b, h, args.seed).step(cfg.steps - 1).astype(np.float64)
        return _oracle_late_rows(cfg, x, rows, qbs)

    for j in range(args.warmup):
        step(j)
    tot_f = tot_t = 0.0
    for j in range(args.steps):
        f, dt = step(j)
        tot_f += f
        tot_t += dt
    value = tot_f / tot_t / 1e12
    cores = len(os.sched_getaffinity(0))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / max(1, args.steps) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(args.config, cfg), "batch": cfg.batch, "heads": cfg.heads,
                   "seq_len": cfg.seq_len, "head_dim": cfg.head_dim, "block": cfg.block},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: the late step (Eq 8) of {len(qbs)} of {cfg.n_blocks} query blocks of "
                                   f"one (batch, head) slice of {cfg.name} over the working set the oracle selects "
                                   "for head 0 (fp64 NumPy; selection and input generation untimed)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(wl.CONFIGS))
    ap.add_argument("--impl", default="wise", choices=["wise", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--selection", default="separate", choices=["fused", "separate"],
                    help="Eq 6 selection fused into the window's discovery launches, or a separate pass")
    ap.add_argument("--block", type=int, default=0, choices=[0, 32, 64, 128],
                    help="support block size (0: the configuration's own)")
    ap.add_argument("--sweep", default=DEFAULT_SWEEP,
                    help="comma-separated configurations of the per-configuration block, or 'none'")
    ap.add_argument("--passes", type=int, default=10, help="balanced passes per configuration")
    ap.add_argument("--reps", type=int, default=4, help="sparse and dense launches per pass")
    ap.add_argument("--copy-streams", type=int, default=1,
                    help="streams the end-to-end run spreads its host-to-device copies over")
    ap.add_argument("--profile-kernel", default=None, choices=["discover", "discover_mass", "sparse", "select"],
                    help="only launch this kernel --steps times on --config (for ncu)")
    args = ap.parse_args()
    if args.profile_kernel:
        profile_kernel(args)
        return
    args.warmup = max(args.warmup, 3) if args.impl == "wise" else args.warmup
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # the CPU oracle arm: rank 0 alone runs and prints; other ranks leave
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)))
        return
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_gpu(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
