"""Benchmark of the WISE hot path on GB300.

One step = one recurrent-attention trajectory of the workload: t_d discovery
steps (dense causal attention; block masses on the last min(4, t_d) steps),
one working-set selection, and T - t_d late steps of block-sparse attention
over the selected support, each step on its own seeded Q/K/V.

`value` is the late-step sparse attention throughput in useful TFLOP/s (4 d
per admissible query-key pair inside the support), measured with CUDA events
on the launching stream inside the timed trajectories. The line also carries
ms per trajectory, the late-step time against the library's own dense kernel
on the same inputs, the roofline of the dominant kernel, an end-to-end figure
through the public API with host buffers, and the fp64 CPU oracle timed on a
bounded sample (cpu_baseline).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 4k] [--impl wise|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
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


def setup_cost_ms(select_ms: float, mass_step_ms, dense_ms: float, window: int) -> float:
    """Cost of building the support: the selection launch plus what each of
    the window's discovery launches costs beyond the plain dense kernel (the
    mass epilogue, or the fused selection); a mass step measured faster than
    the dense kernel adds nothing."""
    extra = 0.0 if mass_step_ms is None else max(0.0, mass_step_ms - dense_ms)
    return select_ms + window * extra


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("attn_kernel.cuh", "ptx.cuh", "select_step.cuh", "internal.h"):
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
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------- GPU arm

def workload(args):
    """The configuration's workload, with the support block size replaced
    when --block asks for another one (the generator plants its evidence in
    blocks of that size)."""
    cfg = wl.CONFIGS[args.config]
    if args.block and args.block != cfg.block:
        cfg = cfg.replace(block=args.block)
    return cfg


def workload_name(args, cfg) -> str:
    base = wl.CONFIGS[args.config]
    return f"wise_{cfg.name}" + (f"_b{cfg.block}" if cfg.block != base.block else "")


def traffic_key(args) -> str:
    base = wl.CONFIGS[args.config]
    return args.config if not args.block or args.block == base.block else f"{args.config}_b{args.block}"


def run_gpu(args, rank, world):
    import torch
    import block_sparse_attention_causal_gb300 as wise

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = workload(args)
    B, H, n, d, blk = cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block
    nb = cfg.n_blocks
    T, td, W = cfg.steps, cfg.t_d, cfg.window
    seed = args.seed + 1000 * rank

    # seeded step inputs, bf16, in pinned host memory and resident in HBM
    steps_np = wl.trajectory_inputs(cfg, range(T), seed=seed)
    host = {}
    dev_in = {}
    for t in range(T):
        x = torch.from_numpy(steps_np[t]).to(torch.bfloat16)
        host[t] = x.pin_memory()
        dev_in[t] = x.to(dev)
    del steps_np

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
    names = ["discover_mass", "discover_select", "discover", "select", "sparse"]
    ev = {k: [] for k in names}

    def call(kind, fn, record):
        if record:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ev[kind].append((a, b))
        else:
            fn()

    # host-to-device copies of a trajectory's step inputs run on rotating copy
    # streams, so that the copy of a later step overlaps the kernels of the
    # current one; each step's kernels wait for their own inputs only
    copy_streams = [torch.cuda.Stream(dev) for _ in range(4)]

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
                    call("discover_select", lambda: wise.discover_select(
                        q, k, v, blk, step=w, window=W, eta=cfg.eta, select_state=sel_state, out=o, lse=lse,
                        mass=masses[w], workspace=ws), record)
                elif w >= 0:
                    call("discover_mass", lambda: wise.discover(q, k, v, blk, out=o, lse=lse, mass=masses[w],
                                                               workspace=ws), record)
                else:
                    call("discover", lambda: wise.discover(q, k, v, blk, want_mass=False, out=o, lse=lse), record)
                launches += 1
                if t == td - 1 and fused:
                    call("select", lambda: wise.select_finalize(sel_state, B, H, n, d, blk, support=support), record)
                    launches += 1
                elif t == td - 1:
                    call("select", lambda: wise.select_support(masses, n, d, blk, cfg.eta, support=support,
                                                               workspace=sel_ws), record)
                    launches += 2
            else:
                call("sparse", lambda: wise.sparse(q, k, v, support, out=o, lse=lse), record)
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
    for k_ in ev:
        ev[k_].clear()
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
    per = {k_: [a.elapsed_time(b) for a, b in v_] for k_, v_ in ev.items()}

    # support statistics from the selected support (identical every trajectory)
    rp = support.row_ptr.cpu().numpy()
    ci = support.col_idx.cpu().numpy()
    sparse_flops = support_flops(rp, ci, nb, blk, d)
    entries = tile_entries(rp, ci, B * H, nb, blk)
    sparse_tile_flops = tile_flops(entries, blk, d)
    dense_flops = wise.dense_flops(B, H, n, d)
    density = float(rp[-1]) / (B * H * nb * (nb + 1) / 2)

    # ------------------------------------------------------------ the library's dense kernel, same late inputs
    dense_ev = []
    late = list(range(td, T))
    for _ in range(2):
        for t in late:
            wise.discover(dev_in[t][0], dev_in[t][1], dev_in[t][2], blk, want_mass=False, out=o, lse=lse)
    barrier()
    for _ in range(args.steps):
        for t in late:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            wise.discover(dev_in[t][0], dev_in[t][1], dev_in[t][2], blk, want_mass=False, out=o, lse=lse)
            b.record(stream)
            dense_ev.append((a, b))
    barrier()
    dense_ms = statistics.median([a.elapsed_time(b) for a, b in dense_ev])

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

    # ------------------------------------------------------------ aggregate over ranks
    sparse_ms = statistics.median(per["sparse"])
    sparse_sum_ms = sum(per["sparse"]) / args.steps
    traj_ms, sparse_sum_ms, e2e_traj_ms = reduce_max_over_ranks([traj_ms, sparse_sum_ms, e2e_traj_ms], world, dev)
    n_late = T - td
    value = whole_job_tflops(n_late * sparse_flops, sparse_sum_ms, world)
    # e2e: the same late-step FLOPs over the whole host-to-host trajectory
    e2e_value = whole_job_tflops(n_late * sparse_flops, e2e_traj_ms, world)

    peaks, peak_kind = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    kern_stats = {}
    for k_, vals_ in per.items():
        if vals_:
            kern_stats[k_] = {"launches": len(vals_), "avg_ms": sum(vals_) / len(vals_),
                              "total_ms_per_step": sum(vals_) / args.steps}
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
    setup_ms = setup_cost_ms(kern_stats["select"]["avg_ms"],
                             kern_stats[mass_kind]["avg_ms"] if mass_kind in kern_stats else None, dense_ms, W)
    dominant = max((k_ for k_ in kern_stats if k_ != "select"), key=lambda k_: kern_stats[k_]["total_ms_per_step"])
    dom = kern_stats[dominant]
    achieved = dom["tflops"]
    kernel_name = {"sparse": "wise_attn_kernel<sparse>", "discover": "wise_attn_kernel<dense>",
                   "discover_mass": "wise_attn_kernel<dense,mass>",
                   "discover_select": "wise_attn_kernel<dense,mass,select>"}[dominant]
    roofline = {"kernel": kernel_name, "bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf,
                "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                "traffic": stored_traffic(dominant, traffic_key(args)),
                "peak_source": f"bf16_tflops ({peak_kind}, burst)",
                "algorithmic": "4*d FLOPs per admissible query-key pair inside the support"}
    sparse_roof = {"achieved": round(kern_stats["sparse"]["tflops"], 2), "peak": peak_tf,
                   "frac": round(kern_stats["sparse"]["tflops"] / peak_tf, 4),
                   "traffic": stored_traffic("sparse", traffic_key(args))}

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(traj_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(args, cfg), "batch": B, "heads": H, "seq_len": n, "head_dim": d,
                   "block": blk, "steps_T": T, "t_d": td, "window": W, "eta": cfg.eta,
                   "selection": "fused into discovery" if fused else "separate pass",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "each trajectory reads T distinct step inputs "
                         f"({T * 3 * B * H * n * d * 2 / 1e9:.2f} GB > 129 MB L2)"},
        "late_step_ms": round(sparse_ms, 4), "dense_step_ms": round(dense_ms, 4),
        "speedup_vs_dense": round(dense_ms / sparse_ms, 3),
        "dense_tflops": round(dense_tflops, 2), "frac_of_bf16_peak": round(value / world / peak_tf, 4),
        "support_density": round(density, 4), "nnz": int(rp[-1]),
        "sparse_useful_tflop_per_step": sparse_flops / 1e12, "dense_tflop_per_step": dense_flops / 1e12,
        "sparse_tile_entries": entries, "sparse_tile_tflop_per_step": sparse_tile_flops / 1e12,
        # setup = the selection launch plus what the window's discovery
        # launches cost beyond the plain dense kernel (masses, fused selection)
        "setup_ms": round(setup_ms, 4),
        "setup_inclusive_speedup": round((n_late * dense_ms) / (setup_ms + n_late * sparse_ms), 3),
        "trajectory_speedup": round(T * dense_ms / traj_ms, 3),
        "kernels": {k_: {kk: (round(vv, 5) if isinstance(vv, float) else vv) for kk, vv in s.items()}
                    for k_, s in kern_stats.items()},
        "roofline": roofline, "roofline_sparse": sparse_roof,
        "clocks": clk.summary(),
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_traj_ms, 3)},
        "gpu_launches": launches,
    }
    result["support_quality"] = support_quality(wise, cfg, dev_in, support, masses, ws, o, lse)
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


# --------------------------------------------------------------------------- oracle (CPU) arm

def _head_support_flops(rows, cfg):
    flops = 0.0
    for qb, row in enumerate(rows):
        for b in row:
            flops += 4.0 * cfg.head_dim * (cfg.block * (cfg.block + 1) / 2 if b == qb else cfg.block ** 2)
    return flops


def _oracle_late_step(cfg, seed, b, h, rows):
    """The fp64 oracle's late step (Eq 8) for one (batch, head) over `rows`;
    returns (useful FLOPs, seconds)."""
    from oracle import wise_oracle as O
    x = wl.HeadGenerator(cfg, b, h, seed).step(cfg.steps - 1).astype(np.float64)
    t0 = time.perf_counter()
    O.causal_attention(x[0], x[1], x[2], cfg.block, support=rows)
    return _head_support_flops(rows, cfg), time.perf_counter() - t0


def _oracle_rows(cfg, seed, b, h):
    """The head's working set as the oracle selects it (discovery masses on the
    window steps, then Eq 6)."""
    from oracle import wise_oracle as O
    g = wl.HeadGenerator(cfg, b, h, seed)
    masses = []
    for t in cfg.window_steps:
        x = g.step(t).astype(np.float64)
        masses.append(O.block_mass(x[0], x[1], cfg.block))
    return O.working_set(masses, cfg.eta)


def cpu_baseline(cfg, seed, rows_by_head, budget_s: float = 10.0):
    """Oracle late steps on the machine's host cores over successive heads (with the
    support the GPU selected for each) until about `budget_s` of CPU work."""
    cores = len(os.sched_getaffinity(0))
    flops = secs = 0.0
    heads = 0
    for (b, h), rows in rows_by_head:
        f, dt = _oracle_late_step(cfg, seed, b, h, rows)
        flops += f
        secs += dt
        heads += 1
        if secs >= budget_s:
            break
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"late step (Eq 8) of {heads} of {cfg.batch * cfg.heads} (batch, head) slices of {cfg.name}, "
                      f"fp64 NumPy oracle over each head's selected support; {secs:.1f} s of CPU work"}


def run_reference(args, rank, world):
    """The oracle arm: per step, one head's late step through the fp64 oracle
    over the support the oracle itself selects (selection untimed)."""
    cfg = workload(args)
    rows = _oracle_rows(cfg, args.seed, 0, 0)
    for _ in range(args.warmup):
        _oracle_late_step(cfg, args.seed, 0, 0, rows)
    tot_f = tot_t = 0.0
    for j in range(args.steps):
        h = j % cfg.heads
        f, dt = _oracle_late_step(cfg, args.seed, 0, h, rows)
        tot_f += f
        tot_t += dt
    value = tot_f / tot_t / 1e12
    cores = len(os.sched_getaffinity(0))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / max(1, args.steps) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(args, cfg), "batch": cfg.batch, "heads": cfg.heads,
                   "seq_len": cfg.seq_len, "head_dim": cfg.head_dim, "block": cfg.block},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: the late step (Eq 8) of one (batch, head) slice of {cfg.name} over "
                                   f"the working set the oracle selects for head 0 (fp64 NumPy, selection untimed)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="4k", choices=sorted(wl.CONFIGS))
    ap.add_argument("--impl", default="wise", choices=["wise", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--selection", default="separate", choices=["fused", "separate"],
                    help="Eq 6 selection fused into the window's discovery launches, or a separate pass")
    ap.add_argument("--block", type=int, default=0, choices=[0, 32, 64, 128],
                    help="support block size (0: the configuration's own)")
    args = ap.parse_args()
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
