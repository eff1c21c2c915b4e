"""The hot path inside a CUDA graph: a whole trajectory (discovery with block
masses over the window, the Eq 6 selection with its CSR and work order, late
sparse steps) is captured once and replayed; the replay must give the same
bits as the eager launches. Runs through the C ABI like every GPU test."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

wise = pytest.importorskip("block_sparse_attention_causal_gb300")


def _trajectory(cfg, xs, bufs):
    B, H, n, d, blk = cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block
    o, lse, masses, ws, sel_ws, support, outs = bufs
    W, td = cfg.window, cfg.t_d
    for t in range(cfg.steps):
        q, k, v = xs[t][0], xs[t][1], xs[t][2]
        if t < td:
            w = t - (td - W)
            if w >= 0:
                wise.discover(q, k, v, blk, out=o, lse=lse, mass=masses[w], workspace=ws)
            else:
                wise.discover(q, k, v, blk, want_mass=False, out=o, lse=lse)
            if t == td - 1:
                wise.select_support(masses, n, d, blk, cfg.eta, support=support, workspace=sel_ws)
        else:
            wise.sparse(q, k, v, support, out=outs[t][0], lse=outs[t][1])


@pytest.mark.parametrize("block", [64, 32])
def test_trajectory_replayed_from_a_cuda_graph_matches_eager(block):
    cfg = wl.CONFIGS["tiny"].replace(name=f"tiny_graph_b{block}", seq_len=512, block=block)
    B, H, n, d, blk = cfg.batch, cfg.heads, cfg.seq_len, cfg.head_dim, cfg.block
    nb = n // blk
    dev = torch.device("cuda", 0)
    bits = wl.trajectory_inputs_bf16(cfg, range(cfg.steps), processes=1)
    xs = {t: torch.from_numpy(bits[t]).view(torch.bfloat16).to(dev) for t in bits}
    o = torch.empty((B, H, n, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=dev)
    masses = torch.zeros((cfg.window, B, H, nb, nb), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, wise.discover_workspace_bytes((B, H, n, d), blk)), dtype=torch.uint8, device=dev)
    # the eager run sizes and allocates the support (and, for blocks of 32, its plan)
    support = wise.select_support(masses, n, d, blk, cfg.eta)
    lib = wise._lib.load()
    desc = wise._lib.make_desc(B, H, n, d, blk)
    sel_ws = torch.empty(max(16, int(lib.wise_select_workspace(desc, cfg.window))), dtype=torch.uint8, device=dev)
    outs = {t: (torch.empty((B, H, n, d), dtype=torch.bfloat16, device=dev),
                torch.empty((B, H, n), dtype=torch.float32, device=dev)) for t in range(cfg.t_d, cfg.steps)}
    bufs = (o, lse, masses, ws, sel_ws, support, outs)
    _trajectory(cfg, xs, bufs)
    wise.check_device()
    eager = {t: (a.clone(), b.clone()) for t, (a, b) in outs.items()}
    eager_rp, eager_ci = support.row_ptr.clone(), support.col_idx.clone()
    for a, b in outs.values():
        a.zero_()
        b.zero_()
    support.row_ptr.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _trajectory(cfg, xs, bufs)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize(dev)
    wise.check_device()
    assert torch.equal(support.row_ptr, eager_rp)
    assert torch.equal(support.col_idx[:int(eager_rp[-1])], eager_ci[:int(eager_rp[-1])])
    for t, (a, b) in outs.items():
        assert torch.equal(a, eager[t][0]) and torch.equal(b, eager[t][1]), t
