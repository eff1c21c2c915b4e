"""Host-side logic of the benchmark: FLOP counting and the multi-rank
aggregation (two gloo ranks on CPU)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_support_flops_counts_admissible_pairs():
    # nb = 3, block 4, one head: rows {0}, {0,1}, {1,2}
    rp = np.array([0, 1, 3, 5], np.int32)
    ci = np.array([0, 0, 1, 1, 2], np.int32)
    d, blk = 8, 4
    brute = 0
    rows = [[0], [0, 1], [1, 2]]
    for q, row in enumerate(rows):
        for i in range(q * blk, (q + 1) * blk):
            for b in row:
                brute += sum(1 for j in range(b * blk, (b + 1) * blk) if j <= i)
    assert bench.support_flops(rp, ci, 3, blk, d) == 4.0 * d * brute


def test_setup_cost_counts_selection_and_window_overhead():
    # selection 0.03 ms; three window steps at 0.13 ms against a 0.12 ms
    # dense kernel: 0.03 + 3 * 0.01
    assert bench.setup_cost_ms(0.03, 0.13, 0.12, 3) == pytest.approx(0.06)
    # no mass steps timed: the selection alone
    assert bench.setup_cost_ms(0.03, None, 0.12, 3) == pytest.approx(0.03)
    # signed: a mass step measured below the dense kernel lowers the figure
    # (timing noise must be able to move it both ways)
    assert bench.setup_cost_ms(0.03, 0.11, 0.12, 3) == pytest.approx(0.0)


def test_median_iqr():
    med, iqr = bench.median_iqr([1.0, 2.0, 3.0, 4.0, 100.0])
    assert med == 3.0 and iqr == pytest.approx(2.0)


def test_reference_sample_spreads_query_blocks():
    assert bench._sample_query_blocks(256, 8) == [0, 36, 73, 109, 146, 182, 219, 255]
    assert bench._sample_query_blocks(4, 8) == [0, 1, 2, 3]


def test_tile_entries_count_what_the_scheduler_forms():
    # one head, nb = 6 blocks of 32: two 128-row tiles, the second ragged
    # (query blocks 4 and 5 only). Tile 0's rows list {0, 1, 2, 3}: one
    # gathered entry; tile 1's list {0, 4, 5}: one.
    rows = [[0], [0, 1], [1, 2], [0, 3], [0, 4], [4, 5]]
    rp = np.cumsum([0] + [len(r) for r in rows]).astype(np.int32)
    ci = np.array(sum(rows, []), np.int32)
    assert bench.tile_entries(rp, ci, 1, 6, 32) == 2
    # six distinct blocks in tile 1 need two entries
    rows2 = [[0], [0, 1], [1, 2], [0, 2, 3], [0, 1, 2, 4], [3, 5]]
    rp2 = np.cumsum([0] + [len(r) for r in rows2]).astype(np.int32)
    ci2 = np.array(sum(rows2, []), np.int32)
    assert bench.tile_entries(rp2, ci2, 1, 6, 32) == 1 + 2
    # blocks of 64: the union of two rows per tile ({0,1}, {0,1,2,3}, {0,4,5});
    # of 128: every listed block
    assert bench.tile_entries(rp, ci, 1, 6, 64) == 2 + 4 + 3
    assert bench.tile_entries(rp, ci, 1, 6, 128) == len(ci)
    assert bench.tile_flops(3, 64, 128) == 4.0 * 128 * 128 * 64 * 3


def test_whole_job_value_is_weak_scaling():
    assert bench.whole_job_tflops(2e12, 1000.0, 1) == pytest.approx(2.0)
    assert bench.whole_job_tflops(2e12, 1000.0, 4) == pytest.approx(8.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vals = bench.reduce_max_over_ranks([1.0 + rank, 5.0 - rank, 2.0], world)
    out[rank] = vals
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0] == [2.0, 5.0, 2.0] and out[1] == [2.0, 5.0, 2.0]
