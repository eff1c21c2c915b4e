"""The seeded input generator: bf16 rounding, determinism, planted structure."""
import numpy as np
import torch

import workloads as wl


def test_bf16_round_matches_torch_rne():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, -1e-30], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(wl.bf16_round(x), ref)
    bits = wl.bf16_bits(wl.bf16_round(x))
    assert np.array_equal(bits, torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_generator_is_deterministic_and_per_head():
    cfg = wl.CONFIGS["tiny"]
    a = wl.HeadGenerator(cfg, 0, 1).step(2)
    b = wl.HeadGenerator(cfg, 0, 1).step(2)
    c = wl.HeadGenerator(cfg, 0, 0).step(2)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    full = wl.step_inputs(cfg, 2)
    assert np.array_equal(full[:, 0, 1], a)


def test_noise_shrinks_with_step_and_evidence_is_planted():
    cfg = wl.CONFIGS["tiny"]
    g = wl.HeadGenerator(cfg, 0, 0)
    d0 = np.abs(g.step(0) - g.base).mean()
    d3 = np.abs(g.step(3) - g.base).mean()
    assert d3 < d0
    assert len(g.evidence_blocks) == cfg.n_evidence
    assert len(set(g.evidence_blocks.tolist())) == cfg.n_evidence


def test_config_table():
    c = wl.CONFIGS["4k"]
    assert (c.batch, c.heads, c.head_dim, c.seq_len, c.block, c.t_d, c.window) == (1, 32, 128, 4096, 128, 3, 3)
    assert wl.CONFIGS["tiny"].window_steps == [0, 1]
    assert wl.CONFIGS["8k_b4"].window_steps == [0, 1, 2, 3]
    assert set(k for k in wl.CONFIGS if k.startswith("sweep")) == {"sweep_2k", "sweep_4k", "sweep_8k", "sweep_16k", "sweep_32k"}


def test_parallel_bf16_generation_matches_the_serial_generator():
    cfg = wl.CONFIGS["tiny"].replace(heads=3)
    serial = wl.trajectory_inputs(cfg, [0, 3])
    for procs in (1, 2):
        bits = wl.trajectory_inputs_bf16(cfg, [0, 3], processes=procs)
        for t in (0, 3):
            assert bits[t].dtype == np.uint16
            assert np.array_equal(bits[t], wl.bf16_bits(serial[t]))
