"""Failure handling on the GPU without a fault.

Every wait in the library's kernels is bounded. The library's self-check
launches one kernel whose only wait is on a barrier nothing arrives on,
through the same wait routine with a 20 ms limit: the wait must run out,
the device error word must read WISE_ERR_DEVICE_TIMEOUT, and the context
must stay usable, so that the next attention call runs clean and matches
the oracle.
"""
import time

import numpy as np
import pytest
import torch

import block_sparse_attention_causal_gb300 as wise
from block_sparse_attention_causal_gb300 import _lib
from oracle import wise_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def test_expired_wait_reports_timeout_and_the_context_stays_usable():
    lib = _lib.load()
    stream = torch.cuda.current_stream()
    assert wise.device_status() == _lib.WISE_OK  # nothing pending from earlier tests
    t0 = time.perf_counter()
    assert lib.wise_wait_expiry_check(stream.cuda_stream) == _lib.WISE_OK
    assert wise.device_status() == _lib.WISE_ERR_DEVICE_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.015 <= elapsed < 1.5, f"the 20 ms wait took {elapsed:.3f} s"
    # the status read cleared the word, and the next launches run clean
    assert wise.device_status() == _lib.WISE_OK
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 1, 2, 384, 128)).astype(np.float32)
    t = torch.from_numpy(x).to(torch.bfloat16)
    xr = t.float().numpy().astype(np.float64)
    q, k, v = (t[i].contiguous().cuda() for i in range(3))
    o, lse, mass = wise.discover(q, k, v, 128, out_dtype=torch.float32)
    assert wise.device_status() == _lib.WISE_OK
    o_ref, lse_ref, r_ref = O.discover(xr[0], xr[1], xr[2], 128)
    assert np.max(np.abs(o.cpu().numpy() - o_ref)) <= 1e-2
    assert np.max(np.abs(mass.cpu().numpy() - r_ref)) <= 1e-3
    # twice in a row: the self-check leaves nothing behind
    assert lib.wise_wait_expiry_check(stream.cuda_stream) == _lib.WISE_OK
    assert wise.device_status() == _lib.WISE_ERR_DEVICE_TIMEOUT
    assert wise.device_status() == _lib.WISE_OK
