"""The binding rejects caller-supplied buffers that the kernels could overrun.

The C ABI takes bare pointers, so the Python layer checks every output,
scratch and support tensor (device, dtype, shape, layout, size) before any
launch. These checks run on the host; the first group needs no GPU, the
second drives the public calls on a GPU with wrong tensors and expects the
raise before anything is launched.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_causal_gb300 as wise
from block_sparse_attention_causal_gb300 import _lib

CPU = torch.device("cpu")


def test_buffer_check_accepts_the_exact_tensor():
    wise._check_buffer("out", torch.empty((1, 2, 256, 64), dtype=torch.float32), torch.float32, (1, 2, 256, 64), CPU)


@pytest.mark.parametrize("bad", [
    torch.empty((1, 2, 256, 64), dtype=torch.bfloat16),        # dtype
    torch.empty((1, 2, 255, 64), dtype=torch.float32),         # shape
    torch.empty((1, 2, 64, 256), dtype=torch.float32),         # transposed shape
    torch.empty((1, 2, 64, 256), dtype=torch.float32).transpose(2, 3),  # right shape, not contiguous
])
def test_buffer_check_rejects(bad):
    with pytest.raises(ValueError):
        wise._check_buffer("out", bad, torch.float32, (1, 2, 256, 64), CPU)


def test_buffer_check_accepts_a_contiguous_view():
    wise._check_buffer("out", torch.empty((2, 2, 256, 64), dtype=torch.float32)[:1], torch.float32,
                       (1, 2, 256, 64), CPU)


def test_buffer_check_rejects_other_device():
    meta = torch.empty((4,), dtype=torch.float32, device="meta")
    with pytest.raises(ValueError, match="expected"):
        wise._check_buffer("lse", meta, torch.float32, (4,), CPU)


def test_workspace_check():
    wise._check_bytes("workspace", torch.empty(100, dtype=torch.uint8), 100, CPU)
    with pytest.raises(ValueError, match="needs 101"):
        wise._check_bytes("workspace", torch.empty(100, dtype=torch.uint8), 101, CPU)
    with pytest.raises(ValueError, match="uint8"):
        wise._check_bytes("workspace", torch.empty(100, dtype=torch.int8), 10, CPU)
    with pytest.raises(ValueError, match="uint8"):
        wise._check_bytes("workspace", torch.empty((10, 10), dtype=torch.uint8), 10, CPU)


def _support(rows_plus_one=9, cols=20, order=2, nnz=1, dtype=torch.int32):
    # batch 1, heads 2, n 256, block 64 -> nb 4, 8 CSR rows, 4 work units
    mk = lambda n: None if n is None else torch.zeros(n, dtype=dtype)
    return wise.Support(mk(rows_plus_one), mk(cols), mk(order), mk(nnz), 1, 2, 256, 64, 64)


def test_support_check():
    wise._check_support("s", _support(order=4), CPU, units=4, capacity=20, need_order=True)
    wise._check_support("s", _support(order=None), CPU, units=4)
    with pytest.raises(ValueError, match="row_ptr"):
        wise._check_support("s", _support(rows_plus_one=8), CPU, units=4)
    with pytest.raises(ValueError, match="row_ptr"):
        wise._check_support("s", _support(rows_plus_one=10), CPU, units=4)
    with pytest.raises(ValueError, match="col_idx"):
        wise._check_support("s", _support(cols=19), CPU, units=4, capacity=20)
    with pytest.raises(ValueError, match="tile_order"):
        wise._check_support("s", _support(order=3), CPU, units=4)
    with pytest.raises(ValueError, match="tile_order"):
        wise._check_support("s", _support(order=None), CPU, units=4, need_order=True)
    with pytest.raises(ValueError, match="nnz"):
        wise._check_support("s", _support(nnz=0), CPU, units=4)
    with pytest.raises(ValueError, match="int32"):
        wise._check_support("s", _support(dtype=torch.int64), CPU, units=2)


def test_schedule_validator(lib):
    d = _lib.make_desc(1, 2, 384, 64, 128)  # 3 query tiles per head -> 6 units
    assert lib.wise_schedule_units(d) == 6
    good = np.array([5, 0, 3, 1, 4, 2], np.int32)
    assert lib.wise_validate_schedule(d, good.ctypes.data) == _lib.WISE_OK
    for bad in ([5, 0, 3, 1, 4, 4],    # duplicate (and 2 missing)
                [5, 0, 3, 1, 4, 6],    # out of range
                [5, 0, 3, 1, 4, -1]):  # negative
        arr = np.array(bad, np.int32)
        assert lib.wise_validate_schedule(d, arr.ctypes.data) == _lib.WISE_ERR_BAD_SUPPORT, bad
    assert lib.wise_validate_schedule(d, None) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert lib.wise_validate_schedule(_lib.make_desc(0, 2, 384, 64, 128), good.ctypes.data) == \
        _lib.WISE_ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------- on a GPU

def _qkv(b=1, h=2, n=256, d=64, seed=0):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((b, h, n, d), generator=g).to(torch.bfloat16).cuda() for _ in range(3)]


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")
def test_public_calls_reject_wrong_buffers():
    q, k, v = _qkv()
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    with pytest.raises(ValueError, match="out"):
        wise.discover(q, k, v, 64, out=torch.empty((1, 2, 256, 64), dtype=torch.bfloat16, device=dev),
                      out_dtype=torch.float32)
    with pytest.raises(ValueError, match="mass"):
        wise.discover(q, k, v, 64, mass=torch.empty((1, 2, 3, 3), **f32))
    with pytest.raises(ValueError, match="lse"):
        wise.discover(q, k, v, 64, lse=torch.empty((1, 2, 255), **f32))
    with pytest.raises(ValueError, match="workspace"):
        wise.discover(q, k, v, 64, workspace=torch.empty(16, dtype=torch.uint8, device=dev))
    with pytest.raises(ValueError, match="out"):
        wise.discover(q, k, v, 64, out=torch.empty((1, 2, 256, 64), dtype=torch.bfloat16, device="cpu"))
    _, _, m = wise.discover(q, k, v, 64)
    sup = wise.select_support(m[None].contiguous(), 256, 64, 64, 0.9)
    with pytest.raises(ValueError, match="out"):
        wise.sparse(q, k, v, sup, out=torch.empty((1, 2, 256, 32), dtype=torch.bfloat16, device=dev))
    short = wise.Support(sup.row_ptr[:-1], sup.col_idx, sup.tile_order, sup.nnz, 1, 2, 256, 64, 64)
    with pytest.raises(ValueError, match="row_ptr"):
        wise.sparse(q, k, v, short)
    host = wise.Support(sup.row_ptr.cpu(), sup.col_idx, sup.tile_order, sup.nnz, 1, 2, 256, 64, 64)
    with pytest.raises(ValueError, match="row_ptr"):
        wise.sparse(q, k, v, host)
    wide = wise.Support(sup.row_ptr.long(), sup.col_idx, sup.tile_order, sup.nnz, 1, 2, 256, 64, 64)
    with pytest.raises(ValueError, match="int32"):
        wise.sparse(q, k, v, wide)
    with pytest.raises(ValueError, match="tile_order"):
        wise.sparse(q, k, v, wise.Support(sup.row_ptr, sup.col_idx, sup.tile_order[:1], sup.nnz, 1, 2, 256, 64, 64))
    with pytest.raises(ValueError, match="col_idx"):
        wise.select_support(m[None].contiguous(), 256, 64, 64, 0.9,
                            support=wise.Support(sup.row_ptr, sup.col_idx[:3], sup.tile_order, sup.nnz,
                                                 1, 2, 256, 64, 64))
    state = wise.new_select_state((1, 2, 256, 64), 64, 2)
    with pytest.raises(ValueError, match="select_state"):
        wise.discover_select(q, k, v, 64, step=0, window=2, eta=0.9, select_state=state[:8])
    with pytest.raises(ValueError, match="select_state"):
        wise.select_finalize(state.cpu(), 1, 2, 256, 64, 64)
    with pytest.raises(ValueError, match="select_state"):
        wise.select_finalize(state[:4], 1, 2, 256, 64, 64)
    wise.check_device()  # nothing was launched by the rejected calls
