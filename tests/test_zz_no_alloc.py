"""The allocation-free selection entry point (wise_select_support_noalloc),
for callers that cannot allocate device memory (a fixed memory plan, a runtime
that owns all device memory, a path that must not call the allocator): through
the C ABI its output
must equal wise_select_support's, on two calls in a row (the shared scratch
array keeps the previous call's contents, which must not leak into the next).
This file is collected last so that a failure here cannot hide other tests."""
import numpy as np
import pytest
import torch

from block_sparse_attention_causal_gb300 import _lib

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def _masses(w, b, h, nb, seed):
    rng = np.random.default_rng(seed)
    m = np.zeros((w, b, h, nb, nb), np.float32)
    for idx in np.ndindex(w, b, h):
        for q in range(nb):
            m[idx][q, :q + 1] = rng.dirichlet(np.full(q + 1, 0.3))
    return torch.from_numpy(m).cuda()


def _select(lib, desc, m, window, eta, noalloc):
    cap = int(lib.wise_support_capacity(desc))
    units = int(lib.wise_schedule_units(desc))
    rows = desc.batch * desc.heads * (desc.seq_len // desc.block)
    rp = torch.full((rows + 1,), -7, dtype=torch.int32, device="cuda")
    ci = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    order = torch.full((units,), -7, dtype=torch.int32, device="cuda")
    nnz = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    if noalloc:
        st = lib.wise_select_support_noalloc(desc, m.data_ptr(), window, eta, 3, rp.data_ptr(), ci.data_ptr(), cap,
                                             order.data_ptr(), nnz.data_ptr(), stream)
    else:
        ws = torch.empty(int(lib.wise_select_workspace(desc, window)), dtype=torch.uint8, device="cuda")
        st = lib.wise_select_support(desc, m.data_ptr(), window, eta, 3, rp.data_ptr(), ci.data_ptr(), cap,
                                     order.data_ptr(), nnz.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    assert st == _lib.WISE_OK
    assert lib.wise_device_status(stream) == _lib.WISE_OK
    n = int(nnz.item())
    return rp.cpu().numpy(), ci[:n].cpu().numpy(), order.cpu().numpy(), n


def test_noalloc_select_matches_workspace_select_twice():
    lib = _lib.load()
    # two different problems back to back: the second must not see the first's scratch
    cases = [((2, 1, 2, 32, 128, 0.9), 1), ((3, 2, 3, 20, 64, 0.8), 2)]
    for (w, b, h, nb, blk, eta), seed in cases:
        desc = _lib.make_desc(b, h, nb * blk, 128, blk)
        m = _masses(w, b, h, nb, seed)
        ref = _select(lib, desc, m, w, eta, noalloc=False)
        got = _select(lib, desc, m, w, eta, noalloc=True)
        for a, r in zip(got[:3], ref[:3]):
            assert np.array_equal(a, r)
        assert got[3] == ref[3]


def test_noalloc_select_rejects_shapes_beyond_its_scratch():
    lib = _lib.load()
    # 8 x 64 x 1024 rows of 32 bitmask words: far beyond 2 MiB of scratch
    desc = _lib.make_desc(8, 64, 1024 * 64, 128, 64)
    assert lib.wise_select_workspace(desc, 1) > (2 << 20)
    st = lib.wise_select_support_noalloc(desc, 16, 1, 0.9, 3, 16, 16, int(lib.wise_support_capacity(desc)), None,
                                         None, torch.cuda.current_stream().cuda_stream)
    assert st == _lib.WISE_ERR_WORKSPACE
