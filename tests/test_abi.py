"""The C-ABI library loads, exports every symbol the header declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

from block_sparse_attention_causal_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "wise.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wise_[a-z_]+)\s*\(", text)))


def test_header_declares_exactly_the_binding_exports():
    assert _declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    version = int(re.search(r"#define WISE_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert lib.wise_abi_version() == version


def test_grouped_query_heads_are_validated(lib):
    """kv_heads must be 0 (= heads) or divide heads; the argument check
    runs before any launch, so no device is needed."""
    dummy = ctypes.c_void_p(16)
    for kv, ok in ((0, True), (1, True), (2, True), (4, True), (3, False), (-1, False), (8, False)):
        d = _lib.make_desc(1, 4, 256, 64, 64, 0.0, 0, kv)
        assert (lib.wise_attn_discover_workspace(d) > 0) == ok, kv
        if not ok:
            st = lib.wise_attn_discover(d, dummy, dummy, dummy, dummy, None, None, None, 0, None)
            assert st == _lib.WISE_ERR_INVALID_ARGUMENT


def test_status_strings(lib):
    for s in range(8):
        assert lib.wise_status_str(s).decode()
    assert lib.wise_status_str(99).decode() == "unknown status"


def _desc(b=1, h=2, n=256, d=64, blk=64, scale=0.0, out=0):
    return _lib.make_desc(b, h, n, d, blk, scale, out)


def test_workspace_and_capacity_queries(lib):
    d = _desc(1, 2, 256, 64, 64)
    nb = 4
    assert lib.wise_support_capacity(d) == 2 * nb * (nb + 1) // 2
    # one 128-row query tile per unit; n = 256 -> two units per (batch, head)
    assert lib.wise_schedule_units(d) == 4
    # lambda scratch: (128/B) * T(T+1)/2 entries of 128 floats (one per row)
    # per (b,h), T = 2 query tiles
    assert lib.wise_attn_discover_workspace(d) == 2 * (2 * 3) * 128 * 4
    assert lib.wise_select_workspace(d, 2) > 0
    assert lib.wise_select_workspace(d, 0) == 0
    assert lib.wise_schedule_units(_desc(1, 1, 128 * 5, 128, 128)) == 5


@pytest.mark.parametrize("bad", [
    dict(b=0), dict(h=0), dict(n=0), dict(n=100), dict(blk=0), dict(scale=-1.0), dict(out=7),
])
def test_invalid_descriptor_rejected(lib, bad):
    d = _desc(**bad)
    assert lib.wise_support_capacity(d) == 0
    st = lib.wise_attn_discover(d, 16, 16, 16, 16, None, None, None, 0, None)
    assert st == _lib.WISE_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("bad", [dict(d=80), dict(d=256), dict(blk=16), dict(blk=256), dict(n=64 * 2048),
                                 dict(blk=32, n=32 * 1056)])
def test_unsupported_shapes_rejected(lib, bad):
    d = _desc(**bad)
    assert lib.wise_attn_discover(d, 16, 16, 16, 16, None, None, None, 0, None) == _lib.WISE_ERR_UNSUPPORTED


def test_block_32_queries(lib):
    # blocks of 32 (the pages' default granularity): four query blocks per
    # 128-row tile; the Eq 5 scratch holds four values per row and 128-key span
    n = 640
    d = _desc(2, 3, n, 64, 32)
    nb, tiles = n // 32, (n + 127) // 128
    assert lib.wise_support_capacity(d) == 2 * 3 * nb * (nb + 1) // 2
    assert lib.wise_schedule_units(d) == 2 * 3 * tiles
    assert lib.wise_attn_discover_workspace(d) == 2 * 3 * 4 * tiles * (tiles + 1) // 2 * 128 * 4
    assert lib.wise_select_workspace(d, 3) > 0


def test_fused_selection_argument_checks(lib):
    d = _desc()  # 1 x 2 heads, n 256, d 64, block 64
    ws = lib.wise_attn_discover_workspace(d)
    st_bytes = lib.wise_select_workspace(d, 2)

    def call(desc=d, q=16, mass=16, ws_=16, wsb=ws, eta=0.9, flags=3, step=0, window=2, state=16, sb=st_bytes):
        return lib.wise_attn_discover_select(desc, q, 16, 16, 16, None, mass, ws_, wsb, eta, flags, step, window,
                                             state, sb, None)
    E = _lib
    assert call(q=None) == E.WISE_ERR_INVALID_ARGUMENT
    assert call(mass=None) == E.WISE_ERR_INVALID_ARGUMENT
    assert call(state=None) == E.WISE_ERR_INVALID_ARGUMENT
    assert call(step=2) == E.WISE_ERR_INVALID_ARGUMENT
    assert call(step=-1) == E.WISE_ERR_INVALID_ARGUMENT
    assert call(window=9, step=0) == E.WISE_ERR_INVALID_ARGUMENT
    assert call(eta=1.0) == E.WISE_ERR_INVALID_ARGUMENT
    assert call(flags=4) == E.WISE_ERR_INVALID_ARGUMENT
    assert call(state=8) == E.WISE_ERR_ALIGNMENT
    assert call(wsb=ws - 1) == E.WISE_ERR_WORKSPACE
    assert call(sb=st_bytes - 1) == E.WISE_ERR_WORKSPACE
    # the epilogue holds a row of up to 256 blocks
    big = _desc(1, 1, 64 * 512, 64, 64)
    assert call(desc=big, wsb=lib.wise_attn_discover_workspace(big),
                sb=lib.wise_select_workspace(big, 2)) == E.WISE_ERR_UNSUPPORTED
    cap = lib.wise_support_capacity(d)
    fin = lambda **kw: lib.wise_select_finalize(d, kw.get("state", 16), kw.get("sb", st_bytes), kw.get("rp", 16), 16,
                                                kw.get("cap", cap), None, None, None)
    assert fin(state=None) == E.WISE_ERR_INVALID_ARGUMENT
    assert fin(rp=None) == E.WISE_ERR_INVALID_ARGUMENT
    assert fin(cap=cap - 1) == E.WISE_ERR_BAD_SUPPORT
    assert fin(sb=16) == E.WISE_ERR_WORKSPACE
    assert fin(state=8) == E.WISE_ERR_ALIGNMENT


def test_null_and_misaligned_pointers_rejected(lib):
    d = _desc()
    assert lib.wise_attn_discover(d, None, 16, 16, 16, None, None, None, 0, None) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert lib.wise_attn_discover(d, 8, 16, 16, 16, None, None, None, 0, None) == _lib.WISE_ERR_ALIGNMENT
    # block masses requested without workspace
    assert lib.wise_attn_discover(d, 16, 16, 16, 16, None, 16, None, 0, None) == _lib.WISE_ERR_WORKSPACE
    assert lib.wise_attn_sparse(d, 16, 16, 16, None, 16, 10, None, 16, None, None) == _lib.WISE_ERR_INVALID_ARGUMENT


def test_gather_plan_argument_checks(lib):
    """The plan of gathered entries exists for blocks of 32 only: its size
    (an int32 count per 128-row tile, 16-byte aligned, then 16 bytes per
    entry, tile t of each slice owning room for t + 1) and the argument
    checks of building and using it (no device work)."""
    d64 = _desc()
    d32 = _lib.make_desc(2, 3, 1024, 64, 32)
    assert lib.wise_gather_plan_bytes(d64) == 0
    tiles, units = 8, 2 * 3 * 8
    assert lib.wise_gather_plan_bytes(d32) == (units * 4 + 15) // 16 * 16 + 2 * 3 * (tiles * (tiles + 1) // 2) * 16
    nbytes = lib.wise_gather_plan_bytes(d32)
    assert lib.wise_gather_plan(d64, 16, 16, 10, 16, 1 << 20, None) == _lib.WISE_ERR_UNSUPPORTED
    assert lib.wise_gather_plan(d32, None, 16, 10, 16, nbytes, None) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert lib.wise_gather_plan(d32, 16, 16, 10, None, nbytes, None) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert lib.wise_gather_plan(d32, 16, 16, 10, 16, nbytes - 1, None) == _lib.WISE_ERR_WORKSPACE
    assert lib.wise_gather_plan(d32, 16, 16, 10, 8, nbytes, None) == _lib.WISE_ERR_ALIGNMENT
    # a plan with another block size, and the usual checks of the sparse step
    assert lib.wise_attn_sparse_planned(d64, 16, 16, 16, 16, 16, 10, None, 16, 16, None, None) == \
        _lib.WISE_ERR_INVALID_ARGUMENT
    assert lib.wise_attn_sparse_planned(d32, 16, 16, 16, None, 16, 10, None, 16, 16, None, None) == \
        _lib.WISE_ERR_INVALID_ARGUMENT
    assert lib.wise_attn_sparse_planned(d32, 16, 16, 16, 16, 16, 10, None, 8, 16, None, None) == \
        _lib.WISE_ERR_ALIGNMENT


def test_select_argument_checks(lib):
    d = _desc()
    cap = lib.wise_support_capacity(d)
    ws = lib.wise_select_workspace(d, 2)
    args = lambda **kw: dict(dict(mass=16, window=2, eta=0.9, flags=3, cap=cap, ws=16, wsb=ws), **kw)

    def call(a):
        return lib.wise_select_support(d, a["mass"], a["window"], a["eta"], a["flags"], 16, 16, a["cap"], None,
                                       None, a["ws"], a["wsb"], None)
    assert call(args(eta=0.0)) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert call(args(eta=1.0)) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert call(args(window=0)) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert call(args(window=9)) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert call(args(flags=4)) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert call(args(mass=None)) == _lib.WISE_ERR_INVALID_ARGUMENT
    assert call(args(cap=cap - 1)) == _lib.WISE_ERR_BAD_SUPPORT
    assert call(args(wsb=ws - 1)) == _lib.WISE_ERR_WORKSPACE


def _host(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data


def test_host_support_validator(lib):
    d = _desc(1, 1, 256, 64, 64)  # nb = 4
    good_rows = [[0], [0, 1], [0, 2], [0, 1, 3]]
    rp = np.cumsum([0] + [len(r) for r in good_rows]).astype(np.int32)
    ci = np.array(sum(good_rows, []), np.int32)
    assert lib.wise_validate_support(d, rp.ctypes.data, ci.ctypes.data, 3) == _lib.WISE_OK
    for bad_rows in ([[0], [1, 0], [0, 2], [0, 3]],      # not ascending
                     [[0], [0, 1], [0, 3], [0, 1, 3]],   # block above the diagonal
                     [[0], [0, 1], [0, 2], [0, 1]]):     # missing diagonal with DIAG
        rp2 = np.cumsum([0] + [len(r) for r in bad_rows]).astype(np.int32)
        ci2 = np.array(sum(bad_rows, []), np.int32)
        assert lib.wise_validate_support(d, rp2.ctypes.data, ci2.ctypes.data, 3) == _lib.WISE_ERR_BAD_SUPPORT
    rows_nodiag = [[0], [0], [0], [0, 1]]
    rp3 = np.cumsum([0] + [len(r) for r in rows_nodiag]).astype(np.int32)
    ci3 = np.array(sum(rows_nodiag, []), np.int32)
    assert lib.wise_validate_support(d, rp3.ctypes.data, ci3.ctypes.data, 1) == _lib.WISE_OK
    assert lib.wise_validate_support(d, rp3.ctypes.data, ci3.ctypes.data, 3) == _lib.WISE_ERR_BAD_SUPPORT
