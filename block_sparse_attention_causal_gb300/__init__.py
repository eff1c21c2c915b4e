"""WISE block-sparse causal attention on GB300 (sm_103a).

Python front end of the C-ABI library ``libwise.so``. The three calls follow
"Attention Routing Stabilizes Early: Working-Set Inference for Recurrent
Language Models" (WISE):

* :func:`discover`        -- early recurrent step: unrestricted causal
  attention (§3 Eq 2) plus the block masses r_qb (§5.1 Eq 5);
* :func:`select_support`  -- once after discovery: the cumulative-mass block
  support of §5.1 Eq 6, unioned over the discovery window, as a CSR;
* :func:`sparse`          -- late recurrent step: attention over the reused
  support only (§5.2 Eqs 7-8);
* :func:`discover_select` / :func:`select_finalize` -- the same discovery and
  selection with each window step's Eq 6 support taken in the discovery
  launch itself (no mass tensors kept across the window, no selection pass).

Torch tensors supply device memory and the stream; every computation runs in
the library's CUDA kernels. There is no CPU path: without the compiled
library on a CUDA device these functions raise.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import torch

from . import _lib
from ._lib import (WISE_BF16, WISE_F32, WISE_SUPPORT_DIAG, WISE_SUPPORT_SINK, WiseError)  # noqa: F401

__all__ = ["discover", "select_support", "sparse", "Support", "device_status", "WiseError", "discover_select",
           "select_finalize", "new_select_state",
           "WISE_SUPPORT_SINK", "WISE_SUPPORT_DIAG", "useful_flops", "dense_flops", "retained_mass",
           "support_jaccard", "select_control", "gather_plan"]

_OUT = {torch.bfloat16: WISE_BF16, torch.float32: WISE_F32}


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_device(name: str, t: torch.Tensor) -> None:
    """The library launches on the current CUDA device's stream and error word,
    so every tensor must live on that device."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{torch.cuda.current_device()} "
                         "(select it with torch.cuda.set_device)")


def _check_buffer(name: str, t: torch.Tensor, dtype: torch.dtype, shape: Sequence[int],
                  device: torch.device) -> None:
    """A caller-supplied output or scratch tensor. The C ABI receives bare
    pointers and cannot see sizes, so a wrong dtype, shape or layout here
    would let a kernel write past the allocation: rejected before any launch."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} must have shape {tuple(int(x) for x in shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_bytes(name: str, t: torch.Tensor, nbytes: int, device: torch.device) -> None:
    """A caller-supplied workspace or selection state: uint8, contiguous, on
    `device`, and at least `nbytes` long."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != torch.uint8 or t.dim() != 1 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 1-D uint8 tensor")
    if t.numel() < nbytes:
        raise ValueError(f"{name} holds {t.numel()} bytes, the call needs {nbytes}")


def _check_int32(name: str, t: torch.Tensor, min_numel: int, device: torch.device, exact: bool = False) -> None:
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != torch.int32 or t.dim() != 1 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 1-D int32 tensor")
    if (t.numel() != min_numel) if exact else (t.numel() < min_numel):
        want = f"exactly {min_numel}" if exact else f"at least {min_numel}"
        raise ValueError(f"{name} has {t.numel()} entries, {want} needed")


def _check_support(name: str, sup: "Support", device: torch.device, units: int, capacity: int = 1,
                   need_order: bool = False) -> None:
    """The CSR tensors of a Support: int32, contiguous, on `device`, with
    row_ptr of exactly batch*heads*nb + 1 entries, col_idx of at least
    `capacity`, and (when present or required) a work order of at least
    `units` entries."""
    rows = sup.batch * sup.heads * sup.n_blocks
    _check_int32(f"{name}.row_ptr", sup.row_ptr, rows + 1, device, exact=True)
    _check_int32(f"{name}.col_idx", sup.col_idx, max(capacity, 1), device)
    _check_int32(f"{name}.nnz", sup.nnz, 1, device)
    if sup.tile_order is not None:
        _check_int32(f"{name}.tile_order", sup.tile_order, units, device)
    elif need_order:
        raise ValueError(f"{name}.tile_order is required here")


def _check_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> int:
    """Validates the operands; returns the number of key/value heads (fewer
    than the query heads for grouped-query attention)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_device(name, t)
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
        if not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous [batch, heads, seq, head_dim] tensor")
    b, h, n, d = q.shape
    hk = k.shape[1]
    if k.shape != v.shape or k.shape != (b, hk, n, d) or hk < 1 or h % hk != 0:
        raise ValueError("k and v must be [batch, kv_heads, seq, head_dim] with kv_heads dividing q's heads")
    return hk


def _desc(shape: Sequence[int], block: int, scale: float, out_dtype: torch.dtype, kv_heads: int = 0) -> _lib.AttnDesc:
    b, h, n, d = shape
    if out_dtype not in _OUT:
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")
    return _lib.make_desc(b, h, n, d, block, scale, _OUT[out_dtype], kv_heads)


def discover_workspace_bytes(shape: Sequence[int], block: int) -> int:
    d = _desc(shape, block, 0.0, torch.bfloat16)
    return int(_lib.load().wise_attn_discover_workspace(d))


def discover(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block: int, *, want_mass: bool = True,
             want_lse: bool = True, out_dtype: torch.dtype = torch.bfloat16, scale: float = 0.0,
             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             mass: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None):
    """Discovery step. Returns (O, LSE or None, block masses [B,H,nb,nb] or None).
    k and v may have fewer heads than q (grouped-query attention)."""
    hk = _check_qkv(q, k, v)
    lib = _lib.load()
    b, h, n, d = q.shape
    desc = _desc(q.shape, block, scale, out_dtype, hk)
    dev = q.device
    if out is None:
        out = torch.empty((b, h, n, d), dtype=out_dtype, device=dev)
    _check_buffer("out", out, out_dtype, (b, h, n, d), dev)
    if want_lse and lse is None:
        lse = torch.empty((b, h, n), dtype=torch.float32, device=dev)
    if want_lse:
        _check_buffer("lse", lse, torch.float32, (b, h, n), dev)
    nb = n // block if block > 0 else 0
    ws_bytes = 0
    if want_mass:
        if mass is None:
            mass = torch.empty((b, h, nb, nb), dtype=torch.float32, device=dev)
        _check_buffer("mass", mass, torch.float32, (b, h, nb, nb), dev)
        ws_bytes = int(lib.wise_attn_discover_workspace(desc))
        if workspace is None:
            workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        _check_bytes("workspace", workspace, ws_bytes, dev)
    else:
        mass = None
    st = lib.wise_attn_discover(desc, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), _ptr(lse),
                                _ptr(mass), _ptr(workspace) if want_mass else None,
                                workspace.numel() if (want_mass and workspace is not None) else 0,
                                _stream_handle(stream))
    _lib.check(st, "wise_attn_discover")
    return out, (lse if want_lse else None), mass


def new_select_state(shape: Sequence[int], block: int, window: int, device="cuda") -> torch.Tensor:
    """Device buffer that carries the working set across the discovery steps
    of one selection window (see :func:`discover_select`)."""
    b, h, n, d = shape
    nbytes = int(_lib.load().wise_select_workspace(_lib.make_desc(b, h, n, d, block), window))
    if nbytes <= 0:
        raise ValueError("unsupported shape or window")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def discover_select(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block: int, *, step: int, window: int,
                    eta: float, select_state: torch.Tensor, flags: int = WISE_SUPPORT_SINK | WISE_SUPPORT_DIAG,
                    want_lse: bool = True, out_dtype: torch.dtype = torch.bfloat16, scale: float = 0.0,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    mass: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None):
    """Discovery step `step` (0-based) of a selection window of `window`
    steps, with the step's Eq 6 support OR-ed into `select_state` in the same
    launch (WISE §5.1 Eq 6, streamed over the window). Returns (O, LSE or
    None, this step's block masses). After the last step,
    :func:`select_finalize` gives the Support."""
    hk = _check_qkv(q, k, v)
    lib = _lib.load()
    b, h, n, d = q.shape
    desc = _desc(q.shape, block, scale, out_dtype, hk)
    dev = q.device
    if out is None:
        out = torch.empty((b, h, n, d), dtype=out_dtype, device=dev)
    _check_buffer("out", out, out_dtype, (b, h, n, d), dev)
    if want_lse and lse is None:
        lse = torch.empty((b, h, n), dtype=torch.float32, device=dev)
    if want_lse:
        _check_buffer("lse", lse, torch.float32, (b, h, n), dev)
    nb = n // block
    if mass is None:
        mass = torch.empty((b, h, nb, nb), dtype=torch.float32, device=dev)
    _check_buffer("mass", mass, torch.float32, (b, h, nb, nb), dev)
    ws_bytes = int(lib.wise_attn_discover_workspace(desc))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    _check_bytes("workspace", workspace, ws_bytes, dev)
    _check_bytes("select_state", select_state, int(lib.wise_select_workspace(desc, window)), dev)
    st = lib.wise_attn_discover_select(desc, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), _ptr(lse),
                                       mass.data_ptr(), workspace.data_ptr(), workspace.numel(), float(eta), flags,
                                       step, window, select_state.data_ptr(), select_state.numel(),
                                       _stream_handle(stream))
    _lib.check(st, "wise_attn_discover_select")
    return out, (lse if want_lse else None), mass


@dataclasses.dataclass
class Support:
    """The reused working set: CSR over rows (batch, head, query block)."""
    row_ptr: torch.Tensor      # int32 [B*H*nb + 1]
    col_idx: torch.Tensor      # int32 [capacity]
    tile_order: Optional[torch.Tensor]  # int32 [units]: late-step work order (None: natural order)
    nnz: torch.Tensor          # int32 [1] (device)
    batch: int
    heads: int
    seq_len: int
    head_dim: int
    block: int
    # blocks of 32: the late steps' gathered entries of every tile, built once
    # from the CSR by gather_plan (None: each late step forms them itself)
    plan: Optional[torch.Tensor] = None

    @property
    def n_blocks(self) -> int:
        return self.seq_len // self.block

    def to_lists(self):
        rp = self.row_ptr.cpu().numpy()
        ci = self.col_idx.cpu().numpy()
        return [ci[rp[r]:rp[r + 1]].tolist() for r in range(len(rp) - 1)]


def select_support(masses: torch.Tensor, seq_len: int, head_dim: int, block: int, eta: float,
                   flags: int = WISE_SUPPORT_SINK | WISE_SUPPORT_DIAG, *,
                   support: Optional[Support] = None, workspace: Optional[torch.Tensor] = None,
                   plan: bool = True, stream: Optional[torch.cuda.Stream] = None) -> Support:
    """Working-set selection from the window's masses [W, B, H, nb, nb] (f32).
    With blocks of 32 (and plan), the late steps' gathered entries are built
    too (gather_plan)."""
    if not masses.is_cuda or masses.dtype != torch.float32 or masses.dim() != 5 or not masses.is_contiguous():
        raise ValueError("masses must be a contiguous float32 CUDA tensor [W, B, H, nb, nb]")
    _check_device("masses", masses)
    lib = _lib.load()
    w, b, h, nb, nb2 = masses.shape
    if nb != nb2 or nb * block != seq_len:
        raise ValueError("mass shape does not match seq_len / block")
    desc = _lib.make_desc(b, h, seq_len, head_dim, block)
    cap = int(lib.wise_support_capacity(desc))
    units = int(lib.wise_schedule_units(desc))
    dev = masses.device
    if support is None:
        support = Support(torch.empty(b * h * nb + 1, dtype=torch.int32, device=dev),
                          torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
                          torch.empty(max(units, 1), dtype=torch.int32, device=dev),
                          torch.empty(1, dtype=torch.int32, device=dev), b, h, seq_len, head_dim, block)
    if (support.batch, support.heads, support.seq_len, support.block) != (b, h, seq_len, block):
        raise ValueError("support was built for a different shape")
    _check_support("support", support, dev, units, cap, need_order=True)
    ws_bytes = int(lib.wise_select_workspace(desc, w))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    _check_bytes("workspace", workspace, ws_bytes, dev)
    st = lib.wise_select_support(desc, masses.data_ptr(), w, float(eta), flags, support.row_ptr.data_ptr(),
                                 support.col_idx.data_ptr(), support.col_idx.numel(),
                                 support.tile_order.data_ptr(), support.nnz.data_ptr(), workspace.data_ptr(),
                                 workspace.numel(), _stream_handle(stream))
    _lib.check(st, "wise_select_support")
    if block == 32 and plan:
        gather_plan(support, stream=stream)
    return support


def gather_plan(support: Support, *, stream: Optional[torch.cuda.Stream] = None) -> Support:
    """For blocks of 32: build (or rebuild) support.plan, the late steps'
    gathered entries of every 128-row tile, from the support's CSR. Call it
    again whenever the CSR changes. Other block sizes have no plan."""
    if support.block != 32:
        support.plan = None
        return support
    lib = _lib.load()
    desc = _lib.make_desc(support.batch, support.heads, support.seq_len, support.head_dim, support.block)
    dev = support.row_ptr.device
    _check_support("support", support, dev, int(lib.wise_schedule_units(desc)))
    nbytes = int(lib.wise_gather_plan_bytes(desc))
    if support.plan is None or support.plan.numel() < nbytes or support.plan.device != dev:
        support.plan = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _check_bytes("plan", support.plan, nbytes, dev)
    st = lib.wise_gather_plan(desc, support.row_ptr.data_ptr(), support.col_idx.data_ptr(), support.col_idx.numel(),
                              support.plan.data_ptr(), support.plan.numel(), _stream_handle(stream))
    _lib.check(st, "wise_gather_plan")
    return support


def sparse(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, support: Support, *, want_lse: bool = True,
           out_dtype: torch.dtype = torch.bfloat16, scale: float = 0.0, out: Optional[torch.Tensor] = None,
           lse: Optional[torch.Tensor] = None, use_schedule: bool = True, use_plan: bool = True,
           stream: Optional[torch.cuda.Stream] = None):
    """Late (reuse) step over the support. Returns (O, LSE or None).
    k and v may have fewer heads than q (grouped-query attention). With
    blocks of 32 and a support.plan (use_plan), the tiles' gathered entries
    are read from the plan; the results are the same bits either way."""
    hk = _check_qkv(q, k, v)
    lib = _lib.load()
    b, h, n, d = q.shape
    if (b, h, n, d) != (support.batch, support.heads, support.seq_len, support.head_dim):
        raise ValueError("support was built for a different shape")
    desc = _desc(q.shape, support.block, scale, out_dtype, hk)
    dev = q.device
    _check_support("support", support, dev, int(lib.wise_schedule_units(desc)))
    if out is None:
        out = torch.empty((b, h, n, d), dtype=out_dtype, device=dev)
    _check_buffer("out", out, out_dtype, (b, h, n, d), dev)
    if want_lse and lse is None:
        lse = torch.empty((b, h, n), dtype=torch.float32, device=dev)
    if want_lse:
        _check_buffer("lse", lse, torch.float32, (b, h, n), dev)
    order = support.tile_order.data_ptr() if (use_schedule and support.tile_order is not None) else None
    if use_plan and support.plan is not None and support.block == 32:
        _check_bytes("support.plan", support.plan, int(lib.wise_gather_plan_bytes(desc)), dev)
        st = lib.wise_attn_sparse_planned(desc, q.data_ptr(), k.data_ptr(), v.data_ptr(), support.row_ptr.data_ptr(),
                                          support.col_idx.data_ptr(), support.col_idx.numel(), order,
                                          support.plan.data_ptr(), out.data_ptr(), _ptr(lse) if want_lse else None,
                                          _stream_handle(stream))
        _lib.check(st, "wise_attn_sparse_planned")
    else:
        st = lib.wise_attn_sparse(desc, q.data_ptr(), k.data_ptr(), v.data_ptr(), support.row_ptr.data_ptr(),
                                  support.col_idx.data_ptr(), support.col_idx.numel(), order, out.data_ptr(),
                                  _ptr(lse) if want_lse else None, _stream_handle(stream))
        _lib.check(st, "wise_attn_sparse")
    return out, (lse if want_lse else None)


def select_finalize(select_state: torch.Tensor, batch: int, heads: int, seq_len: int, head_dim: int, block: int,
                    *, support: Optional["Support"] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> "Support":
    """The Support (CSR and work order) accumulated in `select_state` by a
    window of :func:`discover_select` steps."""
    lib = _lib.load()
    desc = _lib.make_desc(batch, heads, seq_len, head_dim, block)
    nb = seq_len // block
    cap = int(lib.wise_support_capacity(desc))
    units = int(lib.wise_schedule_units(desc))
    if cap <= 0:
        raise ValueError("unsupported shape")
    _check_device("select_state", select_state)
    dev = select_state.device
    _check_bytes("select_state", select_state, int(lib.wise_select_workspace(desc, 1)), dev)
    if support is None:
        support = Support(torch.empty(batch * heads * nb + 1, dtype=torch.int32, device=dev),
                          torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
                          torch.empty(max(units, 1), dtype=torch.int32, device=dev),
                          torch.empty(1, dtype=torch.int32, device=dev), batch, heads, seq_len, head_dim, block)
    if (support.batch, support.heads, support.seq_len, support.block) != (batch, heads, seq_len, block):
        raise ValueError("support was built for a different shape")
    _check_support("support", support, dev, units, cap, need_order=True)
    st = lib.wise_select_finalize(desc, select_state.data_ptr(), select_state.numel(), support.row_ptr.data_ptr(),
                                  support.col_idx.data_ptr(), support.col_idx.numel(),
                                  support.tile_order.data_ptr(), support.nnz.data_ptr(), _stream_handle(stream))
    _lib.check(st, "wise_select_finalize")
    if block == 32:
        gather_plan(support, stream=stream)
    return support


def support_from_lists(rows, batch: int, heads: int, seq_len: int, head_dim: int, block: int,
                       device="cuda") -> Support:
    """A Support from explicit ascending key-block lists (rows ordered batch,
    head, query block). It has no work order: late steps over it use the
    kernel's natural order."""
    rp = [0]
    cols = []
    for r in rows:
        cols.extend(int(x) for x in r)
        rp.append(len(cols))
    return Support(torch.tensor(rp, dtype=torch.int32, device=device),
                   torch.tensor(cols if cols else [0], dtype=torch.int32, device=device),
                   None,
                   torch.tensor([len(cols)], dtype=torch.int32, device=device),
                   batch, heads, seq_len, head_dim, block)


def select_control(masses: torch.Tensor, reference: Support, mode: str, flags: int = 0, *,
                   stream: Optional[torch.cuda.Stream] = None) -> Support:
    """Early-static controls of WISE App. B from one step's masses [B, H, nb, nb]
    (f32) and a reference working set: mode "mass" = MassMatched (Eqs 20-21),
    "size" = SizeMatched (Eq 22). Static-95 (Eq 19) is select_support with a
    window of one step and eta = 0.95."""
    modes = {"mass": _lib.WISE_CONTROL_MASS_MATCHED, "size": _lib.WISE_CONTROL_SIZE_MATCHED}
    if mode not in modes:
        raise ValueError('mode must be "mass" or "size"')
    if not masses.is_cuda or masses.dtype != torch.float32 or masses.dim() != 4 or not masses.is_contiguous():
        raise ValueError("masses must be a contiguous float32 CUDA tensor [B, H, nb, nb]")
    _check_device("masses", masses)
    b, h, nb, _ = masses.shape
    if (b, h, nb) != (reference.batch, reference.heads, reference.n_blocks):
        raise ValueError("masses do not match the reference support's shape")
    lib = _lib.load()
    desc = _lib.make_desc(reference.batch, reference.heads, reference.seq_len, reference.head_dim, reference.block)
    cap = int(lib.wise_support_capacity(desc))
    units = int(lib.wise_schedule_units(desc))
    dev = masses.device
    _check_support("reference", reference, dev, units)
    out = Support(torch.empty(b * h * nb + 1, dtype=torch.int32, device=dev),
                  torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
                  torch.empty(max(units, 1), dtype=torch.int32, device=dev),
                  torch.empty(1, dtype=torch.int32, device=dev), reference.batch, reference.heads,
                  reference.seq_len, reference.head_dim, reference.block)
    ws = torch.empty(max(int(lib.wise_select_workspace(desc, 1)), 16), dtype=torch.uint8, device=dev)
    st = lib.wise_select_control(desc, masses.data_ptr(), modes[mode], reference.row_ptr.data_ptr(),
                                 reference.col_idx.data_ptr(), reference.col_idx.numel(), flags,
                                 out.row_ptr.data_ptr(), out.col_idx.data_ptr(), out.col_idx.numel(),
                                 out.tile_order.data_ptr(), out.nnz.data_ptr(), ws.data_ptr(), ws.numel(),
                                 _stream_handle(stream))
    _lib.check(st, "wise_select_control")
    return out


def retained_mass(masses: torch.Tensor, support: Support, *, stream: Optional[torch.cuda.Stream] = None):
    """Retained future attention mass (WISE App. B metrics) of a support for a
    later step's block masses [B, H, nb, nb] (f32, from :func:`discover`).
    Returns (per-row fractions [B*H*nb] f32, per-batch mean [B] f64)."""
    if not masses.is_cuda or masses.dtype != torch.float32 or masses.dim() != 4 or not masses.is_contiguous():
        raise ValueError("masses must be a contiguous float32 CUDA tensor [B, H, nb, nb]")
    _check_device("masses", masses)
    b, h, nb, _ = masses.shape
    if (b, h, nb) != (support.batch, support.heads, support.n_blocks):
        raise ValueError("masses do not match the support's shape")
    lib = _lib.load()
    desc = _lib.make_desc(support.batch, support.heads, support.seq_len, support.head_dim, support.block)
    _check_support("support", support, masses.device, int(lib.wise_schedule_units(desc)))
    rows = torch.empty(b * h * nb, dtype=torch.float32, device=masses.device)
    mean = torch.empty(b, dtype=torch.float64, device=masses.device)
    st = lib.wise_support_retained_mass(desc, masses.data_ptr(), support.row_ptr.data_ptr(),
                                        support.col_idx.data_ptr(), support.col_idx.numel(), rows.data_ptr(),
                                        mean.data_ptr(), _stream_handle(stream))
    _lib.check(st, "wise_support_retained_mass")
    return rows, mean


def support_jaccard(a: Support, b: Support, *, stream: Optional[torch.cuda.Stream] = None):
    """Rolling working-set stability (WISE App. C.2 Eq 24) between two
    supports of the same shape. Returns (per-row counts [B*H*nb, 2] int32 of
    |A and B|, |A or B|; per-batch summed counts [B, 2] int64; per-batch
    Jaccard index [B] f64)."""
    shape = (a.batch, a.heads, a.seq_len, a.head_dim, a.block)
    if shape != (b.batch, b.heads, b.seq_len, b.head_dim, b.block):
        raise ValueError("supports of different shapes")
    lib = _lib.load()
    desc = _lib.make_desc(*shape)
    rows = a.batch * a.heads * a.n_blocks
    _check_device("a.row_ptr", a.row_ptr)
    dev = a.row_ptr.device
    units = int(lib.wise_schedule_units(desc))
    _check_support("a", a, dev, units)
    _check_support("b", b, dev, units)
    row_counts = torch.empty((rows, 2), dtype=torch.int32, device=dev)
    counts = torch.empty((a.batch, 2), dtype=torch.int64, device=dev)
    jac = torch.empty(a.batch, dtype=torch.float64, device=dev)
    st = lib.wise_support_jaccard(desc, a.row_ptr.data_ptr(), a.col_idx.data_ptr(), a.col_idx.numel(),
                                  b.row_ptr.data_ptr(), b.col_idx.data_ptr(), b.col_idx.numel(),
                                  row_counts.data_ptr(), counts.data_ptr(), jac.data_ptr(), _stream_handle(stream))
    _lib.check(st, "wise_support_jaccard")
    return row_counts, counts, jac


def device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise and read/clear the library's device error word."""
    return int(_lib.load().wise_device_status(_stream_handle(stream)))


def check_device(stream: Optional[torch.cuda.Stream] = None) -> None:
    _lib.check(device_status(stream), "device")


# ---------------------------------------------------------------- FLOP counts

def dense_flops(batch: int, heads: int, seq_len: int, head_dim: int) -> float:
    """Useful FLOPs of causal attention: 4 d per admissible (i, j) pair."""
    return 4.0 * head_dim * batch * heads * seq_len * (seq_len + 1) / 2


def useful_flops(rows_per_bh_counts, block: int, head_dim: int) -> float:
    """Useful FLOPs over a block support: 4 d per admissible pair inside the
    listed blocks (B^2 off the diagonal, B(B+1)/2 on it). `rows_per_bh_counts`
    is a pair (n_offdiag_blocks, n_diag_blocks)."""
    off, diag = rows_per_bh_counts
    return 4.0 * head_dim * (off * block * block + diag * block * (block + 1) / 2)
