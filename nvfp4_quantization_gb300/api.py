"""Python binding of libepq.so: argument marshalling only.

Each function takes torch CUDA tensors, allocates outputs the caller did not
pass (torch is the allocator; the library never allocates), and calls the C
entry point of the same name on the current torch stream.  Every step of the
path runs in the library's kernels.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import EP_ROUND_RNE, EP_ROUND_SR, EpGrouped, check

DEFAULT_ALIGNMENT = 128
DEFAULT_SIGN_MASK = 0xA53C


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def row_bytes(H: int) -> int:
    return int(_lib.lib().ep_nvfp4_row_bytes(int(H)))


def rows_capacity(T: int, k: int, E: int, A: int = DEFAULT_ALIGNMENT) -> int:
    return int(_lib.lib().ep_rows_capacity(int(T), int(k), int(E), int(A)))


@dataclass
class RoutePlan:
    """Device-resident routing plan (all int32 CUDA tensors)."""
    offsets: torch.Tensor     # [E+1]
    counts: torch.Tensor      # [E]
    dest: torch.Tensor        # [T*k]
    T: int
    k: int
    E: int
    A: int
    R_cap: int
    status: torch.Tensor      # uint32-valued int32 [1], EP_DEV_ERR_* bits


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def new_route_workspace(T: int, k: int, E: int, device) -> torch.Tensor:
    """A zero-filled workspace for ep_route_plan (reusable across calls)."""
    nbytes = int(_lib.lib().ep_route_workspace_bytes(int(T), int(k), int(E)))
    return torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device=device)


def ep_route_plan(topk_idx: torch.Tensor, E: int, A: int = DEFAULT_ALIGNMENT, R_cap: int | None = None,
                  plan: RoutePlan | None = None, workspace: torch.Tensor | None = None,
                  status: torch.Tensor | None = None, stream=None) -> RoutePlan:
    """Place every (token, slot) of ``topk_idx`` [T, k] (int32, -1 = dropped)
    in expert-contiguous, A-aligned row order."""
    _need_cuda(topk_idx, "topk_idx", torch.int32)
    T, k = topk_idx.shape
    dev = topk_idx.device
    if R_cap is None:
        R_cap = rows_capacity(T, k, E, A)
    if plan is None:
        plan = RoutePlan(torch.empty(E + 1, dtype=torch.int32, device=dev),
                         torch.empty(E, dtype=torch.int32, device=dev),
                         torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
                         T, k, E, A, R_cap, status if status is not None else new_status(dev))
    if workspace is None:
        workspace = new_route_workspace(T, k, E, dev)
    st = _lib.lib().ep_route_plan(_ptr(topk_idx), T, k, E, A, R_cap, _ptr(plan.offsets), _ptr(plan.counts),
                                  _ptr(plan.dest), _ptr(workspace), workspace.numel() * 4, _ptr(plan.status),
                                  _stream(stream))
    check("ep_route_plan", st)
    return plan


def ep_route_plan_noalloc(topk_idx: torch.Tensor, plan: RoutePlan, stream=None) -> RoutePlan:
    """ep_route_plan into a caller-allocated ``plan``, with no workspace: the
    C entry point uses a fixed scratch array inside the library and allocates
    nothing (for hosts that own all device memory themselves).  Calls whose
    work may overlap on one GPU share that scratch and race."""
    _need_cuda(topk_idx, "topk_idx", torch.int32)
    T, k = topk_idx.shape
    st = _lib.lib().ep_route_plan_noalloc(_ptr(topk_idx), T, k, plan.E, plan.A, plan.R_cap, _ptr(plan.offsets),
                                          _ptr(plan.counts), _ptr(plan.dest), _ptr(plan.status), _stream(stream))
    check("ep_route_plan_noalloc", st)
    return plan


def _need_amax(expert_amax, E: int):
    if expert_amax is not None:
        _need_cuda(expert_amax, "expert_amax", torch.float32)
        if expert_amax.numel() < E:
            raise ValueError("expert_amax needs E entries")


def ep_nvfp4_pack(tokens: torch.Tensor, plan: RoutePlan, rows: torch.Tensor | None = None,
                  rounding: int = EP_ROUND_RNE, seed: int = 0, expert_amax: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """BF16 tokens [T, H] -> packed NVFP4 rows [R_cap, row_bytes(H)] (uint8).
    ``expert_amax`` (f32 [E], filled by the caller, e.g. with zeros) receives
    the max of the token amaxes of each expert's rows."""
    _need_cuda(tokens, "tokens", torch.bfloat16)
    _need_amax(expert_amax, plan.E)
    T, H = tokens.shape
    S = row_bytes(H)
    if rows is None:
        rows = torch.empty((plan.R_cap, S), dtype=torch.uint8, device=tokens.device)
    _need_cuda(rows, "rows", torch.uint8)
    st = _lib.lib().ep_nvfp4_pack(_ptr(tokens), T, H, _ptr(plan.dest), plan.k, _ptr(plan.offsets),
                                  _ptr(plan.counts), plan.E, _ptr(rows), rows.shape[0], _ptr(expert_amax),
                                  int(rounding), int(seed) & ((1 << 64) - 1), _ptr(plan.status), _stream(stream))
    check("ep_nvfp4_pack", st)
    return rows


def ep_nvfp4_dispatch(tokens: torch.Tensor, topk_idx: torch.Tensor, E: int, A: int = DEFAULT_ALIGNMENT,
                      R_cap: int | None = None, plan: RoutePlan | None = None,
                      workspace: torch.Tensor | None = None, rows: torch.Tensor | None = None,
                      rounding: int = EP_ROUND_RNE, seed: int = 0, status: torch.Tensor | None = None,
                      expert_amax: torch.Tensor | None = None, stream=None) -> tuple[RoutePlan, torch.Tensor]:
    """ep_route_plan then ep_nvfp4_pack in one C call (the pack overlaps the
    routing kernel); returns (plan, rows).  ``expert_amax`` (f32 [E]) is
    zeroed and then receives each expert's amax, for ep_nvfp4_direct_receive."""
    _need_cuda(tokens, "tokens", torch.bfloat16)
    _need_amax(expert_amax, E)
    _need_cuda(topk_idx, "topk_idx", torch.int32)
    T, k = topk_idx.shape
    if tokens.shape[0] != T:
        raise ValueError("tokens and topk_idx disagree on T")
    H = tokens.shape[1]
    dev = topk_idx.device
    if R_cap is None:
        R_cap = plan.R_cap if plan is not None else rows_capacity(T, k, E, A)
    if plan is None:
        plan = RoutePlan(torch.empty(E + 1, dtype=torch.int32, device=dev),
                         torch.empty(E, dtype=torch.int32, device=dev),
                         torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
                         T, k, E, A, R_cap, status if status is not None else new_status(dev))
    if workspace is None:
        workspace = new_route_workspace(T, k, E, dev)
    if rows is None:
        rows = torch.empty((R_cap, row_bytes(H)), dtype=torch.uint8, device=dev)
    _need_cuda(rows, "rows", torch.uint8)
    if rows.shape[0] < R_cap:
        raise ValueError("rows has fewer than R_cap rows")
    st = _lib.lib().ep_nvfp4_dispatch(_ptr(topk_idx), _ptr(tokens), T, H, k, E, A, R_cap, _ptr(plan.offsets),
                                      _ptr(plan.counts), _ptr(plan.dest), _ptr(workspace), workspace.numel() * 4,
                                      _ptr(rows), _ptr(expert_amax), int(rounding), int(seed) & ((1 << 64) - 1),
                                      _ptr(plan.status), _stream(stream))
    check("ep_nvfp4_dispatch", st)
    return plan, rows


def ep_nvfp4_unpack(rows: torch.Tensor, H: int, offsets: torch.Tensor, E: int,
                    out: torch.Tensor | None = None, status: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Packed rows -> BF16 [R_cap, H]; rows [0, offsets[E]) are written."""
    _need_cuda(rows, "rows", torch.uint8)
    R_cap = rows.shape[0]
    if out is None:
        out = torch.empty((R_cap, H), dtype=torch.bfloat16, device=rows.device)
    if status is None:
        status = new_status(rows.device)
    st = _lib.lib().ep_nvfp4_unpack(_ptr(rows), R_cap, H, _ptr(offsets), E, _ptr(out), _ptr(status),
                                    _stream(stream))
    check("ep_nvfp4_unpack", st)
    return out


def alloc_grouped(R_cap: int, H: int, E: int, device, rowwise: bool = True) -> dict:
    """Output tensors of the direct receive.  amax_row, amax_col and
    cw_scale_enc are the three rows of one [3, E] tensor, ``metadata``, so a
    single copy moves all three."""
    u8, f32 = torch.uint8, torch.float32
    meta = torch.empty((3, E), dtype=f32, device=device)
    g = dict(cw_codes=torch.empty(R_cap * H // 2, dtype=u8, device=device),
             cw_scales=torch.empty(R_cap * H // 16, dtype=u8, device=device),
             amax_row=meta[0], amax_col=meta[1], cw_scale_enc=meta[2], metadata=meta)
    if rowwise:
        g.update(rw_codes=torch.empty((R_cap, H // 2), dtype=u8, device=device),
                 rw_scales=torch.empty((R_cap, H // 16), dtype=u8, device=device),
                 rw_row_scale=torch.empty(R_cap, dtype=f32, device=device))
    return g


def grouped_struct(g: dict) -> EpGrouped:
    return EpGrouped(*[ctypes.c_void_p(g[n].data_ptr()) if g.get(n) is not None else None
                       for n, _ in EpGrouped._fields_])


def ep_nvfp4_direct_receive(rows: torch.Tensor, H: int, offsets: torch.Tensor, E: int,
                            out: dict | None = None, rounding: int = EP_ROUND_RNE, seed: int = 0,
                            sign_mask: int = DEFAULT_SIGN_MASK, status: torch.Tensor | None = None,
                            rowwise: bool = True, swizzled: bool = False, expert_amax: torch.Tensor | None = None,
                            stream=None) -> dict:
    """Packed rows -> grouped rowwise + columnwise-RHT NVFP4 operands (dict of
    tensors, see ep_nvfp4_grouped in include/epq.h).  ``swizzled`` calls
    ep_nvfp4_direct_receive_swizzled: both scale tensors in the tiled layout
    of block-scaled GEMM operands (H % 128 == 0).  ``expert_amax`` (f32 [E]):
    each expert's amax as the pack or dispatch reduced it; the call then
    skips its own pass over the row trailers."""
    _need_cuda(rows, "rows", torch.uint8)
    _need_amax(expert_amax, E)
    R_cap = rows.shape[0]
    if out is None:
        out = alloc_grouped(R_cap, H, E, rows.device, rowwise)
    if status is None:
        status = new_status(rows.device)
    desc = grouped_struct(out)
    name = "ep_nvfp4_direct_receive_swizzled" if swizzled else "ep_nvfp4_direct_receive"
    st = getattr(_lib.lib(), name)(_ptr(rows), R_cap, H, _ptr(offsets), E, _ptr(expert_amax), ctypes.byref(desc),
                                   int(rounding),
                                   int(seed) & ((1 << 64) - 1), int(sign_mask) & 0xFFFF, _ptr(status),
                                   _stream(stream))
    check(name, st)
    return out


def ep_nvfp4_colwise_rht_bf16(x: torch.Tensor, offsets: torch.Tensor, E: int, amax: torch.Tensor,
                              out: dict | None = None, rounding: int = EP_ROUND_RNE, seed: int = 0,
                              sign_mask: int = DEFAULT_SIGN_MASK, status: torch.Tensor | None = None,
                              stream=None) -> dict:
    """Expert-grouped BF16 rows [R_cap, H] + supplied per-expert amax [E]
    (f32) -> the columnwise RHT operand and its metadata (keys cw_codes,
    cw_scales, amax_row, amax_col, cw_scale_enc)."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(amax, "amax", torch.float32)
    R_cap, H = x.shape
    dev = x.device
    if out is None:
        out = {"cw_codes": torch.empty(R_cap * H // 2, dtype=torch.uint8, device=dev),
               "cw_scales": torch.empty(R_cap * H // 16, dtype=torch.uint8, device=dev),
               "amax_row": torch.empty(E, dtype=torch.float32, device=dev),
               "amax_col": torch.empty(E, dtype=torch.float32, device=dev),
               "cw_scale_enc": torch.empty(E, dtype=torch.float32, device=dev)}
    if status is None:
        status = new_status(dev)
    st = _lib.lib().ep_nvfp4_colwise_rht_bf16(_ptr(x), R_cap, H, _ptr(offsets), E, _ptr(amax), _ptr(out["cw_codes"]),
                                              _ptr(out["cw_scales"]), _ptr(out["amax_row"]), _ptr(out["amax_col"]),
                                              _ptr(out["cw_scale_enc"]), int(rounding), int(seed) & ((1 << 64) - 1),
                                              int(sign_mask) & 0xFFFF, _ptr(status), _stream(stream))
    check("ep_nvfp4_colwise_rht_bf16", st)
    return out


def ep_mxfp8_colwise(x: torch.Tensor, offsets: torch.Tensor, E: int, buf: torch.Tensor | None = None,
                     status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Expert-grouped BF16 rows [R_cap, H] -> one uint8 buffer: the columnwise
    MXFP8 data (expert e: [H][n_e]) then scales (expert e: [H][n_e/32])."""
    _need_cuda(x, "x", torch.bfloat16)
    R_cap, H = x.shape
    if buf is None:
        buf = torch.empty(R_cap * H + R_cap * (H // 32), dtype=torch.uint8, device=x.device)
    if status is None:
        status = new_status(x.device)
    st = _lib.lib().ep_mxfp8_colwise(_ptr(x), R_cap, H, _ptr(offsets), E, _ptr(buf), _ptr(status), _stream(stream))
    check("ep_mxfp8_colwise", st)
    return buf


def ep_mxfp8_pack(tokens: torch.Tensor, plan: RoutePlan, buf: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """BF16 tokens -> one uint8 buffer: data [R_cap, H] then scales [R_cap, H/32]."""
    _need_cuda(tokens, "tokens", torch.bfloat16)
    T, H = tokens.shape
    if buf is None:
        buf = torch.empty(plan.R_cap * H + plan.R_cap * (H // 32), dtype=torch.uint8, device=tokens.device)
    st = _lib.lib().ep_mxfp8_pack(_ptr(tokens), T, H, _ptr(plan.dest), plan.k, _ptr(plan.offsets),
                                  _ptr(plan.counts), plan.E, _ptr(buf), plan.R_cap, _ptr(plan.status),
                                  _stream(stream))
    check("ep_mxfp8_pack", st)
    return buf
