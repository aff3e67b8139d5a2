"""unpermute_combine_gb300 -- GB300 (sm_103a) MoE token dispatch/combine.

A thin binding over libmoe's C ABI (include/moe.h), one Python function per C
entry point with the same name.  It only marshals arguments: it checks
devices, dtypes and shapes, allocates outputs and workspaces with torch, and
passes raw pointers and the current CUDA stream.  Every step of the path runs
in libmoe's CUDA kernels; there is no CPU or PyTorch fallback, and calling any
op without the built library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "MoeError", "library_path", "load_library", "moe_abi_version", "moe_status_string",
    "moe_route_workspace_size", "moe_route", "moe_route_indices", "moe_permute",
    "moe_sort_chunks_workspace_size", "moe_sort_chunks", "moe_chunk_idxs", "moe_combine",
    "moe_combine_backward", "moe_expert_scale", "moe_workspace_status", "RouteResult",
    "moe_route_noalloc", "MOE_ROUTE_NOALLOC_SCRATCH_BYTES", "moe_grouped_swiglu_pack",
    "moe_grouped_swiglu_workspace_size", "moe_grouped_swiglu", "moe_grouped_swiglu_fp8",
    "moe_device_status",
    "moe_route_grouped", "moe_expert_capacity", "moe_route_layout_rows", "moe_route_layout",
    "moe_fill_pad_rows", "moe_quantize_fp8", "moe_dequantize_fp8", "moe_permute_fp8",
    "moe_route_backward", "moe_grouped_swiglu_save", "moe_grouped_swiglu_dgrad",
    "moe_grouped_swiglu_wgrad", "MOE_STATUS_WORKSPACE_BYTES", "moe_selftest_timeout",
    "moe_permute_quantize_fp8",
]

# Bytes of the status-only workspace of the grouped SwiGLU training calls.
MOE_STATUS_WORKSPACE_BYTES = 256

# Size of the library's built-in scratch array used by moe_route_noalloc.
MOE_ROUTE_NOALLOC_SCRATCH_BYTES = 1 << 20

MOE_OK = 0
_DT = {torch.float32: 0, torch.bfloat16: 1}
_DT_MOVE = dict(_DT)
if hasattr(torch, "float8_e4m3fn"):
    _DT_MOVE[torch.float8_e4m3fn] = 2


class MoeError(RuntimeError):
    def __init__(self, name, status):
        self.status = status
        super().__init__(f"{name} failed: {moe_status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libmoe.so (built in-tree by unpermute_combine_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"libmoe.so is not built ({_build.LIB}); run "
                "`python -m unpermute_combine_gb300.build` or __graft_entry__.build()")
        lib = ctypes.CDLL(_build.LIB)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        PSZ = ctypes.POINTER(ctypes.c_size_t)
        sigs = {
            "moe_status_string": ([I], ctypes.c_char_p),
            "moe_abi_version": ([], I),
            "moe_route_workspace_size": ([I64, I, I, PSZ], I),
            "moe_route": ([P, I64, I, I, P, P, P, P, P, P, P, P, P, P, SZ, P], I),
            "moe_route_indices": ([P, P, I64, I, I, P, P, P, P, P, P, P, P, SZ, P], I),
            "moe_route_noalloc": ([P, I64, I, I, P, P, P, P, P, P, P, P, P, P], I),
            "moe_route_layout_rows": ([I64, I, I, I, I, I, ctypes.POINTER(I64)], I),
            "moe_route_layout": ([P, P, I64, I, I, I, I, I, I64, P, P, P, P, P, P, P, SZ, P], I),
            "moe_fill_pad_rows": ([P, I, I64, I64, P, P, I, P], I),
            "moe_expert_capacity": ([I64, I, I, ctypes.c_double, ctypes.POINTER(I64)], I),
            "moe_quantize_fp8": ([P, I64, I64, I, P, P, P], I),
            "moe_dequantize_fp8": ([P, P, I64, I64, I, P, P], I),
            "moe_permute_fp8": ([P, P, I64, I64, I, I, I64, P, P, P, P], I),
            "moe_permute_quantize_fp8": ([P, I64, I64, I, I, I64, P, P, P, P], I),
            "moe_route_backward": ([P, P, P, I64, I, I, P, P], I),
            "moe_route_grouped": ([P, I64, I, I, I, I, P, P, P, P, P, P, P, P, P, P, SZ, P], I),
            "moe_permute": ([P, I, I64, I64, I, I64, P, P, P], I),
            "moe_sort_chunks_workspace_size": ([I, PSZ], I),
            "moe_sort_chunks": ([P, I, I64, I64, P, P, I, P, P, SZ, P], I),
            "moe_chunk_idxs": ([I, I, I, P], I),
            "moe_combine": ([P, I, I64, I64, I, I64, P, P, P, P], I),
            "moe_combine_backward": ([P, P, I, I64, I64, I, I64, P, P, P, P, P], I),
            "moe_expert_scale": ([P, I, I64, I64, I, P, P, P, P], I),
            "moe_workspace_status": ([P, P], I),
            "moe_device_status": ([P], I),
            "moe_selftest_timeout": ([P, SZ, ctypes.c_uint32, P], I),
            "moe_grouped_swiglu_pack": ([P, P, I, I64, I64, P, P, P], I),
            "moe_grouped_swiglu_workspace_size": ([I64, I, I64, I64, PSZ], I),
            "moe_grouped_swiglu": ([P, P, P, P, I64, I, I64, I64, P, P, SZ, P], I),
            "moe_grouped_swiglu_fp8": ([P, P, P, P, P, I64, I, I64, I64, P, P, SZ, P], I),
            "moe_grouped_swiglu_save": ([P, P, P, P, I64, I, I64, I64, P, P, P, P, SZ, P], I),
            "moe_grouped_swiglu_dgrad": ([P, P, P, P, P, I64, I, I64, I64, P, P, P, SZ, P], I),
            "moe_grouped_swiglu_wgrad": ([P, P, P, P, P, I64, I, I64, I64, P, P, P, SZ, P], I),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(int(status)).decode()


def moe_abi_version() -> int:
    return load_library().moe_abi_version()


# ------------------------------------------------------------------ helpers

def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ok(name, status):
    if status != MOE_OK:
        raise MoeError(name, status)


def _cuda(t, name, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t


def _act(t, name):
    _cuda(t, name, ndim=2)
    if t.dtype not in _DT:
        raise ValueError(f"{name} must be float32 or bfloat16, got {t.dtype}")
    return _DT[t.dtype]


def _act_move(t, name):
    _cuda(t, name, ndim=2)
    if t.dtype not in _DT_MOVE:
        raise ValueError(f"{name} must be float32, bfloat16 or float8_e4m3fn, got {t.dtype}")
    return _DT_MOVE[t.dtype]


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def _workspace(nbytes, like, given):
    if given is not None:
        _cuda(given, "workspace", torch.uint8)
        if given.numel() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes, got {given.numel()}")
        return given
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=like.device)


# -------------------------------------------------------------------- route

@dataclass
class RouteResult:
    topk_idx: Optional[torch.Tensor]
    topk_w: Optional[torch.Tensor]
    counts: torch.Tensor
    offsets: torch.Tensor
    group_list: torch.Tensor
    sorted_indices: torch.Tensor
    slot_pos: torch.Tensor
    permuted_probs: Optional[torch.Tensor]
    routing_map: Optional[torch.Tensor]
    workspace: torch.Tensor


def moe_route_workspace_size(T: int, E: int, k: int) -> int:
    n = ctypes.c_size_t(0)
    _ok("moe_route_workspace_size",
        load_library().moe_route_workspace_size(T, E, k, ctypes.byref(n)))
    return n.value


def moe_route(logits: torch.Tensor, k: int, *, routing_map: bool = False,
              workspace: Optional[torch.Tensor] = None, out: Optional[RouteResult] = None,
              stream=None) -> RouteResult:
    """Top-k + softmax over the k scores, counts, offsets/group_list,
    expert-major sorted_indices, slot_pos and permuted_probs (moe.h)."""
    _cuda(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    ws_bytes = moe_route_workspace_size(T, E, k)
    ws = _workspace(ws_bytes, logits, workspace if out is None else out.workspace)
    if out is None:
        i32 = torch.int32
        out = RouteResult(
            topk_idx=_empty((T, k), i32, logits), topk_w=_empty((T, k), torch.float32, logits),
            counts=_empty((E,), i32, logits), offsets=_empty((E + 1,), i32, logits),
            group_list=_empty((E,), i32, logits), sorted_indices=_empty((T * k,), i32, logits),
            slot_pos=_empty((T, k), i32, logits),
            permuted_probs=_empty((T * k,), torch.float32, logits),
            routing_map=_empty((T, E), torch.uint8, logits) if routing_map else None,
            workspace=ws)
    _ok("moe_route", load_library().moe_route(
        _p(logits), T, E, k, _p(out.topk_idx), _p(out.topk_w), _p(out.counts), _p(out.offsets),
        _p(out.group_list), _p(out.sorted_indices), _p(out.slot_pos), _p(out.permuted_probs),
        _p(out.routing_map), _p(ws), ws.numel(), _stream(stream)))
    return out


def moe_route_grouped(logits: torch.Tensor, k: int, n_groups: int, topk_groups: int, *,
                      routing_map: bool = False, workspace: Optional[torch.Tensor] = None,
                      out: Optional[RouteResult] = None, stream=None) -> RouteResult:
    """Group-limited routing: keep the topk_groups best of n_groups consecutive
    expert groups (scored by their largest logit), then route as moe_route."""
    _cuda(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    ws = _workspace(moe_route_workspace_size(T, E, k), logits,
                    workspace if out is None else out.workspace)
    if out is None:
        i32 = torch.int32
        out = RouteResult(
            topk_idx=_empty((T, k), i32, logits), topk_w=_empty((T, k), torch.float32, logits),
            counts=_empty((E,), i32, logits), offsets=_empty((E + 1,), i32, logits),
            group_list=_empty((E,), i32, logits), sorted_indices=_empty((T * k,), i32, logits),
            slot_pos=_empty((T, k), i32, logits),
            permuted_probs=_empty((T * k,), torch.float32, logits),
            routing_map=_empty((T, E), torch.uint8, logits) if routing_map else None,
            workspace=ws)
    _ok("moe_route_grouped", load_library().moe_route_grouped(
        _p(logits), T, E, k, n_groups, topk_groups, _p(out.topk_idx), _p(out.topk_w),
        _p(out.counts), _p(out.offsets), _p(out.group_list), _p(out.sorted_indices),
        _p(out.slot_pos), _p(out.permuted_probs), _p(out.routing_map), _p(ws), ws.numel(),
        _stream(stream)))
    return out


def moe_route_indices(topk_idx: torch.Tensor, topk_w: Optional[torch.Tensor], E: int, *,
                      routing_map: bool = False, workspace: Optional[torch.Tensor] = None,
                      stream=None) -> RouteResult:
    """Index outputs of moe_route from given top-k choices (-1 = empty slot)."""
    _cuda(topk_idx, "topk_idx", torch.int32, 2)
    T, k = topk_idx.shape
    if topk_w is not None:
        _cuda(topk_w, "topk_w", torch.float32, 2)
        if tuple(topk_w.shape) != (T, k):
            raise ValueError("topk_w must match topk_idx")
    ws = _workspace(moe_route_workspace_size(T, E, k), topk_idx, workspace)
    i32 = torch.int32
    r = RouteResult(
        topk_idx=topk_idx, topk_w=topk_w, counts=_empty((E,), i32, topk_idx),
        offsets=_empty((E + 1,), i32, topk_idx), group_list=_empty((E,), i32, topk_idx),
        sorted_indices=_empty((T * k,), i32, topk_idx), slot_pos=_empty((T, k), i32, topk_idx),
        permuted_probs=_empty((T * k,), torch.float32, topk_idx) if topk_w is not None else None,
        routing_map=_empty((T, E), torch.uint8, topk_idx) if routing_map else None,
        workspace=ws)
    _ok("moe_route_indices", load_library().moe_route_indices(
        _p(topk_idx), _p(topk_w), T, E, k, _p(r.counts), _p(r.offsets), _p(r.group_list),
        _p(r.sorted_indices), _p(r.slot_pos), _p(r.permuted_probs), _p(r.routing_map), _p(ws),
        ws.numel(), _stream(stream)))
    return r


def moe_route_noalloc(logits: torch.Tensor, k: int, *, routing_map: bool = False,
                      stream=None) -> RouteResult:
    """moe_route without a workspace, for callers that cannot allocate device
    memory for scratch: the library's built-in scratch array is used instead
    (calls that overlap on the GPU must be serialised).  The outputs are
    allocated here only because this binding returns new tensors; the C entry
    point itself allocates nothing."""
    _cuda(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    i32 = torch.int32
    r = RouteResult(
        topk_idx=_empty((T, k), i32, logits), topk_w=_empty((T, k), torch.float32, logits),
        counts=_empty((E,), i32, logits), offsets=_empty((E + 1,), i32, logits),
        group_list=_empty((E,), i32, logits), sorted_indices=_empty((T * k,), i32, logits),
        slot_pos=_empty((T, k), i32, logits),
        permuted_probs=_empty((T * k,), torch.float32, logits),
        routing_map=_empty((T, E), torch.uint8, logits) if routing_map else None,
        workspace=None)
    _ok("moe_route_noalloc", load_library().moe_route_noalloc(
        _p(logits), T, E, k, _p(r.topk_idx), _p(r.topk_w), _p(r.counts), _p(r.offsets),
        _p(r.group_list), _p(r.sorted_indices), _p(r.slot_pos), _p(r.permuted_probs),
        _p(r.routing_map), _stream(stream)))
    return r


# ------------------------------------------------------------ FP8 dispatch

def moe_route_backward(topk_idx: torch.Tensor, topk_w: torch.Tensor, grad_probs: torch.Tensor,
                       E: int, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """grad_logits [T,E] float32 of the k-softmax router (zero off the chosen
    experts)."""
    _cuda(topk_idx, "topk_idx", torch.int32, 2)
    _cuda(topk_w, "topk_w", torch.float32, 2)
    _cuda(grad_probs, "grad_probs", torch.float32, 2)
    T, k = topk_idx.shape
    if topk_w.shape != (T, k) or grad_probs.shape != (T, k):
        raise ValueError("topk_idx, topk_w and grad_probs must all be [T, k]")
    if out is None:
        out = torch.empty((T, E), dtype=torch.float32, device=topk_idx.device)
    else:
        _cuda(out, "grad_logits", torch.float32, 2)
        if tuple(out.shape) != (T, E):
            raise ValueError("grad_logits must be [T, E]")
    _ok("moe_route_backward", load_library().moe_route_backward(
        _p(topk_idx), _p(topk_w), _p(grad_probs), T, E, k, _p(out), _stream(stream)))
    return out


def moe_quantize_fp8(x: torch.Tensor, block: int = 128, out=None, stream=None):
    """(x_q float8_e4m3fn [T,H], scales float32 [T,H/block]) of bf16 rows;
    out: an optional (x_q, scales) pair to write into."""
    _cuda(x, "x", torch.bfloat16, 2)
    T, H = x.shape
    if out is None:
        q = torch.empty((T, H), dtype=torch.float8_e4m3fn, device=x.device)
        sc = torch.empty((T, H // block if block else 0), dtype=torch.float32, device=x.device)
    else:
        q, sc = out
        _cuda(q, "x_q", torch.float8_e4m3fn, 2)
        _cuda(sc, "scales", torch.float32, 2)
    _ok("moe_quantize_fp8", load_library().moe_quantize_fp8(_p(x), T, H, block, _p(q), _p(sc),
                                                            _stream(stream)))
    return q, sc


def moe_dequantize_fp8(x_q: torch.Tensor, scales: torch.Tensor, block: int = 128,
                       out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """bf16(x_q * scale) per block."""
    _cuda(x_q, "x_q", torch.float8_e4m3fn, 2)
    _cuda(scales, "scales", torch.float32, 2)
    N, H = x_q.shape
    if out is None:
        out = torch.empty((N, H), dtype=torch.bfloat16, device=x_q.device)
    _ok("moe_dequantize_fp8", load_library().moe_dequantize_fp8(
        _p(x_q), _p(scales), N, H, block, _p(out), _stream(stream)))
    return out


def moe_permute_fp8(x_q: torch.Tensor, scales: torch.Tensor, slot_pos: torch.Tensor, out=None,
                    n_rows: Optional[int] = None, stream=None):
    """Move e4m3 rows and their scale rows to the slot rows slot_pos names, in
    one launch; returns (out_q [n_rows,H], out_scales [n_rows,H/block])."""
    _cuda(x_q, "x_q", torch.float8_e4m3fn, 2)
    _cuda(scales, "scales", torch.float32, 2)
    _cuda(slot_pos, "slot_pos", torch.int32, 2)
    T, H = x_q.shape
    k = slot_pos.shape[1]
    if slot_pos.shape[0] != T or scales.shape[0] != T or scales.shape[1] == 0 or \
            H % scales.shape[1] != 0:
        raise ValueError("x_q, scales and slot_pos must have one row per token, "
                         "and scales H/block columns")
    block = H // scales.shape[1]
    if out is None:
        rows = T * k if n_rows is None else n_rows
        oq = torch.empty((rows, H), dtype=torch.float8_e4m3fn, device=x_q.device)
        osc = torch.empty((rows, scales.shape[1]), dtype=torch.float32, device=x_q.device)
    else:
        oq, osc = out
        _cuda(oq, "out_q", torch.float8_e4m3fn, 2)
        _cuda(osc, "out_scales", torch.float32, 2)
        if oq.shape[0] != osc.shape[0] or oq.shape[1] != H or osc.shape[1] != scales.shape[1]:
            raise ValueError("out_q / out_scales shapes do not match x_q / scales")
    _ok("moe_permute_fp8", load_library().moe_permute_fp8(
        _p(x_q), _p(scales), T, H, block, k, oq.shape[0], _p(slot_pos), _p(oq), _p(osc),
        _stream(stream)))
    return oq, osc


def moe_permute_quantize_fp8(x: torch.Tensor, slot_pos: torch.Tensor, block: int = 128,
                             out=None, n_rows: Optional[int] = None, stream=None):
    """Quantize bf16 token rows to e4m3 with per-block scales and move them to
    the slot rows slot_pos names, in one launch (the same bytes as
    moe_quantize_fp8 followed by moe_permute_fp8); returns
    (out_q [n_rows,H] e4m3, out_scales [n_rows,H/block] float32)."""
    _cuda(x, "x", torch.bfloat16, 2)
    _cuda(slot_pos, "slot_pos", torch.int32, 2)
    T, H = x.shape
    k = slot_pos.shape[1]
    if slot_pos.shape[0] != T:
        raise ValueError("slot_pos must have one row per token")
    if block <= 0 or H % block != 0:
        raise ValueError("H must be a multiple of block")
    if out is None:
        rows = T * k if n_rows is None else n_rows
        oq = torch.empty((rows, H), dtype=torch.float8_e4m3fn, device=x.device)
        osc = torch.empty((rows, H // block), dtype=torch.float32, device=x.device)
    else:
        oq, osc = out
        _cuda(oq, "out_q", torch.float8_e4m3fn, 2)
        _cuda(osc, "out_scales", torch.float32, 2)
        if oq.shape[0] != osc.shape[0] or oq.shape[1] != H or osc.shape[1] != H // block:
            raise ValueError("out_q must be [n_rows, H] and out_scales [n_rows, H/block]")
    _ok("moe_permute_quantize_fp8", load_library().moe_permute_quantize_fp8(
        _p(x), T, H, block, k, oq.shape[0], _p(slot_pos), _p(oq), _p(osc), _stream(stream)))
    return oq, osc


# ---------------------------------------------- capacity / padded layout

def moe_expert_capacity(tokens: int, top_k: int, num_experts: int,
                        capacity_factor: float) -> int:
    c = ctypes.c_int64(0)
    _ok("moe_expert_capacity", load_library().moe_expert_capacity(
        tokens, top_k, num_experts, float(capacity_factor), ctypes.byref(c)))
    return c.value


def moe_route_layout_rows(T: int, E: int, k: int, capacity: int = 0, pad: bool = False,
                          alignment: int = 1) -> int:
    n = ctypes.c_int64(0)
    _ok("moe_route_layout_rows", load_library().moe_route_layout_rows(
        T, E, k, capacity, int(bool(pad)), alignment, ctypes.byref(n)))
    return n.value


def moe_route_layout(topk_idx: torch.Tensor, topk_w: Optional[torch.Tensor], E: int, *,
                     capacity: int = 0, pad: bool = False, alignment: int = 1,
                     max_rows: Optional[int] = None, workspace: Optional[torch.Tensor] = None,
                     stream=None) -> RouteResult:
    """Index outputs for a capacity-bounded, padded or aligned layout (moe.h)."""
    _cuda(topk_idx, "topk_idx", torch.int32, 2)
    T, k = topk_idx.shape
    if topk_w is not None:
        _cuda(topk_w, "topk_w", torch.float32, 2)
    if max_rows is None:
        max_rows = moe_route_layout_rows(T, E, k, capacity, pad, alignment)
    ws = _workspace(moe_route_workspace_size(T, E, k), topk_idx, workspace)
    i32 = torch.int32
    r = RouteResult(
        topk_idx=topk_idx, topk_w=topk_w, counts=_empty((E,), i32, topk_idx),
        offsets=_empty((E + 1,), i32, topk_idx), group_list=_empty((E,), i32, topk_idx),
        sorted_indices=_empty((max_rows,), i32, topk_idx), slot_pos=_empty((T, k), i32, topk_idx),
        permuted_probs=_empty((max_rows,), torch.float32, topk_idx) if topk_w is not None else None,
        routing_map=None, workspace=ws)
    _ok("moe_route_layout", load_library().moe_route_layout(
        _p(topk_idx), _p(topk_w), T, E, k, capacity, int(bool(pad)), alignment, max_rows,
        _p(r.counts), _p(r.offsets), _p(r.group_list), _p(r.sorted_indices), _p(r.slot_pos),
        _p(r.permuted_probs), _p(ws), ws.numel(), _stream(stream)))
    return r


def moe_fill_pad_rows(rows: torch.Tensor, offsets: torch.Tensor, counts: torch.Tensor,
                      stream=None) -> torch.Tensor:
    """Zero the padding rows of a padded / aligned permuted buffer."""
    dt = _act_move(rows, "rows")
    _cuda(offsets, "offsets", torch.int32, 1)
    _cuda(counts, "counts", torch.int32, 1)
    E = counts.numel()
    _ok("moe_fill_pad_rows", load_library().moe_fill_pad_rows(
        _p(rows), dt, rows.shape[0], rows.shape[1], _p(offsets), _p(counts), E, _stream(stream)))
    return rows


# ------------------------------------------------------------------ permute

def moe_permute(x: torch.Tensor, slot_pos: torch.Tensor, out: Optional[torch.Tensor] = None,
                n_rows: Optional[int] = None, stream=None) -> torch.Tensor:
    """permuted[slot_pos[t,j]] = x[t]; out has n_rows rows (T*k by default, or
    out's rows); rows no slot names are left as they were."""
    dt = _act_move(x, "x")
    _cuda(slot_pos, "slot_pos", torch.int32, 2)
    T, H = x.shape
    k = slot_pos.shape[1]
    if slot_pos.shape[0] != T:
        raise ValueError("slot_pos must have one row per token")
    if out is None:
        out = _empty((T * k if n_rows is None else n_rows, H), x.dtype, x)
    else:
        _cuda(out, "out", x.dtype, 2)
        if out.shape[1] != H:
            raise ValueError("out must have H columns")
    _ok("moe_permute", load_library().moe_permute(_p(x), dt, T, H, k, out.shape[0], _p(slot_pos),
                                                  _p(out), _stream(stream)))
    return out


# -------------------------------------------------------------- sort_chunks

def moe_sort_chunks_workspace_size(C: int) -> int:
    n = ctypes.c_size_t(0)
    _ok("moe_sort_chunks_workspace_size",
        load_library().moe_sort_chunks_workspace_size(C, ctypes.byref(n)))
    return n.value


def moe_sort_chunks(x: torch.Tensor, split_sizes: torch.Tensor, sorted_idxs: torch.Tensor,
                    out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """out = cat([x.split(split_sizes)[i] for i in sorted_idxs]); split_sizes
    and sorted_idxs are int32 CUDA tensors (no host synchronisation)."""
    dt = _act_move(x, "x")
    _cuda(split_sizes, "split_sizes", torch.int32, 1)
    _cuda(sorted_idxs, "sorted_idxs", torch.int32, 1)
    C = split_sizes.numel()
    if sorted_idxs.numel() != C:
        raise ValueError("split_sizes and sorted_idxs must have the same length")
    N, H = x.shape
    if out is None:
        out = torch.empty_like(x)
    else:
        _cuda(out, "out", x.dtype, 2)
        if out.shape != x.shape:
            raise ValueError("out must match x")
    ws = _workspace(moe_sort_chunks_workspace_size(C), x, workspace)
    _ok("moe_sort_chunks", load_library().moe_sort_chunks(
        _p(x), dt, N, H, _p(split_sizes), _p(sorted_idxs), C, _p(out), _p(ws), ws.numel(),
        _stream(stream)))
    out._moe_workspace = ws  # keeps the status word reachable for moe_workspace_status
    return out


def moe_chunk_idxs(R: int, L: int, inverse: bool = False) -> list:
    """Host helper: rank-major -> expert-major chunk order of an [R x L] split
    matrix (inverse=True: the way back, used with the transposed splits)."""
    buf = (ctypes.c_int32 * (R * L))()
    _ok("moe_chunk_idxs", load_library().moe_chunk_idxs(R, L, int(bool(inverse)), buf))
    return list(buf)


# ------------------------------------------------------------------ combine

def moe_combine(expert_out: torch.Tensor, slot_pos: torch.Tensor,
                topk_w: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """out[t] = sum_j topk_w[t,j] * expert_out[slot_pos[t,j]] (topk_w=None: plain sum)."""
    dt = _act(expert_out, "expert_out")
    _cuda(slot_pos, "slot_pos", torch.int32, 2)
    T, k = slot_pos.shape
    n_rows, H = expert_out.shape
    if topk_w is not None:
        _cuda(topk_w, "topk_w", torch.float32, 2)
        if tuple(topk_w.shape) != (T, k):
            raise ValueError("topk_w must be [T, k]")
    if out is None:
        out = _empty((T, H), expert_out.dtype, expert_out)
    else:
        _cuda(out, "out", expert_out.dtype, 2)
        if tuple(out.shape) != (T, H):
            raise ValueError("out must be [T, H]")
    _ok("moe_combine", load_library().moe_combine(
        _p(expert_out), dt, T, H, k, n_rows, _p(slot_pos), _p(topk_w), _p(out), _stream(stream)))
    return out


def moe_combine_backward(grad_out: torch.Tensor, expert_out: torch.Tensor,
                         slot_pos: torch.Tensor, topk_w: Optional[torch.Tensor] = None,
                         grad_expert_out: Optional[torch.Tensor] = None,
                         grad_probs: Optional[torch.Tensor] = None, stream=None):
    """(grad_expert_out, grad_probs) of the combine; expert_out may have any
    number of rows (T*k, or a padded layout's); rows no slot names are left as
    they were."""
    dt = _act(expert_out, "expert_out")
    _act(grad_out, "grad_out")
    if grad_out.dtype != expert_out.dtype:
        raise ValueError("grad_out and expert_out must share a dtype")
    _cuda(slot_pos, "slot_pos", torch.int32, 2)
    T, k = slot_pos.shape
    n_rows, H = expert_out.shape
    if tuple(grad_out.shape) != (T, H):
        raise ValueError("grad_out must be [T, H]")
    if topk_w is not None:
        _cuda(topk_w, "topk_w", torch.float32, 2)
    if grad_expert_out is None:
        grad_expert_out = torch.empty_like(expert_out)
    else:
        _cuda(grad_expert_out, "grad_expert_out", expert_out.dtype, 2)
    if grad_probs is None:
        grad_probs = _empty((T, k), torch.float32, expert_out)
    else:
        _cuda(grad_probs, "grad_probs", torch.float32, 2)
    _ok("moe_combine_backward", load_library().moe_combine_backward(
        _p(grad_out), _p(expert_out), dt, T, H, k, n_rows, _p(slot_pos), _p(topk_w),
        _p(grad_expert_out), _p(grad_probs), _stream(stream)))
    return grad_expert_out, grad_probs


# ---------------------------------------------------------- stand-in expert

def moe_expert_scale(x_perm: torch.Tensor, offsets: torch.Tensor, scale: torch.Tensor,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[p] = x_perm[p] * scale[e] over the expert segments given by offsets."""
    dt = _act(x_perm, "x_perm")
    _cuda(offsets, "offsets", torch.int32, 1)
    _cuda(scale, "scale", torch.float32, 1)
    E = scale.numel()
    if offsets.numel() != E + 1:
        raise ValueError("offsets must have E+1 entries")
    n, H = x_perm.shape
    if out is None:
        out = torch.empty_like(x_perm)
    _ok("moe_expert_scale", load_library().moe_expert_scale(
        _p(x_perm), dt, n, H, E, _p(offsets), _p(scale), _p(out), _stream(stream)))
    return out


# ----------------------------------------------------------- grouped SwiGLU

def moe_grouped_swiglu_pack(w_up: torch.Tensor, w_down: torch.Tensor, stream=None):
    """One-time weight prepack: w_up [E,H,2I] -> [E,2I,H] (gate/up interleaved
    in 128-row blocks), w_down [E,I,H] -> [E,H,I]; both bf16."""
    _cuda(w_up, "w_up", torch.bfloat16, 3)
    _cuda(w_down, "w_down", torch.bfloat16, 3)
    E, H, I2 = w_up.shape
    I = I2 // 2
    if tuple(w_down.shape) != (E, I, H) or I2 != 2 * I:
        raise ValueError("w_up must be [E,H,2I] and w_down [E,I,H]")
    up_p = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=w_up.device)
    down_p = torch.empty((E, H, I), dtype=torch.bfloat16, device=w_up.device)
    _ok("moe_grouped_swiglu_pack", load_library().moe_grouped_swiglu_pack(
        _p(w_up), _p(w_down), E, H, I, _p(up_p), _p(down_p), _stream(stream)))
    return up_p, down_p


def moe_grouped_swiglu_workspace_size(N: int, E: int, H: int, I: int) -> int:
    n = ctypes.c_size_t(0)
    _ok("moe_grouped_swiglu_workspace_size",
        load_library().moe_grouped_swiglu_workspace_size(N, E, H, I, ctypes.byref(n)))
    return n.value


def moe_grouped_swiglu(x: torch.Tensor, w_up_packed: torch.Tensor, w_down_packed: torch.Tensor,
                       offsets: torch.Tensor, out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y = per-expert SwiGLU FFN over the expert segments of x (see moe.h)."""
    _cuda(x, "x", torch.bfloat16, 2)
    _cuda(w_up_packed, "w_up_packed", torch.bfloat16, 3)
    _cuda(w_down_packed, "w_down_packed", torch.bfloat16, 3)
    _cuda(offsets, "offsets", torch.int32, 1)
    N, H = x.shape
    E, I2, H2 = w_up_packed.shape
    I = I2 // 2
    if H2 != H or tuple(w_down_packed.shape) != (E, H, I) or offsets.numel() != E + 1:
        raise ValueError("packed weights / offsets do not match x")
    if out is None:
        out = torch.empty_like(x)
    ws = _workspace(moe_grouped_swiglu_workspace_size(N, E, H, I), x, workspace)
    _ok("moe_grouped_swiglu", load_library().moe_grouped_swiglu(
        _p(x), _p(w_up_packed), _p(w_down_packed), _p(offsets), N, E, H, I, _p(out), _p(ws),
        ws.numel(), _stream(stream)))
    out._moe_workspace = ws
    return out


def moe_grouped_swiglu_fp8(x_q: torch.Tensor, scales: torch.Tensor, w_up_packed: torch.Tensor,
                           w_down_packed: torch.Tensor, offsets: torch.Tensor,
                           out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """moe_grouped_swiglu on e4m3 rows x_q [N,H] (float8_e4m3fn) and their
    per-128-column scales [N, H/128] float32; returns y [N,H] bf16."""
    _cuda(x_q, "x_q", torch.float8_e4m3fn, 2)
    _cuda(scales, "scales", torch.float32, 2)
    _cuda(w_up_packed, "w_up_packed", torch.bfloat16, 3)
    _cuda(w_down_packed, "w_down_packed", torch.bfloat16, 3)
    _cuda(offsets, "offsets", torch.int32, 1)
    N, H = x_q.shape
    E, I2, H2 = w_up_packed.shape
    I = I2 // 2
    if H2 != H or tuple(w_down_packed.shape) != (E, H, I) or offsets.numel() != E + 1:
        raise ValueError("packed weights / offsets do not match x_q")
    if H % 128 or tuple(scales.shape) != (N, H // 128):
        raise ValueError("scales must be [N, H/128] (block = 128)")
    if out is None:
        out = torch.empty((N, H), dtype=torch.bfloat16, device=x_q.device)
    ws = _workspace(moe_grouped_swiglu_workspace_size(N, E, H, I), x_q, workspace)
    _ok("moe_grouped_swiglu_fp8", load_library().moe_grouped_swiglu_fp8(
        _p(x_q), _p(scales), _p(w_up_packed), _p(w_down_packed), _p(offsets), N, E, H, I,
        _p(out), _p(ws), ws.numel(), _stream(stream)))
    out._moe_workspace = ws
    return out


def moe_grouped_swiglu_save(x: torch.Tensor, w_up_packed: torch.Tensor,
                            w_down_packed: torch.Tensor, offsets: torch.Tensor, out=None,
                            hidden=None, gate_up=None, workspace=None, stream=None):
    """Training forward: (y [N,H], hidden [N,I], gate_up [N,2I]), all bf16."""
    _cuda(x, "x", torch.bfloat16, 2)
    _cuda(w_up_packed, "w_up_packed", torch.bfloat16, 3)
    _cuda(w_down_packed, "w_down_packed", torch.bfloat16, 3)
    _cuda(offsets, "offsets", torch.int32, 1)
    N, H = x.shape
    E, I2, H2 = w_up_packed.shape
    I = I2 // 2
    if H2 != H or tuple(w_down_packed.shape) != (E, H, I) or offsets.numel() != E + 1:
        raise ValueError("packed weights / offsets do not match x")
    out = torch.empty_like(x) if out is None else out
    hidden = x.new_empty((N, I)) if hidden is None else hidden
    gate_up = x.new_empty((N, 2 * I)) if gate_up is None else gate_up
    for t, name, shape in ((out, "y", (N, H)), (hidden, "hidden", (N, I)),
                           (gate_up, "gate_up", (N, 2 * I))):
        _cuda(t, name, torch.bfloat16, 2)
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {list(shape)}")
    ws = _workspace(MOE_STATUS_WORKSPACE_BYTES, x, workspace)
    _ok("moe_grouped_swiglu_save", load_library().moe_grouped_swiglu_save(
        _p(x), _p(w_up_packed), _p(w_down_packed), _p(offsets), N, E, H, I, _p(out), _p(hidden),
        _p(gate_up), _p(ws), ws.numel(), _stream(stream)))
    out._moe_workspace = ws
    return out, hidden, gate_up


def moe_grouped_swiglu_dgrad(dy: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                             offsets: torch.Tensor, gate_up: torch.Tensor, dgate_up=None,
                             dx=None, workspace=None, stream=None):
    """(dgate_up [N,2I], dx [N,H]) bf16; w_up [E,H,2I] and w_down [E,I,H] in
    their original (unpacked) layouts."""
    _cuda(dy, "dy", torch.bfloat16, 2)
    _cuda(w_up, "w_up", torch.bfloat16, 3)
    _cuda(w_down, "w_down", torch.bfloat16, 3)
    _cuda(offsets, "offsets", torch.int32, 1)
    _cuda(gate_up, "gate_up", torch.bfloat16, 2)
    N, H = dy.shape
    E, H2, I2 = w_up.shape
    I = I2 // 2
    if H2 != H or tuple(w_down.shape) != (E, I, H) or offsets.numel() != E + 1 or \
            tuple(gate_up.shape) != (N, 2 * I):
        raise ValueError("weights / offsets / gate_up do not match dy")
    dgate_up = dy.new_empty((N, 2 * I)) if dgate_up is None else dgate_up
    dx = dy.new_empty((N, H)) if dx is None else dx
    _cuda(dgate_up, "dgate_up", torch.bfloat16, 2)
    _cuda(dx, "dx", torch.bfloat16, 2)
    if tuple(dgate_up.shape) != (N, 2 * I) or tuple(dx.shape) != (N, H):
        raise ValueError("dgate_up must be [N,2I] and dx [N,H]")
    ws = _workspace(MOE_STATUS_WORKSPACE_BYTES, dy, workspace)
    _ok("moe_grouped_swiglu_dgrad", load_library().moe_grouped_swiglu_dgrad(
        _p(dy), _p(w_up), _p(w_down), _p(offsets), _p(gate_up), N, E, H, I, _p(dgate_up), _p(dx),
        _p(ws), ws.numel(), _stream(stream)))
    dx._moe_workspace = ws
    return dgate_up, dx


def moe_grouped_swiglu_wgrad(x: torch.Tensor, hidden: torch.Tensor, dy: torch.Tensor,
                             dgate_up: torch.Tensor, offsets: torch.Tensor, dw_up=None,
                             dw_down=None, up: bool = True, down: bool = True, workspace=None,
                             stream=None):
    """(dw_up fp32 [E,H,2I] or None, dw_down fp32 [E,I,H] or None)."""
    _cuda(x, "x", torch.bfloat16, 2)
    _cuda(hidden, "hidden", torch.bfloat16, 2)
    _cuda(dy, "dy", torch.bfloat16, 2)
    _cuda(dgate_up, "dgate_up", torch.bfloat16, 2)
    _cuda(offsets, "offsets", torch.int32, 1)
    N, H = x.shape
    I = hidden.shape[1]
    E = offsets.numel() - 1
    if tuple(hidden.shape) != (N, I) or tuple(dy.shape) != (N, H) or \
            tuple(dgate_up.shape) != (N, 2 * I):
        raise ValueError("x, hidden, dy and dgate_up shapes do not agree")
    f32 = torch.float32
    if up and dw_up is None:
        dw_up = torch.empty((E, H, 2 * I), dtype=f32, device=x.device)
    if down and dw_down is None:
        dw_down = torch.empty((E, I, H), dtype=f32, device=x.device)
    if not up:
        dw_up = None
    if not down:
        dw_down = None
    for t, name, shape in ((dw_up, "dw_up", (E, H, 2 * I)), (dw_down, "dw_down", (E, I, H))):
        if t is not None:
            _cuda(t, name, f32, 3)
            if tuple(t.shape) != shape:
                raise ValueError(f"{name} must be {list(shape)}")
    ws = _workspace(MOE_STATUS_WORKSPACE_BYTES, x, workspace)
    _ok("moe_grouped_swiglu_wgrad", load_library().moe_grouped_swiglu_wgrad(
        _p(x), _p(hidden), _p(dy), _p(dgate_up), _p(offsets), N, E, H, I, _p(dw_up),
        _p(dw_down), _p(ws), ws.numel(), _stream(stream)))
    for t in (dw_up, dw_down):
        if t is not None:
            t._moe_workspace = ws
    return dw_up, dw_down


def moe_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the status word a call left in the
    workspace (0 = MOE_OK, 6 = MOE_ERR_DEVICE_CHECK, 5 = MOE_ERR_TIMEOUT)."""
    _cuda(workspace, "workspace", torch.uint8)
    return load_library().moe_workspace_status(_p(workspace), _stream(stream))


def moe_device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the library's device status
    word (0 = MOE_OK, 5 = MOE_ERR_TIMEOUT from a kernel without a workspace)."""
    return load_library().moe_device_status(_stream(stream))


def moe_selftest_timeout(polls: int = 1024, workspace: Optional[torch.Tensor] = None,
                         device=None, stream=None) -> int:
    """Run the bounded-wait health check (moe.h): a kernel waits on a barrier
    nothing completes, gives up after `polls` polls and records the timeout;
    returns the workspace status it left (5 = MOE_ERR_TIMEOUT expected)."""
    if workspace is None:
        workspace = torch.empty(MOE_STATUS_WORKSPACE_BYTES, dtype=torch.uint8,
                                device=device if device is not None else "cuda")
    _cuda(workspace, "workspace", torch.uint8)
    _ok("moe_selftest_timeout", load_library().moe_selftest_timeout(
        _p(workspace), workspace.numel(), polls, _stream(stream)))
    return moe_workspace_status(workspace, stream)
