"""CPU oracle for the MoE dispatch/combine path -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It wraps ``oracle.c`` (plain C loops, double
accumulation, one rounding per output) with ctypes and numpy; it imports
nothing from the product package and the product package imports nothing
from here.  bf16 tensors are numpy ``uint16`` arrays of bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

F32 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (portable flags only)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(os.path.join(_HERE, f)) > os.path.getmtime(_LIB)
        for f in ("oracle.c", "oracle.h"))
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                        "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            sig = {
                "oracle_bf16_from_double": [P, I64, P],
                "oracle_topk_softmax": [P, I64, I, I, P, P, P],
                "oracle_topk_softmax_grouped": [P, I64, I, I, I, I, P, P, P],
                "oracle_route_indices": [P, P, I64, I, I, P, P, P, P, P, P, P],
                "oracle_permute": [P, I, I64, I64, P, I64, P],
                "oracle_route_backward": [P, P, P, I64, I, I, P],
                "oracle_swiglu_dgrad": [P, P, P, P, P, I, I64, I64, P, I64, P, P, P, P],
                "oracle_swiglu_wgrad_at": [P, P, P, P, P, I, I64, I64, I, P, I64, P],
                "oracle_quantize_fp8": [P, I64, I64, I, P, P],
                "oracle_dequantize_fp8": [P, P, I64, I64, I, P],
                "oracle_e4m3_from_float": [P, I64, P],
                "oracle_route_layout": [P, P, I64, I, I, I, I, I, I64, P, P, P, P, P, P],
                "oracle_chunk_idxs": [I, I, I, P],
                "oracle_sort_chunks": [P, I64, I64, P, P, I, P],
                "oracle_combine": [P, I, I64, I64, I, P, P, P, P],
                "oracle_unpermute": [P, I, I64, I64, P, P, I64, P, P],
                "oracle_combine_backward": [P, P, I, I64, I64, I, P, P, P, P, P],
                "oracle_expert_scale": [P, I, I64, I, P, P, P],
                "oracle_grouped_swiglu": [P, P, P, P, I, I64, I64, P, I64, P, P, P, P],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.oracle_expert_capacity.argtypes = [I64, I, I, ctypes.c_double]
            lib.oracle_expert_capacity.restype = I64
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments (rc={rc})")


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dtype_code(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"expected float32 or uint16 (bf16 bits), got {a.dtype}")


def bf16_from_double(v):
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _check(_load().oracle_bf16_from_double(_ptr(v), v.size, _ptr(out)), "bf16_from_double")
    return out


def topk_softmax(logits, k):
    """Top-k (descending, ties to the lower id) and softmax over the k scores."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    w64 = np.empty((T, k), np.float64)
    _check(_load().oracle_topk_softmax(_ptr(logits), T, E, k, _ptr(idx), _ptr(w), _ptr(w64)),
           "topk_softmax")
    return idx, w, w64


def topk_softmax_grouped(logits, k, n_groups, topk_groups):
    """Group-limited top-k: keep the best topk_groups of n_groups consecutive
    expert groups (scored by their largest logit), then top-k inside them."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    w64 = np.empty((T, k), np.float64)
    _check(_load().oracle_topk_softmax_grouped(_ptr(logits), T, E, k, n_groups, topk_groups,
                                               _ptr(idx), _ptr(w), _ptr(w64)),
           "topk_softmax_grouped")
    return idx, w, w64


def route_indices(topk_idx, topk_w, E):
    """Routing map, counts, offsets, group_list, sorted_indices, slot_pos and
    permuted_probs from top-k choices (-1 = empty slot)."""
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    w = None if topk_w is None else _c(topk_w, np.float32)
    out = {
        "routing_map": np.empty((T, E), np.uint8),
        "counts": np.empty(E, np.int32),
        "offsets": np.empty(E + 1, np.int32),
        "group_list": np.empty(E, np.int32),
        "sorted_indices": np.empty(T * k, np.int32),
        "slot_pos": np.empty((T, k), np.int32),
        "permuted_probs": None if w is None else np.empty(T * k, np.float32),
    }
    _check(_load().oracle_route_indices(
        _ptr(topk_idx), _ptr(w), T, E, k, _ptr(out["routing_map"]), _ptr(out["counts"]),
        _ptr(out["offsets"]), _ptr(out["group_list"]), _ptr(out["sorted_indices"]),
        _ptr(out["slot_pos"]), _ptr(out["permuted_probs"])), "route_indices")
    return out


def e4m3_from_float(v):
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    _check(_load().oracle_e4m3_from_float(_ptr(v), v.size, _ptr(out)), "e4m3_from_float")
    return out


def quantize_fp8(x, block=128):
    """Per-token, per-block e4m3 quantization of bf16 rows (see oracle.h)."""
    x = _c(x, np.uint16)
    T, H = x.shape
    q = np.empty((T, H), np.uint8)
    sc = np.empty((T, H // block), np.float32)
    _check(_load().oracle_quantize_fp8(_ptr(x), T, H, block, _ptr(q), _ptr(sc)), "quantize_fp8")
    return q, sc


def dequantize_fp8(q, scales, block=128):
    q = _c(q, np.uint8)
    sc = _c(scales, np.float32)
    N, H = q.shape
    out = np.empty((N, H), np.uint16)
    _check(_load().oracle_dequantize_fp8(_ptr(q), _ptr(sc), N, H, block, _ptr(out)),
           "dequantize_fp8")
    return out


def expert_capacity(tokens, top_k, num_experts, capacity_factor):
    c = _load().oracle_expert_capacity(int(tokens), int(top_k), int(num_experts),
                                       float(capacity_factor))
    _check(0 if c >= 0 else -1, "expert_capacity")
    return int(c)


def route_layout(topk_idx, topk_w, E, capacity=0, pad=False, alignment=1, max_rows=None):
    """Capacity-bounded / padded / aligned routing layout (see oracle.h)."""
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    if max_rows is None:
        max_rows = E * capacity if pad else T * k + E * (alignment - 1)
    w = None if topk_w is None else _c(topk_w, np.float32)
    out = {
        "counts": np.empty(E, np.int32), "offsets": np.empty(E + 1, np.int32),
        "group_list": np.empty(E, np.int32), "sorted_indices": np.empty(max_rows, np.int32),
        "slot_pos": np.empty((T, k), np.int32),
        "permuted_probs": None if w is None else np.empty(max_rows, np.float32),
    }
    _check(_load().oracle_route_layout(
        _ptr(topk_idx), _ptr(w), T, E, k, int(capacity), int(bool(pad)), int(alignment),
        int(max_rows), _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["group_list"]),
        _ptr(out["sorted_indices"]), _ptr(out["slot_pos"]), _ptr(out["permuted_probs"])),
        "route_layout")
    return out


def route(logits, k):
    """Full routing from logits: top-k, softmax, then route_indices."""
    idx, w, w64 = topk_softmax(logits, k)
    out = route_indices(idx, w, logits.shape[1])
    out.update(topk_idx=idx, topk_w=w, topk_w_f64=w64)
    return out


def permute(x, sorted_indices, n_rows=None):
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint8:
        _dtype_code(x)
    T, H = x.shape
    si = _c(sorted_indices, np.int32)
    n = si.size if n_rows is None else int(n_rows)
    out = np.zeros((n, H), x.dtype)
    _check(_load().oracle_permute(_ptr(x), x.itemsize, T, H, _ptr(si), n, _ptr(out)), "permute")
    return out


def chunk_idxs(R, L, inverse=False):
    idxs = np.empty(R * L, np.int32)
    _check(_load().oracle_chunk_idxs(R, L, int(bool(inverse)), _ptr(idxs)), "chunk_idxs")
    return idxs


def sort_chunks(x, split_sizes, sorted_idxs):
    x = np.ascontiguousarray(x)
    N = x.shape[0]
    row_bytes = x.strides[0] if x.ndim > 1 else x.itemsize
    ss = _c(split_sizes, np.int32)
    si = _c(sorted_idxs, np.int32)
    out = np.zeros_like(x)
    _check(_load().oracle_sort_chunks(_ptr(x), row_bytes, N, _ptr(ss), _ptr(si), ss.size,
                                      _ptr(out)), "sort_chunks")
    return out


def combine(y, slot_pos, topk_w, T=None):
    """out[t] = sum_j topk_w[t,j] * y[slot_pos[t,j]] (double, slot order)."""
    y = np.ascontiguousarray(y)
    code = _dtype_code(y)
    sp = _c(slot_pos, np.int32)
    T_, k = sp.shape
    H = y.shape[1]
    w = None if topk_w is None else _c(topk_w, np.float32)
    out = np.empty((T_, H), y.dtype)
    out64 = np.empty((T_, H), np.float64)
    _check(_load().oracle_combine(_ptr(y), code, T_, H, k, _ptr(sp), _ptr(w), _ptr(out),
                                  _ptr(out64)), "combine")
    return out, out64


def unpermute(y, sorted_indices, probs, T, n_valid):
    """Scatter-add statement of the combine (double, ascending row order)."""
    y = np.ascontiguousarray(y)
    code = _dtype_code(y)
    H = y.shape[1]
    si = _c(sorted_indices, np.int32)
    pr = None if probs is None else _c(probs, np.float32)
    out = np.empty((T, H), y.dtype)
    out64 = np.empty((T, H), np.float64)
    _check(_load().oracle_unpermute(_ptr(y), code, T, H, _ptr(si), _ptr(pr), int(n_valid),
                                    _ptr(out), _ptr(out64)), "unpermute")
    return out, out64


def combine_backward(grad_out, y, slot_pos, topk_w, grad_y_init=None):
    grad_out = np.ascontiguousarray(grad_out)
    y = np.ascontiguousarray(y)
    code = _dtype_code(y)
    assert grad_out.dtype == y.dtype
    sp = _c(slot_pos, np.int32)
    T, k = sp.shape
    H = y.shape[1]
    w = None if topk_w is None else _c(topk_w, np.float32)
    grad_y = np.zeros_like(y) if grad_y_init is None else np.array(grad_y_init, copy=True)
    gp = np.empty((T, k), np.float32)
    gp64 = np.empty((T, k), np.float64)
    _check(_load().oracle_combine_backward(_ptr(grad_out), _ptr(y), code, T, H, k, _ptr(sp),
                                           _ptr(w), _ptr(grad_y), _ptr(gp), _ptr(gp64)),
           "combine_backward")
    return grad_y, gp, gp64


def route_backward(topk_idx, topk_w, grad_probs, E):
    """grad_logits [T,E] float32 of the k-softmax router (zero off the chosen
    experts)."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    w = _c(topk_w, np.float32)
    g = _c(grad_probs, np.float32)
    out = np.empty((T, E), np.float32)
    _check(_load().oracle_route_backward(_ptr(idx), _ptr(w), _ptr(g), T, E, k, _ptr(out)),
           "route_backward")
    return out


def expert_scale(x_perm, offsets, scale):
    x_perm = np.ascontiguousarray(x_perm)
    code = _dtype_code(x_perm)
    off = _c(offsets, np.int32)
    sc = _c(scale, np.float32)
    E = sc.size
    y = np.zeros_like(x_perm)
    _check(_load().oracle_expert_scale(_ptr(x_perm), code, x_perm.shape[1], E, _ptr(off),
                                       _ptr(sc), _ptr(y)), "expert_scale")
    return y


def grouped_swiglu(x, w_up, w_down, offsets, rows=None, save=False):
    """Per-expert GMM1 -> silu(gate)*up -> GMM2 on bf16 bit patterns.
    rows: optional list of row ids to compute (others are left zero).
    save: also return the bf16 gate_up [N,2I] and hidden [N,I]."""
    x = _c(x, np.uint16)
    w_up = _c(w_up, np.uint16)
    w_down = _c(w_down, np.uint16)
    off = _c(offsets, np.int32)
    E, H, I2 = w_up.shape
    I = I2 // 2
    y = np.zeros_like(x)
    y64 = np.zeros(x.shape, np.float64)
    gu = np.zeros((x.shape[0], 2 * I), np.uint16) if save else None
    hid = np.zeros((x.shape[0], I), np.uint16) if save else None
    r = None if rows is None else _c(rows, np.int64)
    n = 0 if r is None else r.size
    _check(_load().oracle_grouped_swiglu(_ptr(x), _ptr(w_up), _ptr(w_down), _ptr(off), E, H, I,
                                         _ptr(r), n, _ptr(y), _ptr(y64), _ptr(gu), _ptr(hid)),
           "grouped_swiglu")
    return (y, y64, gu, hid) if save else (y, y64)


def swiglu_dgrad(dy, w_up, w_down, offsets, gate_up, rows=None):
    """(dgate_up bf16 [N,2I], dgate_up f64, dx bf16 [N,H], dx f64) of the
    grouped SwiGLU backward; rows as in grouped_swiglu."""
    dy = _c(dy, np.uint16)
    w_up = _c(w_up, np.uint16)
    w_down = _c(w_down, np.uint16)
    off = _c(offsets, np.int32)
    gu = _c(gate_up, np.uint16)
    E, H, I2 = w_up.shape
    I = I2 // 2
    N = dy.shape[0]
    dgu = np.zeros((N, 2 * I), np.uint16)
    dgu64 = np.zeros((N, 2 * I), np.float64)
    dx = np.zeros((N, H), np.uint16)
    dx64 = np.zeros((N, H), np.float64)
    r = None if rows is None else _c(rows, np.int64)
    n = 0 if r is None else r.size
    _check(_load().oracle_swiglu_dgrad(_ptr(dy), _ptr(w_up), _ptr(w_down), _ptr(off), _ptr(gu),
                                       E, H, I, _ptr(r), n, _ptr(dgu), _ptr(dgu64), _ptr(dx),
                                       _ptr(dx64)), "swiglu_dgrad")
    return dgu, dgu64, dx, dx64


def swiglu_wgrad_at(which, coords, offsets, H, I, x=None, hidden=None, dy=None, dgate_up=None):
    """Double weight gradients at coords [n,3] = (e, a, b): which 'up' gives
    dW_up[e][h][c], 'down' gives dW_down[e][i][h]."""
    off = _c(offsets, np.int32)
    E = off.size - 1
    co = _c(coords, np.int64).reshape(-1, 3)
    out = np.zeros(co.shape[0], np.float64)
    # keep the converted arrays referenced for the duration of the call
    xs, hs, ds, gs = (None if a is None else _c(a, np.uint16) for a in (x, hidden, dy, dgate_up))
    _check(_load().oracle_swiglu_wgrad_at(
        _ptr(xs), _ptr(hs), _ptr(ds), _ptr(gs), _ptr(off), E, H, I, {"up": 0, "down": 1}[which],
        _ptr(co), co.shape[0], _ptr(out)), "swiglu_wgrad_at")
    return out
