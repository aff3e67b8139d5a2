"""Seeded synthetic inputs for the MoE dispatch/combine path.

This module is the ONLY code shared by the CPU oracle's tests and the CUDA
path's tests and benchmark.  It draws random numbers and lays out arrays; it
holds none of the path's arithmetic (no top-k, no softmax, no ranking, no
gather or reduction).  Everything is numpy with a PCG64 generator seeded per
workload, drawn in a fixed order, so both sides see identical bytes.

Workloads (shapes of the MoE pages' examples; synthetic values, no dataset):
  tiny    T=256,   H=128,  E=8,   k=2  fp32 everything
  mid     T=8192,  H=4096, E=64,  k=2  bf16 activations, fp32 router
  skewed  T=16384, H=7168, E=256, k=8  bf16, Zipf-biased router (DeepSeek-shaped)
  vep8    T=8192,  H=4096, E=64,  k=4  bf16, 8 virtual ranks x 8 local experts
  layer   T=4096,  H=2048, E=64,  k=6, I=1408 bf16 weights for a full MoE layer
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    dtype: str                 # activation dtype: "f32" or "bf16"
    I: int = 0                 # expert intermediate size (layer only)
    zipf_s: float = 0.0        # >0: add 2*log Zipf(s) bias over a seeded expert permutation
    ranks: int = 0             # virtual expert-parallel ranks (vep8 only)
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def N(self) -> int:
        return self.T * self.k


WORKLOADS = {
    "tiny": Workload("tiny", 256, 128, 8, 2, "f32",
                     note="x~N(0,1), W~N(0,1/H); stand-in expert x*(e+1)/8"),
    "mid": Workload("mid", 8192, 4096, 64, 2, "bf16",
                    note="x~N(0,1), W~N(0,1/H): near-uniform routing"),
    "skewed": Workload("skewed", 16384, 7168, 256, 8, "bf16", zipf_s=1.1,
                       note="x~N(0,1), W~N(0,1/H) plus 2*log-Zipf(1.1) expert bias"),
    "vep8": Workload("vep8", 8192, 4096, 64, 4, "bf16", ranks=8,
                     note="8 virtual ranks x 8 local experts, 1024 source tokens each"),
    "layer": Workload("layer", 4096, 2048, 64, 6, "bf16", I=1408,
                      note="expert weights ~N(0, 0.02^2)"),
}


# ------------------------------------------------------------------ bf16 bits

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def as_activation(a32: np.ndarray, dtype: str) -> np.ndarray:
    return np.ascontiguousarray(a32, np.float32) if dtype == "f32" else f32_to_bf16_bits(a32)


def activation_to_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


# ----------------------------------------------------------------- generators

def _normal(rng, shape, std=1.0):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def router_logits(x_act: np.ndarray, W: np.ndarray, bias: np.ndarray | None = None,
                  row_block: int = 2048) -> np.ndarray:
    """Router projection x @ W^T (+ bias) in double, rounded once to float32.

    This is input synthesis: the path starts from the logits, and computing
    them here, once, gives the oracle and the GPU identical bytes."""
    T = x_act.shape[0]
    W64 = W.astype(np.float64)
    out = np.empty((T, W.shape[0]), np.float32)
    for r0 in range(0, T, row_block):
        xb = activation_to_f64(x_act[r0:r0 + row_block])
        lg = xb @ W64.T
        if bias is not None:
            lg += bias[None, :]
        out[r0:r0 + row_block] = lg.astype(np.float32)
    return out


def zipf_bias(E: int, s: float, perm: np.ndarray) -> np.ndarray:
    """bias[perm[i]] = 2 * log(p_i), p_i = (i+1)^-s / sum_j (j+1)^-s."""
    ranks = np.arange(1, E + 1, dtype=np.float64)
    log_p = -s * np.log(ranks) - math.log(np.sum(ranks ** -s))
    bias = np.empty(E, np.float64)
    bias[perm] = 2.0 * log_p
    return bias


_CACHE: dict = {}


def make(name: str, *, T: int | None = None, with_grad: bool = False,
         with_weights: bool = False) -> dict:
    """Inputs of a workload, optionally truncated to its first T tokens.

    Draw order (seed = workload seed): x [T,H], W [E,H], expert permutation
    (zipf workloads), w_up [E,H,2I] and w_down [E,I,H] (layer, if
    requested), grad_out [T,H] (if requested).  Truncation draws the full-size arrays and
    slices, so a prefix of a workload is the same bytes at any size."""
    wl = WORKLOADS[name]
    key = (name, with_grad, with_weights)
    if key not in _CACHE:
        rng = np.random.default_rng(wl.seed)
        x32 = _normal(rng, (wl.T, wl.H))
        W = _normal(rng, (wl.E, wl.H), std=1.0 / math.sqrt(wl.H))
        bias = None
        perm = None
        if wl.zipf_s > 0:
            perm = rng.permutation(wl.E)
            bias = zipf_bias(wl.E, wl.zipf_s, perm)
        x = as_activation(x32, wl.dtype)
        del x32
        d = {"x": x, "W": W, "bias": bias, "expert_perm": perm,
             "logits": router_logits(x, W, bias)}
        if with_weights and wl.I:
            d["w_up"] = f32_to_bf16_bits(_normal(rng, (wl.E, wl.H, 2 * wl.I), std=0.02))
            d["w_down"] = f32_to_bf16_bits(_normal(rng, (wl.E, wl.I, wl.H), std=0.02))
        if with_grad:
            d["grad_out"] = as_activation(_normal(rng, (wl.T, wl.H)), wl.dtype)
        d["scale"] = stand_in_scale(wl.E)
        _CACHE.clear()  # keep at most one full-size workload resident
        _CACHE[key] = d
    d = dict(_CACHE[key])
    if T is not None and T < wl.T:
        for name_ in ("x", "logits", "grad_out"):
            if name_ in d:
                d[name_] = np.ascontiguousarray(d[name_][:T])
    d["workload"] = wl
    return d


def stand_in_scale(E: int) -> np.ndarray:
    """Stand-in expert e multiplies its rows by (e+1)/E."""
    return ((np.arange(E, dtype=np.float64) + 1.0) / E).astype(np.float32)


def random_routing(seed: int, T: int, E: int, k: int, empty_frac: float = 0.0):
    """Random distinct expert choices per token (slot order arbitrary) and
    random positive slot weights; a fraction of slots can be emptied (-1).
    Kernel-level test input: it does not come from any router."""
    rng = np.random.default_rng(seed)
    keys = rng.random((T, E))
    idx = np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)
    w = rng.uniform(0.05, 1.0, (T, k)).astype(np.float32)
    if empty_frac > 0:
        drop = rng.random((T, k)) < empty_frac
        idx[drop] = -1
    return np.ascontiguousarray(idx), np.ascontiguousarray(w)


def random_activation(seed: int, shape, dtype: str, std: float = 1.0):
    rng = np.random.default_rng(seed)
    return as_activation(_normal(rng, shape, std), dtype)


def tie_logits(seed: int, T: int, E: int) -> np.ndarray:
    """Integer-valued logits in [0, 4): many exact ties."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 4, (T, E)).astype(np.float32)
