"""Benchmark of the MoE dispatch/combine hot path on GB300.

One step = one pass of the whole path over one batch of the DeepSeek-shaped
workload (T=16384 tokens, H=7168, E=256 experts, top-8, bf16, Zipf-biased
router): moe_route (top-k + softmax + counts/offsets + expert-major indices),
moe_permute, moe_combine (the expert being the identity, so expert_out is the
permuted buffer) and moe_combine_backward.  value = routed tokens (T*k) per
second over whole steps, inputs resident in HBM.  The step's working set is
about 4.5 GB, far larger than the 129 MB L2, so no L2 flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

After the main step the default run also times, each with its own clock
record, the other workloads under the key "workloads": the full MoE layer
forward (T=4096, H=2048, E=64, k=6, I=1408: route, permute, grouped SwiGLU
on the tensor cores, combine), the virtual expert-parallel sort_chunks
(8 ranks x 8 local experts, forward and inverse) and the two stand-in
pipelines mid (T=8192, H=4096, E=64, k=2) and tiny (T=256, H=128, E=8, k=2,
fp32): route, permute, per-expert scale, combine.  --no-extra skips them.

For N > 1 launch under torchrun: every rank runs an independent replica of
the workload on its own GPU (the path has no cross-GPU exchange), timing is
bracketed by a barrier and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "permute+combine routed-tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "routed-tokens/s"
WORKLOAD = "skewed"
FALLBACK_HBM_GBS = 6800.0
def route_launches(T, E, k, grouped=False, sms=152):
    """Kernels one moe_route call launches: a single cooperative kernel when
    every token block fits on the GPU at once (up to 256 experts, k <= 8, no
    group limit, T <= sms * 128); otherwise top-k + placement, plus a scan
    kernel beyond 256 token blocks."""
    if E <= 256 and k <= 8 and not grouped and 0 < T <= sms * 128:
        return 1
    tpb = min(128, max(32, -(-T // sms))) if E <= 256 else 128
    return 2 + (1 if -(-T // tpb) > 256 else 0)


# ------------------------------------------------------------ host-side logic

def algorithmic_bytes(T, H, E, k, b):
    """Bytes each op must move: every source row read once, every
    destination row written once, plus the 4-byte index/probability arrays."""
    N = T * k
    return {
        "route": T * E * 4 + N * 4 * 5 + E * 4 * 3,
        "permute": T * H * b + N * H * b + N * 4,
        "combine": N * H * b + T * H * b + N * 8,
        "combine_backward": T * H * b + 2 * N * H * b + N * 12,
    }


def layout_bytes(T, H, k, b, kept, rows, live=None):
    """Algorithmic bytes under a capacity / padded / aligned layout: only the
    `kept` slot rows move, the pad-row fill writes the other rows of the
    expert segments (`rows` = offsets[E], the rows the segments span), and
    only the `live` tokens (at least one kept slot; default all T) need their
    x / grad_out row read.  The combine still writes every output row."""
    N = T * k
    live = T if live is None else live
    return {
        "permute": live * H * b + kept * H * b + N * 4 + (rows - kept) * H * b,
        "combine": kept * H * b + T * H * b + N * 8,
        "combine_backward": live * H * b + 2 * kept * H * b + N * 12,
    }


def fp8_bytes(T, H, k, block=128):
    """Algorithmic bytes of the FP8 dispatch stages (bf16 source rows, e4m3
    rows, float scale rows of H/block columns)."""
    N, nb = T * k, H // block
    return {
        "quantize_fp8": T * H * 2 + T * H + T * nb * 4,
        "permute_quantize_fp8": T * H * 2 + N * H + N * nb * 4 + N * 4,
        "permute": T * H + N * H + (T + N) * nb * 4 + 2 * N * 4,
        "dequantize_fp8": N * H + N * nb * 4 + N * H * 2,
    }


def job_value(units_per_rank_step: float, world: int, steps: int, max_elapsed_s: float) -> float:
    """Whole-job throughput: units every rank processed over the slowest rank's time."""
    return units_per_rank_step * world * steps / max_elapsed_s


def reduce_max(value: float, device=None) -> float:
    """Max of a float over the ranks of the default process group (or itself)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Source files that define each timed kernel (a recorded DRAM traffic figure
# stays valid only while these are unchanged).
KERNEL_SOURCES = {
    "route": ("unpermute_combine_gb300/csrc/route.cu", "unpermute_combine_gb300/csrc/common.cuh"),
    "permute": ("unpermute_combine_gb300/csrc/permute.cu", "unpermute_combine_gb300/csrc/common.cuh"),
    "combine": ("unpermute_combine_gb300/csrc/combine.cu", "unpermute_combine_gb300/csrc/common.cuh"),
    "combine_backward": ("unpermute_combine_gb300/csrc/combine.cu",
                         "unpermute_combine_gb300/csrc/common.cuh"),
    "quantize_fp8": ("unpermute_combine_gb300/csrc/fp8.cu", "unpermute_combine_gb300/csrc/common.cuh"),
    "permute_quantize_fp8": ("unpermute_combine_gb300/csrc/fp8.cu",
                             "unpermute_combine_gb300/csrc/pipeline.cuh",
                             "unpermute_combine_gb300/csrc/common.cuh"),
    "swiglu_dgrad": ("unpermute_combine_gb300/csrc/grouped_swiglu.cu",
                     "unpermute_combine_gb300/csrc/pipeline.cuh"),
    "swiglu_wgrad": ("unpermute_combine_gb300/csrc/grouped_swiglu.cu",
                     "unpermute_combine_gb300/csrc/pipeline.cuh"),
    "route_backward": ("unpermute_combine_gb300/csrc/route_bwd.cu",
                       "unpermute_combine_gb300/csrc/common.cuh"),
    "dequantize_fp8": ("unpermute_combine_gb300/csrc/fp8.cu",
                       "unpermute_combine_gb300/csrc/common.cuh"),
}


def source_digest(*files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str, digest: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source (the summary records the source digest)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(rf"^{re.escape(kernel_key)}\s+digest=(\w+)\s+bytes_per_launch=([0-9.eE+]+)",
                  text, re.M)
    if not m or m.group(1) != digest:
        return None
    return float(m.group(2))


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (getattr(self, "out", "") or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm

def layer_flops_bytes(N, H, E, I):
    """Grouped SwiGLU: 2*N*H*2I (GMM1) + 2*N*I*H (GMM2) flops; bytes = both
    weight sets once, x once, hidden written and read once, y once."""
    flops = 6 * N * H * I
    byts = E * (H * 2 * I + I * H) * 2 + N * H * 2 + 2 * N * I * 2 + N * H * 2
    return flops, byts


def train_flops_bytes(N, T, H, E, I, k):
    """The backward GEMMs of the grouped SwiGLU, each 6*N*H*I flops:
    dgrad  = dy @ w_down^T (2NHI) + dgate_up @ w_up^T (4NHI); bytes: dy,
             w_down, gate_up read, dgate_up written and read, w_up, dx;
    wgrad  = hidden^T dy (2NHI) + x^T dgate_up (4NHI); bytes: hidden, dy, x,
             dgate_up read, both fp32 weight gradients written."""
    flops = 6 * N * H * I
    dgrad = (N * H * 2 + E * I * H * 2 + N * 2 * I * 2 * 3 + E * H * 2 * I * 2 + N * H * 2)
    wgrad = (N * I * 2 + N * H * 2 * 2 + N * 2 * I * 2 + E * (I * H + H * 2 * I) * 4)
    return flops, dgrad, wgrad


def parse_layout(spec):
    """'cf=1.25,pad' or 'align=128' -> dict (empty: the plain layout)."""
    out = {}
    for part in (spec or "").split(","):
        part = part.strip()
        if not part:
            continue
        if part == "pad":
            out["pad"] = True
        elif part.startswith("cf="):
            out["cf"] = float(part[3:])
        elif part.startswith("align="):
            out["align"] = int(part[6:])
        else:
            raise ValueError(f"unknown layout option {part!r}")
    if out.get("pad") and not out.get("cf"):
        raise ValueError("pad needs a capacity factor (cf=...)")
    return out


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1700.0, 1900.0, "fallback"


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import unpermute_combine_gb300 as moe
    import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    layer = args.workload == "layer"
    train = layer and bool(args.train)
    d = wl.make(args.workload, with_grad=not layer or train, with_weights=layer, T=args.tokens)
    W = d["workload"]
    T, H, E, k, b = d["x"].shape[0], W.H, W.E, W.k, 2
    N = T * k

    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    h_logits = torch.from_numpy(d["logits"]).pin_memory()
    h_x = bf(d["x"]).pin_memory()
    has_grad = not layer or train
    h_g = bf(d["grad_out"]).pin_memory() if has_grad else None
    logits, x = h_logits.to(dev), h_x.to(dev)
    g = h_g.to(dev) if has_grad else None

    groups = tuple(int(v) for v in args.route_groups.split(":")) if args.route_groups else None
    lay = parse_layout(args.layout)
    cap = moe.moe_expert_capacity(T, k, E, lay["cf"]) if lay.get("cf") else 0
    rows = (moe.moe_route_layout_rows(T, E, k, cap, lay.get("pad", False), lay.get("align", 1))
            if lay else N)
    stream = torch.cuda.Stream(device=dev)
    gp = None
    with torch.cuda.stream(stream):
        r = moe.moe_route(logits, k)
        rl = (moe.moe_route_layout(r.topk_idx, r.topk_w, E, capacity=cap, pad=lay.get("pad", False),
                                   alignment=lay.get("align", 1), max_rows=rows, stream=stream)
              if lay else None)
        xp = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
        fp8 = bool(args.fp8 or args.fp8_split)
        fp8_fused = fp8 and not args.fp8_split and H * 2 <= 16384
        # --fp8-gemm: the layer forward feeds the e4m3 slot rows straight to GMM1
        fp8_gemm = bool(args.fp8_gemm) and fp8_fused and layer and not train and not lay
        if fp8:
            fp8_tok = (torch.empty((T, H), dtype=torch.float8_e4m3fn, device=dev),
                       torch.empty((T, H // 128), dtype=torch.float32, device=dev))
            fp8_rows = (torch.empty((rows, H), dtype=torch.float8_e4m3fn, device=dev),
                        torch.empty((rows, H // 128), dtype=torch.float32, device=dev))
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        if layer:
            # one-time weight layout (model-load step, outside the timed region)
            up_p, down_p = moe.moe_grouped_swiglu_pack(bf(d["w_up"]).to(dev),
                                                       bf(d["w_down"]).to(dev), stream=stream)
            y = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
            gs_ws = torch.empty(moe.moe_grouped_swiglu_workspace_size(rows, E, H, W.I),
                                dtype=torch.uint8, device=dev)
            if train:
                I = W.I
                w_up_d, w_down_d = bf(d["w_up"]).to(dev), bf(d["w_down"]).to(dev)
                hid = torch.empty((rows, I), dtype=torch.bfloat16, device=dev)
                gu = torch.empty((rows, 2 * I), dtype=torch.bfloat16, device=dev)
                gy = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
                gp = torch.empty((T, k), dtype=torch.float32, device=dev)
                dgu = torch.empty((rows, 2 * I), dtype=torch.bfloat16, device=dev)
                dxp = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
                dwu = torch.empty((E, H, 2 * I), dtype=torch.float32, device=dev)
                dwd = torch.empty((E, I, H), dtype=torch.float32, device=dev)
                gx = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
                gl = torch.empty((T, E), dtype=torch.float32, device=dev)
                ws_d = torch.empty(moe.MOE_STATUS_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
                ws_w = torch.empty(moe.MOE_STATUS_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
        else:
            gy = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
            gp = torch.empty((T, k), dtype=torch.float32, device=dev)
    names = (["route", "permute", "grouped_swiglu", "combine"] if layer else
             ["route", "permute", "combine", "combine_backward"])
    if train:
        names += ["combine_backward", "swiglu_dgrad", "swiglu_wgrad", "permute_backward",
                  "route_backward"]
    if fp8:
        names[1:2] = (["permute_quantize_fp8"] if fp8_gemm else
                      ["permute_quantize_fp8", "dequantize_fp8"] if fp8_fused else
                      ["quantize_fp8", "permute", "dequantize_fp8"])
    router_bwd = bool(args.router_bwd) and not layer
    if router_bwd:
        names.append("route_backward")
        with torch.cuda.stream(stream):
            gl = torch.empty((T, E), dtype=torch.float32, device=dev)

    def step(lg, xx, gg, ev=None, ob=None):
        # ob: (out, grad_probs) buffers of this step's results (default: the shared ones)
        o_out, o_gp = ob if ob is not None else (out, gp)
        n_marks = [0]

        def mark():
            if ev is not None:
                ev[n_marks[0]].record(stream)
            n_marks[0] += 1
        mark()
        if groups:
            moe.moe_route_grouped(lg, k, groups[0], groups[1], out=r, stream=stream)
        else:
            moe.moe_route(lg, k, out=r, stream=stream)
        rr = r
        if lay:
            rr = moe.moe_route_layout(r.topk_idx, r.topk_w, E, capacity=cap,
                                      pad=lay.get("pad", False), alignment=lay.get("align", 1),
                                      max_rows=rows, workspace=rl.workspace, stream=stream)
        mark()
        if fp8:
            # FP8 dispatch: quantize, move e4m3 rows and scale rows, and
            # dequantize in place of the expert's input conversion
            if fp8_fused:
                moe.moe_permute_quantize_fp8(xx, rr.slot_pos, 128, out=fp8_rows, stream=stream)
            else:
                moe.moe_quantize_fp8(xx, 128, out=fp8_tok, stream=stream)
                mark()
                moe.moe_permute_fp8(fp8_tok[0], fp8_tok[1], rr.slot_pos, out=fp8_rows,
                                    stream=stream)
            if not fp8_gemm:
                mark()
                moe.moe_dequantize_fp8(fp8_rows[0], fp8_rows[1], 128, out=xp, stream=stream)
        else:
            moe.moe_permute(xx, rr.slot_pos, out=xp, stream=stream)
        if lay:
            moe.moe_fill_pad_rows(xp, rr.offsets, rr.counts, stream=stream)
        mark()
        if train:
            # forward keeping the activations, then the whole layer backward
            moe.moe_grouped_swiglu_save(xp, up_p, down_p, rr.offsets, out=y, hidden=hid,
                                        gate_up=gu, workspace=gs_ws, stream=stream)
            mark()
            moe.moe_combine(y, rr.slot_pos, r.topk_w, out=o_out, stream=stream)
            mark()
            moe.moe_combine_backward(gg, y, rr.slot_pos, r.topk_w, grad_expert_out=gy,
                                     grad_probs=o_gp, stream=stream)
            if lay:     # pad rows of the expert-output gradient must be zero for the GEMMs
                moe.moe_fill_pad_rows(gy, rr.offsets, rr.counts, stream=stream)
            mark()
            moe.moe_grouped_swiglu_dgrad(gy, w_up_d, w_down_d, rr.offsets, gu, dgate_up=dgu,
                                         dx=dxp, workspace=ws_d, stream=stream)
            mark()
            moe.moe_grouped_swiglu_wgrad(xp, hid, gy, dgu, rr.offsets, dw_up=dwu, dw_down=dwd,
                                         workspace=ws_w, stream=stream)
            mark()
            moe.moe_combine(dxp, rr.slot_pos, None, out=gx, stream=stream)   # permute backward
            mark()
            moe.moe_route_backward(r.topk_idx, r.topk_w, o_gp, E, out=gl, stream=stream)
        elif layer:
            if fp8_gemm:
                moe.moe_grouped_swiglu_fp8(fp8_rows[0], fp8_rows[1], up_p, down_p, rr.offsets,
                                           out=y, workspace=gs_ws, stream=stream)
            else:
                moe.moe_grouped_swiglu(xp, up_p, down_p, rr.offsets, out=y, workspace=gs_ws,
                                       stream=stream)
            mark()
            moe.moe_combine(y, rr.slot_pos, r.topk_w, out=o_out, stream=stream)
        else:
            moe.moe_combine(xp, rr.slot_pos, r.topk_w, out=o_out, stream=stream)
            mark()
            moe.moe_combine_backward(gg, xp, rr.slot_pos, r.topk_w, grad_expert_out=gy,
                                     grad_probs=o_gp, stream=stream)
            if router_bwd:
                mark()
                moe.moe_route_backward(r.topk_idx, r.topk_w, o_gp, E, out=gl, stream=stream)
        mark()

    import torch.distributed as dist
    dist_on = dist.is_available() and dist.is_initialized()

    def barrier():
        torch.cuda.synchronize(dev)
        if dist_on:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step(logits, x, g)
    barrier()

    # -------- device-resident timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        barrier()
        t_start.record(stream)
        for i in range(args.steps):
            step(logits, x, g, evs[i])
        t_end.record(stream)
        barrier()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    per = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)) / 1e3
           for j, n in enumerate(names)}
    max_elapsed = reduce_max(elapsed, dev)
    if layer:
        assert moe.moe_workspace_status(gs_ws, stream) == 0, "grouped SwiGLU pipeline timed out"
    if train:
        assert moe.moe_workspace_status(ws_d, stream) == 0, "SwiGLU dgrad pipeline timed out"
        assert moe.moe_workspace_status(ws_w, stream) == 0, "SwiGLU wgrad pipeline timed out"
    if lay:
        assert moe.moe_workspace_status(rl.workspace, stream) == 0, "layout ran out of rows"

    # -------- end to end through the public API from pinned host buffers:
    # every step copies its inputs host -> device and its results device ->
    # host inside the timed region; steps are pipelined over two buffer sets
    # (inputs on one copy stream, the step on its own stream, results on a
    # third), so the copies of step i+1 and i-1 overlap the kernels of step i
    n_sets = 2
    h_out = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(n_sets)]
    h_gp = ([torch.empty((T, k), dtype=torch.float32).pin_memory() for _ in range(n_sets)]
            if has_grad else [None] * n_sets)
    h2d = h_logits.numel() * 4 + h_x.numel() * 2 + (h_g.numel() * 2 if has_grad else 0)
    d2h = h_out[0].numel() * 2 + (h_gp[0].numel() * 4 if has_grad else 0)
    e2e_steps = 0 if args.no_e2e else max(1, min(args.steps, 50))
    e2e_elapsed = float("nan")
    if e2e_steps:
        with torch.cuda.stream(stream):
            d_in = [(torch.empty_like(logits), torch.empty_like(x),
                     torch.empty_like(g) if has_grad else None) for _ in range(n_sets)]
            d_out = [(torch.empty_like(out), torch.empty_like(gp) if has_grad else None)
                     for _ in range(n_sets)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(n_sets)]
        ev_comp = [torch.cuda.Event() for _ in range(n_sets)]
        ev_out = [torch.cuda.Event() for _ in range(n_sets)]

        def e2e_step(i):
            b = i % n_sets
            s_in.wait_event(ev_comp[b])              # step i-2 has read this input set
            with torch.cuda.stream(s_in):
                for dst, src in zip(d_in[b], (h_logits, h_x, h_g)):
                    if dst is not None:
                        dst.copy_(src, non_blocking=True)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])             # step i-2's results have left this set
            step(*d_in[b], ob=d_out[b])
            ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                h_out[b].copy_(d_out[b][0], non_blocking=True)
                if has_grad:
                    h_gp[b].copy_(d_out[b][1], non_blocking=True)
            ev_out[b].record(s_out)

        for i in range(2):
            e2e_step(i)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(e2e_steps):
            e2e_step(i)
        e1.record(s_out)
        barrier()
        e2e_elapsed = reduce_max(e0.elapsed_time(e1) / 1e3, dev)

    if rank != 0:
        return None

    value = job_value(N, world, args.steps, max_elapsed)
    e2e_value = job_value(N, world, e2e_steps, e2e_elapsed) if e2e_steps else None
    peak, peak_kind = measured_peak()
    alg = algorithmic_bytes(T, H, E, k, b)
    if layer:
        fl, by = layer_flops_bytes(N, H, E, W.I)
        alg["grouped_swiglu"] = by
    if train:
        _, bd, bw = train_flops_bytes(N, T, H, E, W.I, k)
        alg["swiglu_dgrad"], alg["swiglu_wgrad"] = bd, bw
        alg["permute_backward"] = alg["combine"] - 4 * N          # unweighted combine
        alg["route_backward"] = T * E * 4 + T * k * 12
    if fp8:
        alg.update(fp8_bytes(T, H, k))
        if fp8_gemm:     # GMM1 reads e4m3 codes and their scales instead of bf16 rows
            alg["grouped_swiglu"] += N * H + N * (H // 128) * 4 - N * H * 2
    if router_bwd:
        alg["route_backward"] = T * E * 4 + T * k * 12
    if lay:
        kept = int(rl.counts.sum().item())
        segs = int(rl.offsets[-1].item())
        live = int((rl.slot_pos >= 0).any(dim=1).sum().item())
        lb = layout_bytes(T, H, k, b, kept, segs, live)
        alg.update({n: v for n, v in lb.items() if n in names})
    kern = {}
    for n in names:
        gbs = alg[n] / per[n] / 1e9
        kern[n] = {"us": round(per[n] * 1e6, 2), "alg_bytes": alg[n], "GB_s": round(gbs, 1),
                   "frac": round(gbs / peak, 4)}
    dominant = max(names, key=lambda n: per[n])
    pc_time = sum(per[n] for n in names if n in ("quantize_fp8", "permute", "dequantize_fp8",
                                                  "permute_quantize_fp8", "combine"))
    if layer:
        t_sus, t_burst, t_kind = measured_tensor_peak()
        gemms = ["grouped_swiglu"] + (["swiglu_dgrad", "swiglu_wgrad"] if train else [])
        for gname in gemms:                       # each is 6*N*H*I flops
            tf_g = fl / per[gname] / 1e12
            kern[gname].update({"TFLOP_s": round(tf_g, 1), "flops": fl,
                                "frac_tensor_sustained": round(tf_g / t_sus, 4),
                                "frac_tensor_burst": round(tf_g / t_burst, 4)})
        top = max(gemms, key=lambda n_: per[n_])
        tf = fl / per[top] / 1e12
        roof = {"bound": "tensor", "kernel": top, "achieved": round(tf, 1),
                "peak": t_sus, "unit": "TFLOP/s", "frac": round(tf / t_sus, 4),
                "peak_source": f"{t_kind} bf16_tflops_sustained (burst {t_burst})",
                "hbm_frac": kern[top]["frac"], "traffic": None}
        workload = (f"layer: T={T} H={H} E={E} k={k} I={W.I} bf16, full MoE layer forward "
                    "(route, permute, grouped SwiGLU on tcgen05, combine)")
        step_desc = "moe_route + moe_permute + moe_grouped_swiglu + moe_combine"
        if train:
            workload = (f"layer: T={T} H={H} E={E} k={k} I={W.I} bf16, MoE layer training step "
                        "(forward keeping activations, then the whole backward)")
            step_desc = ("moe_route + moe_permute + moe_grouped_swiglu_save + moe_combine + "
                         "moe_combine_backward + moe_grouped_swiglu_dgrad + "
                         "moe_grouped_swiglu_wgrad + moe_combine(unweighted: permute backward) + "
                         "moe_route_backward")
    else:
        ach = alg[dominant] / per[dominant] / 1e9
        roof = {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1),
                "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                "peak_source": f"{peak_kind} hbm_gbs",
                "traffic": recorded_traffic(dominant, source_digest(*KERNEL_SOURCES[dominant]))}
        workload = (f"skewed: T={T} H={H} E={E} k={k} bf16, router logits fp32 with "
                    "2*log-Zipf(1.1) expert bias")
        step_desc = "moe_route + moe_permute + moe_combine + moe_combine_backward"
        if groups:
            step_desc = step_desc.replace("moe_route", f"moe_route_grouped({groups[0]} groups, "
                                                       f"{groups[1]} kept)", 1)
    if router_bwd:
        step_desc += " + moe_route_backward"
    if fp8_gemm:
        step_desc = step_desc.replace(
            "moe_permute + moe_grouped_swiglu",
            "moe_permute_quantize_fp8(block 128: bf16 rows -> e4m3 rows + scale rows in the "
            "slots) + moe_grouped_swiglu_fp8(GMM1 from the e4m3 rows)", 1)
        workload = workload.replace("full MoE layer forward", "MoE layer forward with FP8 dispatch")
    elif fp8:
        step_desc = step_desc.replace(
            "moe_permute", ("moe_permute_quantize_fp8(block 128: bf16 rows -> e4m3 rows + scale "
                            "rows in the slots) + moe_dequantize_fp8") if fp8_fused else
            ("moe_quantize_fp8(block 128) + moe_permute_fp8(e4m3 rows + scale rows) + "
             "moe_dequantize_fp8"), 1)
    if lay:
        step_desc = step_desc.replace(" + moe_permute", f" + moe_route_layout(capacity={cap}, "
                                      f"pad={lay.get('pad', False)}, alignment="
                                      f"{lay.get('align', 1)}, rows={rows}) + moe_permute + "
                                      "moe_fill_pad_rows", 1)
    launches = route_launches(T, E, k, bool(groups)) + (1 + 3 + 1 if layer else 3)   # grouped SwiGLU: reset + 2 GEMMs
    if train:
        launches += 1 + 3 + 3 + 1 + 1     # combine bwd, dgrad, wgrad (reset + 2 each), permute bwd, route bwd
        if lay:
            launches += 1                 # pad rows of the expert-output gradient
    if fp8 and not fp8_gemm:
        launches += 1 if fp8_fused else 2   # (quantize,) dequantize
    if router_bwd:
        launches += 1
    if lay:
        launches += 3                     # layout check + scatter, pad-row fill
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; DeepSeek-shaped shapes, no dataset or weights)",
        "config": {"workload": workload, "T": T, "H": H, "E": E, "k": k,
                   "routed_tokens_per_step": N, "step": step_desc,
                   "l2": "no flush: step working set is several GB >> 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "kernels": kern,
        "permute_combine_routed_tokens_per_s": N / pc_time,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "path": "pinned host inputs -> device -> step -> outputs to host, steps "
                        "pipelined over two buffer sets on three streams"},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and not layer:
        line["cpu_baseline"] = cpu_baseline(args.cpu_tokens)
    elif not args.no_cpu_baseline and layer and not train:
        line["cpu_baseline"] = cpu_baseline_layer(args.cpu_layer_tokens)
    return line


# ------------------------------------------------------------ sort_chunks

def vep_bytes(N, H, b, C):
    """sort_chunks, per direction: every row read once and written once, plus
    the split sizes and chunk order (4 bytes each) of every chunk."""
    return 2 * N * H * b + 8 * C


def run_vep8(args, rank, world, local_rank):
    """The rank-major <-> expert-major reorder of an 8-rank x 8-local-expert
    virtual expert-parallel layout: for each virtual rank, moe_sort_chunks
    forward (rank-major receive buffer -> expert-major) and back."""
    import numpy as np
    import torch

    import unpermute_combine_gb300 as moe
    import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    d = wl.make("vep8")
    W = d["workload"]
    R = L = W.ranks
    T, H, k = W.T, W.H, W.k
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    stream = torch.cuda.Stream(device=dev)
    # set-up (untimed): route on the GPU, then each virtual rank's split matrix
    # M_r[src, le] (tokens of source slice src routed to expert r*L + le) and its
    # rank-major receive buffer (for src, then le: those tokens' rows, ascending)
    with torch.cuda.stream(stream):
        r = moe.moe_route(torch.from_numpy(d["logits"]).to(dev), k, stream=stream)
    stream.synchronize()
    idx = r.topk_idx.cpu().numpy()
    x = bf(d["x"]).to(dev)
    per = T // R
    fwd_idx = torch.tensor(moe.moe_chunk_idxs(R, L, False), dtype=torch.int32, device=dev)
    inv_idx = torch.tensor(moe.moe_chunk_idxs(R, L, True), dtype=torch.int32, device=dev)
    ranks = []
    for rr in range(R):
        M = np.zeros((R, L), np.int32)
        rows = []
        for src in range(R):
            toks = np.arange(src * per, (src + 1) * per)
            for le in range(L):
                sel = toks[(idx[toks] == rr * L + le).any(axis=1)]
                M[src, le] = sel.size
                rows.append(sel)
        order = torch.from_numpy(np.concatenate(rows).astype(np.int64)).to(dev)
        buf = x.index_select(0, order)
        ranks.append(dict(buf=buf, em=torch.empty_like(buf), back=torch.empty_like(buf),
                          sp=torch.from_numpy(M.ravel().copy()).to(dev),
                          spt=torch.from_numpy(M.T.ravel().copy()).to(dev),
                          ws_f=torch.empty(moe.moe_sort_chunks_workspace_size(R * L),
                                           dtype=torch.uint8, device=dev),
                          ws_b=torch.empty(moe.moe_sort_chunks_workspace_size(R * L),
                                           dtype=torch.uint8, device=dev)))
    N = sum(int(q["buf"].shape[0]) for q in ranks)
    names = ["sort_chunks", "sort_chunks_inverse"]
    # the virtual ranks' reorders are independent problems: each direction
    # forks them over S streams and joins back onto `stream`, so one call's
    # ramp-up overlaps another's tail
    S = max(1, args.vep_streams)
    side = [torch.cuda.Stream(device=dev) for _ in range(S)] if S > 1 else [stream]

    def direction(srcs, dsts, splits, ws_key, idx):
        if S > 1:
            for st in side:
                st.wait_stream(stream)
        for i, (q, a, b) in enumerate(zip(ranks, srcs, dsts)):
            moe.moe_sort_chunks(a, q[splits], idx, out=b, workspace=q[ws_key],
                                stream=side[i % S])
        if S > 1:
            for st in side:
                stream.wait_stream(st)

    def fwd(bufs=None, ems=None):
        direction(bufs or [q["buf"] for q in ranks], ems or [q["em"] for q in ranks], "sp",
                  "ws_f", fwd_idx)

    def inv(ems=None):
        direction(ems or [q["em"] for q in ranks], [q["back"] for q in ranks], "spt", "ws_b",
                  inv_idx)

    # each direction of the timed step is one CUDA graph of its 8 launches
    for _ in range(2):
        fwd()
        inv()
    stream.synchronize()
    graphs = []
    for fn in (fwd, inv):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs.append(g)

    def step(ev=None, bufs=None, ems=None):
        if ev is not None:
            ev[0].record(stream)
        if bufs is None:
            with torch.cuda.stream(stream):
                graphs[0].replay()
        else:
            fwd(bufs, ems)
        if ev is not None:
            ev[1].record(stream)
        if bufs is None:
            with torch.cuda.stream(stream):
                graphs[1].replay()
        else:
            inv(ems)
        if ev is not None:
            ev[2].record(stream)

    import torch.distributed as dist
    dist_on = dist.is_available() and dist.is_initialized()

    def barrier():
        torch.cuda.synchronize(dev)
        if dist_on:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        barrier()
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        barrier()
    elapsed = t0.elapsed_time(t1) / 1e3
    per_t = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
             / 1e3 for j, n in enumerate(names)}
    for q in ranks:
        assert moe.moe_workspace_status(q["ws_f"], stream) == 0, "sort_chunks plan rejected"
        assert moe.moe_workspace_status(q["ws_b"], stream) == 0, "sort_chunks plan rejected"
    max_elapsed = reduce_max(elapsed, dev)

    # end to end: the rank-major buffers from pinned host memory, the step,
    # the expert-major buffers back to the host, pipelined over two buffer
    # sets on three streams like the main step's end-to-end leg
    n_sets = 2
    h_in = [q["buf"].cpu().pin_memory() for q in ranks]
    h_out = [[torch.empty_like(q["buf"], device="cpu").pin_memory() for q in ranks]
             for _ in range(n_sets)]
    e2e_steps = 0 if args.no_e2e else max(1, min(args.steps, 50))
    e2e_value = None
    if e2e_steps:
        d_in = [[torch.empty_like(q["buf"]) for q in ranks] for _ in range(n_sets)]
        d_em = [[torch.empty_like(q["buf"]) for q in ranks] for _ in range(n_sets)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(n_sets)]
        ev_comp = [torch.cuda.Event() for _ in range(n_sets)]
        ev_out = [torch.cuda.Event() for _ in range(n_sets)]

        def e2e_step(i):
            b = i % n_sets
            s_in.wait_event(ev_comp[b])
            with torch.cuda.stream(s_in):
                for hi, di in zip(h_in, d_in[b]):
                    di.copy_(hi, non_blocking=True)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])
            step(bufs=d_in[b], ems=d_em[b])
            ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                for ho, em in zip(h_out[b], d_em[b]):
                    ho.copy_(em, non_blocking=True)
            ev_out[b].record(s_out)

        for i in range(2):
            e2e_step(i)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(e2e_steps):
            e2e_step(i)
        e1.record(s_out)
        barrier()
        e2e_value = job_value(N, world, e2e_steps, reduce_max(e0.elapsed_time(e1) / 1e3, dev))
    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    alg = vep_bytes(N, H, 2, R * L * R)
    kern = {}
    for n in names:
        gbs = alg / per_t[n] / 1e9
        kern[n] = {"us": round(per_t[n] * 1e6, 2), "alg_bytes": alg, "GB_s": round(gbs, 1),
                   "frac": round(gbs / peak, 4), "launches": R}
    dominant = max(names, key=lambda n_: per_t[n_])
    ach = alg / per_t[dominant] / 1e9
    io = sum(t.numel() * 2 for t in h_in)
    return {
        "metric": METRIC, "value": job_value(N, world, args.steps, max_elapsed), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": max_elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; virtual expert-parallel layout from the GPU route)",
        "config": {"workload": f"vep8: T={T} H={H} E={R * L} k={k} bf16, {R} virtual ranks x "
                               f"{L} local experts, {per}-token source slices",
                   "routed_rows_per_step": N,
                   "step": f"moe_sort_chunks rank-major -> expert-major for each of {R} virtual "
                           "ranks, then expert-major -> rank-major",
                   "launch": f"each direction one CUDA graph of its {R} calls over {S} "
                             f"stream{'s' if S > 1 else ''}",
                   "l2": "no flush: the step moves 537 MB each way, > 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(ach / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs", "traffic": None},
        "kernels": kern,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": io,
                "d2h_bytes_per_step": io, "steps": e2e_steps,
                "path": "pinned rank-major buffers -> device -> step -> expert-major to host, "
                        "steps pipelined over two buffer sets on three streams"},
        "gpu_launches": 2 * R * args.steps,              # one fused launch per call (C <= 1024)
        "clocks": clk.summary(),
        **({} if args.no_cpu_baseline else {"cpu_baseline": cpu_baseline_vep8()}),
    }


# ------------------------------------------------------------------ route alone

def run_route_only(args, rank, world, local_rank):
    """moe_route (or moe_route_grouped) alone on a workload's logits: the
    route's own timing and a small device footprint (logits and the index
    outputs only) for profiling its kernels."""
    import torch

    import unpermute_combine_gb300 as moe
    import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    d = wl.make(args.workload, T=args.tokens)
    W = d["workload"]
    T, E, k = d["logits"].shape[0], W.E, W.k
    logits = torch.from_numpy(d["logits"]).to(dev)
    groups = tuple(int(v) for v in args.route_groups.split(":")) if args.route_groups else None
    stream = torch.cuda.Stream(device=dev)

    def route(out=None):
        if groups:
            return moe.moe_route_grouped(logits, k, groups[0], groups[1], out=out, stream=stream)
        return moe.moe_route(logits, k, out=out, stream=stream)

    with torch.cuda.stream(stream):
        r = route()
    for _ in range(args.warmup):
        route(r)
    torch.cuda.synchronize(dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local_rank) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            evs[i].record(stream)
            route(r)
        evs[args.steps].record(stream)
        torch.cuda.synchronize(dev)
    ts = [evs[i].elapsed_time(evs[i + 1]) * 1e3 for i in range(args.steps)]
    if rank != 0:
        return None
    alg = algorithmic_bytes(T, 1, E, k, 2)["route"]
    us = statistics.median(ts)
    return {"metric": "moe_route microseconds per call", "value": us, "unit": "us",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded)",
            "config": {"workload": f"{args.workload}: T={T} E={E} k={k}, router logits only",
                       "step": ("moe_route_grouped" if groups else "moe_route") +
                               ", back to back on one stream (CUDA events around each call)"},
            "route_us": {"median": us, "min": min(ts), "max": max(ts)},
            "alg_bytes": alg, "GB_s": alg / us / 1e3,
            "gpu_launches": route_launches(T, E, k, bool(groups)) * args.steps,
            "clocks": clk.summary()}


# ------------------------------------------------------- stand-in pipelines

def run_stand_in(args, rank, world, local_rank, name):
    """tiny / mid: moe_route, moe_permute, the stand-in expert (rows of
    expert e scaled by (e+1)/E, moe_expert_scale) and the weighted
    moe_combine, timed per call like the main step."""
    import numpy as np
    import torch

    import unpermute_combine_gb300 as moe
    import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    d = wl.make(name)
    W = d["workload"]
    T, H, E, k = W.T, W.H, W.E, W.k
    N = T * k
    f32 = W.dtype == "f32"
    b = 4 if f32 else 2
    if f32:
        x = torch.from_numpy(d["x"]).to(dev)
    else:
        x = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).to(dev)
    logits = torch.from_numpy(d["logits"]).to(dev)
    scale = torch.from_numpy(d["scale"]).to(dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        r = moe.moe_route(logits, k, stream=stream)
        xp = torch.empty((N, H), dtype=x.dtype, device=dev)
        y = torch.empty_like(xp)
        out = torch.empty((T, H), dtype=x.dtype, device=dev)
    names = ["route", "permute", "expert_scale", "combine"]

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        moe.moe_route(logits, k, out=r, stream=stream)
        mark(1)
        moe.moe_permute(x, r.slot_pos, out=xp, stream=stream)
        mark(2)
        moe.moe_expert_scale(xp, r.offsets, scale, out=y, stream=stream)
        mark(3)
        moe.moe_combine(y, r.slot_pos, r.topk_w, out=out, stream=stream)
        mark(4)

    import torch.distributed as dist
    dist_on = dist.is_available() and dist.is_initialized()

    def barrier():
        torch.cuda.synchronize(dev)
        if dist_on:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        barrier()
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        barrier()
    max_elapsed = reduce_max(t0.elapsed_time(t1) / 1e3, dev)
    per = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
           / 1e3 for j, n in enumerate(names)}
    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    alg = algorithmic_bytes(T, H, E, k, b)
    alg["expert_scale"] = 2 * N * H * b + (E + 1) * 4 + E * 4
    kern = {}
    for n in names:
        gbs = alg[n] / per[n] / 1e9
        kern[n] = {"us": round(per[n] * 1e6, 2), "alg_bytes": alg[n], "GB_s": round(gbs, 1),
                   "frac": round(gbs / peak, 4)}
    dominant = max(names, key=lambda n_: per[n_])
    ach = alg[dominant] / per[dominant] / 1e9
    pc = per["permute"] + per["combine"]
    small = alg[dominant] < 2 * 129e6      # fits in L2 between steps: latency-bound
    return {
        "value": job_value(N, world, args.steps, max_elapsed), "unit": UNIT,
        "ms_per_step": max_elapsed / args.steps * 1e3, "steps": args.steps,
        "warmup": args.warmup, "dtype": W.dtype,
        "config": {"workload": f"{name}: T={T} H={H} E={E} k={k} {W.dtype}, {W.note}",
                   "routed_tokens_per_step": N,
                   "step": "moe_route + moe_permute + moe_expert_scale + moe_combine",
                   "l2": ("no flush; the step's few MB stay in the 129 MB L2: latency-bound, "
                          "read the microseconds" if small else
                          "no flush: permute and combine each move > 129 MB")},
        "roofline": {"bound": "latency" if small else "hbm", "kernel": dominant,
                     "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(ach / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": None},
        "kernels": kern,
        "permute_combine_routed_tokens_per_s": N / pc,
        "gpu_launches": (route_launches(T, E, k) + 3) * args.steps,
        "clocks": clk.summary(),
        **({} if args.no_cpu_baseline else
           {"cpu_baseline": cpu_baseline_stand_in(name, min(T, args.cpu_mid_tokens))}),
    }


EXTRA_WORKLOADS = ("layer", "vep8", "mid", "tiny")


def run_extras(args, rank, world, local_rank):
    """The other workloads, each timed after the main step with its own clock
    record: the full layer forward (grouped SwiGLU on the tensor cores), the
    virtual expert-parallel sort_chunks, and the two stand-in pipelines."""
    out = {}
    for name in EXTRA_WORKLOADS:
        sub = argparse.Namespace(**vars(args))
        sub.workload = name
        sub.steps = max(1, min(args.steps, args.extra_steps))
        sub.no_e2e = True
        sub.train = False
        sub.tokens = None
        if name == "layer":
            line = run_ours(sub, rank, world, local_rank)
        elif name == "vep8":
            line = run_vep8(sub, rank, world, local_rank)
        else:
            line = run_stand_in(sub, rank, world, local_rank, name)
        if line is None:
            continue
        keep = ("value", "unit", "ms_per_step", "steps", "config", "roofline", "kernels",
                "permute_combine_routed_tokens_per_s", "gpu_launches", "clocks",
                "cpu_baseline")
        out[name] = {key: line[key] for key in keep if key in line}
        out[name]["steps"] = sub.steps
    return out


# ------------------------------------------------------------ oracle timing

def cpu_baseline(tokens: int):
    """The CPU oracle, as it stands, on the first `tokens` tokens of the same
    workload: route, permute, combine and combine backward, single-threaded."""
    import numpy as np

    import oracle
    import workloads as wl

    d = wl.make(WORKLOAD, with_grad=True)
    W = d["workload"]
    x, lg, g = d["x"][:tokens], d["logits"][:tokens], d["grad_out"][:tokens]
    t0 = time.perf_counter()
    r = oracle.route(lg, W.k)
    xp = oracle.permute(x, r["sorted_indices"])
    out, _ = oracle.combine(xp, r["slot_pos"], r["topk_w"])
    oracle.combine_backward(g, xp, r["slot_pos"], r["topk_w"])
    dt = time.perf_counter() - t0
    n = tokens * W.k
    return {"value": n / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {tokens} of {W.T} tokens ({n} routed rows), one full step, "
                      f"{dt:.1f} s single-threaded C (host has {os.cpu_count()} cores)"}


def cpu_baseline_layer(tokens: int, threads: int = 0):
    """The CPU oracle on the layer workload's first `tokens` tokens: route,
    permute, the grouped SwiGLU of those tokens' rows, combine.  The grouped
    SwiGLU (all but a sliver of the work) runs the oracle unchanged on
    disjoint row sets in `threads` host threads (default: every core this
    process may use); the other steps are single-threaded."""
    import concurrent.futures as cf

    import numpy as np

    import oracle
    import workloads as wl

    d = wl.make("layer", with_weights=True)
    W = d["workload"]
    x, lg = d["x"][:tokens], d["logits"][:tokens]
    cores = threads or len(os.sched_getaffinity(0))
    t0 = time.perf_counter()
    r = oracle.route(lg, W.k)
    xp = oracle.permute(x, r["sorted_indices"])
    n_rows = xp.shape[0]
    parts = [np.arange(i, n_rows, cores, dtype=np.int64) for i in range(min(cores, n_rows))]
    # the oracle call holds no Python lock while it runs (ctypes), so the
    # row sets are computed in parallel; each row is written by one call
    with cf.ThreadPoolExecutor(max_workers=len(parts)) as ex:
        ys = list(ex.map(lambda rows: oracle.grouped_swiglu(xp, d["w_up"], d["w_down"],
                                                            r["offsets"], rows=rows)[0], parts))
    y = np.zeros_like(xp)
    for rows, yp in zip(parts, ys):
        y[rows] = yp[rows]
    oracle.combine(y, r["slot_pos"], r["topk_w"])
    dt = time.perf_counter() - t0
    n = tokens * W.k
    return {"value": n / dt, "unit": UNIT, "cores": len(parts), "kind": "oracle",
            "sample": f"first {tokens} of {W.T} tokens ({n} routed rows), one layer forward, "
                      f"{dt:.1f} s; the grouped SwiGLU over {len(parts)} host threads "
                      f"(host has {os.cpu_count()} cores)"}


def cpu_baseline_stand_in(name: str, tokens: int):
    """The CPU oracle's route, permute, stand-in expert and combine on the
    first `tokens` tokens of a stand-in workload, single-threaded."""
    import oracle
    import workloads as wl

    d = wl.make(name)
    W = d["workload"]
    x, lg = d["x"][:tokens], d["logits"][:tokens]
    t0 = time.perf_counter()
    passes = n = 0
    while passes == 0 or time.perf_counter() - t0 < 1.0:
        r = oracle.route(lg, W.k)
        xp = oracle.permute(x, r["sorted_indices"])
        y = oracle.expert_scale(xp, r["offsets"], d["scale"])
        oracle.combine(y, r["slot_pos"], r["topk_w"])
        n += tokens * W.k
        passes += 1
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {tokens} of {W.T} tokens, route + permute + stand-in expert + "
                      f"combine, {passes} pass{'es' if passes > 1 else ''} in {dt:.2f} s, "
                      f"single-threaded C (host has {os.cpu_count()} cores)"}


def cpu_baseline_vep8():
    """The CPU oracle's sort_chunks forward and inverse for every virtual
    rank of the virtual expert-parallel layout, single-threaded."""
    import numpy as np

    import oracle
    import workloads as wl

    d = wl.make("vep8")
    W = d["workload"]
    R = L = W.ranks
    per = W.T // R
    idx, _, _ = oracle.topk_softmax(d["logits"], W.k)
    bufs = []
    for rr in range(R):
        M = np.zeros((R, L), np.int32)
        rows = []
        for src in range(R):
            toks = np.arange(src * per, (src + 1) * per)
            for le in range(L):
                sel = toks[(idx[toks] == rr * L + le).any(axis=1)]
                M[src, le] = sel.size
                rows.append(sel)
        bufs.append((M, np.ascontiguousarray(d["x"][np.concatenate(rows)])))
    fwd, inv = oracle.chunk_idxs(R, L, False), oracle.chunk_idxs(R, L, True)
    # one pass takes a fraction of a second: repeat whole passes for >= 2 s
    t0 = time.perf_counter()
    n = passes = 0
    while passes == 0 or time.perf_counter() - t0 < 2.0:
        for M, buf in bufs:
            em = oracle.sort_chunks(buf, M.ravel(), fwd)
            oracle.sort_chunks(em, M.T.ravel(), inv)
            n += buf.shape[0]
        passes += 1
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"all {R} virtual ranks ({n // passes} routed rows), forward + inverse, "
                      f"{passes} passes in {dt:.2f} s, single-threaded C "
                      f"(host has {os.cpu_count()} cores)"}


def run_reference(args, rank):
    """Reference arm: the CPU oracle timed as it stands on host cores."""
    if rank != 0:
        return None
    import workloads as wl
    W = wl.WORKLOADS[WORKLOAD]
    for _ in range(args.warmup):
        cpu_baseline(args.ref_tokens)
    vals = [cpu_baseline(args.ref_tokens) for _ in range(args.steps)]
    n = args.ref_tokens * W.k
    total = sum(n / v["value"] for v in vals)
    value = n * args.steps / total
    cb = dict(vals[-1])
    cb["value"] = value
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": f"{WORKLOAD}: T={W.T} H={W.H} E={W.E} k={W.k} bf16, first "
                                   f"{args.ref_tokens} tokens per step",
                       "T": W.T, "H": W.H, "E": W.E, "k": W.k},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=16384)
    ap.add_argument("--ref-tokens", type=int, default=2048)
    ap.add_argument("--cpu-layer-tokens", type=int, default=1024,
                    help="tokens of the layer workload the CPU oracle baseline runs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-mid-tokens", type=int, default=2048,
                    help="tokens of the stand-in workloads the CPU oracle baseline runs")
    ap.add_argument("--route-only", action="store_true",
                    help="time moe_route alone on the workload's logits (small device "
                         "footprint, for profiling the route kernels)")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the main step (skip the layer, vep8, mid and tiny "
                         "workloads that follow it by default)")
    ap.add_argument("--extra-steps", type=int, default=50,
                    help="timed steps of each extra workload (at most --steps)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="use only the first TOKENS tokens (small cases for profiling)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--train", action="store_true",
                    help="layer workload: time a training step (forward keeping activations, "
                         "combine backward, SwiGLU dgrad and wgrad, permute and router backward)")
    ap.add_argument("--router-bwd", action="store_true",
                    help="append the router k-softmax backward (grad_probs -> grad_logits) "
                         "to the training step")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 dispatch: quantize into the slot rows (one fused launch), "
                         "dequantize")
    ap.add_argument("--fp8-gemm", action="store_true",
                    help="with --workload layer --fp8: GMM1 reads the e4m3 slot rows and block "
                         "scales itself (moe_grouped_swiglu_fp8) instead of a dequantize pass")
    ap.add_argument("--fp8-split", action="store_true",
                    help="FP8 dispatch as separate quantize and e4m3 permute launches")
    ap.add_argument("--layout", default=None, metavar="SPEC",
                    help="capacity / padded / aligned layout, e.g. 'cf=1.25,pad' or 'align=128'")
    ap.add_argument("--route-groups", default=None, metavar="G:KG",
                    help="route with group-limited routing: G expert groups, KG kept")
    ap.add_argument("--vep-streams", type=int, default=4, metavar="S",
                    help="vep8: streams the virtual ranks' calls are forked over")
    ap.add_argument("--workload", choices=["skewed", "layer", "vep8", "mid", "tiny"],
                    default=WORKLOAD,
                    help="skewed: the dispatch/combine step (default); layer: the full MoE "
                         "layer forward with the grouped SwiGLU; vep8: sort_chunks forward "
                         "and inverse on an 8-rank x 8-expert virtual EP layout; mid / tiny: "
                         "route, permute, stand-in expert and combine")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        if args.route_only:
            line = run_route_only(args, rank, world, local_rank)
        elif args.workload in ("mid", "tiny"):
            line = run_stand_in(args, rank, world, local_rank, args.workload)
            if line is not None:
                line = {"metric": METRIC, "n_gpus": world, "higher_is_better": True,
                        "scaling": "weak", "vs_baseline": None,
                        "data": "synthetic (seeded)", **line,
                        "e2e": {"value": None, "unit": UNIT, "h2d_bytes_per_step": 0,
                                "d2h_bytes_per_step": 0,
                                "path": "not measured for the stand-in workloads"}}
        else:
            line = (run_vep8 if args.workload == "vep8" else run_ours)(args, rank, world,
                                                                       local_rank)
        plain = (args.workload == WORKLOAD and not (args.fp8 or args.fp8_split or args.layout or
                                                    args.route_groups or args.router_bwd or
                                                    args.tokens or args.train or
                                                    args.route_only))
        if plain and not args.no_extra:
            extra = run_extras(args, rank, world, local_rank)
            if line is not None:
                line["workloads"] = extra
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
