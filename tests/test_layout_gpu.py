"""Capacity, drop-and-pad and aligned layouts (moe_route_layout,
moe_fill_pad_rows) vs the CPU oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import workloads as wl
from moe_testutil import bf16_ulp_diff, to_dev, to_host, within_one_bf16_ulp

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import unpermute_combine_gb300 as moe  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from unpermute_combine_gb300 import build
    build.build()
    moe.load_library()


def _layout_both(idx, w, E, cap, pad, align):
    rows = moe.moe_route_layout_rows(idx.shape[0], E, idx.shape[1], cap, pad, align)
    r = moe.moe_route_layout(to_dev(idx), to_dev(w), E, capacity=cap, pad=pad, alignment=align,
                             max_rows=rows)
    torch.cuda.synchronize()
    o = oracle.route_layout(idx, w, E, capacity=cap, pad=pad, alignment=align, max_rows=rows)
    return r, o, rows


@pytest.mark.parametrize("T,E,k,cap,pad,align,drop", [
    (1000, 8, 2, 200, False, 1, 0.0),        # capacity drops
    (1000, 8, 2, 300, True, 1, 0.1),         # drop and pad
    (3000, 64, 6, 0, False, 128, 0.0),       # DeepEP-style 128 alignment
    (777, 16, 4, 150, False, 32, 0.2),       # capacity + alignment + empty slots
    (40000, 32, 4, 4500, True, 1, 0.0),      # beyond the fused-scan limit
    (100, 4, 4, 1, True, 1, 0.0),            # capacity 1
    (0, 8, 2, 16, True, 1, 0.0)])
def test_layout_matches_oracle(T, E, k, cap, pad, align, drop):
    idx, w = wl.random_routing(T + E + cap, T, E, k, empty_frac=drop)
    r, o, rows = _layout_both(idx, w, E, cap, pad, align)
    for name in ("counts", "offsets", "group_list", "sorted_indices", "slot_pos", "permuted_probs"):
        assert (to_host(getattr(r, name)) == o[name]).all(), name
    assert moe.moe_workspace_status(r.workspace) == 0


def test_layout_skewed_routing_capacity():
    d = wl.make("skewed")
    W = d["workload"]
    cap = moe.moe_expert_capacity(W.T, W.k, W.E, 1.25)
    assert cap == oracle.expert_capacity(W.T, W.k, W.E, 1.25)
    rows = moe.moe_route_layout_rows(W.T, W.E, W.k, cap, True, 1)
    # the oracle's routing of the DeepSeek-shaped logits, given to both sides
    oi = oracle.route(d["logits"], W.k)
    r = moe.moe_route_layout(to_dev(oi["topk_idx"]), to_dev(oi["topk_w"]), W.E, capacity=cap,
                             pad=True, max_rows=rows)
    torch.cuda.synchronize()
    o = oracle.route_layout(oi["topk_idx"], oi["topk_w"], W.E, capacity=cap, pad=True,
                            max_rows=rows)
    for name in ("counts", "offsets", "sorted_indices", "slot_pos", "permuted_probs"):
        assert (to_host(getattr(r, name)) == o[name]).all(), name
    assert (o["slot_pos"] < 0).sum() > 0          # the skew makes the capacity bite


def test_layout_rows_overflow_is_reported():
    idx, w = wl.random_routing(5, 200, 4, 2)
    r = moe.moe_route_layout(to_dev(idx), to_dev(w), 4, capacity=0, pad=False, alignment=64,
                             max_rows=100)
    assert moe.moe_workspace_status(r.workspace) == 6
    sp = to_host(r.slot_pos)
    assert sp.max() < 100


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_permute_into_padded_layout_and_fill_pads(dtype):
    T, E, k, H = 500, 8, 2, 264
    idx, w = wl.random_routing(9, T, E, k)
    cap = moe.moe_expert_capacity(T, k, E, 1.1)
    r, o, rows = _layout_both(idx, w, E, cap, True, 1)
    x = wl.random_activation(10, (T, H), dtype)
    buf = torch.full((rows, H), 7.0, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                     device="cuda")
    moe.moe_permute(to_dev(x), r.slot_pos, out=buf)
    moe.moe_fill_pad_rows(buf, r.offsets, r.counts)
    got = to_host(buf)
    si = o["sorted_indices"]
    n = int(o["offsets"][E])
    exp = np.zeros_like(got)
    exp[si >= 0] = x[si[si >= 0]]
    assert got[:n].tobytes() == exp[:n].tobytes()


def test_capacity_drops_reach_the_combine():
    T, E, k, H = 600, 8, 4, 512
    idx, w = wl.random_routing(11, T, E, k)
    cap = 200
    r, o, rows = _layout_both(idx, w, E, cap, False, 1)
    y = wl.random_activation(12, (rows, H), "bf16")
    out = to_host(moe.moe_combine(to_dev(y), r.slot_pos, to_dev(w)))
    ref, _ = oracle.combine(y, o["slot_pos"], w)
    assert bf16_ulp_diff(out, ref).max() == 0
    g = wl.random_activation(13, (T, H), "bf16")
    gy, gp = moe.moe_combine_backward(to_dev(g), to_dev(y), r.slot_pos, to_dev(w))
    gy_o, gp_o, gp64 = oracle.combine_backward(g, y, o["slot_pos"], w)
    valid = o["slot_pos"][o["slot_pos"] >= 0]
    assert (to_host(gy)[valid] == gy_o[valid]).all()
    assert (to_host(gp)[o["slot_pos"] < 0] == 0).all()
    assert within_one_bf16_ulp(to_host(gp), gp64).all()


def test_aligned_layout_pipeline_equals_plain_pipeline():
    """Aligned (128-row) expert segments change only where rows sit: the MoE
    layer output must be bit-identical to the plain layout's."""
    d = wl.make("layer", with_weights=True)
    W = d["workload"]
    r = moe.moe_route(to_dev(d["logits"]), W.k)
    up_p, down_p = moe.moe_grouped_swiglu_pack(to_dev(d["w_up"]), to_dev(d["w_down"]))
    x = to_dev(d["x"])
    y = moe.moe_grouped_swiglu(moe.moe_permute(x, r.slot_pos), up_p, down_p, r.offsets)
    plain = moe.moe_combine(y, r.slot_pos, r.topk_w)

    rows = moe.moe_route_layout_rows(W.T, W.E, W.k, 0, False, 128)
    ra = moe.moe_route_layout(r.topk_idx, r.topk_w, W.E, alignment=128, max_rows=rows)
    xa = moe.moe_permute(x, ra.slot_pos, n_rows=rows)
    moe.moe_fill_pad_rows(xa, ra.offsets, ra.counts)
    ya = moe.moe_grouped_swiglu(xa, up_p, down_p, ra.offsets)
    aligned = moe.moe_combine(ya, ra.slot_pos, r.topk_w)
    torch.cuda.synchronize()
    offs = to_host(ra.offsets)
    assert (offs % 128 == 0).all()
    assert torch.equal(plain.view(torch.int16), aligned.view(torch.int16))
