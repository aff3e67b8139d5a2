"""Grouped SwiGLU (tcgen05 tensor cores) vs the CPU oracle through the C ABI.

Bar: relative Frobenius error <= 2e-2 against the oracle's double-accumulated
result (the hidden activation is rounded to bf16 on both sides).  The prepack
is a pure rearrangement and must be bit-exact."""
import numpy as np
import pytest

import oracle
import workloads as wl
from moe_testutil import to_dev, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import unpermute_combine_gb300 as moe  # noqa: E402

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from unpermute_combine_gb300 import build
    build.build()
    moe.load_library()


def _weights(seed, E, H, I, std=0.05):
    rng = np.random.default_rng(seed)
    up = wl.f32_to_bf16_bits((rng.standard_normal((E, H, 2 * I)) * std).astype(np.float32))
    down = wl.f32_to_bf16_bits((rng.standard_normal((E, I, H)) * std).astype(np.float32))
    return up, down


def _rel_frob(got_bits, ref64):
    g = wl.bf16_bits_to_f32(got_bits).astype(np.float64)
    return np.linalg.norm(g - ref64) / max(np.linalg.norm(ref64), 1e-30)


def test_pack_layout_bit_exact():
    E, H, I = 2, 256, 256
    up, down = _weights(1, E, H, I)
    up_p, down_p = moe.moe_grouped_swiglu_pack(to_dev(up), to_dev(down))
    up_p, down_p = to_host(up_p), to_host(down_p)
    # expected: rows of w_up^T, regrouped per 128 hidden columns as [gate | up]
    upT = np.transpose(up, (0, 2, 1))           # [E, 2I, H]
    exp_up = np.empty_like(upT)
    for b in range(I // 128):
        exp_up[:, b * 256:b * 256 + 128] = upT[:, b * 128:(b + 1) * 128]
        exp_up[:, b * 256 + 128:(b + 1) * 256] = upT[:, I + b * 128:I + (b + 1) * 128]
    assert (up_p == exp_up).all()
    assert (down_p == np.transpose(down, (0, 2, 1))).all()


@pytest.mark.parametrize("counts,H,I", [([128], 256, 128),            # one tile
                                        ([130, 0, 300], 256, 128),    # ragged, an empty expert
                                        ([1, 255, 0, 0, 77], 512, 256),
                                        ([0, 0, 64], 256, 384)])
def test_grouped_swiglu_small(counts, H, I):
    E = len(counts)
    N = sum(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rng = np.random.default_rng(N + H + I)
    x = wl.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    up, down = _weights(N + E, E, H, I)
    up_p, down_p = moe.moe_grouped_swiglu_pack(to_dev(up), to_dev(down))
    sentinel = torch.full((N + 3, H), 5.0, dtype=torch.bfloat16, device="cuda")
    y = moe.moe_grouped_swiglu(to_dev(x), up_p, down_p, to_dev(offsets),
                               out=sentinel[:N] if N else None)
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(y._moe_workspace) == 0
    y_o, y64 = oracle.grouped_swiglu(x, up, down, offsets)
    err = _rel_frob(to_host(y), y64)
    assert err <= TOL, err
    # per-expert too, so a wrong segment cannot hide behind a big neighbour
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            assert _rel_frob(to_host(y)[a:b], y64[a:b]) <= TOL
    # rows past the routed rows are untouched
    assert (to_host(sentinel[N:]) == wl.f32_to_bf16_bits(np.full((3, H), 5.0, np.float32))).all()


def test_grouped_swiglu_layer_workload_sampled():
    """Full-size MoE layer workload (T=4096, H=2048, E=64, k=6, I=1408):
    GPU route -> permute -> grouped SwiGLU -> combine, against the oracle on a
    seeded sample of tokens."""
    d = wl.make("layer", with_weights=True)
    W = d["workload"]
    r = moe.moe_route(to_dev(d["logits"]), W.k)
    xp = moe.moe_permute(to_dev(d["x"]), r.slot_pos)
    up_p, down_p = moe.moe_grouped_swiglu_pack(to_dev(d["w_up"]), to_dev(d["w_down"]))
    y = moe.moe_grouped_swiglu(xp, up_p, down_p, r.offsets)
    out = moe.moe_combine(y, r.slot_pos, r.topk_w)
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(y._moe_workspace) == 0

    o = oracle.route(d["logits"], W.k)
    n = int(o["offsets"][W.E])
    xp_o = oracle.permute(d["x"], o["sorted_indices"], n)
    rng = np.random.default_rng(77)
    toks = np.sort(rng.choice(W.T, 24, replace=False))
    rows = o["slot_pos"][toks].ravel()
    y_o, y64 = oracle.grouped_swiglu(xp_o, d["w_up"], d["w_down"], o["offsets"], rows=rows)
    y_gpu = to_host(y)
    assert _rel_frob(y_gpu[rows], y64[rows]) <= TOL
    for p in rows[:12]:
        assert _rel_frob(y_gpu[p:p + 1], y64[p:p + 1]) <= TOL
    # combine of the sampled tokens from the oracle's expert outputs
    sp_local = np.arange(rows.size, dtype=np.int32).reshape(toks.size, W.k)
    out_o, out64 = oracle.combine(np.ascontiguousarray(y_o[rows]), sp_local, o["topk_w"][toks])
    assert _rel_frob(to_host(out)[toks], out64) <= TOL


def test_grouped_swiglu_e1_is_a_dense_ffn():
    """With one expert the layer is a plain SwiGLU FFN; torch (cuBLAS) gives
    an independent reference on the GPU."""
    N, H, I = 384, 512, 256
    rng = np.random.default_rng(5)
    x = wl.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    up, down = _weights(6, 1, H, I)
    up_p, down_p = moe.moe_grouped_swiglu_pack(to_dev(up), to_dev(down))
    y = moe.moe_grouped_swiglu(to_dev(x), up_p, down_p,
                               to_dev(np.array([0, N], np.int32)))
    xf = to_dev(x).float()
    gu = xf @ to_dev(up).float()[0]
    h = (torch.nn.functional.silu(gu[:, :I]) * gu[:, I:]).bfloat16().float()
    ref = (h @ to_dev(down).float()[0]).double().cpu().numpy()
    assert _rel_frob(to_host(y), ref) <= TOL


def _dequant_oracle(q_dev, sc_dev):
    q = q_dev.view(torch.uint8).cpu().numpy()
    return oracle.dequantize_fp8(q, sc_dev.cpu().numpy(), 128)


@pytest.mark.parametrize("counts,H,I", [([128], 512, 128),
                                        ([130, 0, 300], 512, 128),    # ragged, an empty expert
                                        ([1, 255, 0, 0, 77], 1024, 256),
                                        ([0, 0, 64], 512, 384)])
def test_grouped_swiglu_fp8_is_the_bf16_path_on_dequantized_rows(counts, H, I):
    """GMM1 from e4m3 codes and block scales: bit for bit moe_grouped_swiglu
    on moe_dequantize_fp8's rows, and within the bar of the oracle fed the
    oracle's dequantized rows."""
    E = len(counts)
    N = sum(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rng = np.random.default_rng(3 * N + H + I)
    # rows of mixed magnitude, so the block scales differ along a row
    x32 = rng.standard_normal((N, H)).astype(np.float32)
    x32 *= np.exp2(rng.integers(-6, 7, size=(N, H // 128))).repeat(128, axis=1).astype(np.float32)
    x = wl.f32_to_bf16_bits(x32)
    up, down = _weights(N + 2 * E, E, H, I)
    up_p, down_p = moe.moe_grouped_swiglu_pack(to_dev(up), to_dev(down))
    q, sc = moe.moe_quantize_fp8(to_dev(x), 128)
    off = to_dev(offsets)
    sentinel = torch.full((N + 3, H), 5.0, dtype=torch.bfloat16, device="cuda")
    y8 = moe.moe_grouped_swiglu_fp8(q, sc, up_p, down_p, off, out=sentinel[:N] if N else None)
    yd = moe.moe_grouped_swiglu(moe.moe_dequantize_fp8(q, sc, 128), up_p, down_p, off)
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(y8._moe_workspace) == 0
    assert (to_host(y8) == to_host(yd)).all()
    assert (to_host(sentinel[N:]) == wl.f32_to_bf16_bits(np.full((3, H), 5.0, np.float32))).all()
    if N:
        xd_o = _dequant_oracle(q, sc)
        y_o, y64 = oracle.grouped_swiglu(xd_o, up, down, offsets)
        assert _rel_frob(to_host(y8), y64) <= TOL


def test_grouped_swiglu_fp8_layer_workload():
    """Full-size layer workload with FP8 dispatch: GPU route -> fused
    quantize-into-slots -> grouped SwiGLU from the e4m3 rows -> combine; the
    expert outputs equal the bf16 path on the dequantized rows bit for bit,
    and sampled tokens match the oracle on the oracle's dequantized rows."""
    d = wl.make("layer", with_weights=True)
    W = d["workload"]
    r = moe.moe_route(to_dev(d["logits"]), W.k)
    q, sc = moe.moe_permute_quantize_fp8(to_dev(d["x"]), r.slot_pos, 128)
    up_p, down_p = moe.moe_grouped_swiglu_pack(to_dev(d["w_up"]), to_dev(d["w_down"]))
    y8 = moe.moe_grouped_swiglu_fp8(q, sc, up_p, down_p, r.offsets)
    yd = moe.moe_grouped_swiglu(moe.moe_dequantize_fp8(q, sc, 128), up_p, down_p, r.offsets)
    out = moe.moe_combine(y8, r.slot_pos, r.topk_w)
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(y8._moe_workspace) == 0
    assert (to_host(y8) == to_host(yd)).all()

    o = oracle.route(d["logits"], W.k)
    rng = np.random.default_rng(78)
    toks = np.sort(rng.choice(W.T, 16, replace=False))
    rows = o["slot_pos"][toks].ravel()
    xd_o = _dequant_oracle(q, sc)
    y_o, y64 = oracle.grouped_swiglu(xd_o, d["w_up"], d["w_down"], o["offsets"], rows=rows)
    assert _rel_frob(to_host(y8)[rows], y64[rows]) <= TOL
    sp_local = np.arange(rows.size, dtype=np.int32).reshape(toks.size, W.k)
    out_o, out64 = oracle.combine(np.ascontiguousarray(y_o[rows]), sp_local, o["topk_w"][toks])
    assert _rel_frob(to_host(out)[toks], out64) <= TOL
