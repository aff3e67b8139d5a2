"""FP8 dispatch (moe_quantize_fp8, FP8 row movement, moe_dequantize_fp8) vs
the CPU oracle through the C ABI: every byte and every bf16 bit exact."""
import numpy as np
import pytest

import oracle
import workloads as wl
from moe_testutil import to_dev, to_host

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


def _fp8_host(t):
    return t.view(torch.uint8).cpu().numpy()


def _fp8_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda().view(torch.float8_e4m3fn)


def _tricky_rows(seed, T, H):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((T, H)) * np.exp(rng.uniform(-12, 6, (T, 1)))).astype(np.float32)
    x[0, :] = 0.0                                   # all-zero blocks
    x[1, :] = -0.0
    x[2, ::7] = 3e38                                # huge
    x[3, :] = rng.standard_normal(H).astype(np.float32) * 1e-30
    return wl.f32_to_bf16_bits(x)


@pytest.mark.parametrize("T,H,block", [(64, 7168, 128), (33, 4096, 128), (17, 512, 32),
                                       (9, 768, 256), (5, 128, 64)])
def test_quantize_and_dequantize_bit_exact(T, H, block):
    x = _tricky_rows(T + H + block, T, H)
    q, sc = moe.moe_quantize_fp8(to_dev(x), block)
    q_o, sc_o = oracle.quantize_fp8(x, block)
    assert (_fp8_host(q) == q_o).all()
    assert (to_host(sc).view(np.uint32) == sc_o.view(np.uint32)).all()
    dq = to_host(moe.moe_dequantize_fp8(q, sc, block))
    assert (dq == oracle.dequantize_fp8(q_o, sc_o, block)).all()


def test_fp8_dispatch_pipeline_matches_oracle():
    """route -> quantize -> permute the e4m3 rows and their scale rows ->
    dequantize, on the first 2048 tokens of the DeepSeek-shaped workload."""
    d = wl.make("skewed", T=2048)
    W = d["workload"]
    T, H, k, E = 2048, W.H, W.k, W.E
    r = moe.moe_route(to_dev(d["logits"]), k)
    q, sc = moe.moe_quantize_fp8(to_dev(d["x"]), 128)
    qp, scp = moe.moe_permute_fp8(q, sc, r.slot_pos)
    xp = to_host(moe.moe_dequantize_fp8(qp, scp, 128))
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    o = oracle.route(d["logits"], k)
    n = int(o["offsets"][E])
    q_o, sc_o = oracle.quantize_fp8(d["x"], 128)
    qp_o = oracle.permute(q_o, o["sorted_indices"], n)
    scp_o = oracle.permute(sc_o, o["sorted_indices"], n)
    assert (_fp8_host(qp)[:n] == qp_o).all()
    assert (to_host(scp)[:n] == scp_o).all()
    assert (xp[:n] == oracle.dequantize_fp8(qp_o, scp_o, 128)).all()


def test_fp8_rows_through_sort_chunks_and_pad_fill():
    rng = np.random.default_rng(3)
    R, L, H = 3, 4, 256
    M = rng.integers(0, 20, (R, L)).astype(np.int32)
    N = int(M.sum())
    q = rng.integers(0, 256, (N, H)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0                        # no NaN patterns
    fwd = oracle.chunk_idxs(R, L, False)
    em = moe.moe_sort_chunks(_fp8_dev(q), to_dev(M.ravel().copy()), to_dev(fwd))
    assert (_fp8_host(em) == oracle.sort_chunks(q, M.ravel(), fwd)).all()
    offsets = to_dev(np.array([0, 4, 10], np.int32))
    counts = to_dev(np.array([2, 6], np.int32))
    buf = _fp8_dev(np.full((12, H), 0x38, np.uint8))
    moe.moe_fill_pad_rows(buf, offsets, counts)
    got = _fp8_host(buf)
    assert (got[2:4] == 0).all() and (got[:2] == 0x38).all() and (got[4:] == 0x38).all()


@pytest.mark.parametrize("T,H,block,k,E,cap", [
    (1000, 7168, 128, 8, 64, 0),     # 224-byte scale rows ride with the data row
    (513, 4096, 32, 4, 16, 0),       # 512-byte scale rows
    (300, 96, 32, 2, 8, 0),          # 12-byte scale rows: the two-launch path
    (700, 2048, 128, 6, 32, 100),    # capacity drops: unnamed rows stay untouched
    (4, 256, 256, 1, 2, 0),        # 4-byte scale rows
    (50, 20480, 128, 4, 16, 0)])   # 20 KB e4m3 rows: 2 pieces, the scale row with the first
def test_permute_fp8_matches_oracle(T, H, block, k, E, cap):
    idx, w = wl.random_routing(T + H + k, T, E, k)
    rows = moe.moe_route_layout_rows(T, E, k, cap, False, 1)
    r = moe.moe_route_layout(to_dev(idx), to_dev(w), E, capacity=cap, max_rows=rows)
    o = oracle.route_layout(idx, w, E, capacity=cap, max_rows=rows)
    x = _tricky_rows(T * 3 + H, T, H)
    q, sc = moe.moe_quantize_fp8(to_dev(x), block)
    oq = _fp8_dev(np.full((rows, H), 0x3C, np.uint8))
    osc = torch.full((rows, H // block), -2.0, dtype=torch.float32, device="cuda")
    moe.moe_permute_fp8(q, sc, r.slot_pos, out=(oq, osc))
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    q_o, sc_o = oracle.quantize_fp8(x, block)
    si = o["sorted_indices"]
    exp_q = np.full((rows, H), 0x3C, np.uint8)
    exp_s = np.full((rows, H // block), -2.0, np.float32)
    exp_q[si >= 0] = q_o[si[si >= 0]]
    exp_s[si >= 0] = sc_o[si[si >= 0]]
    assert (_fp8_host(oq) == exp_q).all()
    assert (to_host(osc).view(np.uint32) == exp_s.view(np.uint32)).all()


def test_quantize_on_and_near_e4m3_midpoints():
    """Quotients on an e4m3 rounding midpoint (ties to even) or within a few
    float ulps of one, where the code depends on the last bits of the IEEE
    quotient; bit-exact against the oracle."""
    rng = np.random.default_rng(77)
    T, H, block = 512, 4096, 128
    x = rng.standard_normal((T, H)).astype(np.float32)
    # rows 0-15: every block has amax = 448 (scale exactly 1) and its other
    # values on midpoints 2^e (1 + (2m+1)/16), e = -6..7, with random signs
    e = rng.integers(-6, 8, (16, H))
    m = rng.integers(0, 8, (16, H))
    x[:16] = np.ldexp(1.0 + (2 * m + 1) / 16.0, e) * rng.choice([-1.0, 1.0], (16, H))
    x[:16, ::block] = 448.0
    xb = wl.f32_to_bf16_bits(x)
    # the random rows must reach quotients within 8 float ulps of a midpoint
    xf = wl.bf16_bits_to_f32(xb).reshape(T, H // block, block)
    amax = np.abs(xf).max(axis=2, keepdims=True)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q0 = (xf * (np.float32(1.0) / s)).astype(np.float32)
    bits = q0.view(np.uint32)
    mag = bits & 0x7FFFFFFF
    near = (np.abs((bits & 0xFFFFF).astype(np.int64) - 0x80000) <= 8) & (mag >= 0x3C800000)
    assert near[16:].sum() >= 5 and near[:16].sum() > 1000
    q, sc = moe.moe_quantize_fp8(to_dev(xb), block)
    q_o, sc_o = oracle.quantize_fp8(xb, block)
    assert (to_host(sc).view(np.uint32) == sc_o.view(np.uint32)).all()
    assert (_fp8_host(q) == q_o).all()


@pytest.mark.parametrize("T,H,block,k,E,cap", [
    (1000, 7168, 128, 8, 64, 0),     # the DeepSeek row width
    (5000, 2048, 128, 6, 64, 0),     # many tokens per CTA: the ring wraps many times
    (513, 4096, 32, 4, 16, 0),
    (300, 96, 32, 2, 8, 0),          # a 192-byte row
    (700, 2048, 64, 6, 32, 100),     # capacity drops: unnamed rows stay untouched
    (64, 8192, 256, 3, 8, 0),        # the widest row one stage holds
    (4, 512, 128, 1, 2, 0)])         # fewer tokens than CTAs
def test_permute_quantize_fp8_matches_quantize_then_permute(T, H, block, k, E, cap):
    idx, w = wl.random_routing(T + H + 3 * k, T, E, k)
    rows = moe.moe_route_layout_rows(T, E, k, cap, False, 1)
    r = moe.moe_route_layout(to_dev(idx), to_dev(w), E, capacity=cap, max_rows=rows)
    o = oracle.route_layout(idx, w, E, capacity=cap, max_rows=rows)
    x = _tricky_rows(T * 5 + H, T, H)
    oq = _fp8_dev(np.full((rows, H), 0x3C, np.uint8))
    osc = torch.full((rows, H // block), -2.0, dtype=torch.float32, device="cuda")
    moe.moe_permute_quantize_fp8(to_dev(x), r.slot_pos, block, out=(oq, osc))
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    q_o, sc_o = oracle.quantize_fp8(x, block)
    si = o["sorted_indices"]
    exp_q = np.full((rows, H), 0x3C, np.uint8)
    exp_s = np.full((rows, H // block), -2.0, np.float32)
    exp_q[si >= 0] = q_o[si[si >= 0]]
    exp_s[si >= 0] = sc_o[si[si >= 0]]
    assert (_fp8_host(oq) == exp_q).all()
    assert (to_host(osc).view(np.uint32) == exp_s.view(np.uint32)).all()


def test_permute_quantize_fp8_skips_slots_outside_the_rows():
    """Slots naming a row outside [0, n_rows) (negative other than -1, or
    past the buffer) move nothing; every other slot row is the oracle's."""
    T, H, E, k, block = 300, 1024, 16, 4, 128
    idx, w = wl.random_routing(41, T, E, k)
    o = oracle.route_indices(idx, w, E)
    sp = o["slot_pos"].copy()
    rows = T * k
    bad = np.random.default_rng(42).random(sp.shape) < 0.1
    sp[bad] = np.where(np.random.default_rng(43).random(bad.sum()) < 0.5, rows + 5, -7)
    x = _tricky_rows(44, T, H)
    oq = _fp8_dev(np.full((rows, H), 0x3C, np.uint8))
    osc = torch.full((rows, H // block), -2.0, dtype=torch.float32, device="cuda")
    moe.moe_permute_quantize_fp8(to_dev(x), to_dev(sp), block, out=(oq, osc))
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    q_o, sc_o = oracle.quantize_fp8(x, block)
    exp_q = np.full((rows, H), 0x3C, np.uint8)
    exp_s = np.full((rows, H // block), -2.0, np.float32)
    for t in range(T):
        for j in range(k):
            p = sp[t, j]
            if 0 <= p < rows:
                exp_q[p] = q_o[t]
                exp_s[p] = sc_o[t]
    assert (_fp8_host(oq) == exp_q).all()
    assert (to_host(osc).view(np.uint32) == exp_s.view(np.uint32)).all()


def test_shared_memory_limit_only_grows():
    """A kernel's dynamic shared-memory limit is raised for the largest row it
    has seen and never lowered: a wide call, a narrow call, then the wide one
    again must all launch (a narrower call once lowered the limit under the
    wide call's stage size, and the third launch failed)."""
    T, k, E, block = 64, 2, 8, 128
    idx, w = wl.random_routing(7, T, E, k)
    r = moe.moe_route_indices(to_dev(idx), to_dev(w), E)
    for H in (2048, 512, 2048):
        x = _tricky_rows(H + 1, T, H)
        oq, osc = moe.moe_permute_quantize_fp8(to_dev(x), r.slot_pos, block)
        torch.cuda.synchronize()
        q_o, sc_o = oracle.quantize_fp8(x, block)
        si = oracle.route_indices(idx, w, E)["sorted_indices"]
        assert (_fp8_host(oq) == q_o[si]).all()
        assert (to_host(osc).view(np.uint32) == sc_o[si].view(np.uint32)).all()
