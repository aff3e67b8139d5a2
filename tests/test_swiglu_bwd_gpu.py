"""Grouped SwiGLU training path (moe_grouped_swiglu_save / _dgrad / _wgrad)
vs the CPU oracle through the C ABI.

Bounds, from the arithmetic: the GPU accumulates in fp32 on the tensor cores
(order unknown) where the oracle sums in double, then both round once to bf16.
So a bf16 output may differ from the oracle's unrounded double by its own
rounding (half an ulp: 2^-8 relative) and from the oracle's bf16 by one ulp
(2^-7 relative), plus the fp32 accumulation error, bounded by a floor of
2^-10 of the tensor's rms.  Where an output is a product of a stored bf16
intermediate (dx of dgate_up, y of hidden), the measured last-bit differences
of that intermediate are propagated exactly into the bound (sum of
|difference| x |weight|).  The fp32 weight gradients are checked per element
against 8 * K * 2^-24 * sum_p |a_p b_p| (the bound for any summation order of
K products, with headroom for the tensor core's accumulator)."""
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


def _f(bits):
    return wl.bf16_bits_to_f32(np.ascontiguousarray(bits)).astype(np.float64)


def _bf16_close(got_bits, ref64, name, rel=2.0 ** -8, extra=0.0):
    """rel = 2^-8 against an unrounded double (half a bf16 ulp), 2^-7 against
    the oracle's own bf16 (one ulp); extra = a propagated input difference."""
    got = _f(got_bits)
    rms = np.sqrt(np.mean(ref64 ** 2)) if ref64.size else 0.0
    bound = rel * np.abs(ref64) + 2.0 ** -10 * rms + extra + 1e-30
    bad = np.abs(got - ref64) > bound
    assert not bad.any(), f"{name}: {bad.sum()} of {bad.size} outside the bound"


def _dx_extra(dgu_gpu_bits, dgu_o_bits, w_up_bits, offsets, rows):
    """sum_c |dgate_up_gpu - dgate_up_oracle|[p,c] * |w_up[e][h][c]|: how far
    the stored dgate_up's last-bit differences can move dx[p,h]."""
    out = np.zeros((len(rows), w_up_bits.shape[1]))
    d = np.abs(_f(dgu_gpu_bits) - _f(dgu_o_bits))
    for i, p in enumerate(rows):
        e = int(np.searchsorted(offsets, p, side="right") - 1)
        out[i] = np.abs(_f(w_up_bits[e])) @ d[i]
    return out * (1 + 2.0 ** -20)


def _case(seed, counts, H, I, scale=0.05):
    rng = np.random.default_rng(seed)
    E = len(counts)
    N = int(sum(counts))
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = wl.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    up = wl.f32_to_bf16_bits((rng.standard_normal((E, H, 2 * I)) * scale).astype(np.float32))
    down = wl.f32_to_bf16_bits((rng.standard_normal((E, I, H)) * scale).astype(np.float32))
    dy = wl.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    return dict(E=E, N=N, H=H, I=I, offsets=offsets, x=x, up=up, down=down, dy=dy)


def _wgrad_bound(P, Q, offsets, which_coords):
    """8 * K_e * 2^-24 * sum_p |P[p,a] Q[p,b]| at each coordinate (e, a, b)."""
    out = np.empty(len(which_coords))
    for i, (e, a, b) in enumerate(which_coords):
        r0, r1 = offsets[e], offsets[e + 1]
        s = np.abs(P[r0:r1, a] * Q[r0:r1, b]).sum()
        out[i] = 8 * max(r1 - r0, 1) * 2.0 ** -24 * s + 1e-30
    return out


CASES = [
    (1, [37, 0, 129, 300], 256, 128),     # ragged, empty expert, 64-row tails, half N tile
    (2, [64, 200, 1, 63], 512, 384),      # 1.5 N tiles, single-row expert
    (3, [130], 256, 256),                  # one expert
    # last stages of 16, 48, 32, 16, 17, 33 rows: whole 16-row MMA groups with
    # no zeroed tail next to ragged ones
    (4, [16, 48, 96, 80, 17, 33], 256, 128),
]


@pytest.mark.parametrize("seed,counts,H,I", CASES)
def test_forward_save_matches_forward_and_oracle(seed, counts, H, I):
    c = _case(seed, counts, H, I)
    up_p, down_p = moe.moe_grouped_swiglu_pack(to_dev(c["up"]), to_dev(c["down"]))
    xd, off = to_dev(c["x"]), to_dev(c["offsets"])
    y0 = moe.moe_grouped_swiglu(xd, up_p, down_p, off)
    y, hid, gu = moe.moe_grouped_swiglu_save(xd, up_p, down_p, off)
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(y._moe_workspace) == 0
    assert torch.equal(y0.view(torch.int16), y.view(torch.int16))     # same arithmetic
    _, y64, gu_o, hid_o = oracle.grouped_swiglu(c["x"], c["up"], c["down"], c["offsets"],
                                                save=True)
    _bf16_close(to_host(gu), _f(gu_o), "gate_up", rel=2.0 ** -7)
    _bf16_close(to_host(hid), _f(hid_o), "hidden", rel=2.0 ** -7)


@pytest.mark.parametrize("seed,counts,H,I", CASES)
def test_dgrad_matches_oracle(seed, counts, H, I):
    c = _case(seed, counts, H, I)
    _, _, gu_o, _ = oracle.grouped_swiglu(c["x"], c["up"], c["down"], c["offsets"], save=True)
    dgu, dx = moe.moe_grouped_swiglu_dgrad(to_dev(c["dy"]), to_dev(c["up"]), to_dev(c["down"]),
                                           to_dev(c["offsets"]), to_dev(gu_o))
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(dx._moe_workspace) == 0
    dgu_o, dgu64, dx_o, dx64 = oracle.swiglu_dgrad(c["dy"], c["up"], c["down"], c["offsets"], gu_o)
    dgu_h = to_host(dgu)
    _bf16_close(dgu_h, dgu64, "dgate_up")
    # dx is a product of the stored (bf16) dgate_up: compare with the oracle's
    # dx from its own dgate_up, allowing for dgate_up's last-bit differences
    extra = _dx_extra(dgu_h, dgu_o, c["up"], c["offsets"], np.arange(c["N"]))
    _bf16_close(to_host(dx), dx64, "dx", extra=extra)


@pytest.mark.parametrize("seed,counts,H,I", CASES)
def test_wgrad_matches_oracle(seed, counts, H, I):
    c = _case(seed, counts, H, I)
    E, off = c["E"], c["offsets"]
    _, _, gu_o, hid_o = oracle.grouped_swiglu(c["x"], c["up"], c["down"], off, save=True)
    dgu_o, *_ = oracle.swiglu_dgrad(c["dy"], c["up"], c["down"], off, gu_o)
    dw_up, dw_down = moe.moe_grouped_swiglu_wgrad(to_dev(c["x"]), to_dev(hid_o), to_dev(c["dy"]),
                                                 to_dev(dgu_o), to_dev(off))
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(dw_up._moe_workspace) == 0
    got_up, got_down = to_host(dw_up), to_host(dw_down)
    rng = np.random.default_rng(seed)
    for which, got, P, Q, A, B in (("up", got_up, c["x"], dgu_o, H, 2 * I),
                                   ("down", got_down, hid_o, c["dy"], I, H)):
        coords = [(e, int(rng.integers(A)), int(rng.integers(B))) for e in range(E)
                  for _ in range(64)]
        # every corner of every tile row / column block too
        coords += [(e, a, b) for e in range(E) for a in (0, A - 1) for b in (0, B - 1)]
        kw = dict(x=c["x"], dgate_up=dgu_o) if which == "up" else dict(hidden=hid_o, dy=c["dy"])
        ref = oracle.swiglu_wgrad_at(which, coords, off, H, I, **kw)
        g = np.array([got[e, a, b] for e, a, b in coords], np.float64)
        bound = _wgrad_bound(_f(P), _f(Q), off, coords)
        assert (np.abs(g - ref) <= bound).all(), which
        for e in range(E):
            if off[e] == off[e + 1]:
                assert (got[e] == 0).all()                      # empty expert


def test_layer_workload_training_path():
    """DeepSeek-style layer (T=4096, H=2048, E=64, k=6, I=1408) at full size:
    the GPU training chain (save -> dgrad -> wgrad) vs the oracle on sampled
    rows and weight-gradient coordinates."""
    d = wl.make("layer", with_weights=True)
    W = d["workload"]
    r = moe.moe_route(to_dev(d["logits"]), W.k)
    o = oracle.route(d["logits"], W.k)
    off = o["offsets"]
    assert (to_host(r.offsets) == off).all()                # same row layout on both sides
    N = int(off[-1])
    xp = moe.moe_permute(to_dev(d["x"]), r.slot_pos)
    up, down = to_dev(d["w_up"]), to_dev(d["w_down"])
    up_p, down_p = moe.moe_grouped_swiglu_pack(up, down)
    y, hid, gu = moe.moe_grouped_swiglu_save(xp, up_p, down_p, r.offsets)
    dy_h = wl.f32_to_bf16_bits(np.random.default_rng(9).standard_normal((N, W.H)).astype(np.float32))
    dy = to_dev(dy_h)
    dgu, dx = moe.moe_grouped_swiglu_dgrad(dy, up, down, r.offsets, gu)
    dw_up, dw_down = moe.moe_grouped_swiglu_wgrad(xp, hid, dy, dgu, r.offsets)
    torch.cuda.synchronize()
    for t in (y, dx, dw_up):
        assert moe.moe_workspace_status(t._moe_workspace) == 0
    x_o = oracle.permute(d["x"], o["sorted_indices"], N)     # the oracle's expert input
    x_h = to_host(xp)
    rows = np.random.default_rng(10).choice(N, 48, replace=False)
    rows = np.concatenate([rows, off[1:-1][off[1:-1] < N][:8], [N - 1]]).astype(np.int64)
    _, y64, gu_o, hid_o = oracle.grouped_swiglu(x_o, d["w_up"], d["w_down"], off, rows=rows,
                                                save=True)
    _bf16_close(to_host(gu)[rows], _f(gu_o[rows]), "gate_up", rel=2.0 ** -7)
    # y from the GPU's own hidden: each hidden may sit one bf16 ulp from the
    # oracle's, moving y by up to sum_i ulp(h_i) |w_down[e][i][h]|
    hid_d = np.abs(_f(to_host(hid)[rows]) - _f(hid_o[rows]))
    y_extra = np.stack([hid_d[i] @ np.abs(_f(d["w_down"][int(np.searchsorted(off, p, "right") - 1)]))
                        for i, p in enumerate(rows)]) * (1 + 2.0 ** -20)
    _bf16_close(to_host(y)[rows], y64[rows], "y", extra=y_extra)
    # dgrad of the sampled rows: the GPU ran it on its own gate_up, the oracle
    # on its own; the gate_up difference propagates into dgate_up and dx, so
    # feed the oracle's gate_up through the GPU dgrad too for a tight check
    dgu_o, dgu64, _, dx64 = oracle.swiglu_dgrad(dy_h, d["w_up"], d["w_down"], off, gu_o, rows=rows)
    gu_mix = to_host(gu)
    gu_mix[rows] = gu_o[rows]
    dgu2, dx2 = moe.moe_grouped_swiglu_dgrad(dy, up, down, r.offsets, to_dev(gu_mix))
    dgu2_h = to_host(dgu2)
    _bf16_close(dgu2_h[rows], dgu64[rows], "dgate_up")
    extra = _dx_extra(dgu2_h[rows], dgu_o[rows], d["w_up"], off, rows)
    _bf16_close(to_host(dx2)[rows], dx64[rows], "dx", extra=extra)
    # wgrad at sampled coordinates: the oracle's weight gradient (double sum
    # over the expert's rows) of the GPU chain's own activations, so only the
    # wgrad kernel's arithmetic is under test here
    rng = np.random.default_rng(11)
    hid_h, dgu_h = to_host(hid), to_host(dgu)
    for which, got, P, Q, A, B in (("up", to_host(dw_up), x_h, dgu_h, W.H, 2 * W.I),
                                   ("down", to_host(dw_down), hid_h, dy_h, W.I, W.H)):
        coords = [(int(rng.integers(W.E)), int(rng.integers(A)), int(rng.integers(B)))
                  for _ in range(200)]
        ref = oracle.swiglu_wgrad_at(which, np.array(coords), off, W.H, W.I, x=x_h, hidden=hid_h,
                                     dy=dy_h, dgate_up=dgu_h)
        g = np.array([got[e, a, b] for e, a, b in coords], np.float64)
        bound = _wgrad_bound(_f(P), _f(Q), off, coords)
        assert (np.abs(g - ref) <= bound).all(), which


def test_training_on_an_aligned_layout_equals_the_plain_layout():
    """Expert segments padded to 64 rows with zero pad rows (the layout that
    spares the wgrad its partial stages): every row output is bit-identical
    to the plain layout's, and the weight gradients agree within the fp32
    summation bound (same products, different K stages)."""
    rng = np.random.default_rng(21)
    T, H, I, E, k = 700, 256, 128, 8, 2
    idx, w = wl.random_routing(22, T, E, k)
    x = to_dev(wl.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)))
    up_h = wl.f32_to_bf16_bits((rng.standard_normal((E, H, 2 * I)) * 0.05).astype(np.float32))
    down_h = wl.f32_to_bf16_bits((rng.standard_normal((E, I, H)) * 0.05).astype(np.float32))
    g = to_dev(wl.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)))
    up, down = to_dev(up_h), to_dev(down_h)
    up_p, down_p = moe.moe_grouped_swiglu_pack(up, down)

    def chain(r, rows):
        xp = moe.moe_permute(x, r.slot_pos, n_rows=rows)
        moe.moe_fill_pad_rows(xp, r.offsets, r.counts)
        y, hid, gu = moe.moe_grouped_swiglu_save(xp, up_p, down_p, r.offsets)
        gy, _ = moe.moe_combine_backward(g, y, r.slot_pos, to_dev(w))
        moe.moe_fill_pad_rows(gy, r.offsets, r.counts)
        dgu, dx = moe.moe_grouped_swiglu_dgrad(gy, up, down, r.offsets, gu)
        dwu, dwd = moe.moe_grouped_swiglu_wgrad(xp, hid, gy, dgu, r.offsets)
        torch.cuda.synchronize()
        for t_ in (y, dx, dwu):
            assert moe.moe_workspace_status(t_._moe_workspace) == 0
        return dict(xp=to_host(xp), y=to_host(y), gu=to_host(gu), hid=to_host(hid),
                    gy=to_host(gy), dgu=to_host(dgu), dx=to_host(dx), dwu=to_host(dwu),
                    dwd=to_host(dwd), sp=to_host(r.slot_pos))

    plain_rows = T * k
    rp = moe.moe_route_layout(to_dev(idx), to_dev(w), E, max_rows=plain_rows)
    a_rows = moe.moe_route_layout_rows(T, E, k, 0, False, 64)
    ra = moe.moe_route_layout(to_dev(idx), to_dev(w), E, alignment=64, max_rows=a_rows)
    p, a = chain(rp, plain_rows), chain(ra, a_rows)
    assert (to_host(ra.offsets) % 64 == 0).all()
    # the same token slot lands on row sp_plain[t,j] and row sp_aligned[t,j]
    sp_p, sp_a = p["sp"].ravel(), a["sp"].ravel()
    for name in ("y", "gu", "hid", "dgu", "dx"):
        assert (p[name][sp_p] == a[name][sp_a]).all(), name
    for name, P, Q in (("dwu", "xp", "dgu"), ("dwd", "hid", "gy")):
        Pf, Qf = _f(p[P][sp_p]), _f(p[Q][sp_p])
        e_of = idx.ravel()
        diff = np.abs(p[name].astype(np.float64) - a[name].astype(np.float64))
        for e in range(E):
            rows_e = e_of == e
            bound = 8 * max(rows_e.sum(), 1) * 2.0 ** -24 * (np.abs(Pf[rows_e]).T @ np.abs(Qf[rows_e]))
            assert (diff[e] <= bound + 1e-30).all(), (name, e)


def test_invalid_offsets_are_reported_and_writes_stay_in_bounds():
    """Offsets past the buffer or decreasing: every call reports
    MOE_ERR_DEVICE_CHECK and no row outside the buffers is written (the
    outputs are views into larger buffers whose guard rows must survive)."""
    rng = np.random.default_rng(31)
    N, H, I, E = 256, 256, 128, 3
    bad = to_dev(np.array([0, 100, 400, 300], np.int32))   # past N, then decreasing
    x = to_dev(wl.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32)))
    up = to_dev(wl.f32_to_bf16_bits((rng.standard_normal((E, H, 2 * I)) * 0.05).astype(np.float32)))
    down = to_dev(wl.f32_to_bf16_bits((rng.standard_normal((E, I, H)) * 0.05).astype(np.float32)))
    up_p, down_p = moe.moe_grouped_swiglu_pack(up, down)
    guard = 64
    sentinel = 12345

    def big(cols):
        t = torch.full((N + guard, cols), sentinel, dtype=torch.int16, device="cuda")
        return t.view(torch.bfloat16)

    yb, hb, gb = big(H), big(I), big(2 * I)
    y, hid, gu = moe.moe_grouped_swiglu_save(x, up_p, down_p, bad, out=yb[:N], hidden=hb[:N],
                                             gate_up=gb[:N])
    assert moe.moe_workspace_status(y._moe_workspace) == 6
    dgb, dxb = big(2 * I), big(H)
    dgu, dx = moe.moe_grouped_swiglu_dgrad(x, up, down, bad, gu, dgate_up=dgb[:N], dx=dxb[:N])
    assert moe.moe_workspace_status(dx._moe_workspace) == 6
    dwu, dwd = moe.moe_grouped_swiglu_wgrad(x, hid, x, dgu, bad)
    assert moe.moe_workspace_status(dwu._moe_workspace) == 6
    torch.cuda.synchronize()
    for b in (yb, hb, gb, dgb, dxb):
        assert (b.view(torch.int16)[N:] == sentinel).all()
    # pad-row fill with a negative offset writes nothing before the buffer
    rows = big(H)
    moe.moe_fill_pad_rows(rows[8:8 + 100], to_dev(np.array([-5, 10, 20], np.int32)),
                          to_dev(np.array([0, 3], np.int32)))
    torch.cuda.synchronize()
    assert (rows.view(torch.int16)[:8] == sentinel).all()
    assert (rows.view(torch.int16)[8 + 20:] == sentinel).all()
