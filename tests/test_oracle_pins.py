"""Pins for the CPU oracle: the pages' worked examples, closed forms,
invariants and brute force on tiny inputs.  No GPU.  Each test is chosen so a
plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a wrong tie rule) fails it."""
import itertools
import math

import numpy as np
import pytest

import oracle
import workloads as wl


# ------------------------------------------------------------ worked examples

def test_dispatcher_worked_example(golden):
    g = golden("dispatcher_permute_example.json")
    T, E = g["num_tokens"], g["num_experts"]
    r = oracle.route_indices(np.array(g["topk_idx_k2"]), None, E)
    assert r["routing_map"].tolist() == g["routing_map"]
    assert r["routing_map"].T.tolist() == g["routing_map_T"]
    n = int(r["offsets"][E])
    assert r["sorted_indices"][:n].tolist() == g["sorted_indices"]
    assert (r["sorted_indices"][n:] == -1).all()
    # row t of tokens holds the value t in every column, so rows name tokens
    tokens = np.repeat(np.arange(T, dtype=np.float32)[:, None], 5, axis=1)
    permuted = oracle.permute(tokens, r["sorted_indices"], n)
    assert permuted[:, 0].astype(int).tolist() == g["permuted_input_token_rows"]
    assert r["counts"].tolist() == [2, 3, 2]
    assert r["group_list"].tolist() == [2, 5, 7]
    assert r["offsets"].tolist() == [0, 2, 5, 7]
    # token 3's second slot is empty
    assert r["slot_pos"][3, 1] == -1


def test_group_list_example(golden):
    g = golden("moe_ops_group_list.json")
    counts = g["tokens_per_expert"]
    experts = np.concatenate([np.full(c, e) for e, c in enumerate(counts)])
    rng = np.random.default_rng(3)
    rng.shuffle(experts)  # token order must not matter for the counts
    r = oracle.route_indices(experts[:, None].astype(np.int32), None, len(counts))
    assert r["counts"].tolist() == counts
    assert r["group_list"].tolist() == g["group_list"]
    seg = [[int(r["offsets"][e]), int(r["offsets"][e + 1])] for e in range(len(counts))]
    assert seg == g["segments"]


def test_k1_example(golden):
    g = golden("moe_ops_k1_example.json")
    ex = np.array(g["expert_of_token"], np.int32)[:, None]
    r = oracle.route_indices(ex, None, 2)
    order = [g["tokens"][t] for t in r["sorted_indices"]]
    assert order == g["expert_major_tokens"]


def _letters_to_rows(letters):
    return np.array([[ord(c)] * 3 for c in letters], np.float32)


def test_rank_major_example(golden):
    g = golden("moe_ops_rank_major.json")
    M = np.array(g["splits_rank_by_expert"], np.int32)
    R, L = M.shape
    rank_major = _letters_to_rows(g["rank_major"])
    fwd = oracle.chunk_idxs(R, L, inverse=False)
    em = oracle.sort_chunks(rank_major, M.ravel(), fwd)
    assert [chr(int(v)) for v in em[:, 0]] == g["expert_major"]
    # the permute indices of the page: expert-major row i came from rank-major row idx[i]
    idx = [g["rank_major"].index(c) for c in g["expert_major"]]
    assert idx == g["permute_indices"]
    assert M.sum(axis=0).tolist() == g["tokens_per_expert"]
    # unpermute with the transposed splits restores rank-major order
    inv = oracle.chunk_idxs(R, L, inverse=True)
    back = oracle.sort_chunks(em, M.T.ravel(), inv)
    assert [chr(int(v)) for v in back[:, 0]] == g["rank_major"]


def test_weighted_merge_example(golden):
    g = golden("moe_ops_weighted_merge.json")
    E, H = 4, 3
    out_1 = np.array([1.0, -2.0, 4.0], np.float32)
    out_3 = np.array([10.0, 20.0, -5.0], np.float32)
    topk = np.array([g["experts"]], np.int32)
    w = np.array([g["weights"]], np.float32)
    r = oracle.route_indices(topk, w, E)
    y = np.zeros((2, H), np.float32)
    y[r["slot_pos"][0, 0]] = out_1
    y[r["slot_pos"][0, 1]] = out_3
    out, out64 = oracle.combine(y, r["slot_pos"], w)
    expected = [0.7 * 1 + 0.3 * 10, 0.7 * -2 + 0.3 * 20, 0.7 * 4 + 0.3 * -5]   # 3.7, 4.6, 1.3
    np.testing.assert_allclose(out64[0], expected, rtol=1e-7)
    # the weights are float32 roundings of 0.7 and 0.3: allow a couple of float32 ulps
    np.testing.assert_allclose(out[0], np.array(expected, np.float32), rtol=3e-7)


# ------------------------------------------------------------- bf16 rounding

def test_bf16_rounding_matches_torch_for_float_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormals
        (rng.standard_normal(2000) * 1e37).astype(np.float32),
        np.array([0.0, -0.0, 3.3895314e38, 3.4e38, -3.4e38, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8],
                 np.float32),
    ])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_double(v.astype(np.float64))
    assert (got == ref).all()


def test_bf16_rounding_single_rounding_from_double():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: ties to even -> 1.0.
    # A hair above the midpoint must round up, although float32 would first
    # round it back onto the midpoint (the double-rounding trap).
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 3 * 2.0 ** -8,
                  -(1.0 + 2.0 ** -8 + 2.0 ** -40), 2.0 ** -133, 2.0 ** -134, 2.0 ** -134 * 3,
                  3.3961776e38, 1e300])
    got = oracle.bf16_from_double(v).tolist()
    assert got == [0x3F80, 0x3F81, 0x3F82, 0xBF81, 0x0001, 0x0000, 0x0002, 0x7F80, 0x7F80]


# -------------------------------------------------------------- top-k, softmax

def test_topk_brute_force_tiny():
    for seed in range(40):
        rng = np.random.default_rng(seed)
        T, E = int(rng.integers(1, 7)), int(rng.integers(1, 6))
        if seed % 2:
            logits = rng.integers(0, 3, (T, E)).astype(np.float32)     # many ties
        else:
            logits = rng.standard_normal((T, E)).astype(np.float32)
        for k in range(1, E + 1):
            idx, w, w64 = oracle.topk_softmax(logits, k)
            for t in range(T):
                chosen = idx[t].tolist()
                assert len(set(chosen)) == k
                # every chosen expert beats every other one: larger logit,
                # or an equal logit and a lower id
                for e in chosen:
                    for f in set(range(E)) - set(chosen):
                        assert (logits[t, e] > logits[t, f]) or (
                            logits[t, e] == logits[t, f] and e < f)
                # slots in descending logit order, equal logits by ascending id
                for a, b in zip(chosen, chosen[1:]):
                    assert (logits[t, a] > logits[t, b]) or (
                        logits[t, a] == logits[t, b] and a < b)
                # and the chosen set is the best of all k-subsets by that rule
                best = max(itertools.combinations(range(E), k),
                           key=lambda s: sorted(((logits[t, e], -e) for e in s), reverse=True))
                assert set(best) == set(chosen)


def test_softmax_closed_forms():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((64, 16)).astype(np.float32) * 3
    idx, w, w64 = oracle.topk_softmax(logits, 1)
    assert (w == 1.0).all()
    idx, w, w64 = oracle.topk_softmax(logits, 2)
    s = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
    sig = 1.0 / (1.0 + np.exp(-(s[:, 0] - s[:, 1])))       # 2-way softmax = logistic
    np.testing.assert_allclose(w64[:, 0], sig, rtol=1e-14)
    np.testing.assert_allclose(w64[:, 1], 1 - sig, rtol=1e-12, atol=1e-15)
    idx, w, w64 = oracle.topk_softmax(logits, 6)
    s = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
    np.testing.assert_allclose(w64.sum(axis=1), 1.0, rtol=1e-14)
    for a, b in [(0, 1), (2, 5), (1, 4)]:
        np.testing.assert_allclose(w64[:, a] / w64[:, b], np.exp(s[:, a] - s[:, b]), rtol=1e-12)
    assert (np.diff(w64, axis=1) <= 0).all()
    # shift invariance: adding a constant to a token's logits changes nothing
    idx2, w2, _ = oracle.topk_softmax(logits + np.float32(8), 6)
    assert (idx2 == idx).all()
    np.testing.assert_allclose(w2, w, atol=1e-6)


# ------------------------------------------------------------ router backward

def test_route_backward_hand_example():
    # w = (3/4, 1/4), g = (1, 0): sum w g = 3/4, grads 3/4*(1-3/4), 1/4*(0-3/4)
    # w = (1/2, 1/2), g = (2, -2): sum w g = 0, grads 1 and -1
    idx = np.array([[2, 0], [1, 3]], np.int32)
    w = np.array([[0.75, 0.25], [0.5, 0.5]], np.float32)
    g = np.array([[1.0, 0.0], [2.0, -2.0]], np.float32)
    got = oracle.route_backward(idx, w, g, 4)
    exp = np.array([[-0.1875, 0, 0.1875, 0], [0, 1, 0, -1]], np.float32)
    assert (got == exp).all()


def test_route_backward_matches_finite_differences_of_the_router():
    """d/ds of L = sum_j g_j w_j(s), with w from the oracle's own k-softmax."""
    rng = np.random.default_rng(41)
    T, E, k = 24, 12, 4
    # distinct logits 0.375 apart on a 2^-3 grid: s +- 2^-10 is exact and
    # keeps the selection and its order
    logits = np.stack([rng.permutation(E) * 0.375 - 2.0 for _ in range(T)]).astype(np.float32)
    g = rng.standard_normal((T, k)).astype(np.float32)
    idx, w, _ = oracle.topk_softmax(logits, k)
    grad = oracle.route_backward(idx, w, g, E)
    h = 2.0 ** -10

    def loss(lg):
        i2, _, w64 = oracle.topk_softmax(lg, k)
        assert (i2 == idx).all()
        return (w64 * g.astype(np.float64)).sum(axis=1)

    for e in range(E):
        lp, lm = logits.copy(), logits.copy()
        lp[:, e] += np.float32(h)
        lm[:, e] -= np.float32(h)
        fd = (loss(lp) - loss(lm)) / (2 * h)
        np.testing.assert_allclose(grad[:, e], fd, atol=2e-5)


def test_route_backward_invariants():
    rng = np.random.default_rng(42)
    T, E = 200, 64
    logits = rng.standard_normal((T, E)).astype(np.float32)
    for k in (1, 2, 8):
        idx, w, _ = oracle.topk_softmax(logits, k)
        g = rng.standard_normal((T, k)).astype(np.float32)
        grad = oracle.route_backward(idx, w, g, E)
        chosen = np.zeros((T, E), bool)
        np.put_along_axis(chosen, idx, True, axis=1)
        assert (grad[~chosen] == 0).all()                   # only chosen experts
        if k == 1:
            assert (grad == 0).all()                        # w = 1 identically
            continue
        # softmax is shift invariant: the gradient sums to zero over a token
        scale = np.abs(w * g).sum(axis=1)
        assert (np.abs(grad.sum(axis=1)) <= 1e-6 * scale + 1e-30).all()
        if k == 2:
            # logistic closed form w1 w2 (g1 - g2), which assumes w1 + w2 = 1;
            # the float weights miss that by an ulp, hence the scaled bound
            a = np.take_along_axis(grad, idx, axis=1)
            w0, w1 = w[:, 0].astype(np.float64), w[:, 1].astype(np.float64)
            g0, g1 = g[:, 0].astype(np.float64), g[:, 1].astype(np.float64)
            ref = w0 * w1 * (g0 - g1)
            bound = 1e-6 * w0 * (np.abs(g0) + np.abs(g1)) + 1e-30
            assert (np.abs(a[:, 0] - ref) <= bound).all()
            assert (np.abs(a[:, 1] + ref) <= bound).all()
    # equal upstream gradients carry no signal through a softmax
    idx, w, _ = oracle.topk_softmax(logits, 8)
    grad = oracle.route_backward(idx, w, np.full((T, 8), 3.0, np.float32), E)
    assert np.abs(grad).max() <= 3e-6


def test_route_backward_empty_slots_and_bad_ids():
    idx = np.array([[1, -1, 0]], np.int32)
    w = np.array([[0.5, 0.0, 0.5]], np.float32)
    g = np.array([[1.0, 7.0, 3.0]], np.float32)
    got = oracle.route_backward(idx, w, g, 3)
    # sum w g = 0.5 + 1.5 = 2 over the valid slots: expert 1 gets 0.5*(1-2),
    # expert 0 gets 0.5*(3-2), expert 2 (the empty slot's) nothing
    assert (got == np.array([[0.5, -0.5, 0.0]], np.float32)).all()
    for bad in ([[1, 3, 0]], [[1, 1, 0]], [[1, -2, 0]]):
        with pytest.raises(ValueError):
            oracle.route_backward(np.array(bad, np.int32), w, g, 3)


def test_grouped_topk_with_all_groups_is_plain_topk():
    rng = np.random.default_rng(21)
    logits = rng.standard_normal((50, 24)).astype(np.float32)
    for n_groups in (1, 2, 3, 4, 6, 8, 24):
        idx, w, _ = oracle.topk_softmax_grouped(logits, 5, n_groups, n_groups)
        idx0, w0, _ = oracle.topk_softmax(logits, 5)
        assert (idx == idx0).all() and (w == w0).all()


def test_grouped_topk_brute_force_tiny():
    for seed in range(30):
        rng = np.random.default_rng(400 + seed)
        n_groups = int(rng.integers(2, 5))
        gsize = int(rng.integers(1, 4))
        E = n_groups * gsize
        G = int(rng.integers(1, n_groups + 1))
        k = int(rng.integers(1, G * gsize + 1))
        T = 4
        if seed % 2:
            logits = rng.integers(0, 3, (T, E)).astype(np.float32)      # ties
        else:
            logits = rng.standard_normal((T, E)).astype(np.float32)
        idx, w, w64 = oracle.topk_softmax_grouped(logits, k, n_groups, G)
        for t in range(T):
            score = [max(logits[t, g * gsize:(g + 1) * gsize]) for g in range(n_groups)]
            # the kept groups: the best G by (score desc, id asc), over all G-subsets
            best = max(itertools.combinations(range(n_groups), G),
                       key=lambda s: sorted(((score[g], -g) for g in s), reverse=True))
            allowed = [e for e in range(E) if e // gsize in best]
            ref = sorted(allowed, key=lambda e: (-logits[t, e], e))[:k]
            assert idx[t].tolist() == ref
            np.testing.assert_allclose(w64[t].sum(), 1.0, rtol=1e-14)


def test_grouped_topk_rejects_bad_shapes():
    z = np.zeros((2, 12), np.float32)
    with pytest.raises(ValueError):
        oracle.topk_softmax_grouped(z, 2, 5, 2)      # 12 experts do not split into 5 groups
    with pytest.raises(ValueError):
        oracle.topk_softmax_grouped(z, 7, 4, 2)      # 2 groups of 3 cannot give 7 experts


def test_topk_rejects_bad_k():
    with pytest.raises(ValueError):
        oracle.topk_softmax(np.zeros((2, 4), np.float32), 5)


# ------------------------------------------------------------------- routing

def _brute_force_sorted(topk_idx, E):
    """Stable sort of all valid (expert, token) pairs, expert major."""
    pairs = sorted((int(e), t) for t, row in enumerate(topk_idx) for e in row if e >= 0)
    return [t for _, t in pairs]


def test_route_invariants_and_brute_force():
    for seed, (T, E, k, drop) in enumerate([(1, 1, 1, 0.0), (5, 4, 2, 0.0), (6, 5, 5, 0.0),
                                            (37, 9, 3, 0.2), (200, 16, 4, 0.1), (0, 3, 2, 0.0)]):
        idx, w = wl.random_routing(seed, T, E, k, drop)
        r = oracle.route_indices(idx, w, E)
        valid = idx >= 0
        n = int(valid.sum())
        assert r["counts"].sum() == n == r["offsets"][E] == (r["group_list"][-1] if E else 0)
        assert r["sorted_indices"][:n].tolist() == _brute_force_sorted(idx, E)
        assert (r["sorted_indices"][n:] == -1).all() and (r["permuted_probs"][n:] == 0).all()
        assert (r["routing_map"].sum(axis=1) == valid.sum(axis=1)).all()
        for t in range(T):
            for j in range(k):
                p = r["slot_pos"][t, j]
                if idx[t, j] < 0:
                    assert p == -1
                    continue
                e = idx[t, j]
                assert r["offsets"][e] <= p < r["offsets"][e + 1]
                assert r["sorted_indices"][p] == t
                assert r["permuted_probs"][p] == w[t, j]
        for e in range(E):
            seg = r["sorted_indices"][r["offsets"][e]:r["offsets"][e + 1]]
            assert (np.diff(seg) > 0).all()


def test_route_rejects_duplicates_and_bad_ids():
    with pytest.raises(ValueError):
        oracle.route_indices(np.array([[1, 1]], np.int32), None, 3)
    with pytest.raises(ValueError):
        oracle.route_indices(np.array([[0, 3]], np.int32), None, 3)


def test_route_all_tokens_one_expert():
    T, E = 50, 6
    r = oracle.route_indices(np.full((T, 1), 4, np.int32), None, E)
    assert r["counts"].tolist() == [0, 0, 0, 0, T, 0]
    assert r["sorted_indices"].tolist() == list(range(T))
    assert r["slot_pos"][:, 0].tolist() == list(range(T))


# ------------------------------------------------------------------ FP8

def test_e4m3_encoding_table():
    v = np.array([0.0, -0.0, 1.0, -1.0, 0.5, 448.0, 500.0, -1e9, 2.0 ** -6, 2.0 ** -9,
                  7 * 2.0 ** -9, 1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 240.0, 17.0, 18.0],
                 np.float32)
    got = oracle.e4m3_from_float(v).tolist()
    # 1.0625 is the midpoint of 1.0 and 1.125: ties to even -> 1.0 (0x38);
    # 1.1875 is the midpoint of 1.125 and 1.25 -> 1.25 (0x3A); 2^-10 ties to 0;
    # 3*2^-10 ties to 2*2^-10 -> 0x02; 17 ties 16|18 -> 16 (0x58); 500 saturates
    assert got == [0x00, 0x80, 0x38, 0xB8, 0x30, 0x7E, 0x7E, 0xFE, 0x08, 0x01, 0x07, 0x38,
                   0x3A, 0x00, 0x02, 0x77, 0x58, 0x59]


def test_e4m3_matches_torch_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8")
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(50000) * 30, rng.standard_normal(5000) * 1e-2,
                        rng.uniform(-448, 448, 5000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (oracle.e4m3_from_float(v) == ref).all()


def test_fp8_quantize_round_trip_bounds():
    x = wl.random_activation(6, (40, 512), "bf16")
    x[3, :128] = 0                                     # an all-zero block
    q, sc = oracle.quantize_fp8(x, 128)
    assert sc.shape == (40, 4) and sc[3, 0] == 1.0 and (q[3, :128] == 0).all()
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    amax = np.abs(xf.reshape(40, 4, 128)).max(axis=2)
    np.testing.assert_array_equal(sc[amax > 0], (amax[amax > 0] / 448.0).astype(np.float32))
    dq = wl.bf16_bits_to_f32(oracle.dequantize_fp8(q, sc, 128)).astype(np.float64)
    s = np.repeat(sc.astype(np.float64), 128, axis=1)
    # e4m3 keeps 4 significant bits: error <= 2^-4 relative, plus the
    # subnormal quantum 2^-9 * scale, plus the final bf16 rounding
    err = np.abs(dq - xf)
    assert (err <= np.abs(xf) * 2.0 ** -4 + s * 2.0 ** -10 + np.abs(dq) * 2.0 ** -8 + 1e-30).all()
    # the block maximum maps to +-448
    qa = np.abs(q.reshape(40, 4, 128).astype(np.int32) & 0x7F).max(axis=2)
    assert (qa[amax > 0] == 0x7E).all()


# ------------------------------------------------ capacity / padded layout

def test_capacity_worked_example(golden):
    g = golden("moe_ops_capacity.json")
    assert g["tokens_per_rank"] * g["top_k"] // g["num_experts"] == g["average_per_expert"]
    assert oracle.expert_capacity(g["tokens_per_rank"], g["top_k"], g["num_experts"],
                                  g["capacity_factor"]) == g["capacity"]
    assert oracle.expert_capacity(1000, 3, 7, 1.0) == 429          # ceil(428.57...)
    assert oracle.expert_capacity(100, 2, 8, 1.0) == 25


def test_layout_without_limits_is_the_plain_route():
    idx, w = wl.random_routing(31, 200, 12, 3, empty_frac=0.1)
    a = oracle.route_indices(idx, w, 12)
    b = oracle.route_layout(idx, w, 12, capacity=0, pad=False, alignment=1, max_rows=600)
    for name in ("counts", "offsets", "group_list", "sorted_indices", "slot_pos", "permuted_probs"):
        assert (a[name] == b[name]).all(), name


def test_layout_capacity_drops_the_latest_tokens():
    # all 10 tokens pick expert 2 first and expert 0 second; capacity 4
    idx = np.tile(np.array([[2, 0]], np.int32), (10, 1))
    w = np.tile(np.array([[0.75, 0.25]], np.float32), (10, 1))
    r = oracle.route_layout(idx, w, 3, capacity=4, pad=False, alignment=1, max_rows=20)
    assert r["counts"].tolist() == [4, 0, 4]
    assert r["offsets"].tolist() == [0, 4, 4, 8]
    assert r["sorted_indices"][:8].tolist() == [0, 1, 2, 3, 0, 1, 2, 3]
    assert (r["slot_pos"][4:] == -1).all()                 # tokens 4..9 dropped everywhere
    assert r["slot_pos"][:4, 0].tolist() == [4, 5, 6, 7] and r["slot_pos"][:4, 1].tolist() == [0, 1, 2, 3]


def test_layout_pad_and_alignment_segments():
    idx, w = wl.random_routing(32, 300, 8, 2)
    cap = oracle.expert_capacity(300, 2, 8, 1.25)
    p = oracle.route_layout(idx, w, 8, capacity=cap, pad=True)
    assert p["offsets"].tolist() == [e * cap for e in range(9)]
    a = oracle.route_layout(idx, w, 8, capacity=0, pad=False, alignment=128)
    assert (a["offsets"] % 128 == 0).all()
    assert (np.diff(a["offsets"]) >= a["counts"]).all() and (np.diff(a["offsets"]) - a["counts"] < 128).all()
    plain = oracle.route_indices(idx, w, 8)
    assert (a["counts"] == plain["counts"]).all()
    for lay in (p, a):
        n = int(lay["offsets"][-1])
        si = lay["sorted_indices"]
        for e in range(8):
            s0, c = lay["offsets"][e], lay["counts"][e]
            seg = si[s0:lay["offsets"][e + 1]]
            assert (np.diff(seg[:c]) > 0).all() and (seg[c:] == -1).all()
        assert (si[n:] == -1).all()
        sp = lay["slot_pos"]
        assert (si[sp[sp >= 0]] == np.nonzero(sp >= 0)[0]).all()


def test_layout_rejects_overflowing_rows():
    idx, w = wl.random_routing(33, 50, 4, 2)
    with pytest.raises(ValueError):
        oracle.route_layout(idx, w, 4, capacity=0, pad=False, alignment=64, max_rows=100)


# ------------------------------------------------------------------- combine

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_permute_then_combine_k1_is_identity(dtype):
    T, H, E = 33, 19, 5
    x = wl.random_activation(4, (T, H), dtype)
    idx, _ = wl.random_routing(5, T, E, 1)
    r = oracle.route_indices(idx, None, E)
    y = oracle.permute(x, r["sorted_indices"], T)
    out, _ = oracle.combine(y, r["slot_pos"], np.ones((T, 1), np.float32))
    assert out.tobytes() == x.tobytes()
    out2, _ = oracle.combine(y, r["slot_pos"], None)
    assert out2.tobytes() == x.tobytes()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_combine_equals_scatter_add_unpermute(dtype):
    T, H, E, k = 41, 24, 7, 3
    idx, w = wl.random_routing(6, T, E, k, empty_frac=0.15)
    r = oracle.route_indices(idx, w, E)
    n = int(r["offsets"][E])
    y = wl.random_activation(7, (T * k, H), dtype)
    out, out64 = oracle.combine(y, r["slot_pos"], w)
    out2, out2_64 = oracle.unpermute(y, r["sorted_indices"], r["permuted_probs"], T, n)
    np.testing.assert_allclose(out64, out2_64, rtol=1e-13, atol=1e-13)


def test_combine_stand_in_closed_form():
    d = wl.make("tiny")
    w_ = d["workload"]
    r = oracle.route(d["logits"], w_.k)
    n = int(r["offsets"][w_.E])
    xp = oracle.permute(d["x"], r["sorted_indices"], n)
    y = oracle.expert_scale(xp, r["offsets"], d["scale"])
    out, out64 = oracle.combine(y, r["slot_pos"], r["topk_w"])
    # stand-in expert e scales by (e+1)/E, so out[t] = x[t] * sum_j w_j (e_j+1)/E;
    # each y row is rounded to float32 once, hence a relative 2^-24 slack
    factor = (r["topk_w"].astype(np.float64) * (r["topk_idx"] + 1) / w_.E).sum(axis=1)
    np.testing.assert_allclose(out64, d["x"].astype(np.float64) * factor[:, None],
                               rtol=2.0 ** -23)


def test_combine_backward_exact_small_integers():
    # Dyadic inputs keep every product and sum exact in float32, so the
    # gradients can be checked against their definitions exactly.
    rng = np.random.default_rng(8)
    T, H, E, k = 9, 6, 5, 3
    idx, _ = wl.random_routing(9, T, E, k, empty_frac=0.2)
    w = (rng.integers(1, 16, (T, k)) / 16).astype(np.float32)
    r = oracle.route_indices(idx, w, E)
    y = rng.integers(-8, 9, (T * k, H)).astype(np.float32)
    g = rng.integers(-8, 9, (T, H)).astype(np.float32)
    sentinel = np.full_like(y, 777.0)
    gy, gp, gp64 = oracle.combine_backward(g, y, r["slot_pos"], w, grad_y_init=sentinel)
    for t in range(T):
        for j in range(k):
            p = r["slot_pos"][t, j]
            if p < 0:
                assert gp[t, j] == 0
                continue
            assert (gy[p] == w[t, j] * g[t]).all()
            assert gp[t, j] == float(np.dot(g[t].astype(np.float64), y[p]))
    n = int(r["offsets"][E])
    assert (gy[n:] == 777.0).all()


def test_combine_backward_is_the_adjoint():
    rng = np.random.default_rng(10)
    T, H, E, k = 64, 48, 8, 4
    idx, w = wl.random_routing(11, T, E, k, empty_frac=0.1)
    r = oracle.route_indices(idx, w, E)
    y = rng.standard_normal((T * k, H)).astype(np.float32)
    g = rng.standard_normal((T, H)).astype(np.float32)
    out, out64 = oracle.combine(y, r["slot_pos"], w)
    gy, gp, gp64 = oracle.combine_backward(g, y, r["slot_pos"], w)
    n = int(r["offsets"][E])
    lhs = float(np.sum(g.astype(np.float64) * out64))             # <g, C y>
    rhs = float(np.sum(gy[:n].astype(np.float64) * y[:n]))        # <C^T g, y>
    # grad_y rows are rounded to float32 once each: relative 2^-24 per term
    scale = float(np.sum(np.abs(gy[:n].astype(np.float64) * y[:n])))
    assert abs(lhs - rhs) <= 1e-6 * scale + 1e-9
    # d<g,out>/dw[t,j] = <g_t, y_p>, and out is linear in w
    assert abs(np.sum(gp64 * w) - lhs) <= 1e-9 * np.sum(np.abs(gp64 * w)) + 1e-12


def test_combine_backward_finite_difference_in_weights():
    rng = np.random.default_rng(12)
    T, H, E, k = 7, 10, 6, 3
    idx, w = wl.random_routing(13, T, E, k)
    r = oracle.route_indices(idx, w, E)
    y = rng.standard_normal((T * k, H)).astype(np.float32)
    g = rng.standard_normal((T, H)).astype(np.float32)
    _, gp, gp64 = oracle.combine_backward(g, y, r["slot_pos"], w)
    _, base = oracle.combine(y, r["slot_pos"], w)
    L0 = np.sum(g.astype(np.float64) * base)
    for t in range(T):
        for j in range(k):
            w2 = w.copy()
            w2[t, j] += np.float32(1.0)
            step = float(w2[t, j]) - float(w[t, j])   # the float32 step actually taken
            _, o2 = oracle.combine(y, r["slot_pos"], w2)
            # the loss is linear in w, so a finite step gives the derivative exactly
            slope = (np.sum(g.astype(np.float64) * o2) - L0) / step
            assert abs(slope - gp64[t, j]) <= 1e-9 * (1 + abs(slope))


def test_expert_scale_closed_form():
    x = wl.random_activation(14, (10, 4), "bf16")
    offsets = np.array([0, 3, 3, 10], np.int32)
    y = oracle.expert_scale(x, offsets, np.array([0.5, 4.0, 0.25], np.float32))
    xf = wl.bf16_bits_to_f32(x)
    yf = wl.bf16_bits_to_f32(y)
    assert (yf[:3] == xf[:3] * 0.5).all() and (yf[3:] == xf[3:] * 0.25).all()


# --------------------------------------------------------------- sort_chunks

def test_sort_chunks_round_trip_and_expert_major_brute_force():
    for seed, (R, L) in enumerate([(3, 4), (8, 8), (1, 5), (5, 1), (2, 7)]):
        rng = np.random.default_rng(100 + seed)
        M = rng.integers(0, 5, (R, L)).astype(np.int32)   # asymmetric in general
        M[0, 0] = 0                                        # an empty chunk
        N = int(M.sum())
        rows = np.arange(N * 3, dtype=np.float32).reshape(N, 3)
        em = oracle.sort_chunks(rows, M.ravel(), oracle.chunk_idxs(R, L, False))
        # brute force: rank-major blocks (r, l) in row order; expert-major
        # lists them local expert first, source rank second
        starts = np.concatenate([[0], np.cumsum(M.ravel())])
        block = {(r, l): rows[starts[r * L + l]:starts[r * L + l + 1]]
                 for r in range(R) for l in range(L)}
        expected = np.concatenate([block[(r, l)] for l in range(L) for r in range(R)])
        assert (em == expected).all()
        back = oracle.sort_chunks(em, M.T.ravel(), oracle.chunk_idxs(R, L, True))
        assert (back == rows).all()


def test_chunk_idxs_are_mutually_inverse():
    for R, L in [(2, 2), (8, 8), (3, 5)]:
        f = oracle.chunk_idxs(R, L, False)
        i = oracle.chunk_idxs(R, L, True)
        assert sorted(f.tolist()) == list(range(R * L))
        # position of chunk c in the forward order, read through the inverse order
        assert [int(f[v]) for v in i] == list(range(R * L)) or \
               [int(i[v]) for v in f] == list(range(R * L))


def test_sort_chunks_rejects_bad_splits():
    x = np.zeros((5, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.sort_chunks(x, np.array([2, 2], np.int32), np.array([1, 0], np.int32))
    with pytest.raises(ValueError):
        oracle.sort_chunks(x, np.array([2, 3], np.int32), np.array([1, 1], np.int32))


# ----------------------------------------------------------- grouped SwiGLU

def _numpy_swiglu(x_bits, up_bits, down_bits):
    x = wl.bf16_bits_to_f32(x_bits).astype(np.float64)
    up = wl.bf16_bits_to_f32(up_bits).astype(np.float64)
    down = wl.bf16_bits_to_f32(down_bits).astype(np.float64)
    I = up.shape[1] // 2
    gu = x @ up
    gate, u = gu[:, :I], gu[:, I:]
    h = gate / (1 + np.exp(-gate)) * u
    h = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(h.astype(np.float32))).astype(np.float64)
    return h @ down


def test_grouped_swiglu_reduces_to_dense_ffn():
    rng = np.random.default_rng(15)
    E, H, I = 3, 32, 24
    counts = [5, 0, 7]
    N = sum(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = wl.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    up = wl.f32_to_bf16_bits((rng.standard_normal((E, H, 2 * I)) * 0.2).astype(np.float32))
    down = wl.f32_to_bf16_bits((rng.standard_normal((E, I, H)) * 0.2).astype(np.float32))
    y, y64 = oracle.grouped_swiglu(x, up, down, offsets)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if a == b:
            continue
        ref = _numpy_swiglu(x[a:b], up[e], down[e])
        err = np.linalg.norm(y64[a:b] - ref) / np.linalg.norm(ref)
        assert err < 1e-3
    # sampled rows give the same values as the full computation
    ys, _ = oracle.grouped_swiglu(x, up, down, offsets, rows=np.array([11, 0, 6]))
    assert (ys[[11, 0, 6]] == y[[11, 0, 6]]).all()


# ------------------------------------------------- grouped SwiGLU backward

def _swiglu_case(seed=16):
    rng = np.random.default_rng(seed)
    E, H, I = 3, 24, 16
    counts = [6, 0, 9]
    N = sum(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = wl.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    up = wl.f32_to_bf16_bits((rng.standard_normal((E, H, 2 * I)) * 0.3).astype(np.float32))
    down = wl.f32_to_bf16_bits((rng.standard_normal((E, I, H)) * 0.3).astype(np.float32))
    dy = wl.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    y, y64, gu, hid = oracle.grouped_swiglu(x, up, down, offsets, save=True)
    return dict(E=E, H=H, I=I, N=N, offsets=offsets, x=x, up=up, down=down, dy=dy, y64=y64,
                gu=gu, hid=hid)


def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def test_forward_saves_the_stored_activations():
    c = _swiglu_case()
    gu, hid, I = _f64(c["gu"]), _f64(c["hid"]), c["I"]
    # hidden is silu(gate) * up of the unrounded gate_up; from the rounded
    # one it agrees to a few bf16 quanta
    ref = gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]
    assert np.abs(hid - ref).max() <= 2 ** -6 * np.abs(ref).max()


def test_swiglu_dgrad_matches_autograd():
    """dgate_up (before rounding) is the autograd gradient of
    sum(dy * (silu(gate)*up) @ w_down[e]) at the stored gate / up."""
    torch = pytest.importorskip("torch")
    c = _swiglu_case()
    dgu, dgu64, dx, dx64 = oracle.swiglu_dgrad(c["dy"], c["up"], c["down"], c["offsets"], c["gu"])
    I, off = c["I"], c["offsets"]
    for e in range(c["E"]):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        gu = torch.tensor(_f64(c["gu"][a:b]), requires_grad=True)
        h = torch.nn.functional.silu(gu[:, :I]) * gu[:, I:]
        y = h @ torch.tensor(_f64(c["down"][e]))
        (y * torch.tensor(_f64(c["dy"][a:b]))).sum().backward()
        np.testing.assert_allclose(dgu64[a:b], gu.grad.numpy(), rtol=1e-11, atol=1e-14)
    # the stored dgate_up is its bf16 rounding
    assert (dgu == wl.f32_to_bf16_bits(dgu64.astype(np.float32))).mean() > 0.99


def test_swiglu_dx_is_the_adjoint_of_gmm1():
    torch = pytest.importorskip("torch")
    c = _swiglu_case()
    dgu, _, dx, dx64 = oracle.swiglu_dgrad(c["dy"], c["up"], c["down"], c["offsets"], c["gu"])
    off = c["offsets"]
    xv = torch.zeros((c["N"], c["H"]), dtype=torch.float64, requires_grad=True)
    loss = 0
    for e in range(c["E"]):
        a, b = off[e], off[e + 1]
        loss = loss + (torch.tensor(_f64(dgu[a:b])) * (xv[a:b] @ torch.tensor(_f64(c["up"][e])))).sum()
    loss.backward()
    np.testing.assert_allclose(dx64, xv.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_swiglu_wgrad_up_matches_autograd():
    torch = pytest.importorskip("torch")
    c = _swiglu_case()
    dgu, *_ = oracle.swiglu_dgrad(c["dy"], c["up"], c["down"], c["offsets"], c["gu"])
    E, H, I, off = c["E"], c["H"], c["I"], c["offsets"]
    wv = torch.zeros((E, H, 2 * I), dtype=torch.float64, requires_grad=True)
    loss = 0
    for e in range(E):
        a, b = off[e], off[e + 1]
        loss = loss + (torch.tensor(_f64(dgu[a:b])) * (torch.tensor(_f64(c["x"][a:b])) @ wv[e])).sum()
    loss.backward()
    coords = np.array([(e, h, j) for e in range(E) for h in range(H) for j in range(2 * I)])
    got = oracle.swiglu_wgrad_at("up", coords, off, H, I, x=c["x"], dgate_up=dgu)
    np.testing.assert_allclose(got.reshape(E, H, 2 * I), wv.grad.numpy(), rtol=1e-12, atol=1e-14)
    assert (got.reshape(E, H, 2 * I)[1] == 0).all()                 # the empty expert


def test_swiglu_wgrad_down_by_exact_finite_differences():
    """y is linear in w_down at fixed hidden: changing one weight by delta
    changes sum(dy * y) by exactly delta * dW_down (up to double rounding)."""
    c = _swiglu_case()
    off, H, I = c["offsets"], c["H"], c["I"]
    base = (_f64(c["dy"]) * c["y64"]).sum()
    rng = np.random.default_rng(5)
    picks = [(e, int(rng.integers(I)), int(rng.integers(H))) for e in (0, 2) for _ in range(6)]
    got = oracle.swiglu_wgrad_at("down", picks, off, H, I, hidden=c["hid"], dy=c["dy"])
    for (e, i, h), g in zip(picks, got):
        down = c["down"].copy()
        old = wl.bf16_bits_to_f32(down[e, i, h:h + 1])[0]
        down[e, i, h] = wl.f32_to_bf16_bits(np.array([old + 0.5], np.float32))[0]
        delta = float(wl.bf16_bits_to_f32(down[e, i, h:h + 1])[0]) - float(old)
        _, y64 = oracle.grouped_swiglu(c["x"], c["up"], down, off)
        change = (_f64(c["dy"]) * y64).sum() - base
        assert change == pytest.approx(delta * g, rel=1e-9, abs=1e-12)
