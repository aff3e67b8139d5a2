"""Router backward (moe_route_backward) vs the CPU oracle through the C ABI:
every float bit-exact (both sides: double, slot-order sum, one rounding)."""
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
    moe.moe_device_status()


def _both(idx, w, g, E):
    got = to_host(moe.moe_route_backward(to_dev(idx), to_dev(w), to_dev(g), E))
    assert moe.moe_device_status() == 0
    return got, oracle.route_backward(idx, w, g, E)


@pytest.mark.parametrize("name", ["tiny", "mid", "skewed", "vep8", "layer"])
def test_route_backward_on_routed_workloads(name):
    d = wl.make(name)
    W = d["workload"]
    idx, w, _ = oracle.topk_softmax(d["logits"], W.k)      # the workload's routing
    g = np.random.default_rng(len(name)).standard_normal((W.T, W.k)).astype(np.float32)
    got, exp = _both(idx, w, g, W.E)
    assert got.view(np.uint32).tobytes() == exp.view(np.uint32).tobytes()


@pytest.mark.parametrize("T,E,k,empty", [
    (1, 8, 2, 0.0), (33, 7, 3, 0.0),        # ragged warp; E not a multiple of 4
    (1000, 64, 6, 0.3),                     # empty (-1) slots
    (257, 1024, 32, 0.0), (96, 5, 5, 0.0),  # k = E
    (500, 16, 1, 0.0)])                     # k = 1: all zero
def test_route_backward_edge_shapes(T, E, k, empty):
    idx, w = wl.random_routing(T + E + k, T, E, k, empty_frac=empty)
    g = np.random.default_rng(T).standard_normal((T, k)).astype(np.float32) * 10
    got, exp = _both(idx, w, g, E)
    assert got.view(np.uint32).tobytes() == exp.view(np.uint32).tobytes()


def test_route_backward_after_the_combine_backward():
    """grad_probs as a backward produces them (the oracle's own chain on the
    DeepSeek-shaped routing), given to both sides."""
    d = wl.make("skewed", T=2048, with_grad=True)
    W = d["workload"]
    o = oracle.route(d["logits"], W.k)
    n = int(o["offsets"][W.E])
    xp = oracle.permute(d["x"], o["sorted_indices"], n)
    _, gp, _ = oracle.combine_backward(d["grad_out"], xp, o["slot_pos"], o["topk_w"])
    gl = to_host(moe.moe_route_backward(to_dev(o["topk_idx"]), to_dev(o["topk_w"]), to_dev(gp),
                                        W.E))
    exp = oracle.route_backward(o["topk_idx"], o["topk_w"], gp, W.E)
    assert gl.view(np.uint32).tobytes() == exp.view(np.uint32).tobytes()


def test_route_backward_reports_bad_ids():
    idx = np.array([[0, 5], [1, 1], [2, -1], [3, 0]], np.int32)   # 5 >= E, a repeat
    w = np.full((4, 2), 0.5, np.float32)
    g = np.array([[1, 2], [3, 4], [5, 6], [7, 8]], np.float32)
    got = to_host(moe.moe_route_backward(to_dev(idx), to_dev(w), to_dev(g), 4))
    assert moe.moe_device_status() == 6
    assert moe.moe_device_status() == 0                          # reading clears it
    good = oracle.route_backward(idx[2:], w[2:], g[2:], 4)
    assert (got[2:] == good).all()
    assert got[0, 1:].tolist() == [0, 0, 0]                       # only the valid id
