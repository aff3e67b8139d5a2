"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace -- a plugin living inside a
fixed, pre-reserved memory budget with no allocator of its own, or code that
must not call cudaMalloc because it can synchronise the device.  For them
moe_route_noalloc uses a scratch array built into the library.  These tests
call it through the C ABI (ctypes, raw device pointers) twice in a row and
check that it gives exactly what moe_route gives with a workspace.  The file
is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import unpermute_combine_gb300 as moe  # noqa: E402

MOE_OK, MOE_ERR_UNSUPPORTED = 0, 2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from unpermute_combine_gb300 import build
    build.build()
    return moe.load_library()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(lib, logits, k, stream):
    T, E = logits.shape
    dev = logits.device
    out = {
        "topk_idx": torch.full((T, k), -7, dtype=torch.int32, device=dev),
        "topk_w": torch.full((T, k), -7.0, dtype=torch.float32, device=dev),
        "counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
        "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        "group_list": torch.full((E,), -7, dtype=torch.int32, device=dev),
        "sorted_indices": torch.full((T * k,), -7, dtype=torch.int32, device=dev),
        "slot_pos": torch.full((T, k), -7, dtype=torch.int32, device=dev),
        "permuted_probs": torch.full((T * k,), -7.0, dtype=torch.float32, device=dev),
        "routing_map": torch.full((T, E), 7, dtype=torch.uint8, device=dev),
    }
    rc = lib.moe_route_noalloc(
        _p(logits), T, E, k, _p(out["topk_idx"]), _p(out["topk_w"]), _p(out["counts"]),
        _p(out["offsets"]), _p(out["group_list"]), _p(out["sorted_indices"]),
        _p(out["slot_pos"]), _p(out["permuted_probs"]), _p(out["routing_map"]),
        ctypes.c_void_p(stream.cuda_stream))
    return rc, out


def test_noalloc_route_matches_route_on_two_calls_in_a_row(lib):
    stream = torch.cuda.current_stream()
    # two different problems back to back: the second call reuses the
    # scratch the first one left behind
    # (40000 tokens: more than 256 token blocks, so the route runs its scan
    # kernel and keeps per-block prefixes in the shared array as well)
    for T, E, k, seed in [(16384, 256, 8, 11), (3001, 64, 6, 12), (16384, 256, 8, 13),
                          (40000, 256, 8, 14)]:
        g = np.random.default_rng(seed)
        logits = torch.from_numpy(g.standard_normal((T, E)).astype(np.float32)).cuda()
        rc, got = _call_noalloc(lib, logits, k, stream)
        assert rc == MOE_OK, moe.moe_status_string(rc)
        ref = moe.moe_route(logits, k, routing_map=True)
        torch.cuda.synchronize()
        for name in ("topk_idx", "counts", "offsets", "group_list", "sorted_indices",
                     "slot_pos", "routing_map"):
            assert torch.equal(got[name], getattr(ref, name)), name
        # same kernels on the same input: the weights agree to the last bit,
        # well inside the 1e-6 the routing tests allow
        assert (got["topk_w"] - ref.topk_w).abs().max().item() <= 1e-6
        assert (got["permuted_probs"] - ref.permuted_probs).abs().max().item() <= 1e-6


def test_noalloc_route_rejects_problems_beyond_its_scratch(lib):
    need = moe.moe_route_workspace_size(1 << 20, 1024, 8)
    assert need > moe.MOE_ROUTE_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x1000)   # never touched: the size check comes first
    rc = lib.moe_route_noalloc(fake, 1 << 20, 1024, 8, fake, fake, fake, fake, fake, fake,
                               fake, fake, None, None)
    assert rc == MOE_ERR_UNSUPPORTED
