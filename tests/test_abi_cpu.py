"""libmoe's C ABI without a GPU: the library builds and loads, exports every
entry point include/moe.h declares, and its host-side validation rejects bad
arguments before anything is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import unpermute_combine_gb300 as moe
from unpermute_combine_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return moe.load_library()


def declared_symbols():
    names = set()
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert "moe_route" in names and "moe_combine_backward" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    assert moe.moe_abi_version() == 2
    assert moe.moe_status_string(0) == "MOE_OK"
    assert moe.moe_status_string(6) == "MOE_ERR_DEVICE_CHECK"
    assert moe.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_chunk_idxs_host_helper_matches_oracle(lib):
    for R, L in [(2, 2), (8, 8), (3, 5), (1, 7)]:
        for inv in (False, True):
            assert moe.moe_chunk_idxs(R, L, inv) == oracle.chunk_idxs(R, L, inv).tolist()


def test_workspace_sizes(lib):
    a = moe.moe_route_workspace_size(16384, 256, 8)
    assert a % 256 == 0 and a >= 256 + 128 * 257 * 4
    assert moe.moe_route_workspace_size(0, 8, 2) >= 256
    assert moe.moe_sort_chunks_workspace_size(64) >= 256 + 4 * (2 * 65 + 64)


def _status(fn, *args):
    return fn(*args)


def test_host_validation_rejects_before_launch(lib):
    sz = ctypes.c_size_t()
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: validation fails first
    # k > E, k > 32, E > 1024, negative T
    assert lib.moe_route_workspace_size(10, 4, 5, ctypes.byref(sz)) == 2
    assert lib.moe_route_workspace_size(10, 64, 33, ctypes.byref(sz)) == 2
    assert lib.moe_route_workspace_size(10, 2048, 2, ctypes.byref(sz)) == 2
    assert lib.moe_route_workspace_size(-1, 8, 2, ctypes.byref(sz)) == 1
    assert lib.moe_route_workspace_size(10, 8, 2, None) == 1
    # missing outputs
    assert lib.moe_route(fake, 10, 8, 2, fake, fake, None, fake, fake, fake, fake, fake, None,
                         fake, 1 << 20, None) == 1
    # misaligned / too small workspace
    assert lib.moe_route(fake, 10, 8, 2, fake, fake, fake, fake, fake, fake, fake, fake, None,
                         P(0x1004), 1 << 20, None) == 3
    assert lib.moe_route(fake, 10, 8, 2, fake, fake, fake, fake, fake, fake, fake, fake, None,
                         P(0x1000), 16, None) == 3
    # bad dtype, bad k, null pointers
    assert lib.moe_permute(fake, 7, 10, 16, 2, 20, fake, fake, None) == 1
    assert lib.moe_permute(fake, 1, 10, 16, 33, 330, fake, fake, None) == 2
    assert lib.moe_permute(None, 1, 10, 16, 2, 20, fake, fake, None) == 1
    assert lib.moe_permute(fake, 1, 10, 16, 2, -1, fake, fake, None) == 1
    assert lib.moe_combine(fake, 1, 10, 16, 0, 20, fake, None, fake, None) == 1
    assert lib.moe_combine_backward(fake, fake, 1, 10, 16, 2, 20, fake, None, fake, None,
                                    None) == 1
    assert lib.moe_sort_chunks(fake, 1, 10, 16, fake, fake, 0, fake, fake, 1 << 20, None) == 1
    assert lib.moe_sort_chunks(fake, 1, 10, 16, fake, fake, 4, fake, P(0x1001), 1 << 20,
                               None) == 3
    assert lib.moe_chunk_idxs(0, 4, 0, None) == 1
    assert lib.moe_expert_scale(fake, 1, 10, 16, 0, fake, fake, fake, None) == 1
    assert lib.moe_workspace_status(P(0x1003), None) == 3
    # FP8: block sizes, divisibility and alignment
    assert lib.moe_quantize_fp8(fake, 4, 256, 48, fake, fake, None) == 2
    assert lib.moe_quantize_fp8(fake, 4, 200, 128, fake, fake, None) == 1
    assert lib.moe_quantize_fp8(P(0x1008), 4, 256, 128, fake, fake, None) == 1
    assert lib.moe_quantize_fp8(fake, 4, 256, 128, P(0x1004), fake, None) == 1
    assert lib.moe_dequantize_fp8(fake, fake, 4, 256, 128, P(0x1008), None) == 1
    assert lib.moe_dequantize_fp8(None, None, 0, 256, 128, None, None) == 0
    assert lib.moe_permute_fp8(fake, fake, 4, 256, 100, 2, 8, fake, fake, fake, None) == 2
    assert lib.moe_permute_fp8(fake, fake, 4, 200, 128, 2, 8, fake, fake, fake, None) == 1
    assert lib.moe_permute_fp8(fake, None, 4, 256, 128, 2, 8, fake, fake, fake, None) == 1
    assert lib.moe_permute_fp8(fake, fake, 4, 256, 128, 33, 8, fake, fake, fake, None) == 2
    assert lib.moe_permute_fp8(None, None, 0, 256, 128, 2, 0, None, None, None, None) == 0
    # router backward
    assert lib.moe_route_backward(fake, fake, fake, 10, 4, 5, fake, None) == 1
    assert lib.moe_route_backward(fake, fake, fake, 10, 2048, 2, fake, None) == 2
    assert lib.moe_route_backward(fake, fake, fake, 10, 64, 33, fake, None) == 2
    assert lib.moe_route_backward(fake, None, fake, 10, 8, 2, fake, None) == 1
    assert lib.moe_route_backward(None, None, None, 0, 8, 2, None, None) == 0
    # empty problems are valid no-ops and launch nothing
    assert lib.moe_permute(None, 1, 0, 16, 2, 0, None, None, None) == 0
    assert lib.moe_combine(None, 1, 0, 16, 2, 0, None, None, None, None) == 0
    assert lib.moe_combine(None, 1, 5, 0, 2, 10, fake, None, None, None) == 0
    # layout helpers are host-only
    assert lib.moe_route_layout_rows(100, 8, 2, 30, 1, 1, ctypes.byref(ctypes.c_int64())) == 0
    assert lib.moe_route_layout_rows(100, 8, 2, 0, 1, 1, ctypes.byref(ctypes.c_int64())) == 1
    cap = ctypes.c_int64()
    assert lib.moe_expert_capacity(1024, 2, 8, ctypes.c_double(1.25), ctypes.byref(cap)) == 0
    assert cap.value == 320


def test_binding_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        moe.moe_route(torch.zeros((4, 8)), 2)
    with pytest.raises(ValueError):
        moe.moe_combine(torch.zeros((8, 4)), torch.zeros((4, 2), dtype=torch.int32))


def test_timeout_selftest_validates_before_launch(lib):
    P = ctypes.c_void_p
    # no, misaligned or too small a workspace; a poll count of 0 or past the
    # pipelines' own limit (2^20)
    assert lib.moe_selftest_timeout(None, 256, 16, None) == 3
    assert lib.moe_selftest_timeout(P(0x1010), 256, 16, None) == 3
    assert lib.moe_selftest_timeout(P(0x1000), 128, 16, None) == 3
    assert lib.moe_selftest_timeout(P(0x1000), 256, 0, None) == 1
    assert lib.moe_selftest_timeout(P(0x1000), 256, (1 << 20) + 1, None) == 1


def test_permute_quantize_fp8_validates_before_launch(lib):
    P = ctypes.c_void_p
    f = P(0x1000)
    # block not 32/64/128/256; H not a multiple of block; k out of range;
    # H beyond one shared-memory stage; a missing or misaligned buffer
    assert lib.moe_permute_quantize_fp8(f, 4, 480, 48, 2, 8, f, f, f, None) == 2
    assert lib.moe_permute_quantize_fp8(f, 4, 200, 128, 2, 8, f, f, f, None) == 1
    assert lib.moe_permute_quantize_fp8(f, 4, 256, 128, 0, 8, f, f, f, None) == 1
    assert lib.moe_permute_quantize_fp8(f, 4, 256, 128, 33, 8, f, f, f, None) == 1
    assert lib.moe_permute_quantize_fp8(f, 4, 16384, 128, 2, 8, f, f, f, None) == 2
    assert lib.moe_permute_quantize_fp8(f, 4, 256, 128, 2, 8, None, f, f, None) == 1
    assert lib.moe_permute_quantize_fp8(P(0x1008), 4, 256, 128, 2, 8, f, f, f, None) == 1
    assert lib.moe_permute_quantize_fp8(f, 4, 256, 128, 2, 8, f, P(0x1008), f, None) == 1
    assert lib.moe_permute_quantize_fp8(f, 0, 256, 128, 2, 8, None, None, None, None) == 0


def test_grouped_swiglu_fp8_validates_before_launch(lib):
    """Shapes the FP8 expert FFN cannot take are refused on the host."""
    P = ctypes.c_void_p
    f = P(0x1000)                                      # never dereferenced
    ws = P(0x2000)
    big = ctypes.c_size_t(1 << 40)
    call = lib.moe_grouped_swiglu_fp8
    assert call(f, f, f, f, f, 64, 4, 256, 128, f, ws, big, None) == 2   # H not a multiple of 512
    assert call(f, f, f, f, f, 64, 4, 512, 100, f, ws, big, None) == 2   # I not a multiple of 128
    assert call(f, f, f, f, f, 64, 0, 512, 128, f, ws, big, None) == 1   # no experts
    assert call(f, None, f, f, f, 64, 4, 512, 128, f, ws, big, None) == 1
    assert call(f, f, f, f, f, 64, 4, 512, 128, f, None, big, None) == 3
    assert call(f, f, f, f, f, 64, 4, 512, 128, f, ws, 16, None) == 3
    assert call(f, P(0x1004), f, f, f, 64, 4, 512, 128, f, ws, big, None) == 1   # scales unaligned
