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


def test_route_variants_validate_before_launch(lib):
    """moe_route_grouped, moe_route_indices, moe_route_layout and
    moe_fill_pad_rows refuse bad groups, sizes, pointers and workspaces on
    the host."""
    P = ctypes.c_void_p
    f = P(0x1000)                                      # never dereferenced
    ws = P(0x2000)
    big = ctypes.c_size_t(1 << 40)

    def grouped(E, k, g, kg, counts=f, ws_=ws, nbytes=big):
        return lib.moe_route_grouped(f, 64, E, k, g, kg, f, f, counts, f, f, f, f, f, None,
                                     ws_, nbytes, None)
    assert grouped(64, 2, 0, 1) == 1                   # no groups
    assert grouped(64, 2, 8, 9) == 1                   # more kept groups than groups
    assert grouped(10, 2, 4, 2) == 1                   # E not a multiple of the groups
    assert grouped(128, 2, 64, 4) == 2                 # more than 32 groups
    assert grouped(64, 9, 8, 1) == 1                   # k above the kept groups' experts
    assert grouped(64, 2, 8, 4, counts=None) == 1
    assert grouped(64, 2, 8, 4, ws_=None) == 3
    assert grouped(64, 2, 8, 4, ws_=P(0x2010)) == 3    # workspace not 256-byte aligned
    assert grouped(64, 2, 8, 4, nbytes=16) == 3

    def indices(E, k, idx=f, w=f, probs=f, counts=f, ws_=ws):
        return lib.moe_route_indices(idx, w, 64, E, k, counts, f, f, f, f, probs, None,
                                     ws_, big, None)
    assert indices(4, 5) == 2                          # k > E
    assert indices(0, 1) == 1
    assert indices(8, 2, counts=None) == 1
    assert indices(8, 2, idx=None) == 1
    assert indices(8, 2, w=None) == 1                  # permuted_probs without weights
    assert indices(8, 2, ws_=P(0x2080)) == 3

    def layout(cap, pad, align, max_rows=256, E=8, sorted_=f, slot=f, nbytes=big):
        return lib.moe_route_layout(f, f, 64, E, 2, cap, pad, align, max_rows, f, f, f,
                                    sorted_, slot, f, ws, nbytes, None)
    assert layout(0, 0, 0) == 1                        # alignment below 1
    assert layout(0, 1, 1) == 1                        # padding needs a capacity
    assert layout(-1, 0, 1) == 1
    assert layout(16, 1, 1, max_rows=-1) == 1
    assert layout(1 << 21, 1, 1, E=1024) == 2          # E * capacity rows >= 2^31
    assert layout(16, 1, 1, sorted_=None) == 1
    assert layout(16, 1, 1, slot=None) == 1
    assert layout(16, 1, 1, nbytes=16) == 3

    def fill(dtype, max_rows, H, E, rows=f, offsets=f):
        return lib.moe_fill_pad_rows(rows, dtype, max_rows, H, offsets, f, E, None)
    assert fill(3, 64, 16, 4) == 1                     # no such dtype
    assert fill(1, 64, 16, 0) == 1
    assert fill(1, 64, 16, 1025) == 2
    assert fill(1, 64, 16, 4, offsets=None) == 1
    assert fill(1, 64, 16, 4, rows=None) == 1
    assert fill(1, 0, 16, 4, rows=None) == 0           # nothing to fill: no launch
    assert fill(2, 64, 0, 4, rows=None) == 0


def test_grouped_swiglu_family_validates_before_launch(lib):
    """The grouped SwiGLU forward, its pack, save, dgrad and wgrad refuse
    shapes the tensor-core tiles cannot take, missing or unaligned buffers and
    short workspaces on the host; the workspace size is the status header
    plus the bf16 hidden rows."""
    P = ctypes.c_void_p
    f = P(0x1000)                                      # never dereferenced
    odd = P(0x1008)                                    # not 16-byte aligned
    ws = P(0x2000)
    big = ctypes.c_size_t(1 << 40)
    sz = ctypes.c_size_t()
    size = lib.moe_grouped_swiglu_workspace_size
    assert size(64, 4, 256, 128, ctypes.byref(sz)) == 0 and sz.value == 256 + 64 * 128 * 2
    assert size(0, 4, 256, 128, ctypes.byref(sz)) == 0 and sz.value == 256 + 256
    assert size(64, 4, 128, 128, ctypes.byref(sz)) == 2      # H not a multiple of 256
    assert size(64, 4, 256, 64, ctypes.byref(sz)) == 2       # I not a multiple of 128
    assert size(64, 0, 256, 128, ctypes.byref(sz)) == 1
    assert size(64, 1025, 256, 128, ctypes.byref(sz)) == 2
    assert size(-1, 4, 256, 128, ctypes.byref(sz)) == 1
    assert size(1 << 31, 4, 256, 128, ctypes.byref(sz)) == 2
    assert size(64, 4, 256, 128, None) == 1

    fwd = lib.moe_grouped_swiglu
    assert fwd(f, f, f, None, 64, 4, 256, 128, f, ws, big, None) == 1    # no offsets
    assert fwd(None, f, f, f, 64, 4, 256, 128, f, ws, big, None) == 1
    assert fwd(f, f, f, f, 64, 4, 256, 128, f, None, big, None) == 3
    assert fwd(f, f, f, f, 64, 4, 256, 128, f, P(0x2010), big, None) == 3
    assert fwd(f, f, f, f, 64, 4, 256, 128, f, ws, 16640 - 1, None) == 3
    assert fwd(odd, f, f, f, 64, 4, 256, 128, f, ws, big, None) == 1

    pack = lib.moe_grouped_swiglu_pack
    assert pack(f, f, 0, 256, 128, f, f, None) == 1
    assert pack(f, f, 4, 100, 128, f, f, None) == 2
    assert pack(None, f, 4, 256, 128, f, f, None) == 1

    save = lib.moe_grouped_swiglu_save
    assert save(f, f, f, f, 64, 4, 256, 128, f, None, f, ws, big, None) == 1   # no hidden
    assert save(f, f, f, f, 64, 4, 256, 128, f, f, f, None, big, None) == 3
    assert save(f, f, f, f, 64, 4, 256, 128, f, f, f, ws, 16, None) == 3
    assert save(f, f, f, f, 64, 4, 256, 128, f, f, odd, ws, big, None) == 1

    dgrad = lib.moe_grouped_swiglu_dgrad
    assert dgrad(f, f, f, f, f, 64, 4, 256, 128, f, None, ws, big, None) == 1   # no dx
    assert dgrad(f, f, f, f, f, 64, 4, 256, 128, f, f, None, big, None) == 3
    assert dgrad(odd, f, f, f, f, 64, 4, 256, 128, f, f, ws, big, None) == 1

    wgrad = lib.moe_grouped_swiglu_wgrad
    assert wgrad(f, f, f, f, None, 64, 4, 256, 128, f, f, ws, big, None) == 1  # no offsets
    assert wgrad(None, f, f, f, f, 64, 4, 256, 128, f, None, ws, big, None) == 1
    assert wgrad(f, f, None, f, f, 64, 4, 256, 128, None, f, ws, big, None) == 1
    assert wgrad(f, f, f, f, f, 64, 4, 256, 128, f, f, None, big, None) == 3
    assert wgrad(f, f, f, f, f, 64, 4, 256, 128, P(0x1004), None, ws, big, None) == 1
