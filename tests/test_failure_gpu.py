"""Failure detection on the GPU without a fault: a bounded wait on a barrier
that nothing completes gives up, the kernel returns with MOE_ERR_TIMEOUT in
its status word, and the context stays usable for ordinary calls."""
import time

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


@pytest.mark.parametrize("polls", [1, 1024])
def test_a_wait_that_runs_out_reports_timeout_and_returns(polls):
    ws = torch.zeros(moe.MOE_STATUS_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    t0 = time.monotonic()
    assert moe.moe_selftest_timeout(polls, workspace=ws) == 5          # MOE_ERR_TIMEOUT
    assert time.monotonic() - t0 < 30.0
    header = to_host(ws).view(np.uint32)
    assert header[0] == 5 and header[1] == polls                      # status, detail


def test_context_is_usable_after_a_timeout():
    assert moe.moe_selftest_timeout(256) == 5
    # ordinary calls afterwards: route + permute + combine, bit-exact vs the
    # oracle (the combine weights are the oracle's, given to both sides)
    d = wl.make("tiny")
    W = d["workload"]
    o = oracle.route(d["logits"], W.k)
    r = moe.moe_route(to_dev(d["logits"]), W.k)
    xp = moe.moe_permute(to_dev(d["x"]), r.slot_pos)
    out = to_host(moe.moe_combine(xp, r.slot_pos, to_dev(o["topk_w"])))
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert (to_host(r.slot_pos) == o["slot_pos"]).all()
    xp_o = oracle.permute(d["x"], o["sorted_indices"], int(o["offsets"][W.E]))
    assert to_host(xp).tobytes() == xp_o.tobytes()
    ref, _ = oracle.combine(xp_o, o["slot_pos"], o["topk_w"])
    assert out.tobytes() == ref.tobytes()
