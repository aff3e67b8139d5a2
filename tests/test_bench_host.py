"""bench.py's host-side logic without a GPU: the max-over-ranks timing and
whole-job value of the replica mode over two gloo ranks, the algorithmic byte
counts, clock parsing and the reference arm's rank gating."""
import os
import socket
import types

import pytest

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = 1.0 + rank                    # rank 1 is the slow replica
    m = bench.reduce_max(elapsed)
    v = bench.job_value(131072, world, 10, m)
    q.put((rank, m, v))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_report_the_slowest_rank_over_gloo():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [2.0, 2.0]
    # whole-job throughput: both ranks' units over the slowest rank's time
    assert got[0][2] == pytest.approx(131072 * 2 * 10 / 2.0)


def test_reduce_max_without_a_process_group_is_identity():
    assert bench.reduce_max(3.5) == 3.5


def test_algorithmic_bytes_at_the_deepseek_shape():
    a = bench.algorithmic_bytes(16384, 7168, 256, 8, 2)
    N = 16384 * 8
    assert a["permute"] == 16384 * 7168 * 2 + N * 7168 * 2 + 4 * N
    assert abs(a["permute"] / 1e6 - 2114.45) < 0.01
    assert abs(a["combine_backward"] / 1e6 - 3994.55) < 0.01
    assert a["combine"] - a["permute"] == 4 * N


def test_fp8_bytes_at_the_deepseek_shape():
    f = bench.fp8_bytes(16384, 7168, 8)
    T, H, N, nb = 16384, 7168, 16384 * 8, 56
    assert f["quantize_fp8"] == 3 * T * H + 4 * T * nb
    # the FP8 permute writes half the bf16 permute's row bytes
    bf = bench.algorithmic_bytes(T, H, 256, 8, 2)["permute"]
    assert f["permute"] < 0.52 * bf
    assert f["dequantize_fp8"] == 3 * N * H + 4 * N * nb
    # fused: bf16 rows read once, e4m3 + scale rows written to every slot
    assert f["permute_quantize_fp8"] == 2 * T * H + N * H + 4 * N * nb + 4 * N
    assert f["permute_quantize_fp8"] < f["quantize_fp8"] + f["permute"]


def test_layout_bytes_count_only_kept_rows():
    T, H, k, b = 16384, 7168, 8, 2
    full = bench.algorithmic_bytes(T, H, 256, k, b)
    same = bench.layout_bytes(T, H, k, b, T * k, T * k)
    assert same == {n: full[n] for n in same}
    capped = bench.layout_bytes(T, H, k, b, 50000, 163840)
    assert capped["combine"] == 50000 * H * b + T * H * b + 8 * T * k
    assert capped["permute"] == T * H * b + 163840 * H * b + 4 * T * k
    sparse = bench.layout_bytes(T, H, k, b, 50000, 163840, live=9000)
    assert sparse["combine_backward"] == 9000 * H * b + 2 * 50000 * H * b + 12 * T * k
    assert sparse["combine"] == capped["combine"]


def test_vep_bytes_at_the_virtual_ep_shape():
    # 32768 routed rows of 4096 bf16 each way: 536.9 MB per direction
    assert abs(bench.vep_bytes(32768, 4096, 2, 512) / 1e6 - 536.9) < 0.1


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.out = ("0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
             "0, 1980, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active\n"
             "0, 2010, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    s = c.summary()
    assert s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_reference_arm_runs_on_rank_zero_only():
    args = types.SimpleNamespace(steps=1, warmup=3, ref_tokens=8)
    assert bench.run_reference(args, rank=1) is None


def test_recorded_traffic_is_void_for_a_changed_source(tmp_path, monkeypatch):
    d = bench.source_digest(*bench.KERNEL_SOURCES["combine_backward"])
    assert bench.recorded_traffic("combine_backward", "0" * 16) is None
    got = bench.recorded_traffic("combine_backward", d)
    assert got is None or got > 1e9


def test_parse_layout():
    assert bench.parse_layout(None) == {}
    assert bench.parse_layout("cf=1.25,pad") == {"cf": 1.25, "pad": True}
    assert bench.parse_layout("align=128") == {"align": 128}
    with pytest.raises(ValueError):
        bench.parse_layout("pad")
    with pytest.raises(ValueError):
        bench.parse_layout("bogus=1")
