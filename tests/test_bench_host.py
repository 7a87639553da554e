"""bench.py's host logic: rank aggregation under gloo (world size 2) and helpers."""

import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    got = bench.max_over_ranks(dist, 1.5 + rank)
    bench.barrier(dist)
    out.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=5) for _ in range(2))
    assert results == [(0, 2.5), (1, 2.5)]


def test_single_rank_needs_no_process_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.0) == 3.0


def test_clock_sampler_parses_nvidia_smi_rows():
    s = bench.ClockSampler(None)

    class FakeProc:
        def terminate(self):
            pass

        def communicate(self, timeout=None):
            rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
                    "0, 1980, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active"]
            return "\n".join(rows), ""

    s.proc = FakeProc()
    c = s.stop()
    assert c["samples"] == 2 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]


def test_profiled_traffic_requires_a_current_summary(tmp_path, monkeypatch):
    path = tmp_path / "summary.md"
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", {"bf16": str(path)})
    assert bench.profiled_traffic(32) is None
    path.write_text(f"source_sha256_16: {bench.kernel_source_hash()}\n"
                    "dram_bytes_per_launch_full_batch: 1000\n")
    assert bench.profiled_traffic(32) == 1000
    path.write_text("source_sha256_16: 0000000000000000\ndram_bytes_per_launch_full_batch: 1000\n")
    assert bench.profiled_traffic(32) is None


def test_peak_falls_back_when_no_measurement(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    v, src = bench.measured_hbm_peak()
    assert v == bench.FALLBACK_HBM_GBS and src.startswith("fallback")


def test_fp8_prefill_profile_hash_covers_its_kernel():
    """The fp8 prefill kernel lives in its own header: a change there must
    invalidate its profile and not the bf16 prefill one."""
    assert "prefill_fp8.cuh" in bench.PREFILL_FP8_SOURCES
    assert "prefill_fp8.cuh" not in bench.PREFILL_SOURCES
    assert bench.kernel_source_hash("prefill_fp8") != bench.kernel_source_hash("prefill")
    assert bench.kernel_source_hash("prefill") != bench.kernel_source_hash("decode")
