"""bench.py's host logic: rank aggregation under gloo (world size 2) and helpers."""

import json
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


def test_profiled_traffic_requires_a_current_record(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    path = tmp_path / "profiles" / (bench.PROFILE_RECORDS["bf16"] + ".json")
    assert bench.profiled_traffic(32) is None
    rec = {"source_path": "decode", "source_sha256_16": bench.kernel_source_hash("decode"),
           "dram_bytes_per_launch_full_batch": 1000}
    path.write_text(json.dumps(rec))
    assert bench.profiled_traffic(32) == 1000 and bench.profiled_traffic(8) == 250
    path.write_text(json.dumps(dict(rec, source_sha256_16="0000000000000000")))
    assert bench.profiled_traffic(32) is None
    # a record of the prefill sources does not stand for the decode kernel
    path.write_text(json.dumps(dict(rec, source_path="prefill",
                                    source_sha256_16=bench.kernel_source_hash("prefill"))))
    assert bench.profiled_traffic(32) is None


def test_committed_records_are_machine_written():
    """Every profiles/*.json has the fields --record-profile writes."""
    import glob
    for f in glob.glob(os.path.join(bench.ROOT, "profiles", "*.json")):
        rec = json.load(open(f))
        for key in ("profile", "report", "command", "source_path", "source_sha256_16",
                    "launches", "dram_bytes_per_launch", "dram_bytes_per_launch_full_batch"):
            assert key in rec, (f, key)
        assert rec["source_path"] in bench.SOURCE_SETS


def test_peak_falls_back_when_no_measurement(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    v, src = bench.measured_hbm_peak()
    assert v == bench.FALLBACK_HBM_GBS and src.startswith("fallback")


def test_prefill_profile_hashes_cover_their_kernels():
    """The E4M3 prefill kernel and the per-row top-k live in their own headers:
    a change there must invalidate their profiles and not the bf16 prefill one."""
    assert "prefill_fp8.cuh" in bench.PREFILL_FP8_SOURCES
    assert "prefill_fp8.cuh" not in bench.PREFILL_SOURCES
    assert "rows_topk.cuh" in bench.ROWS_TOPK_SOURCES
    assert "rows_topk.cuh" not in bench.PREFILL_SOURCES
    hashes = {p: bench.kernel_source_hash(p) for p in bench.SOURCE_SETS}
    assert len(set(hashes.values())) == len(hashes)
