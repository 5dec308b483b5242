"""The benchmark's multi-process path on the CPU: two gloo ranks, as torchrun would start them.

Every rank steps its own full parameter list (replicas), the job's time is the slowest rank's (a MAX all-reduce),
and the job's value counts every rank's parameters. The reference arm prints only on rank 0."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slow = bench.slowest_rank_ms(times[rank], dist, "cpu")
        out[rank] = (slow, bench.job_value(world, 1000, 10, slow))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_job_value():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, [1.5, 4.0], out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 4.0
    assert out[0][1] == pytest.approx(world * 1000 * 10 / 4.0e-3)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    wl = workloads.WORKLOADS["tiny"]

    class Args:
        steps, warmup, gpus = 1, 3, 2
    for rank, expect in (("1", ""), ("0", '"impl": "reference"')):
        monkeypatch.setenv("RANK", rank)
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(Args(), wl)
        assert (expect in buf.getvalue()) if expect else buf.getvalue() == ""


def test_hbm_peak_from_measured_peaks_file(tmp_path):
    """The roofline's denominator is read from the peaks record whatever its layout, else the fallback is used."""
    import bench
    cases = [({"hbm_gbs": 6781.0}, 6781.0), ({"hbm": {"copy_gbs": 6781.5}}, 6781.5),
             ({"peaks": {"hbm_copy_GBps": 6700}}, 6700.0), ({"hbm_tbs": 6.781}, 6781.0),
             ({"bf16_tflops": 1900.0, "hbm_gbs": 6790}, 6790.0), ({"bf16_tflops": 1900.0}, None), ({}, None)]
    for record, want in cases:
        p = tmp_path / "peaks.json"
        p.write_text(json.dumps(record))
        v, src = bench.hbm_peak(str(p))
        if want is None:
            assert src == "fallback" and v == bench.FALLBACK_HBM_GBS, record
        else:
            assert src == "measured" and abs(v - want) < 1e-6, (record, v)
    assert bench.hbm_peak(str(tmp_path / "missing.json"))[1] == "fallback"


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """The roofline's DRAM traffic comes from the committed ncu summary only while that summary names the current
    AdamW kernel source by its hash; any other hash, a missing figure or a missing file gives null."""
    import bench
    monkeypatch.chdir(ROOT)
    sha = bench.kernel_source_sha()
    assert len(sha) == 16 and int(sha, 16) >= 0 and sha == bench.kernel_source_sha()
    p = tmp_path / "profile.md"
    monkeypatch.setattr(bench, "PROFILE", str(p))
    p.write_text(f"kernel_source_sha256_16: {sha}\n\ndram_bytes_per_launch_full_size: 3.4577e+09\n")
    assert bench.profiled_traffic() == 3.4577e9
    other = ("0" if sha[0] != "0" else "1") + sha[1:]
    p.write_text(f"kernel_source_sha256_16: {other}\n\ndram_bytes_per_launch_full_size: 3.4577e+09\n")
    assert bench.profiled_traffic() is None
    p.write_text(f"kernel_source_sha256_16: {sha}\n")
    assert bench.profiled_traffic() is None
    monkeypatch.setattr(bench, "PROFILE", str(tmp_path / "missing.md"))
    assert bench.profiled_traffic() is None


def test_byte_model_of_every_benchmarked_step():
    """The bytes per parameter the benchmark's GB/s and roofline fractions are computed from, for each step it times:
    AdamW reads w, g, m, v and writes w, m, v (28 B with float32 moments, 20 packed, 24 with m packed alone; 26 with
    binary16 gradients), plus the norm's read of g; with the norm fused into the gradient's add, that kernel reads g
    and a and writes g instead (12 B) and the norm reads nothing more; SGD moves w and g (and its buffer)."""
    import dataclasses
    import bench
    import workloads
    W = workloads.WORKLOADS
    small = W["gpt2_small"]
    assert bench.adamw_bytes_per_param(small) == 28 and bench.step_bytes_per_param(small) == 32
    assert bench.adamw_bytes_per_param(W["gpt2_small_bf16"]) == 20 and bench.step_bytes_per_param(W["gpt2_xl"]) == 24
    assert bench.adamw_bytes_per_param(dataclasses.replace(small, moments="bf16x2_m")) == 24
    assert bench.adamw_bytes_per_param(W["fp16_scaled"]) == 26 and bench.step_bytes_per_param(W["fp16_scaled"]) == 28
    assert bench.step_bytes_per_param(small, zero_grad=True) == 36
    assert bench.step_bytes_per_param(small, opt="accumulate") == 12 + 28
    assert bench.step_bytes_per_param(W["fp16_scaled"], opt="accumulate") == 6 + 26
    assert bench.adamw_bytes_per_param(small, opt="sgd") == 12 and bench.adamw_bytes_per_param(small, opt="momentum") == 20
