"""Host logic of the multi-rank benchmark path on CPU (gloo, world size 2):
ranks are independent replicas, the job time is the slowest rank's, and the
job throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [120.0, 180.0][rank]
    job_ms = bench.max_over_ranks(ms, world, torch.device("cpu"))
    per_step, value = bench.job_throughput(job_ms, 10, 32768, world)
    q.put((rank, job_ms, per_step, value, bench.dist_env()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job_ms, per_step, value, env in res:
        assert job_ms == 180.0
        assert per_step == pytest.approx(18.0)
        assert value == pytest.approx(2 * 32768 / 0.018)
        assert env == (rank, 2, 0)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(12.5, 1, torch.device("cpu")) == 12.5
    assert bench.job_throughput(100.0, 10, 1000, 1) == (10.0, pytest.approx(1000 / 0.01))


def test_clock_summary_uses_the_timed_region(monkeypatch):
    """The clock record covers the samples taken inside the timed region, or the two around
    it when the region is shorter than the sampling interval; throttle reasons are the union."""
    s = bench.ClockSampler(0)

    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            pass

    s.proc = FakeProc()
    monkeypatch.setattr(bench.time, "sleep", lambda _: None)
    row = "{}, 2070, 900.0, 0x0, Not Active, Not Active, {}, Not Active"
    s.lines = [(1.00, row.format(1500, "Not Active")), (1.05, row.format(2070, "Active")),
               (1.10, row.format(2060, "Not Active")), (1.20, row.format(1400, "Not Active"))]
    inside = s.stop((1.04, 1.11))
    assert inside["samples"] == 2 and inside["window"] == "timed region"
    assert inside["sm_mhz"] == 2065.0 and inside["reasons"] == ["sw_thermal_slowdown"]
    short = s.stop((1.06, 1.07))
    assert short["samples"] == 2 and short["window"] == "samples bracketing the timed region"
    assert short["sm_mhz"] == 2065.0
    assert s.stop(None)["samples"] == 4


def test_tensor_peak_follows_the_power_cap():
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    p, src = bench.tensor_peak(peaks, "fallback", {"reasons": ["sw_power_cap"]})
    assert p == 1700.0 and "sustained" in src
    p, src = bench.tensor_peak(peaks, "fallback", {"reasons": []})
    assert p == 1900.0 and "burst" in src


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the fp64 oracle on the host cores) prints one JSON line
    with the contract's keys, the same metric and unit as the CUDA arm, and an e2e object that
    moves no bytes."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    d = json.loads(lines[-1])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == bench.WORKLOADS["mha32k"].name
