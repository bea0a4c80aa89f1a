"""CCA prefill benchmark: global-aware pooling + fused core/local attention.

One step = one full prefill pass (cca_pool then cca_attn_fwd) over one batch
of synthetic inputs already resident in HBM.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mha32k|mha128k|gqa64k]
                  [--impl cca|reference] [--no-e2e] [--no-cpu-baseline] [--no-sweep]

Besides the headline workload, the default run times the 128K MHA workload, the
GQA 64K workload (with both GQA pooling modes) and the 12 points of the g x w
sweep, each over at least 10 timed steps and 0.3 s, each with the clock record
of its own timed region and the tensor peak that record selects.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (no data-path collective: batches are independent), so the
scaling is weak; the only collectives are the timing barrier and the
max-over-ranks of the elapsed time.  `--impl reference` times the fp64 CPU
oracle on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sparse_long_context_cca_gb300 import workloads as W  # noqa: E402

WORKLOADS = {"mha32k": W.MHA_32K, "mha128k": W.MHA_128K, "gqa64k": W.GQA_64K}
METRIC = "CCA prefill tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129e6


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
        tf = d.get("bf16_tflops")
        tfs = d.get("bf16_tflops_sustained", tf)
        if hbm and tf:
            return {"hbm_gbs": float(hbm), "bf16_tflops": float(tf),
                    "bf16_tflops_sustained": float(tfs)}, "measured"
    except (OSError, ValueError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(peaks, peak_src, clocks):
    """Dense bf16 peak for a kernel timed over a region with this clock record: the
    sustained (power-capped) figure when power capping was active in the region, else
    the burst figure."""
    if "sw_power_cap" in (clocks.get("reasons") or []):
        return peaks["bf16_tflops_sustained"], f"{peak_src} dense bf16 (sustained: power cap active in the timed region)"
    return peaks["bf16_tflops"], f"{peak_src} dense bf16 (burst)"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.25)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self, window=None):
        """Stop sampling; the clock summary over `window` (see summary)."""
        if self.proc is None:
            return self.summary(window)
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        return self.summary(window)

    def summary(self, window=None):
        """Clock summary over the samples taken inside `window` (host monotonic times
        bracketing one timed region).  When the region is shorter than the sampling
        interval and no sample falls inside it, the two samples around it are used."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in list(self.lines):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((t, float(parts[0]), float(parts[1]),
                             {n for n, v in zip(names, parts[4:8]) if v.lower().startswith("active")}))
            except ValueError:
                continue
        where = "whole measurement"
        if window is not None and rows:
            lo, hi = window
            inside = [r for r in rows if lo <= r[0] <= hi]
            if inside:
                rows, where = inside, "timed region"
            else:
                before = [r for r in rows if r[0] < lo][-1:]
                after = [r for r in rows if r[0] > hi][:1]
                rows, where = before + after, "samples bracketing the timed region"
        sm = [r[1] for r in rows]
        reasons = set().union(*[r[3] for r in rows]) if rows else set()
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in rows) if rows else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": where}


def kernel_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel_file: str, workload_key: str):
    """Per-launch DRAM bytes recorded from an ncu capture of this kernel source,
    or None when no capture exists for the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    sha = kernel_sha(kernel_file)
    for ln in lines:
        parts = ln.split()
        if len(parts) >= 4 and not ln.startswith("#") and parts[0] == workload_key and parts[1] == sha:
            return float(parts[2]) + float(parts[3])
    return None


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's elapsed time (the job's time); identity at world == 1."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(total_ms: float, steps: int, tokens_per_rank_step: int, world: int):
    """(ms per step, whole-job tokens/s): every rank processes its own batch each step."""
    ms_per_step = total_ms / steps
    return ms_per_step, tokens_per_rank_step * world / (ms_per_step / 1e3)


def nvtx_push(name: str):
    """Names the enclosed host region for a timeline profiler (NVTX); a no-op without one."""
    try:
        torch.cuda.nvtx.range_push(name)
    except Exception:
        pass


def nvtx_pop():
    try:
        torch.cuda.nvtx.range_pop()
    except Exception:
        pass


def time_steps(fn, steps, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    return start, end


def bench_config(wl, world):
    """The workload description both arms print as `config`."""
    return {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "N": wl.N, "d": wl.d,
            "g": wl.g, "w": wl.w, "global_batch": wl.B * world, "seq_len": wl.N,
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (%.0f MB of Q/K/V vs 129 MB), no flush" % (
                (wl.B * wl.Hq + 2 * wl.B * wl.Hkv) * wl.N * wl.d * 2 / 1e6)}


MIN_ROW_STEPS = 10
MIN_ROW_SECONDS = 0.3


def row_steps(est_ms: float) -> int:
    """Timed steps of a secondary row: at least MIN_ROW_STEPS and MIN_ROW_SECONDS (so that
    the row's own clock record holds several samples), at most 300."""
    return int(min(300, max(MIN_ROW_STEPS, -(-MIN_ROW_SECONDS * 1e3 // max(est_ms, 1e-3)))))


def run_cca(args, rank, world, local):
    from sparse_long_context_cca_gb300 import api
    from sparse_long_context_cca_gb300.inputs import make_qkv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    api.load_library()
    wl = WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()

    def measure(wl, steps, warmup, pool_mode=0):
        """Times `steps` prefill steps (cca_pool + cca_attn_fwd) after `warmup` untimed ones.
        steps=None picks the count from the warm-up's own timing (row_steps).  Returns
        (total ms, mean pooling ms, mean attention ms, steps, host window)."""
        Q, K, V = make_qkv(wl, dev)
        G = wl.N // wl.g
        Kc = torch.empty((wl.B, wl.Hkv, G, wl.d), dtype=Q.dtype, device=dev)
        Vc = torch.empty_like(Kc)
        O = torch.empty_like(Q)
        LSE = torch.empty((wl.B, wl.Hq, wl.N), dtype=torch.float32, device=dev)

        def step(e=None):
            if e is not None:
                e[0].record(stream)
            api.cca_pool(Q, K, V, wl.g, Kc, Vc, stream=stream, pool_mode=pool_mode)
            if e is not None:
                e[1].record(stream)
            api.cca_attn_fwd(Q, K, V, Kc, Vc, wl.g, wl.w, O, LSE, stream=stream)
            if e is not None:
                e[2].record(stream)

        w0 = torch.cuda.Event(enable_timing=True)
        w1 = torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for _ in range(warmup):
            step()
        w1.record(stream)
        torch.cuda.synchronize()
        if steps is None:
            steps = row_steps(w0.elapsed_time(w1) / max(1, warmup))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        h0 = time.monotonic()
        nvtx_push(f"timed prefill steps: {wl.name}")
        t0.record(stream)
        for k in range(steps):
            step(ev[k])
        t1.record(stream)
        nvtx_pop()
        torch.cuda.synchronize()
        h1 = time.monotonic()
        if world > 1:
            torch.distributed.barrier()
        total_ms = t0.elapsed_time(t1)
        pool_ms = [a.elapsed_time(b) for a, b, _ in ev]
        attn_ms = [b.elapsed_time(c) for _, b, c in ev]
        assert torch.isfinite(LSE).all()
        del Q, K, V, O, LSE, Kc, Vc
        torch.cuda.empty_cache()
        return total_ms, statistics.mean(pool_ms), statistics.mean(attn_ms), steps, (h0, h1)

    def row(wl, pool_mode=0, note=None):
        """One secondary workload with its own clock record and peak."""
        tot, pm, am, steps, win = measure(wl, None, 3, pool_mode)
        ck = sampler.summary(win)
        tp, tp_src = tensor_peak(peaks, peak_src, ck)
        flops, pbytes = W.attn_flops(wl), W.pool_bytes(wl)
        r = {"workload": wl.name, "steps": steps, "warmup": 3, "ms_per_step": tot / steps,
             "tokens_per_s": wl.B * wl.N / (tot / steps / 1e3),
             "attn_ms": am, "attn_eff_tflops": flops / (am / 1e3) / 1e12,
             "attn_frac": flops / (am / 1e3) / 1e12 / tp, "attn_peak": tp, "attn_peak_source": tp_src,
             "pool_ms": pm, "pool_gbs": pbytes / (pm / 1e3) / 1e9,
             "pool_frac": pbytes / (pm / 1e3) / 1e9 / peaks["hbm_gbs"],
             "attn_flops": flops, "pool_bytes": pbytes, "clocks": ck}
        if pool_mode:
            r["pool_mode"] = pool_mode
        if note:
            r["note"] = note
        return r

    sampler = ClockSampler(local)
    sampler.start()
    total_ms, pool_ms, attn_ms, _, window = measure(wl, args.steps, args.warmup)
    clocks = sampler.summary(window)
    tpeak, tpeak_src = tensor_peak(peaks, peak_src, clocks)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step, value = job_throughput(total_ms, args.steps, wl.B * wl.N, world)
    flops = W.attn_flops(wl)
    pbytes = W.pool_bytes(wl)
    attn_tflops = flops / (attn_ms / 1e3) / 1e12
    pool_gbs = pbytes / (pool_ms / 1e3) / 1e9
    kfile = os.path.join(ROOT, "sparse_long_context_cca_gb300", "csrc", "attn_tc.cu")
    pfile = os.path.join(ROOT, "sparse_long_context_cca_gb300", "csrc", "pool.cu")
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normal Q/K/V, 1% heavy-hitter keys)",
        "config": bench_config(wl, world),
        "attn_eff_tflops": attn_tflops,
        "attn_ms": attn_ms, "pool_ms": pool_ms,
        "pool_gbs": pool_gbs,
        "roofline": {"bound": "tensor", "kernel": "attn_bf16_tc_kernel", "achieved": attn_tflops,
                     "peak": tpeak, "unit": "TFLOP/s",
                     "frac": attn_tflops / tpeak,
                     "peak_source": tpeak_src,
                     "traffic": recorded_traffic(kfile, args.workload),
                     "algorithmic_unit": "4*d FLOP per (query, visible key, head): %.4g FLOP per launch" % flops},
        "pool_roofline": {"bound": "hbm", "kernel": "pool_kernel", "achieved": pool_gbs,
                          "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": pool_gbs / peaks["hbm_gbs"],
                          "peak_source": f"{peak_src} copy bandwidth",
                          "traffic": recorded_traffic(pfile, args.workload),
                          "algorithmic_bytes": pbytes},
        "clocks": clocks,
        "gpu_launches": 2 * args.steps,
    }
    if args.also_128k and wl is not W.MHA_128K:
        r = row(W.MHA_128K)
        r["attn_traffic"] = recorded_traffic(kfile, "mha128k")
        r["pool_traffic"] = recorded_traffic(pfile, "mha128k")
        out["mha128k"] = r
    if args.sweep:
        # the other synthetic workloads: GQA 64K (both GQA pooling modes) and the g x w sweep
        rows = [row(W.GQA_64K) if wl is not W.GQA_64K else None,
                row(W.GQA_64K, pool_mode=3, note="alternative GQA pooling: per-head softmax weights "
                                                 "averaged over the 4 heads sharing a KV head")]
        out["gqa64k"] = [x for x in rows if x is not None]
        out["sweep"] = [row(w3) for w3 in W.sweep()]
        # the tiny fp32 workload (the parity configuration): fp32 attention runs on CUDA cores
        # (a 1e-4 output tolerance rules out tf32 tensor cores); 256 tokens are launch-bound
        tot, pm, am, n, win = measure(W.TINY_F32, None, 3)
        out["tiny_f32"] = {"workload": W.TINY_F32.name, "steps": n, "warmup": 3, "us_per_step": tot / n * 1e3,
                           "tokens_per_s": W.TINY_F32.B * W.TINY_F32.N / (tot / n / 1e3),
                           "pool_us": pm * 1e3, "attn_us": am * 1e3, "clocks": sampler.summary(win),
                           "note": "fp32 on CUDA cores; at 256 tokens each kernel is bound by its launch"}
    if args.decode:
        out["decode"] = decode_bench(wl, dev, stream, 50, peaks)
        if args.also_128k and wl is not W.MHA_128K:
            out["decode_128k"] = decode_bench(W.MHA_128K, dev, stream, 50, peaks)
        out["decode_layers"] = decode_layers_bench(wl, dev, 16, 20, peaks)
        if args.also_128k and wl is not W.MHA_128K:
            out["decode_layers_128k"] = decode_layers_bench(W.MHA_128K, dev, 16, 20, peaks)
        if args.sweep and wl is not W.GQA_64K:
            # grouped-query decode: each CTA reads its KV head's rows once for the 4 query heads
            out["decode_gqa64k"] = decode_bench(W.GQA_64K, dev, stream, 50, peaks)
            out["decode_layers_gqa64k"] = decode_layers_bench(W.GQA_64K, dev, 16, 20, peaks)
    if args.backward:
        bw = backward_bench(wl, dev, stream, 10, peaks)
        bw["clocks"] = sampler.summary(bw.pop("window"))
        bp, bp_src = tensor_peak(peaks, peak_src, bw["clocks"])
        bw["frac"], bw["peak"], bw["peak_source"] = bw["eff_tflops"] / bp, bp, bp_src
        out["backward"] = bw
    if args.comparator:
        out["full_attention_comparator"] = comparator(wl, dev, stream, max(3, args.steps // 4), ms_per_step)
        # the same comparison at the other context lengths the pages compare (each against its
        # own CCA step time from the rows above)
        if "mha128k" in out:
            out["full_attention_comparator_128k"] = comparator(W.MHA_128K, dev, stream, 3,
                                                               out["mha128k"]["ms_per_step"])
        if out.get("gqa64k"):
            out["full_attention_comparator_gqa64k"] = comparator(W.GQA_64K, dev, stream, 3,
                                                                 out["gqa64k"][0]["ms_per_step"])
    sampler.stop()
    if not args.no_e2e:
        out["e2e"] = e2e(wl, dev, stream, max(3, args.steps // 2), world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    return out


def decode_bench(wl, dev, stream, iters, peaks):
    """One decoding step at the last position of the workload (the token that sees the
    most cores): cca_decode_fwd over the caches, timed with CUDA events."""
    from sparse_long_context_cca_gb300 import api
    from sparse_long_context_cca_gb300.inputs import make_qkv
    Q, K, V = make_qkv(wl, dev)
    Kc, Vc = api.cca_pool(Q, K, V, wl.g, stream=stream)
    pos = wl.N - 1
    q = Q[:, :, pos].contiguous()
    del Q
    O = torch.empty_like(q)
    LSE = torch.empty((wl.B, wl.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(api.decode_workspace_size(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, wl.g, wl.w, q.dtype),
                     dtype=torch.uint8, device=dev)
    # The caches of one step (49 MB at 32K) fit in the 129 MB L2, so every timed step
    # starts from a flushed L2: a 512 MB write on the same stream just before it, then a
    # read of another 512 MB, so that the L2 holds clean lines (as between two decode steps
    # of a model, which mostly read other layers' caches and weights) and the step's reads
    # do not also pay for writing back the flush's dirty lines.  Each step has its own pair
    # of events; the flush (about 0.16 ms) keeps the GPU busy while the host enqueues the
    # next step, so the pair measures the step on the device, not the host's launch overhead.
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    sweep = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    for _ in range(5):
        api.cca_decode_fwd(q, K, V, Kc, Vc, pos, wl.g, wl.w, O, LSE, ws, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    nvtx_push(f"timed decode steps: {wl.name}")
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            flush.fill_(1)
            torch.sum(sweep, 0, out=sink)
            e0.record(stream)
            api.cca_decode_fwd(q, K, V, Kc, Vc, pos, wl.g, wl.w, O, LSE, ws, stream=stream)
            e1.record(stream)
    nvtx_pop()
    torch.cuda.synchronize()
    step_us = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev)
    us = sum(step_us) / len(step_us)
    del flush, sweep, sink
    lo = max(0, pos - wl.w + 1)
    keys = lo // wl.g + (pos - lo + 1)
    e = 2 if wl.dtype == "bf16" else 4
    nbytes = wl.B * wl.Hkv * keys * 2 * wl.d * e + 2 * wl.B * wl.Hq * wl.d * e
    del K, V, Kc, Vc
    torch.cuda.empty_cache()
    return {"what": f"one decode step at position {pos} ({keys} visible keys per head), split-KV + combine",
            "us_per_step": us, "us_median": step_us[len(step_us) // 2], "steps": iters,
            "l2": "flushed before every step (512 MB write, then a 512 MB read so the L2 holds clean lines); "
                  "per-step CUDA events (1.024 us ticks)",
            "tokens_per_s": wl.B / (us * 1e-6),
            "gbs": nbytes / (us * 1e-6) / 1e9, "hbm_frac": nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
            "algorithmic_bytes": nbytes,
            "kernel_launches_per_step": api.decode_kernels(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, wl.g, wl.w, q.dtype, pos)}


def decode_layers_bench(wl, dev, n_layers, replays, peaks):
    """The decode step of a whole model's attention: the same position decoded through
    n_layers layers, each with its own caches, the 2 * n_layers launches captured in one
    CUDA graph and replayed.  A replay reads n_layers times the one-step bytes (790 MB at
    32K, 2.4 GB at 128K), far more than the L2 holds, so every layer's caches come from
    HBM as in a model; the graph removes the host's per-call cost, so the launches follow
    one another as closely as the stream allows."""
    from sparse_long_context_cca_gb300 import api
    pos = wl.N - 1
    e = 2 if wl.dtype == "bf16" else 4
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed + 7)
    G = wl.N // wl.g
    layers = []
    for _ in range(n_layers):
        # seeded random caches of the workload's shape (their values do not change the work)
        t = [torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).mul_(wl.d ** -0.25).to(dt)
             for shape in ((wl.B, wl.Hq, wl.d), (wl.B, wl.Hkv, wl.N, wl.d), (wl.B, wl.Hkv, wl.N, wl.d),
                           (wl.B, wl.Hkv, G, wl.d), (wl.B, wl.Hkv, G, wl.d))]
        q, K, V, Kc, Vc = t
        O = torch.empty_like(q)
        LSE = torch.empty((wl.B, wl.Hq), dtype=torch.float32, device=dev)
        ws = torch.empty(api.decode_workspace_size(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, wl.g, wl.w, dt),
                         dtype=torch.uint8, device=dev)
        layers.append((q, K, V, Kc, Vc, O, LSE, ws))
    for (q, K, V, Kc, Vc, O, LSE, ws) in layers:  # eager once: per-device setup outside the capture
        api.cca_decode_fwd(q, K, V, Kc, Vc, pos, wl.g, wl.w, O, LSE, ws)
    torch.cuda.synchronize()
    ref = [(O.clone(), LSE.clone()) for (_, _, _, _, _, O, LSE, _) in layers]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for (q, K, V, Kc, Vc, O, LSE, ws) in layers:
            api.cca_decode_fwd(q, K, V, Kc, Vc, pos, wl.g, wl.w, O, LSE, ws)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    same = all(torch.equal(O, r[0]) and torch.equal(LSE, r[1])
               for (_, _, _, _, _, O, LSE, _), r in zip(layers, ref))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
    cur = torch.cuda.current_stream()
    nvtx_push(f"timed decode graph replays ({n_layers} layers): {wl.name}")
    for e0, e1 in ev:
        e0.record(cur)
        graph.replay()
        e1.record(cur)
    nvtx_pop()
    torch.cuda.synchronize()
    rep_us = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev)
    us = rep_us[len(rep_us) // 2] / n_layers
    lo = max(0, pos - wl.w + 1)
    keys = lo // wl.g + (pos - lo + 1)
    nbytes = wl.B * wl.Hkv * keys * 2 * wl.d * e + 2 * wl.B * wl.Hq * wl.d * e
    del layers, ref, graph
    torch.cuda.empty_cache()
    return {"what": f"the decode step at position {pos} through {n_layers} layers, each with its own caches, "
                    f"captured as one CUDA graph ({2 * n_layers} launches) and replayed; per-layer figures",
            "us_per_layer": us, "replays": replays, "replay_us_median": rep_us[len(rep_us) // 2],
            "bytes_per_replay": nbytes * n_layers,
            "l2": "not flushed: a replay reads far more than the L2 holds, every layer's caches from HBM",
            "gbs": nbytes / (us * 1e-6) / 1e9, "hbm_frac": nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
            "replay_matches_eager_bitwise": same,
            "kernel_launches_per_layer": api.decode_kernels(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, wl.g, wl.w, dt, pos)}


def backward_bench(wl, dev, stream, iters, peaks):
    """Backward pass (dQ, dK, dV of sum(dO * O)) of the whole prefill step."""
    from sparse_long_context_cca_gb300 import api
    from sparse_long_context_cca_gb300.inputs import make_qkv
    Q, K, V = make_qkv(wl, dev)
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, wl.g, wl.w, stream=stream)
    dO = torch.randn(Q.shape, device=dev, generator=torch.Generator(device=dev).manual_seed(5)).to(Q.dtype)
    grads = api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, wl.g, wl.w, stream=stream)
    for _ in range(2):  # warm-up
        api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, wl.g, wl.w, dQ=grads[0], dK=grads[1], dV=grads[2],
                            stream=stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    nvtx_push(f"timed backward: {wl.name}")
    h0 = time.monotonic()
    e0.record(stream)
    for _ in range(iters):
        api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, wl.g, wl.w, dQ=grads[0], dK=grads[1], dV=grads[2],
                            stream=stream)
    e1.record(stream)
    nvtx_pop()
    torch.cuda.synchronize()
    h1 = time.monotonic()
    ms = e0.elapsed_time(e1) / iters
    flops = 2.5 * W.attn_flops(wl)
    del Q, K, V, O, LSE, Kc, Vc, dO, grads
    torch.cuda.empty_cache()
    eff = flops / (ms / 1e3) / 1e12
    return {"what": "backward of pooling + fused attention: tcgen05 dQ kernel, tcgen05 dK/dV kernel over the "
                    "core tiles, the pooling backward as per-token scalars (CUDA cores, fp32), then the "
                    "dK/dV kernel over the raw-token tiles adding the pooling terms as it writes each row",
            "ms": ms, "eff_tflops": eff,
            "frac_of_bf16_burst": eff / peaks["bf16_tflops"] if peaks.get("bf16_tflops") else None,
            "algorithmic_unit": "10*d FLOP per (query, visible key, head): q.k, dO.v, dQ, dK, dV",
            "kernel_launches": 4, "iterations": iters, "warmup": 3, "window": (h0, h1)}


def comparator(wl, dev, stream, steps, cca_ms_per_step):
    """Dense causal softmax attention over the same Q, K, V with the same kernel (g = 1,
    w = N), timed like the CCA step: the attention-level counterpart of the pages'
    CCA-versus-full-attention prefill comparison."""
    from sparse_long_context_cca_gb300 import api
    from sparse_long_context_cca_gb300.inputs import make_qkv
    Q, K, V = make_qkv(wl, dev)
    O = torch.empty_like(Q)
    LSE = torch.empty((wl.B, wl.Hq, wl.N), dtype=torch.float32, device=dev)
    for _ in range(2):
        api.causal_attention(Q, K, V, O=O, LSE=LSE, stream=stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        api.causal_attention(Q, K, V, O=O, LSE=LSE, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flops = 4.0 * wl.d * wl.N * (wl.N + 1) / 2 * wl.B * wl.Hq
    del Q, K, V, O, LSE
    torch.cuda.empty_cache()
    return {"what": "causal softmax attention over all N keys, same kernel (g=1, w=N)",
            "attn_ms": ms, "eff_tflops": flops / (ms / 1e3) / 1e12,
            "cca_speedup": ms / cca_ms_per_step,
            "note": "CCA step = pooling + fused attention; speed-up = full attention time / CCA step time"}


def e2e(wl, dev, stream, steps, world):
    """Same metric through the library's host-buffer entry point, cca_prefill_host: every
    step copies Q, K, V from pinned host memory, pools, attends and copies O and LSE back
    to pinned host memory; the library pipelines these over slices of KV heads."""
    from sparse_long_context_cca_gb300 import api
    from sparse_long_context_cca_gb300.inputs import make_qkv
    Qd, Kd, Vd = make_qkv(wl, dev)
    hQ, hK, hV = (t.cpu().pin_memory() for t in (Qd, Kd, Vd))
    del Qd, Kd, Vd
    torch.cuda.empty_cache()
    hO = torch.empty(hQ.shape, dtype=hQ.dtype).pin_memory()
    hL = torch.empty((wl.B, wl.Hq, wl.N), dtype=torch.float32).pin_memory()
    ws = torch.empty(api.prefill_host_workspace_size(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, wl.g, wl.w, hQ.dtype),
                     dtype=torch.uint8, device=dev)

    def step():
        api.cca_prefill_host(hQ, hK, hV, wl.g, wl.w, out=(hO, hL, None, None), workspace=ws, stream=stream)

    for _ in range(2):
        step()
    stream.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    stream.synchronize()
    dt = (time.perf_counter() - t0) / steps
    h2d = sum(t.numel() * t.element_size() for t in (hQ, hK, hV))
    d2h = hO.numel() * hO.element_size() + hL.numel() * 4
    del ws
    torch.cuda.empty_cache()
    return {"value": wl.B * wl.N * world / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3, "steps": steps,
            "api": "cca_prefill_host (copies pipelined with the kernels over 8 slices of KV heads)",
            "h2d_gbs": h2d / dt / 1e9, "d2h_gbs": d2h / dt / 1e9}


def oracle_sample(wl, seconds_budget, row_frac=1.0):
    """Times the fp64 oracle on whole heads of the workload (pooling of the head's
    KV head + attention of every row), as many heads as fit the budget.  With
    row_frac < 1 it times one head's pooling and an evenly spaced fraction of its
    rows instead, and scales the rows' time to the whole head.
    Returns (tokens/s scaled to all heads, threads, description)."""
    import oracle
    from sparse_long_context_cca_gb300.inputs import make_qkv
    small = wl.small(B=1, Hq=wl.Hq // wl.Hkv, Hkv=1)  # one KV head with its query heads
    Q, K, V = make_qkv(small, "cpu")
    q, k, v = oracle.widen(Q[:, :1]), oracle.widen(K), oracle.widen(V)
    stride = max(1, int(round(1.0 / row_frac))) if row_frac < 1.0 else 1
    if stride > 1:
        rows = [(0, 0, i) for i in range(stride // 2, wl.N, stride)]
        t0 = time.perf_counter()
        Kc, Vc = oracle.pool(oracle.widen(Q), k, v, wl.g)
        t1 = time.perf_counter()
        oracle.attn_rows(q, k, v, Kc, Vc, wl.g, wl.w, rows)
        t2 = time.perf_counter()
        per_head = (t1 - t0) + (t2 - t1) * wl.N / len(rows)
        step_seconds = per_head * wl.B * wl.Hq
        desc = (f"pooling of one KV head of {wl.name} and 1 in {stride} of its {wl.N} rows for one query "
                f"head ({len(rows)} rows, {t2 - t0:.2f} s), rows scaled to the head, the head to {wl.B * wl.Hq} heads")
        return wl.B * wl.N / step_seconds, oracle.threads(), desc, step_seconds
    heads_done = 0
    t_used = 0.0
    while True:
        t0 = time.perf_counter()
        Kc, Vc = oracle.pool(oracle.widen(Q), k, v, wl.g)
        oracle.attn(q, k, v, Kc, Vc, wl.g, wl.w)
        t_used += time.perf_counter() - t0
        heads_done += 1
        if t_used >= seconds_budget or heads_done >= wl.B * wl.Hq:
            break
    per_head = t_used / heads_done
    step_seconds = per_head * wl.B * wl.Hq
    desc = (f"{heads_done} whole head(s) of {wl.name} (pooling of its KV head + all {wl.N} rows), "
            f"{t_used:.1f} s, scaled by {wl.B * wl.Hq}/{heads_done} heads")
    return wl.B * wl.N / step_seconds, oracle.threads(), desc, step_seconds


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        outp = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in outp.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(wl, seconds):
    v, cores, desc, _ = oracle_sample(wl, seconds)
    return {"value": v, "unit": "tokens/s", "cores": cores, "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "kind": "oracle", "sample": desc}


def run_reference(args, rank, world):
    """The fp64 oracle on the host cores, on the same workload as the CUDA arm.  Each step
    times a bounded sample of the workload (whole heads, or a fraction of one head's rows
    when the run is long) and scales it to the whole workload: `value` is that scaled
    tokens/s, `ms_per_step` the wall time each sampled step really took, and
    `extrapolated_ms_per_step` the time the whole workload would take."""
    if rank != 0:
        return None
    wl = WORKLOADS[args.workload]
    # One whole head per step (~0.5 s on 16 cores at 32K) while the run stays near 100 steps;
    # beyond that each step samples a proportional fraction of a head's rows, so that the
    # run stays within about a minute.
    frac = min(1.0, 100.0 / max(1, args.steps + args.warmup))
    vals = []
    for _ in range(args.warmup):
        oracle_sample(wl, 0.0, frac)
    desc = cores = None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, cores, desc, _ = oracle_sample(wl, 0.0, frac)
        vals.append(v)
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "extrapolated_ms_per_step": wl.B * wl.N / value * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": bench_config(wl, world),
            "runs_on": "host CPU, rank 0 (the fp64 oracle)",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "cpu_model": cpu_model(),
                             "nproc": os.cpu_count(), "kind": "oracle",
                             "sample": "each step: " + desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1, help="GPUs of this node (one rank each under torchrun)")
    ap.add_argument("--steps", type=int, default=300, help="timed steps of the headline workload")
    ap.add_argument("--warmup", type=int, default=5, help="untimed steps before them (at least 3)")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="mha32k", help="the headline workload")
    ap.add_argument("--impl", choices=["cca", "reference"], default="cca",
                    help="cca: the library on the GPU; reference: the fp64 oracle on the host cores")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer (copies included) measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the oracle on the host")
    ap.add_argument("--no-128k", dest="also_128k", action="store_false", help="skip the 128K rows")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="host time budget of the oracle sample")
    ap.add_argument("--no-comparator", dest="comparator", action="store_false",
                    help="skip the dense causal attention comparison")
    ap.add_argument("--no-decode", dest="decode", action="store_false", help="skip the decode rows")
    ap.add_argument("--no-backward", dest="backward", action="store_false", help="skip the backward row")
    ap.add_argument("--heads", type=int, default=0, help="query heads of the workload (a head slice)")
    ap.add_argument("--batch", type=int, default=0, help="batch of the workload")
    ap.add_argument("--g", type=int, default=0, help="group size of the workload")
    ap.add_argument("--w", type=int, default=0, help="window of the workload")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false",
                    help="skip the GQA 64K rows (prefill and decode), the 12 g x w sweep points and the tiny fp32 row")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.heads or args.g or args.w or args.batch:
        # a slice or variant of the named workload (e.g. a head slice for a profiler run)
        base = WORKLOADS[args.workload]
        r = base.Hq // base.Hkv
        hq = args.heads or base.Hq
        if hq % r:
            ap.error(f"--heads must be a multiple of {r}")
        wl = base.small(B=args.batch or base.B, Hq=hq, Hkv=hq // r, g=args.g or base.g, w=args.w or base.w)
        wl = wl.small(name=f"{base.name.split(' ')[0]} B{wl.B} Hq{wl.Hq} Hkv{wl.Hkv} d{wl.d} N{wl.N} g{wl.g} w{wl.w}")
        if wl.N % wl.g:
            ap.error("N must be a multiple of g")
        args.workload = "custom"
        WORKLOADS["custom"] = wl
    rank, world, local = dist_env()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    out = run_cca(args, rank, world, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
