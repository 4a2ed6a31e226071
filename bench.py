#!/usr/bin/env python
"""Benchmark of the fused exact attention forward on GB300.

One step = one pass of the hot path over one batch: ``fa_fwd`` on the headline
workload (B=8, H=32, Nq=Nk=2048, d=128, non-causal, bf16; seeded synthetic
N(0,1) inputs). Prints ONE JSON line (rank 0) with TFLOPS (4*B*H*Nq*Nk*d per
step, halved for causal), the roofline of the kernel against the measured
dense bf16 peak, the same metric end to end from pinned host buffers, SM
clocks sampled during the timed region, the float64 CPU oracle timed on a
bounded sample, and timings of the other workloads (causal, long sequence,
d=256, split-KV + combine sweep).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With ``--gpus N`` > 1 and no torchrun environment the script starts N ranks
itself; under ``torchrun`` WORLD_SIZE must equal N. Each rank runs the same
per-GPU workload (weak scaling, no data exchange: heads are independent);
timing takes the max over ranks.
``--impl reference`` times the float64 oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "exact_attention_80_gb300", "csrc")
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------------ distributed helpers

def dist_env():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend: str):
    import torch.distributed as dist

    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def dist_barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist

        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def dist_max(value: float, world: int, device=None) -> float:
    """Max of a float over ranks (the slowest rank sets the job time)."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(value: float, world: int, device=None) -> float:
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling); rank 0 keeps the base seed."""
    return base_seed + 7919 * rank


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampler around the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.6)  # nvidia-smi start-up

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        time.sleep(2 * self.period_ms / 1000.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        """Median SM clock under load: the samples drawing at least half the
        highest power seen (the sampled window also holds the sampler's start-up
        and the device sleep that queues the timed launches, both near idle).
        Throttle reasons from every sample."""
        rows, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx, pw = float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            rows.append((sm, pw))
            smax.append(mx)
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        peak_w = max(pw for _, pw in rows)
        loaded = [(sm, pw) for sm, pw in rows if pw >= 0.5 * peak_w]
        return {"sm_mhz": statistics.median(sm for sm, _ in loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_under_load": round(statistics.median(pw for _, pw in loaded), 1)}


# ------------------------------------------------------------------ helpers

def sustained_bf16_peak():
    """The measured bf16 GEMM rate held for seconds under the power cap, or None."""
    try:
        with open(PEAKS_FILE, encoding="utf-8") as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(PEAKS_FILE, encoding="utf-8") as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


# Sources that do not build or launch the forward kernels (the split merge, the
# allocation-free wrapper, the backward): a change there leaves their recorded
# DRAM traffic valid.
NOT_FORWARD = ("fa_combine.cu", "fa_noalloc.cu", "fa_bwd.cu")


def kernel_source_hash() -> str:
    """Hash of the sources of the forward kernels and their launch."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")) and name not in NOT_FORWARD:
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, only if it was taken
    on the current kernel sources (else None)."""
    try:
        with open(TRAFFIC_FILE, encoding="utf-8") as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    for e in rec.get("entries", []):
        if (e.get("kernel") == kernel and e.get("workload") == workload
                and e.get("source_hash") == kernel_source_hash()):
            return float(e["dram_bytes_per_launch"])
    return None


def kernel_name(fa, B: int, H: int, Nq: int, d: int, sms: int, Nk: int | None = None,
                causal: bool = False) -> str:
    """The forward kernel fa_fwd launches for this shape: the one-tile kernel at
    d = 256; at d = 64 and 128 the two-tile kernel, with persistent CTAs when its
    work units fill four waves of one CTA per SM and span at most 16 key tiles of
    128 (32 for non-causal d = 128) (include/fa.h, fa_fwd)."""
    if d == 256:
        return f"fa_fwd_tp_kernel<{d}>"
    key_tiles = -(-(Nq if Nk is None else Nk) // 128)
    short_units = key_tiles <= 16 or (d == 128 and not causal and key_tiles <= 32)
    if short_units and fa.fa_fwd_grid_ctas(B, H, Nq, d, 1) >= 4 * sms:
        return f"fa_fwd_tmp_kernel<{d}>"
    return f"fa_fwd_tm_kernel<{d}>"


def blas_threads():
    """The BLAS pool's thread count as threadpoolctl reports it, or None where
    threadpoolctl is not installed."""
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return None


def cpu_threads() -> int:
    return blas_threads() or os.cpu_count() or 1


def oracle_sample(cfg: dict, budget_s: float, seed: int, max_heads: int | None = None):
    """Time the float64 oracle over whole (b, h) heads of the workload until the
    budget is spent. Returns (tflops, heads, seconds)."""
    import oracle
    from exact_attention_80_gb300.inputs import f32, make_qkv, metric_flops, to_f64

    d = cfg["d"]
    q, k, v = make_qkv(1, 1, cfg["Nq"], cfg["Nk"], d, seed)
    qf, kf, vf = to_f64(q)[0, 0], to_f64(k)[0, 0], to_f64(v)[0, 0]
    scale = f32(1.0 / math.sqrt(d))
    heads, t0 = 0, time.perf_counter()
    while True:
        oracle.attention_f64(qf, kf, vf, scale, cfg["causal"])
        heads += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_heads is not None and heads >= max_heads):
            break
    flops = heads * metric_flops(1, 1, cfg["Nq"], cfg["Nk"], d, cfg["causal"])
    return flops / el / 1e12, heads, el


# ------------------------------------------------------------------ our arm

def time_launches(fn, steps: int, stream, queue_ahead: bool = False):
    """CUDA events bracketing every step on `stream`; returns per-step ms.

    With ``queue_ahead`` the stream first runs a device-side sleep long enough
    for the host to enqueue every step, so kernels shorter than the host's
    launch time run back to back and the events time the device work, not the
    gaps between launches."""
    import torch

    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    if queue_ahead:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(200_000 * steps)  # ~0.1 ms of SM cycles per step
    evs[0].record(stream)
    for i in range(steps):
        fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]


def time_alternating(fa_fn, fb_fn, steps: int, stream):
    """Per-launch ms of `fa_fn` and `fb_fn` run alternately (a, b, a, b, ...) in
    one sequence queued behind a device sleep, an event between every two
    launches; returns the two lists. A drift of the clock over the run then
    moves both alike, so their per-pair differences stay meaningful."""
    import torch

    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps + 1)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(400_000 * steps)
    evs[0].record(stream)
    for i in range(steps):
        fa_fn()
        evs[2 * i + 1].record(stream)
        fb_fn()
        evs[2 * i + 2].record(stream)
    torch.cuda.synchronize()
    ta = [evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(steps)]
    tb = [evs[2 * i + 1].elapsed_time(evs[2 * i + 2]) for i in range(steps)]
    return ta, tb


def time_back_to_back(fn, steps: int, stream) -> float:
    """Mean ms per call of `steps` calls queued behind a device sleep and
    bracketed by one pair of CUDA events (nothing between the calls)."""
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(200_000 * steps)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def spread_us(times_ms) -> dict:
    """Median, 10th and 90th percentile of per-launch times, in microseconds."""
    xs = sorted(times_ms)
    n = len(xs)

    def q(f):
        return round(xs[min(n - 1, int(f * (n - 1) + 0.5))] * 1e3, 1)

    return {"median_us": round(statistics.median(xs) * 1e3, 1), "p10_us": q(0.1), "p90_us": q(0.9)}


def fill_splits(fa, B, H, Nq, d, sms):
    """The largest split count whose split-KV grid still fits one CTA per SM."""
    best = 1
    for S in range(1, fa.FA_MAX_SPLITS + 1):
        if fa.fa_fwd_grid_ctas(B, H, Nq, d, S) <= sms:
            best = S
    return best


def device_qkv(c: dict, gen, device):
    """Seeded N(0,1) bf16 Q, K, V of workload ``c`` drawn on the device. A
    workload with ``outlier_frac`` (the large-head-dim one) gets the recipe of
    ``inputs.make_qkv`` on the device generator: per (b, h), floor(frac * Nk)
    distinct key rows chosen by a seeded permutation are scaled by 8 in fp32
    before the bf16 rounding."""
    import torch

    B, H, Nq, Nk, d = c["B"], c["H"], c["Nq"], c["Nk"], c["d"]
    gen.manual_seed(c["seed"])
    q = torch.randn((B, H, Nq, d), generator=gen, device=device)
    k = torch.randn((B, H, Nk, d), generator=gen, device=device)
    v = torch.randn((B, H, Nk, d), generator=gen, device=device)
    frac = c.get("outlier_frac", 0.0)
    if frac > 0.0:
        count = int(math.floor(frac * Nk))
        rows = torch.rand((B * H, Nk), generator=gen, device=device).argsort(dim=1)[:, :count]
        kh = k.view(B * H, Nk, d)
        kh.scatter_(1, rows[:, :, None].expand(-1, -1, d),
                    kh.gather(1, rows[:, :, None].expand(-1, -1, d)) * 8.0)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def extra_workloads(device, stream, reps: int = 20):
    """TFLOPS of the other benchmark workloads (seeded device-side N(0,1) bf16)."""
    import torch

    import exact_attention_80_gb300 as fa
    from exact_attention_80_gb300.inputs import CONFIGS, metric_flops

    out = {}
    gen = torch.Generator(device=device)
    # Chunked prefill against a key cache: 4096 new queries over 8192 keys with the
    # bottom-right causal mask (FLOPs from the visible pairs).
    configs = dict(CONFIGS)
    configs["prefill_bottom_right"] = dict(B=1, H=32, Nq=4096, Nk=8192, d=128,
                                           causal="bottom_right", seed=1006)
    for name in ("c1", "c2_causal", "c3", "c3_causal", "c4", "prefill_bottom_right", "c5"):
        c = configs[name]
        B, H, Nq, Nk, d, causal = c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["causal"]
        q, k, v = device_qkv(c, gen, device)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), device=device)
        flops = metric_flops(B, H, Nq, Nk, d, causal)
        if name != "c5":
            fn = lambda: fa.fa_fwd(q, k, v, o, lse, causal, stream=stream)  # noqa: E731
            for _ in range(3):
                fn()
            times = time_launches(fn, reps, stream, queue_ahead=True)
            ms = statistics.median(times)
            sp = spread_us(times)
            out[name] = {"tflops": round(flops / ms / 1e9, 1), "us": round(ms * 1e3, 1),
                         "p10_us": sp["p10_us"], "p90_us": sp["p90_us"]}
            if name == "c1":
                # A launch-bound call: also the mean over calls issued back to back
                # with no event between them (as a loop of small attention calls
                # runs), where one call's launch overlaps the previous one's end.
                out[name]["us_back_to_back"] = round(time_back_to_back(fn, 200, stream) * 1e3, 2)
            if c.get("outlier_frac"):
                out[name]["inputs"] = (f"N(0,1) bf16, {c['outlier_frac']:.0%} of K rows per head "
                                       "scaled x8 (seeded permutation)")
        else:
            sweep = {}
            # The printed split counts, plus the largest whose grid fits one CTA per SM.
            sms = torch.cuda.get_device_properties(device).multi_processor_count
            fill = fill_splits(fa, B, H, Nq, d, sms)
            for S in sorted({1, 2, 3, 4, 16, 64, fill}):
                ws = torch.empty(fa.fa_splitkv_workspace_bytes(B, H, Nq, d, S) // 4,
                                 device=device)
                f_split = lambda: fa.fa_fwd_splitkv(q, k, v, ws, S, causal, stream=stream)  # noqa
                f_comb = lambda: fa.fa_combine(ws, o, lse, B, H, Nq, d, S, stream=stream)  # noqa
                for _ in range(3):
                    f_split()
                    f_comb()
                t_c = time_launches(f_comb, reps, stream, queue_ahead=True)
                # The decode step as a caller runs it: split, then merge, back to
                # back (the merge's launch overlaps the split's tail), timed
                # alternately with the split alone.
                t_s, t_sc = time_alternating(f_split, lambda: (f_split(), f_comb()), reps, stream)
                ms_s, ms_c, ms_sc = (statistics.median(t) for t in (t_s, t_c, t_sc))
                ms_in_seq = statistics.median([b - a for a, b in zip(t_s, t_sc)])
                sp_sc = spread_us(t_sc)
                kv_bytes = 2 * B * H * Nk * d * 2 + 2 * B * H * Nq * d * 2
                part = S * B * H * Nq * (d + 2) * 4
                comb_bytes = part + B * H * Nq * (d * 2 + 4)
                sweep[str(S)] = {
                    "tflops": round(flops / (ms_s + ms_c) / 1e9, 1),
                    "split_us": round(ms_s * 1e3, 1), "combine_us": round(ms_c * 1e3, 1),
                    "split_gbs": round((kv_bytes + part) / ms_s / 1e6, 1),
                    "combine_gbs": round(comb_bytes / ms_c / 1e6, 1),
                    "split_then_combine_us": round(ms_sc * 1e3, 1),
                    "split_then_combine_p10_p90_us": [sp_sc["p10_us"], sp_sc["p90_us"]],
                    "combine_in_sequence_us": round(ms_in_seq * 1e3, 1),
                    "tflops_in_sequence": round(flops / ms_sc / 1e9, 1)}
            out[name] = sweep
        del q, k, v, o, lse
    out["c3_tile_sweep"] = tile_sweep(device, stream, reps)
    out["varlen_causal"] = varlen_workload(device, stream, reps)
    out["c2_fp8"] = fp8_workload(device, stream, reps)
    out["c4_fp8"] = fp8_workload(device, stream, reps, shape=(8, 16, 8191, 256), causal=True,
                                 seed=1011)
    out["c2_fp8_d64"] = fp8_workload(device, stream, reps, shape=(8, 32, 2048, 64), seed=1012)
    out["c5_fp8"] = fp8_decode_workload(device, stream, reps)
    out["c2_bwd"] = bwd_workload(device, stream, reps)
    out["c2_bwd_d64"] = bwd_workload(device, stream, reps, d=64)
    out["bwd_d256"] = bwd_workload(device, stream, reps, d=256, shape=(2, 16, 4096))
    return out


def tile_sweep(device, stream, reps):
    """The long-sequence workload (B=1, H=8, N=8192, d=128), both masks, at each
    query-tile size a CTA can own: 256 rows (two 128-row tiles, fa_fwd's
    choice), 128 rows (one tile, fa_fwd_rows) and 64 rows (one tile of M = 64
    MMAs, fa_fwd_rows)."""
    import torch

    import exact_attention_80_gb300 as fa
    from exact_attention_80_gb300.inputs import CONFIGS, metric_flops

    res = {}
    gen = torch.Generator(device=device)
    for name in ("c3", "c3_causal"):
        c = CONFIGS[name]
        B, H, Nq, Nk, d, causal = c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["causal"]
        q, k, v = device_qkv(c, gen, device)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), device=device)
        flops = metric_flops(B, H, Nq, Nk, d, causal)
        line = {}
        for rows in (256, 128, 64):
            fn = lambda: fa.fa_fwd_rows(q, k, v, o, lse, rows, causal, stream=stream)  # noqa: E731
            for _ in range(3):
                fn()
            ms = statistics.median(time_launches(fn, reps, stream, queue_ahead=True))
            line[f"rows_{rows}"] = {"tflops": round(flops / ms / 1e9, 1), "us": round(ms * 1e3, 1),
                                    "ctas": B * H * -(-Nq // rows)}
        res[name] = line
        del q, k, v, o, lse
    return res


def bwd_workload(device, stream, reps, d=128, shape=(8, 32, 2048)):
    """The backward (fa_bwd) on a (B, H, N) shape (default the C2 one) at head
    dim d, both masks, on seeded device-side N(0,1) bf16 inputs and upstream
    gradient; FLOPs 2.5x the forward's metric (five GEMMs against two). The
    three launches of one call are timed together."""
    import torch

    import exact_attention_80_gb300 as fa
    from exact_attention_80_gb300.inputs import metric_flops

    B, H, N = shape
    gen = torch.Generator(device=device).manual_seed(1010)
    q, k, v, do = (torch.randn((B, H, N, d), generator=gen, device=device).to(torch.bfloat16)
                   for _ in range(4))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d) // 4, device=device)
    res = {}
    for causal in (False, True):
        o, lse = fa.attention(q, k, v, causal=causal, stream=stream)
        fn = lambda: fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, causal, stream=stream)  # noqa: E731
        for _ in range(3):
            fn()
        ms = statistics.median(time_launches(fn, reps, stream, queue_ahead=True))
        flops = 2.5 * metric_flops(B, H, N, N, d, causal)
        res["causal" if causal else "non_causal"] = {"tflops": round(flops / ms / 1e9, 1),
                                                     "us": round(ms * 1e3, 1)}
        del o, lse
    return res


def fp8_decode_workload(device, stream, reps):
    """The C5 decode shape (B=1, H=8, Nq=128, Nk=131072, d=128) with e4m3 Q, K, V
    (descales 2^-5) through fa_fwd_fp8_splitkv + fa_combine, at 16 splits and at
    the largest split count whose grid fits one CTA per SM. K and V are half the
    bytes of bf16; split_gbs counts the bytes the split kernel moves."""
    import torch

    import exact_attention_80_gb300 as fa
    from exact_attention_80_gb300.inputs import metric_flops

    B, H, Nq, Nk, d = 1, 8, 128, 131072, 128
    ds = 2.0 ** -5
    gen = torch.Generator(device=device).manual_seed(1009)
    q8, k8, v8 = ((torch.randn(shape, generator=gen, device=device) / ds)
                  .clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
                  for shape in ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d)))
    o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, H, Nq), device=device)
    flops = metric_flops(B, H, Nq, Nk, d, False)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    fill = fill_splits(fa, B, H, Nq, d, sms)
    res = {}
    for S in sorted({16, fill}):
        ws = torch.empty(fa.fa_splitkv_workspace_bytes(B, H, Nq, d, S) // 4, device=device)
        f_split = lambda: fa.fa_fwd_fp8_splitkv(q8, k8, v8, ds, ds, ds, ws, S, False, stream=stream)  # noqa
        f_comb = lambda: fa.fa_combine(ws, o, lse, B, H, Nq, d, S, stream=stream)  # noqa
        for _ in range(3):
            f_split()
            f_comb()
        ms_s = statistics.median(time_launches(f_split, reps, stream, queue_ahead=True))
        ms_c = statistics.median(time_launches(f_comb, reps, stream, queue_ahead=True))
        moved = 2 * B * H * Nk * d + B * H * Nq * d + S * B * H * Nq * (d + 2) * 4
        res[str(S)] = {"tflops": round(flops / (ms_s + ms_c) / 1e9, 1),
                       "split_us": round(ms_s * 1e3, 1), "combine_us": round(ms_c * 1e3, 1),
                       "split_gbs": round(moved / ms_s / 1e6, 1)}
    return res


def fp8_workload(device, stream, reps, shape=(8, 32, 2048, 128), causal=False, seed=1008):
    """A workload shape (default C2: B=8, H=32, N=2048, d=128, non-causal) with
    e4m3 Q, K, V (N(0,1) / 2^-5 rounded to e4m3, descales 2^-5), through
    fa_fwd_fp8. Its roofline peak is the measured bf16 peak times 2, the nominal
    fp8/bf16 dense ratio."""
    import torch

    import exact_attention_80_gb300 as fa
    from exact_attention_80_gb300.inputs import metric_flops

    B, H, N, d = shape
    ds = 2.0 ** -5
    gen = torch.Generator(device=device).manual_seed(seed)
    q8, k8, v8 = ((torch.randn((B, H, N, d), generator=gen, device=device) / ds)
                  .clamp(-448.0, 448.0).to(torch.float8_e4m3fn) for _ in range(3))
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, H, N), device=device)
    fn = lambda: fa.fa_fwd_fp8(q8, k8, v8, ds, ds, ds, o, lse, causal, stream=stream)  # noqa: E731
    for _ in range(3):
        fn()
    ms = statistics.median(time_launches(fn, reps, stream, queue_ahead=True))
    tflops = metric_flops(B, H, N, N, d, causal) / ms / 1e9
    peak_tf, _, kind = measured_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    kernel = kernel_name(fa, B, H, N, d, sms, N, causal).replace("_kernel", "8_kernel")
    return {"tflops": round(tflops, 1), "us": round(ms * 1e3, 1), "kernel": kernel,
            "shape": f"B={B} H={H} N={N} d={d} {'causal' if causal else 'non-causal'}",
            "roofline_frac": round(tflops / (2.0 * peak_tf), 4),
            "peak": f"2 x {kind} bf16 burst = {2.0 * peak_tf:.1f} TFLOP/s"}


def varlen_workload(device, stream, reps):
    """Ragged batch: 16 packed sequences with seeded lengths in [512, 4096],
    H=32, d=128, top-left causal; FLOPs 4*H*d times the visible pairs."""
    import random

    import torch

    import exact_attention_80_gb300 as fa

    rnd = random.Random(1007)
    lens = [rnd.randint(512, 4096) for _ in range(16)]
    H, d = 32, 128
    total = sum(lens)
    gen = torch.Generator(device=device).manual_seed(1007)
    q = torch.randn((total, H, d), generator=gen, device=device).to(torch.bfloat16)
    k = torch.randn((total, H, d), generator=gen, device=device).to(torch.bfloat16)
    v = torch.randn((total, H, d), generator=gen, device=device).to(torch.bfloat16)
    cu = torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32, device=device)
    o = torch.empty_like(q)
    lse = torch.empty((H, total), device=device)
    fn = lambda: fa.fa_fwd_varlen(q, k, v, o, lse, cu, cu, max(lens), True, stream=stream)  # noqa: E731
    for _ in range(3):
        fn()
    ms = statistics.median(time_launches(fn, reps, stream, queue_ahead=True))
    flops = 4.0 * H * d * sum(n * (n + 1) / 2 for n in lens)
    return {"tflops": round(flops / ms / 1e9, 1), "us": round(ms * 1e3, 1), "sequences": len(lens),
            "tokens": total}


def run_case(args) -> None:
    """Runs one workload's kernels alone, ``--warmup`` untimed then ``--steps``
    timed calls, and prints their mean device time: the target of an ncu
    capture, which then sees only these launches. Cases:

    ``fwd:<workload>``        fa_fwd on a benchmark workload (c1 .. c4)
    ``rows:<workload>:<R>``   fa_fwd_rows with R query rows per CTA (one unit per CTA)
    ``split:<S>``             fa_fwd_splitkv + fa_combine on c5 with S splits
    ``fp8[:<d>]``             fa_fwd_fp8 on the c2 shape at head dim d (default 128;
                              e4m3, descales 2^-5)
    ``bwd:<B>x<H>x<N>[x<d>][:causal]``  fa_bwd (d = 128 unless given)
    """
    import torch

    import exact_attention_80_gb300 as fa
    from exact_attention_80_gb300.inputs import CONFIGS

    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    fa.load_library()
    stream = torch.cuda.current_stream(device)
    gen = torch.Generator(device=device)
    kind, _, arg = args.case.partition(":")
    fns = {}
    if kind == "fwd":
        c = CONFIGS[arg]
        q, k, v = device_qkv(c, gen, device)
        o, lse = torch.empty_like(q), torch.empty(q.shape[:3], device=device)
        fns["fa_fwd"] = lambda: fa.fa_fwd(q, k, v, o, lse, c["causal"], stream=stream)
    elif kind == "rows":
        wl, _, rows = arg.partition(":")
        c = CONFIGS[wl]
        q, k, v = device_qkv(c, gen, device)
        o, lse = torch.empty_like(q), torch.empty(q.shape[:3], device=device)
        fns["fa_fwd_rows"] = lambda: fa.fa_fwd_rows(q, k, v, o, lse, int(rows), c["causal"], stream=stream)
    elif kind == "split":
        c = CONFIGS["c5"]
        S = int(arg)
        B, H, Nq, d = c["B"], c["H"], c["Nq"], c["d"]
        q, k, v = device_qkv(c, gen, device)
        o, lse = torch.empty_like(q), torch.empty(q.shape[:3], device=device)
        ws = torch.empty(fa.fa_splitkv_workspace_bytes(B, H, Nq, d, S) // 4, device=device)
        fns["fa_fwd_splitkv"] = lambda: fa.fa_fwd_splitkv(q, k, v, ws, S, False, stream=stream)
        fns["fa_combine"] = lambda: fa.fa_combine(ws, o, lse, B, H, Nq, d, S, stream=stream)
    elif kind == "fp8":
        ds = 2.0 ** -5
        d = int(arg) if arg else 128
        gen.manual_seed(1008)
        q8, k8, v8 = ((torch.randn((8, 32, 2048, d), generator=gen, device=device) / ds)
                      .clamp(-448.0, 448.0).to(torch.float8_e4m3fn) for _ in range(3))
        o = torch.empty((8, 32, 2048, d), dtype=torch.bfloat16, device=device)
        lse = torch.empty((8, 32, 2048), device=device)
        fns["fa_fwd_fp8"] = lambda: fa.fa_fwd_fp8(q8, k8, v8, ds, ds, ds, o, lse, False, stream=stream)
    elif kind == "bwd":
        shape, _, mask = arg.partition(":")
        dims = [int(x) for x in shape.split("x")]
        B, H, N = dims[:3]
        d = dims[3] if len(dims) > 3 else 128
        causal = mask == "causal"
        gen.manual_seed(1010)
        q, k, v, do = (torch.randn((B, H, N, d), generator=gen, device=device).to(torch.bfloat16)
                       for _ in range(4))
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d) // 4, device=device)
        o, lse = fa.attention(q, k, v, causal=causal, stream=stream)
        fns["fa_bwd"] = lambda: fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, causal, stream=stream)
    else:
        raise SystemExit(f"unknown case {args.case!r}")
    for _ in range(args.warmup):
        for fn in fns.values():
            fn()
    torch.cuda.synchronize()
    times = {name: statistics.mean(time_launches(fn, args.steps, stream)) for name, fn in fns.items()}
    if fa.fa_device_status(clear=True, stream=stream) != fa.FA_OK:
        raise RuntimeError("device status reports a timed-out wait")
    print(f"case {args.case}: " + ", ".join(f"{n} {t * 1e3:.1f} us" for n, t in times.items()))


def workload_config(wl: str, world: int) -> dict:
    """The ``config`` object of both arms' JSON lines for workload ``wl``."""
    from exact_attention_80_gb300.inputs import CONFIGS

    c = CONFIGS[wl]
    B, H, Nq, Nk, d, causal = c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["causal"]
    in_bytes = (B * H * Nq * d + 2 * B * H * Nk * d) * 2
    cfg = {"workload": f"{wl}: B={B} H={H} Nq={Nq} Nk={Nk} d={d} "
                       f"{'causal' if causal else 'non-causal'}",
           "B": B, "H": H, "Nq": Nq, "Nk": Nk, "d": d, "causal": causal,
           "seed": c["seed"], "per_rank_batch": B,
           "l2": (f"inputs larger than L2 ({in_bytes / 2**20:.0f} MiB of Q/K/V per rank vs "
                  f"{L2_BYTES / 2**20:.0f} MiB L2); no flush") if in_bytes > L2_BYTES else
                 "inputs smaller than L2",
           "parallelism": f"replicas x{world} (independent heads, no exchange)"}
    if c.get("outlier_frac"):
        cfg["outliers"] = f"{c['outlier_frac']:.0%} of K rows per head scaled x8"
    return cfg


def run_ours(args):
    import numpy as np
    import torch

    import exact_attention_80_gb300 as fa
    import oracle
    from exact_attention_80_gb300.inputs import CONFIGS, f32, make_qkv, metric_flops, to_f64

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist_init("nccl")
    fa.load_library()
    stream = torch.cuda.current_stream(device)

    wl = args.workload
    c = CONFIGS[wl]
    B, H, Nq, Nk, d, causal = c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["causal"]
    seed = shard_seed(c["seed"], rank)
    q_h, k_h, v_h = make_qkv(B, H, Nq, Nk, d, seed, outlier_frac=c.get("outlier_frac", 0.0))
    scale = f32(1.0 / math.sqrt(d))
    q, k, v = q_h.to(device), k_h.to(device), v_h.to(device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=device)
    flops = metric_flops(B, H, Nq, Nk, d, causal)

    step = lambda: fa.fa_fwd(q, k, v, o, lse, causal, scale, stream=stream)  # noqa: E731

    # ---- timed region (device-resident inputs)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    dist_barrier(world, device)
    torch.cuda.synchronize()
    # The K steps back to back between one pair of CUDA events (queued behind a
    # device sleep so that the host's launch rate does not show): an event
    # between launches would serialise each launch against the previous one's
    # end.
    local_ms = time_back_to_back(step, args.steps, stream) * args.steps
    torch.cuda.synchronize()
    dist_barrier(world, device)
    if sampler:
        sampler.stop()
    total_ms = dist_max(local_ms, world, device)
    status = fa.fa_device_status(clear=True, stream=stream)
    if status != fa.FA_OK:
        raise RuntimeError(f"device status {fa.fa_status_string(status)}")
    ms_per_step = total_ms / args.steps
    value = dist_sum(flops, world, device) * args.steps / (total_ms / 1e3) / 1e12
    avg_launch_ms = local_ms / args.steps
    # Spread of the per-launch time (median, p10, p90): a separate pass with an
    # event after every launch, outside the timed region.
    launch_spread = spread_us(time_launches(step, min(args.steps, 200), stream, queue_ahead=True))

    # ---- numeric check outside the timed window: one whole (b, h) head, chosen
    # by the seed, element by element against the oracle
    rng = np.random.default_rng(seed)
    b, h = int(rng.integers(B)), int(rng.integers(H))
    ro, rl = oracle.attention_f64(to_f64(q_h[b, h]), to_f64(k_h[b, h]), to_f64(v_h[b, h]), scale,
                                  causal)
    got = o[b, h].float().cpu().numpy().astype(np.float64)
    worst = float(np.abs(got - ro).max())
    rel = float(np.linalg.norm(got - ro) / np.linalg.norm(ro))
    lse_err = float(np.abs(lse[b, h].cpu().numpy() - rl).max())
    if not (worst <= 2e-2 and rel <= 5e-3 and lse_err <= 1e-3):
        raise RuntimeError(f"bench parity check failed on head ({b}, {h}): max-abs {worst:.3e}, "
                           f"rel-L2 {rel:.3e}, LSE {lse_err:.3e}")

    # ---- end to end through the public API from pinned host buffers
    qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    op = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lp = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    def e2e_step():
        # Host-to-device copies of one slice of the batch overlap the kernel of
        # the previous slice and the copy back of the one before.
        fa.fa_fwd_from_host(qp, kp, vp, op, lp, q, k, v, o, lse, causal, scale,
                            chunks=args.e2e_chunks, stream=stream)

    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_err = float((op.float() - o.float().cpu()).abs().max())
    if e2e_err != 0.0:
        raise RuntimeError(f"end-to-end output differs from the device-resident one ({e2e_err:.3e})")
    dist_barrier(world, device)
    e2e_ms = dist_max(sum(time_launches(e2e_step, e2e_steps, stream)), world, device) / e2e_steps
    e2e_value = dist_sum(flops, world, device) / (e2e_ms / 1e3) / 1e12
    e2e_launches = len(fa.head_slices(B * H, args.e2e_chunks))
    h2d = (qp.numel() + kp.numel() + vp.numel()) * 2
    d2h = op.numel() * 2 + lp.numel() * 4

    extras = extra_workloads(device, stream) if (rank == 0 and not args.no_extras) else None
    dist_barrier(world, device)

    if rank != 0:
        return None
    peak_tf, _, peak_kind = measured_peaks()
    achieved = flops / (avg_launch_ms / 1e3) / 1e12
    clocks = sampler.summary() if sampler else None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        tf, heads, secs = oracle_sample(c, args.cpu_budget, seed)
        cpu = {"value": round(tf, 6), "unit": "TFLOPS", "cores": cpu_threads(), "kind": "oracle",
               "os_cpu_count": os.cpu_count(), "blas_threads": blas_threads(),
               "sample": f"{heads} passes of the float64 NumPy oracle over one seeded "
                         f"{c['Nq']}x{c['Nk']} d={d} head of {wl} (the same synthetic head each "
                         f"time, all its queries against all its keys), {secs:.1f} s"}
    kname = kernel_name(fa, B, H, Nq, d, torch.cuda.get_device_properties(device).multi_processor_count,
                        Nk, bool(causal))
    line = {
        "metric": "attention fwd TFLOPS (bf16, 4*B*H*Nq*Nk*d, halved for causal)",
        "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": workload_config(wl, world),
        "roofline": {"bound": "tensor", "kernel": kname,
                     "achieved": round(achieved, 1), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tf, 4),
                     "peak_kind": f"{peak_kind} bf16 burst (kernel timed alone)",
                     # The timed region (2000 launches back to back, about 0.75 s)
                     # runs under the power cap, like the sustained GEMM figure:
                     # the fraction of that, for context.
                     "frac_of_sustained": (round(achieved / sustained_bf16_peak(), 4)
                                           if sustained_bf16_peak() else None),
                     "traffic": recorded_traffic(kname, wl),
                     "flops_per_launch": flops},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "how": f"fa_fwd_from_host: the heads in {e2e_launches} slices (the last two a half "
                       "and a quarter of the others), host-to-device copies, kernels and "
                       "device-to-host copies on three streams"},
        "gpu_launches": args.steps,
        "per_launch": launch_spread,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "parity_whole_head": {"head": [b, h], "max_abs": worst, "rel_l2": rel, "lse_abs": lse_err},
        "other_workloads": extras,
    }
    return line


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The float64 oracle as the reference arm, on the host cores, rank 0 only.
    Each step is a bounded sample of the workload: a block of 256 query rows of
    one (b, h) head against all of its keys."""
    import oracle
    from exact_attention_80_gb300.inputs import CONFIGS, f32, make_qkv, to_f64

    rank, world, _ = dist_env()
    if rank != 0:
        return None
    wl = args.workload
    c = CONFIGS[wl]
    B, H, Nq, Nk, d, causal = c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["causal"]
    q, k, v = make_qkv(1, 1, Nq, Nk, d, c["seed"])
    qf, kf, vf = to_f64(q)[0, 0], to_f64(k)[0, 0], to_f64(v)[0, 0]
    scale = f32(1.0 / math.sqrt(d))
    rows_per_step = min(256, Nq)
    n_blocks = -(-Nq // rows_per_step)

    def step(i):
        r0 = (i % n_blocks) * rows_per_step
        rows = list(range(r0, min(r0 + rows_per_step, Nq)))
        oracle.attention_rows_f64(qf, kf, vf, scale, causal, rows)
        return len(rows)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    rows_done = sum(step(i) for i in range(args.steps))
    secs = time.perf_counter() - t0
    flops = 4.0 * rows_done * Nk * d / (2 if causal else 1)
    value = flops / secs / 1e12
    return {
        "impl": "reference",
        "metric": "attention fwd TFLOPS (bf16, 4*B*H*Nq*Nk*d, halved for causal)",
        "value": round(value, 6), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16, upcast to float64)",
        "config": workload_config(wl, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cpu_threads(),
                         "kind": "oracle", "os_cpu_count": os.cpu_count(), "blas_threads": blas_threads(),
                         "sample": f"each step = {rows_per_step} query rows of one (b,h) head "
                                   f"of {wl} against all {Nk} keys (float64 NumPy oracle)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def launch_ranks(n: int, argv: list[str]) -> int:
    """Re-runs this script as ``n`` ranks on this node (one per GPU) under
    torch.distributed.run with a loopback rendezvous; returns its exit code."""
    import socket

    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c2")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of float64 oracle work for cpu_baseline")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="slices of consecutive (b, h) heads whose copies overlap the kernels end "
                         "to end")
    ap.add_argument("--case", default=None,
                    help="run one workload's kernels only, for an ncu capture (see run_case)")
    args = ap.parse_args(argv)
    if args.case:
        run_case(args)
        return 0
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    world_env = os.environ.get("WORLD_SIZE")
    if world_env is None and args.gpus > 1:
        # One process per GPU: start the ranks here rather than run as one.
        return launch_ranks(args.gpus, argv)
    if int(world_env or "1") != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world_env}: launch one rank per GPU "
              f"(or leave WORLD_SIZE unset and let --gpus start them)", file=sys.stderr)
        return 2
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    if args.impl == "ours" and int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist

        if dist.is_initialized():
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
