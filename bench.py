"""Benchmark of the fused attention forward on one GB300 (or N replicas).

One step = one pass of the hot path over one batch.  Default workload
("long"): B=1, H=16, N=65536, d=128, bf16 Q/K/V drawn from N(0,1), causal,
scale 1/sqrt(128) -- the largest single-GPU configuration of the
attention-forward benchmark, one fa_fwd launch per step.  The FP8 workloads
("fp8_1k", "fp8_4k", "fp8_16k") make a step the whole FP8 path: quantise Q
and K (block scales + Hadamard) and V (block scales), then fa_fwd_fp8.

Timing: W untimed warm-up steps, then K timed steps; before each step L2 is
flushed outside the timed events by writing a 512 MB buffer and then reading
another 512 MB buffer (so the lines left in L2 are clean and no write-back of
the flush lands inside the timed region); each step is bracketed by CUDA
events on the stream the kernels are launched on; the reported time is the
sum over the K steps, the max over ranks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extra] [--ablate]

--ablate times the kernel variants of libfa_ablate.so (one design choice of
the attention kernel switched each) on a few workloads instead.

Multi-GPU (torchrun): every rank runs the same workload on its own GPU
(independent problems, no data-path collective): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import attn_inputs as gen  # noqa: E402

METRIC = "attention fwd TFLOPS (BF16, FP8) and % of GB300 dense tensor peak, 1 GPU"
KERNEL_SOURCES = ["exact_attention_forward_09_gb300/csrc/attn_fwd.cuh",
                  "exact_attention_forward_09_gb300/csrc/ptx.cuh"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SHAPES = {"long": (1, 16, 65536, 128, True), "mid": (4, 16, 2048, 128, False),
          "sweep4k": (4, 16, 4096, 128, False), "sweep16k": (1, 16, 16384, 128, False),
          "sweep8k_d64": (2, 32, 8192, 64, False), "sweep512": (32, 16, 512, 128, False),
          "fp8_1k": (16, 16, 1024, 128, False), "fp8_4k": (4, 16, 4096, 128, False),
          "fp8_16k": (1, 16, 16384, 128, False)}
FLUSH_BYTES = 512 * 1024 * 1024


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    ent = t.get(workload)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed
    region (50 ms period)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,power.limit")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons, limit = [], 0.0, [], set(), None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = max(smax, float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(n)
                if len(parts) > 9:
                    try:
                        limit = float(parts[9])
                    except ValueError:
                        pass
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None, "power_limit_w": limit}


class Flusher:
    """Leaves L2 cold and clean: write a buffer larger than L2, then read
    another one (the written lines are evicted, and written back, by the read,
    outside the timed region)."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(FLUSH_BYTES // 4, device=device, dtype=torch.float32)
        self.r = torch.ones(FLUSH_BYTES // 4, device=device, dtype=torch.float32)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


# ------------------------------------------------------------ our arm -------
def run_ours(args, rank, world, device):
    import ctypes

    import torch
    import exact_attention_forward_09_gb300 as fa

    B, H, N, d, causal = args.B, args.H, args.N, args.d, args.causal
    scale = 1.0 / math.sqrt(d)
    fp8 = args.fp8
    dtype = torch.float32 if fp8 else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(1 + rank)
    q = torch.randn((B, H, N, d), device=device, dtype=torch.float32, generator=g).to(dtype)
    k = torch.randn((B, H, N, d), device=device, dtype=torch.float32, generator=g).to(dtype)
    v = torch.randn((B, H, N, d), device=device, dtype=torch.float32, generator=g).to(dtype)
    o = torch.empty((B, H, N, d), device=device, dtype=torch.bfloat16)
    lse = torch.empty((B, H, N), device=device, dtype=torch.float32)
    flush = Flusher(device)
    stream = torch.cuda.current_stream(device)
    flops = gen.flops(B, H, N, d, causal)
    signs = gen.hadamard_signs(d, 4)
    keep = (ctypes.c_int8 * d)(*[int(x) for x in signs])
    if fp8:
        nb = (N + 127) // 128
        q8, k8, v8 = (torch.empty((B, H, N, d), device=device, dtype=torch.uint8) for _ in range(3))
        qs, ks, vs = (torch.empty((B, H, nb), device=device, dtype=torch.float32) for _ in range(3))
    launches_per_step = 4 if fp8 else 1

    # one step = the whole hot path on one batch: FP8 quantises Q and K
    # (block scales + Hadamard) and V (block scales) in one fa_quant_fp8_qkv
    # call (three launches on internal streams, joined back), then runs
    # attention; `mid` marks the start of the attention launch (the dominant
    # kernel)
    def step(qi, ki, vi, mid=None):
        if fp8:
            lib = fa.lib()
            sp = torch.cuda.current_stream(device).cuda_stream
            st = lib.fa_quant_fp8_qkv(qi.data_ptr(), ki.data_ptr(), vi.data_ptr(), q8.data_ptr(), k8.data_ptr(),
                                      v8.data_ptr(), qs.data_ptr(), ks.data_ptr(), vs.data_ptr(), B, H, H, N, N, d,
                                      ctypes.cast(keep, ctypes.c_void_p), sp)
            assert st == 0
            if mid is not None:
                mid.record(stream)
            fa.fwd_fp8(q8, k8, v8, qs, ks, vs, causal=causal, scale=scale, out=o, lse=lse)
        else:
            if mid is not None:
                mid.record(stream)
            fa.fwd(qi, ki, vi, causal=causal, scale=scale, out=o, lse=lse)

    for _ in range(args.warmup):
        flush()
        step(q, k, v)
    fa.check_device_error(device)
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    sampler = ClockSampler(device.index if device.index is not None else 0)
    _barrier(world)
    torch.cuda.synchronize(device)
    sampler.start()
    time.sleep(0.1)
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        step(q, k, v, mid=ev[i][1])
        ev[i][2].record(stream)
    torch.cuda.synchronize(device)
    _barrier(world)
    clocks = sampler.stop()
    fa.check_device_error(device)
    times_ms = [a.elapsed_time(c) for a, _, c in ev]
    total_ms = _max_over_ranks(sum(times_ms), world, device)
    launch_ms = sum(b.elapsed_time(c) for _, b, c in ev) / len(ev)   # the attention launch alone

    # end to end through the public API: pinned host inputs -> device, kernel,
    # result back to pinned host memory, every step.  bf16/fp16: one
    # fa_fwd_host call on the host buffers (it overlaps the copies of one
    # chunk of heads with the kernel of the previous one); FP8: the inputs
    # are copied, quantised and attended, and the result copied back.
    qh = q.cpu().pin_memory()
    kh = k.cpu().pin_memory()
    vh = v.cpu().pin_memory()
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    if fp8:
        qd, kd, vd = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def e2e_step():
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            step(qd, kd, vd)
            oh.copy_(o, non_blocking=True)
            lh.copy_(lse, non_blocking=True)
    else:
        ws = torch.empty((fa.fwd_host_workspace_bytes(B, H, H, N, N, d),), dtype=torch.uint8, device=device)

        def e2e_step():
            fa.fwd_host(qh, kh, vh, causal=causal, scale=scale, out=oh, lse=lh, workspace=ws, device=device)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, min(args.steps, 10))
    e0.record(stream)
    t_host = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    # host time to enqueue the steps: when it nears the device time, the
    # end-to-end figure is bound by the host (a shared CPU), not the GPU
    enqueue_ms = (time.perf_counter() - t_host) * 1e3 / n_e2e
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), world, device) / n_e2e
    h2d = 3 * q.numel() * q.element_size()
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
    # the host link as this run sees it (one pinned tensor each way, alone):
    # e2e can only hide the copies while they take less than the kernels
    link = {}
    for name, dst, src in (("h2d", q, qh), ("d2h", oh, o)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize(device)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize(device)
        link[name] = round(3 * src.numel() * src.element_size() / (c0.elapsed_time(c1) * 1e-3) / 1e9, 1)
    del qh, kh, vh, oh, lh

    extra, fp8_point, short_n = {}, None, None
    if rank == 0 and not args.no_extra:
        del q, k, v, o, lse
        torch.cuda.empty_cache()
        fp8_point = run_fp8_point(device, flush)
        short_n = run_short_n(device, flush)
        extra = run_extra(device, flush)

    return dict(times_ms=times_ms, total_ms=total_ms, launch_ms=launch_ms, flops=flops, clocks=clocks,
                launches_per_step=launches_per_step, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, link=link,
                enqueue_ms=enqueue_ms, extra=extra,
                fp8_point=fp8_point, short_n=short_n)


def _launch_times(fn, steps, device, flush):
    """Event-timed durations (ms) of `steps` calls of fn, each after an L2 flush."""
    import torch
    stream = torch.cuda.current_stream(device)
    ts = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize(device)
        ts.append(a.elapsed_time(b))
    return ts


def _time_launches(fn, steps, device, flush):
    """Median of the flushed launch durations (ms): one slow launch (the first
    after a shape change, a clock step) does not move the point."""
    return statistics.median(_launch_times(fn, steps, device, flush))


def run_fp8_point(device, flush):
    """The FP8 half of the metric, on the largest FP8 configuration (B=1,
    H=16, N=16384, d=128): attention alone against the FP8 peak, and the
    whole FP8 step (Q, K and V quantised in one fa_quant_fp8_qkv call, then
    attention)."""
    import torch
    import exact_attention_forward_09_gb300 as fa

    peaks, src = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * 2.0
    B, H, N, d, _ = SHAPES["fp8_16k"]
    g = torch.Generator(device=device)
    g.manual_seed(11)
    x = [torch.randn((B, H, N, d), device=device, generator=g) for _ in range(3)]
    signs = gen.hadamard_signs(d, 4)
    q8, qs = fa.quant_fp8(x[0], signs=signs)
    k8, ks = fa.quant_fp8(x[1], signs=signs)
    v8, vs = fa.quant_fp8(x[2])
    o = torch.empty((B, H, N, d), device=device, dtype=torch.bfloat16)
    lse = torch.empty((B, H, N), device=device, dtype=torch.float32)
    attn = lambda: fa.fwd_fp8(q8, k8, v8, qs, ks, vs, out=o, lse=lse)

    def whole():
        fa.quant_fp8_qkv(x[0], x[1], x[2], signs=signs)
        attn()

    attn()
    # 200 flushed launches (about 0.3 s) with the clocks sampled meanwhile
    sampler = ClockSampler(device.index if device.index is not None else 0)
    torch.cuda.synchronize(device)
    sampler.start()
    time.sleep(0.1)
    ts = _launch_times(attn, 200, device, flush)
    clocks = sampler.stop()
    ms, ms_mean = statistics.median(ts), sum(ts) / len(ts)
    ms_step = _time_launches(whole, 10, device, flush)
    fl = gen.flops(B, H, N, d, False)
    tf = fl / (ms * 1e-3) / 1e12
    fa.check_device_error(device)
    return {"workload": f"fp8_16k: B={B} H={H} N={N} d={d} non-causal, Q/K block scales + Hadamard, V block scales",
            "value": tf, "unit": "TFLOPS", "ms": ms, "ms_mean": ms_mean, "timing": "median of 200 flushed launches",
            "clocks": clocks,
            "peak": fp8_peak, "frac": tf / fp8_peak,
            "peak_source": f"{src} bf16 burst (cuBLAS GEMM) x 2, the nominal dense fp8:bf16 ratio",
            "kernel": f"attn_fwd_kernel<e4m3,{d},non-causal>", "traffic": load_traffic("fp8_16k"),
            "step_ms": ms_step, "step_tflops": fl / (ms_step * 1e-3) / 1e12}


def run_short_n(device, flush):
    """Short sequences, where the forward sits at or below the ridge: HBM
    GB/s on the algorithmic bytes (Q, K, V read once, O written once, LSE)
    against the measured HBM bandwidth, beside TFLOPS."""
    import torch
    import exact_attention_forward_09_gb300 as fa

    peaks, _ = load_peaks()
    g = torch.Generator(device=device)
    g.manual_seed(12)
    out = {}
    for N, causal in ((512, False), (512, True), (1024, True)):
        B, H, d = gen.TOTAL_TOKENS // N, 16, 128
        q, k, v = (torch.randn((B, H, N, d), device=device, generator=g).to(torch.bfloat16) for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), device=device, dtype=torch.float32)
        fn = lambda: fa.fwd(q, k, v, causal=causal, out=o, lse=lse)
        fn()
        ms = _time_launches(fn, 10, device, flush)
        nbytes = 4 * q.numel() * 2 + lse.numel() * 4
        gbs = nbytes / (ms * 1e-3) / 1e9
        tf = gen.flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12
        out[f"N{N}_d128{'_causal' if causal else ''}"] = {
            "B": B, "H": H, "ms": round(ms, 4), "hbm_gbs": round(gbs, 1),
            "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3), "tflops": round(tf, 1),
            "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 3), "bytes": nbytes}
    out["note"] = "algorithmic bytes = Q+K+V read + O written (bf16) + LSE (fp32); peak = measured HBM copy bandwidth"
    return out


def run_extra(device, flush):
    """Secondary points (not the headline): the 16K-token sweep at every
    (N, H, d) causal and not, the mid workload (bf16, fp16), FP8 at N=4096,
    the quantiser's bandwidth, split-KV decode and the backward."""
    import torch
    import exact_attention_forward_09_gb300 as fa

    peaks, _ = load_peaks()
    out = {}
    g = torch.Generator(device=device)
    g.manual_seed(7)

    def bf(B, H, N, d, causal, dtype=torch.bfloat16, reps=5):
        q, k, v = (torch.randn((B, H, N, d), device=device, generator=g).to(dtype) for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), device=device, dtype=torch.float32)
        fn = lambda: fa.fwd(q, k, v, causal=causal, out=o, lse=lse)
        fn()
        ms = _time_launches(fn, reps, device, flush)
        tf = gen.flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12
        return {"ms": round(ms, 4), "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 3)}

    out["mid"] = bf(4, 16, 2048, 128, False)
    out["mid_causal"] = bf(4, 16, 2048, 128, True)
    out["mid_fp16"] = bf(4, 16, 2048, 128, False, torch.float16)
    sweep = {}
    for (_, B, H, N, d, _) in gen.sweep_configs():
        for causal in (False, True):
            r = bf(B, H, N, d, causal, reps=3)
            sweep[f"N{N}_d{d}{'_causal' if causal else ''}"] = [r["tflops"], r["frac_of_bf16_peak"]]
    out["sweep_16k_tokens"] = {"points": sweep, "format": "[TFLOPS, fraction of the bf16 peak]"}

    # FP8 at N = 4096 (attention) and the quantiser's bandwidth on that input
    fp8_peak = peaks["bf16_tflops"] * 2.0
    B, H, N, d = 4, 16, 4096, 128
    x = [torch.randn((B, H, N, d), device=device, generator=g) for _ in range(3)]
    signs = gen.hadamard_signs(d, 4)
    q8, qs = fa.quant_fp8(x[0], signs=signs)
    k8, ks = fa.quant_fp8(x[1], signs=signs)
    v8, vs = fa.quant_fp8(x[2])
    o = torch.empty((B, H, N, d), device=device, dtype=torch.bfloat16)
    lse = torch.empty((B, H, N), device=device, dtype=torch.float32)
    fn = lambda: fa.fwd_fp8(q8, k8, v8, qs, ks, vs, out=o, lse=lse)
    fn()
    ms = _time_launches(fn, 5, device, flush)
    tf = gen.flops(B, H, N, d, False) / (ms * 1e-3) / 1e12
    qbytes = x[0].numel() * 5  # 4 B read + 1 B written per element
    quant = {}
    cos, sin = (torch.from_numpy(t).to(device) for t in gen.rope_tables(N, d))
    for name, qfn, extra_b in (("block", lambda: fa.quant_fp8(x[2]), 0),
                               ("block_hadamard", lambda: fa.quant_fp8(x[0], signs=signs), 0),
                               ("per_tensor", lambda: fa.quant_fp8(x[2], per_tensor=True), 0),
                               ("rope_half_hadamard", lambda: fa.quant_fp8(x[0], signs=signs,
                                                                          rope=(cos, sin, fa.FA_ROPE_HALF)),
                                (cos.numel() + sin.numel()) * 4),
                               ("rope_half", lambda: fa.quant_fp8(x[0], rope=(cos, sin, fa.FA_ROPE_HALF)),
                                (cos.numel() + sin.numel()) * 4)):
        qms = _time_launches(qfn, 5, device, flush)
        gbs = (qbytes + extra_b) / (qms * 1e-3) / 1e9
        quant[name] = {"us": round(qms * 1e3, 1), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3)}
    # the FP8 workload's quantisation: Q and K with the rotation, V without,
    # in one fa_quant_fp8_qkv call (three launches on internal streams)
    qms = _time_launches(lambda: fa.quant_fp8_qkv(x[0], x[1], x[2], signs=signs), 5, device, flush)
    gbs = 3 * qbytes / (qms * 1e-3) / 1e9
    quant["qkv_one_call"] = {"us": round(qms * 1e3, 1), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3)}
    out["fp8_N4096_d128"] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac_of_fp8_peak": round(tf / fp8_peak, 3)}
    out["quantiser_N4096_d128"] = quant
    del x, q8, k8, v8, o, lse

    # decode-like: one query row per head against a long key/value cache,
    # GQA 4 (split-KV with the group's query heads packed), against the
    # unsplit grouped-query path on the same shape; HBM-bound, so the figure
    # is the K/V bytes read per second
    B, Hq, Hkv, Nk, d = 8, 32, 8, 32768, 128
    q = torch.randn((B, Hq, 1, d), device=device, generator=g).to(torch.bfloat16)
    k, v = (torch.randn((B, Hkv, Nk, d), device=device, generator=g).to(torch.bfloat16) for _ in range(2))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, 1), device=device, dtype=torch.float32)
    need = fa.splitkv_workspace_bytes(B, Hq, Hkv, 1, Nk, d)
    ws = torch.empty((max(need, 1),), dtype=torch.uint8, device=device)
    kv_bytes = 2 * B * Hkv * Nk * d * 2
    dec = {}
    for name, fn in (("splitkv", lambda: fa.fwd_splitkv(q, k, v, out=o, lse=lse, workspace=ws)),
                     ("unsplit_gqa", lambda: fa.fwd_gqa(q, k, v, out=o, lse=lse))):
        fn()
        ms = _time_launches(fn, 5, device, flush)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        dec[name] = {"ms": round(ms, 4), "kv_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3)}
    dec["workload"] = f"B={B} Hq={Hq} Hkv={Hkv} Nq=1 Nk={Nk} d={d} bf16, K/V {kv_bytes / 1e9:.2f} GB"
    out["decode"] = dec
    del q, k, v, o, lse, ws

    # backward (dQ, dK, dV) from the forward's O and LSE; FLOPs counted as
    # 2.5x the forward's (five matrix products against two)
    bwd = {}
    for name, (B, H, N, d, causal) in (("mid", (4, 16, 2048, 128, False)), ("mid_causal", (4, 16, 2048, 128, True)),
                                       ("N8192", (2, 16, 8192, 128, False)),
                                       ("N8192_causal", (2, 16, 8192, 128, True)),
                                       ("N2048_d64", (4, 32, 2048, 64, False)),
                                       ("N8192_d64", (2, 32, 8192, 64, False))):
        q, k, v, do = (torch.randn((B, H, N, d), device=device, generator=g).to(torch.bfloat16) for _ in range(4))
        o, lse = fa.fwd(q, k, v, causal=causal)
        ws = torch.empty((fa.bwd_workspace_bytes(B, H, N, d),), dtype=torch.uint8, device=device)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fn = lambda: fa.bwd(q, k, v, o, lse, do, causal=causal, dq=dq, dk=dk, dv=dv, workspace=ws)
        fn()
        ms = _time_launches(fn, 5, device, flush)
        tf = 2.5 * gen.flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12
        bwd[name] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 3)}
    bwd["workload"] = ("bf16, 16K tokens per point; d=128: H=16, d=64: H=32; mid: B=4 N=2048, N8192: B=2; "
                       "dq, dk, dv from dO ~ N(0,1); one call per timed step after an L2 flush")
    out["backward"] = bwd
    fa.check_device_error(device)
    return out


ABLATE_VARIANTS = {0: "shipped kernel", 1: "split softmax (two warpgroups per Q tile, 64 keys each)",
                   2: "eager rescale (no lazy threshold)", 4: "P handed over whole (not in two halves)",
                   8: "one Q tile per CTA, S double-buffered (no two-tile alternation)",
                   16: "no work stealing", 32: "separate P (Q K^T of the next tile starts once S is read)",
                   64: "polynomial exponentials on the FMA pipe for 1/8 (d=128 bf16) or 3/8 (FP8, d=64) of P",
                   128: "early partial Q K^T (keys beyond P's columns issued at P's first half)",
                   256: "direct O stores from registers (no staging boxes, no bulk tensor stores)"}
ABLATE_BUILT = {(False, False, 128): (0, 1, 2, 4, 8, 16, 64, 128, 256), (False, True, 128): (0, 1, 8, 16, 256),
                (True, False, 128): (0, 1, 2, 4, 8, 16, 64, 128, 256), (False, False, 64): (0, 1, 32, 64, 128, 256),
                (False, True, 64): (0, 32)}


def run_ablate(args, device):
    """Time the kernel variants of libfa_ablate.so (include/fa_ablate.h): each
    switches one design choice of the attention kernel; TFLOPS and the ratio
    to the shipped kernel, per workload."""
    import ctypes

    import torch
    import exact_attention_forward_09_gb300 as fa
    from exact_attention_forward_09_gb300 import build as fa_build

    fa.lib()  # the product library must be present too (same build)
    lib = ctypes.CDLL(fa_build.LIB_ABLATE)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.fa_ablate_fwd.argtypes = [i32, i32, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, f32, vp, vp, vp, vp]
    lib.fa_ablate_fwd.restype = i32
    flush = Flusher(device)
    g = torch.Generator(device=device)
    g.manual_seed(13)
    out = {}
    for name, (B, H, N, d, causal, fp8) in (("N16384_bf16", (1, 16, 16384, 128, False, False)),
                                            ("mid_bf16", (4, 16, 2048, 128, False, False)),
                                            ("N16384_bf16_causal", (1, 16, 16384, 128, True, False)),
                                            ("mid_bf16_causal", (4, 16, 2048, 128, True, False)),
                                            ("N16384_fp8", (1, 16, 16384, 128, False, True)),
                                            ("N4096_fp8", (4, 16, 4096, 128, False, True)),
                                            ("N8192_d64_bf16", (2, 32, 8192, 64, False, False)),
                                            ("N2048_d64_bf16", (8, 32, 2048, 64, False, False)),
                                            ("N8192_d64_bf16_causal", (2, 32, 8192, 64, True, False))):
        if fp8:
            x = [torch.randn((B, H, N, d), device=device, generator=g) for _ in range(3)]
            signs = gen.hadamard_signs(d, 4)
            q, qs = fa.quant_fp8(x[0], signs=signs)
            k, ks = fa.quant_fp8(x[1], signs=signs)
            v, vs = fa.quant_fp8(x[2])
            ds = (qs.data_ptr(), ks.data_ptr(), vs.data_ptr())
        else:
            q, k, v = (torch.randn((B, H, N, d), device=device, generator=g).to(torch.bfloat16) for _ in range(3))
            ds = (None, None, None)
        o = torch.empty((B, H, N, d), device=device, dtype=torch.bfloat16)
        lse = torch.empty((B, H, N), device=device, dtype=torch.float32)
        res = {}
        for var in ABLATE_BUILT[(fp8, causal, d)]:
            def fn(var=var):
                st = lib.fa_ablate_fwd(var, int(fp8), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), B, H, N, d, int(causal), 1.0 / math.sqrt(d), *ds,
                                       torch.cuda.current_stream(device).cuda_stream)
                assert st == 0, st
            fn()
            ms = _time_launches(fn, args.steps, device, flush)
            res[var] = {"variant": ABLATE_VARIANTS[var], "ms": round(ms, 4),
                        "tflops": round(gen.flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12, 1)}
        base = res[0]["tflops"]
        for var in res:
            res[var]["vs_shipped"] = round(res[var]["tflops"] / base, 3)
        out[name] = {"shape": f"B={B} H={H} N={N} d={d} {'causal' if causal else 'non-causal'} "
                              f"{'e4m3' if fp8 else 'bf16'}", "variants": res}
        fa.check_device_error(device)
    print(json.dumps({"ablation": out, "steps_per_point": args.steps,
                      "l2": "flushed before every timed launch (512 MB write, then 512 MB read)"}), flush=True)


def whole_job_tflops(flops_per_rank_step: float, world: int, total_ms_max: float, steps: int) -> float:
    """Whole-job throughput: every rank runs `steps` steps of `flops_per_rank_step`
    (independent problems); the job takes the slowest rank's time."""
    return flops_per_rank_step * world * steps / (total_ms_max * 1e-3) / 1e12


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, world, device):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------- CPU oracle timing -----
def sampled_rows(N: int, count: int) -> list:
    """`count` query rows spread evenly over [0, N) (first and last included)."""
    count = max(1, min(count, N))
    if count == 1:
        return [N - 1]
    return sorted({round(i * (N - 1) / (count - 1)) for i in range(count)})


def row_flops(rows, N: int, d: int, causal: bool) -> float:
    """FLOPs of the sampled rows: 4 d per visible (query, key) pair."""
    if causal:
        return float(sum(4.0 * d * (r + 1) for r in rows))
    return 4.0 * d * N * len(rows)


def time_oracle(B, H, N, d, causal, budget_s: float):
    """Time the fp64 oracle as it stands on a bounded sample of the workload:
    R query rows of one head spread evenly over the sequence, R chosen from a
    small calibration run so that the measured run takes about `budget_s`.
    Returns (TFLOPS, seconds, sample text, threads)."""
    import oracle

    threads = oracle.max_threads()
    q, k, v = gen.qkv_normal((1, 1, N, d), 99)
    scale = 1.0 / math.sqrt(d)
    cal = sampled_rows(N, min(N, 64))
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, causal=causal, scale=scale, rows=cal)
    t1 = max(time.perf_counter() - t0, 1e-6)
    per_flop = t1 / row_flops(cal, N, d, causal)
    want = budget_s / per_flop
    count = min(N, max(len(cal), int(len(cal) * want / row_flops(cal, N, d, causal))))
    rows = sampled_rows(N, count)
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, causal=causal, scale=scale, rows=rows)
    el = time.perf_counter() - t0
    fl = row_flops(rows, N, d, causal)
    sample = (f"{len(rows)} of {N} query rows of 1 of {B * H} heads, spread evenly, fp64 C oracle; "
              f"FLOPs counted as 4 d per visible (query, key) pair")
    return fl / el / 1e12, el, sample, threads


def run_reference(args, rank, world):
    """The oracle timed as it stands: each step is a bounded sample (query
    rows of one head of the workload).  Rank 0 only."""
    import oracle

    if rank != 0:
        return
    B, H, N, d, causal = args.B, args.H, args.N, args.d, args.causal
    threads = oracle.max_threads()
    q, k, v = gen.qkv_normal((1, 1, N, d), 97)
    scale = 1.0 / math.sqrt(d)
    rows = sampled_rows(N, 1024)
    for _ in range(args.warmup):
        oracle.attn_fwd(q, k, v, causal=causal, scale=scale, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attn_fwd(q, k, v, causal=causal, scale=scale, rows=rows)
    el = time.perf_counter() - t0
    fl = row_flops(rows, N, d, causal) * args.steps
    val = fl / el / 1e12
    sample = (f"{len(rows)} of {N} query rows (spread evenly) of 1 of {B * H} heads per step, fp64 C oracle; "
              f"FLOPs counted as 4 d per visible (query, key) pair")
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(args),
        "cpu_baseline": {"value": val, "unit": "TFLOPS", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def _config(args):
    kind = ("fp32 inputs quantised to e4m3 in the step (Q, K: block scales + Hadamard; V: block scales), "
            "then FP8 attention" if getattr(args, "fp8", False) else "bf16")
    return {"workload": f"{args.workload}: B={args.B} H={args.H} N={args.N} d={args.d} {kind} "
                        f"{'causal' if args.causal else 'non-causal'} scale=1/sqrt(d)",
            "B": args.B, "H": args.H, "N": args.N, "d": args.d, "causal": bool(args.causal),
            "l2": "flushed before every timed step (512 MB write, then 512 MB read: cold, clean L2; "
                  "outside the timed events)",
            "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long", choices=sorted(SHAPES))
    ap.add_argument("--causal", action="store_true", help="causal masks (the long workload is always causal)")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ablate", action="store_true",
                    help="time the kernel variants of libfa_ablate.so instead (one GPU, one JSON line)")
    args = ap.parse_args()
    args.fp8 = args.workload.startswith("fp8")
    args.B, args.H, args.N, args.d, always_causal = SHAPES[args.workload]
    args.causal = bool(args.causal or always_causal)
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    if args.ablate:
        if rank == 0:
            run_ablate(args, device)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    res = run_ours(args, rank, world, device)

    if rank == 0:
        peaks, peak_src = load_peaks()
        tflops = whole_job_tflops(res["flops"], world, res["total_ms"], args.steps)
        achieved = res["flops"] / (res["launch_ms"] * 1e-3) / 1e12
        e2e_tflops = res["flops"] * world / (res["e2e_ms"] * 1e-3) / 1e12
        cpu_tf, cpu_s, cpu_sample, cpu_threads = time_oracle(args.B, args.H, args.N, args.d, args.causal,
                                                              args.cpu_budget)
        traffic = load_traffic(args.workload + ("_causal" if args.causal and args.workload != "long" else ""))
        if args.fp8:
            peak = peaks["bf16_tflops"] * 2.0
            peak_source = f"{peak_src} bf16 burst (cuBLAS GEMM) x 2, the nominal dense fp8:bf16 ratio"
            kernel = f"attn_fwd_kernel<e4m3,{args.d},{'causal' if args.causal else 'non-causal'}>"
        else:
            peak = peaks["bf16_tflops"]
            peak_source = f"{peak_src} bf16 burst (cuBLAS GEMM)"
            kernel = f"attn_fwd_kernel<bf16,{args.d},{'causal' if args.causal else 'non-causal'}>"
        line = {
            "metric": METRIC, "value": tflops, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["total_ms"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if args.fp8 else "bf16", "data": "synthetic",
            "config": _config(args),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_source, "kernel": kernel,
                         "algorithmic_flops_per_launch": res["flops"],
                         "frac_of_sustained": achieved / (peak * peaks.get("bf16_tflops_sustained", peak)
                                                          / peaks["bf16_tflops"])},
            "cpu_baseline": {"value": cpu_tf, "unit": "TFLOPS", "cores": cpu_threads, "kind": "oracle",
                             "sample": cpu_sample, "seconds": round(cpu_s, 2)},
            "e2e": {"value": e2e_tflops, "unit": "TFLOPS", "h2d_bytes_per_step": res["h2d"],
                    "d2h_bytes_per_step": res["d2h"],
                    "call": "copies + quantiser + fa_fwd_fp8" if args.fp8 else "fa_fwd_host on pinned host buffers",
                    "host_link_gbs": res["link"], "ms_per_step": res["e2e_ms"],
                    "host_enqueue_ms_per_step": round(res["enqueue_ms"], 3)},
            "gpu_launches": args.steps * res["launches_per_step"],
            "clocks": res["clocks"],
            "fp8": res["fp8_point"],
            "short_n_hbm": res["short_n"],
            "extra": res["extra"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
