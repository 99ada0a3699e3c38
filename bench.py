"""Benchmark of the fine-grained FP8 GEMM hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  quantize_1x128(X) -> quantize_128x128(W) -> gemm_fp8_blockscaled(UE8M0 scales)
with X = 4096 x 7168 bf16 activations and W = 7168 x 7168 bf16 weights drawn
N(0,1) with 1-in-1024 outliers x400 (the FP8 prefill workload: M=4096,
N=K=7168).  The metric is TFLOPS (2*M*N*K per step / step time) and the GEMM
kernel's fraction of the GB300 dense FP8 tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs its own batch (weak
scaling, no collective on the data path); value = all ranks' FLOPs / max time.
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload (rank 0 only).
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
sys.path.insert(0, ROOT)

M_TOK, N_OUT, K_IN = 4096, 7168, 7168
FLOPS_PER_STEP = 2.0 * M_TOK * N_OUT * K_IN
WORKLOAD = "fp8 block-scaled NT GEMM M=4096 N=7168 K=7168, UE8M0 scales (quantize 1x128 + 128x128 + GEMM)"
L2_FLUSH_BYTES = 256 << 20

# DRAM traffic of the GEMM kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum per launch), valid only for the kernel sources it was
# taken from (sha256 over GEMM_SOURCES).  See profiles/.
NCU_TRAFFIC = {"src_sha": "99bb47b52f5de29e", "bytes_per_launch": 151203328}


# sources the block-scaled GEMM kernel and its launch are compiled from
GEMM_SOURCES = ("api.cu", "device_common.cuh", "fgf8_internal.h", "gemm_launch.cuh", "gemm_mxf8.cu",
                "gemm_persistent.cuh", "ptx.cuh")


def _strip_comments(text: str) -> str:
    """C/C++ source without comments and blank space (string literals kept), so
    that editing a comment does not count as changing the kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join("".join(out).split())


class L2Flush:
    """Flushes L2 between timed iterations: a 256 MiB write, then a 256 MiB read of
    a second buffer.  The read evicts the dirty lines the write left (their
    write-back happens here, outside the timed events) and leaves clean ones, so the
    next timed kernel does not pay for another kernel's write-backs."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def _src_sha() -> str:
    h = hashlib.sha256()
    for p in [os.path.join(ROOT, "fine_grained_fp8_persistent_gb300", "csrc", f) for f in GEMM_SOURCES]:
        with open(p, encoding="utf-8") as f:
            h.update(os.path.basename(p).encode())
            h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), \
            float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling during the timed region (SM clock, throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None
        self.skip = 0

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # the timed region starts only once nvidia-smi is producing samples
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0:
            time.sleep(0.01)
        self.skip = len(self.lines)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines[self.skip:]:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(value: float, world: int, device) -> float:
    """Largest `value` over all ranks (the slowest rank's time sets the job's)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_tflops(steps: int, world: int, t_max_ms: float) -> float:
    """Whole-job throughput: each of `world` ranks ran `steps` steps of its own
    batch (weak scaling) in at most `t_max_ms`."""
    return FLOPS_PER_STEP * steps * world / (t_max_ms * 1e-3) / 1e12


# ============================================================================ ours
def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    import __graft_entry__ as ge
    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world > 1:
        ge.build()
    from fine_grained_fp8_persistent_gb300 import binding as fg
    from fine_grained_fp8_persistent_gb300 import inputs

    UE = fg.SCALE_UE8M0
    # inputs resident in HBM before the timed region (each rank its own batch)
    x_cpu = inputs.normal_bf16((M_TOK, K_IN), seed=1000 + rank, outliers=True)
    w_cpu = inputs.normal_bf16((N_OUT, K_IN), seed=2000, outliers=True)
    x = x_cpu.to(dev)
    w = w_cpu.to(dev)
    xq = torch.empty((M_TOK, K_IN), dtype=torch.uint8, device=dev)
    wq = torch.empty((N_OUT, K_IN), dtype=torch.uint8, device=dev)
    sfa_shape, sfa_dt = fg.sfa_shape(M_TOK, K_IN, UE)
    sfb_shape, sfb_dt = fg.sfb_shape(1, N_OUT, K_IN, UE)
    sfa = torch.empty(sfa_shape, dtype=sfa_dt, device=dev)
    sfb = torch.empty(sfb_shape, dtype=sfb_dt, device=dev)
    d = torch.empty((M_TOK, N_OUT), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    side = torch.cuda.Stream(device=dev)

    def step():
        # the two quantizers are independent and neither saturates HBM alone: the
        # weights go on a side stream, the activations on this one; the GEMM waits
        # for both
        side.wait_stream(stream)
        fg.quantize_128x128(w, UE, wq, sfb, stream=side)
        fg.quantize_1x128(x, UE, xq, sfa, stream=stream)
        stream.wait_stream(side)
        ev_q.record(stream)
        fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, UE, out=d, stream=stream)

    ev_q = torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    rc, bits = fg.check_status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {bits:#x} after warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit()
                           else local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush()                           # L2 flush between timed steps (outside the events)
        starts[i].record(stream)
        ev_q = mids[i]
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    gemm_tile = fg.last_tile()
    if world > 1:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    gemm_ms = [m.elapsed_time(e) for m, e in zip(mids, ends)]
    total_ms = sum(step_ms)
    rc, bits = fg.check_status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {bits:#x} after the timed steps")

    t_max_ms = _max_over_ranks(total_ms, world, dev)
    value = _job_tflops(args.steps, world, t_max_ms)

    e2e = None if args.no_e2e else _e2e(args, fg, x_cpu, w_cpu, dev, stream, side, d)
    variants = _variants(fg, dev, stream, args.variant) if rank == 0 and not args.no_variants else None
    cpu = _cpu_baseline(args) if rank == 0 and world == 1 and not args.no_cpu else None

    bf16_peak, bf16_sust, hbm, src = _peaks()
    fp8_peak = 2.0 * bf16_peak
    gemm_avg_ms = statistics.mean(gemm_ms)
    achieved = FLOPS_PER_STEP / (gemm_avg_ms * 1e-3) / 1e12
    traffic = NCU_TRAFFIC["bytes_per_launch"] if NCU_TRAFFIC["src_sha"] == _src_sha() else None
    if rank == 0:
        line = {
            "metric": "TFLOPS (FP8 block-scaled NT GEMM step, fraction of GB300 dense FP8 tensor peak)",
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(t_max_ms / args.steps, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "e4m3 x e4m3 -> f32 accumulate (bf16 out)",
            "data": "synthetic (seeded N(0,1) bf16, 1/1024 outliers x400)",
            "config": {"workload": WORKLOAD, "M": M_TOK, "N": N_OUT, "K": K_IN,
                       "scale_format": "ue8m0", "per_rank_batch_tokens": M_TOK,
                       "l2": "flushed between steps (256 MiB write, then 256 MiB read, outside the timed events)",
                       "parallelism": f"replicas x{world} (independent batches, no collective)"},
            "gemm_ms": round(gemm_avg_ms, 4),
            "quantize_ms": round(statistics.mean(s - g for s, g in zip(step_ms, gemm_ms)), 4),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(fp8_peak, 1),
                         "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
                         "traffic": traffic,
                         "peak_note": f"FP8 dense = 2 x bf16 burst GEMM peak ({bf16_peak} TFLOP/s, {src}); "
                                      f"vs sustained: {round(achieved / (2 * bf16_sust), 4)}",
                         "kernel": f"gemm_persistent ({gemm_tile})"},
            "e2e": e2e,
            "gpu_launches": 3 * args.steps,
            "clocks": clocks,
            "wall_s_timed_region": round(wall, 3),
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if variants is not None:
            line["variants"] = variants
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _e2e(args, fg, x_cpu, w_cpu, dev, stream, side, d_device) -> dict:
    """Same step through the public API from pinned HOST buffers: every step copies
    its X and W to the device, quantizes both, runs the GEMM and copies D back, all
    inside the timed region.  Steps are pipelined over two buffer sets: the
    host-to-device copies of step i + 1 run while step i computes and its result
    travels back (separate copy streams, one per direction), as a serving loop
    would; the weight path (its copy and quantizer) runs beside the activation
    path as in the device-resident step."""
    import torch
    UE = fg.SCALE_UE8M0
    xh = x_cpu.pin_memory()
    wh = w_cpu.pin_memory()
    nbuf = 2
    dh = [torch.empty((M_TOK, N_OUT), dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    # device buffers allocated once, outside the timed loop
    xd = [torch.empty_like(xh, device=dev) for _ in range(nbuf)]
    wd = [torch.empty_like(wh, device=dev) for _ in range(nbuf)]
    xq = [torch.empty((M_TOK, K_IN), dtype=torch.uint8, device=dev) for _ in range(nbuf)]
    wq = [torch.empty((N_OUT, K_IN), dtype=torch.uint8, device=dev) for _ in range(nbuf)]
    sh, dt = fg.sfa_shape(M_TOK, K_IN, UE)
    sfa = [torch.empty(sh, dtype=dt, device=dev) for _ in range(nbuf)]
    sh, dt = fg.sfb_shape(1, N_OUT, K_IN, UE)
    sfb = [torch.empty(sh, dtype=dt, device=dev) for _ in range(nbuf)]
    d = [torch.empty((M_TOK, N_OUT), dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    h2d_x = torch.cuda.Stream(device=dev)
    h2d_w = torch.cuda.Stream(device=dev)
    d2h = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_free = [ev() for _ in range(nbuf)]     # the quantizers of the step that used this set are done
    out_free = [ev() for _ in range(nbuf)]    # the result of the step that used this set is on the host
    x_in, w_in, w_q, d_ready = [ev() for _ in range(nbuf)], [ev() for _ in range(nbuf)], \
        [ev() for _ in range(nbuf)], [ev() for _ in range(nbuf)]
    started = [False] * nbuf

    def one(i):
        b = i % nbuf
        for s_ in (h2d_x, h2d_w):
            if started[b]:
                s_.wait_event(in_free[b])
        with torch.cuda.stream(h2d_x):
            xd[b].copy_(xh, non_blocking=True)
            x_in[b].record(h2d_x)
        with torch.cuda.stream(h2d_w):
            wd[b].copy_(wh, non_blocking=True)
            w_in[b].record(h2d_w)
        side.wait_event(w_in[b])
        if started[b]:
            side.wait_event(d_ready[b])   # the GEMM of the step before has read wq[b]
        fg.quantize_128x128(wd[b], UE, wq[b], sfb[b], stream=side)
        w_q[b].record(side)
        stream.wait_event(x_in[b])
        fg.quantize_1x128(xd[b], UE, xq[b], sfa[b], stream=stream)
        stream.wait_event(w_q[b])
        in_free[b].record(stream)
        if started[b]:
            stream.wait_event(out_free[b])
        fg.gemm_fp8_blockscaled(xq[b], sfa[b], wq[b], sfb[b], UE, out=d[b], stream=stream)
        d_ready[b].record(stream)
        d2h.wait_event(d_ready[b])
        with torch.cuda.stream(d2h):
            dh[b].copy_(d[b], non_blocking=True)
            out_free[b].record(d2h)
        started[b] = True

    for i in range(2 * nbuf):
        one(i)
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 20))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for s_ in (h2d_x, h2d_w, side, stream, d2h):
        s_.synchronize()
    e0.record(h2d_x)
    h2d_w.wait_event(e0)
    for i in range(steps):
        one(i)
    # the run ends when the last result is on the host
    stream.wait_stream(d2h)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # same inputs, deterministic kernels: the result read back to the host must be
    # bit-identical to the device-resident step's
    same = bool(torch.equal(dh[(steps - 1) % nbuf].to(dev), d_device))
    return {"value": round(FLOPS_PER_STEP / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": xh.numel() * 2 + wh.numel() * 2,
            "d2h_bytes_per_step": dh[0].numel() * 2,
            "pipelined": "two buffer sets; copies of step i+1 overlap step i",
            "result_matches_device_step": same}


def _variants(fg, dev, stream, only=None) -> dict:
    """Kernel-only throughput of every other configuration on its own workload,
    each against the roofline that bounds it: the dense FP8 (2 x bf16) or bf16
    tensor peak for the large GEMMs, the HBM copy bandwidth for the skinny and
    masked-decode GEMMs and the quantizers (algorithmic bytes: every operand,
    scale table and output once; padding rows and empty experts excluded)."""
    import torch
    from fine_grained_fp8_persistent_gb300 import inputs
    out = {}
    bf16_peak, _, hbm, src = _peaks()
    fp8_peak = 2.0 * bf16_peak

    def timeit(fn, iters=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        es = [torch.cuda.Event(enable_timing=True) for _ in range(2 * iters)]
        flush = L2Flush(dev)
        tot = 0.0
        for i in range(iters):
            flush()
            es[2 * i].record(stream)
            fn()
            es[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        for i in range(iters):
            tot += es[2 * i].elapsed_time(es[2 * i + 1])
        return tot / iters

    def record(name, ms, flops, byts, bound):
        r = {"ms": round(ms, 4), "bound": bound}
        if flops:
            r["TFLOP/s"] = round(flops / (ms * 1e-3) / 1e12, 1)
        r["GB/s"] = round(byts / (ms * 1e-3) / 1e9, 1)
        if bound == "tensor_fp8":
            r["frac"] = round(r["TFLOP/s"] / fp8_peak, 4)
        elif bound == "tensor_fp4":
            r["frac"] = round(r["TFLOP/s"] / (6.0 * bf16_peak), 4)
        elif bound == "tensor_bf16":
            r["frac"] = round(r["TFLOP/s"] / bf16_peak, 4)
        elif bound == "hbm":
            r["frac"] = round(r["GB/s"] / hbm, 4)
        r["tile"] = fg.last_tile() if flops else None
        out[name] = r

    def want(name):
        # a group (e.g. "grouped_contiguous") is wanted when the requested name
        # lies inside it, a single variant when its name starts with the request
        return only is None or name.startswith(only) or only.startswith(name)

    def sf_bytes(rows, k, fmt):
        return rows * (k // 128) * 4 if fmt == fg.SCALE_F32 else rows * ((k // 128 + 3) // 4) * 4

    # FP8 block-scaled dense: the 128 x 128 x 256 case, the M = 64 decode and the
    # M = 4096 case with FP32 scales
    w = inputs.normal_bf16((N_OUT, K_IN), 2, outliers=True).to(dev)
    x = inputs.normal_bf16((M_TOK, K_IN), 1, outliers=True).to(dev)
    small_a = inputs.normal_bf16((128, 256), 0).to(dev)
    small_b = inputs.normal_bf16((128, 256), 1).to(dev)
    xq, sfa = fg.quantize_1x128(small_a, fg.SCALE_F32)
    wq, sfb = fg.quantize_128x128(small_b, fg.SCALE_F32)
    d = torch.empty((128, 128), dtype=torch.bfloat16, device=dev)
    if want("fp8_f32scale_128x128x256"):
        ms = timeit(lambda: fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, fg.SCALE_F32, out=d))
        record("fp8_f32scale_128x128x256", ms, 2.0 * 128 * 128 * 256, 2 * 128 * 256 + 128 * 128 * 2, "latency")
    for name, m, fmt in (("fp8_ue8m0_64x7168x7168", 64, fg.SCALE_UE8M0),
                         ("fp8_f32scale_64x7168x7168", 64, fg.SCALE_F32),
                         ("fp8_f32scale_4096x7168x7168", M_TOK, fg.SCALE_F32)):
        if not want(name):
            continue
        xq, sfa = fg.quantize_1x128(x[:m].contiguous(), fmt)
        wq, sfb = fg.quantize_128x128(w, fmt)
        d = torch.empty((m, N_OUT), dtype=torch.bfloat16, device=dev)
        ms = timeit(lambda: fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, fmt, out=d))
        byts = m * K_IN + N_OUT * K_IN + m * N_OUT * 2 + sf_bytes(m, K_IN, fmt) + sf_bytes(N_OUT, K_IN, fmt)
        record(name, ms, 2.0 * m * N_OUT * K_IN, byts, "hbm" if m < 1024 else "tensor_fp8")
    # the UE8M0 GEMM with its output quantized 1x128 (next layer's activations) in
    # the epilogue, against the GEMM followed by quantize_1x128 of its bf16 output
    if want("fused_quant") or want("gemm_then_quantize"):
        ue = fg.SCALE_UE8M0
        xq, sfa = fg.quantize_1x128(x, ue)
        wq, sfb = fg.quantize_128x128(w, ue)
        dq = torch.empty((M_TOK, N_OUT), dtype=torch.uint8, device=dev)
        shape, dt = fg.sfa_shape(M_TOK, N_OUT, ue)
        sfd = torch.empty(shape, dtype=dt, device=dev)
        d = torch.empty((M_TOK, N_OUT), dtype=torch.bfloat16, device=dev)
        byts = M_TOK * K_IN + N_OUT * K_IN + M_TOK * N_OUT + sf_bytes(M_TOK, K_IN, ue) + sf_bytes(N_OUT, K_IN, ue)
        if want("fused_quant"):
            ms = timeit(lambda: fg.gemm_fp8_blockscaled_quant(xq, sfa, wq, sfb, ue, ue, dq=dq, sfd=sfd))
            record("fused_quant_ue8m0_4096x7168x7168", ms, 2.0 * M_TOK * N_OUT * K_IN, byts, "tensor_fp8")
            f32 = fg.SCALE_F32
            xq32, sfa32 = fg.quantize_1x128(x, f32)
            wq32, sfb32 = fg.quantize_128x128(w, f32)
            ms = timeit(lambda: fg.gemm_fp8_blockscaled_quant(xq32, sfa32, wq32, sfb32, f32, ue, dq=dq, sfd=sfd))
            record("fused_quant_f32scale_4096x7168x7168", ms, 2.0 * M_TOK * N_OUT * K_IN,
                   byts - sf_bytes(M_TOK, K_IN, ue) - sf_bytes(N_OUT, K_IN, ue)
                   + sf_bytes(M_TOK, K_IN, f32) + sf_bytes(N_OUT, K_IN, f32), "tensor_fp8")
            del xq32, wq32
        if want("gemm_then_quantize"):
            def unfused():
                fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, ue, out=d)
                fg.quantize_1x128(d, ue, xq=dq, sfa=sfd)
            ms = timeit(unfused)
            record("gemm_then_quantize_ue8m0_4096x7168x7168", ms, 2.0 * M_TOK * N_OUT * K_IN,
                   byts + 4 * M_TOK * N_OUT, "tensor_fp8")
        del dq, sfd, d
    del x, xq, wq

    # 16-bit dense 4096^3
    if want("f16_4096x4096x4096"):
        a = inputs.uniform_16bit((4096, 4096), 3).to(dev)
        b = inputs.uniform_16bit((4096, 4096), 4).to(dev)
        d16 = torch.empty((4096, 4096), dtype=torch.float16, device=dev)
        ms = timeit(lambda: fg.gemm_f16(a, b, out=d16))
        record("f16_4096x4096x4096", ms, 2.0 * 4096 ** 3, 3 * 4096 * 4096 * 2, "tensor_bf16")
        del a, b, d16

    # 4-bit block-scaled dense GEMM (MXFP4, NVFP4) on the FP8 prefill shape, and the
    # 4-bit quantizer on the activations; FP4 peak = 6 x the bf16 peak (nominal
    # dense 13.5 vs 2.25 PFLOP/s)
    if want("fp4") or want("quantize_fp4"):
        xf = inputs.normal_bf16((M_TOK, K_IN), 13, outliers=True).to(dev)
        wf = inputs.normal_bf16((N_OUT, K_IN), 14, outliers=True).to(dev)
        d4 = torch.empty((M_TOK, N_OUT), dtype=torch.bfloat16, device=dev)
        for fmt, tag, sv in ((fg.FP4_MX, "mxfp4", 32), (fg.FP4_NV, "nvfp4", 16)):
            xq4, sfa4 = fg.quantize_fp4(xf, fmt)
            wq4, sfb4 = fg.quantize_fp4(wf, fmt)
            if want(f"fp4_{tag}"):
                ms = timeit(lambda: fg.gemm_fp4_blockscaled(xq4, sfa4, wq4, sfb4, fmt, out=d4))
                byts = (M_TOK + N_OUT) * K_IN // 2 + (M_TOK + N_OUT) * K_IN // sv + M_TOK * N_OUT * 2
                record(f"fp4_{tag}_4096x7168x7168", ms, 2.0 * M_TOK * N_OUT * K_IN, byts, "tensor_fp4")
            if want(f"quantize_fp4_{tag}"):
                ms = timeit(lambda: fg.quantize_fp4(xf, fmt, xq=xq4, sf=sfa4))
                record(f"quantize_fp4_{tag}_4096x7168", ms, 0, M_TOK * K_IN * 2 + M_TOK * K_IN // 2 + M_TOK * K_IN // sv,
                       "hbm")
        del xf, wf, d4, xq4, wq4

    # grouped contiguous: 8 experts, N = 4096, K = 7168, counts multinomial(8192)
    if not want("grouped_contiguous"):
        return _variants_tail(fg, dev, timeit, record, sf_bytes, want, out)
    G, N, K = 8, 4096, 7168
    counts = inputs.expert_counts(8192, G, 7)
    m_idx, total = inputs.contiguous_layout(counts, fg.mk_alignment_for_contiguous())
    ac = inputs.normal_bf16((total, K), 8, outliers=True).to(dev)
    bc = inputs.normal_bf16((G, N, K), 9, outliers=True).to(dev)
    m_idx = m_idx.to(dev)
    valid = sum(counts)
    for fmt, tag in ((fg.SCALE_UE8M0, "ue8m0"), (fg.SCALE_F32, "f32scale")):
        if not want(f"grouped_contiguous_{tag}"):
            continue
        aq, sfa = fg.quantize_1x128(ac, fmt)
        bq, sfb = fg.quantize_128x128(bc, fmt)
        dc = torch.empty((total, N), dtype=torch.bfloat16, device=dev)
        ms = timeit(lambda: fg.grouped_fp8_contiguous(aq, sfa, bq, sfb, m_idx, fmt, out=dc))
        byts = valid * K + G * N * K + valid * N * 2 + sf_bytes(valid, K, fmt) + G * sf_bytes(N, K, fmt)
        record(f"grouped_contiguous_{tag}_8x4096x7168_m{valid}", ms, 2.0 * valid * N * K, byts, "tensor_fp8")
    del ac, bc
    return _variants_tail(fg, dev, timeit, record, sf_bytes, want, out)


def _variants_tail(fg, dev, timeit, record, sf_bytes, want, out) -> dict:
    """The masked-decode and quantizer variants (see _variants)."""
    import torch
    from fine_grained_fp8_persistent_gb300 import inputs
    # grouped masked decode: 32 experts, Mmax = 256, N = 7168, K = 2048, FP32 scales
    if not want("grouped_masked"):
        return _quantizer_variants(fg, dev, timeit, record, sf_bytes, want, out)
    G, MM, N, K = 32, 256, 7168, 2048
    mm = inputs.masked_rows(G, MM, 10)
    am = inputs.normal_bf16((G, MM, K), 11, outliers=True).to(dev)
    bm = inputs.normal_bf16((G, N, K), 12, outliers=True).to(dev)
    mm_dev = mm.to(dev)
    dm = torch.empty((G, MM, N), dtype=torch.bfloat16, device=dev)
    sm_ = int(mm.sum())
    live = int((mm > 0).sum())
    for fmt, tag in ((fg.SCALE_F32, "f32scale"), (fg.SCALE_UE8M0, "ue8m0")):
        name = f"grouped_masked_{tag}_32x256x7168x2048_m{sm_}"
        if not want(name):
            continue
        sh, dt = fg.sfa_shape(MM, K, fmt)
        aq = torch.empty((G, MM, K), dtype=torch.uint8, device=dev)
        sfa = torch.empty((G, *sh), dtype=dt, device=dev)
        for g in range(G):
            fg.quantize_1x128(am[g], fmt, aq[g], sfa[g])
        bq, sfb = fg.quantize_128x128(bm, fmt)
        ms = timeit(lambda: fg.grouped_fp8_masked(aq, sfa, bq, sfb, mm_dev, fmt, out=dm))
        byts = sm_ * K + live * N * K + sm_ * N * 2 + sf_bytes(sm_, K, fmt) + live * sf_bytes(N, K, fmt)
        record(name, ms, 2.0 * sm_ * N * K, byts, "hbm")
        del aq, bq
    del am, bm, dm
    return _quantizer_variants(fg, dev, timeit, record, sf_bytes, want, out)


def _quantizer_variants(fg, dev, timeit, record, sf_bytes, want, out) -> dict:
    """The two quantizers on the bench shapes (UE8M0)."""
    from fine_grained_fp8_persistent_gb300 import inputs
    if want("quantize_1x128_4096x7168"):
        xb = inputs.normal_bf16((M_TOK, K_IN), 5, outliers=True).to(dev)
        ms = timeit(lambda: fg.quantize_1x128(xb, fg.SCALE_UE8M0))
        record("quantize_1x128_4096x7168", ms, 0, M_TOK * K_IN * 3 + sf_bytes(M_TOK, K_IN, 1), "hbm")
    if want("quantize_128x128_7168x7168"):
        wb = inputs.normal_bf16((N_OUT, K_IN), 6, outliers=True).to(dev)
        ms = timeit(lambda: fg.quantize_128x128(wb, fg.SCALE_UE8M0))
        record("quantize_128x128_7168x7168", ms, 0, N_OUT * K_IN * 3 + sf_bytes(N_OUT, K_IN, 1), "hbm")
    return out


# ============================================================================ oracle (CPU)
def _oracle_sample(rows: int):
    """One bounded sample of the workload on the CPU oracle: quantize `rows`
    activation rows (1x128) and the whole weight (128x128), then compute those
    rows of D.  Returns (seconds, FLOPs of the GEMM part)."""
    import numpy as np
    import oracle
    from fine_grained_fp8_persistent_gb300 import inputs
    x = inputs.normal_bf16((rows, K_IN), seed=1000, outliers=True).float().numpy()
    w = inputs.normal_bf16((N_OUT, K_IN), seed=2000, outliers=True).float().numpy()
    t0 = time.perf_counter()
    aq, sfa = oracle.quantize_1x128(x, oracle.SCALE_UE8M0)
    bq, sfb = oracle.quantize_128x128(w, oracle.SCALE_UE8M0)
    oracle.gemm_fp8(aq, sfa, bq, sfb, oracle.SCALE_UE8M0)
    return time.perf_counter() - t0, 2.0 * rows * N_OUT * K_IN


def _sample_rows(seconds: float) -> int:
    """Output rows of one oracle sample that takes about `seconds` on this host
    (calibrated on an 8-row sample)."""
    t8, _ = _oracle_sample(8)
    return int(max(1, min(M_TOK, round(8 * seconds / max(t8, 1e-3)))))


def _cpu_baseline(args) -> dict:
    import oracle
    oracle.build()
    rows = args.cpu_rows if args.cpu_rows > 0 else _sample_rows(args.cpu_seconds)
    secs, flops = _oracle_sample(rows)
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{rows} of {M_TOK} output rows: quantize {rows}x{K_IN} (1x128) + "
                      f"{N_OUT}x{K_IN} (128x128) + GEMM {rows}x{N_OUT}x{K_IN}, UE8M0, fp64 oracle",
            "seconds": round(secs, 2)}


def run_reference(args) -> None:
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    oracle.build()
    # each step is a bounded sample, sized so the whole run takes about
    # --ref-seconds on the host cores
    rows = args.cpu_rows if args.cpu_rows > 0 else \
        _sample_rows(args.ref_seconds / (args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_sample(rows)
    tot = 0.0
    flops = 0.0
    for _ in range(args.steps):
        s, f = _oracle_sample(rows)
        tot += s
        flops += f
    value = flops / tot / 1e12
    cores = oracle.num_threads()
    sample = (f"{rows} of {M_TOK} output rows per step: quantize {rows}x{K_IN} (1x128) + "
              f"{N_OUT}x{K_IN} (128x128) + GEMM {rows}x{N_OUT}x{K_IN}, UE8M0, fp64 oracle")
    line = {
        "impl": "reference",
        "metric": "TFLOPS (FP8 block-scaled NT GEMM step, fraction of GB300 dense FP8 tensor peak)",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 codes, f64 accumulate", "data": "synthetic (seeded N(0,1) bf16, 1/1024 outliers x400)",
        "config": {"workload": WORKLOAD, "M": M_TOK, "N": N_OUT, "K": K_IN, "scale_format": "ue8m0",
                   "parallelism": "CPU oracle on the host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="output rows in one oracle sample (0: sized from --cpu-seconds / --ref-seconds)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target length of the cpu_baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=120.0, help="target length of an --impl reference run")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--no-variants", action="store_true", help="skip the extra kernel lines")
    ap.add_argument("--variant", default=None, help="run only the variants whose name starts with this")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
