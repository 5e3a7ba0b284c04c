#!/usr/bin/env python
"""Benchmark: chunked Q8_0-KV causal prefill attention on GB300.

One step = the whole hot path over one synthetic problem with inputs resident
in HBM: q8kv_quantize(K), q8kv_quantize(V), attn_state_init, one
attn_chunk_step per KV chunk (on slices of the whole-sequence Q8_0 buffers),
attn_finalize.  Default workload: m64k (1 x 65,536 tokens, 32 heads x 64,
causal, 8 KV chunks of 8,192).

Prints one JSON line (rank 0).  value = causal attention TFLOP/s of the whole
job: 4*D*B*H*M(M+1)/2 flops per replica per step, summed over ranks, divided
by the max-over-ranks time of the timed steps.  With --gpus N > 1 every rank
runs an independent replica (the path does not shard; weak scaling).

--impl reference times the CPU oracle (fp64 numpy, worker pool on the host
cores) on a bounded prefix of the same workload and prints the same line with
"impl": "reference".
"""

import argparse
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

METRIC = "causal Q8_0-KV prefill attention TFLOP/s & % FP16 tensor peak; tokens/s"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ host side --

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="m64k")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) leg")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle CPU baseline")
    p.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi clocks")
    p.add_argument("--other-workloads", default="m512,m2k_out,b8_m2k,m1m,m16k_d128",
                   help="comma-separated workloads also timed (one GPU only) and reported under "
                        "'workloads'; empty to skip")
    return p.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def dist_barrier(dist):
    if dist is not None:
        dist.barrier()


def dist_max(dist, x):
    """Max of a float over ranks (identity for one rank)."""
    if dist is None:
        return float(x)
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def quantize_record(B, M, H, D, ms, peaks, peak_src):
    """HBM roofline of the two q8kv_quantize launches of a step (K and V):
    fp32 read (4 B per value) plus Q8_0 written (34 B per 32 values)."""
    n_bytes = 2 * B * M * H * (D * 4 + (D // 32) * 34)
    gbs = n_bytes / (ms * 1e-3) / 1e9 if ms > 0 else None
    hbm = float(peaks.get("hbm_gbs"))
    return {"kernel": "q8kv_quantize (K and V)", "bound": "hbm", "ms_per_step": ms,
            "algorithmic_bytes": n_bytes, "achieved": gbs, "peak": hbm, "unit": "GB/s",
            "frac": gbs / hbm if gbs else None, "peak_kind": f"HBM copy, {peak_src}"}


def hbm_record(kernel, n_bytes, ms, peaks, peak_src, algorithmic):
    """HBM roofline of one launch per step of an HBM-bound kernel."""
    gbs = n_bytes / (ms * 1e-3) / 1e9 if ms > 0 else None
    hbm = float(peaks.get("hbm_gbs"))
    return {"kernel": kernel, "bound": "hbm", "ms_per_step": ms, "algorithmic_bytes": n_bytes,
            "algorithmic": algorithmic, "achieved": gbs, "peak": hbm, "unit": "GB/s",
            "frac": gbs / hbm if gbs else None, "peak_kind": f"HBM copy, {peak_src}"}


def make_record(*, value, n_gpus, steps, warmup, ms_per_step, config, extra):
    rec = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": n_gpus, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded torch.randn on the device)",
        "config": config,
    }
    rec.update(extra)
    return rec


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [s for s in sm if mx and s > 0.3 * max(mx)]
        return {"sm_mhz": statistics.median(busy or sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


def profile_traffic(kernel_src):
    """DRAM bytes per launch of the chunk-step kernel from the committed ncu
    summary, or None when the kernel source changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "chunk_step_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        with open(kernel_src, "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
        if rec.get("kernel_sha256_16") != h:
            return None, "stale"
        return rec, "ok"
    except Exception:
        return None, "absent"


def step_hbm_bytes(w):
    """Algorithmic HBM bytes of one step of workload w (head_dim D; the figures
    in brackets are D = 64): quantise K and V (4D B fp32 in + D/32*34 B Q8_0 out
    per head row each [256 + 68]), state init (4(2 + D) B per state row [264]),
    one chunk step per KV chunk (per state row it touches: 2D B of Q and
    2 x 4(2 + D) B of state [128 + 528]; per chunk key and head: 2 x D/32*34 B
    of Q8_0 K and V [136]), finalise (4(1 + D) B in + 2D B out per state row
    [260 + 128])."""
    B, M, H, D = w.batch, w.tokens, w.heads, w.head_dim
    row8 = D // 32 * 34
    state = 4 * (2 + D)
    rows = B * H * M
    total = 2 * rows * (4 * D + row8) + rows * state + rows * (4 * (1 + D) + 2 * D)
    for s0 in range(0, M, w.chunk):
        n = min(w.chunk, M - s0)
        total += B * H * (M - s0) * (2 * D + 2 * state) + B * H * n * 2 * row8
    return total


def time_workload(name, steps, warmup, peaks, peak_src, flush_l2, sample_clocks):
    """Time the whole step of another workload on the current device: each
    step bracketed by its own CUDA events (and, for problems smaller than L2,
    preceded by a write of a 256 MB buffer outside the events).  Returns its
    record for the 'workloads' key."""
    import torch
    from chunked_prefill_attention_gb300 import q8attn as Q, workloads as W
    w = W.WORKLOADS[name]
    dev = torch.cuda.current_device()
    B, M, H, D = w.batch, w.tokens, w.heads, w.head_dim
    q, k, v = W.make_inputs(w, device=torch.device("cuda", dev))
    stride = Q.plane_stride(M, D)
    k8 = torch.empty((B, H, stride), dtype=torch.uint8, device=q.device)
    v8 = torch.empty((B, H, stride), dtype=torch.uint8, device=q.device)
    st = Q.State(B, H, M, q.device, init=False, head_dim=D)
    out = torch.empty((B, M, H, D), dtype=torch.float16, device=q.device)
    chunks = [(s0, min(w.chunk, M - s0)) for s0 in range(0, M, w.chunk)]
    stream = torch.cuda.current_stream()
    scratch = torch.empty((256 << 20,), dtype=torch.uint8, device=q.device) if flush_l2 else None

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        Q.q8kv_quantize(k, k8, stride)
        Q.q8kv_quantize(v, v8, stride)
        Q.attn_state_init(st)
        if ev is not None:
            ev[1].record(stream)
        for s0, n in chunks:
            Q.attn_chunk_step(q, k8, v8, s0, n, st, k_offset_bytes=s0 * Q.row_bytes(D))
        if ev is not None:
            ev[2].record(stream)
        Q.attn_finalize(st, out)
        if ev is not None:
            ev[3].record(stream)

    def timed(one_step, n_events):
        for _ in range(warmup):
            one_step()
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)] for _ in range(steps)]
        for s in range(steps):
            if scratch is not None:
                scratch.zero_()
            one_step(evs[s])
        torch.cuda.synchronize()
        rc, status = Q.device_status()
        if rc != 0:
            raise RuntimeError(f"device status {status:#x} after timing {name}")
        return evs

    tensor_bound = w.tokens >= 65536 or D == 128
    clocks = ClockSampler(dev) if sample_clocks else None
    if clocks:
        clocks.start()
    evs = timed(step, 4)
    ms_calls = sum(e[0].elapsed_time(e[3]) for e in evs) / steps
    chunk_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / steps
    ms, graph_note = ms_calls, None
    if not tensor_bound:
        # the same step captured once into a CUDA graph (q8a_prefill_graph) and
        # replayed with one launch: the kernels no longer wait on the host
        g = Q.PrefillGraph(q, k, v, w.chunk)

        def graph_step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            g.launch(stream)
            if ev is not None:
                ev[1].record(stream)

        gevs = timed(graph_step, 2)
        ms = sum(e[0].elapsed_time(e[1]) for e in gevs) / steps
        graph_note = "one q8a_prefill_graph replay per step (the same %d launches)" % (4 + len(chunks))
        g.close()
    clk = clocks.stop() if clocks else None
    tflops = w.causal_flops / (ms * 1e-3) / 1e12
    rec = {"workload": w.describe(), "ms_per_step": ms, "tflops": tflops,
           "tokens_per_s": B * M / (ms * 1e-3), "steps": steps, "warmup": warmup,
           "l2": ("L2 flushed before each step (256 MB write outside the timed events)" if flush_l2
                  else "inputs larger than L2")}
    if graph_note:
        rec["launch"] = graph_note
        rec["ms_per_step_launch_by_launch"] = ms_calls
    if tensor_bound:
        peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
        achieved = w.causal_flops / (chunk_ms * 1e-3) / 1e12
        rec["roofline"] = {"bound": "tensor", "kernel": "attn_chunk_step", "achieved": achieved,
                           "peak": peak, "unit": UNIT, "frac": achieved / peak,
                           "peak_kind": f"dense bf16/fp16 {peak_src} sustained",
                           "ms_attn_chunks_per_step": chunk_ms}
    else:
        hbm = float(peaks.get("hbm_gbs"))
        n_bytes = step_hbm_bytes(w)
        gbs = n_bytes / (ms * 1e-3) / 1e9
        rec["roofline"] = {"bound": "hbm", "kernel": "whole step (%d kernels)" % (4 + len(chunks)),
                           "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                           "algorithmic_bytes": n_bytes, "peak_kind": f"HBM copy, {peak_src}"}
    rec["clocks"] = clk
    del q, k, v, k8, v8, st, out, scratch
    torch.cuda.empty_cache()
    return rec


# ------------------------------------------------------------------ our arm --

def run_ours(args):
    import torch
    from chunked_prefill_attention_gb300 import _build, q8attn as Q, workloads as W

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dist = dist_init(world, "nccl")
    _build.ensure_built()
    w = W.WORKLOADS[args.workload]
    dev = torch.device("cuda", local_rank)
    B, M, H, D = w.batch, w.tokens, w.heads, w.head_dim
    q, k, v = W.make_inputs(w, device=dev)
    stride = Q.plane_stride(M, D)
    k8 = torch.empty((B, H, stride), dtype=torch.uint8, device=dev)
    v8 = torch.empty((B, H, stride), dtype=torch.uint8, device=dev)
    st = Q.State(B, H, M, dev, init=False, head_dim=D)
    out = torch.empty((B, M, H, D), dtype=torch.float16, device=dev)
    chunks = [(s0, min(w.chunk, M - s0)) for s0 in range(0, M, w.chunk)]
    stream = torch.cuda.current_stream(dev)

    def step(ev=None, qev=None):
        if qev is not None:
            qev[0].record(stream)
        Q.q8kv_quantize(k, k8, stride)
        Q.q8kv_quantize(v, v8, stride)
        if qev is not None:
            qev[1].record(stream)
        Q.attn_state_init(st)
        if qev is not None:
            qev[2].record(stream)
        for i, (s0, n) in enumerate(chunks):
            if ev is not None:
                ev[i][0].record(stream)
            Q.attn_chunk_step(q, k8, v8, s0, n, st, k_offset_bytes=s0 * Q.row_bytes(D))
            if ev is not None:
                ev[i][1].record(stream)
        if qev is not None:
            qev[3].record(stream)
        Q.attn_finalize(st, out)
        if qev is not None:
            qev[4].record(stream)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    rc, status = Q.device_status()
    if rc != 0:
        raise RuntimeError(f"device status {status:#x} after warm-up")

    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in chunks]
           for _ in range(args.steps)]
    qevs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(5)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = None if args.no_clocks else ClockSampler(local_rank)
    dist_barrier(dist)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    t0.record(stream)
    for s in range(args.steps):
        step(evs[s], qevs[s])
    t1.record(stream)
    torch.cuda.synchronize()
    dist_barrier(dist)
    clk = clocks.stop() if clocks else None
    ms = t0.elapsed_time(t1) / args.steps
    chunk_ms = sum(a.elapsed_time(b) for per in evs for a, b in per) / args.steps
    quant_ms = sum(e[0].elapsed_time(e[1]) for e in qevs) / args.steps
    init_ms = sum(e[1].elapsed_time(e[2]) for e in qevs) / args.steps
    fin_ms = sum(e[3].elapsed_time(e[4]) for e in qevs) / args.steps
    launches_chunk = len(chunks)
    ms_max = dist_max(dist, ms)
    rc, status = Q.device_status()
    if rc != 0:
        raise RuntimeError(f"device status {status:#x} after the timed steps")

    flops = w.causal_flops
    value = world * flops / (ms_max * 1e-3) / 1e12
    tokens_s = world * B * M / (ms_max * 1e-3)
    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    peak_burst = float(peaks.get("bf16_tflops"))
    achieved = flops / (chunk_ms * 1e-3) / 1e12          # all chunk launches of one step
    traffic_rec, traffic_state = profile_traffic(
        os.path.join(ROOT, "chunked_prefill_attention_gb300", "csrc", "chunk_step.cu"))
    traffic = None
    if traffic_rec is not None and traffic_rec.get("workload") == w.name:
        traffic = traffic_rec.get("dram_bytes_per_launch")

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        qh = q.cpu().pin_memory()
        kh = k.cpu().pin_memory()
        vh = v.cpu().pin_memory()
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        bufs = Q.PipelineBuffers(B, M, H, dev, w.chunk, head_dim=D)

        def e2e_step():
            # attn_prefill_pipelined: K/V chunk copies overlap quantise + chunk steps
            Q.attn_prefill_pipelined(qh, kh, vh, oh, bufs)

        e2e_step()
        torch.cuda.synchronize()
        dist_barrier(dist)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        dist_barrier(dist)
        e_ms = dist_max(dist, a.elapsed_time(b) / args.steps)
        e2e = {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": int(qh.nbytes + kh.nbytes + vh.nbytes),
               "d2h_bytes_per_step": int(oh.nbytes)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, q, k, v, budget_s=30.0)

    others = {}
    names = [n for n in args.other_workloads.split(",") if n and n != w.name]
    if world == 1 and names:
        bufs = None
        del q, k, v, k8, v8, out
        torch.cuda.empty_cache()
        for name in names:
            big = W.WORKLOADS[name].tokens >= 1 << 20
            others[name] = time_workload(name, 2 if big else 20, 1 if big else 3, peaks, peak_src,
                                         flush_l2=W.WORKLOADS[name].tokens < 65536,
                                         sample_clocks=big and not args.no_clocks)

    n_launch = args.steps * (3 + len(chunks) + 1)
    config = {
        "workload": w.describe(), "batch": B, "tokens": M, "heads": H, "head_dim": D,
        "kv_chunk": w.chunk, "kv_chunks": len(chunks), "replicas": world,
        "l2": "inputs larger than L2: K, V fp32 %.2f GB, Q fp16 %.2f GB, Q8_0 KV %.2f GB, state %.2f GB"
              % (2 * B * M * H * D * 4 / 1e9, B * M * H * D * 2 / 1e9, 2 * B * H * stride / 1e9,
                 (st.m.nbytes + st.l.nbytes + st.o.nbytes) / 1e9),
    }
    attn_ms = chunk_ms + init_ms + fin_ms   # the step without the two quantise launches
    extra = {
        "tokens_per_s": tokens_s,
        "pct_fp16_peak": 100.0 * value / (world * peak_sus),
        "ms_attn_chunks_per_step": chunk_ms,
        # the metric's own time base: every attn_chunk_step launch + init + finalise
        "attention": {"ms_per_step": attn_ms, "tflops": flops / (attn_ms * 1e-3) / 1e12,
                      "tokens_per_s": B * M / (attn_ms * 1e-3),
                      "excludes": "the two q8kv_quantize launches (reported under quantize)"},
        # one exponential per unmasked score, over the chunk launches
        "exp_per_s": w.causal_pairs / (chunk_ms * 1e-3),
        "roofline": {"bound": "tensor", "kernel": "attn_chunk_step", "achieved": achieved,
                     "peak": peak_sus, "unit": UNIT, "frac": achieved / peak_sus,
                     "peak_kind": f"dense bf16/fp16 {peak_src} sustained (burst {peak_burst})",
                     "algorithmic": "4*D flops per unmasked (query, key) pair; %d launches/step" % launches_chunk,
                     "traffic": traffic, "traffic_note": traffic_state},
        "quantize": quantize_record(B, M, H, D, quant_ms, peaks, peak_src),
        "state_init": hbm_record("attn_state_init", B * H * M * 4 * (2 + D), init_ms, peaks, peak_src,
                                 "%d B written per state row (m, l, %d O)" % (4 * (2 + D), D)),
        "finalize": hbm_record("attn_finalize", B * H * M * (4 * (1 + D) + 2 * D), fin_ms, peaks, peak_src,
                               "%d B read (l, %d O) + %d B fp16 written per state row"
                               % (4 * (1 + D), D, 2 * D)),
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": n_launch,
        "cpu_baseline": cpu,
        "workloads": others or None,
    }
    rec = make_record(value=value, n_gpus=world, steps=args.steps, warmup=args.warmup,
                      ms_per_step=ms_max, config=config, extra=extra)
    if rank == 0:
        print(json.dumps(rec), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------ Mode B (burst) arm --

def run_burst(args):
    """Mode B speculative burst verification: the context's Q8_0 KV cache is
    resident (quantised before timing); one step = state init for the 64
    candidates, attn_chunk_step_split over the whole context, finalise.  value =
    Q8_0 KV bytes read per step / step time (GB/s), against the measured HBM
    copy bandwidth."""
    import torch
    from chunked_prefill_attention_gb300 import _build, q8attn as Q, workloads as W

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dist = dist_init(world, "nccl")
    _build.ensure_built()
    b = W.BURSTS[args.workload]
    dev = torch.device("cuda", local_rank)
    q, k, v = W.make_burst_inputs(b, device=dev)
    M, H = b.context, b.heads
    k8 = Q.q8kv_quantize(k)
    v8 = Q.q8kv_quantize(v)
    del k, v
    torch.cuda.empty_cache()
    st = Q.State(1, H, b.queries, dev, init=False)
    out = torch.empty((1, b.queries, H, b.head_dim), dtype=torch.float16, device=dev)
    # CTAs per key range: one per (b, h), or with grouped-query packing one per
    # (b, K/V head) and 256 (candidate, head) rows
    group = H // b.kv_h
    packed = group >= 2 and 128 % group == 0 and b.head_dim == 64
    ctas = b.kv_h * -(-b.queries * group // 256) if packed else H
    split = b.split_keys or Q.split_keys_for(ctas, M, torch.cuda.get_device_properties(dev).multi_processor_count)
    ws = torch.empty(Q.split_workspace_floats(1, H, b.queries, M, split), dtype=torch.float32,
                     device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        Q.attn_state_init(st)
        if b.kv_h != H:
            Q.attn_chunk_step_split_gqa(q, k8, v8, 0, M, st, split, workspace=ws, q_pos0=M, causal=False)
        else:
            Q.attn_chunk_step_split(q, k8, v8, 0, M, st, split, workspace=ws, q_pos0=M,
                                    causal=False)
        Q.attn_finalize(st, out)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    rc, status = Q.device_status()
    if rc != 0:
        raise RuntimeError(f"device status {status:#x} after warm-up")
    clocks = None if args.no_clocks else ClockSampler(local_rank)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(dist)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    dist_barrier(dist)
    clk = clocks.stop() if clocks else None
    ms = dist_max(dist, t0.elapsed_time(t1) / args.steps)
    rc, status = Q.device_status()
    if rc != 0:
        raise RuntimeError(f"device status {status:#x} after the timed steps")
    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs"))
    gbs = world * b.kv_bytes / (ms * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        qh = q.cpu().pin_memory()
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        def e2e_step():
            q.copy_(qh, non_blocking=True)
            step()
            oh.copy_(out, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            e2e_step()
        c.record(stream)
        torch.cuda.synchronize()
        e_ms = dist_max(dist, a.elapsed_time(c) / args.steps)
        e2e = {"value": world * b.kv_bytes / (e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": int(qh.nbytes), "d2h_bytes_per_step": int(oh.nbytes)}
    config = {"workload": b.describe(), "batch": 1, "tokens": M, "queries": b.queries, "heads": H,
              "head_dim": b.head_dim, "split_keys": split, "key_ranges": -(-M // split), "replicas": world,
              "l2": "Q8_0 KV %.2f GB, larger than L2" % (b.kv_bytes / 1e9)}
    tflops = world * b.flops / (ms * 1e-3) / 1e12
    peak_t = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    hbm_roof = {"bound": "hbm", "kernel": "attn_chunk_step_split + merge", "achieved": gbs,
                "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "peak_kind": f"HBM copy bandwidth, {peak_src}",
                "algorithmic": "2*H_kv*M*(D/32*34) bytes of Q8_0 K and V per step", "traffic": None}
    tensor_roof = {"bound": "tensor", "kernel": "attn_chunk_step_split + merge", "achieved": tflops,
                   "peak": peak_t, "unit": "TFLOP/s", "frac": tflops / peak_t,
                   "peak_kind": f"dense bf16/fp16 {peak_src} sustained",
                   "algorithmic": "4*D flops per (candidate, context key) pair and query head", "traffic": None}
    # the binding resource: a grouped-query burst reads each K/V plane once for
    # several query heads, so it can be bound by the tensor work instead
    extra = {
        "candidate_tokens_per_s": world * b.queries / (ms * 1e-3),
        "tflops": tflops,
        "roofline": hbm_roof if hbm_roof["frac"] >= tensor_roof["frac"] else tensor_roof,
        "roofline_other": tensor_roof if hbm_roof["frac"] >= tensor_roof["frac"] else hbm_roof,
        "clocks": clk, "e2e": e2e, "gpu_launches": args.steps * 4, "cpu_baseline": None,
    }
    rec = make_record(value=gbs, n_gpus=world, steps=args.steps, warmup=args.warmup,
                      ms_per_step=ms, config=config, extra=extra)
    rec["metric"] = "Mode B speculative burst verification over a Q8_0 KV cache: KV GB/s"
    rec["unit"] = "GB/s"
    if rank == 0:
        print(json.dumps(rec), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------- CPU oracle --

def _oracle_prefix(qn, kn, vn, n_tok, pool):
    """Run the oracle's whole path on the first n_tok tokens: quantise K and V,
    then plain causal attention for every row of every (b, h) plane."""
    B, M, H, D = qn.shape
    kq = pool.map(_quant_slice, [kn[:, :n_tok, h:h + 1] for h in range(H)])
    vq = pool.map(_quant_slice, [vn[:, :n_tok, h:h + 1] for h in range(H)])
    tasks = []
    rows = list(range(n_tok))
    import numpy as np
    for b in range(B):
        for h in range(H):
            tasks.append((qn[b, :n_tok, h].astype(np.float64), np.asarray(rows), kq[h][b, 0], vq[h][b, 0],
                          1.0 / math.sqrt(D), True, 0))
    from oracle.runner import _attn_task
    pool.map(_attn_task, tasks, chunksize=1)


def _quant_slice(x):
    from oracle import q8_0
    return q8_0.quantize_kv(x)


def _oracle_pool():
    from oracle import runner as oracle_runner
    return oracle_runner.pool(), oracle_runner.workers()


def cpu_baseline(w, q, k, v, budget_s=20.0):
    """The oracle (as it stands) on the host cores, on a prefix of the
    workload sized to take about `budget_s` seconds."""
    pool, cores = _oracle_pool()
    n_tok = 1024
    cap = min(w.tokens, 32768)
    qn = q[:, :cap].cpu().numpy()
    kn = k[:, :cap].cpu().numpy()
    vn = v[:, :cap].cpu().numpy()
    while True:
        t = time.perf_counter()
        _oracle_prefix(qn, kn, vn, n_tok, pool)
        dt = time.perf_counter() - t
        if dt * 3.5 > budget_s or 2 * n_tok > qn.shape[1]:
            break
        n_tok *= 2
    flops = 4 * w.head_dim * w.batch * w.heads * n_tok * (n_tok + 1) // 2
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "seconds": dt,
            "sample": f"first {n_tok} tokens of {w.name} (all {w.heads} heads): oracle Q8_0 quantise of "
                      f"K and V + fp64 plain causal attention of every row, numpy, {cores} spawn workers"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import torch
    from chunked_prefill_attention_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    pool, cores = _oracle_pool()
    total = max(1, args.steps + args.warmup)
    n_tok = 2048 if total <= 20 else 1024
    q, k, v = W.make_inputs(w, device="cpu", tokens=n_tok)
    qn, kn, vn = q.numpy(), k.numpy(), v.numpy()
    for _ in range(args.warmup):
        _oracle_prefix(qn, kn, vn, n_tok, pool)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_prefix(qn, kn, vn, n_tok, pool)
    dt = (time.perf_counter() - t) / max(args.steps, 1)
    flops = 4 * w.head_dim * w.batch * w.heads * n_tok * (n_tok + 1) // 2
    value = flops / dt / 1e12
    sample = (f"per step: first {n_tok} tokens of {w.name} (all {w.heads} heads): oracle Q8_0 quantise of K "
              f"and V + fp64 plain causal attention of every row, numpy, {cores} spawn workers")
    config = {"workload": w.describe(), "batch": w.batch, "tokens": w.tokens, "heads": w.heads,
              "head_dim": w.head_dim, "kv_chunk": w.chunk, "replicas": 1, "l2": "n/a (host CPU)"}
    extra = {"impl": "reference", "dtype": "f64",
             "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
             "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
             "gpu_launches": 0}
    rec = make_record(value=value, n_gpus=world, steps=args.steps, warmup=args.warmup,
                      ms_per_step=dt * 1e3, config=config, extra=extra)
    rec["dtype"] = "f64"
    rec["data"] = "synthetic (seeded torch.randn on the host)"
    print(json.dumps(rec), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload.startswith("burst_"):
        run_burst(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
