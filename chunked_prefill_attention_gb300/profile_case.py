"""Run a few attn_chunk_step launches of a reduced prefill problem, for kernel
profiling with Nsight Compute.

The problem keeps the m64k draw (Q, K, V ~ N(0,1), seed 3, 32 heads x 64) at
--tokens tokens split in KV chunks of --chunk keys.  The script quantises K
and V, initialises the state and folds every chunk once (warm-up), then
launches the chunk-step kernel for chunk --index another --reps times on the
same state.  With --tokens 16384 --chunk 8192 --index 1 each profiled launch
is 64 query tiles x 32 heads over 8,192 keys (a full-tile chunk plus its
diagonal), and the device holds about 0.3 GB, above the 129 MB L2.

  ncu --set full --clock-control none -k regex:chunk_step_kernel -s 2 -c 1 \\
      python -m chunked_prefill_attention_gb300.profile_case

With --quantize TOKENS it runs q8kv_quantize instead: the K of the m64k draw
at TOKENS tokens (65536: 537 MB of fp32 in, 143 MB of Q8_0 out, above L2), one
warm-up launch and then --reps launches.

  ncu --set full --clock-control none -k regex:q8kv_quantize -s 1 -c 1 \\
      python -m chunked_prefill_attention_gb300.profile_case --quantize 65536

With --pipelined it runs attn_prefill_pipelined on the m64k draw at --tokens
tokens in chunks of --chunk from page-locked host buffers (one warm-up call,
then --reps calls), so that the DRAM counters of its chunk-step launches can be
set beside those of the device-resident step (where the whole K and V are
quantised before the first chunk step):

  ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none \\
      -k regex:chunk_step_kernel -s 8 -c 8 \\
      python -m chunked_prefill_attention_gb300.profile_case --pipelined --tokens 65536 --reps 1

With --head-dim 128 the chunk-step case takes the m16k_d128 draw (seed 6, 32
heads x 128) instead; --tokens 16384 --chunk 4096 --index 1 profiles a launch
of keys 4,096..8,191 against query rows 4,096..16,383 (0.7 GB on the device):

  ncu --set full --clock-control none -k regex:chunk_step_d128 -s 4 -c 1 \\
      python -m chunked_prefill_attention_gb300.profile_case --head-dim 128 --chunk 4096

With --burst CONTEXT it runs Mode B burst verification instead: the 64
candidates of the burst_m1m draw against a CONTEXT-token, 32-head Q8_0 cache
in key ranges of --split keys (attn_chunk_step_split, paired launches), one
warm-up call and then --reps calls.  --burst 131072 holds 0.57 GB of Q8_0 KV.

  ncu --set full --clock-control none -k regex:chunk_step_kernel -s 1 -c 1 \\
      python -m chunked_prefill_attention_gb300.profile_case --burst 131072
"""

import argparse


def main(argv=None):
    import torch

    from chunked_prefill_attention_gb300 import _build, q8attn as Q, workloads as W

    p = argparse.ArgumentParser()
    p.add_argument("--tokens", type=int, default=16384)
    p.add_argument("--chunk", type=int, default=8192)
    p.add_argument("--index", type=int, default=1)
    p.add_argument("--reps", type=int, default=2)
    p.add_argument("--burst", type=int, default=0)
    p.add_argument("--split", type=int, default=8192)
    p.add_argument("--quantize", type=int, default=0)
    p.add_argument("--pipelined", action="store_true")
    p.add_argument("--head-dim", type=int, default=64, choices=(64, 128))
    a = p.parse_args(argv)
    _build.ensure_built()
    if a.pipelined:
        return pipelined(a)
    if a.burst > 0:
        return burst(a)
    if a.quantize > 0:
        return quantize(a)
    w = W.WORKLOADS["m64k" if a.head_dim == 64 else "m16k_d128"]
    q, k, v = W.make_inputs(w, device="cuda", tokens=a.tokens)
    B, M, H, D = q.shape
    rb = Q.row_bytes(D)
    k8 = Q.q8kv_quantize(k)
    v8 = Q.q8kv_quantize(v)
    st = Q.State(B, H, M, q.device, head_dim=D)
    starts = list(range(0, M, a.chunk))
    for s0 in starts:
        Q.attn_chunk_step(q, k8, v8, s0, min(a.chunk, M - s0), st, k_offset_bytes=s0 * rb)
    s0 = starts[a.index]
    n = min(a.chunk, M - s0)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(a.reps):
        Q.attn_chunk_step(q, k8, v8, s0, n, st, k_offset_bytes=s0 * rb)
    ev[1].record()
    torch.cuda.synchronize()
    rc, status = Q.device_status()
    ms = ev[0].elapsed_time(ev[1]) / a.reps
    rows = M - (s0 // 128) * 128
    print(f"chunk {a.index} (keys {s0}..{s0 + n - 1}, query rows {s0 // 128 * 128}..{M - 1}): "
          f"{ms:.3f} ms per launch, status {rc}")


def pipelined(a):
    import torch

    from chunked_prefill_attention_gb300 import q8attn as Q, workloads as W

    w = W.WORKLOADS["m64k"]
    q, k, v = W.make_inputs(w, device="cuda", tokens=a.tokens)
    B, M, H, D = q.shape
    qh, kh, vh = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    del q, k, v
    oh = torch.empty((B, M, H, D), dtype=torch.float16).pin_memory()
    bufs = Q.PipelineBuffers(B, M, H, torch.device("cuda"), a.chunk)
    Q.attn_prefill_pipelined(qh, kh, vh, oh, bufs)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(a.reps):
        Q.attn_prefill_pipelined(qh, kh, vh, oh, bufs)
    ev[1].record()
    torch.cuda.synchronize()
    rc, _ = Q.device_status()
    ms = ev[0].elapsed_time(ev[1]) / max(a.reps, 1)
    print(f"pipelined prefill {B}x{M}x{H}x{D}, chunks of {a.chunk}: {ms:.3f} ms per call, status {rc}")


def quantize(a):
    import torch

    from chunked_prefill_attention_gb300 import q8attn as Q, workloads as W

    w = W.WORKLOADS["m64k"]
    _, k, _ = W.make_inputs(w, device="cuda", tokens=a.quantize)
    k8 = Q.q8kv_quantize(k)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(a.reps):
        Q.q8kv_quantize(k, k8)
    ev[1].record()
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / a.reps
    B, M, H, D = k.shape
    n_bytes = B * M * H * (D * 4 + 68)
    print(f"quantize {B}x{M}x{H}x{D}: {ms:.4f} ms per launch, {n_bytes / (ms * 1e-3) / 1e9:.0f} GB/s")


def burst(a):
    import torch

    from chunked_prefill_attention_gb300 import q8attn as Q, workloads as W

    b = W.BURSTS["burst_m1m"]
    q, k, v = W.make_burst_inputs(b, device="cuda", context=a.burst)
    M = a.burst
    k8 = Q.q8kv_quantize(k)
    v8 = Q.q8kv_quantize(v)
    del k, v
    ws = torch.empty(Q.split_workspace_floats(1, b.heads, b.queries, M, a.split), dtype=torch.float32,
                     device="cuda")
    st = Q.State(1, b.heads, b.queries, q.device)

    def call():
        Q.attn_state_init(st)
        Q.attn_chunk_step_split(q, k8, v8, 0, M, st, a.split, workspace=ws, q_pos0=M, causal=False)

    call()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(a.reps):
        call()
    ev[1].record()
    torch.cuda.synchronize()
    rc, _ = Q.device_status()
    ms = ev[0].elapsed_time(ev[1]) / a.reps
    kv_bytes = 2 * b.heads * M * Q.ROW_BYTES
    print(f"burst: {b.queries} candidates x {b.heads} heads against {M} keys, ranges of {a.split}: "
          f"{ms:.3f} ms per call, {kv_bytes / (ms * 1e-3) / 1e9:.0f} GB/s of Q8_0 KV, status {rc}")


if __name__ == "__main__":
    main()
