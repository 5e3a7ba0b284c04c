"""Seeded random problem shapes through every entry point, against the oracle:
batch, tokens, heads, head dimension, chunk length, mask, query offset and the
call used (chunk by chunk, captured graph, split key ranges, pipelined from host
buffers) are drawn from a fixed generator, so each case is reproducible from
its index.  Q8_0 bytes must match bit for bit and the output must be within the
parity tolerance ("Out-of-Core Flash Streaming & Speculative Decode (1M
Context)", §3: the chunked result equals the plain definition)."""

import numpy as np
import pytest
import torch

from tests.conftest import cuda_available
from tests.parity import assert_device_clean, compare, gpu_bytes, oracle_out, seeded

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

N_CASES = 24


def _case(i):
    rng = np.random.default_rng(1000 + i)
    D = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 3))
    H = int(rng.integers(1, 5))
    M = int(rng.integers(1, 1400))
    align = 4 if D == 64 else 2
    chunk = int(rng.integers(1, 700) // align * align) or align
    path = ["steps", "graph", "split", "pipelined"][i % 4]
    causal = bool(rng.integers(0, 4)) if path != "split" else bool(rng.integers(0, 2))
    if path == "pipelined":
        chunk = max(4, chunk // 4 * 4)
    n_q, q_pos0 = M, 0
    if not causal and path in ("steps", "split") and rng.integers(0, 2):
        n_q, q_pos0 = int(rng.integers(1, 200)), M   # candidates after the context
    split = int(rng.integers(1, 9)) * 128
    return dict(D=D, B=B, H=H, M=M, chunk=chunk, path=path, causal=causal, n_q=n_q, q_pos0=q_pos0,
                split=split, seed=2000 + 3 * i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(lib, i):
    from chunked_prefill_attention_gb300 import q8attn as Q
    c = _case(i)
    D, B, H, M, chunk, n_q, q_pos0 = c["D"], c["B"], c["H"], c["M"], c["chunk"], c["n_q"], c["q_pos0"]
    q = seeded((B, n_q, H, D), c["seed"], "cuda", torch.float16)
    k = seeded((B, M, H, D), c["seed"] + 1, "cuda")
    v = seeded((B, M, H, D), c["seed"] + 2, "cuda")
    rb = Q.row_bytes(D)
    if c["path"] == "graph":
        g = Q.PrefillGraph(q, k, v, chunk, causal=c["causal"])
        out = g.launch().clone()
        k8, v8 = g.k8, g.v8
        torch.cuda.synchronize()
        g.close()
    elif c["path"] == "pipelined":
        qh, kh, vh = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
        oh = torch.zeros((B, M, H, D), dtype=torch.float16).pin_memory()
        bufs = Q.PipelineBuffers(B, M, H, q.device, chunk, head_dim=D)
        Q.attn_prefill_pipelined(qh, kh, vh, oh, bufs, causal=c["causal"])
        torch.cuda.current_stream().synchronize()
        out, k8, v8 = oh, bufs.k8, bufs.v8
    else:
        k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
        st = Q.State(B, H, n_q, q.device, head_dim=D)
        for s0 in range(0, M, chunk):
            n = min(chunk, M - s0)
            if c["path"] == "split":
                Q.attn_chunk_step_split(q, k8, v8, s0, n, st, c["split"], q_pos0=q_pos0, causal=c["causal"],
                                        k_offset_bytes=s0 * rb)
            else:
                Q.attn_chunk_step(q, k8, v8, s0, n, st, q_pos0=q_pos0, causal=c["causal"],
                                  k_offset_bytes=s0 * rb)
        out = Q.attn_finalize(st)
    assert_device_clean()
    want, wk8, wv8 = oracle_out(q, k, v, causal=c["causal"], q_pos0=q_pos0)
    assert np.array_equal(gpu_bytes(k8, M, D), wk8) and np.array_equal(gpu_bytes(v8, M, D), wv8), c
    compare(out.cpu().numpy(), want, f"case {i}: {c}")
