"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, compare."""

import math

import numpy as np
import torch

from chunked_prefill_attention_gb300 import q8attn as Q
from oracle import runner as oracle_runner

# Attention tolerance: fp16 output with fp32 accumulation against the fp64
# oracle on identical dequantised KV.
MAX_ABS = 2e-3
REL_L2 = 1e-3


def gpu_bytes(planes, n_tokens, head_dim=64):
    """uint8 [B, H, stride] device planes -> numpy [B, H, n_tokens, head_dim/32*34]."""
    B, H, _ = planes.shape
    rb = Q.row_bytes(head_dim)
    return planes[:, :, :n_tokens * rb].reshape(B, H, n_tokens, rb).cpu().numpy()


def run_gpu(q, k, v, chunk, causal=True, scale=None, q_pos0=0, order=None):
    """Quantise K, V and fold every chunk (in `order`) on the GPU.
    Returns (out fp16 [B, n_q, H, 64] on device, k8, v8, state)."""
    B, n_q, H, D = q.shape
    M = k.shape[1]
    k8 = Q.q8kv_quantize(k)
    v8 = Q.q8kv_quantize(v)
    st = Q.State(B, H, n_q, q.device, head_dim=D)
    starts = list(range(0, M, chunk))
    if order is not None:
        starts = [starts[i] for i in order]
    for s0 in starts:
        Q.attn_chunk_step(q, k8, v8, s0, min(chunk, M - s0), st, q_pos0=q_pos0, scale=scale,
                          causal=causal, k_offset_bytes=s0 * Q.row_bytes(D))
    out = Q.attn_finalize(st)
    assert_device_clean()
    return out, k8, v8, st


def assert_device_clean():
    """No device-side wait ran out since the last check (clears the word)."""
    rc, status = Q.device_status(clear=True)
    assert rc == Q.Q8A_OK, f"device status word {status:#x}: a device-side wait ran out"


def oracle_out(q, k, v, causal=True, scale=None, rows=None, q_pos0=0):
    """Oracle quantisation of the same fp32 K, V and plain attention.
    Returns (out fp64 [B, rows, H, 64], k8 bytes, v8 bytes)."""
    qn = q.cpu().numpy()
    k8 = oracle_runner.quantize_kv(k.cpu().numpy())
    v8 = oracle_runner.quantize_kv(v.cpu().numpy())
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    out = oracle_runner.attention(qn, k8, v8, scale, causal=causal, rows=rows, q_pos0=q_pos0)
    return out, k8, v8


def compare(got, want, what=""):
    """got: fp16/fp32 array, want: fp64 oracle.  Asserts the tolerance and
    returns (max_abs, rel_l2, |want| at the worst element)."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    i = int(np.argmax(err))
    max_abs = float(err.flat[i])
    rel = float(np.sqrt(np.sum(err ** 2) / max(np.sum(want ** 2), 1e-300)))
    msg = f"{what}: max|err| {max_abs:.3e} at |out| {abs(want.flat[i]):.3f}, rel-L2 {rel:.3e}"
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    assert max_abs <= MAX_ABS, msg
    assert rel <= REL_L2, msg
    return max_abs, rel, abs(float(want.flat[i]))


def seeded(shape, seed, device, dtype=torch.float32, scale=1.0):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * scale).to(dtype)
