"""attn_chunk_step_gqa (query heads sharing K/V heads) against the oracle's
grouped-query mapping: query head h of H reads K/V head h // (H / H_kv).
Grouping is an extension beyond the source pages; the oracle's mapping is
pinned in test_oracle_pins.py."""

import numpy as np
import pytest
import torch

from tests.conftest import cuda_available
from tests.parity import assert_device_clean, compare, seeded

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _run(q, k, v, chunk, causal=True, q_pos0=0):
    from chunked_prefill_attention_gb300 import q8attn as Q
    B, n_q, H, _ = q.shape
    M = k.shape[1]
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(B, H, n_q, q.device)
    for s0 in range(0, M, chunk):
        Q.attn_chunk_step_gqa(q, k8, v8, s0, min(chunk, M - s0), st, q_pos0=q_pos0, causal=causal,
                              k_offset_bytes=s0 * 68)
    out = Q.attn_finalize(st)
    assert_device_clean()
    return out, k8, v8


def _oracle(q, k8, v8, M, causal=True, q_pos0=0):
    from oracle import runner
    from tests.parity import gpu_bytes
    return runner.attention(q.cpu().numpy(), gpu_bytes(k8, M), gpu_bytes(v8, M), 0.125, causal=causal,
                            q_pos0=q_pos0)


@pytest.mark.parametrize("B,M,H,H_kv,chunk", [(1, 1000, 8, 2, 256), (2, 600, 4, 1, 600), (1, 777, 6, 3, 384)])
def test_gqa_causal_prefill(lib, B, M, H, H_kv, chunk):
    from oracle import runner
    q = seeded((B, M, H, 64), M + 70, "cuda", torch.float16)
    k = seeded((B, M, H_kv, 64), M + 71, "cuda")
    v = seeded((B, M, H_kv, 64), M + 72, "cuda")
    out, k8, v8 = _run(q, k, v, chunk)
    from tests.parity import gpu_bytes
    assert np.array_equal(gpu_bytes(k8, M), runner.quantize_kv(k.cpu().numpy()))
    compare(out.cpu().numpy(), _oracle(q, k8, v8, M), f"gqa B{B} M{M} H{H}/{H_kv}")


def test_gqa_burst_rectangular(lib):
    """64 candidates after a 3,000-token context, 8 query heads on 2 K/V heads,
    no mask (one query tile: the paired launch)."""
    M, H, H_kv = 3000, 8, 2
    q = seeded((1, 64, H, 64), 81, "cuda", torch.float16)
    k = seeded((1, M, H_kv, 64), 82, "cuda")
    v = seeded((1, M, H_kv, 64), 83, "cuda")
    out, k8, v8 = _run(q, k, v, M, causal=False, q_pos0=M)
    compare(out.cpu().numpy(), _oracle(q, k8, v8, M, causal=False, q_pos0=M), "gqa burst")


def test_gqa_with_equal_head_counts_is_the_plain_step(lib):
    """kv_heads == heads takes the same path as attn_chunk_step: bitwise equal."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    M, H = 700, 4
    q = seeded((1, M, H, 64), 91, "cuda", torch.float16)
    k8 = Q.q8kv_quantize(seeded((1, M, H, 64), 92, "cuda"))
    v8 = Q.q8kv_quantize(seeded((1, M, H, 64), 93, "cuda"))
    a = Q.State(1, H, M, q.device)
    b = Q.State(1, H, M, q.device)
    Q.attn_chunk_step(q, k8, v8, 0, M, a)
    Q.attn_chunk_step_gqa(q, k8, v8, 0, M, b)
    assert_device_clean()
    assert torch.equal(a.m, b.m) and torch.equal(a.l, b.l) and torch.equal(a.o, b.o)


@pytest.mark.parametrize("D,M,H,H_kv,split,n_q,B", [(64, 20000, 8, 2, 2048, 64, 1), (128, 5000, 6, 3, 1024, 64, 1),
                                                     (64, 3000, 4, 1, 384, 64, 1), (64, 4000, 16, 2, 512, 70, 2),
                                                     (64, 2500, 8, 4, 1024, 64, 1), (64, 1800, 8, 1, 256, 33, 1),
                                                     (64, 1000, 6, 2, 128, 64, 1)])
def test_gqa_split_burst(lib, D, M, H, H_kv, split, n_q, B):
    """Burst verification for a grouped-query model: candidates after the
    context, the keys folded in parallel ranges over the shared K/V planes.  At
    head_dim 64 with a group of 2, 4 or 8 heads the tiles take (candidate,
    head) pairs of one group (70 candidates x 8 heads: a ragged last tile whose
    extra rows read the next sequence's queries and stay inactive; a group of
    3 is not a divisor of 128 and keeps one head per tile)."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    from oracle import runner
    from tests.parity import gpu_bytes
    q = seeded((B, n_q, H, D), M + D, "cuda", torch.float16)
    k = seeded((B, M, H_kv, D), M + D + 1, "cuda")
    v = seeded((B, M, H_kv, D), M + D + 2, "cuda")
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(B, H, n_q, q.device, head_dim=D)
    Q.attn_chunk_step_split_gqa(q, k8, v8, 0, M, st, split, q_pos0=M, causal=False)
    out = Q.attn_finalize(st)
    assert_device_clean()
    want = runner.attention(q.cpu().numpy(), gpu_bytes(k8, M, D), gpu_bytes(v8, M, D), 1.0 / np.sqrt(D),
                            causal=False, q_pos0=M)
    compare(out.cpu().numpy(), want, f"gqa split burst D{D} H{H}/{H_kv}")


def test_gqa_split_causal_matches_unsplit(lib):
    """Causal chunks folded with the grouped-query split and without it agree
    within the parity tolerance, and the split output matches the oracle."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    M, H, H_kv, chunk = 1100, 6, 2, 512
    q = seeded((1, M, H, 64), 95, "cuda", torch.float16)
    k = seeded((1, M, H_kv, 64), 96, "cuda")
    v = seeded((1, M, H_kv, 64), 97, "cuda")
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, M, q.device)
    for s0 in range(0, M, chunk):
        Q.attn_chunk_step_split_gqa(q, k8, v8, s0, min(chunk, M - s0), st, 256, k_offset_bytes=s0 * 68)
    out = Q.attn_finalize(st)
    assert_device_clean()
    compare(out.cpu().numpy(), _oracle(q, k8, v8, M), "gqa causal split")
