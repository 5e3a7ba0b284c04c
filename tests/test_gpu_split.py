"""attn_chunk_step_split (the chunk's keys folded in parallel ranges, each into
its own partial state, then merged) against the oracle: Mode B burst
verification -- 64 candidate queries after the context, rectangular
full-context attention ("Out-of-Core Flash Streaming & Speculative Decode (1M
Context)", §4) -- and causal prefill with ragged ranges."""

import math

import numpy as np
import pytest
import torch

from tests.conftest import cuda_available
from tests.parity import assert_device_clean, compare, gpu_bytes, oracle_out, seeded

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _kv(B, M, H, seed, scale=1.0):
    k = seeded((B, M, H, 64), seed, "cuda", scale=scale)
    v = seeded((B, M, H, 64), seed + 1, "cuda", scale=scale)
    return k, v


@pytest.mark.parametrize("M,H,split", [(4096, 4, 512), (3000, 2, 384), (700, 3, 128)])
def test_burst_verification_rectangular(lib, M, H, split):
    """64 candidate queries at positions M .. M+63 see every context key."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    q = seeded((1, 64, H, 64), M + 1, "cuda", torch.float16)
    k, v = _kv(1, M, H, M + 2)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, 64, q.device)
    Q.attn_chunk_step_split(q, k8, v8, 0, M, st, split, q_pos0=M, causal=False)
    out = Q.attn_finalize(st)
    assert_device_clean()
    want, wk8, wv8 = oracle_out(q, k, v, causal=False, q_pos0=M)
    assert np.array_equal(gpu_bytes(k8, M), wk8) and np.array_equal(gpu_bytes(v8, M), wv8)
    compare(out.cpu().numpy(), want, f"burst M{M} split{split}")


@pytest.mark.parametrize("M,chunk,split", [(1000, 1000, 256), (1029, 512, 128), (2048, 2048, 1024)])
def test_causal_prefill_split(lib, M, chunk, split):
    """Causal prefill with every chunk split: later ranges are invisible to the
    early rows of a chunk, whose partials the merge must skip."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    H = 3
    q = seeded((1, M, H, 64), M + 11, "cuda", torch.float16)
    k, v = _kv(1, M, H, M + 12)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, M, q.device)
    for s0 in range(0, M, chunk):
        Q.attn_chunk_step_split(q, k8, v8, s0, min(chunk, M - s0), st, split, k_offset_bytes=s0 * 68)
    out = Q.attn_finalize(st)
    assert_device_clean()
    want, *_ = oracle_out(q, k, v)
    compare(out.cpu().numpy(), want, f"causal split M{M} chunk{chunk} split{split}")


def test_split_matches_unsplit(lib):
    """Split and unsplit forms of the same update.  Each keeps its own
    softmax reference m (the row max, or up to 8 ln 2 below it), so the two
    m agree within 8 ln 2 and l e^m (the sum of e^S over the keys) agrees to
    the rounding of the weights; the weights are rounded to fp16 against each
    key range's own reference before the merge, so the outputs agree within
    the parity tolerance rather than bit for bit."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    M, H = 2304, 2
    q = seeded((1, 64, H, 64), 41, "cuda", torch.float16)
    k, v = _kv(1, M, H, 42, scale=1.5)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    a = Q.State(1, H, 64, q.device)
    b = Q.State(1, H, 64, q.device)
    Q.attn_chunk_step(q, k8, v8, 0, M, a, q_pos0=M, causal=False)
    Q.attn_chunk_step_split(q, k8, v8, 0, M, b, 256, q_pos0=M, causal=False)
    assert_device_clean()
    lazy = 8 * math.log(2)
    assert torch.all(torch.abs(a.m - b.m) <= lazy + 1e-4)
    assert torch.allclose(a.l * torch.exp(a.m - b.m), b.l, rtol=1e-3, atol=0)
    oa, ob = Q.attn_finalize(a).float(), Q.attn_finalize(b).float()
    assert torch.max(torch.abs(oa - ob)).item() <= 2e-3
    want, *_ = oracle_out(q, k, v, causal=False, q_pos0=M)
    compare(ob.cpu().numpy(), want, "split")


def test_split_continues_a_state(lib):
    """An unsplit chunk, then a split one, into the same state."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    M, H = 1536, 2
    q = seeded((1, M, H, 64), 51, "cuda", torch.float16)
    k, v = _kv(1, M, H, 52)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, M, q.device)
    Q.attn_chunk_step(q, k8, v8, 0, 512, st)
    ws = torch.empty(Q.split_workspace_floats(1, H, M, 1024, 256), dtype=torch.float32, device="cuda")
    Q.attn_chunk_step_split(q, k8, v8, 512, 1024, st, 256, workspace=ws, k_offset_bytes=512 * 68)
    out = Q.attn_finalize(st)
    assert_device_clean()
    want, *_ = oracle_out(q, k, v)
    compare(out.cpu().numpy(), want, "unsplit then split")


def test_burst_verification_long_context(lib):
    """64 candidates against a 131,072-token, 32-head Q8_0 context, in 64
    key ranges of 2,048 keys."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    from oracle import runner as oracle_runner
    M, H = 131072, 32
    q = seeded((1, 64, H, 64), 61, "cuda", torch.float16)
    k, v = _kv(1, M, H, 62)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, 64, q.device)
    Q.attn_chunk_step_split(q, k8, v8, 0, M, st, 2048, q_pos0=M, causal=False)
    out = Q.attn_finalize(st).cpu().numpy()
    assert_device_clean()
    wk8 = oracle_runner.quantize_kv(k.cpu().numpy())
    assert np.array_equal(gpu_bytes(k8, M), wk8)
    del k
    wv8 = oracle_runner.quantize_kv(v.cpu().numpy())
    assert np.array_equal(gpu_bytes(v8, M), wv8)
    del v
    want = oracle_runner.attention(q.cpu().numpy(), wk8, wv8, 0.125, causal=False, q_pos0=M)
    compare(out, want, "burst 131072")


@pytest.mark.parametrize("n_q,M,chunk", [(100, 1900, 640), (1, 1000, 1000), (128, 2000, 1024)])
def test_paired_launch_continues_a_state(lib, n_q, M, chunk):
    """One query tile without the causal mask runs in paired mode (the two
    softmax pipelines take the even and odd key tiles and merge at the end).
    Here the chunks are folded one after another into the same state, so tile
    A starts from the state of the previous chunks; odd tile counts and a
    ragged last chunk (1900 = 640 + 640 + 620) included."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    H = 3
    q = seeded((1, n_q, H, 64), n_q + M, "cuda", torch.float16)
    k, v = _kv(1, M, H, n_q + M + 1)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, n_q, q.device)
    for s0 in range(0, M, chunk):
        Q.attn_chunk_step(q, k8, v8, s0, min(chunk, M - s0), st, q_pos0=M, causal=False,
                          k_offset_bytes=s0 * 68)
    out = Q.attn_finalize(st)
    assert_device_clean()
    want, *_ = oracle_out(q, k, v, causal=False, q_pos0=M)
    compare(out.cpu().numpy(), want, f"paired n_q{n_q} M{M} chunk{chunk}")


def test_burst_verification_bench_shape(lib):
    """The burst benchmark's own case: the 64 seeded candidates of the burst
    workload against its 1,048,576-token, 32-head context, folded in the key
    ranges the benchmark picks (whole waves on this device: 19 ranges of 55,296
    keys on 152 SMs) with a caller workspace, exactly as the benchmark launches
    it.
    The oracle checks the Q8_0 bytes and the output of three of the heads."""
    from chunked_prefill_attention_gb300 import q8attn as Q, workloads as W
    from oracle import runner as oracle_runner
    b = W.BURSTS["burst_m1m"]
    M, H = b.context, b.heads
    q, k, v = W.make_burst_inputs(b, device="cuda")
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, b.queries, q.device)
    split = b.split_keys or Q.split_keys_for(H, M, torch.cuda.get_device_properties(0).multi_processor_count)
    ws = torch.empty(Q.split_workspace_floats(1, H, b.queries, M, split), dtype=torch.float32,
                     device="cuda")
    Q.attn_chunk_step_split(q, k8, v8, 0, M, st, split, workspace=ws, q_pos0=M, causal=False)
    out = Q.attn_finalize(st).cpu().numpy()
    assert_device_clean()
    heads = [0, 17, 31]
    qn = q.cpu().numpy()
    for h in heads:
        wk8 = oracle_runner.quantize_kv(k[:, :, h:h + 1].contiguous().cpu().numpy())
        assert np.array_equal(k8[:, h:h + 1, :M * 68].reshape(1, 1, M, 68).cpu().numpy(), wk8)
        wv8 = oracle_runner.quantize_kv(v[:, :, h:h + 1].contiguous().cpu().numpy())
        assert np.array_equal(v8[:, h:h + 1, :M * 68].reshape(1, 1, M, 68).cpu().numpy(), wv8)
        want = oracle_runner.attention(qn[:, :, h:h + 1], wk8, wv8, 0.125, causal=False, q_pos0=M)
        res = compare(out[:, :, h:h + 1], want, f"burst_m1m head {h}")
        print(f"\n[burst_m1m head {h}] max|err| {res[0]:.3e} (|out| {res[2]:.2f}), rel-L2 {res[1]:.3e}")


def test_grouped_query_burst_bench_shape(lib):
    """The grouped-query burst benchmark's case: 64 candidates of 32 query
    heads on 8 K/V heads against a 1,048,576-token context, launched as the
    benchmark does (packed tiles of (candidate, head) pairs, wave-sized key
    ranges); the oracle checks the Q8_0 bytes of two K/V heads and the output
    of three query heads."""
    from chunked_prefill_attention_gb300 import q8attn as Q, workloads as W
    from oracle import runner as oracle_runner
    b = W.BURSTS["burst_m1m_gqa8"]
    M, H, H_kv = b.context, b.heads, b.kv_h
    g = H // H_kv
    q, k, v = W.make_burst_inputs(b, device="cuda")
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, b.queries, q.device)
    ctas = H_kv * -(-b.queries * g // 256)
    split = Q.split_keys_for(ctas, M, torch.cuda.get_device_properties(0).multi_processor_count)
    Q.attn_chunk_step_split_gqa(q, k8, v8, 0, M, st, split, q_pos0=M, causal=False)
    out = Q.attn_finalize(st).cpu().numpy()
    assert_device_clean()
    qn = q.cpu().numpy()
    for h in [0, 13, 31]:
        kvh = h // g
        wk8 = oracle_runner.quantize_kv(k[:, :, kvh:kvh + 1].contiguous().cpu().numpy())
        wv8 = oracle_runner.quantize_kv(v[:, :, kvh:kvh + 1].contiguous().cpu().numpy())
        if h in (0, 31):
            assert np.array_equal(k8[:, kvh:kvh + 1, :M * 68].reshape(1, 1, M, 68).cpu().numpy(), wk8)
            assert np.array_equal(v8[:, kvh:kvh + 1, :M * 68].reshape(1, 1, M, 68).cpu().numpy(), wv8)
        want = oracle_runner.attention(qn[:, :, h:h + 1], wk8, wv8, 0.125, causal=False, q_pos0=M)
        res = compare(out[:, :, h:h + 1], want, f"burst_m1m_gqa8 head {h}")
        print(f"\n[burst_m1m_gqa8 head {h}] max|err| {res[0]:.3e} (|out| {res[2]:.2f}), rel-L2 {res[1]:.3e}")
