"""attn_state_init / attn_chunk_step / attn_finalize on the GPU vs the oracle:
small and ragged shapes, masks, chunk orders and the state round trip."""

import numpy as np
import pytest
import torch

from tests.conftest import cuda_available
from tests.parity import assert_device_clean, compare, gpu_bytes, oracle_out, run_gpu, seeded

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _inputs(B, M, H, seed, kv_scale=1.0, n_q=None):
    n_q = M if n_q is None else n_q
    q = seeded((B, n_q, H, 64), seed, "cuda", torch.float16)
    k = seeded((B, M, H, 64), seed + 1, "cuda", scale=kv_scale)
    v = seeded((B, M, H, 64), seed + 2, "cuda", scale=kv_scale)
    return q, k, v


@pytest.mark.parametrize("B,M,H,chunk", [
    (1, 1, 1, 1), (1, 2, 2, 2), (1, 7, 3, 4), (1, 64, 2, 64), (1, 128, 2, 128),
    (1, 129, 2, 128), (1, 130, 2, 128), (2, 200, 3, 64), (1, 257, 4, 256), (1, 300, 2, 100),
    (1, 383, 2, 384), (1, 512, 4, 512), (2, 640, 2, 256), (1, 1000, 2, 500), (1, 1029, 1, 1029),
])
def test_causal_parity_small(lib, B, M, H, chunk):
    q, k, v = _inputs(B, M, H, seed=M * 7 + B)
    out, k8, v8, _ = run_gpu(q, k, v, chunk)
    want, wk8, wv8 = oracle_out(q, k, v)
    assert np.array_equal(gpu_bytes(k8, M), wk8) and np.array_equal(gpu_bytes(v8, M), wv8)
    compare(out.cpu().numpy(), want, f"B{B} M{M} H{H} chunk{chunk}")


def test_outlier_channels(lib):
    """Two K channels x20 per head: the Q.K path must use exact dequantised K."""
    q, k, v = _inputs(1, 700, 4, seed=11)
    k[..., 3] *= 20
    k[..., 35] *= 20
    out, *_ = run_gpu(q, k, v, 256)
    want, *_ = oracle_out(q, k, v)
    compare(out.cpu().numpy(), want, "outliers")


def test_noncausal_rectangular(lib):
    q, k, v = _inputs(1, 333, 3, seed=21, n_q=70)
    out, *_ = run_gpu(q, k, v, 128, causal=False)
    want, *_ = oracle_out(q, k, v, causal=False)
    compare(out.cpu().numpy(), want, "non-causal")


def test_queries_after_context(lib):
    """64 query rows placed after 448 keys (q_pos0 = 448): every key visible
    to every query under the causal rule."""
    q, k, v = _inputs(1, 448, 2, seed=31, n_q=64)
    out, *_ = run_gpu(q, k, v, 128, q_pos0=448)
    want, *_ = oracle_out(q, k, v, q_pos0=448)
    compare(out.cpu().numpy(), want, "q_pos0=448")


def test_queries_inside_context(lib):
    """Queries are the last 200 rows of a 520-token sequence (q_pos0 = 320)."""
    q, k, v = _inputs(1, 520, 2, seed=41, n_q=200)
    out, *_ = run_gpu(q, k, v, 128, q_pos0=320)
    want, *_ = oracle_out(q, k, v, q_pos0=320)
    compare(out.cpu().numpy(), want, "q_pos0=320")


def test_other_scale(lib):
    q, k, v = _inputs(1, 300, 2, seed=51)
    out, *_ = run_gpu(q, k, v, 128, scale=0.3)
    want, *_ = oracle_out(q, k, v, scale=0.3)
    compare(out.cpu().numpy(), want, "scale 0.3")


def test_chunk_order_any(lib):
    q, k, v = _inputs(1, 768, 2, seed=61, kv_scale=2.0)
    ref, *_ = run_gpu(q, k, v, 128)
    for order in ([5, 4, 3, 2, 1, 0], [2, 0, 5, 1, 3, 4]):
        out, *_ = run_gpu(q, k, v, 128, order=order)
        want, *_ = oracle_out(q, k, v)
        compare(out.cpu().numpy(), want, f"order {order}")
        assert torch.max(torch.abs(out.float() - ref.float())).item() < 2e-3


def test_chunked_matches_single_chunk(lib):
    """With chunk boundaries on 128-key tile boundaries every row sees the same
    fp32 scores in the same key tiles, so m and l are bit-identical whether the
    keys come in one chunk or several.  O differs only in where its high and
    residual accumulator halves are added (at each chunk boundary), i.e. by
    fp32 rounding."""
    q, k, v = _inputs(2, 1024, 3, seed=71)
    a, *_, sa = run_gpu(q, k, v, 1024)
    for chunk in (256, 128):
        b, *_, sb = run_gpu(q, k, v, chunk)
        assert torch.equal(sa.m, sb.m) and torch.equal(sa.l, sb.l)
        diff = (sa.o - sb.o).abs() / sa.l[..., None]
        assert diff.max().item() <= 1e-5
        assert torch.max(torch.abs(a.float() - b.float())).item() <= 2e-3


def test_state_checkpoint_resume_bitwise(lib):
    from chunked_prefill_attention_gb300 import q8attn as Q
    q, k, v = _inputs(1, 1024, 2, seed=81)
    full, k8, v8, _ = run_gpu(q, k, v, 256)
    st = Q.State(1, 2, 1024, "cuda")
    for s0 in (0, 256):
        Q.attn_chunk_step(q, k8, v8, s0, 256, st, k_offset_bytes=s0 * 68)
    saved = [t.cpu() for t in (st.m, st.l, st.o)]
    del st
    st2 = Q.State(1, 2, 1024, "cuda", init=False)
    st2.m.copy_(saved[0]); st2.l.copy_(saved[1]); st2.o.copy_(saved[2])
    for s0 in (512, 768):
        Q.attn_chunk_step(q, k8, v8, s0, 256, st2, k_offset_bytes=s0 * 68)
    assert torch.equal(Q.attn_finalize(st2), full)
    assert_device_clean()


def test_separate_chunk_buffers_with_ragged_tail(lib):
    """Chunks in their own buffers (not slices): sizes not multiples of 4 use
    the plain-copy tail path."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    q, k, v = _inputs(1, 301, 2, seed=91)
    st = Q.State(1, 2, 301, "cuda")
    for s0, n in ((0, 101), (101, 150), (251, 50)):
        k8 = Q.q8kv_quantize(k[:, s0:s0 + n].contiguous())
        v8 = Q.q8kv_quantize(v[:, s0:s0 + n].contiguous())
        Q.attn_chunk_step(q, k8, v8, s0, n, st)
    out = Q.attn_finalize(st)
    assert_device_clean()
    want, *_ = oracle_out(q, k, v)
    compare(out.cpu().numpy(), want, "separate buffers")


def test_state_init_and_finalize_values(lib):
    from chunked_prefill_attention_gb300 import q8attn as Q
    st = Q.State(2, 3, 37, "cuda")
    assert torch.all(torch.isneginf(st.m)) and torch.all(st.l == 0) and torch.all(st.o == 0)
    out = Q.attn_finalize(st)
    assert out.shape == (2, 37, 3, 64) and torch.all(out == 0)
    st.l.fill_(4.0)
    st.o.copy_(torch.arange(64, device="cuda", dtype=torch.float32).expand_as(st.o))
    out = Q.attn_finalize(st)
    assert torch.equal(out[1, 5, 2].float(), (torch.arange(64, device="cuda") / 4.0).half().float())


@pytest.mark.parametrize("D", [64, 128])
def test_finalize_is_the_rounded_quotient(lib, D):
    """attn_finalize gives fp16(RN_fp32(O / l)): the fp32 quotient it forms
    without a divide per value equals the IEEE quotient (torch's division),
    bit for bit, over a wide spread of O and l; rows with l == 0 give 0."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    g = torch.Generator(device="cuda")
    g.manual_seed(D)
    st = Q.State(2, 5, 300, "cuda", head_dim=D)
    st.l.copy_(torch.exp(torch.rand(st.l.shape, generator=g, device="cuda") * 20.0 - 2.0))
    st.l[0, 1, :7] = 0.0
    st.o.copy_(torch.randn(st.o.shape, generator=g, device="cuda") * st.l[..., None] *
               torch.rand(st.o.shape, generator=g, device="cuda") * 8.0)
    out = Q.attn_finalize(st)
    want = torch.where(st.l[..., None] > 0, st.o / st.l[..., None], torch.zeros_like(st.o))
    want = want.permute(0, 2, 1, 3).half()
    assert torch.equal(out, want)
    assert torch.all(out[0, :7, 1] == 0)


def test_rows_before_chunk_keep_state(lib):
    """A causal chunk starting at key 256 leaves the state of rows 0..255 untouched."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    q, k, v = _inputs(1, 512, 2, seed=101)
    k8 = Q.q8kv_quantize(k)
    v8 = Q.q8kv_quantize(v)
    st = Q.State(1, 2, 512, "cuda")
    Q.attn_chunk_step(q, k8, v8, 0, 256, st)
    before = [t.clone() for t in (st.m, st.l, st.o)]
    Q.attn_chunk_step(q, k8, v8, 256, 256, st, k_offset_bytes=256 * 68)
    assert torch.equal(st.m[:, :, :256], before[0][:, :, :256])
    assert torch.equal(st.l[:, :, :256], before[1][:, :, :256])
    assert torch.equal(st.o[:, :, :256], before[2][:, :, :256])
    assert_device_clean()
