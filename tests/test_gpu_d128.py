"""head_dim 128 (four Q8_0 blocks, 136 bytes per head row): quantised bytes
bit-exact against the oracle, attention within max|err| <= 2e-3 and rel-L2 <=
1e-3 of the oracle on identical dequantised KV -- causal prefill in chunks
(including an 8,192-token case), ragged sizes that take the plain-copy tail,
rectangular attention after a context, grouped-query attention, chunk order.
The oracle quantises a head row of any multiple of 32 channels in channel
order and computes the plain definition in fp64."""

import numpy as np
import pytest
import torch

from tests.conftest import cuda_available
from oracle import runner as oracle_runner
from tests.parity import assert_device_clean, compare, gpu_bytes, oracle_out, run_gpu, seeded

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]
D = 128


def _inputs(B, M, H, seed, H_kv=None, n_q=None):
    H_kv = H if H_kv is None else H_kv
    n_q = M if n_q is None else n_q
    q = seeded((B, n_q, H, D), seed, "cuda", torch.float16)
    k = seeded((B, M, H_kv, D), seed + 1, "cuda")
    v = seeded((B, M, H_kv, D), seed + 2, "cuda")
    return q, k, v


@pytest.mark.parametrize("B,M,H", [(1, 1, 1), (1, 7, 3), (2, 9, 8), (1, 100, 9), (2, 1000, 16)])
def test_d128_quantize_bytes(lib, B, M, H):
    from chunked_prefill_attention_gb300 import q8attn as Q
    x = seeded((B, M, H, D), 300 + M, "cuda")
    x[..., 5] *= 40.0                          # an outlier channel in block 0
    x[0, 0, 0, 64:96] = 0.0                    # an all-zero block
    out = Q.q8kv_quantize(x)
    assert out.shape[-1] == Q.plane_stride(M, D)
    want = oracle_runner.quantize_kv(x.cpu().numpy())
    assert want.shape[-1] == 136
    assert np.array_equal(gpu_bytes(out, M, D), want)


def test_d128_quantize_input_only_16_byte_aligned(lib):
    from chunked_prefill_attention_gb300 import q8attn as Q
    B, M, H = 1, 37, 5
    base = seeded((B * M * H * D + 4,), 313, "cuda")
    x = base[4:].view(B, M, H, D)
    want = oracle_runner.quantize_kv(x.cpu().numpy())
    assert np.array_equal(gpu_bytes(Q.q8kv_quantize(x), M, D), want)


@pytest.mark.parametrize("B,M,H,chunk", [
    (1, 1, 1, 1), (1, 2, 2, 2), (1, 63, 2, 64), (1, 64, 2, 64), (1, 65, 2, 64), (1, 129, 2, 128),
    (2, 200, 3, 64), (1, 300, 2, 100), (1, 333, 2, 110), (1, 1000, 2, 500), (2, 1030, 4, 256),
])
def test_d128_causal_parity_small(lib, B, M, H, chunk):
    """Chunk starts are even (a 136-byte row offset is 16-byte aligned only
    then); a ragged last tile of odd length has a byte count that is not a
    multiple of 16 (copied with plain loads).  Launches over one query tile run
    the paired kernel (both pipelines on its rows, merged at the end); launches
    over two or more run the two-query-tile kernel, including odd tile counts
    (300, 333 and 1030 tokens) and chunks whose first visible tile is not 0."""
    q, k, v = _inputs(B, M, H, seed=M * 5 + B)
    out, k8, v8, _ = run_gpu(q, k, v, chunk)
    want, wk8, wv8 = oracle_out(q, k, v)
    assert np.array_equal(gpu_bytes(k8, M, D), wk8) and np.array_equal(gpu_bytes(v8, M, D), wv8)
    compare(out.cpu().numpy(), want, f"d128 B{B} M{M} H{H} chunk {chunk}")


def test_d128_causal_8192_tokens(lib):
    """A causal 8,192-token prefill over 8 heads in four chunks of 2,048."""
    q, k, v = _inputs(1, 8192, 8, seed=8192)
    out, *_ = run_gpu(q, k, v, 2048)
    want, *_ = oracle_out(q, k, v)
    res = compare(out.cpu().numpy(), want, "d128 causal 8192")
    print(f"\n[d128 causal 8192] max|err| {res[0]:.3e} (|out| {res[2]:.2f}), rel-L2 {res[1]:.3e}")


@pytest.mark.parametrize("n_q,M,q_pos0", [(64, 4096, 4096), (128, 1000, 1000), (200, 777, 0)])
def test_d128_rectangular(lib, n_q, M, q_pos0):
    """No causal mask: candidate rows after a context (as in burst
    verification), and a plain rectangular case."""
    q, k, v = _inputs(1, M, 4, seed=n_q + M, n_q=n_q)
    out, *_ = run_gpu(q, k, v, 512, causal=False, q_pos0=q_pos0)
    want, *_ = oracle_out(q, k, v, causal=False, q_pos0=q_pos0)
    compare(out.cpu().numpy(), want, f"d128 rectangular n_q {n_q} M {M}")


@pytest.mark.parametrize("H,H_kv", [(8, 2), (4, 1)])
def test_d128_grouped_query(lib, H, H_kv):
    from chunked_prefill_attention_gb300 import q8attn as Q
    B, M = 2, 2048
    q, k, v = _inputs(B, M, H, seed=41 + H_kv, H_kv=H_kv)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(B, H, M, q.device, head_dim=D)
    for s0 in range(0, M, 512):
        Q.attn_chunk_step_gqa(q, k8, v8, s0, 512, st, k_offset_bytes=s0 * Q.row_bytes(D))
    out = Q.attn_finalize(st)
    assert_device_clean()
    wk8 = oracle_runner.quantize_kv(k.cpu().numpy())
    wv8 = oracle_runner.quantize_kv(v.cpu().numpy())
    want = oracle_runner.attention(q.cpu().numpy(), wk8, wv8, 1.0 / np.sqrt(D))
    compare(out.cpu().numpy(), want, f"d128 GQA H{H} H_kv{H_kv}")


def test_d128_chunk_order(lib):
    q, k, v = _inputs(1, 768, 2, seed=91)
    want, *_ = oracle_out(q, k, v)
    for order in ([0, 1, 2], [2, 0, 1]):
        out, *_ = run_gpu(q, k, v, 256, order=order)
        compare(out.cpu().numpy(), want, f"d128 order {order}")


@pytest.mark.parametrize("M,H,split", [(4096, 4, 512), (3000, 2, 384), (20000, 8, 2048)])
def test_d128_burst_split(lib, M, H, split):
    """Burst verification at head_dim 128: 64 candidates after the context,
    no mask, the keys folded in parallel ranges (the paired kernel per range)
    and merged."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    q, k, v = _inputs(1, M, H, seed=M + split, n_q=64)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, 64, q.device, head_dim=D)
    Q.attn_chunk_step_split(q, k8, v8, 0, M, st, split, q_pos0=M, causal=False)
    out = Q.attn_finalize(st)
    assert_device_clean()
    want, *_ = oracle_out(q, k, v, causal=False, q_pos0=M)
    compare(out.cpu().numpy(), want, f"d128 burst M{M} split{split}")


@pytest.mark.parametrize("M,chunk,split", [(1000, 1000, 256), (1030, 512, 128)])
def test_d128_causal_split(lib, M, chunk, split):
    """Causal prefill with every chunk split at head_dim 128: later ranges are
    invisible to the early rows of a chunk, whose partials the merge skips."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    H = 3
    q, k, v = _inputs(1, M, H, seed=M + 7)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st = Q.State(1, H, M, q.device, head_dim=D)
    for s0 in range(0, M, chunk):
        Q.attn_chunk_step_split(q, k8, v8, s0, min(chunk, M - s0), st, split,
                                k_offset_bytes=s0 * Q.row_bytes(D))
    out = Q.attn_finalize(st)
    assert_device_clean()
    want, *_ = oracle_out(q, k, v)
    compare(out.cpu().numpy(), want, f"d128 causal split M{M} chunk{chunk} split{split}")


def test_d128_static_split_matches_workspace_split(lib):
    """The allocation-free split at head_dim 128 runs the same kernels on the
    same inputs as the split with a caller workspace: identical state."""
    import ctypes
    from chunked_prefill_attention_gb300 import q8attn as Q
    M, H = 5000, 4
    q, k, v = _inputs(1, M, H, seed=77, n_q=64)
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    a = Q.State(1, H, 64, q.device, head_dim=D)
    b = Q.State(1, H, 64, q.device, head_dim=D)
    Q.attn_chunk_step_split(q, k8, v8, 0, M, a, 1024, q_pos0=M, causal=False)
    rc = lib.attn_chunk_step_split_static(
        ctypes.c_void_p(q.data_ptr()), M, ctypes.c_void_p(k8.data_ptr()), ctypes.c_void_p(v8.data_ptr()),
        k8.shape[-1], 0, M, ctypes.c_void_p(b.m.data_ptr()), ctypes.c_void_p(b.l.data_ptr()),
        ctypes.c_void_p(b.o.data_ptr()), 1, H, 64, D, 1.0 / np.sqrt(D), 0, 1024,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == Q.Q8A_OK
    torch.cuda.synchronize()
    assert_device_clean()
    assert torch.equal(a.m, b.m) and torch.equal(a.l, b.l) and torch.equal(a.o, b.o)
