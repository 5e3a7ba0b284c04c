"""attn_prefill_pipelined: the whole prefill from host buffers with the K/V
chunk copies overlapped with the device work.  Its output must be bit-identical
to the device-resident path (same kernels, same chunk order) and within the
parity tolerance of the oracle."""

import pytest
import torch

from tests.conftest import cuda_available
from tests.parity import assert_device_clean, compare, oracle_out, seeded

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("B,M,H,chunk", [(1, 1000, 2, 256), (2, 768, 3, 128), (1, 2048, 4, 2048),
                                         (2, 2600, 3, 256), (1, 17000, 2, 8192), (2, 5000, 3, 2048),
                                         (1, 1500, 2, 2048)])
def test_pipelined_matches_device_path(lib, B, M, H, chunk):
    """The K/V slots hold two chunks: with M > 2 * chunk each slot is refilled
    several times (one case streams 11 chunks through them).  Q follows chunk
    0's K and V in row blocks, and chunk 0's step runs per block (blocks of
    256 rows for the small chunks, 8,192 for the 17,000-token case, with a
    ragged last block).  When chunk 0 is a multiple of 1,024 tokens (or the
    whole sequence) its K, V and query rows cross in leads of 1,024 tokens,
    each folded as it arrives (two batch entries with later row blocks; a
    single 1,500-token chunk whose last lead holds a partial query tile)."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    q = seeded((B, M, H, 64), M + 71, "cuda", torch.float16)
    k = seeded((B, M, H, 64), M + 72, "cuda")
    v = seeded((B, M, H, 64), M + 73, "cuda")
    ref, *_ = Q.prefill_attention(q, k, v, chunk)
    qh, kh, vh = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    oh = torch.empty((B, M, H, 64), dtype=torch.float16).pin_memory()
    bufs = Q.PipelineBuffers(B, M, H, q.device, chunk)
    assert bufs.kv_slots.numel() == 4 * B * min(chunk, M) * H * 64   # two chunks of K and V
    for _ in range(2):   # twice on the same buffers: the calls must be ordered
        oh.zero_()
        Q.attn_prefill_pipelined(qh, kh, vh, oh, bufs)
        torch.cuda.current_stream().synchronize()
        assert_device_clean()
        assert torch.equal(oh, ref.cpu())
    want, *_ = oracle_out(q, k, v)
    compare(oh.numpy(), want, f"pipelined B{B} M{M}")


@pytest.mark.parametrize("B,M,H,chunk", [(1, 900, 2, 256), (2, 520, 3, 512)])
def test_pipelined_without_causal_mask(lib, B, M, H, chunk):
    """Without the causal mask every chunk updates every row, so the output is
    finalised and copied back once at the end."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    q = seeded((B, M, H, 64), M + 81, "cuda", torch.float16)
    k = seeded((B, M, H, 64), M + 82, "cuda")
    v = seeded((B, M, H, 64), M + 83, "cuda")
    ref, *_ = Q.prefill_attention(q, k, v, chunk, causal=False)
    qh, kh, vh = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    oh = torch.zeros((B, M, H, 64), dtype=torch.float16).pin_memory()
    bufs = Q.PipelineBuffers(B, M, H, q.device, chunk)
    Q.attn_prefill_pipelined(qh, kh, vh, oh, bufs, causal=False)
    torch.cuda.current_stream().synchronize()
    assert_device_clean()
    assert torch.equal(oh, ref.cpu())
    want, *_ = oracle_out(q, k, v, causal=False)
    compare(oh.numpy(), want, f"pipelined non-causal B{B} M{M}")


@pytest.mark.parametrize("B,M,H,chunk,causal", [(1, 1000, 2, 256, True), (2, 1800, 3, 512, True),
                                                (1, 9000, 2, 4096, True), (1, 700, 2, 256, False)])
def test_pipelined_head_dim_128(lib, B, M, H, chunk, causal):
    """head_dim 128 (136-byte Q8_0 rows): slots of twice the floats, chunk 0's
    query blocks folded by the two-query-tile kernel (and a one-tile last
    block by the paired kernel), bit-identical to the device path."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    D = 128
    q = seeded((B, M, H, D), M + 91, "cuda", torch.float16)
    k = seeded((B, M, H, D), M + 92, "cuda")
    v = seeded((B, M, H, D), M + 93, "cuda")
    ref, *_ = Q.prefill_attention(q, k, v, chunk, causal=causal)
    qh, kh, vh = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    oh = torch.zeros((B, M, H, D), dtype=torch.float16).pin_memory()
    bufs = Q.PipelineBuffers(B, M, H, q.device, chunk, head_dim=D)
    assert bufs.kv_slots.numel() == 4 * B * min(chunk, M) * H * D
    Q.attn_prefill_pipelined(qh, kh, vh, oh, bufs, causal=causal)
    torch.cuda.current_stream().synchronize()
    assert_device_clean()
    assert torch.equal(oh, ref.cpu())
    want, *_ = oracle_out(q, k, v, causal=causal)
    compare(oh.numpy(), want, f"pipelined d128 B{B} M{M} causal {causal}")
