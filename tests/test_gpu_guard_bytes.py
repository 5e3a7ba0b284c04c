"""Guard bytes around every buffer a call writes: each output tensor is a view
into a larger allocation whose head, tail (and, for the Q8_0 planes, the
padding between planes) hold a sentinel pattern; after the calls the sentinels
must be intact.  A kernel that writes outside its tensors -- a wrong stride, a
ragged tile, an off-by-one row -- changes them.  Shapes are ragged on purpose
(partial query and key tiles, padded plane strides, both head sizes)."""

import pytest
import torch

from tests.conftest import cuda_available
from tests.parity import assert_device_clean, seeded

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

GUARD = 4096   # bytes on each side; a multiple of 256 keeps every view aligned
SENTINEL = 0xA5


class Guarded:
    """A byte buffer of `n` usable bytes between two guard regions."""

    def __init__(self, n):
        self.n = n
        self.raw = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        return self.raw[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        return bool(torch.all(head == SENTINEL)) and bool(torch.all(tail == SENTINEL))


def _state(B, H, n_q, D):
    from chunked_prefill_attention_gb300 import q8attn as Q
    gm, gl, go = Guarded(B * H * n_q * 4), Guarded(B * H * n_q * 4), Guarded(B * H * n_q * D * 4)
    st = Q.State.__new__(Q.State)
    st.m = gm.view(torch.float32, (B, H, n_q))
    st.l = gl.view(torch.float32, (B, H, n_q))
    st.o = go.view(torch.float32, (B, H, n_q, D))
    return st, [gm, gl, go]


def _planes(B, H, M, D, pad):
    """Q8_0 planes with `pad` extra bytes per plane (a padded stride)."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    stride = Q.plane_stride(M, D) + pad
    g = Guarded(B * H * stride)
    return g, g.view(torch.uint8, (B, H, stride)), stride


def _padding_intact(planes, M, D):
    from chunked_prefill_attention_gb300 import q8attn as Q
    return bool(torch.all(planes[:, :, M * Q.row_bytes(D):] == SENTINEL))


@pytest.mark.parametrize("D,B,M,H,chunk,causal", [(64, 2, 333, 3, 100, True), (64, 1, 700, 2, 256, False),
                                                  (128, 2, 301, 3, 110, True), (128, 1, 520, 2, 256, False)])
def test_chunk_steps_write_only_their_tensors(lib, D, B, M, H, chunk, causal):
    from chunked_prefill_attention_gb300 import q8attn as Q
    q = seeded((B, M, H, D), M + D, "cuda", torch.float16)
    k = seeded((B, M, H, D), M + D + 1, "cuda")
    v = seeded((B, M, H, D), M + D + 2, "cuda")
    gk, k8, stride = _planes(B, H, M, D, pad=48)
    gv, v8, _ = _planes(B, H, M, D, pad=48)
    Q.q8kv_quantize(k, k8, stride)
    Q.q8kv_quantize(v, v8, stride)
    st, gst = _state(B, H, M, D)
    Q.attn_state_init(st)
    for s0 in range(0, M, chunk):
        Q.attn_chunk_step(q, k8, v8, s0, min(chunk, M - s0), st, causal=causal, stride=stride,
                          k_offset_bytes=s0 * Q.row_bytes(D))
    gout = Guarded(B * M * H * D * 2)
    out = gout.view(torch.float16, (B, M, H, D))
    Q.attn_finalize(st, out)
    torch.cuda.synchronize()
    assert_device_clean()
    assert gk.intact() and gv.intact() and all(g.intact() for g in gst) and gout.intact()
    assert _padding_intact(k8, M, D) and _padding_intact(v8, M, D)
    assert torch.all(torch.isfinite(out.float()))


@pytest.mark.parametrize("D", [64, 128])
def test_split_writes_only_its_tensors(lib, D):
    from chunked_prefill_attention_gb300 import q8attn as Q
    M, H, n_q, split = 1500, 3, 70, 256
    q = seeded((1, n_q, H, D), 5 + D, "cuda", torch.float16)
    k = seeded((1, M, H, D), 6 + D, "cuda")
    v = seeded((1, M, H, D), 7 + D, "cuda")
    k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
    st, gst = _state(1, H, n_q, D)
    Q.attn_state_init(st)
    n_ws = Q.split_workspace_floats(1, H, n_q, M, split, D)
    gws = Guarded(n_ws * 4)
    ws = gws.view(torch.float32, (n_ws,))
    Q.attn_chunk_step_split(q, k8, v8, 0, M, st, split, workspace=ws, q_pos0=M, causal=False)
    torch.cuda.synchronize()
    assert_device_clean()
    assert gws.intact() and all(g.intact() for g in gst)


@pytest.mark.parametrize("D", [64, 128])
def test_pipelined_and_graph_write_only_their_tensors(lib, D):
    from chunked_prefill_attention_gb300 import q8attn as Q
    B, M, H, chunk = 1, 900, 2, 256
    q = seeded((B, M, H, D), 9 + D, "cuda", torch.float16)
    k = seeded((B, M, H, D), 10 + D, "cuda")
    v = seeded((B, M, H, D), 11 + D, "cuda")
    # pipelined: guard the slots, the planes, the state and both outputs
    bufs = Q.PipelineBuffers(B, M, H, q.device, chunk, head_dim=D)
    n_slot = bufs.kv_slots.numel()
    gslot = Guarded(n_slot * 4)
    bufs.kv_slots = gslot.view(torch.float32, (n_slot,))
    gk, bufs.k8, _ = _planes(B, H, M, D, pad=0)
    gv, bufs.v8, _ = _planes(B, H, M, D, pad=0)
    bufs.state, gst = _state(B, H, M, D)
    gq, gout = Guarded(B * M * H * D * 2), Guarded(B * M * H * D * 2)
    bufs.q = gq.view(torch.float16, (B, M, H, D))
    bufs.out = gout.view(torch.float16, (B, M, H, D))
    oh = torch.zeros((B, M, H, D), dtype=torch.float16).pin_memory()
    Q.attn_prefill_pipelined(q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory(), oh, bufs)
    torch.cuda.current_stream().synchronize()
    assert_device_clean()
    assert all(g.intact() for g in [gslot, gk, gv, gq, gout] + gst)
    # the captured graph on the same inputs gives the pipelined output bit for bit
    g = Q.PrefillGraph(q, k, v, chunk)
    ref = g.launch().clone()
    torch.cuda.synchronize()
    assert torch.equal(ref.cpu(), oh)
    g.close()
