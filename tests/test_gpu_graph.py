"""q8a_prefill_graph: a whole device-resident prefill (quantise K and V, state
init, the chunk steps in order, finalise -- "Out-of-Core Flash Streaming &
Speculative Decode (1M Context)", §3) captured once into a CUDA graph and
replayed.  A replay runs the same kernels with the same arguments as the calls
made one by one, so its outputs, Q8_0 bytes and state are bit-identical to
theirs; the output is also checked against the oracle."""

import numpy as np
import pytest
import torch

from tests.conftest import cuda_available
from tests.parity import assert_device_clean, compare, gpu_bytes, oracle_out

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _eager(q, k, v, chunk, causal=True):
    from chunked_prefill_attention_gb300 import q8attn as Q
    B, M, H, D = q.shape
    st = Q.State(B, H, M, q.device, init=False, head_dim=D)
    out, k8, v8 = Q.prefill_attention(q, k, v, chunk, causal=causal, state=st)
    return out, k8, v8, st


def _same(g, eager, M, D):
    out, k8, v8, st = eager
    rb = M * (D // 32 * 34)
    assert torch.equal(g.out, out)
    assert torch.equal(g.k8[..., :rb], k8[..., :rb]) and torch.equal(g.v8[..., :rb], v8[..., :rb])
    assert torch.equal(g.state.m, st.m) and torch.equal(g.state.l, st.l) and torch.equal(g.state.o, st.o)


@pytest.mark.parametrize("name,batch,tokens", [("m512", 1, 512), ("m2k_out", 1, 2048), ("b8_m2k", 2, 1024),
                                               ("m16k_d128", 1, 1024)])
def test_graph_replay_matches_calls_and_oracle(lib, name, batch, tokens):
    from chunked_prefill_attention_gb300 import q8attn as Q, workloads as W
    w = W.WORKLOADS[name]
    q, k, v = W.make_inputs(w, device="cuda", batch=batch, tokens=tokens)
    D = q.shape[-1]
    chunk = min(w.chunk, 256)
    g = Q.PrefillGraph(q, k, v, chunk)
    g.launch()
    torch.cuda.synchronize()
    assert_device_clean()
    _same(g, _eager(q, k, v, chunk), tokens, D)
    want, wk8, wv8 = oracle_out(q, k, v)
    assert np.array_equal(gpu_bytes(g.k8, tokens, D), wk8) and np.array_equal(gpu_bytes(g.v8, tokens, D), wv8)
    compare(g.out.cpu().numpy(), want, f"graph {name} B{batch} M{tokens}")
    g.close()


def test_graph_replays_new_inputs_in_place(lib):
    """The graph reads its buffers at replay time: new Q, K and V written into
    them give the new prefill; replays of the same inputs give the same bits."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    from tests.parity import seeded
    B, M, H = 1, 1000, 3
    q = seeded((B, M, H, 64), 71, "cuda", torch.float16)
    k = seeded((B, M, H, 64), 72, "cuda")
    v = seeded((B, M, H, 64), 73, "cuda")
    g = Q.PrefillGraph(q, k, v, 384)
    first = g.launch().clone()
    again = g.launch().clone()
    torch.cuda.synchronize()
    assert torch.equal(first, again)
    q.copy_(seeded((B, M, H, 64), 74, "cuda", torch.float16))
    k.copy_(seeded((B, M, H, 64), 75, "cuda", scale=2.0))
    v.copy_(seeded((B, M, H, 64), 76, "cuda"))
    g.launch()
    torch.cuda.synchronize()
    assert_device_clean()
    _same(g, _eager(q, k, v, 384), M, 64)
    assert not torch.equal(g.out, first)
    want, *_ = oracle_out(q, k, v)
    compare(g.out.cpu().numpy(), want, "graph replay, new inputs")
    g.close()


def test_graph_without_mask_and_on_another_stream(lib):
    """Rectangular attention (causal = 0) and a replay on a side stream."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    from tests.parity import seeded
    B, M, H = 2, 700, 2
    q = seeded((B, M, H, 64), 81, "cuda", torch.float16)
    k = seeded((B, M, H, 64), 82, "cuda")
    v = seeded((B, M, H, 64), 83, "cuda")
    g = Q.PrefillGraph(q, k, v, 128, causal=False)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g.launch(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert_device_clean()
    _same(g, _eager(q, k, v, 128, causal=False), M, 64)
    want, *_ = oracle_out(q, k, v, causal=False)
    compare(g.out.cpu().numpy(), want, "graph, no mask")
    g.close()


def test_graph_create_reports_a_failing_call_and_leaves_no_capture(lib):
    """A captured call that rejects its arguments (here a K buffer that is only
    4-byte aligned) makes the create fail with that call's code and no handle;
    the capture is ended, so a following create and replay work."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    from tests.parity import seeded
    B, M, H = 1, 256, 2
    q = seeded((B, M, H, 64), 91, "cuda", torch.float16)
    k_buf = seeded((B * M * H * 64 + 4,), 92, "cuda")
    v = seeded((B, M, H, 64), 93, "cuda")
    k_bad = k_buf[1:1 + B * M * H * 64].view(B, M, H, 64)
    with pytest.raises(Q.Q8AttnError) as err:
        Q.PrefillGraph(q, k_bad, v, 128)
    assert err.value.code == Q.Q8A_ERR_MISALIGNED
    k = k_bad.clone()
    g = Q.PrefillGraph(q, k, v, 128)
    g.launch()
    torch.cuda.synchronize()
    assert_device_clean()
    _same(g, _eager(q, k, v, 128), M, 64)
    g.close()


def test_graph_as_the_first_call_of_a_process(lib):
    """A process whose first library call is the captured prefill (so the
    kernels' one-time launch set-up happens while the graph is being recorded)
    gets the same bits as the calls made one by one, at both head sizes."""
    import subprocess
    import sys
    from tests.conftest import ROOT
    code = r"""
import torch
from chunked_prefill_attention_gb300 import q8attn as Q
from tests.parity import seeded
for D, chunk in ((64, 128), (128, 256)):
    B, M, H = 1, 600, 2
    q = seeded((B, M, H, D), 11 + D, "cuda", torch.float16)
    k = seeded((B, M, H, D), 12 + D, "cuda")
    v = seeded((B, M, H, D), 13 + D, "cuda")
    g = Q.PrefillGraph(q, k, v, chunk)
    g.launch()
    torch.cuda.synchronize()
    ref, *_ = Q.prefill_attention(q, k, v, chunk)
    assert torch.equal(g.out, ref), D
    g.close()
print("ok")
"""
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
