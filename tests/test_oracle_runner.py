"""Pins for oracle/runner.py, the whole-problem driver that every GPU parity
test compares against.  Each check compares the runner with the plain
functions it assembles (per-plane `attention.attention_unchunked`, serial
`q8_0.quantize_kv`), which are pinned themselves in test_oracle_pins.py, so a
slip in the runner's own bookkeeping -- which plane lands where in the output,
which K/V head a query head reads, how the parallel quantise pieces are joined
-- fails here on the CPU.  CPU only."""

import math

import numpy as np
import pytest

from oracle import attention as att
from oracle import q8_0, runner


def _problem(B, H, H_kv, n_q, M, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, n_q, H, 64)).astype(np.float16)
    k = rng.standard_normal((B, M, H_kv, 64)).astype(np.float32)
    v = rng.standard_normal((B, M, H_kv, 64)).astype(np.float32)
    # distinct scales per (b, head) so that every plane's output differs clearly
    k *= (1.0 + 0.25 * np.arange(B * H_kv, dtype=np.float32)).reshape(B, 1, H_kv, 1)
    v += np.arange(B * H_kv, dtype=np.float32).reshape(B, 1, H_kv, 1)
    return q, q8_0.quantize_kv(k), q8_0.quantize_kv(v)


def _per_plane(q, k8, v8, scale, causal, q_pos0):
    """The definition, one (b, h) plane at a time: query head h of H reads K/V
    head h // (H // H_kv) ("grouped-query" extension; H_kv = H is multi-head)."""
    B, n_q, H, D = q.shape
    H_kv = k8.shape[1]
    out = np.zeros((B, n_q, H, D))
    for b in range(B):
        for h in range(H):
            g = h // (H // H_kv)
            out[b, :, h] = att.attention_unchunked(
                q[b, :, h], q8_0.dequantize_kv(k8[b, g]), q8_0.dequantize_kv(v8[b, g]), scale,
                causal=causal, q_pos0=q_pos0)
    return out


def runner_attention_agrees(rm, H_kv=2, causal=True, seed=21):
    """rm.attention against the per-plane definition on B = 2, H = 4, with a
    query offset and a shuffled subset of rows."""
    B, H, n_q, q_pos0 = 2, 4, 40, 16
    M = q_pos0 + n_q
    q, k8, v8 = _problem(B, H, H_kv, n_q, M, seed)
    scale = 1.0 / math.sqrt(64)
    rows = np.random.default_rng(seed + 1).permutation(n_q)[:27]
    got = rm.attention(q, k8, v8, scale, causal=causal, rows=rows, q_pos0=q_pos0)
    want = _per_plane(q, k8, v8, scale, causal, q_pos0)[:, rows]
    return got.shape == want.shape and np.allclose(got, want, rtol=0, atol=1e-13)


def runner_quantize_agrees(rm):
    """The parallel quantise (token ranges on worker processes, B = 2, a ragged
    last range) gives the serial quantiser's bytes."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal((2, 4100, 32, 64)).astype(np.float32)
    x[1] *= 3.0
    assert 2 * 4100 * 32 >= 65536      # large enough to take the parallel path
    got = rm.quantize_kv(x, parallel=True)
    return got.shape == (2, 32, 4100, 68) and np.array_equal(got, q8_0.quantize_kv(x))


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("H_kv", [4, 2, 1])
def test_runner_attention_is_the_per_plane_definition(H_kv, causal):
    assert runner_attention_agrees(runner, H_kv=H_kv, causal=causal)


def test_runner_parallel_quantise_is_the_serial_quantiser():
    assert runner_quantize_agrees(runner)


def test_runner_planes_differ():
    """The check above can see a plane mix-up only if the planes differ."""
    q, k8, v8 = _problem(2, 4, 2, 8, 8, 5)
    out = _per_plane(q, k8, v8, 0.125, True, 0)
    for i in range(8):
        for j in range(i + 1, 8):
            assert not np.allclose(out[i // 4, :, i % 4], out[j // 4, :, j % 4])
