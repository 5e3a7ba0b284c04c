"""Why the chunk step splits the dequantised K and V into an fp16 high part and
an fp16 residual, at twice the tensor-core work of plain fp16 operands.

The chunk step's arithmetic is emulated here in numpy on the oracle's Q8_0
bytes (the same seeded draws as the GPU workloads, fewer tokens and heads):
scores from the K operand in fp32, the eager running max per 128-key tile,
beta = 2^(S * scale * log2 e - m * log2 e) in fp32, P = fp16(beta), l summed
from beta in fp32, O accumulated in fp32 tile by tile, and O / l rounded to
fp16 at the end -- the online softmax of "Out-of-Core Flash Streaming &
Speculative Decode (1M Context)", §3, in the order the kernel takes it.  Each
operand is either exact (d * q, which the high part plus the residual
represent without error) or d * q rounded once to fp16.  The result is
compared with the oracle's plain attention over the same dequantised K and V
against the GPU parity tolerance.

What it shows: the exact operands stay well inside the tolerance on every
workload's distribution; fp16 K breaks it on the outlier workload (channels
scaled x20, |K| up to about 80, where fp16 keeps 11 bits); fp16 V stays
inside it there, but uses nearly all of it.  CPU only, about ten seconds."""

import math

import numpy as np
import pytest

from chunked_prefill_attention_gb300 import workloads as W
from oracle import attention, q8_0
from tests.parity import MAX_ABS, REL_L2


def _f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def _f16(x):
    return np.asarray(x, dtype=np.float16).astype(np.float64)


def _emulate_head(q, k, v, k_fp16, v_fp16, scale=0.125):
    """One causal head, keys folded in 128-key tiles (the chunk boundaries do
    not change this arithmetic: the kernel carries m, l and O in fp32 across
    them).  q fp16 values, k and v dequantised, all float64 [M, D]."""
    M = q.shape[0]
    kk = _f16(k) if k_fp16 else k
    vv = _f16(v) if v_fp16 else v
    s_all = _f32(q @ kk.T)
    c = float(np.float32(scale * math.log2(math.e)))
    m = np.full(M, -np.inf)
    l = np.zeros(M)
    o = np.zeros((M, q.shape[1]))
    rows = np.arange(M)
    for t0 in range(0, M, 128):
        t1 = min(t0 + 128, M)
        s = s_all[:, t0:t1].copy()
        s[np.arange(t0, t1)[None, :] > rows[:, None]] = -np.inf
        m_new = np.maximum(m, _f32(s.max(axis=1) * scale))
        with np.errstate(invalid="ignore"):
            alpha = np.where(m_new > m, np.where(np.isneginf(m), 0.0, np.exp2((m - m_new) * math.log2(math.e))),
                             1.0)
        m = m_new
        mlog = np.where(np.isneginf(m), 0.0, _f32(m * math.log2(math.e)))
        beta = _f32(np.exp2(_f32(s * c - mlog[:, None])))
        o = _f32(o * alpha[:, None] + _f16(beta) @ vv[t0:t1])
        l = _f32(l * alpha + beta.sum(axis=1))
    return _f16(_f32(o / l[:, None]))


def _errors(name, tokens, heads, k_fp16, v_fp16):
    w = W.WORKLOADS[name]
    q, k, v = (t.numpy() for t in W.make_inputs(w, tokens=tokens))
    k8 = q8_0.quantize_kv(k[:, :, :heads])
    v8 = q8_0.quantize_kv(v[:, :, :heads])
    worst, num, den = 0.0, 0.0, 0.0
    for h in range(heads):
        kh, vh = q8_0.dequantize_kv(k8[0, h]), q8_0.dequantize_kv(v8[0, h])
        qh = q[0, :, h].astype(np.float64)
        want = attention.attention_unchunked(qh, kh, vh, 0.125)
        err = np.abs(_emulate_head(qh, kh, vh, k_fp16, v_fp16) - want)
        worst = max(worst, float(err.max()))
        num += float(np.sum(err ** 2))
        den += float(np.sum(want ** 2))
    return worst, math.sqrt(num / den)


CASES = [("m512", 512, 16), ("m2k_out", 2048, 8), ("b8_m2k", 2048, 4), ("m64k", 2048, 4)]


@pytest.mark.parametrize("name,tokens,heads", CASES)
def test_exact_operands_within_tolerance(name, tokens, heads):
    worst, rel = _errors(name, tokens, heads, False, False)
    assert worst <= 0.7 * MAX_ABS and rel <= 0.5 * REL_L2, (name, worst, rel)


def test_fp16_k_breaks_tolerance_on_outlier_channels():
    worst, rel = _errors("m2k_out", 2048, 8, True, False)
    assert worst > MAX_ABS, worst
    assert rel > REL_L2, rel


def test_fp16_v_leaves_no_margin_on_outlier_channels():
    exact, _ = _errors("m2k_out", 2048, 8, False, False)
    worst, _ = _errors("m2k_out", 2048, 8, False, True)
    assert worst > 0.9 * MAX_ABS, worst
    assert worst > 1.5 * exact, (worst, exact)
