"""Why the chunk step splits the dequantised K and V into an fp16 high part and
an fp16 residual, at twice the tensor-core work of plain fp16 operands.

The chunk step's arithmetic is emulated here in numpy on the oracle's Q8_0
bytes (the same seeded draws as the GPU workloads, fewer tokens and heads):
scores from the K operand in fp32, per 128-key tile a reference m that moves
to the tile max only when that exceeds m by more than 8 ln 2,
beta = 2^(S * scale * log2 e - m * log2 e) in fp32, P = fp16(beta), l summed
from beta in fp32 plus, per tile, fp16(beta) - beta of the tile's largest
score, O accumulated in fp32 tile by tile, and O / l rounded to fp16 at the
end -- the online softmax of "Out-of-Core Flash Streaming & Speculative Decode
(1M Context)", §3, in the order the kernel takes it.  Each
operand is either exact (d * q, which the high part plus the residual
represent without error) or d * q rounded once to fp16.  The result is
compared with the oracle's plain attention over the same dequantised K and V
against the GPU parity tolerance.

What it shows: the exact operands stay well inside the tolerance on every
workload's distribution; fp16 K breaks it on the outlier workload (channels
scaled x20, |K| up to about 80, where fp16 keeps 11 bits); fp16 V stays
inside it there, but uses nearly all of it.  It also shows why l takes the
tile max's weight as fp16 rounds it: without that term, a row dominated by one
key divides that key's fp16-rounded weight by its unrounded one, which doubles
the worst error on peaked draws.  CPU only, about twenty seconds."""

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


LAZY = 8 * math.log(2)   # the reference moves when a tile max exceeds it by more


def _emulate_head(q, k, v, k_fp16, v_fp16, scale=0.125, max_term=True):
    """One causal head, keys folded in 128-key tiles (the chunk boundaries do
    not change this arithmetic: the kernel carries m, l and O in fp32 across
    them).  q fp16 values, k and v dequantised, all float64 [M, D].
    max_term=False leaves out l's fp16(beta) - beta term of the tile max."""
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
        smax = s.max(axis=1)
        t_nat = _f32(smax * scale)
        move = t_nat > m + LAZY
        m_new = np.where(move, t_nat, m)
        with np.errstate(invalid="ignore"):
            alpha = np.where(move, np.where(np.isneginf(m), 0.0, np.exp2((m - m_new) * math.log2(math.e))), 1.0)
        m = m_new
        mlog = np.where(np.isneginf(m), 0.0, _f32(m * math.log2(math.e)))
        beta = _f32(np.exp2(_f32(s * c - mlog[:, None])))
        o = _f32(o * alpha[:, None] + _f16(beta) @ vv[t0:t1])
        lsum = beta.sum(axis=1)
        if max_term:
            bmax = np.where(np.isneginf(smax), 0.0, _f32(np.exp2(_f32(smax * c - mlog))))
            lsum = lsum + (_f16(bmax) - bmax)
        l = _f32(l * alpha + lsum)
    return _f16(_f32(o / l[:, None]))


def _errors_of(q, k, v, heads, k_fp16, v_fp16, max_term=True):
    k8 = q8_0.quantize_kv(k[:, :, :heads])
    v8 = q8_0.quantize_kv(v[:, :, :heads])
    worst, num, den = 0.0, 0.0, 0.0
    for h in range(heads):
        kh, vh = q8_0.dequantize_kv(k8[0, h]), q8_0.dequantize_kv(v8[0, h])
        qh = q[0, :, h].astype(np.float64)
        want = attention.attention_unchunked(qh, kh, vh, 0.125)
        err = np.abs(_emulate_head(qh, kh, vh, k_fp16, v_fp16, max_term=max_term) - want)
        worst = max(worst, float(err.max()))
        num += float(np.sum(err ** 2))
        den += float(np.sum(want ** 2))
    return worst, math.sqrt(num / den)


def _errors(name, tokens, heads, k_fp16, v_fp16):
    q, k, v = (t.numpy() for t in W.make_inputs(W.WORKLOADS[name], tokens=tokens))
    return _errors_of(q, k, v, heads, k_fp16, v_fp16)


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


def test_l_needs_the_rounded_weight_of_the_tile_max():
    """A peaked draw (K ~ N(0, 9), V ~ N(0, 4)) where rows are dominated by
    one key: with l summing only the fp32 weights, the dominant key's fp16
    weight over its fp32 one shows up in the output; with the tile max's
    rounding added to l the error is about half of that."""
    rng = np.random.default_rng(5)
    M, D, H = 2048, 64, 2
    q = rng.standard_normal((1, M, H, D)).astype(np.float16).astype(np.float32)
    k = (rng.standard_normal((1, M, H, D)) * 3.0).astype(np.float32)
    v = (rng.standard_normal((1, M, H, D)) * 2.0).astype(np.float32)
    with_term, _ = _errors_of(q, k, v, H, False, False, max_term=True)
    without, _ = _errors_of(q, k, v, H, False, False, max_term=False)
    assert without > 1.5 * with_term, (without, with_term)
