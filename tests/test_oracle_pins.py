"""Pins for the CPU oracle: checks against what the pages print, closed forms,
invariants and brute force, so that a plausible slip in the oracle fails here.
CPU only."""

import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import q8_0, attention as att

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _block(values):
    x = np.zeros(32, dtype=np.float32)
    for k, v in values.items():
        x[int(k)] = np.float32(v)
    return x


# ---------------------------------------------------------------- format ----

def test_block_layout_matches_page():
    g = _golden("page_constants.json")["block"]
    assert q8_0.BLOCK_VALUES == g["values"]
    assert q8_0.BLOCK_BYTES == g["bytes"] == g["values"] * 1 + 2
    assert q8_0.ROW_BYTES == 2 * g["bytes"]
    # 64 -> 34 bytes per 32 values: 46.875 %, printed as 46.88 % and 47 %
    red = 100.0 * (1 - g["bytes"] / g["fp16_bytes"])
    assert red == 46.875
    assert round(red, 2) == g["reduction_percent_printed"]
    assert round(red) == g["reduction_percent_rounded_printed"]


def test_pack_byte_offsets():
    d16 = np.array([[np.float16(1.5), np.float16(-2.0)]])
    q = np.zeros((1, 2, 32), dtype=np.int8)
    q[0, 0, 0], q[0, 0, 31], q[0, 1, 0], q[0, 1, 31] = 7, -1, -128 + 1, 127
    raw = q8_0.pack_rows(d16, q)[0]
    assert raw.shape == (68,)
    assert raw[0:2].tobytes() == np.float16(1.5).tobytes()          # scale first, little-endian
    assert raw[2] == 7 and raw[33] == 255                              # codes at 2..33
    assert raw[34:36].tobytes() == np.float16(-2.0).tobytes()         # second block at 34
    assert raw[36] == 129 and raw[67] == 127
    d2, q2 = q8_0.unpack_rows(raw[None])
    assert np.array_equal(d2.view(np.uint16), d16.view(np.uint16)) and np.array_equal(q2, q)


@pytest.mark.parametrize("case", _golden("page_constants.json")["kv_sizes"]["cases"],
                         ids=lambda c: c["printed"])
def test_kv_sizes_match_printed_totals(case):
    f = q8_0.kv_cache_bytes if case["what"] == "q8_0" else q8_0.fp16_kv_cache_bytes
    b = f(case["layers"], case["heads"], case["tokens"], case["head_dim"])
    scaled = b / case["unit"]
    if case["rounding"] == "truncate":
        shown = math.floor(scaled * 10 ** case["digits"]) / 10 ** case["digits"]
    else:
        shown = round(scaled, case["digits"])
    assert shown * case["unit"] == pytest.approx(case["printed_bytes_rounded"])


def test_kv_size_exact_bytes():
    # 2 tensors * 32 heads * 65,536 tokens * 68 bytes
    assert q8_0.kv_cache_bytes(1, 32, 65536, 64) == 285_212_672
    assert q8_0.kv_cache_bytes(1, 32, 1048576, 64) == 4_563_402_752
    assert q8_0.kv_cache_bytes(16, 32, 1048576, 64) == 16 * 4_563_402_752
    assert q8_0.fp16_kv_cache_bytes(1, 32, 1048576, 64) == 8_589_934_592


# ------------------------------------------------------------- quantiser ----

@pytest.mark.parametrize("case", _golden("q8_0_blocks.json")["cases"], ids=lambda c: c["name"])
def test_quantiser_hand_checked_blocks(case):
    x = _block(case["values"])
    d16, q = q8_0.quantize_blocks(x)
    assert float(d16[0]) == case["d16"]
    want = np.zeros(32, dtype=np.int8)
    for k, v in case["codes"].items():
        want[int(k)] = v
    assert np.array_equal(q[0], want), (q[0], want)


def _random_blocks(n, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n, 64)) * scale).astype(np.float32)
    # heavy tails and a few tiny blocks so scales span many binades
    x[::7] *= np.float32(30.0)
    x[3::11] *= np.float32(1e-3)
    return x


def test_quantiser_round_trip_bound():
    x = _random_blocks(4000, 1)
    d16, q = q8_0.quantize_blocks(x)
    xb = x.reshape(-1, 2, 32).astype(np.float64)
    d = d16.astype(np.float64)[..., None]
    err = np.abs(xb - d * q.astype(np.float64))
    assert np.all(err <= d / 2 * (1 + 2.0 ** -16))


def test_quantiser_uses_full_code_range():
    x = _random_blocks(4000, 2)
    d16, q = q8_0.quantize_blocks(x)
    normal = d16.astype(np.float64) >= 2.0 ** -14
    peak = np.max(np.abs(q.astype(np.int32)), axis=-1)
    assert np.all(peak[normal] == 127)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)


def test_quantiser_idempotent_on_dequantised_blocks():
    x = _random_blocks(3000, 3)
    d16, q = q8_0.quantize_blocks(x)
    y = q8_0.dequantize_blocks(d16, q).astype(np.float32)   # d16*q is exact in fp32
    d2, q2 = q8_0.quantize_blocks(y.reshape(x.shape))
    normal = d16 >= np.float16(2.0 ** -14)
    assert np.array_equal(d2.view(np.uint16)[normal], d16.view(np.uint16)[normal])
    assert np.array_equal(q2[normal], q[normal])


def test_quantiser_sign_symmetry():
    x = _random_blocks(500, 4)
    d1, q1 = q8_0.quantize_blocks(x)
    d2, q2 = q8_0.quantize_blocks(-x)
    assert np.array_equal(d1.view(np.uint16), d2.view(np.uint16))
    assert np.array_equal(q1.astype(np.int32), -q2.astype(np.int32))


def test_quantiser_scale_is_amax_over_127_in_fp16():
    # brute force per block with Python floats: d16 = nearest fp16 to fl32(amax/127)
    x = _random_blocks(200, 5)
    d16, _ = q8_0.quantize_blocks(x)
    for i in range(x.shape[0]):
        for b in range(2):
            amax = max(abs(float(v)) for v in x[i, 32 * b:32 * b + 32])
            d32 = np.float32(amax) / np.float32(127)
            assert np.float16(d32) == d16[i, b]


def test_quantize_kv_layout_is_head_major():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, 5, 3, 64)).astype(np.float32)   # [B, M, H, D]
    raw = q8_0.quantize_kv(x)
    assert raw.shape == (2, 3, 5, 68)
    for b, m, h in itertools.product(range(2), range(5), range(3)):
        d16, q = q8_0.quantize_blocks(x[b, m, h])
        assert np.array_equal(raw[b, h, m], q8_0.pack_rows(d16[None], q[None])[0])
    y = q8_0.dequantize_kv(raw)
    assert y.shape == (2, 3, 5, 64)
    assert np.max(np.abs(y - x.transpose(0, 2, 1, 3))) <= np.max(np.abs(x)) / 127



def test_quantize_kv_head_dim_128_is_four_blocks_in_channel_order():
    """A 128-channel head row is four blocks, channels 0-31, 32-63, 64-95,
    96-127, each quantised on its own: 136 bytes, the 34-byte block four times."""
    rng = np.random.default_rng(16)
    x = rng.standard_normal((1, 3, 2, 128)).astype(np.float32)
    x[0, 1, 0, 64:96] *= 40.0       # one block with a much larger scale
    raw = q8_0.quantize_kv(x)
    assert raw.shape == (1, 2, 3, 136)
    for m, h, j in itertools.product(range(3), range(2), range(4)):
        d16, q = q8_0.quantize_blocks(x[0, m, h, 32 * j:32 * j + 32])
        assert np.array_equal(raw[0, h, m, 34 * j:34 * j + 34], q8_0.pack_rows(d16[None], q[None])[0])
    y = q8_0.dequantize_kv(raw)
    assert y.shape == (1, 2, 3, 128)
    # each block's round trip is bounded by its own scale
    for m, h, j in itertools.product(range(3), range(2), range(4)):
        blk = x[0, m, h, 32 * j:32 * j + 32]
        assert np.max(np.abs(y[0, h, m, 32 * j:32 * j + 32] - blk)) <= np.max(np.abs(blk)) / 127
    assert q8_0.kv_cache_bytes(1, 32, 1, 128) == 2 * 32 * 136
    with pytest.raises(ValueError):
        q8_0.quantize_kv(np.zeros((1, 1, 1, 48), dtype=np.float32))


# ------------------------------------------------------------- attention ----

def _brute(q, k, v, scale, causal=True, q_pos0=0):
    """Triple loop in pure Python floats: out_i = sum_j w_ij v_j,
    w_ij = exp(s_ij) / sum_j' exp(s_ij') over visible keys."""
    n_q, d = len(q), len(q[0])
    out = []
    for i in range(n_q):
        vis = [j for j in range(len(k)) if (not causal) or j <= q_pos0 + i]
        if not vis:
            out.append([0.0] * d)
            continue
        s = {j: scale * sum(float(q[i][t]) * float(k[j][t]) for t in range(d)) for j in vis}
        mx = max(s.values())
        e = {j: math.exp(s[j] - mx) for j in vis}
        z = sum(e.values())
        out.append([sum(e[j] * float(v[j][t]) for j in vis) / z for t in range(d)])
    return np.array(out)


@pytest.mark.parametrize("m,d,causal,q_pos0", [(1, 4, True, 0), (3, 5, True, 0), (8, 8, True, 0),
                                               (6, 4, False, 0), (5, 3, True, 2), (4, 128, True, 0)])
def test_attention_matches_brute_force(m, d, causal, q_pos0):
    rng = np.random.default_rng(m * 10 + d)
    n_k = m + q_pos0
    q = rng.standard_normal((m, d))
    k = rng.standard_normal((n_k, d))
    v = rng.standard_normal((n_k, d))
    scale = 1 / math.sqrt(d)
    want = _brute(q, k, v, scale, causal, q_pos0)
    assert np.allclose(att.attention_unchunked(q, k, v, scale, causal, q_pos0), want, rtol=0, atol=1e-13)
    rows = np.arange(m)[::-1]
    assert np.allclose(att.attention_rows(q[rows], k, v, rows, scale, causal, q_pos0), want[rows], rtol=0, atol=1e-13)
    for kb in (1, 2, 3):   # key blocks smaller than the rows: same two-pass result
        got = att.attention_rows(q[rows], k, v, rows, scale, causal, q_pos0, block=2, key_block=kb)
        assert np.allclose(got, want[rows], rtol=0, atol=1e-13)
    for c in (1, 2, 3):
        got = att.attention_chunked(q, k, v, c, scale, causal, q_pos0)
        assert np.allclose(got, want, rtol=0, atol=1e-13)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(0)
    q, k, v = (rng.standard_normal((1, 64)) for _ in range(3))
    assert np.array_equal(att.attention_unchunked(q, k, v, 0.125), v)


def test_first_row_is_first_value():
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((50, 64)) for _ in range(3))
    out = att.attention_unchunked(q, k, v, 0.125)
    assert np.array_equal(out[0], v[0])


def test_equal_keys_give_causal_running_mean():
    rng = np.random.default_rng(2)
    n = 40
    q = rng.standard_normal((n, 64))
    k = np.repeat(rng.standard_normal((1, 64)), n, axis=0)
    v = rng.standard_normal((n, 64))
    want = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    assert np.allclose(att.attention_unchunked(q, k, v, 0.125), want, atol=1e-13)
    assert np.allclose(att.attention_chunked(q, k, v, 7, 0.125), want, atol=1e-13)


def test_zero_query_gives_uniform_average():
    rng = np.random.default_rng(3)
    n = 33
    q = np.zeros((n, 64))
    k = rng.standard_normal((n, 64))
    v = rng.standard_normal((n, 64))
    want = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    assert np.allclose(att.attention_unchunked(q, k, v, 0.125), want, atol=1e-13)


def test_constant_values_give_constant_output():
    rng = np.random.default_rng(4)
    n = 30
    q, k = rng.standard_normal((n, 64)), rng.standard_normal((n, 64))
    v = np.tile(rng.standard_normal((1, 64)), (n, 1))
    assert np.allclose(att.attention_unchunked(q, k, v, 0.125), v, atol=1e-13)


def test_scale_is_one_over_sqrt_d():
    # two keys whose dot products with q differ by 8*ln 3: with scale 1/sqrt(64)
    # the weights are 3/4 and 1/4 exactly
    d = 64
    q = np.zeros((2, d)); q[1, 0] = 1.0
    k = np.zeros((2, d)); k[1, 0] = 8 * math.log(3.0)
    v = np.zeros((2, d)); v[0, 0] = 1.0; v[1, 1] = 1.0
    out = att.attention_unchunked(q, k, v, 1 / math.sqrt(d))
    assert out[1, 0] == pytest.approx(0.25, abs=1e-15)
    assert out[1, 1] == pytest.approx(0.75, abs=1e-15)


def test_dominant_logit_gives_one_hot():
    rng = np.random.default_rng(5)
    n = 12
    q = np.zeros((n, 64)); q[:, 0] = 1.0
    k = rng.standard_normal((n, 64)) * 0.01
    k[4, 0] = 2000.0    # scaled logit 250 for every row that can see key 4
    v = rng.standard_normal((n, 64))
    out = att.attention_unchunked(q, k, v, 0.125)
    assert np.allclose(out[4:], np.tile(v[4], (n - 4, 1)), atol=1e-12)


def test_softmax_weights_sum_to_one_and_respect_the_mask():
    rng = np.random.default_rng(6)
    n = 24
    q, k = rng.standard_normal((n, 16)) * 3, rng.standard_normal((n, 16)) * 3
    v = np.eye(n)      # output row i = the weights of row i
    w = att.attention_unchunked(q, k, v, 0.25)
    assert np.all(np.abs(w.sum(axis=1) - 1) < 1e-12)
    assert np.all(w >= 0)
    assert np.all(np.triu(w, 1) == 0)
    w2 = att.attention_chunked(q, k, v, 5, 0.25)
    assert np.all(np.abs(w2.sum(axis=1) - 1) < 1e-12)


@pytest.mark.parametrize("chunk", [1, 3, 16, 37, 64, 200])
def test_chunked_equals_unchunked(chunk):
    rng = np.random.default_rng(chunk)
    n = 150
    q = rng.standard_normal((n, 64))
    k = rng.standard_normal((n, 64)) * 2
    v = rng.standard_normal((n, 64))
    want = att.attention_unchunked(q, k, v, 0.125)
    got = att.attention_chunked(q, k, v, chunk, 0.125)
    assert np.max(np.abs(got - want)) < 1e-12


def test_chunk_order_does_not_matter():
    rng = np.random.default_rng(11)
    n = 96
    q = rng.standard_normal((n, 64))
    k = rng.standard_normal((n, 64)) * 3   # big logits so later chunks raise the max
    v = rng.standard_normal((n, 64))
    want = att.attention_unchunked(q, k, v, 0.125)
    for order in ([3, 1, 0, 2], [2, 3, 1, 0], [0, 1, 2, 3]):
        got = att.attention_chunked(q, k, v, 24, 0.125, order=order)
        assert np.max(np.abs(got - want)) < 1e-12


def test_future_chunk_leaves_state_untouched():
    # the causal skip: a chunk whose keys all lie after every query changes nothing
    rng = np.random.default_rng(12)
    q, k, v = (rng.standard_normal((16, 64)) for _ in range(3))
    st = att.state_init(8, 64)
    att.chunk_step(st, q[:8], k[:8], v[:8], 0, 0.125)
    before = {n: a.copy() for n, a in st.items()}
    att.chunk_step(st, q[:8], k[8:], v[8:], 8, 0.125)
    for n in before:
        assert np.array_equal(before[n], st[n])


def test_state_checkpoint_resume_is_exact():
    rng = np.random.default_rng(13)
    n = 64
    q, k, v = (rng.standard_normal((n, 64)) for _ in range(3))
    st = att.state_init(n, 64)
    for s0 in range(0, n, 16):
        att.chunk_step(st, q, k[s0:s0 + 16], v[s0:s0 + 16], s0, 0.125)
    st2 = att.state_init(n, 64)
    for s0 in range(0, 32, 16):
        att.chunk_step(st2, q, k[s0:s0 + 16], v[s0:s0 + 16], s0, 0.125)
    saved = {n_: np.array(a) for n_, a in st2.items()}
    st3 = {n_: a.copy() for n_, a in saved.items()}
    for s0 in range(32, n, 16):
        att.chunk_step(st3, q, k[s0:s0 + 16], v[s0:s0 + 16], s0, 0.125)
    for n_ in st:
        assert np.array_equal(st[n_], st3[n_])


def test_row_without_visible_key_finalises_to_zero():
    st = att.state_init(3, 4)
    assert np.array_equal(att.finalize(st), np.zeros((3, 4)))
    # queries at positions 0..2, keys at 5..6: nothing visible
    rng = np.random.default_rng(14)
    q, k, v = rng.standard_normal((3, 4)), rng.standard_normal((2, 4)), rng.standard_normal((2, 4))
    att.chunk_step(st, q, k, v, 5, 0.5)
    assert np.all(np.isneginf(st["m"])) and np.all(st["l"] == 0)
    assert np.array_equal(att.finalize(st), np.zeros((3, 4)))


# ---- grouped-query attention (an extension: the pages describe one K/V head
# per query head; query head h of H reads K/V head h // (H / H_kv)) ----------

def _gqa_case(H, H_kv, M=48, seed=7):
    from oracle import runner
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, M, H, 64)).astype(np.float16)
    k = rng.standard_normal((1, M, H_kv, 64)).astype(np.float32)
    v = rng.standard_normal((1, M, H_kv, 64)).astype(np.float32)
    return q, runner.quantize_kv(k, parallel=False), runner.quantize_kv(v, parallel=False)


@pytest.mark.parametrize("H,H_kv", [(4, 2), (6, 3), (4, 1)])
def test_gqa_equals_multi_head_on_repeated_kv(H, H_kv):
    """Grouped heads give exactly what multi-head attention gives when every
    K/V plane is repeated for the H / H_kv query heads of its group."""
    from oracle import runner
    q, k8, v8 = _gqa_case(H, H_kv)
    got = runner.attention(q, k8, v8, 0.125)
    rep = H // H_kv
    want = runner.attention(q, np.repeat(k8, rep, axis=1), np.repeat(v8, rep, axis=1), 0.125)
    assert np.array_equal(got, want)
    # and not what an interleaved (h % H_kv) assignment would give
    if H_kv > 1 and rep > 1:
        inter = runner.attention(q, np.tile(k8, (1, rep, 1, 1)), np.tile(v8, (1, rep, 1, 1)), 0.125)
        assert not np.allclose(got, inter)


def test_mqa_identical_queries_give_identical_heads():
    """One K/V head shared by all query heads: heads with the same queries
    produce the same output."""
    from oracle import runner
    q, k8, v8 = _gqa_case(4, 1)
    q[:, :, 1] = q[:, :, 0]
    q[:, :, 3] = q[:, :, 0]
    out = runner.attention(q, k8, v8, 0.125)
    assert np.array_equal(out[:, :, 1], out[:, :, 0]) and np.array_equal(out[:, :, 3], out[:, :, 0])
    assert not np.allclose(out[:, :, 2], out[:, :, 0])


def test_gqa_rejects_ungrouped_heads():
    from oracle import runner
    q, k8, v8 = _gqa_case(4, 2)
    with pytest.raises(ValueError):
        runner.attention(q[:, :, :3], k8, v8, 0.125)
