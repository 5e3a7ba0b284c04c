"""Planted mistakes: each case copies one oracle module, plants a plausible
slip in the copy (on the CPU, never in the real module) and checks that the pin
checks below catch it.  This shows the pins can tell a right oracle from a
subtly wrong one."""

import json
import math
import os
import types

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _mutant(module, old, new):
    path = os.path.join(ROOT, "oracle", module + ".py")
    with open(path) as f:
        src = f.read()
    assert old in src, f"mutation anchor not found in {module}: {old!r}"
    mod = types.ModuleType("mutant_" + module)
    exec(compile(src.replace(old, new), path + " (mutant)", "exec"), mod.__dict__)
    return mod


def _quant_pins_pass(qm):
    with open(os.path.join(ROOT, "tests", "golden", "q8_0_blocks.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        x = np.zeros(32, dtype=np.float32)
        for k, v in c["values"].items():
            x[int(k)] = v
        d16, q = qm.quantize_blocks(x)
        want = np.zeros(32, dtype=np.int8)
        for k, v in c["codes"].items():
            want[int(k)] = v
        if float(d16[0]) != c["d16"] or not np.array_equal(q[0], want):
            return False
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, 2, 3, 64)).astype(np.float32)
    raw = qm.quantize_kv(x)
    d16, q = qm.unpack_rows(raw[0, 0, 0][None])
    d_ref, q_ref = qm.quantize_blocks(x[0, 0, 0])
    if not (np.array_equal(d16[0].view(np.uint16), d_ref.view(np.uint16)) and np.array_equal(q[0], q_ref)):
        return False
    if raw[0, 0, 0, 0:2].tobytes() != d_ref[0].tobytes():
        return False
    return True


def _brute(q, k, v, scale):
    out = []
    for i in range(len(q)):
        s = [scale * float(np.dot(q[i], k[j])) for j in range(i + 1)]
        mx = max(s)
        e = [math.exp(t - mx) for t in s]
        out.append(sum(e[j] * v[j] for j in range(i + 1)) / sum(e))
    return np.array(out)


def _attention_pins_pass(am):
    rng = np.random.default_rng(1)
    n, d = 10, 8
    q = rng.standard_normal((n, d))
    k = rng.standard_normal((n, d)) * 2
    v = rng.standard_normal((n, d))
    scale = 1 / math.sqrt(d)
    want = _brute(q, k, v, scale)
    for got in (am.attention_unchunked(q, k, v, scale),
                am.attention_rows(q[::-1], k, v, np.arange(n)[::-1], scale)[::-1],
                am.attention_rows(q, k, v, np.arange(n), scale, block=3, key_block=4),
                am.attention_chunked(q, k, v, 3, scale),
                am.attention_chunked(q, k, v, 4, scale, order=[2, 0, 1])):
        if not np.allclose(got, want, atol=1e-12, rtol=0):
            return False
    return True


QUANT_MUTANTS = [
    ("divide by 128", "amax / np.float32(127.0)", "amax / np.float32(128.0)"),
    ("round half to even", "np.floor(np.abs(r64) + 0.5)", "np.round(np.abs(r64))"),
    ("codes from the fp32 scale", "dd = d16.astype(np.float32)[..., None]", "dd = d32[..., None]"),
    ("truncate instead of round", "np.floor(np.abs(r64) + 0.5)", "np.floor(np.abs(r64))"),
    ("codes before scale in the block", "out[..., 0:2] = d16", "out[..., 32:34] = d16"),
    ("amax without abs", "np.max(np.abs(xb), axis=-1)", "np.max(xb, axis=-1)"),
]

ATTN_MUTANTS = [
    ("alpha sign flipped", "np.exp(np.where(live, m_old - m_safe, 0.0))", "np.exp(np.where(live, m_safe - m_old, 0.0))"),
    ("mask off by one", "return k_pos[None, :] <= q_pos[:, None]", "return k_pos[None, :] < q_pos[:, None]"),
    ("l not rescaled", "l_new = l_old * alpha + np.sum(beta, axis=1)", "l_new = l_old + np.sum(beta, axis=1)"),
    ("O not rescaled", "o_new = o_old * alpha[:, None] + beta @ v_c", "o_new = o_old + beta @ v_c"),
    ("scale applied twice", "s = (q @ k.T) * scale", "s = (q @ k.T) * scale * scale"),
    ("row block reads keys transposed", "return np.where(vis, (qb @ kb.T) * scale, -np.inf), vis",
     "return np.where(vis, (qb @ kb[::-1].T) * scale, -np.inf), vis"),
    ("row block drops a key block from the sum", "for k0 in range(0, n_k, key_block):            # pass 2",
     "for k0 in range(key_block, n_k, key_block):            # pass 2"),
    ("max not subtracted per row", "beta = np.where(vis & live[:, None], np.exp(s - m_safe[:, None]), 0.0)",
     "beta = np.where(vis & live[:, None], np.exp(s - m_safe[None, :1]), 0.0)"),
    ("finalise multiplies", "state[\"O\"] / np.where(pos, l, 1.0)[:, None]", "state[\"O\"] * np.where(pos, l, 1.0)[:, None]"),
]


def test_unmutated_oracle_passes_the_checks():
    import oracle.q8_0 as qm
    import oracle.attention as am
    assert _quant_pins_pass(qm)
    assert _attention_pins_pass(am)


@pytest.mark.parametrize("name,old,new", QUANT_MUTANTS, ids=[m[0] for m in QUANT_MUTANTS])
def test_quantiser_mutant_is_caught(name, old, new):
    try:
        ok = _quant_pins_pass(_mutant("q8_0", old, new))
    except Exception:
        ok = False
    assert not ok, f"planted mistake not caught: {name}"


@pytest.mark.filterwarnings("ignore:invalid value encountered:RuntimeWarning")   # a mutant may produce NaN
@pytest.mark.parametrize("name,old,new", ATTN_MUTANTS, ids=[m[0] for m in ATTN_MUTANTS])
def test_attention_mutant_is_caught(name, old, new):
    try:
        ok = _attention_pins_pass(_mutant("attention", old, new))
    except Exception:
        ok = False
    assert not ok, f"planted mistake not caught: {name}"


def _runner_pins_pass(rm):
    """The runner checks of test_oracle_runner.py on a mutant runner.  The
    mutant keeps the real worker pool and task functions (spawned workers can
    only import the real module); every planted slip below sits in the code that
    runs in this process."""
    from oracle import runner
    from tests import test_oracle_runner as pins
    rm.pool, rm._attn_task, rm._quant_task = runner.pool, runner._attn_task, runner._quant_task
    return (pins.runner_attention_agrees(rm, H_kv=2, causal=True)
            and pins.runner_attention_agrees(rm, H_kv=1, causal=False)
            and pins.runner_quantize_agrees(rm))


RUNNER_MUTANTS = [
    ("plane assembly swaps batch and head", "out[i // H, :, i % H] = r", "out[i % B, :, i // B] = r"),
    ("interleaved head groups", "g = h // group", "g = h % H_kv"),
    ("quantise pieces joined in reverse token order",
     "parts.append(np.concatenate(pool().map(_quant_task, tasks), axis=2))",
     "parts.append(np.concatenate(pool().map(_quant_task, tasks)[::-1], axis=2))"),
    ("quantise batch entries swapped", "return np.concatenate(parts, axis=0)",
     "return np.concatenate(parts[::-1], axis=0)"),
    ("causal key range cut one short",
     "min(k8.shape[2], q_pos0 + int(rows.max()) + 1)", "min(k8.shape[2], q_pos0 + int(rows.max()))"),
]


def test_unmutated_runner_passes_the_checks():
    assert _runner_pins_pass(_mutant("runner", "", ""))


@pytest.mark.parametrize("name,old,new", RUNNER_MUTANTS, ids=[m[0] for m in RUNNER_MUTANTS])
def test_runner_mutant_is_caught(name, old, new):
    try:
        ok = _runner_pins_pass(_mutant("runner", old, new))
    except Exception:
        ok = False
    assert not ok, f"planted mistake not caught: {name}"
