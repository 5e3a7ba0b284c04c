"""q8kv_quantize on the GPU vs the oracle: bit-exact bytes."""

import numpy as np
import pytest
import torch

from tests.conftest import cuda_available
from oracle import runner as oracle_runner
from tests.parity import gpu_bytes, seeded

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _check(x, lib, stride=None):
    from chunked_prefill_attention_gb300 import q8attn as Q
    B, M, H, _ = x.shape
    out = Q.q8kv_quantize(x, stride=stride)
    got = gpu_bytes(out, M)
    want = oracle_runner.quantize_kv(x.cpu().numpy())
    assert got.shape == want.shape
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        b, h, t, byte = bad[0]
        raise AssertionError(f"{len(bad)} bytes differ; first at b={b} h={h} t={t} byte={byte}: "
                             f"gpu {got[b, h, t]} oracle {want[b, h, t]}")
    return out


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 3, 2), (2, 5, 3), (1, 17, 8), (3, 100, 9),
                                   (1, 1001, 12), (2, 64, 32), (1, 130, 32)])
def test_quantize_shapes(lib, shape):
    B, M, H = shape
    x = seeded((B, M, H, 64), 100 + M, "cuda")
    _check(x, lib)


def test_quantize_special_values(lib):
    B, M, H = 1, 64, 8
    x = seeded((B, M, H, 64), 7, "cuda")
    x[0, 0] = 0.0                                   # all-zero blocks
    x[0, 1] *= 1e-6                                 # subnormal fp16 scales
    x[0, 2] *= 3e-8                                 # scales that underflow to 0
    x[0, 3] = torch.round(x[0, 3] * 8) / 8          # many exact ties
    x[0, 4, :, 0] = 127.0                           # d = 1 exactly, ties at .5
    x[0, 4, :, 1:32] = torch.arange(31, device="cuda", dtype=torch.float32) - 15.5
    x[0, 5] *= 1000.0                               # large values
    x[0, 6, :, 5] = -60000.0                        # near the fp16 range
    x[0, 7] = -x[0, 7].abs()                        # one-signed blocks
    _check(x, lib)


def test_quantize_codes_next_to_half_integer_quotients(lib):
    """Blocks whose scale is exactly d (amax = 127 d) and whose other values lie
    within three ulps of (k + 1/2) d: the code is decided by the last bit of
    the quotient x / d, so it must be the correctly rounded one."""
    rng = np.random.default_rng(11)
    M, H = 256, 16
    x = np.empty((1, M, H, 64), dtype=np.float32)
    for blk in range(2):
        e = rng.integers(-12, 8, size=(M, H))
        d = np.float16(np.ldexp(1.0 + rng.integers(0, 1024, size=(M, H)) / 1024.0, e)).astype(np.float32)
        k = rng.integers(0, 127, size=(M, H, 31)).astype(np.float32)
        base = ((k + 0.5) * d[..., None]).astype(np.float32)
        ulps = rng.integers(-3, 4, size=(M, H, 31))
        v = base.copy()
        for step in range(3):
            up = ulps > step
            dn = ulps < -step
            v = np.where(up, np.nextafter(v, np.float32(np.inf)), v)
            v = np.where(dn, np.nextafter(v, np.float32(-np.inf)), v)
        sign = np.where(rng.random((M, H, 31)) < 0.5, -1.0, 1.0).astype(np.float32)
        x[0, :, :, 32 * blk] = 127.0 * d
        x[0, :, :, 32 * blk + 1:32 * blk + 32] = v * sign
    _check(torch.from_numpy(x).cuda(), lib)


def test_quantize_padded_stride_leaves_padding(lib):
    from chunked_prefill_attention_gb300 import q8attn as Q
    B, M, H = 2, 7, 3
    x = seeded((B, M, H, 64), 9, "cuda")
    stride = 7 * 68 + 4 + 60        # 540 -> pad to 544 (multiple of 16)
    stride = (stride + 15) // 16 * 16
    out = torch.full((B, H, stride), 0xAB, dtype=torch.uint8, device="cuda")
    Q.q8kv_quantize(x, out=out, stride=stride)
    assert torch.all(out[:, :, M * 68:] == 0xAB)
    got = gpu_bytes(out, M)
    assert np.array_equal(got, oracle_runner.quantize_kv(x.cpu().numpy()))


@pytest.mark.parametrize("name", ["m512", "m2k_out", "b8_m2k", "m64k"])
def test_quantize_workloads_full(lib, name):
    from chunked_prefill_attention_gb300 import workloads
    w = workloads.WORKLOADS[name]
    _, k, v = workloads.make_inputs(w, device="cuda")
    _check(k, lib)
    _check(v, lib)


def test_quantize_m1m_sampled_windows(lib):
    """The 1,048,576-token problem: GPU quantises everything; the oracle checks
    token windows at both ends, around every chunk boundary and at seeded
    random places (quantisation is independent per row)."""
    from chunked_prefill_attention_gb300 import q8attn as Q, workloads
    w = workloads.WORKLOADS["m1m"]
    _, k, v = workloads.make_inputs(w, device="cuda")
    M = w.tokens
    g = torch.Generator().manual_seed(w.seed)
    starts = {0, M - 256} | {c * w.chunk - 128 for c in range(1, w.n_chunks)}
    starts |= set((torch.randint(0, M - 256, (24,), generator=g) // 16 * 16).tolist())
    for x in (k, v):
        out = Q.q8kv_quantize(x)
        for s0 in sorted(starts):
            got = out[:, :, s0 * 68:(s0 + 256) * 68].reshape(1, w.heads, 256, 68).cpu().numpy()
            want = oracle_runner.quantize_kv(x[:, s0:s0 + 256].cpu().numpy())
            assert np.array_equal(got, want), f"window at token {s0}"
        del out


def test_quantize_scale_overflow_gives_zero_codes(lib):
    """A block with amax beyond 65504 * 127 has its scale rounded to +inf in
    fp16; the oracle's codes are then x / inf = 0 (outside the documented
    input range, but still bit-exact)."""
    B, M, H = 1, 32, 4
    x = seeded((B, M, H, 64), 17, "cuda")
    x[0, 3, 1, :32] = 1.0e7 * torch.sign(x[0, 3, 1, :32])
    x[0, 9, 2, 32:] = -9.0e6
    out = _check(x, lib)
    raw = gpu_bytes(out, M)
    assert raw[0, 1, 3, 0:2].tobytes() == np.float16(np.inf).tobytes()
    assert not raw[0, 1, 3, 2:34].any()


@pytest.mark.parametrize("offset_floats", [4, 8])
def test_quantize_input_only_16_byte_aligned(lib, offset_floats):
    """An input 16 but not 32 bytes aligned is read with 128-bit loads; the
    bytes are the same."""
    B, M, H = 2, 50, 3
    base = seeded((B * M * H * 64 + offset_floats,), 23, "cuda")
    x = base[offset_floats:].view(B, M, H, 64)
    assert x.data_ptr() % 16 == 0
    _check(x, lib)
