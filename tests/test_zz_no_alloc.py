"""attn_chunk_step_split_static: the split chunk step for callers that cannot
allocate device memory at call time, such as code inside a host framework that
owns the device allocator, or a loop that cannot take the implicit device
synchronisation of cudaMalloc (its partial states live in a fixed scratch array
inside the library).  Checked through the C ABI against attn_chunk_step_split
with a workspace of the caller's own, on two different problems in a row (the
shared scratch keeps the first call's contents when the second one runs), and
against the oracle; and checked to take no device memory once loaded.  This
file is collected last on purpose."""

import ctypes
import math

import pytest
import torch

from tests.conftest import cuda_available
from tests.parity import MAX_ABS, assert_device_clean, seeded


def _call_static(lib, q, k8, v8, kv_start, kv_len, st, split, q_pos0, causal, k_off=0):
    B, n_q, H, D = q.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
    return lib.attn_chunk_step_split_static(
        ctypes.c_void_p(q.data_ptr()), q_pos0, ctypes.c_void_p(k8.data_ptr() + k_off),
        ctypes.c_void_p(v8.data_ptr() + k_off), k8.shape[-1], kv_start, kv_len,
        ctypes.c_void_p(st.m.data_ptr()), ctypes.c_void_p(st.l.data_ptr()),
        ctypes.c_void_p(st.o.data_ptr()), B, H, n_q, D, 1.0 / math.sqrt(D), int(causal), split, stream)


def test_static_scratch_limit_is_checked(lib):
    """Too large a split is refused before anything reaches the device."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    cap = lib.q8a_static_split_scratch_floats()
    assert cap == 8 * 1024 * 1024
    P = ctypes.c_void_p
    A16 = P(0x100000)
    # 1 x 32 heads x 4096 queries x 1,048,576 keys in ranges of 128: far beyond the scratch
    rc = lib.attn_chunk_step_split_static(A16, 0, A16, A16, 68 * 1048576, 0, 1048576, A16, A16, A16,
                                          1, 32, 4096, 64, 0.125, 0, 128, P(0))
    assert rc == Q.Q8A_ERR_INVALID_ARG
    assert b"static scratch" in lib.q8a_last_error()
    assert lib.attn_chunk_step_split_static(A16, 0, A16, A16, 68 * 128, 0, 128, A16, A16, A16, 1, 2,
                                            64, 64, 0.125, 0, 100, P(0)) == Q.Q8A_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")
def test_static_split_matches_workspace_split_twice(lib):
    """Two different problems in a row: the static scratch still holds the
    first problem's partials when the second runs.  The static call runs the
    same kernels on the same inputs as the workspace call, so m, l, O and the
    output must be identical; both are also checked against the oracle."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    from tests.parity import compare, oracle_out
    cases = [
        # 64 candidates after a 4,096-token context, rectangular mask
        dict(M=4096, H=4, n_q=64, q_pos0=4096, causal=False, split=512, chunk=4096, seed=901),
        # causal prefill of 1,000 tokens in two chunks, each split in ranges of 256
        dict(M=1000, H=3, n_q=1000, q_pos0=0, causal=True, split=256, chunk=512, seed=911),
    ]
    for c in cases:
        M, H, n_q = c["M"], c["H"], c["n_q"]
        q = seeded((1, n_q, H, 64), c["seed"], "cuda", torch.float16)
        k = seeded((1, M, H, 64), c["seed"] + 1, "cuda")
        v = seeded((1, M, H, 64), c["seed"] + 2, "cuda")
        k8, v8 = Q.q8kv_quantize(k), Q.q8kv_quantize(v)
        ref = Q.State(1, H, n_q, q.device)
        got = Q.State(1, H, n_q, q.device)
        for s0 in range(0, M, c["chunk"]):
            n = min(c["chunk"], M - s0)
            Q.attn_chunk_step_split(q, k8, v8, s0, n, ref, c["split"], q_pos0=c["q_pos0"],
                                    causal=c["causal"], k_offset_bytes=s0 * 68)
            rc = _call_static(lib, q, k8, v8, s0, n, got, c["split"], c["q_pos0"], c["causal"],
                              k_off=s0 * 68)
            assert rc == Q.Q8A_OK, lib.q8a_last_error()
        want, out = Q.attn_finalize(ref), Q.attn_finalize(got)
        assert_device_clean()
        assert torch.equal(ref.m, got.m) and torch.equal(ref.l, got.l) and torch.equal(ref.o, got.o)
        assert torch.equal(out, want)
        oracle, _, _ = oracle_out(q, k, v, causal=c["causal"], q_pos0=c["q_pos0"])
        compare(out.cpu().numpy(), oracle, f"static split M={M} n_q={n_q}")


@pytest.mark.gpu
@pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")
def test_static_split_takes_no_device_memory(lib):
    """After a first call (which loads the kernels and makes the scratch
    resident), further calls leave the free device memory unchanged."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    M, H, n_q = 2048, 2, 64
    q = seeded((1, n_q, H, 64), 931, "cuda", torch.float16)
    k8 = Q.q8kv_quantize(seeded((1, M, H, 64), 932, "cuda"))
    v8 = Q.q8kv_quantize(seeded((1, M, H, 64), 933, "cuda"))
    st = Q.State(1, H, n_q, q.device)
    assert _call_static(lib, q, k8, v8, 0, M, st, 256, M, False) == Q.Q8A_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        Q.attn_state_init(st)
        assert _call_static(lib, q, k8, v8, 0, M, st, 256, M, False) == Q.Q8A_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert_device_clean()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
