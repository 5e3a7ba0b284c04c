"""The C-ABI library builds, loads and exports every symbol that
include/q8attn.h declares; argument validation answers before any CUDA call.
Runs without a GPU (no call here reaches a kernel launch)."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "q8attn.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_four_calls():
    names = _declared_functions()
    for n in ("q8kv_quantize", "attn_state_init", "attn_chunk_step", "attn_finalize"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from chunked_prefill_attention_gb300 import q8attn
    names = _declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"
        assert n in q8attn.SIGNATURES, f"binding lacks {n}"
    assert lib.q8a_abi_version() == 7


def test_plane_stride(lib):
    assert lib.q8a_plane_stride_bytes(512) == 512 * 68
    assert lib.q8a_plane_stride_bytes(1) == 80
    assert lib.q8a_plane_stride_bytes(3) == 208
    assert lib.q8a_plane_stride_bytes(0) == 0
    assert lib.q8a_plane_stride_bytes(-1) == -1


P = ctypes.c_void_p
A16 = P(0x100000)     # 16-byte aligned fake addresses: never dereferenced,
A4 = P(0x100004)      # validation fails before any launch


def _err(lib):
    return lib.q8a_last_error().decode()


def test_quantize_validation(lib):
    from chunked_prefill_attention_gb300 import q8attn as Q
    s = P(0)
    assert lib.q8kv_quantize(A16, A16, 1, 4, 2, 32, 272, s) == Q.Q8A_ERR_UNSUPPORTED
    assert "head_dim" in _err(lib)
    assert lib.q8kv_quantize(A16, A16, -1, 4, 2, 64, 272, s) == Q.Q8A_ERR_INVALID_ARG
    assert lib.q8kv_quantize(A16, A16, 1, -4, 2, 64, 272, s) == Q.Q8A_ERR_INVALID_ARG
    assert lib.q8kv_quantize(A16, A16, 1, 4, 0, 64, 272, s) == Q.Q8A_ERR_INVALID_ARG
    assert lib.q8kv_quantize(P(0), A16, 1, 4, 2, 64, 272, s) == Q.Q8A_ERR_INVALID_ARG
    assert lib.q8kv_quantize(A16, A16, 1, 4, 2, 64, 271, s) == Q.Q8A_ERR_INVALID_ARG   # < 4*68
    assert lib.q8kv_quantize(A16, A16, 1, 4, 2, 64, 280, s) == Q.Q8A_ERR_MISALIGNED   # % 16
    assert lib.q8kv_quantize(A4, A16, 1, 4, 2, 64, 288, s) == Q.Q8A_ERR_MISALIGNED
    # head_dim 128: 136-byte rows
    assert lib.q8kv_quantize(A16, A16, 1, 4, 2, 128, 543, s) == Q.Q8A_ERR_INVALID_ARG  # < 4*136
    assert lib.q8kv_quantize(A16, A16, 1, 4, 2, 128, 552, s) == Q.Q8A_ERR_MISALIGNED  # % 16
    assert lib.q8kv_quantize(A16, A16, 1, 4, 2, 96, 544, s) == Q.Q8A_ERR_UNSUPPORTED
    # empty problems are no-ops that never touch the device
    assert lib.q8kv_quantize(A16, A16, 0, 4, 2, 64, 288, s) == Q.Q8A_OK
    assert lib.q8kv_quantize(P(0), P(0), 1, 0, 2, 64, 0, s) == Q.Q8A_OK


def test_state_and_finalize_validation(lib):
    from chunked_prefill_attention_gb300 import q8attn as Q
    s = P(0)
    assert lib.attn_state_init(A16, A16, A16, 1, 2, 8, 96, s) == Q.Q8A_ERR_UNSUPPORTED
    assert lib.attn_finalize(A16, A16, A16, 1, 2, 8, 32, s) == Q.Q8A_ERR_UNSUPPORTED
    assert lib.attn_state_init(P(0), A16, A16, 1, 2, 8, 64, s) == Q.Q8A_ERR_INVALID_ARG
    assert lib.attn_state_init(A16, A16, A4, 1, 2, 8, 64, s) == Q.Q8A_ERR_MISALIGNED
    assert lib.attn_state_init(A16, A16, A16, 1, 2, -8, 64, s) == Q.Q8A_ERR_INVALID_ARG
    assert lib.attn_state_init(P(0), P(0), P(0), 1, 2, 0, 64, s) == Q.Q8A_OK
    assert lib.attn_finalize(A16, A16, A4, 1, 2, 8, 64, s) == Q.Q8A_ERR_MISALIGNED
    assert lib.attn_finalize(A16, P(0), A16, 1, 2, 8, 64, s) == Q.Q8A_ERR_INVALID_ARG
    assert lib.attn_finalize(P(0), P(0), P(0), 0, 2, 8, 64, s) == Q.Q8A_OK


def test_chunk_step_validation(lib):
    from chunked_prefill_attention_gb300 import q8attn as Q
    s = P(0)

    def call(q=A16, q_pos0=0, k=A16, v=A16, stride=8704, kv_start=0, kv_len=128, m=A16, l=A16,
             o=A16, batch=1, heads=2, n_q=128, hd=64, scale=0.125, causal=1):
        return lib.attn_chunk_step(q, q_pos0, k, v, stride, kv_start, kv_len, m, l, o, batch, heads,
                                   n_q, hd, scale, causal, s)

    assert call(hd=32) == Q.Q8A_ERR_UNSUPPORTED
    assert call(hd=128, stride=128 * 136 - 16) == Q.Q8A_ERR_INVALID_ARG   # 136-byte rows
    assert call(hd=128, kv_len=0, k=P(0), v=P(0)) == Q.Q8A_OK
    assert call(k=P(0)) == Q.Q8A_ERR_INVALID_ARG
    assert call(stride=8703) == Q.Q8A_ERR_INVALID_ARG
    assert call(stride=8712) == Q.Q8A_ERR_MISALIGNED
    assert call(k=P(0x100008)) == Q.Q8A_ERR_MISALIGNED
    assert call(o=A4) == Q.Q8A_ERR_MISALIGNED
    assert call(scale=0.0) == Q.Q8A_ERR_INVALID_ARG
    assert call(scale=float("nan")) == Q.Q8A_ERR_INVALID_ARG
    assert call(kv_start=-1) == Q.Q8A_ERR_INVALID_ARG
    assert call(q_pos0=-3) == Q.Q8A_ERR_INVALID_ARG
    assert call(kv_len=-1) == Q.Q8A_ERR_INVALID_ARG
    # no-ops: empty chunk, no queries, or every query before the chunk (causal)
    assert call(kv_len=0, k=P(0), v=P(0)) == Q.Q8A_OK
    assert call(n_q=0) == Q.Q8A_OK
    assert call(kv_start=128, n_q=128) == Q.Q8A_OK


def test_gqa_step_validation(lib):
    """attn_chunk_step_gqa rejects a head count that is not a multiple of the
    K/V head count before any CUDA call; otherwise it validates like
    attn_chunk_step."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    s = P(0)

    def call(heads=4, kv_heads=2, k=A16, kv_len=128, hd=64, n_q=128):
        return lib.attn_chunk_step_gqa(A16, 0, k, A16, 8704, 0, kv_len, A16, A16, A16, 1, heads,
                                       kv_heads, n_q, hd, 0.125, 1, s)

    assert call(kv_heads=0) == Q.Q8A_ERR_INVALID_ARG
    assert call(kv_heads=-2) == Q.Q8A_ERR_INVALID_ARG
    assert call(heads=6, kv_heads=4) == Q.Q8A_ERR_INVALID_ARG
    assert call(heads=2, kv_heads=4) == Q.Q8A_ERR_INVALID_ARG
    assert call(hd=32) == Q.Q8A_ERR_UNSUPPORTED
    assert call(k=P(0)) == Q.Q8A_ERR_INVALID_ARG
    assert call(kv_len=0, k=P(0)) == Q.Q8A_OK
    assert call(n_q=0) == Q.Q8A_OK


def test_split_step_validation(lib):
    """attn_chunk_step_split rejects bad range sizes and workspaces before it
    touches the device."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    s = P(0)
    need = lib.q8a_split_workspace_floats(1, 2, 128, 1000, 256)
    assert need == 4 * 1 * 2 * 128 * 66
    assert lib.q8a_split_workspace_floats(1, 2, 128, 1000, 0) == -1
    assert lib.q8a_split_workspace_floats(-1, 2, 128, 1000, 256) == -1

    def call(split=256, ws=A16, ws_n=need, kv_len=1000, stride=68000, causal=0):
        return lib.attn_chunk_step_split(A16, 0, A16, A16, stride, 0, kv_len, A16, A16, A16, 1, 2, 128,
                                         64, 0.125, causal, split, ws, ws_n, s)

    assert call(split=0) == Q.Q8A_ERR_INVALID_ARG
    assert call(split=100) == Q.Q8A_ERR_INVALID_ARG
    assert call(ws=P(0)) == Q.Q8A_ERR_INVALID_ARG
    assert call(ws_n=need - 1) == Q.Q8A_ERR_INVALID_ARG
    assert call(ws=P(0x100008)) == Q.Q8A_ERR_MISALIGNED
    assert call(split=128, kv_len=128 * 70000, stride=68 * 128 * 70000,
                ws_n=1 << 62) == Q.Q8A_ERR_UNSUPPORTED
    assert call(kv_len=0, ws=P(0), ws_n=0) == Q.Q8A_OK


def test_pipelined_prefill_validation(lib):
    """attn_prefill_pipelined checks sizes and pointers before any CUDA call."""
    from chunked_prefill_attention_gb300 import q8attn as Q

    def call(chunk=256, hd=64, q=A16, B=1, M=512, slots=A16, slot_floats=None):
        if slot_floats is None:
            slot_floats = lib.q8a_prefill_slot_floats(B, 2, min(chunk, M) if chunk > 0 else 1)
        return lib.attn_prefill_pipelined(q, A16, A16, A16, B, 2, M, hd, chunk, 0.125, 1, A16, slots,
                                          slot_floats, A16, A16, 34816, A16, A16, A16, A16, P(0), P(0))

    assert lib.q8a_prefill_slot_floats(2, 3, 100) == 4 * 2 * 100 * 3 * 64
    assert lib.q8a_prefill_slot_floats(1, 0, 100) == -1
    assert call(chunk=0) == Q.Q8A_ERR_INVALID_ARG
    assert call(chunk=6) == Q.Q8A_ERR_INVALID_ARG
    assert call(hd=32) == Q.Q8A_ERR_UNSUPPORTED
    # head_dim 128 needs twice the slot floats of head_dim 64
    assert call(hd=128) == Q.Q8A_ERR_INVALID_ARG and b"kv_slots" in lib.q8a_last_error()
    assert lib.q8a_prefill_slot_floats_for(2, 3, 100, 128) == 4 * 2 * 100 * 3 * 128
    assert lib.q8a_prefill_slot_floats_for(2, 3, 100, 64) == lib.q8a_prefill_slot_floats(2, 3, 100)
    assert lib.q8a_prefill_slot_floats_for(2, 3, 100, 96) == -1
    assert call(q=P(0)) == Q.Q8A_ERR_INVALID_ARG
    assert call(slots=P(0)) == Q.Q8A_ERR_INVALID_ARG
    # two slots of one 256-token chunk are needed, whatever the sequence length
    assert call(slot_floats=lib.q8a_prefill_slot_floats(1, 2, 256) - 1) == Q.Q8A_ERR_INVALID_ARG
    assert b"kv_slots" in lib.q8a_last_error()
    assert call(slots=P(0x100008)) == Q.Q8A_ERR_MISALIGNED
    assert call(B=0) == Q.Q8A_OK
    assert call(M=0) == Q.Q8A_OK


def test_prefill_graph_validation(lib):
    """q8a_prefill_graph_create checks its arguments before any CUDA call and
    leaves the handle NULL on failure; launch and destroy accept NULL safely."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    h = P(0x1234)

    def create(*, ptrs=A16, stride=16 * 68, B=1, H=2, M=16, D=64, chunk=8, scale=0.125, out=True):
        return lib.q8a_prefill_graph_create(ptrs, A16, A16, A16, A16, stride, A16, A16, A16, A16, B, H, M, D,
                                            chunk, scale, 1, ctypes.byref(h) if out else None)

    assert create(out=False) == Q.Q8A_ERR_INVALID_ARG
    assert "graph_out" in _err(lib)
    for kw in (dict(B=-1), dict(H=0), dict(M=-1), dict(chunk=0), dict(chunk=6), dict(ptrs=P(0)),
               dict(stride=15 * 68), dict(stride=16 * 68 + 4), dict(scale=0.0)):
        h.value = 0x1234
        assert create(**kw) == Q.Q8A_ERR_INVALID_ARG, kw
        assert not h.value, kw
    assert create(D=32) == Q.Q8A_ERR_UNSUPPORTED
    assert "head_dim" in _err(lib)
    assert create(D=128, chunk=3, stride=Q.plane_stride(16, 128)) == Q.Q8A_ERR_INVALID_ARG
    assert "chunk" in _err(lib)
    assert lib.q8a_prefill_graph_launch(None, None) == Q.Q8A_ERR_INVALID_ARG
    assert lib.q8a_prefill_graph_destroy(None) == Q.Q8A_OK


def test_runtime_knobs_validation(lib):
    from chunked_prefill_attention_gb300 import q8attn as Q
    assert lib.q8a_set_wait_timeout_ns(10) == Q.Q8A_ERR_INVALID_ARG
    assert lib.q8a_set_wait_timeout_ns(2_000_000_000) == Q.Q8A_OK
    assert lib.q8a_test_inject(7) == Q.Q8A_ERR_INVALID_ARG
    assert lib.q8a_test_inject(0) == Q.Q8A_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from chunked_prefill_attention_gb300 import q8attn
    monkeypatch.setattr(q8attn, "_lib", None)
    monkeypatch.setattr(q8attn, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        q8attn.load()


def test_head_dim_128_strides_and_split_sizes(lib):
    """head_dim 128 rows are four 34-byte blocks; the split calls size their
    partial states by the head dimension and check the workspace before any
    CUDA call."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    assert lib.q8a_plane_stride_bytes_for(100, 128) == (100 * 136 + 15) // 16 * 16
    assert lib.q8a_plane_stride_bytes_for(100, 64) == lib.q8a_plane_stride_bytes(100)
    assert lib.q8a_plane_stride_bytes_for(100, 96) == -1
    assert lib.q8a_plane_stride_bytes_for(-1, 128) == -1
    need = lib.q8a_split_workspace_floats_for(1, 2, 64, 512, 128, 128)
    assert need == 4 * 1 * 2 * 64 * 130
    assert lib.q8a_split_workspace_floats_for(1, 2, 64, 512, 128, 64) == lib.q8a_split_workspace_floats(1, 2, 64, 512, 128)
    assert lib.q8a_split_workspace_floats_for(1, 2, 64, 512, 128, 96) == -1
    s = P(0)
    rc = lib.attn_chunk_step_split(A16, 0, A16, A16, 136 * 512, 0, 512, A16, A16, A16, 1, 2, 64, 96,
                                   0.125, 0, 128, A16, 1 << 20, s)
    assert rc == Q.Q8A_ERR_UNSUPPORTED and b"head_dim" in lib.q8a_last_error()
    # enough for head_dim 64 but not for 128
    rc = lib.attn_chunk_step_split(A16, 0, A16, A16, 136 * 512, 0, 512, A16, A16, A16, 1, 2, 64, 128,
                                   0.125, 0, 128, A16, lib.q8a_split_workspace_floats(1, 2, 64, 512, 128), s)
    assert rc == Q.Q8A_ERR_INVALID_ARG and b"workspace" in lib.q8a_last_error()
    rc = lib.attn_chunk_step_split_static(A16, 0, A16, A16, 136 * 512, 0, 512, A16, A16, A16, 1, 2, 64,
                                          96, 0.125, 0, 128, s)
    assert rc == Q.Q8A_ERR_UNSUPPORTED

def test_status_before_any_launch_is_ok(lib):
    """The sync-free check makes no CUDA call without a stream: before any
    chunk step has run (nothing registered, nothing failed) it answers OK."""
    from chunked_prefill_attention_gb300 import q8attn as Q
    assert lib.q8a_status(None) == Q.Q8A_OK
