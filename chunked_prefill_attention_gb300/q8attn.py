"""Python binding of libq8attn.so (ctypes).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors; their device pointers
and the current torch stream are handed to the C ABI declared in
include/q8attn.h.  There is no CPU fallback: if the library is missing or fails
to load, every call raises.
"""

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# Q8ATTN_LIBRARY selects another in-tree build of the same library (the
# sanitizer build the host-code tests load); it is never a fallback.
LIB_PATH = os.environ.get("Q8ATTN_LIBRARY") or os.path.join(_HERE, "libq8attn.so")

Q8A_OK = 0
Q8A_ERR_INVALID_ARG = -1
Q8A_ERR_MISALIGNED = -2
Q8A_ERR_UNSUPPORTED = -3
Q8A_ERR_CUDA = -4
Q8A_ERR_TIMEOUT = -5
ROW_BYTES = 68
HEAD_DIM = 64

# name -> (restype, argtypes); mirrors include/q8attn.h
_I64, _I32, _U32, _U64, _P, _F = (ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64,
                                  ctypes.c_void_p, ctypes.c_float)
SIGNATURES = {
    "q8a_abi_version": (_U32, []),
    "q8a_last_error": (ctypes.c_char_p, []),
    "q8a_plane_stride_bytes": (_I64, [_I64]),
    "q8a_plane_stride_bytes_for": (_I64, [_I64, _I32]),
    "q8kv_quantize": (ctypes.c_int, [_P, _P, _I64, _I64, _I32, _I32, _I64, _P]),
    "attn_state_init": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _I64, _I32, _P]),
    "attn_chunk_step": (ctypes.c_int, [_P, _I64, _P, _P, _I64, _I64, _I64, _P, _P, _P, _I64, _I32,
                                       _I64, _I32, _F, _I32, _P]),
    "attn_chunk_step_gqa": (ctypes.c_int, [_P, _I64, _P, _P, _I64, _I64, _I64, _P, _P, _P, _I64,
                                           _I32, _I32, _I64, _I32, _F, _I32, _P]),
    "attn_chunk_step_split": (ctypes.c_int, [_P, _I64, _P, _P, _I64, _I64, _I64, _P, _P, _P, _I64,
                                             _I32, _I64, _I32, _F, _I32, _I64, _P, _I64, _P]),
    "attn_chunk_step_split_gqa": (ctypes.c_int, [_P, _I64, _P, _P, _I64, _I64, _I64, _P, _P, _P, _I64,
                                                 _I32, _I32, _I64, _I32, _F, _I32, _I64, _P, _I64, _P]),
    "q8a_split_workspace_floats": (_I64, [_I64, _I32, _I64, _I64, _I64]),
    "q8a_split_workspace_floats_for": (_I64, [_I64, _I32, _I64, _I64, _I64, _I32]),
    "attn_chunk_step_split_static": (ctypes.c_int, [_P, _I64, _P, _P, _I64, _I64, _I64, _P, _P, _P,
                                                    _I64, _I32, _I64, _I32, _F, _I32, _I64, _P]),
    "q8a_static_split_scratch_floats": (_I64, []),
    "attn_finalize": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _I64, _I32, _P]),
    "attn_prefill_pipelined": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I32, _I64, _I32, _I64, _F, _I32,
                                              _P, _P, _I64, _P, _P, _I64, _P, _P, _P, _P, _P, _P]),
    "q8a_prefill_slot_floats": (_I64, [_I64, _I32, _I64]),
    "q8a_prefill_slot_floats_for": (_I64, [_I64, _I32, _I64, _I32]),
    "q8a_prefill_graph_create": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I64, _I32,
                                                _I64, _I32, _I64, _F, _I32, ctypes.POINTER(_P)]),
    "q8a_prefill_graph_launch": (ctypes.c_int, [_P, _P]),
    "q8a_prefill_graph_destroy": (ctypes.c_int, [_P]),
    "q8a_device_status": (ctypes.c_int, [_P, ctypes.POINTER(_U32), _I32]),
    "q8a_status": (ctypes.c_int, [_P]),
    "q8a_set_wait_timeout_ns": (ctypes.c_int, [_U64]),
    "q8a_test_inject": (ctypes.c_int, [_I32]),
}

_lib = None


class Q8AttnError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"q8attn error {code}: {msg}")
        self.code = code


def load():
    """Load the in-tree shared library (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(rc):
    if rc != Q8A_OK:
        raise Q8AttnError(rc, load().q8a_last_error().decode())


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def row_bytes(head_dim):
    """Bytes of one Q8_0 head row: head_dim / 32 blocks of 34 bytes."""
    return head_dim // 32 * 34


def plane_stride(n_tokens, head_dim=HEAD_DIM):
    return int(load().q8a_plane_stride_bytes_for(n_tokens, head_dim))


def q8kv_quantize(x, out=None, stride=None):
    """x: fp32 CUDA [B, M, H, D] (D = 64 or 128) -> uint8 [B, H, stride] Q8_0
    planes (rows of D/32*34 B)."""
    B, M, H, D = x.shape
    if stride is None:
        stride = plane_stride(M, D)
    if out is None:
        out = torch.empty((B, H, stride), dtype=torch.uint8, device=x.device)
    _check(load().q8kv_quantize(_ptr(x), _ptr(out), B, M, H, D, stride, _stream(x)))
    return out


class State:
    """Persistent per-row online-softmax state (fp32): m, l [B, H, n_q]; O [B, H, n_q, D]."""

    def __init__(self, batch, heads, n_q, device, init=True, head_dim=HEAD_DIM):
        self.m = torch.empty((batch, heads, n_q), dtype=torch.float32, device=device)
        self.l = torch.empty((batch, heads, n_q), dtype=torch.float32, device=device)
        self.o = torch.empty((batch, heads, n_q, head_dim), dtype=torch.float32, device=device)
        if init:
            attn_state_init(self)

    @property
    def shape(self):
        return self.m.shape

    @property
    def head_dim(self):
        return self.o.shape[-1]


def attn_state_init(state):
    B, H, n = state.shape
    _check(load().attn_state_init(_ptr(state.m), _ptr(state.l), _ptr(state.o), B, H, n, state.head_dim,
                                  _stream(state.m)))
    return state


def attn_chunk_step(q, k8, v8, kv_start, kv_len, state, q_pos0=0, scale=None, causal=True,
                    stride=None, k_offset_bytes=0):
    """Fold KV keys [kv_start, kv_start + kv_len) into `state`.

    q: fp16 [B, n_q, H, D]; k8, v8: uint8 Q8_0 planes [B, H, stride] whose byte
    `k_offset_bytes` is the chunk's key 0 (so a whole-sequence buffer is passed
    with k_offset_bytes = kv_start * row_bytes(D))."""
    B, n_q, H, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stride is None:
        stride = k8.shape[-1]
    lib = load()
    kp = ctypes.c_void_p(k8.data_ptr() + k_offset_bytes)
    vp = ctypes.c_void_p(v8.data_ptr() + k_offset_bytes)
    _check(lib.attn_chunk_step(_ptr(q), q_pos0, kp, vp, stride, kv_start, kv_len, _ptr(state.m),
                               _ptr(state.l), _ptr(state.o), B, H, n_q, D, scale, int(bool(causal)),
                               _stream(q)))
    return state


def attn_chunk_step_gqa(q, k8, v8, kv_start, kv_len, state, q_pos0=0, scale=None, causal=True,
                        stride=None, k_offset_bytes=0):
    """attn_chunk_step for grouped-query attention: k8, v8 hold kv_heads =
    k8.shape[1] planes per batch entry and query head h reads plane
    h // (H // kv_heads)."""
    B, n_q, H, D = q.shape
    kv_heads = k8.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stride is None:
        stride = k8.shape[-1]
    lib = load()
    kp = ctypes.c_void_p(k8.data_ptr() + k_offset_bytes)
    vp = ctypes.c_void_p(v8.data_ptr() + k_offset_bytes)
    _check(lib.attn_chunk_step_gqa(_ptr(q), q_pos0, kp, vp, stride, kv_start, kv_len, _ptr(state.m),
                                   _ptr(state.l), _ptr(state.o), B, H, kv_heads, n_q, D, scale,
                                   int(bool(causal)), _stream(q)))
    return state


def split_workspace_floats(batch, heads, n_q, kv_len, split_keys, head_dim=HEAD_DIM):
    n = int(load().q8a_split_workspace_floats_for(batch, heads, n_q, kv_len, split_keys, head_dim))
    if n < 0:
        raise Q8AttnError(Q8A_ERR_INVALID_ARG, "invalid sizes for the split workspace")
    return n


def split_keys_for(bh, kv_len, sms, max_waves=8, min_keys=2048):
    """Key-range length for attn_chunk_step_split.  The split launch runs one
    CTA per (batch, head) and key range, one CTA per SM, so the range count n
    is chosen to make n * bh a whole number of waves: the fewest waves (up to
    max_waves) whose CTA count bh divides, keeping ranges of at least min_keys
    keys; the length is rounded up to whole 128-key tiles.  Without such a
    count, ranges of 8,192 keys."""
    if bh <= 0 or kv_len <= 0 or sms <= 0:
        raise ValueError("bh, kv_len and sms must be positive")
    for waves in range(1, max_waves + 1):
        if (waves * sms) % bh == 0:
            n = waves * sms // bh
            length = -(-(-(-kv_len // n)) // 128) * 128
            if length >= min_keys:
                return length
    return 8192


def attn_chunk_step_split(q, k8, v8, kv_start, kv_len, state, split_keys, workspace=None, q_pos0=0,
                          scale=None, causal=True, stride=None, k_offset_bytes=0):
    """attn_chunk_step with the chunk's keys folded in parallel ranges of
    `split_keys` keys and merged.  `workspace`: fp32 CUDA tensor of at least
    split_workspace_floats(...) elements (allocated here when None)."""
    B, n_q, H, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stride is None:
        stride = k8.shape[-1]
    need = split_workspace_floats(B, H, n_q, kv_len, split_keys, D)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.float32, device=q.device)
    lib = load()
    kp = ctypes.c_void_p(k8.data_ptr() + k_offset_bytes)
    vp = ctypes.c_void_p(v8.data_ptr() + k_offset_bytes)
    _check(lib.attn_chunk_step_split(_ptr(q), q_pos0, kp, vp, stride, kv_start, kv_len,
                                     _ptr(state.m), _ptr(state.l), _ptr(state.o), B, H, n_q, D,
                                     scale, int(bool(causal)), split_keys, _ptr(workspace),
                                     workspace.numel(), _stream(q)))
    return state


def attn_chunk_step_split_gqa(q, k8, v8, kv_start, kv_len, state, split_keys, workspace=None, q_pos0=0,
                              scale=None, causal=True, stride=None, k_offset_bytes=0):
    """attn_chunk_step_split with k8, v8 holding H_kv planes per sequence
    ([B, H_kv, stride]); query head h reads plane h // (H // H_kv)."""
    B, n_q, H, D = q.shape
    H_kv = k8.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stride is None:
        stride = k8.shape[-1]
    need = split_workspace_floats(B, H, n_q, kv_len, split_keys, D)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.float32, device=q.device)
    kp = ctypes.c_void_p(k8.data_ptr() + k_offset_bytes)
    vp = ctypes.c_void_p(v8.data_ptr() + k_offset_bytes)
    _check(load().attn_chunk_step_split_gqa(_ptr(q), q_pos0, kp, vp, stride, kv_start, kv_len,
                                            _ptr(state.m), _ptr(state.l), _ptr(state.o), B, H, H_kv, n_q, D,
                                            scale, int(bool(causal)), split_keys, _ptr(workspace),
                                            workspace.numel(), _stream(q)))
    return state


def attn_finalize(state, out=None):
    """O / l -> fp16 [B, n_q, H, D]."""
    B, H, n = state.shape
    if out is None:
        out = torch.empty((B, n, H, state.head_dim), dtype=torch.float16, device=state.m.device)
    _check(load().attn_finalize(_ptr(state.l), _ptr(state.o), _ptr(out), B, H, n, state.head_dim,
                                _stream(state.m)))
    return out


def prefill_attention(q, k, v, chunk, scale=None, causal=True, k8=None, v8=None, state=None, out=None):
    """The whole path: quantise K and V, initialise the state, fold every KV
    chunk of `chunk` keys in order, finalise.  Returns (out, k8, v8)."""
    B, M, H, D = q.shape
    k8 = q8kv_quantize(k, k8)
    v8 = q8kv_quantize(v, v8)
    if state is None:
        state = State(B, H, M, q.device, init=True, head_dim=D)
    else:
        attn_state_init(state)
    for s0 in range(0, M, chunk):
        n = min(chunk, M - s0)
        attn_chunk_step(q, k8, v8, s0, n, state, scale=scale, causal=causal,
                        k_offset_bytes=s0 * row_bytes(D))
    out = attn_finalize(state, out)
    return out, k8, v8


class PrefillGraph:
    """prefill_attention captured once into a CUDA graph
    (q8a_prefill_graph_create) and replayed with one launch per call.  The
    graph keeps the tensors' addresses: their contents may change between
    launches, so a new prefill of the same shape writes its Q, K and V into
    .q/.k/.v (the caller's tensors) and launches again."""

    def __init__(self, q, k, v, chunk, scale=None, causal=True):
        B, M, H, D = q.shape
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        self.q, self.k, self.v = q, k, v
        self.stride = plane_stride(M, D)
        self.k8 = torch.empty((B, H, self.stride), dtype=torch.uint8, device=q.device)
        self.v8 = torch.empty((B, H, self.stride), dtype=torch.uint8, device=q.device)
        self.state = State(B, H, M, q.device, init=False, head_dim=D)
        self.out = torch.empty((B, M, H, D), dtype=torch.float16, device=q.device)
        self._h = None
        h = ctypes.c_void_p()
        st = self.state
        with torch.cuda.device(q.device):
            _check(load().q8a_prefill_graph_create(
                _ptr(q), _ptr(k), _ptr(v), _ptr(self.k8), _ptr(self.v8), self.stride, _ptr(st.m),
                _ptr(st.l), _ptr(st.o), _ptr(self.out), B, H, M, D, chunk, scale, int(bool(causal)),
                ctypes.byref(h)))
        self._h = h

    def launch(self, stream=None):
        """Enqueue one replay on `stream` (default: the current stream); returns .out."""
        s = stream if stream is not None else torch.cuda.current_stream(self.out.device)
        with torch.cuda.device(self.out.device):
            _check(load().q8a_prefill_graph_launch(self._h, ctypes.c_void_p(s.cuda_stream)))
        return self.out

    def close(self):
        if self._h is not None and _lib is not None:
            _lib.q8a_prefill_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        self.close()


class PipelineBuffers:
    """Device buffers of attn_prefill_pipelined for one problem size and chunk:
    Q and the output (whole sequence), two chunk slots of fp32 K and V, the
    Q8_0 planes of the whole sequence and the state."""

    def __init__(self, batch, n_tokens, heads, device, chunk, head_dim=HEAD_DIM):
        shape = (batch, n_tokens, heads, head_dim)
        self.chunk = chunk
        self.q = torch.empty(shape, dtype=torch.float16, device=device)
        self.out = torch.empty(shape, dtype=torch.float16, device=device)
        n_slot = int(load().q8a_prefill_slot_floats_for(batch, heads, min(chunk, n_tokens), head_dim))
        if n_slot < 0:
            raise Q8AttnError(Q8A_ERR_INVALID_ARG, "invalid sizes for the prefill slots")
        self.kv_slots = torch.empty((n_slot,), dtype=torch.float32, device=device)
        self.stride = plane_stride(n_tokens, head_dim)
        self.k8 = torch.empty((batch, heads, self.stride), dtype=torch.uint8, device=device)
        self.v8 = torch.empty((batch, heads, self.stride), dtype=torch.uint8, device=device)
        self.state = State(batch, heads, n_tokens, device, init=False, head_dim=head_dim)
        self.copy_stream = torch.cuda.Stream(device=device)


def attn_prefill_pipelined(q_host, k_host, v_host, out_host, bufs, scale=None, causal=True):
    """The whole prefill from host tensors (page-locked for overlap) in chunks of
    bufs.chunk tokens: K/V chunk copies on bufs.copy_stream into two device
    slots overlap quantise + chunk step on the current stream; the output lands
    in out_host once the current stream drains."""
    B, M, H, D = q_host.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = bufs.state
    _check(load().attn_prefill_pipelined(
        _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(out_host), B, H, M, D, bufs.chunk, scale,
        int(bool(causal)), _ptr(bufs.q), _ptr(bufs.kv_slots), bufs.kv_slots.numel(), _ptr(bufs.k8),
        _ptr(bufs.v8), bufs.stride, _ptr(st.m), _ptr(st.l), _ptr(st.o), _ptr(bufs.out),
        _stream(bufs.q), ctypes.c_void_p(bufs.copy_stream.cuda_stream)))
    return out_host


def device_status(clear=True, stream=None):
    """(rc, status word) of the current device; synchronises the stream."""
    st = ctypes.c_uint32(0)
    s = ctypes.c_void_p(stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    rc = load().q8a_device_status(s, ctypes.byref(st), 1 if clear else 0)
    return rc, st.value


def status(stream=None):
    """Return code of the sync-free status check (q8a_status): Q8A_OK, or
    Q8A_ERR_TIMEOUT once a kernel has recorded a run-out wait."""
    s = ctypes.c_void_p(stream.cuda_stream if stream is not None else None)
    return load().q8a_status(s)


def set_wait_timeout_ns(ns):
    _check(load().q8a_set_wait_timeout_ns(int(ns)))


def test_inject(kind):
    _check(load().q8a_test_inject(int(kind)))
