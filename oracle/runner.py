"""Runs the CPU oracle over whole problems, in parallel worker processes.

Test infrastructure (used by tests/, smoke() and the benchmark's CPU-baseline
leg only): this calls only the oracle modules and numpy.  Worker pools use the
`spawn` start method so that no worker is forked from a process that already
holds a CUDA context.  Each task is one (batch, head) plane or one slice of a
tensor, so the per-task memory stays bounded.
"""

import atexit
import multiprocessing as mp
import os

import numpy as np

_POOL = None


_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def workers():
    return max(1, len(os.sched_getaffinity(0)))


def pool():
    """One BLAS thread per worker: the pool itself supplies the parallelism.
    The limit must be in the environment when a worker starts, because the
    worker imports numpy (and so sizes its BLAS thread pool) while it unpickles
    its task function, before any initializer runs."""
    global _POOL
    if _POOL is None:
        saved = {v: os.environ.get(v) for v in _BLAS_VARS}
        os.environ.update({v: "1" for v in _BLAS_VARS})
        try:
            _POOL = mp.get_context("spawn").Pool(workers())
            atexit.register(_close_pool)
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old
    return _POOL


def _close_pool():
    """Stop the workers before the interpreter tears down the pool's queues."""
    global _POOL
    if _POOL is not None:
        _POOL.terminate()
        _POOL.join()
        _POOL = None


def _quant_task(x):
    from oracle import q8_0
    return q8_0.quantize_kv(x)


def quantize_kv(x, parallel=True):
    """oracle.quantize_kv over fp32 [B, M, H, 64], split by token ranges."""
    from oracle import q8_0
    B, M, H, D = x.shape
    if not parallel or M * H * B < (1 << 16):
        return q8_0.quantize_kv(x)
    step = max(1, (1 << 22) // (H * D))     # ~16 MB of fp32 per task
    parts = []
    for b in range(B):
        tasks = [np.ascontiguousarray(x[b:b + 1, s:s + step]) for s in range(0, M, step)]
        parts.append(np.concatenate(pool().map(_quant_task, tasks), axis=2))
    return np.concatenate(parts, axis=0)


def _attn_task(args):
    q_rows, rows, k8, v8, scale, causal, q_pos0 = args
    from oracle import q8_0, attention
    k = q8_0.dequantize_kv(k8)
    v = q8_0.dequantize_kv(v8)
    return attention.attention_rows(q_rows, k, v, rows, scale, causal, q_pos0, block=256, key_block=8192)


def attention(q, k8, v8, scale, causal=True, rows=None, q_pos0=0):
    """Plain-definition attention on oracle-quantised KV, per (b, h) plane.

    q: fp16 numpy [B, n_q, H, 64]; k8, v8: uint8 [B, H_kv, M, 68] (oracle
    bytes) with H a multiple of H_kv.  Query head h attends over K/V head
    h // (H // H_kv): grouped-query attention, which the source pages do not
    describe; it is the standard definition (H_kv = H is ordinary multi-head
    attention, H_kv = 1 multi-query attention).
    rows: optional query-row indices (same for every plane).
    Returns fp64 [B, len(rows) or n_q, H, 64]."""
    B, n_q, H, D = q.shape
    H_kv = k8.shape[1]
    if H_kv <= 0 or H % H_kv != 0:
        raise ValueError(f"query heads {H} are not a multiple of K/V heads {H_kv}")
    group = H // H_kv
    rows = np.arange(n_q) if rows is None else np.asarray(rows, dtype=np.int64)
    tasks = []
    for b in range(B):
        for h in range(H):
            g = h // group
            kv_need = k8.shape[2] if not causal else min(k8.shape[2], q_pos0 + int(rows.max()) + 1)
            tasks.append((q[b, rows, h].astype(np.float64), rows, k8[b, g, :kv_need], v8[b, g, :kv_need],
                          scale, causal, q_pos0))
    res = pool().map(_attn_task, tasks, chunksize=1)
    out = np.zeros((B, rows.size, H, D), dtype=np.float64)
    for i, r in enumerate(res):
        out[i // H, :, i % H] = r
    return out
