"""Causal softmax attention over dequantised KV, plain and chunked (oracle; test
infrastructure), all in fp64.

Sources:
  * "Out-of-Core Flash Streaming & Speculative Decode (1M Context)", §3
    "Chunked FlashAttention: Exact Mathematical Derivation": scores
    S_ij = Q_i . K_cj / sqrt(D); per chunk c the running maximum m_i, the
    running denominator l_i and the unnormalised output O_i are updated by
    steps 1-6 (tile max, new max, rescale factor alpha = e^(m_old - m_new),
    weights beta_j = e^(S_ij - m_new), l <- l*alpha + sum beta,
    O <- O*alpha + sum beta_j V_j), and the answer is O_i / l_i after the last
    chunk.  The page states the chunked result equals in-memory attention.
  * same page, §4 "Mode A vs. Mode B": prefill uses a triangular causal mask.

Readings where the page is silent (listed in the design notes):
  * initial state m = -inf, l = 0, O = 0; when the new maximum is still -inf
    (no visible key so far) alpha = 1 and every beta = 0, so no 0*inf or
    (-inf)-(-inf) is ever formed.
  * causal masking uses absolute positions: query row r sits at q_pos0 + r,
    key j of a chunk at kv_start + j; the key is visible iff its position is
    <= the query's.  A row with no visible key in a chunk keeps its state.
  * finalising a row whose l is 0 (it never saw a key) gives 0.

The plain definition (`attention_unchunked`, `attention_rows`) is what the
GPU path is compared with; the recurrence (`attention_chunked`, `state_init`,
`chunk_step`, `finalize`) restates the page's steps literally and is pinned to
the plain definition by the chunked == unchunked invariant.
"""

import numpy as np


def _visible(q_pos, k_pos, causal):
    """Boolean mask [n_q, n_k]: key visible to query."""
    if not causal:
        return np.ones((q_pos.size, k_pos.size), dtype=bool)
    return k_pos[None, :] <= q_pos[:, None]


def attention_unchunked(q, k, v, scale, causal=True, q_pos0=0, kv_pos0=0):
    """Plain softmax attention: out_i = sum_j softmax_j(scale * q_i . k_j) v_j
    over the keys visible to row i; fp64, two passes (max, then exp-sum).

    q: [n_q, D]; k, v: [n_k, D] (any float dtype, promoted to fp64).
    Returns fp64 [n_q, D]; a row that sees no key is 0.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    q_pos = q_pos0 + np.arange(q.shape[0])
    k_pos = kv_pos0 + np.arange(k.shape[0])
    vis = _visible(q_pos, k_pos, causal)
    s = (q @ k.T) * scale
    s = np.where(vis, s, -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    any_vis = np.isfinite(m)
    m = np.where(any_vis, m, 0.0)
    p = np.where(vis, np.exp(s - m), 0.0)
    den = np.sum(p, axis=1, keepdims=True)
    out = (p @ v) / np.where(any_vis, den, 1.0)
    return np.where(any_vis, out, 0.0)


def attention_rows(q_rows, k, v, rows, scale, causal=True, q_pos0=0, block=256, key_block=16384):
    """The plain definition for a subset of query rows (large problems).

    q_rows: [len(rows), D], the queries of `rows`; k, v: [n_k, D] with key j
    at position j; query row r sits at position q_pos0 + r.  Returns fp64
    [len(rows), D] in the order of `rows`.

    Same two passes as `attention_unchunked` -- first the row maximum over the
    visible keys, then sum_j e^(s_j - max) and sum_j e^(s_j - max) v_j -- with
    each pass walking the keys in blocks of `key_block` so that memory stays
    bounded for very long rows.  Only the order of the fp64 additions differs.
    """
    rows = np.asarray(rows, dtype=np.int64)
    q_rows = np.asarray(q_rows)
    out = np.zeros((rows.size, v.shape[1]), dtype=np.float64)
    order = np.argsort(rows, kind="stable")
    for s0 in range(0, rows.size, block):
        idx = order[s0:s0 + block]
        r = rows[idx]
        n_k = k.shape[0]
        if causal:
            n_k = int(min(n_k, q_pos0 + r.max() + 1))
        n_k = max(n_k, 0)
        qb = np.asarray(q_rows[idx], dtype=np.float64)
        q_pos = q_pos0 + r

        def scores(k0, k1):
            kb = np.asarray(k[k0:k1], dtype=np.float64)
            vis = _visible(q_pos, np.arange(k0, k1), causal)
            return np.where(vis, (qb @ kb.T) * scale, -np.inf), vis

        m = np.full(r.size, -np.inf)
        for k0 in range(0, n_k, key_block):            # pass 1: row maximum
            s, _ = scores(k0, min(n_k, k0 + key_block))
            m = np.maximum(m, np.max(s, axis=1))
        any_vis = np.isfinite(m)
        m = np.where(any_vis, m, 0.0)
        den = np.zeros(r.size)
        num = np.zeros((r.size, v.shape[1]))
        for k0 in range(0, n_k, key_block):            # pass 2: exp-sum and weighted sum
            k1 = min(n_k, k0 + key_block)
            s, vis = scores(k0, k1)
            p = np.where(vis, np.exp(s - m[:, None]), 0.0)
            den += np.sum(p, axis=1)
            num += p @ np.asarray(v[k0:k1], dtype=np.float64)
        o = num / np.where(any_vis, den, 1.0)[:, None]
        out[idx] = np.where(any_vis[:, None], o, 0.0)
    return out


# ---- the page's recurrence, step by step -----------------------------------

def state_init(n_q, d):
    """Initial persistent state: m = -inf, l = 0, O = 0 (fp64)."""
    return {"m": np.full(n_q, -np.inf), "l": np.zeros(n_q), "O": np.zeros((n_q, d))}


def chunk_step(state, q, k_c, v_c, kv_start, scale, causal=True, q_pos0=0):
    """Fold one KV chunk (keys at positions kv_start .. kv_start+n_c-1) into the
    state, following steps 1-6 of the chunked derivation.  Updates in place."""
    q = np.asarray(q, dtype=np.float64)
    k_c = np.asarray(k_c, dtype=np.float64)
    v_c = np.asarray(v_c, dtype=np.float64)
    m_old, l_old, o_old = state["m"], state["l"], state["O"]
    vis = _visible(q_pos0 + np.arange(q.shape[0]), kv_start + np.arange(k_c.shape[0]), causal)
    # 1. local tile scores
    s = np.where(vis, (q @ k_c.T) * scale, -np.inf)
    # 2. local tile maximum (-inf for a row with no visible key)
    m_tile = np.max(s, axis=1) if k_c.shape[0] else np.full(q.shape[0], -np.inf)
    # 3. updated global maximum
    m_new = np.maximum(m_old, m_tile)
    live = np.isfinite(m_new)
    m_safe = np.where(live, m_new, 0.0)
    # 4. rescaling factors (alpha = 1, beta = 0 while nothing is visible)
    alpha = np.where(live, np.exp(np.where(live, m_old - m_safe, 0.0)), 1.0)
    beta = np.where(vis & live[:, None], np.exp(s - m_safe[:, None]), 0.0)
    # 5. updated normaliser
    l_new = l_old * alpha + np.sum(beta, axis=1)
    # 6. updated unnormalised output
    o_new = o_old * alpha[:, None] + beta @ v_c
    state["m"], state["l"], state["O"] = m_new, l_new, o_new
    return state


def finalize(state):
    """Attention_i = O_i / l_i; a row with l == 0 gives 0."""
    l = state["l"]
    pos = l > 0
    return np.where(pos[:, None], state["O"] / np.where(pos, l, 1.0)[:, None], 0.0)


def attention_chunked(q, k, v, chunk, scale, causal=True, q_pos0=0, order=None):
    """Run the recurrence over KV chunks of `chunk` keys (key j at position j),
    in the given chunk order (default ascending), then finalise."""
    n_k = k.shape[0]
    starts = list(range(0, n_k, chunk))
    if order is not None:
        starts = [starts[i] for i in order]
    st = state_init(q.shape[0], v.shape[1])
    for s0 in starts:
        chunk_step(st, q, k[s0:s0 + chunk], v[s0:s0 + chunk], s0, scale, causal, q_pos0)
    return finalize(st)
