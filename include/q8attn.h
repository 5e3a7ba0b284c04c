/*
 * q8attn.h -- C ABI of libq8attn.so: causal FlashAttention prefill over a
 * Q8_0-quantised KV cache, computed chunk by chunk with a persistent
 * online-softmax state, for NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *   [ARCH]   "Core Architecture & The 4-Brick Pipeline", §5 "Brick 4:
 *            Barrier-Free FlashAttention & Dynamic Q8_0 KV Cache", part 2
 *            "Dynamic Q8_0 KV Cache Compression".
 *   [STREAM] "Out-of-Core Flash Streaming & Speculative Decode (1M Context)",
 *            §2 (the double-buffered streaming of KV chunks), §3 "Chunked
 *            FlashAttention: Exact Mathematical Derivation" and §4 "Mode A vs.
 *            Mode B Execution Modes".
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or synchronises on its own (q8a_device_status, which
 *     says so, synchronises its stream; the first chunk-step call of the process
 *     pins one page of the library's own memory for q8a_status); every compute
 *     call is one or more asynchronous kernel launches on `stream` (a
 *     cudaStream_t passed as void*; NULL is the legacy default stream).
 *   - Return value: Q8A_OK (0) or a negative Q8A_ERR_* code.  Arguments are
 *     validated on the host before any CUDA call, so argument errors are
 *     reported without touching the device.  q8a_last_error() returns a
 *     thread-local message for the last failing call of the calling thread.
 *   - Sizes of zero are allowed and make the call a no-op; negative sizes are
 *     Q8A_ERR_INVALID_ARG.
 *   - head_dim D is 64 (two Q8_0 blocks per head row) for every call, and
 *     128 (four blocks) for q8kv_quantize, attn_state_init, attn_chunk_step,
 *     attn_chunk_step_gqa, attn_chunk_step_split (and its allocation-free
 *     form), attn_finalize, attn_prefill_pipelined and the captured prefill.
 *   - Layouts (all row-major, contiguous):
 *       Q, out    fp16  [B][n_q][H][D]           token-major
 *       x (K, V)  fp32  [B][n_tokens][H][D]      token-major
 *       K8, V8    Q8_0  [B][H] planes of n_tokens rows of D/32*34 bytes (68 at
 *                 D = 64, 136 at D = 128); plane (b, h) starts
 *                 `plane_stride_bytes * (b*H + h)` bytes after the base.  A row
 *                 is block 0 (channels 0..31), block 1 (32..63), ...; each
 *                 34-byte block is an fp16 scale d (little-endian) followed by
 *                 32 int8 codes.
 *       m, l      fp32  [B][H][n_q]
 *       O         fp32  [B][H][n_q][D]
 *   - Device wait budget: every wait inside a kernel is bounded (default 2 s,
 *     see q8a_set_wait_timeout_ns).  A wait that runs out stops the kernel's
 *     blocks cleanly and records Q8A_ERR_TIMEOUT in a per-device status word
 *     that q8a_device_status() reads; the CUDA context stays usable.
 */
#ifndef Q8ATTN_H_
#define Q8ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Raised whenever an entry point is added or its contract changes.  2: the
 * split, allocation-free split, pipelined and grouped-query calls.  3: the
 * pipelined call streams K and V through two chunk slots (kv_slots).  4:
 * head_dim 128 and q8a_plane_stride_bytes_for.  5: the captured prefill
 * (q8a_prefill_graph_*).  6: attn_prefill_pipelined and the split calls at
 * head_dim 128, q8a_prefill_slot_floats_for, q8a_split_workspace_floats_for and
 * attn_chunk_step_split_gqa.  7: q8a_status. */
#define Q8A_ABI_VERSION 7u

enum {
  Q8A_OK = 0,
  Q8A_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad stride or shape */
  Q8A_ERR_MISALIGNED = -2,  /* a pointer or stride lacks the required alignment */
  Q8A_ERR_UNSUPPORTED = -3, /* a head_dim the call does not support, or a size beyond int32 tiles */
  Q8A_ERR_CUDA = -4,        /* a CUDA runtime or driver call failed */
  Q8A_ERR_TIMEOUT = -5      /* a device-side wait ran out of budget */
};

#define Q8A_ROW_BYTES 68 /* one 64-channel head row: two 34-byte Q8_0 blocks */
#define Q8A_HEAD_DIM 64  /* the head dimension every call supports */

/* ABI version of the loaded library (Q8A_ABI_VERSION). */
uint32_t q8a_abi_version(void);

/* Thread-local description of the last error returned to this thread ("" if none). */
const char *q8a_last_error(void);

/* Smallest valid plane stride for n_tokens rows: n_tokens*68 rounded up to 16. */
int64_t q8a_plane_stride_bytes(int64_t n_tokens);

/* The same for head_dim 64 or 128: n_tokens * head_dim/32*34 rounded up to 16;
 * -1 for a negative n_tokens or another head_dim. */
int64_t q8a_plane_stride_bytes_for(int64_t n_tokens, int32_t head_dim);

/*
 * q8kv_quantize -- dynamic Q8_0 quantisation of one K or V tensor [ARCH].
 *
 * For every (b, t, h) row of x and each of its two 32-channel blocks:
 *   amax = max |x| over the block;  d = fp16_rn(amax / 127)  (IEEE fp32 divide);
 *   q_i  = round_half_away_from_zero(x_i / d)  (IEEE fp32 divide by the stored
 *          fp16 d), clamped to [-127, 127];  d == 0 gives all-zero codes.
 * The result is bit-exact and deterministic.  Inputs must be finite with
 * |x| <= 65504*127 (larger values are not detected).
 *
 *   x                  fp32 [B][n_tokens][H][D], 16-byte aligned.
 *   q8_out             Q8_0 planes [B][H], row t of plane (b,h) at byte
 *                      plane_stride*(b*H+h) + (D/32*34)*t; 16-byte aligned.
 *   out_plane_stride_bytes  >= n_tokens*D/32*34 and a multiple of 16.
 * Errors: Q8A_ERR_INVALID_ARG, Q8A_ERR_MISALIGNED, Q8A_ERR_UNSUPPORTED, Q8A_ERR_CUDA.
 */
int q8kv_quantize(const float *x, void *q8_out, int64_t batch, int64_t n_tokens,
                  int32_t heads, int32_t head_dim, int64_t out_plane_stride_bytes,
                  void *stream);

/*
 * attn_state_init -- the persistent per-row state before the first chunk
 * [STREAM §3]: m_i = -inf, l_i = 0, O_i = 0 for every (b, h, row).
 *   m, l  fp32 [B][H][n_q] (4-byte aligned);  o fp32 [B][H][n_q][D] (16-byte aligned).
 */
int attn_state_init(float *m, float *l, float *o, int64_t batch, int32_t heads,
                    int64_t n_q, int32_t head_dim, void *stream);

/*
 * attn_chunk_step -- fold one KV chunk into the state [STREAM §3, steps 1-6]:
 *   S_ij = scale * Q_i . K_j;   m~_i = max_j S_ij;   m'_i = max(m_i, m~_i);
 *   alpha = e^(m_i - m'_i);     beta_ij = e^(S_ij - m'_i);
 *   l'_i = alpha*l_i + sum_j beta_ij;   O'_i = alpha*O_i + sum_j beta_ij V_j.
 * The kernels take m' as a reference that moves to the new max only when that
 * exceeds m by more than 8 ln 2 (otherwise m' = m and alpha = 1): any reference
 * gives the same O / l, and this one keeps O's rescaling rare.  So after a call
 * a row that has seen a key holds l = sum e^(S - m) and O = sum e^(S - m) V
 * over the keys folded so far, with max S - 8 ln 2 <= m <= max S.
 * K and V are the dequantised Q8_0 values d*q.  Only visible keys take part:
 * query row r has position q_pos0 + r, chunk key j has position kv_start + j,
 * and with `causal` the key is visible iff its position <= the query's (the
 * triangular mask of [STREAM §4] Mode A).  A row that sees no key of this
 * chunk keeps its state unchanged; key tiles above the diagonal are skipped
 * ([ARCH] causal skipping).  Chunks may be folded in any order; the result is
 * the same up to floating-point rounding.
 *
 *   q            fp16 [B][n_q][H][D], 16-byte aligned (rows of this call's queries).
 *   k_q8, v_q8   key 0 of this chunk in plane (b=0, h=0); plane (b,h) starts
 *                kv_plane_stride_bytes*(b*H+h) later; 16-byte aligned.
 *   kv_plane_stride_bytes  >= kv_len*D/32*34 and a multiple of 16.  (A slice of
 *                a whole-sequence Q8_0 buffer uses that buffer's stride and a
 *                pointer advanced by kv_start*D/32*34 bytes, which is 16-byte
 *                aligned when kv_start is a multiple of 4 at D = 64, of 2 at
 *                D = 128.)
 *   kv_start     absolute position of the chunk's first key (>= 0).
 *   kv_len       number of keys in the chunk (0 makes the call a no-op).
 *   m, l, o      the state, updated in place (layouts above; o 16-byte aligned).
 *   scale        logit scale (1/sqrt(64) = 0.125 for the standard model); > 0.
 *   causal       nonzero for the causal mask, 0 for full (rectangular) attention.
 * Numerics: Q is fp16; each dequantised key and value d*q is split exactly
 * into an fp16 high part and an fp16 residual, so Q.K and P.V are formed from
 * exact operands on the tensor cores with fp32 accumulation; the weights
 * P = e^(S - m) (at most 2^8) are rounded to fp16 once, and l takes each key
 * tile's largest weight as rounded (so a row dominated by one key divides by
 * exactly that key's weight); m, l and O stay fp32 in the state.
 * At D = 128 a CTA folds one 128-row query tile with its two softmax pipelines
 * taking alternate 64-key tiles and merges their states at the end (the same
 * recurrence), so results match D = 64's numerics.
 * Errors: Q8A_ERR_INVALID_ARG, Q8A_ERR_MISALIGNED, Q8A_ERR_UNSUPPORTED, Q8A_ERR_CUDA.
 */
int attn_chunk_step(const void *q, int64_t q_pos0, const void *k_q8, const void *v_q8,
                    int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len,
                    float *m, float *l, float *o, int64_t batch, int32_t heads,
                    int64_t n_q, int32_t head_dim, float scale, int32_t causal,
                    void *stream);

/*
 * attn_chunk_step_gqa -- attn_chunk_step for grouped-query attention: `heads`
 * query heads share `kv_heads` K/V heads, query head h reading K/V head
 * h / (heads / kv_heads) (so kv_heads = heads is attn_chunk_step and
 * kv_heads = 1 is multi-query attention).  Grouping is not on the source pages;
 * it is the standard layout of models whose KV cache has fewer heads than the
 * queries, and it shrinks the Q8_0 cache by heads / kv_heads.  Arguments as for
 * attn_chunk_step, except that k_q8 and v_q8 hold batch * kv_heads planes
 * (plane (b, g) starts kv_plane_stride_bytes*(b*kv_heads+g) later) while q and
 * the state keep `heads` heads.
 * Errors: as attn_chunk_step; Q8A_ERR_INVALID_ARG also when kv_heads <= 0 or
 * heads is not a multiple of kv_heads.
 */
int attn_chunk_step_gqa(const void *q, int64_t q_pos0, const void *k_q8, const void *v_q8,
                        int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len,
                        float *m, float *l, float *o, int64_t batch, int32_t heads,
                        int32_t kv_heads, int64_t n_q, int32_t head_dim, float scale,
                        int32_t causal, void *stream);

/*
 * attn_chunk_step_split -- the same update as attn_chunk_step for query rows
 * that are few against a long chunk, such as Mode B speculative burst
 * verification ([STREAM §4]: K = 64 candidate queries against the whole
 * context, rectangular full-context mask, bound by reading the KV cache once).
 * The chunk's keys are cut into ranges of split_keys keys that are folded in
 * parallel, each into an empty partial state (m_s, l_s, O_s) in `workspace`;
 * a second kernel then folds the partials into (m, l, O) with the same
 * recurrence ([STREAM §3] steps 3-6, with a partial's max, weight sum and
 * weighted values in place of a chunk's).  The result equals attn_chunk_step's
 * up to floating-point rounding.  Arguments as for attn_chunk_step, plus:
 *   split_keys        keys per range, a positive multiple of 128.
 *   workspace         caller-owned fp32 scratch, 16-byte aligned, of at least
 *                     q8a_split_workspace_floats_for(batch, heads, n_q, kv_len,
 *                     split_keys, head_dim) floats; its contents are
 *                     overwritten.  Calls sharing one workspace must be ordered
 *                     on one stream.
 * At head_dim 128 each key range is folded by the paired kernel (one 128-row
 * query tile per CTA, its two pipelines on alternate 64-key tiles).
 *   workspace_floats  its size in floats.
 * Two kernel launches on `stream`.  Errors: as attn_chunk_step; Q8A_ERR_INVALID_ARG
 * also for a bad split_keys or a missing or too small workspace;
 * Q8A_ERR_UNSUPPORTED beyond 65,535 key ranges.
 * If q8a_device_status later reports Q8A_ERR_TIMEOUT for work that includes
 * this call, some key ranges may not have written their partial states and the
 * merge may have folded stale workspace contents into (m, l, O): the state is
 * then undefined and must be re-initialised with attn_state_init.
 */
int attn_chunk_step_split(const void *q, int64_t q_pos0, const void *k_q8, const void *v_q8,
                          int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len,
                          float *m, float *l, float *o, int64_t batch, int32_t heads,
                          int64_t n_q, int32_t head_dim, float scale, int32_t causal,
                          int64_t split_keys, float *workspace, int64_t workspace_floats,
                          void *stream);

/*
 * attn_chunk_step_split_gqa -- attn_chunk_step_split for grouped-query
 * attention: `heads` query heads on `kv_heads` K/V planes, query head h
 * reading plane h / (heads / kv_heads), as for attn_chunk_step_gqa (burst
 * verification of a model whose KV cache has fewer heads than its queries).
 * The workspace is sized by the query heads (q8a_split_workspace_floats_for
 * with `heads`).  Errors: as attn_chunk_step_split; Q8A_ERR_INVALID_ARG also
 * when kv_heads <= 0 or heads is not a multiple of kv_heads.
 */
int attn_chunk_step_split_gqa(const void *q, int64_t q_pos0, const void *k_q8, const void *v_q8,
                              int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len,
                              float *m, float *l, float *o, int64_t batch, int32_t heads,
                              int32_t kv_heads, int64_t n_q, int32_t head_dim, float scale,
                              int32_t causal, int64_t split_keys, float *workspace,
                              int64_t workspace_floats, void *stream);

/* Floats of workspace attn_chunk_step_split needs at head_dim 64:
 * ceil(kv_len / split_keys) * batch * heads * n_q * 66; -1 for invalid sizes. */
int64_t q8a_split_workspace_floats(int64_t batch, int32_t heads, int64_t n_q, int64_t kv_len,
                                   int64_t split_keys);

/* The same at head_dim 64 or 128: ceil(kv_len / split_keys) * batch * heads *
 * n_q * (head_dim + 2); -1 for invalid sizes or another head_dim. */
int64_t q8a_split_workspace_floats_for(int64_t batch, int32_t heads, int64_t n_q, int64_t kv_len,
                                       int64_t split_keys, int32_t head_dim);

/*
 * attn_chunk_step_split_static -- attn_chunk_step_split for callers that
 * cannot allocate device memory when they make the call: for instance code
 * embedded in a host framework that owns the device allocator and forbids
 * other allocations, or a latency-critical loop that cannot afford the
 * implicit device synchronisation of cudaMalloc / cudaFree.  It allocates
 * nothing: the partial states live in a fixed scratch array inside the
 * library: q8a_static_split_scratch_floats() floats = 32 MiB, held until the
 * process exits on each GPU where the library's kernels are loaded (with the
 * default lazy module loading, each GPU where one of them first runs; with
 * CUDA_MODULE_LOADING=EAGER, every visible GPU when the library is loaded).
 * The source pages have no counterpart: this is an interface convenience, not
 * part of the method.
 *   Arguments, result and errors: as attn_chunk_step_split without the
 *   workspace.  A call whose partial states would need more floats than the
 *   scratch holds (q8a_split_workspace_floats_for(...) > the scratch size) is
 *   rejected with Q8A_ERR_INVALID_ARG before anything is launched; use larger
 *   key ranges or attn_chunk_step_split with a workspace of your own.
 *   The first call on a device looks up the scratch's device address on that
 *   (current) device, and looks it up again when the device's context has
 *   changed since (after cudaDeviceReset).
 *   Every call on a device shares the one scratch array, which keeps the last
 *   call's contents; each call writes every partial it later reads, so no
 *   clearing is needed, but calls whose kernels can overlap on the GPU (other
 *   streams, other host threads) race on it: order them on one stream.  After
 *   a timeout the state is undefined, as for attn_chunk_step_split.
 */
int attn_chunk_step_split_static(const void *q, int64_t q_pos0, const void *k_q8,
                                 const void *v_q8, int64_t kv_plane_stride_bytes,
                                 int64_t kv_start, int64_t kv_len, float *m, float *l, float *o,
                                 int64_t batch, int32_t heads, int64_t n_q, int32_t head_dim,
                                 float scale, int32_t causal, int64_t split_keys, void *stream);

/* Size of the static scratch of attn_chunk_step_split_static, in floats. */
int64_t q8a_static_split_scratch_floats(void);

/*
 * attn_finalize -- out_i = O_i / l_i after the last chunk [STREAM §3]; a row
 * with l_i == 0 (it saw no key) gives 0.  out is fp16 (round to nearest even),
 * [B][n_q][H][D], 16-byte aligned; l 4-byte aligned; o 16-byte aligned.
 */
int attn_finalize(const float *l, const float *o, void *out, int64_t batch, int32_t heads,
                  int64_t n_q, int32_t head_dim, void *stream);

/*
 * attn_prefill_pipelined -- the whole prefill from host buffers ([STREAM §2]
 * "Double-Buffered Ping-Pong Execution": the next KV chunk is read into the
 * second of two fixed slots while the current one is folded into the state).
 * Q is copied to the device, then for each chunk of `chunk` tokens its fp32 K
 * and V are copied on `copy_stream` into slot c % 2 of `kv_slots` while
 * `compute_stream` quantises and folds the chunks before it (q8kv_quantize of
 * the slot into the Q8_0 planes, attn_chunk_step with kv_start = the chunk's
 * first token, q_pos0 = 0); a slot is refilled only after the quantise that
 * read it.  Q crosses after chunk 0's K and V, in blocks of up to 8,192 rows,
 * and chunk 0's step runs block by block as they arrive; with `causal` and a
 * chunk 0 of a multiple of 1,024 tokens (or the whole sequence), chunk 0's K,
 * V and query rows cross together in leads of 1,024 tokens, each quantised and
 * folded (its rows against chunk 0's keys up to them) as it arrives.  The fp32
 * inputs so take 2 x 2 x B x chunk x H x 64 floats of device
 * memory whatever the sequence length.  With `causal` no later chunk touches a
 * chunk's own query rows, so those rows are finalised right after its step and
 * copied back to the host on copy_stream while the device works on the later
 * chunks; without it, attn_finalize and one copy back run at the end.  The
 * result is bit-identical to quantising the whole K and V, folding the same
 * chunks in order and finalising.
 *   q_host, out_host   fp16 [B][n_tokens][H][D] in host memory (D = head_dim,
 *                      64 or 128);
 *   k_host, v_host     fp32 [B][n_tokens][H][D] in host memory;
 *                      page-locked host memory lets the copies overlap the
 *                      device work (pageable memory works, without overlap).
 *   q_dev, out_dev     device buffers of the layout and size of q_host;
 *   kv_slots           device fp32 scratch, 16-byte aligned, of at least
 *                      q8a_prefill_slot_floats_for(batch, heads, min(chunk,
 *                      n_tokens), head_dim) floats (kv_slot_floats);
 *                      overwritten;
 *   k8, v8, plane_stride_bytes    the Q8_0 planes of the whole sequence (as for
 *                      q8kv_quantize): the cache this prefill produces;
 *   m, l, o            the state (as for attn_state_init; initialised here);
 *   chunk              tokens per chunk, a positive multiple of 4;
 *   compute_stream, copy_stream   two streams (the same stream is allowed and
 *                      then nothing overlaps).  Everything is enqueued
 *                      asynchronously; the copy stream first waits for the
 *                      work already on the compute stream, so back-to-back calls
 *                      on the same buffers are ordered.  The output is on the
 *                      host once compute_stream has drained.
 * The call creates and releases five CUDA events; it allocates no memory.
 * Errors: Q8A_ERR_INVALID_ARG (sizes, null pointers, too small kv_slots),
 * Q8A_ERR_UNSUPPORTED (head_dim), Q8A_ERR_MISALIGNED, those of the calls above,
 * Q8A_ERR_CUDA (a copy, event or stream call failed).
 */
int attn_prefill_pipelined(const void *q_host, const float *k_host, const float *v_host,
                           void *out_host, int64_t batch, int32_t heads, int64_t n_tokens,
                           int32_t head_dim, int64_t chunk, float scale, int32_t causal,
                           void *q_dev, float *kv_slots, int64_t kv_slot_floats, void *k8,
                           void *v8, int64_t plane_stride_bytes, float *m, float *l, float *o,
                           void *out_dev, void *compute_stream, void *copy_stream);

/* Floats of kv_slots attn_prefill_pipelined needs at head_dim 64: 4 * batch *
 * chunk * heads * 64 (two slots of one chunk's fp32 K and V); -1 for invalid
 * sizes. */
int64_t q8a_prefill_slot_floats(int64_t batch, int32_t heads, int64_t chunk);

/* The same at head_dim 64 or 128: 4 * batch * chunk * heads * head_dim; -1 for
 * invalid sizes or another head_dim. */
int64_t q8a_prefill_slot_floats_for(int64_t batch, int32_t heads, int64_t chunk, int32_t head_dim);

/*
 * q8a_prefill_graph_create -- capture one whole device-resident prefill into a
 * CUDA graph, to be replayed with q8a_prefill_graph_launch ([STREAM §3]: the
 * chunks folded in order into the persistent state, then the final division).
 * The graph holds, in this order, the launches of: q8kv_quantize of k into k8
 * and of v into v8; attn_state_init of (m, l, o); attn_chunk_step for the
 * chunks [s0, s0 + chunk) of the sequence in order (kv_start = s0, q_pos0 = 0,
 * the chunk's slice of k8 and v8); attn_finalize of (l, o) into out.  A replay
 * computes exactly what those calls compute when made one by one on a stream,
 * with one host launch instead of one per kernel, so short prefills do not
 * leave the device waiting on the host between kernels.
 *   q, out        fp16 [B][n_tokens][H][D] device buffers, 16-byte aligned;
 *   k, v          fp32 [B][n_tokens][H][D] device buffers, 16-byte aligned;
 *   k8, v8        the Q8_0 planes written by the replay (layout and stride as
 *                 for q8kv_quantize);
 *   m, l, o       the state (layouts above);
 *   chunk         tokens per chunk: a positive multiple of 4 at D = 64, of 2
 *                 at D = 128;
 *   scale, causal as for attn_chunk_step;
 *   graph_out     receives the handle (NULL on failure).
 * The graph keeps the pointers and sizes it was created with (and the device
 * wait budget then in force): the caller keeps every buffer alive and in place
 * until q8a_prefill_graph_destroy, and may change their contents between
 * replays.  The launches are recorded on a private stream of the current
 * device; nothing runs during the call, and no device buffer is allocated.
 * Errors: Q8A_ERR_INVALID_ARG (null pointers, sizes, chunk, stride, scale),
 * Q8A_ERR_UNSUPPORTED (head_dim), Q8A_ERR_MISALIGNED and the other errors of
 * the captured calls, Q8A_ERR_CUDA (stream capture or instantiation failed).
 */
typedef struct q8a_prefill_graph q8a_prefill_graph;
int q8a_prefill_graph_create(const void *q, const float *k, const float *v, void *k8, void *v8,
                             int64_t plane_stride_bytes, float *m, float *l, float *o, void *out,
                             int64_t batch, int32_t heads, int64_t n_tokens, int32_t head_dim,
                             int64_t chunk, float scale, int32_t causal,
                             q8a_prefill_graph **graph_out);

/* Enqueue one replay of the captured prefill on `stream` (asynchronous).  The
 * current device must be the one the graph was created on.  Replays on one
 * stream run one after another.
 * Errors: Q8A_ERR_INVALID_ARG (null handle, other device), Q8A_ERR_CUDA. */
int q8a_prefill_graph_launch(q8a_prefill_graph *graph, void *stream);

/* Release the graph (NULL is allowed).  Replays already enqueued finish first
 * (CUDA keeps the graph's resources until they have run). */
int q8a_prefill_graph_destroy(q8a_prefill_graph *graph);

/*
 * q8a_device_status -- read (and optionally clear) the status word of the
 * current device: 0 when no device-side wait has run out since the last clear.
 * Synchronises `stream`.  Returns Q8A_OK, Q8A_ERR_TIMEOUT (when the word is
 * nonzero; *status_out then holds it: bit 0 set, bits 8..15 the role that gave
 * up first: 1 softmax, 2 dequantisation, 3 producer, 4 MMA issue, 5 final drain)
 * or Q8A_ERR_CUDA.  status_out may be NULL.
 */
int q8a_device_status(void *stream, uint32_t *status_out, int32_t clear);

/*
 * q8a_status -- the sync-free status check: whether any kernel of this library
 * has recorded a device-side wait that ran out since the last clear, read from
 * a host-mapped word without synchronising anything and without blocking.  A
 * block of a kernel whose wait ran out copies the device's status code (as
 * q8a_device_status reports it) into that word once its roles have stopped;
 * the store reaches the host while the kernel runs, so the answer covers the
 * library's kernels that have run so far on any stream, not work still queued.  The word is one page of the
 * library's own memory, registered with CUDA (cudaHostRegister, mapped and
 * portable) by the first chunk-step call of the process; nothing is allocated.
 * q8a_device_status with `clear` clears it too.
 *   stream   if not NULL, also asks cudaStreamQuery(stream), which does not
 *            block, and reports a CUDA error that the stream's work raised.
 * Returns Q8A_OK, Q8A_ERR_TIMEOUT (a wait ran out; q8a_last_error() names the
 * role), Q8A_ERR_CUDA (from cudaStreamQuery) or Q8A_ERR_UNSUPPORTED (the page
 * could not be registered: use q8a_device_status).
 */
int q8a_status(void *stream);

/* Budget of every device-side wait, in nanoseconds (default 2e9; minimum 1e6).
 * Applies to launches made after the call, from any thread. */
int q8a_set_wait_timeout_ns(uint64_t ns);

/*
 * q8a_test_inject -- test hook for the timeout path.  kind 1 makes the NEXT
 * attn_chunk_step launch skip the query-tile load (and its barrier arrival) in
 * its first block, so that block's waits run out, it stops cleanly and the
 * status word reports Q8A_ERR_TIMEOUT.  kind 0 clears a pending injection.
 * No memory fault, trap or unbounded wait is involved.
 */
int q8a_test_inject(int32_t kind);

#ifdef __cplusplus
}
#endif

#endif /* Q8ATTN_H_ */
