// pipeline.cu -- the whole prefill from host buffers, with the host-to-device
// copy of each KV chunk overlapped with the device work on the chunks before
// it.
//
// This is the GB300 form of the pages' out-of-core streaming ("Out-of-Core
// Flash Streaming & Speculative Decode (1M Context)", §2 "Double-Buffered
// Ping-Pong Execution": while the GPU folds chunk c into the persistent state,
// the next chunk is already being read into the second of two fixed slots).
// Here the source is pinned host memory instead of flash, the copies run on a
// copy stream into two device slots of one chunk's fp32 K and V each (so the
// fp32 inputs take device memory in proportion to the chunk, not the
// sequence), and each chunk's Q8_0 quantisation and chunk step wait on that
// chunk's copy through an event; a slot is refilled only after the quantise
// that read it.  Host code only: every step of the computation is one of the
// library's kernels.

#include <cstdio>

#include "../../include/q8attn.h"
#include "internal.h"

namespace {

constexpr const char* kFn = "attn_prefill_pipelined";

int cuda_err(cudaError_t e, const char* what) {
  char msg[256];
  std::snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorName(e));
  return q8a::set_error(Q8A_ERR_CUDA, kFn, msg);
}

}  // namespace

extern "C" {

int64_t q8a_prefill_slot_floats_for(int64_t batch, int32_t heads, int64_t chunk, int32_t head_dim) {
  if (batch < 0 || heads <= 0 || chunk <= 0 || (head_dim != 64 && head_dim != 128)) return -1;
  return 4 * batch * chunk * heads * head_dim;   // 2 slots x (K, V) x [B][chunk][H][D]
}

int64_t q8a_prefill_slot_floats(int64_t batch, int32_t heads, int64_t chunk) {
  return q8a_prefill_slot_floats_for(batch, heads, chunk, Q8A_HEAD_DIM);
}

int attn_prefill_pipelined(const void* q_host, const float* k_host, const float* v_host,
                           void* out_host, int64_t batch, int32_t heads, int64_t n_tokens,
                           int32_t head_dim, int64_t chunk, float scale, int32_t causal,
                           void* q_dev, float* kv_slots, int64_t kv_slot_floats, void* k8, void* v8,
                           int64_t plane_stride_bytes, float* m, float* l, float* o, void* out_dev,
                           void* compute_stream, void* copy_stream) {
  q8a::NvtxRange nvtx_range("attn_prefill_pipelined");
  if (head_dim != 64 && head_dim != 128)
    return q8a::set_error(Q8A_ERR_UNSUPPORTED, kFn, "head_dim must be 64 or 128");
  if (batch < 0 || heads <= 0 || n_tokens < 0 || chunk <= 0 || chunk % 4 != 0)
    return q8a::set_error(Q8A_ERR_INVALID_ARG, kFn,
                          "sizes must be >= 0, heads > 0 and chunk a positive multiple of 4");
  if (batch == 0 || n_tokens == 0) return Q8A_OK;
  if (!q_host || !k_host || !v_host || !out_host || !q_dev || !kv_slots || !k8 || !v8 || !m ||
      !l || !o || !out_dev)
    return q8a::set_error(Q8A_ERR_INVALID_ARG, kFn, "null pointer");
  // a chunk longer than the sequence only needs the sequence's tokens in a slot
  const int64_t slot_tokens = chunk < n_tokens ? chunk : n_tokens;
  if (kv_slot_floats < q8a_prefill_slot_floats_for(batch, heads, slot_tokens, head_dim))
    return q8a::set_error(Q8A_ERR_INVALID_ARG, kFn,
                          "kv_slots holds fewer than q8a_prefill_slot_floats_for(batch, heads, "
                          "min(chunk, n_tokens), head_dim) floats");
  if (reinterpret_cast<uintptr_t>(kv_slots) % 16 != 0)
    return q8a::set_error(Q8A_ERR_MISALIGNED, kFn, "kv_slots needs 16-byte alignment");
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t xs = static_cast<cudaStream_t>(copy_stream);
  const int64_t row_floats = static_cast<int64_t>(heads) * head_dim;   // one token, all heads
  const int64_t q8_row = head_dim / 32 * 34;                           // bytes of one Q8_0 head row
  // slot s holds K at kv_slots + 2*s*part and V at kv_slots + (2*s+1)*part, each
  // [B][slot_tokens][H][D] (a shorter last chunk keeps the per-sequence stride)
  const int64_t part = batch * slot_tokens * row_floats;

  // ev: a chunk's inputs are on the device (copy stream -> compute stream);
  // ev_q: a block of query rows is on the device (copy -> compute);
  // ev_fin: a row block of the output is final (compute stream -> copy stream);
  // ev_free[s]: slot s has been quantised and may be refilled (compute -> copy).
  cudaEvent_t ev = nullptr, ev_q = nullptr, ev_fin = nullptr, ev_free[2] = {nullptr, nullptr};
  cudaEvent_t* all[5] = {&ev, &ev_q, &ev_fin, &ev_free[0], &ev_free[1]};
  auto release = [&]() {
    for (cudaEvent_t* p : all)   // released once the recorded work is done
      if (*p) cudaEventDestroy(*p);
  };
  for (cudaEvent_t* p : all) {
    cudaError_t ce = cudaEventCreateWithFlags(p, cudaEventDisableTiming);
    if (ce != cudaSuccess) {
      release();
      return cuda_err(ce, "cudaEventCreateWithFlags");
    }
  }
  cudaError_t e = cudaSuccess;
  int rc = Q8A_OK;
  auto bail = [&](int code) {
    release();
    return code;
  };
  const size_t out_row_bytes = static_cast<size_t>(row_floats) * 2;   // one token, all heads, fp16
  // copy query rows [r0, r0 + n) of every sequence back to the host on `st`
  auto copy_out_rows = [&](int64_t r0, int64_t n, cudaStream_t st) -> cudaError_t {
    for (int64_t b = 0; b < batch; ++b) {
      const size_t off = static_cast<size_t>(b * n_tokens + r0) * out_row_bytes;
      cudaError_t ce = cudaMemcpyAsync(static_cast<uint8_t*>(out_host) + off,
                                       static_cast<const uint8_t*>(out_dev) + off,
                                       static_cast<size_t>(n) * out_row_bytes,
                                       cudaMemcpyDeviceToHost, st);
      if (ce != cudaSuccess) return ce;
    }
    return cudaSuccess;
  };
  // Earlier work on the compute stream may still read the device buffers that
  // the copies below overwrite: the copy stream starts after it.
  if ((e = cudaEventRecord(ev, cs)) != cudaSuccess) return bail(cuda_err(e, "cudaEventRecord"));
  if ((e = cudaStreamWaitEvent(xs, ev, 0)) != cudaSuccess) return bail(cuda_err(e, "cudaStreamWaitEvent"));
  if ((rc = attn_state_init(m, l, o, batch, heads, n_tokens, head_dim, cs)) != Q8A_OK) return bail(rc);
  // Q follows chunk 0's K and V on the copy stream in blocks of q_block rows
  // (a multiple of 256, two 128-row query tiles); chunk 0's step runs block by
  // block as the rows arrive, so only chunk 0's K and V and the first block of
  // Q cross the link before the device starts.
  const int64_t q_block = ((chunk < 8192 ? chunk : 8192) + 255) / 256 * 256;
  // leads of chunk 0 (causal): a multiple of 256 rows (two query tiles) whose
  // Q8_0 rows start 16-byte aligned at either head_dim
  constexpr int64_t kLead = 1024;
  const size_t q_row_bytes = static_cast<size_t>(row_floats) * 2;   // one token, all heads, fp16

  // With the causal mask (q_pos0 = 0) no later chunk touches the query rows of
  // chunk c, so they are final once its step has run: they are finalised then,
  // and copied back on the copy stream behind the next chunk's inputs, while
  // the device works on the chunks after it.
  int64_t prev_r0 = -1, prev_n = 0;   // row block finalised but not yet copied back
  int64_t c = 0;                      // chunk index; chunk c uses slot c % 2
  for (int64_t s0 = 0; s0 < n_tokens; s0 += chunk, ++c) {
    const int64_t n = (n_tokens - s0 < chunk) ? n_tokens - s0 : chunk;
    const int slot = static_cast<int>(c & 1);
    float* ks = kv_slots + 2 * slot * part;
    float* vs = ks + part;
    const size_t bytes = static_cast<size_t>(n * row_floats) * sizeof(float);
    const uint8_t* kc = static_cast<const uint8_t*>(k8) + s0 * q8_row;
    const uint8_t* vc = static_cast<const uint8_t*>(v8) + s0 * q8_row;
    if (c == 0 && causal && (n % kLead == 0 || n == n_tokens)) {
      // Chunk 0 with the mask: its K, V and query rows cross in leads of kLead
      // tokens, and as each lead arrives it is quantised and its rows are
      // folded with chunk 0's keys up to them (the later keys of the chunk are
      // masked for them), so the device starts after one lead instead of the
      // whole chunk.  The same key tiles in the same order as one chunk-0 step.
      for (int64_t j0 = 0; j0 < n; j0 += kLead) {
        const int64_t nj = (n - j0 < kLead) ? n - j0 : kLead;
        const size_t kv_bytes = static_cast<size_t>(nj * row_floats) * sizeof(float);
        for (int64_t b = 0; b < batch; ++b) {
          const int64_t src = (b * n_tokens + j0) * row_floats;
          const int64_t dst = (b * slot_tokens + j0) * row_floats;
          const size_t qoff = static_cast<size_t>(b * n_tokens + j0) * q_row_bytes;
          if ((e = cudaMemcpyAsync(ks + dst, k_host + src, kv_bytes, cudaMemcpyHostToDevice, xs)) != cudaSuccess ||
              (e = cudaMemcpyAsync(vs + dst, v_host + src, kv_bytes, cudaMemcpyHostToDevice, xs)) != cudaSuccess ||
              (e = cudaMemcpyAsync(static_cast<uint8_t*>(q_dev) + qoff, static_cast<const uint8_t*>(q_host) + qoff,
                                   static_cast<size_t>(nj) * q_row_bytes, cudaMemcpyHostToDevice, xs)) !=
                  cudaSuccess)
            return bail(cuda_err(e, "copy of a lead of chunk 0"));
        }
        if ((e = cudaEventRecord(ev, xs)) != cudaSuccess || (e = cudaStreamWaitEvent(cs, ev, 0)) != cudaSuccess)
          return bail(cuda_err(e, "cudaEventRecord / cudaStreamWaitEvent"));
        for (int64_t b = 0; b < batch; ++b) {
          const int64_t off = (b * slot_tokens + j0) * row_floats;
          uint8_t* kq = static_cast<uint8_t*>(k8) + b * heads * plane_stride_bytes + j0 * q8_row;
          uint8_t* vq = static_cast<uint8_t*>(v8) + b * heads * plane_stride_bytes + j0 * q8_row;
          if ((rc = q8kv_quantize(ks + off, kq, 1, nj, heads, head_dim, plane_stride_bytes, cs)) != Q8A_OK ||
              (rc = q8kv_quantize(vs + off, vq, 1, nj, heads, head_dim, plane_stride_bytes, cs)) != Q8A_OK)
            return bail(rc);
        }
        if ((rc = q8a::chunk_step_tiles(q_dev, 0, kc, vc, plane_stride_bytes, 0, j0 + nj, m, l, o, batch, heads,
                                        n_tokens, head_dim, scale, causal, j0 / 128, (j0 + nj + 127) / 128,
                                        true, cs)) != Q8A_OK)
          return bail(rc);
      }
      if ((e = cudaEventRecord(ev_free[slot], cs)) != cudaSuccess) return bail(cuda_err(e, "cudaEventRecord"));
      // the rows after chunk 0 in blocks, each folded with the whole chunk as it arrives
      for (int64_t r0 = n; r0 < n_tokens; r0 += q_block) {
        const int64_t nr = (n_tokens - r0 < q_block) ? n_tokens - r0 : q_block;
        for (int64_t b = 0; b < batch; ++b) {
          const size_t off = static_cast<size_t>(b * n_tokens + r0) * q_row_bytes;
          if ((e = cudaMemcpyAsync(static_cast<uint8_t*>(q_dev) + off, static_cast<const uint8_t*>(q_host) + off,
                                   static_cast<size_t>(nr) * q_row_bytes, cudaMemcpyHostToDevice, xs)) !=
              cudaSuccess)
            return bail(cuda_err(e, "copy of a block of Q"));
        }
        if ((e = cudaEventRecord(ev_q, xs)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(cs, ev_q, 0)) != cudaSuccess)
          return bail(cuda_err(e, "cudaEventRecord / cudaStreamWaitEvent"));
        if ((rc = q8a::chunk_step_tiles(q_dev, 0, kc, vc, plane_stride_bytes, s0, n, m, l, o, batch, heads,
                                        n_tokens, head_dim, scale, causal, r0 / 128, (r0 + nr + 127) / 128,
                                        true, cs)) != Q8A_OK)
          return bail(rc);
      }
      if ((e = q8a::launch_finalize_rows(l, o, out_dev, batch, heads, n_tokens, head_dim, s0, n, cs)) !=
          cudaSuccess)
        return bail(cuda_err(e, "finalize of a row block"));
      if ((e = cudaEventRecord(ev_fin, cs)) != cudaSuccess) return bail(cuda_err(e, "cudaEventRecord"));
      prev_r0 = s0;
      prev_n = n;
      continue;
    }
    // the slot's previous chunk (c - 2) must have been quantised before it is refilled
    if (c >= 2 && (e = cudaStreamWaitEvent(xs, ev_free[slot], 0)) != cudaSuccess)
      return bail(cuda_err(e, "cudaStreamWaitEvent"));
    for (int64_t b = 0; b < batch; ++b) {
      const int64_t src = (b * n_tokens + s0) * row_floats;
      const int64_t dst = b * slot_tokens * row_floats;
      if ((e = cudaMemcpyAsync(ks + dst, k_host + src, bytes, cudaMemcpyHostToDevice, xs)) != cudaSuccess ||
          (e = cudaMemcpyAsync(vs + dst, v_host + src, bytes, cudaMemcpyHostToDevice, xs)) != cudaSuccess)
        return bail(cuda_err(e, "copy of a K/V chunk"));
    }
    // the chunk (and, before it on the copy stream, Q after chunk 0) is on the device once ev fires
    if ((e = cudaEventRecord(ev, xs)) != cudaSuccess) return bail(cuda_err(e, "cudaEventRecord"));
    if (prev_r0 >= 0) {
      if ((e = cudaStreamWaitEvent(xs, ev_fin, 0)) != cudaSuccess ||
          (e = copy_out_rows(prev_r0, prev_n, xs)) != cudaSuccess)
        return bail(cuda_err(e, "copy of an output row block"));
      prev_r0 = -1;
    }
    if ((e = cudaStreamWaitEvent(cs, ev, 0)) != cudaSuccess) return bail(cuda_err(e, "cudaStreamWaitEvent"));
    for (int64_t b = 0; b < batch; ++b) {
      const int64_t off = b * slot_tokens * row_floats;
      uint8_t* kq = static_cast<uint8_t*>(k8) + b * heads * plane_stride_bytes + s0 * q8_row;
      uint8_t* vq = static_cast<uint8_t*>(v8) + b * heads * plane_stride_bytes + s0 * q8_row;
      if ((rc = q8kv_quantize(ks + off, kq, 1, n, heads, head_dim, plane_stride_bytes, cs)) != Q8A_OK ||
          (rc = q8kv_quantize(vs + off, vq, 1, n, heads, head_dim, plane_stride_bytes, cs)) != Q8A_OK)
        return bail(rc);
    }
    if ((e = cudaEventRecord(ev_free[slot], cs)) != cudaSuccess) return bail(cuda_err(e, "cudaEventRecord"));
    if (c == 0) {
      for (int64_t r0 = 0; r0 < n_tokens; r0 += q_block) {
        const int64_t nr = (n_tokens - r0 < q_block) ? n_tokens - r0 : q_block;
        for (int64_t b = 0; b < batch; ++b) {
          const size_t off = static_cast<size_t>(b * n_tokens + r0) * q_row_bytes;
          if ((e = cudaMemcpyAsync(static_cast<uint8_t*>(q_dev) + off,
                                   static_cast<const uint8_t*>(q_host) + off,
                                   static_cast<size_t>(nr) * q_row_bytes, cudaMemcpyHostToDevice, xs)) !=
              cudaSuccess)
            return bail(cuda_err(e, "copy of a block of Q"));
        }
        if ((e = cudaEventRecord(ev_q, xs)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(cs, ev_q, 0)) != cudaSuccess)
          return bail(cuda_err(e, "cudaEventRecord / cudaStreamWaitEvent"));
        if ((rc = q8a::chunk_step_tiles(q_dev, 0, kc, vc, plane_stride_bytes, s0, n, m, l, o, batch, heads,
                                        n_tokens, head_dim, scale, causal, r0 / 128, (r0 + nr + 127) / 128,
                                        true, cs)) != Q8A_OK)
          return bail(rc);
      }
    } else if ((rc = q8a::chunk_step_tiles(q_dev, 0, kc, vc, plane_stride_bytes, s0, n, m, l, o, batch, heads,
                                           n_tokens, head_dim, scale, causal, 0, (n_tokens + 127) / 128, true,
                                           cs)) != Q8A_OK) {
      return bail(rc);
    }
    if (causal) {
      if ((e = q8a::launch_finalize_rows(l, o, out_dev, batch, heads, n_tokens, head_dim, s0, n, cs)) !=
          cudaSuccess)
        return bail(cuda_err(e, "finalize of a row block"));
      if ((e = cudaEventRecord(ev_fin, cs)) != cudaSuccess) return bail(cuda_err(e, "cudaEventRecord"));
      prev_r0 = s0;
      prev_n = n;
    }
  }
  if (causal) {
    // the last row block, then the compute stream waits for every copy back
    if ((e = cudaStreamWaitEvent(xs, ev_fin, 0)) != cudaSuccess ||
        (e = copy_out_rows(prev_r0, prev_n, xs)) != cudaSuccess)
      return bail(cuda_err(e, "copy of an output row block"));
    if ((e = cudaEventRecord(ev, xs)) != cudaSuccess) return bail(cuda_err(e, "cudaEventRecord"));
    if ((e = cudaStreamWaitEvent(cs, ev, 0)) != cudaSuccess) return bail(cuda_err(e, "cudaStreamWaitEvent"));
    return bail(Q8A_OK);
  }
  // without the mask: the copy stream's last work (the slot copies) is done
  // before the compute stream's quantise of them, so nothing else to wait for
  if ((rc = attn_finalize(l, o, out_dev, batch, heads, n_tokens, head_dim, cs)) != Q8A_OK) return bail(rc);
  if ((e = copy_out_rows(0, n_tokens, cs)) != cudaSuccess) return bail(cuda_err(e, "copy of the output"));
  return bail(Q8A_OK);
}

}  // extern "C"
