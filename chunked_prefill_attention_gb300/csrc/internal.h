// internal.h -- launchers shared by the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

namespace q8a {

// An NVTX range around one ABI call, so that Nsight tools show the library's
// calls on the timeline; without a tool attached it does nothing.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};


// Programmatic dependent launch of the library's kernels: while a PdlScope is
// alive on the calling thread (the captured prefill sets one during stream
// capture), every kernel is launched with programmatic stream serialization,
// so the device may schedule it while its predecessor's last CTAs run; each
// kernel waits for the predecessor's completion before touching memory.
bool pdl_enabled();
struct PdlScope {
  PdlScope();
  ~PdlScope();
  PdlScope(const PdlScope&) = delete;
  PdlScope& operator=(const PdlScope&) = delete;
  bool prev;
};

// kernel<<<grid, block, smem, stream>>>(args...), with programmatic stream
// serialization when pdl_enabled().
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

constexpr int kHeadDim = 64;
constexpr int kRowBytes = 68;  // one head row: two 34-byte Q8_0 blocks

// q8kv_quantize: fp32 [B][M][H][D] -> Q8_0 planes [B][H] of D/32*34-byte rows
// (D = head_dim, 64 or 128).
cudaError_t launch_quantize(const float* x, uint8_t* out, int64_t batch, int64_t n_tokens,
                            int32_t heads, int32_t head_dim, int64_t plane_stride,
                            cudaStream_t stream);

// attn_state_init over `rows` = B*H*n_q state rows of head_dim O channels.
cudaError_t launch_state_init(float* m, float* l, float* o, int64_t rows, int32_t head_dim,
                              cudaStream_t stream);

// attn_finalize: fp32 O, l -> fp16 out [B][n_q][H][D].
cudaError_t launch_finalize(const float* l, const float* o, void* out, int64_t batch,
                            int32_t heads, int64_t n_q, int32_t head_dim, cudaStream_t stream);
// The same for query rows row0 .. row0+n_rows-1 of every (b, h) plane only.
cudaError_t launch_finalize_rows(const float* l, const float* o, void* out, int64_t batch,
                                 int32_t heads, int64_t n_q, int32_t head_dim, int64_t row0,
                                 int64_t n_rows, cudaStream_t stream);

// Arguments of one chunk-step launch (everything but the Q tensor map).
struct ChunkArgs {
  const uint8_t* q;       // Q fp16 [B][n_q][H][D] (the head_dim 128 kernel reads rows directly)
  const uint8_t* k8;      // chunk key 0 of plane (0,0)
  const uint8_t* v8;
  float* m;
  float* l;
  float* o;
  int64_t plane_stride;   // bytes between (b,h) planes of k8 / v8
  int64_t q_pos0;         // position of query row 0
  int64_t kv_start;       // position of chunk key 0
  int64_t kv_len;         // keys in the chunk (> 0)
  int64_t n_q;            // query rows per (b,h)
  int32_t heads;
  int32_t kv_heads;       // K/V heads (planes per batch entry); heads is a multiple of it
  int32_t bh;             // batch * heads
  int32_t tile0;          // first 128-row query tile launched
  int32_t n_qtiles;       // 128-row query tiles launched per (b,h), from tile0 on
  float scale;            // logit scale
  float scale_log2;       // scale * log2(e)
  int32_t causal;
  int32_t inject;         // test hook: 1 = first block skips its query-tile load
  int32_t head_dim;       // 64 or 128
  int32_t pair;           // 1: one query tile, no causal mask -- the CTA's two softmax
                          // pipelines share the rows and split the key tiles (even / odd)
  int32_t pack;           // grouped-query bursts (head_dim 64, no causal mask): a tile's
                          // rows are (query row, query head) pairs of the `pack` query
                          // heads that share one K/V plane, row = query row * pack +
                          // head in the group; bh then counts (batch, K/V head) units
                          // and n_qtiles the 128-row tiles of n_q * pack rows; 0 = off
  int32_t head_group;     // (b, h) units per group in the CTA order (1..8): as many as
                          // keep the group's K and V of the chunk within 16 MiB of L2
  int32_t l2_keep_kv;     // 1: Q and the running state go through L2 with the evict-first
                          // policy (whole 32-byte sectors), so that the chunk's Q8_0 rows,
                          // quantised just before the step, stay in L2 for every CTA
                          // that reads them (the pipelined prefill; head_dim 64)
  uint64_t timeout_ns;    // budget of every device-side wait
  uint32_t* host_status;  // device address of the host-mapped failure word, or null
  // Split form (split_keys > 0): block row y of the grid folds keys
  // [y*split_keys, min((y+1)*split_keys, kv_len)) of the chunk into an empty
  // partial state at part_m/part_l/part_o + y * (bh*n_q) rows; the partials
  // are merged into m/l/o by launch_split_merge.
  int64_t split_keys;
  int32_t n_splits;
  float* part_m;
  float* part_l;
  float* part_o;
};

// The tensor map must describe Q as fp16 {H*64, n_q, B} with a {64, 128, 1}
// box and 128-byte swizzle.
cudaError_t launch_chunk_step(const CUtensorMap& qmap, const ChunkArgs& args, cudaStream_t stream);

// The head_dim 128 chunk step: Q as fp16 {H*128, n_q, B} with a {64, 128, 1}
// box and 128-byte swizzle; n_qtiles counts 128-row query tiles (one per CTA);
// no split form.
cudaError_t launch_chunk_step_d128(const CUtensorMap& qmap, const ChunkArgs& args, cudaStream_t stream);

// attn_chunk_step for the 128-row query tiles [tile_begin, tile_end) only;
// l2_keep_kv sets ChunkArgs::l2_keep_kv (the chunk was quantised just before,
// and o is 32-byte aligned).
int chunk_step_tiles(const void* q, int64_t q_pos0, const void* k_q8, const void* v_q8,
                     int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len, float* m,
                     float* l, float* o, int64_t batch, int32_t heads, int64_t n_q, int32_t head_dim,
                     float scale, int32_t causal, int64_t tile_begin, int64_t tile_end,
                     bool l2_keep_kv, cudaStream_t stream);

// Device address of the host-mapped failure word that q8a_status reads (the
// first call registers the library's page for it), or null when the page could
// not be registered.
uint32_t* host_status_word();

// Record `msg` as the calling thread's last error (q8a_last_error) and return code.
int set_error(int code, const char* fn, const char* msg);
// Clear the calling thread's last error and return Q8A_OK (a call that succeeded).
int clear_error();

// A launcher that refuses a launch configuration describes why here (thread
// local; "" when the last refusal had no note).
const char* launch_note();
void set_launch_note(const char* fmt, ...);

// Merge the n_splits partial states of a split chunk step into (m, l, o).
cudaError_t launch_split_merge(const ChunkArgs& args, cudaStream_t stream);

// Status word of the current device (bit 0: a device-side wait ran out).
cudaError_t read_device_status(cudaStream_t stream, uint32_t* status, bool clear);

}  // namespace q8a
