// api.cu -- the extern "C" entry points of libq8attn.so (declared in
// include/q8attn.h): host-side argument validation, the Q tensor map, and the
// launches.  Every argument is checked before the first CUDA call, so argument
// errors never touch the device.

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/q8attn.h"
#include "internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}
int ok() {
  g_err[0] = '\0';
  return Q8A_OK;
}
thread_local char g_note[256] = "";

int cuda_fail(cudaError_t e, const char* what) {
  const int rc = fail(Q8A_ERR_CUDA, "%s: %s (%s)%s%s", what, cudaGetErrorName(e), cudaGetErrorString(e),
                      g_note[0] ? ": " : "", g_note);
  g_note[0] = '\0';
  return rc;
}
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int32_t> g_inject{0};

// cuTensorMapEncodeTiled, fetched once through the runtime (no link to libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

int q8a::set_error(int code, const char* fn, const char* msg) {
  return fail(code, "%s: %s", fn, msg);
}

int q8a::clear_error() { return ok(); }

namespace {
thread_local bool g_pdl = false;
}  // namespace
bool q8a::pdl_enabled() { return g_pdl; }
q8a::PdlScope::PdlScope() : prev(g_pdl) { g_pdl = true; }
q8a::PdlScope::~PdlScope() { g_pdl = prev; }

// The host-mapped failure word: one page of this library's memory, registered
// with CUDA on first use (registration pins it; nothing is allocated).  A
// kernel whose wait runs out stores its status code there as well as in the
// device word, so q8a_status reads it without a CUDA call.
namespace {
alignas(4096) uint32_t g_host_status_page[4096 / sizeof(uint32_t)];
std::mutex g_host_status_mu;
std::atomic<int> g_host_status_state{0};   // 0 not tried, 1 registered, 2 registration failed
uint32_t* g_host_status_dev = nullptr;
}  // namespace

uint32_t* q8a::host_status_word() {
  const int st = g_host_status_state.load(std::memory_order_acquire);
  if (st != 0) return st == 1 ? g_host_status_dev : nullptr;
  std::lock_guard<std::mutex> lock(g_host_status_mu);
  if (g_host_status_state.load(std::memory_order_relaxed) == 0) {
    // registration is not a stream operation; relaxed capture mode keeps it
    // legal while this or another thread is capturing a stream
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    int result = 2;
    if (cudaHostRegister(g_host_status_page, sizeof(g_host_status_page),
                         cudaHostRegisterMapped | cudaHostRegisterPortable) == cudaSuccess) {
      void* dev = nullptr;
      if (cudaHostGetDevicePointer(&dev, g_host_status_page, 0) == cudaSuccess) {
        g_host_status_dev = static_cast<uint32_t*>(dev);
        result = 1;
      } else {
        cudaHostUnregister(g_host_status_page);
      }
    }
    if (result != 1) cudaGetLastError();   // the failure is reported by q8a_status, not later calls
    cudaThreadExchangeStreamCaptureMode(&mode);
    g_host_status_state.store(result, std::memory_order_release);
  }
  return g_host_status_state.load(std::memory_order_relaxed) == 1 ? g_host_status_dev : nullptr;
}

const char* q8a::launch_note() { return g_note; }

void q8a::set_launch_note(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_note, sizeof(g_note), fmt, ap);
  va_end(ap);
}

namespace {

// allow_128: the call also supports head_dim 128 (four Q8_0 blocks per row).
int check_common(int64_t batch, int32_t heads, int32_t head_dim, const char* fn, bool allow_128) {
  if (batch < 0) return fail(Q8A_ERR_INVALID_ARG, "%s: batch must be >= 0 (got %lld)", fn, (long long)batch);
  if (heads <= 0) return fail(Q8A_ERR_INVALID_ARG, "%s: heads must be > 0 (got %d)", fn, heads);
  if (head_dim != 64 && !(allow_128 && head_dim == 128))
    return fail(Q8A_ERR_UNSUPPORTED, "%s: head_dim must be 64%s (got %d)", fn, allow_128 ? " or 128" : "",
                head_dim);
  return Q8A_OK;
}

// Bytes of one Q8_0 head row: head_dim / 32 blocks of 34 bytes.
int64_t row_bytes(int32_t head_dim) { return static_cast<int64_t>(head_dim / 32) * 34; }

}  // namespace

extern "C" {

uint32_t q8a_abi_version(void) { return Q8A_ABI_VERSION; }

const char* q8a_last_error(void) { return g_err; }

int64_t q8a_plane_stride_bytes(int64_t n_tokens) {
  if (n_tokens < 0) return -1;
  return (n_tokens * Q8A_ROW_BYTES + 15) / 16 * 16;
}

int64_t q8a_plane_stride_bytes_for(int64_t n_tokens, int32_t head_dim) {
  if (n_tokens < 0 || (head_dim != 64 && head_dim != 128)) return -1;
  return (n_tokens * row_bytes(head_dim) + 15) / 16 * 16;
}

int q8kv_quantize(const float* x, void* q8_out, int64_t batch, int64_t n_tokens, int32_t heads,
                  int32_t head_dim, int64_t out_plane_stride_bytes, void* stream) {
  q8a::NvtxRange nvtx_range("q8kv_quantize");
  const char* fn = "q8kv_quantize";
  if (int rc = check_common(batch, heads, head_dim, fn, true)) return rc;
  if (n_tokens < 0) return fail(Q8A_ERR_INVALID_ARG, "%s: n_tokens must be >= 0", fn);
  if (batch == 0 || n_tokens == 0) return ok();
  if (!x || !q8_out) return fail(Q8A_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (out_plane_stride_bytes < n_tokens * row_bytes(head_dim))
    return fail(Q8A_ERR_INVALID_ARG, "%s: plane stride %lld < n_tokens*%lld = %lld", fn,
                (long long)out_plane_stride_bytes, (long long)row_bytes(head_dim),
                (long long)(n_tokens * row_bytes(head_dim)));
  if (!aligned(x, 16) || !aligned(q8_out, 16) || out_plane_stride_bytes % 16)
    return fail(Q8A_ERR_MISALIGNED, "%s: x, q8_out and the plane stride must be 16-byte aligned", fn);
  cudaError_t e = q8a::launch_quantize(x, static_cast<uint8_t*>(q8_out), batch, n_tokens, heads,
                                       head_dim, out_plane_stride_bytes,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

int attn_state_init(float* m, float* l, float* o, int64_t batch, int32_t heads, int64_t n_q,
                    int32_t head_dim, void* stream) {
  q8a::NvtxRange nvtx_range("attn_state_init");
  const char* fn = "attn_state_init";
  if (int rc = check_common(batch, heads, head_dim, fn, true)) return rc;
  if (n_q < 0) return fail(Q8A_ERR_INVALID_ARG, "%s: n_q must be >= 0", fn);
  if (batch == 0 || n_q == 0) return ok();
  if (!m || !l || !o) return fail(Q8A_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned(m, 4) || !aligned(l, 4) || !aligned(o, 16))
    return fail(Q8A_ERR_MISALIGNED, "%s: m, l need 4-byte and o 16-byte alignment", fn);
  cudaError_t e = q8a::launch_state_init(m, l, o, batch * heads * n_q, head_dim,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

namespace {

// Validation, query-tile range and Q tensor map shared by the two chunk-step
// entry points.  Returns Q8A_OK with *empty set when the call has nothing to do.
int prepare_chunk_step(const char* fn, const void* q, int64_t q_pos0, const void* k_q8,
                       const void* v_q8, int64_t kv_plane_stride_bytes, int64_t kv_start,
                       int64_t kv_len, float* m, float* l, float* o, int64_t batch, int32_t heads,
                       int64_t n_q, int32_t head_dim, float scale, int32_t causal,
                       CUtensorMap* qmap, q8a::ChunkArgs* a, bool* empty) {
  *empty = false;
  if (int rc = check_common(batch, heads, head_dim, fn, true)) return rc;
  if (n_q < 0 || kv_len < 0) return fail(Q8A_ERR_INVALID_ARG, "%s: n_q and kv_len must be >= 0", fn);
  if (q_pos0 < 0 || kv_start < 0) return fail(Q8A_ERR_INVALID_ARG, "%s: positions must be >= 0", fn);
  if (!(scale > 0.0f) || !std::isfinite(scale))
    return fail(Q8A_ERR_INVALID_ARG, "%s: scale must be finite and > 0", fn);
  if (batch == 0 || n_q == 0 || kv_len == 0) {
    *empty = true;
    return Q8A_OK;
  }
  if (!q || !k_q8 || !v_q8 || !m || !l || !o) return fail(Q8A_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (kv_plane_stride_bytes < kv_len * row_bytes(head_dim))
    return fail(Q8A_ERR_INVALID_ARG, "%s: plane stride %lld < kv_len*%lld = %lld", fn,
                (long long)kv_plane_stride_bytes, (long long)row_bytes(head_dim),
                (long long)(kv_len * row_bytes(head_dim)));
  if (!aligned(q, 16) || !aligned(k_q8, 16) || !aligned(v_q8, 16) || kv_plane_stride_bytes % 16 ||
      !aligned(o, 16) || !aligned(m, 4) || !aligned(l, 4))
    return fail(Q8A_ERR_MISALIGNED,
                "%s: q, k_q8, v_q8, o and the plane stride need 16-byte alignment; m, l 4-byte", fn);
  if (kv_len > 0x7FFFFFFFll || n_q > 0x7FFFFFFFll || (int64_t)heads * head_dim * 2 * n_q >= (1ll << 40))
    return fail(Q8A_ERR_UNSUPPORTED, "%s: sizes beyond the supported range", fn);

  // Query tiles that can see any key of this chunk.
  int64_t first_row = 0;
  if (causal) {
    first_row = kv_start - q_pos0;
    if (first_row >= n_q) {   // every query precedes the chunk
      *empty = true;
      return Q8A_OK;
    }
    if (first_row < 0) first_row = 0;
  }
  const int64_t tile0 = first_row / 128;
  const int64_t n_qtiles = (n_q + 127) / 128 - tile0;
  if (n_qtiles * batch * heads > 0x7FFFFFFFll)
    return fail(Q8A_ERR_UNSUPPORTED, "%s: too many query tiles for one launch", fn);

  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(Q8A_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", fn);
  std::memset(qmap, 0, sizeof(*qmap));
  // the box is 64 channels (128 bytes, one swizzle atom) wide at either head_dim;
  // a head_dim 128 query tile takes two loads
  const cuuint64_t hd = static_cast<cuuint64_t>(head_dim);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(heads) * hd, static_cast<cuuint64_t>(n_q),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(heads) * hd * 2,
                                 static_cast<cuuint64_t>(heads) * hd * 2 * static_cast<cuuint64_t>(n_q)};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult cr = enc(qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(q), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(Q8A_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed (%d)", fn, (int)cr);

  *a = q8a::ChunkArgs{};
  a->q = static_cast<const uint8_t*>(q);
  a->k8 = static_cast<const uint8_t*>(k_q8);
  a->v8 = static_cast<const uint8_t*>(v_q8);
  a->m = m;
  a->l = l;
  a->o = o;
  a->plane_stride = kv_plane_stride_bytes;
  a->q_pos0 = q_pos0;
  a->kv_start = kv_start;
  a->kv_len = kv_len;
  a->n_q = n_q;
  a->heads = heads;
  a->kv_heads = heads;
  a->bh = static_cast<int32_t>(batch * heads);
  a->tile0 = static_cast<int32_t>(tile0);
  a->n_qtiles = static_cast<int32_t>(n_qtiles);
  a->scale = scale;
  a->scale_log2 = scale * 1.4426950408889634f;
  a->causal = causal ? 1 : 0;
  a->pair = (!causal && n_qtiles == 1) ? 1 : 0;
  a->head_dim = head_dim;
  {
    const int64_t kv_head_bytes = 2 * kv_len * row_bytes(head_dim);   // one head's K and V of the chunk
    const int64_t g = (int64_t{16} << 20) / kv_head_bytes;
    a->head_group = static_cast<int32_t>(g < 1 ? 1 : (g > 8 ? 8 : g));
  }
  a->timeout_ns = g_timeout_ns.load();
  a->host_status = q8a::host_status_word();
  return Q8A_OK;
}

}  // namespace

int attn_chunk_step(const void* q, int64_t q_pos0, const void* k_q8, const void* v_q8,
                    int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len, float* m,
                    float* l, float* o, int64_t batch, int32_t heads, int64_t n_q, int32_t head_dim,
                    float scale, int32_t causal, void* stream) {
  q8a::NvtxRange nvtx_range("attn_chunk_step");
  const char* fn = "attn_chunk_step";
  CUtensorMap qmap;
  q8a::ChunkArgs a;
  bool empty = false;
  if (int rc = prepare_chunk_step(fn, q, q_pos0, k_q8, v_q8, kv_plane_stride_bytes, kv_start,
                                  kv_len, m, l, o, batch, heads, n_q, head_dim, scale, causal,
                                  &qmap, &a, &empty))
    return rc;
  if (empty) return ok();
  a.inject = g_inject.exchange(0);
  cudaError_t e = head_dim == 128 ? q8a::launch_chunk_step_d128(qmap, a, static_cast<cudaStream_t>(stream))
                                  : q8a::launch_chunk_step(qmap, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

}  // extern "C"

// attn_chunk_step restricted to the 128-row query tiles [tile_begin, tile_end)
// (rows outside them are left as they are); the pipelined prefill uses it to
// start the first chunk's step on the query rows that have arrived.
int q8a::chunk_step_tiles(const void* q, int64_t q_pos0, const void* k_q8, const void* v_q8,
                          int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len, float* m,
                          float* l, float* o, int64_t batch, int32_t heads, int64_t n_q,
                          int32_t head_dim, float scale, int32_t causal, int64_t tile_begin,
                          int64_t tile_end, bool l2_keep_kv, cudaStream_t stream) {
  const char* fn = "attn_chunk_step";
  CUtensorMap qmap;
  q8a::ChunkArgs a;
  bool empty = false;
  if (int rc = prepare_chunk_step(fn, q, q_pos0, k_q8, v_q8, kv_plane_stride_bytes, kv_start,
                                  kv_len, m, l, o, batch, heads, n_q, head_dim, scale, causal,
                                  &qmap, &a, &empty))
    return rc;
  if (empty) return ok();
  const int64_t t0 = tile_begin > a.tile0 ? tile_begin : a.tile0;
  const int64_t t1 = tile_end < a.tile0 + a.n_qtiles ? tile_end : a.tile0 + a.n_qtiles;
  if (t1 <= t0) return ok();
  // at head_dim 64 a CTA folds two consecutive tiles: a range ending inside the
  // query rows must hold an even number of them, or its last CTA would also fold
  // the first tile after the range
  if (head_dim == 64 && (t1 - t0) % 2 != 0 && t1 * 128 < n_q)
    return fail(Q8A_ERR_INVALID_ARG, "%s: an interior range of an odd number of query tiles", fn);
  a.tile0 = static_cast<int32_t>(t0);
  a.n_qtiles = static_cast<int32_t>(t1 - t0);
  a.l2_keep_kv = (l2_keep_kv && head_dim == 64 && aligned(o, 32)) ? 1 : 0;
  cudaError_t e = head_dim == 128 ? q8a::launch_chunk_step_d128(qmap, a, stream)
                                  : q8a::launch_chunk_step(qmap, a, stream);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

extern "C" {

int64_t q8a_split_workspace_floats_for(int64_t batch, int32_t heads, int64_t n_q, int64_t kv_len,
                                       int64_t split_keys, int32_t head_dim) {
  if (batch < 0 || heads <= 0 || n_q < 0 || kv_len < 0 || split_keys <= 0 ||
      (head_dim != 64 && head_dim != 128))
    return -1;
  const int64_t n_splits = (kv_len + split_keys - 1) / split_keys;
  return n_splits * batch * heads * n_q * (head_dim + 2);
}

int64_t q8a_split_workspace_floats(int64_t batch, int32_t heads, int64_t n_q, int64_t kv_len,
                                   int64_t split_keys) {
  return q8a_split_workspace_floats_for(batch, heads, n_q, kv_len, split_keys, Q8A_HEAD_DIM);
}

int attn_chunk_step_gqa(const void* q, int64_t q_pos0, const void* k_q8, const void* v_q8,
                        int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len, float* m,
                        float* l, float* o, int64_t batch, int32_t heads, int32_t kv_heads,
                        int64_t n_q, int32_t head_dim, float scale, int32_t causal, void* stream) {
  q8a::NvtxRange nvtx_range("attn_chunk_step_gqa");
  const char* fn = "attn_chunk_step_gqa";
  if (kv_heads <= 0 || heads <= 0 || heads % kv_heads != 0)
    return fail(Q8A_ERR_INVALID_ARG, "%s: heads (%d) must be a positive multiple of kv_heads (%d)",
                fn, (int)heads, (int)kv_heads);
  CUtensorMap qmap;
  q8a::ChunkArgs a;
  bool empty = false;
  if (int rc = prepare_chunk_step(fn, q, q_pos0, k_q8, v_q8, kv_plane_stride_bytes, kv_start,
                                  kv_len, m, l, o, batch, heads, n_q, head_dim, scale, causal,
                                  &qmap, &a, &empty))
    return rc;
  if (empty) return ok();
  a.kv_heads = kv_heads;
  a.inject = g_inject.exchange(0);
  cudaError_t e = head_dim == 128 ? q8a::launch_chunk_step_d128(qmap, a, static_cast<cudaStream_t>(stream))
                                  : q8a::launch_chunk_step(qmap, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

}  // extern "C"

namespace {

// Q as the packed A operand of grouped-query bursts: a 3-D view {64 channels,
// heads, batch * n_q rows} of the fp16 [B][n_q][H][64] tensor with a box of
// {64, group, 128 / group}, so one box is 128 rows ordered (query row, head of
// the group), 128-byte swizzled like the plain query tile.
int encode_q_packed(const char* fn, const void* q, int64_t batch, int32_t heads, int64_t n_q,
                    int32_t group, CUtensorMap* qmap) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(Q8A_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", fn);
  std::memset(qmap, 0, sizeof(*qmap));
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch * n_q)};
  const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(heads) * 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(128 / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult cr = enc(qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(Q8A_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed (%d)", fn, (int)cr);
  return Q8A_OK;
}

// The split step behind attn_chunk_step_split (kv_heads = heads) and
// attn_chunk_step_split_gqa.
int split_step(const char* fn, const void* q, int64_t q_pos0, const void* k_q8, const void* v_q8,
               int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len, float* m, float* l,
               float* o, int64_t batch, int32_t heads, int32_t kv_heads, int64_t n_q, int32_t head_dim,
               float scale, int32_t causal, int64_t split_keys, float* workspace,
               int64_t workspace_floats, void* stream) {
  if (kv_heads <= 0 || heads <= 0 || heads % kv_heads != 0)
    return fail(Q8A_ERR_INVALID_ARG, "%s: heads (%d) must be a positive multiple of kv_heads (%d)",
                fn, (int)heads, (int)kv_heads);
  if (head_dim != 64 && head_dim != 128)
    return fail(Q8A_ERR_UNSUPPORTED, "%s: head_dim must be 64 or 128 (got %d)", fn, head_dim);
  if (split_keys <= 0 || split_keys % 128 != 0)
    return fail(Q8A_ERR_INVALID_ARG, "%s: split_keys must be a positive multiple of 128 (got %lld)",
                fn, (long long)split_keys);
  // the workspace is checked before anything touches the device
  int64_t n_splits = 0, rows = 0;
  if (batch > 0 && heads > 0 && n_q > 0 && kv_len > 0) {
    n_splits = (kv_len + split_keys - 1) / split_keys;
    if (n_splits > 65535) return fail(Q8A_ERR_UNSUPPORTED, "%s: more than 65535 key ranges", fn);
    rows = batch * heads * n_q;
    const int64_t need = n_splits * rows * (head_dim + 2);
    if (!workspace) return fail(Q8A_ERR_INVALID_ARG, "%s: null workspace", fn);
    if (workspace_floats < need)
      return fail(Q8A_ERR_INVALID_ARG, "%s: workspace of %lld floats < %lld needed", fn,
                  (long long)workspace_floats, (long long)need);
    if (!aligned(workspace, 16))
      return fail(Q8A_ERR_MISALIGNED, "%s: workspace needs 16-byte alignment", fn);
  }
  CUtensorMap qmap;
  q8a::ChunkArgs a;
  bool empty = false;
  if (int rc = prepare_chunk_step(fn, q, q_pos0, k_q8, v_q8, kv_plane_stride_bytes, kv_start,
                                  kv_len, m, l, o, batch, heads, n_q, head_dim, scale, causal,
                                  &qmap, &a, &empty))
    return rc;
  if (empty) return ok();
  // workspace: partial O [n_splits][rows][D], then m [n_splits][rows], then l
  a.split_keys = split_keys;
  a.n_splits = static_cast<int32_t>(n_splits);
  a.part_o = workspace;
  a.part_m = workspace + n_splits * rows * head_dim;
  a.part_l = a.part_m + n_splits * rows;
  a.kv_heads = kv_heads;
  q8a::ChunkArgs merge = a;   // the merge walks every (batch, query head, row)
  // Few query rows over grouped K/V heads (a burst): the tiles take (query row,
  // query head) pairs of one K/V group, so each dequantised key tile serves
  // all the group's heads instead of one.
  const int32_t group = heads / kv_heads;
  if (head_dim == 64 && !causal && group >= 2 && 128 % group == 0) {
    if (int rc = encode_q_packed(fn, q, batch, heads, n_q, group, &qmap)) return rc;
    a.pack = group;
    a.bh = static_cast<int32_t>(batch * kv_heads);
    a.tile0 = 0;
    a.n_qtiles = static_cast<int32_t>((n_q * group + 127) / 128);
    a.pair = 0;
  }
  a.inject = g_inject.exchange(0);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = head_dim == 128 ? q8a::launch_chunk_step_d128(qmap, a, st) : q8a::launch_chunk_step(qmap, a, st);
  if (e == cudaSuccess) e = q8a::launch_split_merge(merge, st);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

}  // namespace

extern "C" {

int attn_chunk_step_split(const void* q, int64_t q_pos0, const void* k_q8, const void* v_q8,
                          int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len,
                          float* m, float* l, float* o, int64_t batch, int32_t heads, int64_t n_q,
                          int32_t head_dim, float scale, int32_t causal, int64_t split_keys,
                          float* workspace, int64_t workspace_floats, void* stream) {
  q8a::NvtxRange nvtx_range("attn_chunk_step_split");
  return split_step("attn_chunk_step_split", q, q_pos0, k_q8, v_q8, kv_plane_stride_bytes, kv_start, kv_len, m,
                    l, o, batch, heads, heads, n_q, head_dim, scale, causal, split_keys, workspace,
                    workspace_floats, stream);
}

int attn_chunk_step_split_gqa(const void* q, int64_t q_pos0, const void* k_q8, const void* v_q8,
                              int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len,
                              float* m, float* l, float* o, int64_t batch, int32_t heads,
                              int32_t kv_heads, int64_t n_q, int32_t head_dim, float scale,
                              int32_t causal, int64_t split_keys, float* workspace,
                              int64_t workspace_floats, void* stream) {
  q8a::NvtxRange nvtx_range("attn_chunk_step_split_gqa");
  return split_step("attn_chunk_step_split_gqa", q, q_pos0, k_q8, v_q8, kv_plane_stride_bytes, kv_start,
                    kv_len, m, l, o, batch, heads, kv_heads, n_q, head_dim, scale, causal, split_keys,
                    workspace, workspace_floats, stream);
}

}  // extern "C"

// ---- allocation-free split step ----------------------------------------------
// Scratch for attn_chunk_step_split_static: the partial states live in this
// fixed array, which takes 32 MiB on each GPU where the library's kernels are
// loaded (under lazy module loading, the GPUs where one of them first runs)
// until the process exits.  In host code the symbol is only a stand-in; its
// device address is looked up once per device with that device current, and
// again whenever the device's current context has changed (after a device
// reset the module is loaded anew and the array may sit elsewhere).
namespace {

constexpr int64_t kStaticSplitFloats = 8ll * 1024 * 1024;   // 32 MiB
__device__ __align__(256) float g_static_split_scratch[kStaticSplitFloats];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
float* g_static_ptr[kMaxDevices] = {};
CUcontext g_static_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current_fn() {
  static std::once_flag once;
  static CtxGetCurrentFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch on the current device.
int static_scratch(const char* fn, float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  if (dev < 0 || dev >= kMaxDevices)
    return fail(Q8A_ERR_UNSUPPORTED, "%s: device ordinal %d beyond %d", fn, dev, kMaxDevices);
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (!get_ctx) return fail(Q8A_ERR_CUDA, "%s: cuCtxGetCurrent unavailable", fn);
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (!ctx || !g_static_ptr[dev] || g_static_ctx[dev] != ctx) {
    // the lookup itself makes the device's primary context current
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_split_scratch);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return fail(Q8A_ERR_CUDA, "%s: no current CUDA context", fn);
    g_static_ptr[dev] = static_cast<float*>(p);
    g_static_ctx[dev] = ctx;
  }
  *out = g_static_ptr[dev];
  return Q8A_OK;
}

}  // namespace

extern "C" {

int64_t q8a_static_split_scratch_floats(void) { return kStaticSplitFloats; }

int attn_chunk_step_split_static(const void* q, int64_t q_pos0, const void* k_q8, const void* v_q8,
                                 int64_t kv_plane_stride_bytes, int64_t kv_start, int64_t kv_len,
                                 float* m, float* l, float* o, int64_t batch, int32_t heads,
                                 int64_t n_q, int32_t head_dim, float scale, int32_t causal,
                                 int64_t split_keys, void* stream) {
  q8a::NvtxRange nvtx_range("attn_chunk_step_split_static");
  const char* fn = "attn_chunk_step_split_static";
  if (head_dim != 64 && head_dim != 128)
    return fail(Q8A_ERR_UNSUPPORTED, "%s: head_dim must be 64 or 128 (got %d)", fn, head_dim);
  if (split_keys <= 0 || split_keys % 128 != 0)
    return fail(Q8A_ERR_INVALID_ARG, "%s: split_keys must be a positive multiple of 128 (got %lld)",
                fn, (long long)split_keys);
  float* ws = nullptr;
  if (batch > 0 && heads > 0 && n_q > 0 && kv_len > 0) {
    const int64_t need = q8a_split_workspace_floats_for(batch, heads, n_q, kv_len, split_keys, head_dim);
    if (need > kStaticSplitFloats)
      return fail(Q8A_ERR_INVALID_ARG,
                  "%s: the partial states need %lld floats, more than the %lld of the static "
                  "scratch; use larger key ranges or attn_chunk_step_split",
                  fn, (long long)need, (long long)kStaticSplitFloats);
    if (int rc = static_scratch(fn, &ws)) return rc;
  }
  return attn_chunk_step_split(q, q_pos0, k_q8, v_q8, kv_plane_stride_bytes, kv_start, kv_len, m, l,
                               o, batch, heads, n_q, head_dim, scale, causal, split_keys, ws,
                               kStaticSplitFloats, stream);
}

int attn_finalize(const float* l, const float* o, void* out, int64_t batch, int32_t heads,
                  int64_t n_q, int32_t head_dim, void* stream) {
  q8a::NvtxRange nvtx_range("attn_finalize");
  const char* fn = "attn_finalize";
  if (int rc = check_common(batch, heads, head_dim, fn, true)) return rc;
  if (n_q < 0) return fail(Q8A_ERR_INVALID_ARG, "%s: n_q must be >= 0", fn);
  if (batch == 0 || n_q == 0) return ok();
  if (!l || !o || !out) return fail(Q8A_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned(l, 4) || !aligned(o, 16) || !aligned(out, 16))
    return fail(Q8A_ERR_MISALIGNED, "%s: l needs 4-byte, o and out 16-byte alignment", fn);
  cudaError_t e = q8a::launch_finalize(l, o, out, batch, heads, n_q, head_dim,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

int q8a_device_status(void* stream, uint32_t* status_out, int32_t clear) {
  uint32_t s = 0;
  cudaError_t e = q8a::read_device_status(static_cast<cudaStream_t>(stream), &s, clear != 0);
  if (e == cudaSuccess && clear) __atomic_store_n(&g_host_status_page[0], 0u, __ATOMIC_RELEASE);
  if (status_out) *status_out = s;
  if (e != cudaSuccess) return cuda_fail(e, "q8a_device_status");
  if (s != 0)
    return fail(Q8A_ERR_TIMEOUT, "q8a_device_status: a device-side wait ran out (status 0x%x, role %u)",
                s, (s >> 8) & 0xFFu);
  return ok();
}

int q8a_status(void* stream) {
  if (g_host_status_state.load(std::memory_order_acquire) == 2)
    return fail(Q8A_ERR_UNSUPPORTED, "q8a_status: the host-mapped status word could not be registered; "
                                     "use q8a_device_status");
  if (stream) {
    const cudaError_t e = cudaStreamQuery(static_cast<cudaStream_t>(stream));   // does not block
    if (e != cudaSuccess && e != cudaErrorNotReady) return cuda_fail(e, "q8a_status");
  }
  const uint32_t s = __atomic_load_n(&g_host_status_page[0], __ATOMIC_ACQUIRE);
  if (s != 0)
    return fail(Q8A_ERR_TIMEOUT, "q8a_status: a device-side wait ran out (status 0x%x, role %u)", s,
                (s >> 8) & 0xFFu);
  return ok();
}

int q8a_set_wait_timeout_ns(uint64_t ns) {
  if (ns < 1000000ull) return fail(Q8A_ERR_INVALID_ARG, "q8a_set_wait_timeout_ns: minimum is 1e6 ns");
  g_timeout_ns.store(ns);
  return ok();
}

int q8a_test_inject(int32_t kind) {
  if (kind != 0 && kind != 1) return fail(Q8A_ERR_INVALID_ARG, "q8a_test_inject: kind must be 0 or 1");
  g_inject.store(kind);
  return ok();
}

}  // extern "C"
