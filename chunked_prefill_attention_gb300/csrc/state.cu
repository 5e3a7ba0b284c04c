// state.cu -- the persistent online-softmax state before the first chunk and
// the final normalisation after the last one ("Out-of-Core Flash Streaming &
// Speculative Decode (1M Context)", §3: m, l, O kept in global memory between
// chunks; Attention_i = O_i / l_i after chunk C-1).
//
// Both kernels are HBM streams: init writes 4 * (2 + D) B per (row, head)
// (264 B at head_dim 64); finalise reads 4 * (1 + D) B and writes 2 * D B.
// Finalise maps D / 8 threads to one D-float O row (two 128-bit loads each) and
// writes 8 fp16 (one 128-bit store) per thread, so both the head-major fp32
// reads and the token-major fp16 writes are whole 128-byte lines.

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace q8a {
namespace {

constexpr int kThreads = 256;

__host__ __device__ __forceinline__ int64_t i64min_host(int64_t a, int64_t b) { return a < b ? a : b; }

__global__ void __launch_bounds__(kThreads)
state_init_kernel(float* __restrict__ m, float* __restrict__ l, float4* __restrict__ o,
                  int64_t rows, int32_t head_dim) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t start = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = start; i < rows * (head_dim / 4); i += stride) o[i] = z;
  for (int64_t i = start; i < rows; i += stride) {
    m[i] = -INFINITY;
    l[i] = 0.0f;
  }
}

// kD / 8 threads per state row, 8 channels each.
template <int kD>
__global__ void __launch_bounds__(kThreads)
finalize_kernel(const float* __restrict__ l, const float4* __restrict__ o, uint4* __restrict__ out,
                int64_t n_q, int32_t heads, int64_t row0, int64_t n_rows, int64_t rows) {
  // rows = B*H*n_rows state rows: query rows row0 .. row0+n_rows-1 of every plane
  pdl_launch_dependents();
  pdl_wait();
  constexpr int kParts = kD / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; g < rows * kParts;
       g += stride) {
    const int64_t k = g / kParts;       // (b*H + h)*n_rows + (r - row0)
    const int part = static_cast<int>(g % kParts);
    const int64_t r = row0 + k % n_rows;
    const int64_t bh = k / n_rows;
    const int64_t row = bh * n_q + r;   // (b*H + h)*n_q + r
    const int64_t h = bh % heads;
    const int64_t b = bh / heads;
    const float lv = __ldg(l + row);
    const float4 a = __ldg(o + row * (kD / 4) + 2 * part);
    const float4 c = __ldg(o + row * (kD / 4) + 2 * part + 1);
    // o / l rounded to fp32 without a divide per value: with r = RN(1 / l),
    // q0 = RN(o r) and the exact residual o - q0 l (one fma), RN(q0 + res r) is
    // the correctly rounded quotient (Markstein's correction) for every normal
    // quotient; a subnormal one rounds to an fp16 zero either way.
    const bool seen = lv > 0.0f;
    const float rc = seen ? __frcp_rn(lv) : 0.0f;
    const float2 r2 = make_float2(rc, rc);
    const float2 nl2 = make_float2(-lv, -lv);
    float2 y[4] = {make_float2(a.x, a.y), make_float2(a.z, a.w), make_float2(c.x, c.y), make_float2(c.z, c.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 q0 = __fmul2_rn(y[i], r2);
      const float2 res = __ffma2_rn(q0, nl2, y[i]);
      y[i] = seen ? __ffma2_rn(res, r2, q0) : make_float2(0.0f, 0.0f);
    }
    uint4 pk;
    __half2 h0 = __floats2half2_rn(y[0].x, y[0].y);
    __half2 h1 = __floats2half2_rn(y[1].x, y[1].y);
    __half2 h2 = __floats2half2_rn(y[2].x, y[2].y);
    __half2 h3 = __floats2half2_rn(y[3].x, y[3].y);
    pk.x = *reinterpret_cast<uint32_t*>(&h0);
    pk.y = *reinterpret_cast<uint32_t*>(&h1);
    pk.z = *reinterpret_cast<uint32_t*>(&h2);
    pk.w = *reinterpret_cast<uint32_t*>(&h3);
    out[((b * n_q + r) * heads + h) * kParts + part] = pk;
  }
}

// Merge of the split partial states into the state, one (b, h, row) per kD / 8
// threads (8 channels each).  It is the chunk recurrence applied with a
// partial's (m_s, l_s, O_s) in place of a chunk's row max, weight sum and
// weighted values:  m' = max(m, m_s...),  l' = l e^(m - m') + sum_s l_s e^(m_s - m'),
// O' = O e^(m - m') + sum_s O_s e^(m_s - m').  A partial is read only when its
// key range holds a key the row can see (the chunk-step kernel writes exactly
// those rows).
template <int kD>
__global__ void __launch_bounds__(kThreads)
split_merge_kernel(float* __restrict__ m, float* __restrict__ l, float4* __restrict__ o,
                   const float* __restrict__ pm, const float* __restrict__ pl,
                   const float4* __restrict__ po, int64_t rows, int64_t n_q, int64_t q_pos0,
                   int64_t kv_start, int64_t split_keys, int32_t n_splits, int32_t causal) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  constexpr int kParts = kD / 8;      // threads per row (8 or 16: a row never spans two warps)
  constexpr int kRowF4 = kD / 4;      // float4 per O row
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; g < rows * kParts;
       g += stride) {
    const int64_t row = g / kParts;   // (b*H + h)*n_q + r
    const int part = static_cast<int>(g % kParts);
    const int64_t pos = q_pos0 + row % n_q;
    // splits whose first key the row can see (all of them without the mask)
    int ns = n_splits;
    if (causal) {
      const int64_t vis = pos - kv_start;   // keys 0 .. vis of the chunk are visible
      ns = vis < 0 ? 0 : static_cast<int>(i64min_host(n_splits, vis / split_keys + 1));
    }
    if (ns == 0) continue;
    const float m0 = m[row];   // every read of this row's m and l happens here
    const float l0 = l[row];
    float mx = m0;
    for (int s = 0; s < ns; ++s) mx = fmaxf(mx, pm[s * rows + row]);
    if (mx == -INFINITY) continue;
    const float f = (m0 == -INFINITY) ? 0.0f : expf(m0 - mx);
    float lv = l0 * f;
    float4 a = o[row * kRowF4 + 2 * part], c = o[row * kRowF4 + 2 * part + 1];
    float y[8] = {a.x * f, a.y * f, a.z * f, a.w * f, c.x * f, c.y * f, c.z * f, c.w * f};
    for (int s = 0; s < ns; ++s) {
      const float ms = pm[s * rows + row];
      if (ms == -INFINITY) continue;
      const float w = expf(ms - mx);
      lv = fmaf(pl[s * rows + row], w, lv);
      const float4 pa = po[(s * rows + row) * kRowF4 + 2 * part];
      const float4 pc = po[(s * rows + row) * kRowF4 + 2 * part + 1];
      y[0] = fmaf(pa.x, w, y[0]); y[1] = fmaf(pa.y, w, y[1]);
      y[2] = fmaf(pa.z, w, y[2]); y[3] = fmaf(pa.w, w, y[3]);
      y[4] = fmaf(pc.x, w, y[4]); y[5] = fmaf(pc.y, w, y[5]);
      y[6] = fmaf(pc.z, w, y[6]); y[7] = fmaf(pc.w, w, y[7]);
    }
    o[row * kRowF4 + 2 * part] = make_float4(y[0], y[1], y[2], y[3]);
    o[row * kRowF4 + 2 * part + 1] = make_float4(y[4], y[5], y[6], y[7]);
    // the row's lanes took the same path; all have read m and l by now
    __syncwarp(((1u << kParts) - 1u) << ((threadIdx.x & 31) & ~(kParts - 1)));
    if (part == 0) {
      m[row] = mx;
      l[row] = lv;
    }
  }
}

int grid_for(int64_t work) {
  int64_t blocks = (work + kThreads - 1) / kThreads;
  const int64_t cap = 152 * 16;   // a few waves of resident blocks; grid-stride beyond
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_state_init(float* m, float* l, float* o, int64_t rows, int32_t head_dim,
                              cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  return launch_kernel(state_init_kernel, dim3(grid_for(rows * (head_dim / 4))), dim3(kThreads), 0, stream, m, l,
                       reinterpret_cast<float4*>(o), rows, head_dim);
}

cudaError_t launch_finalize(const float* l, const float* o, void* out, int64_t batch,
                            int32_t heads, int64_t n_q, int32_t head_dim, cudaStream_t stream) {
  return launch_finalize_rows(l, o, out, batch, heads, n_q, head_dim, 0, n_q, stream);
}

cudaError_t launch_finalize_rows(const float* l, const float* o, void* out, int64_t batch,
                                 int32_t heads, int64_t n_q, int32_t head_dim, int64_t row0,
                                 int64_t n_rows, cudaStream_t stream) {
  const int64_t rows = batch * heads * n_rows;
  if (rows <= 0) return cudaSuccess;
  if (head_dim != 64 && head_dim != 128) return cudaErrorInvalidValue;
  auto kernel = head_dim == 64 ? finalize_kernel<64> : finalize_kernel<128>;
  return launch_kernel(kernel, dim3(grid_for(rows * (head_dim / 8))), dim3(kThreads), 0, stream, l,
                       reinterpret_cast<const float4*>(o), reinterpret_cast<uint4*>(out), n_q, heads, row0,
                       n_rows, rows);
}

cudaError_t launch_split_merge(const ChunkArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.bh) * a.n_q;
  if (rows <= 0 || a.n_splits <= 0) return cudaSuccess;
  if (a.head_dim != 64 && a.head_dim != 128) return cudaErrorInvalidValue;
  auto kernel = a.head_dim == 64 ? split_merge_kernel<64> : split_merge_kernel<128>;
  return launch_kernel(kernel, dim3(grid_for(rows * (a.head_dim / 8))), dim3(kThreads), 0, stream, a.m, a.l,
                       reinterpret_cast<float4*>(a.o), a.part_m, a.part_l,
                       reinterpret_cast<const float4*>(a.part_o), rows, a.n_q, a.q_pos0, a.kv_start,
                       a.split_keys, a.n_splits, a.causal);
}

}  // namespace q8a
