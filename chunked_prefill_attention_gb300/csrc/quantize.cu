// quantize.cu -- dynamic Q8_0 quantisation of a K or V tensor.
//
// Block format and rule ("Core Architecture & The 4-Brick Pipeline", §5 part 2
// "Dynamic Q8_0 KV Cache Compression"): 32 values -> one fp16 scale d plus 32
// int8 codes, 34 bytes; symmetric 8-bit.  Here d = fp16_rn(amax / 127) with an
// IEEE fp32 divide, and q = round_half_away(x / d) with an IEEE fp32 divide by
// the stored fp16 d, clamped to [-127, 127] (d == 0 -> all codes 0).
//
// The quotient x / d is formed as the correctly rounded fp32 quotient without a
// divide per value: with y = RN(1/d) (one __frcp_rn per block), q0 = RN(x*y) is
// within one ulp of x/d, the residual r = x - q0*d is exact as one fma, and
// RN(q0 + r*y) is RN(x/d) -- Markstein's correction theorem for division
// with a fused multiply-add (P. Markstein, IBM J. Res. Dev. 34(1), 1990; also
// Muller et al., "Handbook of Floating-Point Arithmetic", on fma-based
// division).  The theorem needs a normal quotient; a quotient below 2^-126 is
// far below 0.5 and rounds to code 0 either way.
//
// Memory plan (HBM-bound: 256 B read + 68 B written per 64-value head row):
// one block handles 16 tokens x 8 heads.  Each half-warp quantises one head
// row: its 16 lanes load the row's 256 bytes with one 128-bit load each, the 8
// lanes of a 32-value block reduce amax with three xor-shuffles, and every lane
// emits 4 codes.  Rows are assembled in shared memory so that each head's 16
// consecutive output rows (1088 contiguous bytes of the head-major plane) are
// written back as coalesced 32-bit words.
// This translation unit must not be built with fast-math (IEEE divides).

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace q8a {
namespace {

constexpr int kTok = 16;    // tokens per block
constexpr int kHeads = 8;   // heads per block
constexpr int kThreads = 256;
constexpr int kRowsPerHalfWarp = kTok * kHeads / (kThreads / 16);  // 8

// RN(x / d) for d > 0, from y = RN(1 / d) (see the note above).
__device__ __forceinline__ float div_rn_by(float x, float d, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q0, d, x);
  return __fmaf_rn(r, y, q0);
}

__device__ __forceinline__ uint32_t quant4(float4 v, float d, float y) {
  const float x[4] = {v.x, v.y, v.z, v.w};
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int q = 0;
    if (d > 0.0f) {
      float r = roundf(div_rn_by(x[i], d, y));   // round half away from zero
      r = fminf(fmaxf(r, -127.0f), 127.0f);
      q = static_cast<int>(r);
    }
    packed |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * i);
  }
  return packed;
}

__global__ void __launch_bounds__(kThreads)
q8kv_quantize_kernel(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t n_tokens,
                     int32_t heads, int64_t plane_stride, int32_t tok_tiles, int32_t head_tiles) {
  __shared__ __align__(16) uint8_t stage[kHeads][kTok * kRowBytes];

  const int64_t blk = blockIdx.x;
  const int ht = static_cast<int>(blk % head_tiles);
  const int64_t rest = blk / head_tiles;
  const int64_t tt = rest % tok_tiles;
  const int64_t b = rest / tok_tiles;
  const int64_t t0 = tt * kTok;
  const int h0 = ht * kHeads;
  const int n_tok = static_cast<int>(i64min(kTok, n_tokens - t0));
  const int n_h = min(kHeads, heads - h0);

  const int hw = threadIdx.x >> 4;   // half-warp: one head row at a time
  const int ln = threadIdx.x & 15;   // lane in half-warp: 4 consecutive channels
  const int blkid = ln >> 3;         // 32-value block of the row (0 or 1)

  // Issue all loads first: rows hw, hw+16, ... (row rr -> token rr/8, head rr%8)
  float4 v[kRowsPerHalfWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerHalfWarp; ++i) {
    const int rr = hw + 16 * i;
    const int tok = rr >> 3, hh = rr & 7;
    v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tok < n_tok && hh < n_h) {
      const float* src = x + (((b * n_tokens + t0 + tok) * heads + h0 + hh) * kHeadDim + 4 * ln);
      v[i] = __ldg(reinterpret_cast<const float4*>(src));
    }
  }
#pragma unroll
  for (int i = 0; i < kRowsPerHalfWarp; ++i) {
    const int rr = hw + 16 * i;
    const int tok = rr >> 3, hh = rr & 7;
    float a = fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w)));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
    const __half d16 = __float2half_rn(__fdiv_rn(a, 127.0f));
    const float d = __half2float(d16);
    const float y = d > 0.0f ? __frcp_rn(d) : 0.0f;
    const uint32_t codes = quant4(v[i], d, y);
    if (tok < n_tok && hh < n_h) {
      uint8_t* row = &stage[hh][tok * kRowBytes];
      const int off = 34 * blkid + 2 + 4 * (ln & 7);   // 2-byte aligned
      *reinterpret_cast<uint16_t*>(row + off) = static_cast<uint16_t>(codes & 0xFFFFu);
      *reinterpret_cast<uint16_t*>(row + off + 2) = static_cast<uint16_t>(codes >> 16);
      if ((ln & 7) == 0) *reinterpret_cast<__half*>(row + 34 * blkid) = d16;
    }
  }
  __syncthreads();

  // Write back: head hh's rows t0..t0+n_tok-1 are contiguous in its plane;
  // warp hh copies them as 32-bit words.
  static_assert(kThreads / 32 == kHeads, "one warp per head of the block");
  const int hh = threadIdx.x >> 5;
  if (hh < n_h) {
    const int words = n_tok * (kRowBytes / 4);
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + (b * heads + h0 + hh) * plane_stride +
                                                t0 * kRowBytes);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(stage[hh]);
    for (int wi = threadIdx.x & 31; wi < words; wi += 32) dst[wi] = src[wi];
  }
}

}  // namespace

cudaError_t launch_quantize(const float* x, uint8_t* out, int64_t batch, int64_t n_tokens,
                            int32_t heads, int64_t plane_stride, cudaStream_t stream) {
  const int64_t tok_tiles = (n_tokens + kTok - 1) / kTok;
  const int64_t head_tiles = (heads + kHeads - 1) / kHeads;
  const int64_t blocks = batch * tok_tiles * head_tiles;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF || tok_tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  q8kv_quantize_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
      x, out, n_tokens, heads, plane_stride, static_cast<int32_t>(tok_tiles),
      static_cast<int32_t>(head_tiles));
  return cudaGetLastError();
}

}  // namespace q8a
