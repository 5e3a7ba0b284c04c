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
// Memory plan (HBM-bound: 4 B read per value + 34 B written per 32 values):
// one block handles 16 tokens (8 at head_dim 128) x 8 heads, one warp per head
// and one thread per 32-value block.  A thread loads its block's
// 128 contiguous bytes with four 256-bit loads (eight 128-bit loads when x is
// only 16-byte aligned), reduces amax in registers, forms d and the reciprocal
// once, and emits its 32 codes as eight 32-bit words into its head's staging
// rows in shared memory.  The warp then writes its head's consecutive rows
// (1088 contiguous, 16-byte-aligned bytes of the head-major plane) back with
// 128-bit stores (32-bit stores for a ragged last tile); no block-wide barrier,
// so the warps of a block load, convert and store independently.
// This translation unit must not be built with fast-math (IEEE divides).

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace q8a {
namespace {

constexpr int kHeads = 8;       // heads per block, one warp each
constexpr int kThreads = 256;
static_assert(kThreads / 32 == kHeads, "one warp per head of the block");
constexpr int kStageBytes = 1088;   // one head's rows of a tile: 16 x 68 or 8 x 136 bytes

// Two codes from two values, each as the low byte of a word: q = RN(x / d) by
// the corrected quotient above (packed fp32x2), rounded half away from zero and
// clamped to [-127, 127], every step exact in fp32:
//   floor(RZ(a + 0.5)) is a rounded half away from zero for 0 <= a < 2^23
//     (a + 0.5 is exact for a >= 0.5; below, round-toward-zero keeps it < 1);
//   clamping t to 127.5 first clamps floor(t) to 127 (and catches a >= 2^23);
//   RZ(t + 2^23) - 2^23 is floor(t) for 0.5 <= t < 2^23;
//   RN(s + 1.5 * 2^23) holds the integer s (|s| <= 127) in its low byte, in
//     two's complement.
// With y = 0 and nd = 0 (scale 0, or +inf in fp16 when amax exceeds
// 65504 * 127, where x / inf = 0) both codes are 0.
__device__ __forceinline__ uint2 code_pair(float2 x, float2 nd2, float2 y2) {
  const float2 q0 = __fmul2_rn(x, y2);
  const float2 r = __ffma2_rn(q0, nd2, x);
  const float2 qq = __ffma2_rn(r, y2, q0);
  float2 t = __fadd2_rz(make_float2(fabsf(qq.x), fabsf(qq.y)), make_float2(0.5f, 0.5f));
  t = make_float2(fminf(t.x, 127.5f), fminf(t.y, 127.5f));
  const float2 m = __fadd2_rz(t, make_float2(8388608.0f, 8388608.0f));
  const float2 f = __fadd2_rn(m, make_float2(-8388608.0f, -8388608.0f));
  const float2 u = __fadd2_rn(make_float2(copysignf(f.x, qq.x), copysignf(f.y, qq.y)),
                              make_float2(12582912.0f, 12582912.0f));
  return make_uint2(__float_as_uint(u.x), __float_as_uint(u.y));
}

// 256-bit read-only load of eight consecutive floats (32-byte aligned).  The
// input is read once, so its lines go first when L2 needs room (`policy` is
// the evict-first policy); the Q8_0 rows written here stay for the chunk step
// that reads them next.
__device__ __forceinline__ void ldg256(const float* p, float* v, uint64_t policy) {
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                 "=f"(v[6]), "=f"(v[7])
               : "l"(p), "l"(policy));
}
// 128-bit read-only load with the same policy.
__device__ __forceinline__ float4 ldg128(const float* p, uint64_t policy) {
  float4 f;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
               : "l"(p), "l"(policy));
  return f;
}

// kD: channels per head row (64 or 128: kD / 32 Q8_0 blocks, kD / 32 * 34
// bytes per row).  A warp quantises kTok = 32 / blocks consecutive tokens of one
// head, one lane per block (lane = blocks * token + block).
// kWide: x is 32-byte aligned and every block is loaded with 256-bit loads
// (every block starts a multiple of 128 bytes after x); otherwise 128-bit loads.
template <int kD, bool kWide>
__global__ void __launch_bounds__(kThreads)
q8kv_quantize_kernel(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t n_tokens,
                     int32_t heads, int64_t plane_stride, int32_t tok_tiles, int32_t head_tiles) {
  constexpr int kBlk = kD / 32;
  constexpr int kRow = kBlk * 34;
  constexpr int kTok = 32 / kBlk;
  static_assert(kTok * kRow == kStageBytes, "staging rows of one head");
  __shared__ __align__(16) uint8_t stage[kHeads][kStageBytes];
  pdl_launch_dependents();
  pdl_wait();

  const int64_t blk = blockIdx.x;
  const int ht = static_cast<int>(blk % head_tiles);
  const int64_t rest = blk / head_tiles;
  const int64_t tt = rest % tok_tiles;
  const int64_t b = rest / tok_tiles;
  const int64_t t0 = tt * kTok;
  const int h0 = ht * kHeads;
  const int n_tok = static_cast<int>(i64min(kTok, n_tokens - t0));
  const int n_h = min(kHeads, heads - h0);

  // warp -> head hh of the tile; lane -> (token tok, 32-value block bb)
  const int hh = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (hh >= n_h) return;
  const int tok = lane / kBlk, bb = lane % kBlk;
  const bool valid = tok < n_tok;
  float v[32];
  if (valid) {
    const float* src = x + (((b * n_tokens + t0 + tok) * heads + h0 + hh) * kD + 32 * bb);
    const uint64_t pol = l2_evict_first_policy();
    if (kWide) {
#pragma unroll
      for (int i = 0; i < 4; ++i) ldg256(src + 8 * i, v + 8 * i, pol);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 f = ldg128(src + 4 * i, pol);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.0f;
  }
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));
  const __half d16 = __float2half_rn(__fdiv_rn(a, 127.0f));
  const float d = __half2float(d16);
  const bool finite_nonzero = d > 0.0f && d <= 65504.0f;
  const float y = finite_nonzero ? __frcp_rn(d) : 0.0f;
  const float nd = finite_nonzero ? -d : 0.0f;
  const float2 y2 = make_float2(y, y), nd2 = make_float2(nd, nd);
  uint32_t w[8];   // codes 4k .. 4k+3, little-endian
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint2 c01 = code_pair(make_float2(v[4 * k], v[4 * k + 1]), nd2, y2);
    const uint2 c23 = code_pair(make_float2(v[4 * k + 2], v[4 * k + 3]), nd2, y2);
    w[k] = __byte_perm(__byte_perm(c01.x, c01.y, 0x0040), __byte_perm(c23.x, c23.y, 0x0040), 0x5410);
  }
  const uint32_t dbits = __half_as_ushort(d16);
  if (valid) {
    // block bb of the row: d at 34 * bb, codes at 34 * bb + 2.  Rows start
    // 4-byte aligned; an even block starts 4-byte aligned (codes at 2 mod 4),
    // an odd one 2 mod 4 (codes 4-byte aligned).
    uint8_t* blk_at = &stage[hh][tok * kRow + 34 * bb];
    if ((bb & 1) == 0) {
      uint32_t* p = reinterpret_cast<uint32_t*>(blk_at);
      p[0] = dbits | (w[0] << 16);
#pragma unroll
      for (int k = 0; k < 7; ++k) p[1 + k] = __funnelshift_r(w[k], w[k + 1], 16);
      *reinterpret_cast<uint16_t*>(blk_at + 32) = static_cast<uint16_t>(w[7] >> 16);
    } else {
      *reinterpret_cast<uint16_t*>(blk_at) = static_cast<uint16_t>(dbits);
      uint32_t* p = reinterpret_cast<uint32_t*>(blk_at + 2);
#pragma unroll
      for (int k = 0; k < 8; ++k) p[k] = w[k];
    }
  }
  __syncwarp();

  // Write back: head hh's rows t0 .. t0+n_tok-1 are contiguous in its plane
  // (byte t0 * kRow = tt * 1088, a multiple of 16).
  uint8_t* dst = out + (b * heads + h0 + hh) * plane_stride + t0 * kRow;
  if (n_tok == kTok) {
    const uint4* s4 = reinterpret_cast<const uint4*>(stage[hh]);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int i = lane; i < kStageBytes / 16; i += 32) d4[i] = s4[i];
  } else {
    const uint32_t* s1 = reinterpret_cast<const uint32_t*>(stage[hh]);
    uint32_t* d1 = reinterpret_cast<uint32_t*>(dst);
    for (int i = lane; i < n_tok * (kRow / 4); i += 32) d1[i] = s1[i];
  }
}

template <int kD>
cudaError_t launch_quantize_d(const float* x, uint8_t* out, int64_t batch, int64_t n_tokens,
                              int32_t heads, int64_t plane_stride, cudaStream_t stream) {
  constexpr int kTok = 32 / (kD / 32);
  const int64_t tok_tiles = (n_tokens + kTok - 1) / kTok;
  const int64_t head_tiles = (heads + kHeads - 1) / kHeads;
  const int64_t blocks = batch * tok_tiles * head_tiles;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF || tok_tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const bool wide = (reinterpret_cast<uintptr_t>(x) & 31u) == 0;
  auto kernel = wide ? q8kv_quantize_kernel<kD, true> : q8kv_quantize_kernel<kD, false>;
  return launch_kernel(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream, x, out, n_tokens,
                       heads, plane_stride, static_cast<int32_t>(tok_tiles), static_cast<int32_t>(head_tiles));
}

}  // namespace

cudaError_t launch_quantize(const float* x, uint8_t* out, int64_t batch, int64_t n_tokens,
                            int32_t heads, int32_t head_dim, int64_t plane_stride,
                            cudaStream_t stream) {
  if (head_dim == 64) return launch_quantize_d<64>(x, out, batch, n_tokens, heads, plane_stride, stream);
  if (head_dim == 128) return launch_quantize_d<128>(x, out, batch, n_tokens, heads, plane_stride, stream);
  return cudaErrorInvalidValue;
}

}  // namespace q8a
