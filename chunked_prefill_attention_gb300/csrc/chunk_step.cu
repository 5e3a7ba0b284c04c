// chunk_step.cu -- one KV chunk of causal FlashAttention over a Q8_0 KV cache,
// folded into the persistent fp32 state (m, l, O) in HBM.
//
// What is computed ("Out-of-Core Flash Streaming & Speculative Decode (1M
// Context)", §3 "Chunked FlashAttention: Exact Mathematical Derivation",
// steps 1-6): for each query row i and the visible keys j of the chunk,
//   S_ij = scale * Q_i.K_j,  m' = max(m, max_j S_ij),  alpha = e^(m - m'),
//   beta_j = e^(S_ij - m'),  l' = alpha l + sum beta,  O' = alpha O + sum beta_j V_j.
// K and V are the dequantised Q8_0 blocks ("Core Architecture & The 4-Brick
// Pipeline", §5 part 2); key tiles entirely above the causal diagonal are
// skipped (same section, "Causal Skipping").
//
// GB300 design.  One CTA = two 128-row query tiles (A, B) of one (batch, head)
// that share every dequantised key/value tile.  16 warps in four warpgroups:
//   WG0, WG1   softmax of tile A / tile B (200 registers each after setmaxnreg):
//              thread i owns query row i of its tile (TMEM lane i), loads its S
//              row with tcgen05.ld, masks (diagonal and tail tiles only), takes
//              the row max (3-input max), forms beta = ex2(S*c - m*log2e) with
//              packed fp32x2 arithmetic, folds the V block scales into the fp16
//              weights P'_b = fp16(beta * d_b) (so V codes stay exact), writes P'
//              over its S row, rescales its O row in TMEM when the max moved,
//              and keeps m and l in registers.  It round-trips (m, l, O) with HBM
//              before the first and after the last tile.
//   WG2        dequant (one thread per key row): K = d*q is split exactly into
//              K_hi = fp16(d*q) and K_lo = fp16(d*q - K_hi) with half2 multiply /
//              fma on codes converted by the exponent-bias trick, so that
//              Q.K_hi + Q.K_lo reproduces Q.K from exact fp16 operands; V codes
//              are converted to fp16 exactly and the two V block scales are kept
//              aside as fp32.  K tiles are K-major with 128-byte swizzle, V tiles
//              MN-major with 64-byte swizzle.
//   WG3        warp 12: producer -- TMA tensor loads of the two fp16 Q tiles and
//              cp.async.bulk of the raw 68-byte-row K/V tiles (8704 B each,
//              contiguous in the head-major planes) into a 3-stage ring;
//              warp 13: MMA issuer (one thread): S_X = Q_X K_hi^T + Q_X K_lo^T
//              (M=128, N=128, 8 MMAs of K=16) and O_X,b += P'_X,b V_b (M=128,
//              N=32, A read from TMEM), issued in the order PV_A(t), QK_A(t+1),
//              PV_B(t), QK_B(t+1) so that each softmax warpgroup works while the
//              tensor core runs the other tile's MMAs.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,320), O_B [320,384).
// Every mbarrier wait is bounded by a wall-clock budget; a wait that runs out
// records the failing role in a per-device status word, every role then
// leaves its loop, waits (again bounded) for its own copies / MMAs in flight,
// and the CTA frees its TMEM and exits.

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace q8a {

__device__ uint32_t g_status;

namespace {

constexpr int BM = 128;                // query rows per tile
constexpr int NQT = 2;                 // query tiles per CTA
constexpr int BN = 128;                // keys per tile
constexpr int RAWB = BN * kRowBytes;   // raw bytes of one K (or V) tile: 8704
constexpr int NR = 3;                  // raw ring stages
constexpr int ND = 2;                  // dequantised ring stages
constexpr int kThreads = 512;
constexpr int kRegSoftmax = 200;       // 2 x 128 x 200 + 2 x 128 x 56 = 65536
constexpr int kRegOther = 56;
static_assert(2 * 128 * kRegSoftmax + 2 * 128 * kRegOther == 65536, "register split");

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_Q = 0;                            // NQT x (128 x 128 B), SW128 K-major
constexpr int DEQ_BYTES = 49152;
constexpr int DQ_KHI = 0, DQ_KLO = 16384, DQ_V0 = 32768, DQ_V1 = 40960;
constexpr int OFF_DEQ = NQT * 16384;
constexpr int OFF_DV = OFF_DEQ + ND * DEQ_BYTES;    // fp32 V scales [ND][64 pairs][4]
constexpr int OFF_RAW = OFF_DV + ND * 1024;         // [NR][K raw | V raw]
constexpr int OFF_BAR = OFF_RAW + NR * 2 * RAWB;
// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_RAWFULL = 1;                 // NR
constexpr int B_RAWEMPTY = B_RAWFULL + NR;   // NR
constexpr int B_DEQFULL = B_RAWEMPTY + NR;   // ND
constexpr int B_DEQEMPTY = B_DEQFULL + ND;   // ND
constexpr int B_SFULL = B_DEQEMPTY + ND;     // NQT
constexpr int B_PFULL = B_SFULL + NQT;       // NQT
constexpr int B_PVDONE = B_PFULL + NQT;      // NQT
constexpr int B_DRAIN = B_PVDONE + NQT;
constexpr int NBAR = B_DRAIN + 1;
constexpr int OFF_CTL = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_CTL + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;        // alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_RAW % 16 == 0 && RAWB % 16 == 0, "bulk copy alignment");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_S = 0;      // + 128 * tile
constexpr uint32_t T_O = 256;    // + 64 * tile

constexpr float kLog2e = 1.4426950408889634f;

// role ids recorded in the status word when a wait runs out
enum : uint32_t { R_SOFTMAX = 1, R_DEQUANT = 2, R_PRODUCER = 3, R_MMA = 4, R_DRAIN = 5 };

struct Ctl {
  uint32_t tmem_base;
  uint32_t abort;
};

// Warp-uniform bounded wait on an mbarrier phase.  All 32 lanes call it
// together.  Returns false when the CTA is aborting (honour_abort) or the
// budget ran out; in the latter case the first failure is recorded.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctl* ctl,
                                         uint64_t budget_ns, uint32_t role, bool honour_abort) {
  if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
  const int lane = threadIdx.x & 31;
  uint64_t t0 = 0;
  if (lane == 0) t0 = global_timer_ns();
  while (true) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xFFFFFFFFu, ok)) return true;
    int stop = 0;
    if (lane == 0) {
      if (honour_abort && *reinterpret_cast<volatile uint32_t*>(&ctl->abort) != 0u) {
        stop = 1;
      } else if (global_timer_ns() - t0 > budget_ns) {
        stop = 2;
        *reinterpret_cast<volatile uint32_t*>(&ctl->abort) = 1u;
        atomicCAS(&g_status, 0u, 1u | (role << 8));
      }
    }
    stop = __shfl_sync(0xFFFFFFFFu, stop, 0);
    if (stop) return false;
  }
}

template <uint32_t N>
__device__ __forceinline__ void reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Four signed int8 codes -> two half2 (exact): flip the sign bit to get
// u = q + 128 in [0, 255], place u under the fp16 exponent of 1024 (0x64uu is
// 1024 + u exactly) and subtract 1152.
__device__ __forceinline__ void codes_to_half2(uint32_t w, __half2& lo, __half2& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x7362);
  const __half2 bias = __half2half2(__ushort_as_half(0x6480));   // 1152
  lo = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  hi = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Per-CTA work description.
struct Unit {
  int64_t bh, b, h, r0;   // (batch*heads index), first row of tile A
  int T[NQT];             // KV tiles each query tile needs (0 = inactive)
  int T_all;              // max over tiles
};

__device__ __forceinline__ Unit make_unit(const ChunkArgs& a) {
  Unit u;
  const int64_t idx = blockIdx.x;
  u.bh = idx / a.n_qtiles;   // n_qtiles counts 256-row units here
  const int64_t qu = a.n_qtiles - 1 - (idx % a.n_qtiles);   // heavy units first
  u.b = u.bh / a.heads;
  u.h = u.bh % a.heads;
  u.r0 = static_cast<int64_t>(a.tile0) * BM + qu * (NQT * BM);
  u.T_all = 0;
#pragma unroll
  for (int x = 0; x < NQT; ++x) {
    const int64_t rx = u.r0 + x * BM;
    u.T[x] = 0;
    if (rx < a.n_q) {
      const int64_t r_last = i64min(rx + BM - 1, a.n_q - 1);
      int64_t n_vis = a.kv_len;
      if (a.causal) n_vis = i64min(n_vis, a.q_pos0 + r_last - a.kv_start + 1);
      u.T[x] = n_vis > 0 ? static_cast<int>((n_vis + BN - 1) / BN) : 0;
    }
    u.T_all = max(u.T_all, u.T[x]);
  }
  return u;
}

// ------------------------------------------------------------------ roles --

__device__ __forceinline__ void producer_role(const CUtensorMap* qmap, const ChunkArgs& a, const Unit& u,
                              uint8_t* smem, uint32_t sbase, Ctl* ctl) {
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const bool skip_q = (a.inject == 1) && (blockIdx.x == 0);
  if (lane == 0) {
    prefetch_tensormap(qmap);
    if (!skip_q) {
      uint32_t nq = 0;
#pragma unroll
      for (int x = 0; x < NQT; ++x) nq += (u.T[x] > 0) ? 1u : 0u;
      mbar_arrive_expect_tx(bar(B_QFULL), nq * BM * 128);
#pragma unroll
      for (int x = 0; x < NQT; ++x)
        if (u.T[x] > 0)
          tma_load_3d(sbase + OFF_Q + x * 16384, qmap, bar(B_QFULL),
                      static_cast<int32_t>(u.h * kHeadDim), static_cast<int32_t>(u.r0 + x * BM),
                      static_cast<int32_t>(u.b));
    }
  }
  int last_bulk[NR];
#pragma unroll
  for (int s = 0; s < NR; ++s) last_bulk[s] = -1;

  const uint8_t* kp = a.k8 + u.bh * a.plane_stride;
  const uint8_t* vp = a.v8 + u.bh * a.plane_stride;
  for (int t = 0; t < u.T_all; ++t) {
    const int sr = t % NR;
    if (!wait_bar(bar(B_RAWEMPTY + sr), ((t / NR) & 1) ^ 1, ctl, a.timeout_ns, R_PRODUCER, true))
      break;
    const int64_t k0 = static_cast<int64_t>(t) * BN;
    const int n = static_cast<int>(i64min(BN, a.kv_len - k0));
    const uint32_t bytes = static_cast<uint32_t>(n) * kRowBytes;
    const uint32_t dk = sbase + OFF_RAW + sr * 2 * RAWB;
    if ((bytes & 15u) == 0u) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_RAWFULL + sr), 2u * bytes);
        bulk_load(dk, kp + k0 * kRowBytes, bytes, bar(B_RAWFULL + sr));
        bulk_load(dk + RAWB, vp + k0 * kRowBytes, bytes, bar(B_RAWFULL + sr));
      }
#pragma unroll
      for (int s = 0; s < NR; ++s)
        if (s == sr) last_bulk[s] = t;
    } else {
      // ragged tail whose byte count is not a multiple of 16: plain 4-byte copies
      const uint32_t* sk = reinterpret_cast<const uint32_t*>(kp + k0 * kRowBytes);
      const uint32_t* sv = reinterpret_cast<const uint32_t*>(vp + k0 * kRowBytes);
      uint32_t* wk = reinterpret_cast<uint32_t*>(smem + OFF_RAW + sr * 2 * RAWB);
      uint32_t* wv = wk + RAWB / 4;
      const int words = n * (kRowBytes / 4);
      for (int w = lane; w < words; w += 32) {
        wk[w] = __ldg(sk + w);
        wv[w] = __ldg(sv + w);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_RAWFULL + sr));
      // nothing asynchronous is outstanding on this stage any more
#pragma unroll
      for (int s = 0; s < NR; ++s)
        if (s == sr) last_bulk[s] = -1;
    }
  }
  // Never leave with a copy in flight: wait (bounded, even when aborting) for the
  // bulk copy still outstanding on each stage (the stage's latest use, when that
  // use was a bulk copy), and for the Q tiles.
#pragma unroll
  for (int s = 0; s < NR; ++s) {
    if (last_bulk[s] >= 0)
      wait_bar(bar(B_RAWFULL + s), (last_bulk[s] / NR) & 1, ctl, a.timeout_ns, R_DRAIN, false);
  }
  if (!skip_q) wait_bar(bar(B_QFULL), 0, ctl, a.timeout_ns, R_DRAIN, false);
}

__device__ __forceinline__ void dequant_role(const ChunkArgs& a, const Unit& u, uint8_t* smem, uint32_t sbase,
                             Ctl* ctl) {
  const int k = threadIdx.x - 256;   // key row of the tile owned by this thread
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int ksw = k & 7;             // 128-byte swizzle phase of this K row
  const int vsw = (k >> 1) & 3;      // 64-byte swizzle phase of this V row
  for (int t = 0; t < u.T_all; ++t) {
    const int sr = t % NR, sd = t % ND;
    if (!wait_bar(bar(B_RAWFULL + sr), (t / NR) & 1, ctl, a.timeout_ns, R_DEQUANT, true)) break;
    if (!wait_bar(bar(B_DEQEMPTY + sd), ((t / ND) & 1) ^ 1, ctl, a.timeout_ns, R_DEQUANT, true))
      break;
    const int n_valid = static_cast<int>(i64min(BN, a.kv_len - static_cast<int64_t>(t) * BN));
    uint8_t* dq = smem + OFF_DEQ + sd * DEQ_BYTES;
    // V scales, interleaved per key pair: {d0[2p], d0[2p+1], d1[2p], d1[2p+1]}
    float* dvs = reinterpret_cast<float*>(smem + OFF_DV + sd * 1024) + (k >> 1) * 4 + (k & 1);
    uint4* khi_row = reinterpret_cast<uint4*>(dq + DQ_KHI + k * 128);
    uint4* klo_row = reinterpret_cast<uint4*>(dq + DQ_KLO + k * 128);
    uint8_t* v0_row = dq + DQ_V0 + (k >> 3) * 512 + (k & 7) * 64;
    uint8_t* v1_row = dq + DQ_V1 + (k >> 3) * 512 + (k & 7) * 64;
    if (k < n_valid) {
      const uint32_t* rk = reinterpret_cast<const uint32_t*>(smem + OFF_RAW + sr * 2 * RAWB + k * kRowBytes);
      const uint32_t* rv = rk + RAWB / 4;
      // ---- K: block 0 = bytes 0..33 (words 0..8), block 1 = bytes 34..67 (words 8..16)
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = rk[8 * blk + i];
        const unsigned short dbits =
            blk == 0 ? static_cast<unsigned short>(w[0] & 0xFFFFu) : static_cast<unsigned short>(w[0] >> 16);
        const __half2 d2 = __half2half2(__ushort_as_half(dbits));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          // codes 8c .. 8c+7 of this block
          uint32_t c0, c1;
          if (blk == 0) {
            c0 = __byte_perm(w[2 * c], w[2 * c + 1], 0x5432);
            c1 = __byte_perm(w[2 * c + 1], w[2 * c + 2], 0x5432);
          } else {
            c0 = w[1 + 2 * c];
            c1 = w[2 + 2 * c];
          }
          __half2 q0, q1, q2, q3;
          codes_to_half2(c0, q0, q1);
          codes_to_half2(c1, q2, q3);
          const __half2 h0 = __hmul2(q0, d2), h1 = __hmul2(q1, d2);
          const __half2 h2 = __hmul2(q2, d2), h3 = __hmul2(q3, d2);
          const __half2 l0 = __hfma2(q0, d2, __hneg2(h0)), l1 = __hfma2(q1, d2, __hneg2(h1));
          const __half2 l2 = __hfma2(q2, d2, __hneg2(h2)), l3 = __hfma2(q3, d2, __hneg2(h3));
          const int pc = (4 * blk + c) ^ ksw;
          khi_row[pc] = make_uint4(h2u(h0), h2u(h1), h2u(h2), h2u(h3));
          klo_row[pc] = make_uint4(h2u(l0), h2u(l1), h2u(l2), h2u(l3));
        }
      }
      // ---- V: codes to fp16 (exact), scales aside
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = rv[8 * blk + i];
        const unsigned short dbits =
            blk == 0 ? static_cast<unsigned short>(w[0] & 0xFFFFu) : static_cast<unsigned short>(w[0] >> 16);
        dvs[2 * blk] = __half2float(__ushort_as_half(dbits));
        uint8_t* vrow = blk == 0 ? v0_row : v1_row;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t c0, c1;
          if (blk == 0) {
            c0 = __byte_perm(w[2 * c], w[2 * c + 1], 0x5432);
            c1 = __byte_perm(w[2 * c + 1], w[2 * c + 2], 0x5432);
          } else {
            c0 = w[1 + 2 * c];
            c1 = w[2 + 2 * c];
          }
          __half2 q0, q1, q2, q3;
          codes_to_half2(c0, q0, q1);
          codes_to_half2(c1, q2, q3);
          *reinterpret_cast<uint4*>(vrow + 16 * (c ^ vsw)) = make_uint4(h2u(q0), h2u(q1), h2u(q2), h2u(q3));
        }
      }
    } else {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        khi_row[c] = z;
        klo_row[c] = z;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        *reinterpret_cast<uint4*>(v0_row + 16 * c) = z;
        *reinterpret_cast<uint4*>(v1_row + 16 * c) = z;
      }
      dvs[0] = 0.0f;
      dvs[2] = 0.0f;
    }
    fence_proxy_async_smem();
    mbar_arrive(bar(B_DEQFULL + sd));
    mbar_arrive(bar(B_RAWEMPTY + sr));
  }
}

__device__ __forceinline__ void mma_role(const ChunkArgs& a, const Unit& u, uint32_t sbase, uint32_t tmem,
                         Ctl* ctl) {
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  constexpr uint32_t kIdescQK = idesc_f16_f32(128, 128, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, 32, 0, 1);

  auto issue_qk = [&](int x, int t) {
    const uint32_t dq = sbase + OFF_DEQ + (t % ND) * DEQ_BYTES;
    const uint32_t d_tmem = tmem + T_S + 128 * x;
    const uint32_t qa = sbase + OFF_Q + x * 16384;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const uint32_t kb = dq + (part ? DQ_KLO : DQ_KHI);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = smem_desc(qa + 32 * kk, 1024, 1024, kSwizzle128);
        const uint64_t bd = smem_desc(kb + 32 * kk, 1024, 1024, kSwizzle128);
        mma_ss(d_tmem, ad, bd, kIdescQK, (part | kk) != 0 ? 1u : 0u);
      }
    }
  };
  auto issue_pv = [&](int x, int t) {
    const uint32_t dq = sbase + OFF_DEQ + (t % ND) * DEQ_BYTES;
    const uint32_t p_tmem = tmem + T_S + 128 * x;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const uint32_t vb = dq + (blk ? DQ_V1 : DQ_V0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t bd = smem_desc(vb + 1024 * kk, 512, 512, kSwizzle64);
        mma_ts(tmem + T_O + 64 * x + 32 * blk, p_tmem + 64 * blk + 8 * kk, bd, kIdescPV, 1u);
      }
    }
  };

  bool ok = wait_bar(bar(B_QFULL), 0, ctl, a.timeout_ns, R_MMA, true);
  if (ok) ok = wait_bar(bar(B_DEQFULL + 0), 0, ctl, a.timeout_ns, R_MMA, true);
  if (ok) {
    if (lane == 0) {
      tc_fence_after();
#pragma unroll
      for (int x = 0; x < NQT; ++x)
        if (u.T[x] > 0) {
          issue_qk(x, 0);
          mma_commit(bar(B_SFULL + x));
        }
    }
    __syncwarp();
    for (int t = 0; t < u.T_all && ok; ++t) {
#pragma unroll
      for (int x = 0; x < NQT; ++x) {
        if (t >= u.T[x]) continue;
        if (!wait_bar(bar(B_PFULL + x), t & 1, ctl, a.timeout_ns, R_MMA, true)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          issue_pv(x, t);
          mma_commit(bar(B_PVDONE + x));
          // release the dequantised stage after the last PV that reads it
          bool last = true;
#pragma unroll
          for (int y = x + 1; y < NQT; ++y) last = last && (t >= u.T[y]);
          if (last) mma_commit(bar(B_DEQEMPTY + t % ND));
        }
        __syncwarp();
        if (t + 1 < u.T[x]) {
          // K of tile t+1 dequantised, and S_x no longer read as P' by PV_x(t)
          if (!wait_bar(bar(B_DEQFULL + (t + 1) % ND), ((t + 1) / ND) & 1, ctl, a.timeout_ns, R_MMA,
                        true) ||
              !wait_bar(bar(B_PVDONE + x), t & 1, ctl, a.timeout_ns, R_MMA, true)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            tc_fence_after();
            issue_qk(x, t + 1);
            mma_commit(bar(B_SFULL + x));
          }
          __syncwarp();
        }
      }
    }
  }
  // Never leave with an MMA in flight.
  if (lane == 0) mma_commit(bar(B_DRAIN));
  __syncwarp();
  wait_bar(bar(B_DRAIN), 0, ctl, a.timeout_ns, R_DRAIN, false);
}

__device__ __forceinline__ void softmax_role(const ChunkArgs& a, const Unit& u, int x, uint8_t* smem,
                             uint32_t sbase, uint32_t tmem, Ctl* ctl) {
  const int row = threadIdx.x & 127;       // TMEM lane
  const int wq = (threadIdx.x >> 5) & 3;   // warp's lane quarter
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int T = u.T[x];
  if (T == 0) return;

  const int64_t rg = u.r0 + x * BM + row;
  const int64_t pos = a.q_pos0 + rg;
  const bool active = rg < a.n_q && (!a.causal || pos >= a.kv_start);
  const int64_t sidx = u.bh * a.n_q + rg;
  const uint32_t t_s = tmem + lane_off + T_S + 128 * x;
  const uint32_t t_o = tmem + lane_off + T_O + 64 * x;

  float m_run = -INFINITY, l_run = 0.0f;
  {
    uint32_t oa[32], ob[32];
    if (active) {
      m_run = a.m[sidx];
      l_run = a.l[sidx];
      const float4* src = reinterpret_cast<const float4*>(a.o + sidx * kHeadDim);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 p = src[i];
        oa[4 * i + 0] = __float_as_uint(p.x);
        oa[4 * i + 1] = __float_as_uint(p.y);
        oa[4 * i + 2] = __float_as_uint(p.z);
        oa[4 * i + 3] = __float_as_uint(p.w);
        const float4 y = src[8 + i];
        ob[4 * i + 0] = __float_as_uint(y.x);
        ob[4 * i + 1] = __float_as_uint(y.y);
        ob[4 * i + 2] = __float_as_uint(y.z);
        ob[4 * i + 3] = __float_as_uint(y.w);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) oa[i] = ob[i] = 0u;
    }
    tmem_st32(t_o, oa);
    tmem_st32(t_o + 32, ob);
    tmem_wait_st();
  }

  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  bool ok = true;
  for (int t = 0; t < T; ++t) {
    const int sd = t % ND;
    if (!wait_bar(bar(B_SFULL + x), t & 1, ctl, a.timeout_ns, R_SOFTMAX, true) ||
        !wait_bar(bar(B_DEQFULL + sd), (t / ND) & 1, ctl, a.timeout_ns, R_SOFTMAX, true)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t s[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(t_s + 32 * c, s[c]);
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_wait_ld(s[c]);

    const int64_t k0 = static_cast<int64_t>(t) * BN;
    const bool need_mask = (k0 + BN > a.kv_len) ||
                           (a.causal && a.kv_start + k0 + BN - 1 > a.q_pos0 + u.r0 + x * BM);
    if (need_mask) {
      int64_t lim = a.kv_len - 1 - k0;
      if (a.causal) lim = i64min(lim, pos - a.kv_start - k0);
      const int li = static_cast<int>(i64max(-1, i64min(lim, BN - 1)));
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (32 * c + j > li) s[c][j] = __float_as_uint(-INFINITY);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int j = 0; j < 32; j += 2)
        mx = max3(mx, __uint_as_float(s[c][j]), __uint_as_float(s[c][j + 1]));
    const float m_new = fmaxf(m_run, mx * a.scale);
    float alpha = 1.0f, mlog = 0.0f;
    if (m_new != -INFINITY) {
      alpha = ex2_approx((m_run - m_new) * kLog2e);
      mlog = m_new * kLog2e;
    }
    const float2 nm2 = make_float2(-mlog, -mlog);
    const float4* dv = reinterpret_cast<const float4*>(smem + OFF_DV + sd * 1024);
    float2 rs = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t pa[16], pb[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const float2 sv = make_float2(__uint_as_float(s[c][2 * jj]), __uint_as_float(s[c][2 * jj + 1]));
        const float2 e = __ffma2_rn(sv, sl2, nm2);
        const float2 bt = make_float2(ex2_approx(e.x), ex2_approx(e.y));
        rs = __fadd2_rn(rs, bt);
        const float4 d = dv[16 * c + jj];
        const float2 p0 = __fmul2_rn(bt, make_float2(d.x, d.y));
        const float2 p1 = __fmul2_rn(bt, make_float2(d.z, d.w));
        pa[jj] = pack_half2(p0.x, p0.y);
        pb[jj] = pack_half2(p1.x, p1.y);
      }
      tmem_st16(t_s + 16 * c, pa);
      tmem_st16(t_s + 64 + 16 * c, pb);
    }
    if (t > 0) {
      if (!wait_bar(bar(B_PVDONE + x), (t - 1) & 1, ctl, a.timeout_ns, R_SOFTMAX, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
    }
    if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
      uint32_t oa[32], ob[32];
      tmem_ld32(t_o, oa);
      tmem_ld32(t_o + 32, ob);
      tmem_wait_ld(oa);
      tmem_wait_ld(ob);
      const float2 al = make_float2(alpha, alpha);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float2 va = __fmul2_rn(make_float2(__uint_as_float(oa[i]), __uint_as_float(oa[i + 1])), al);
        float2 vb = __fmul2_rn(make_float2(__uint_as_float(ob[i]), __uint_as_float(ob[i + 1])), al);
        oa[i] = __float_as_uint(va.x);
        oa[i + 1] = __float_as_uint(va.y);
        ob[i] = __float_as_uint(vb.x);
        ob[i + 1] = __float_as_uint(vb.y);
      }
      tmem_st32(t_o, oa);
      tmem_st32(t_o + 32, ob);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar(B_PFULL + x));
    l_run = fmaf(l_run, alpha, rs.x + rs.y);   // same ops per tile with or without chunking
    m_run = m_new;
  }
  if (ok) {
    if (wait_bar(bar(B_PVDONE + x), (T - 1) & 1, ctl, a.timeout_ns, R_SOFTMAX, true)) {
      tc_fence_after();
      uint32_t oa[32], ob[32];
      tmem_ld32(t_o, oa);
      tmem_ld32(t_o + 32, ob);
      tmem_wait_ld(oa);
      tmem_wait_ld(ob);
      if (active) {
        a.m[sidx] = m_run;
        a.l[sidx] = l_run;
        float4* dst = reinterpret_cast<float4*>(a.o + sidx * kHeadDim);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          dst[i] = make_float4(__uint_as_float(oa[4 * i]), __uint_as_float(oa[4 * i + 1]),
                               __uint_as_float(oa[4 * i + 2]), __uint_as_float(oa[4 * i + 3]));
          dst[8 + i] = make_float4(__uint_as_float(ob[4 * i]), __uint_as_float(ob[4 * i + 1]),
                                   __uint_as_float(ob[4 * i + 2]), __uint_as_float(ob[4 * i + 3]));
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_step_kernel(const __grid_constant__ CUtensorMap qmap, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + OFF_CTL);
  const int warp = threadIdx.x >> 5;
  const int wg = warp >> 2;

  const Unit u = make_unit(a);
  if (u.T_all == 0) return;   // uniform over the CTA: no visible key for these rows

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t count = 1;
      if (i >= B_RAWEMPTY && i < B_RAWEMPTY + NR) count = 128;   // dequant threads
      if (i >= B_DEQFULL && i < B_DEQFULL + ND) count = 128;     // dequant threads
      if (i >= B_PFULL && i < B_PFULL + NQT) count = 128;        // softmax threads of a tile
      mbar_init(sbase + OFF_BAR + 8u * i, count);
    }
    ctl->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(sbase + OFF_CTL, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (wg < 2) {
    reg_alloc<kRegSoftmax>();
    softmax_role(a, u, wg, smem, sbase, tmem, ctl);
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
    return;
  }
  reg_dealloc<kRegOther>();
  if (wg == 2) {
    dequant_role(a, u, smem, sbase, ctl);
  } else if (warp == 12) {
    producer_role(&qmap, a, u, smem, sbase, ctl);
  } else if (warp == 13) {
    mma_role(a, u, sbase, tmem, ctl);
  }
  tc_fence_before();
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_chunk_step(const CUtensorMap& qmap, const ChunkArgs& args, cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(chunk_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  // the host counts 128-row query tiles; a CTA takes NQT of them
  ChunkArgs units = args;
  units.n_qtiles = (args.n_qtiles + NQT - 1) / NQT;
  const int64_t blocks = static_cast<int64_t>(units.n_qtiles) * units.bh;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  chunk_step_kernel<<<static_cast<unsigned>(blocks), kThreads, SMEM_BYTES, stream>>>(qmap, units);
  return cudaGetLastError();
}

cudaError_t read_device_status(cudaStream_t stream, uint32_t* status, bool clear) {
  uint32_t host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_status, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && clear) {
    static const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice,
                                stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  }
  if (status) *status = host;
  return e;
}

}  // namespace q8a
