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
// sharing every dequantised 128-key tile.  16 warps in four warpgroups:
//   WG0, WG1   softmax of tile A / tile B: thread i owns query row i of its tile
//              (TMEM lane i).  Per key tile it reads its 128-score S row from
//              TMEM in two passes of 32-column chunks (row max first, then the
//              weights), each chunk loaded while the previous one is worked on
//              and both passes kept as rolled loops (the kernel's hot code must
//              stay small enough for the instruction caches), masks
//              diagonal and tail tiles, forms beta = ex2(S*c - m*log2e) with
//              packed fp32x2 arithmetic, folds the V block scales into the fp16
//              weights P'_b = fp16(beta * d_b) (so V codes stay exact), writes P'
//              over the same S columns, rescales its O row in TMEM when the max
//              moved, and keeps m and l in registers.  It round-trips (m, l, O)
//              with HBM before the first and after the last key tile.
//   WG2        dequant, one thread per key row: K = d*q is split exactly into
//              K_hi = fp16(d*q) and K_lo = fp16(d*q - K_hi) with half2 multiply /
//              fma on codes converted by the exponent-bias trick, so that
//              Q.K_hi + Q.K_lo reproduces Q.K from exact fp16 operands; V codes
//              become fp16 exactly and the V block scales are kept aside as fp32.
//              K tiles are K-major with 128-byte swizzle, V tiles MN-major with
//              64-byte swizzle.
//   WG3        warp 12: producer -- TMA tensor loads of the two fp16 Q tiles and
//              cp.async.bulk of the raw 68-byte-row K/V tiles (8704 B each,
//              contiguous in the head-major planes) into a 2-stage ring;
//              warp 13: MMA issuer (one thread), event driven: it polls the
//              barriers without blocking and issues whatever is ready, so neither
//              softmax warpgroup waits behind the other.
// MMA shapes (measured on this part: an M=128, K=16 instruction costs about
// 55 cycles up to N=64 and 65 cycles at N=128, so narrow instructions waste the
// tensor pipe): S_X = Q_X K_hi^T + Q_X K_lo^T with N=128 (8 instructions per key
// tile); O_X,b += P'_X,b V_b with N=32, A read from TMEM, the two V blocks
// interleaved so consecutive instructions update independent accumulators.
// TMEM columns: three S buffers [0,128), [128,256), [256,384) used round-robin
// by the sequence QK_A(0), QK_B(0), QK_A(1), QK_B(1), ... (so the next S of each
// tile is computed while both softmaxes run); O_A [384,448), O_B [448,512).
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
constexpr int NR = 2;                  // raw ring stages
constexpr int ND = 3;                  // dequantised ring stages
constexpr int NSB = 3;                 // S buffers in TMEM, shared by the query tiles
constexpr int kThreads = 512;
constexpr int kRegSoftmax = 152;       // setmaxnreg split: 2 x 128 x 152 + 2 x 128 x 104 = 65536
constexpr int kRegOther = 104;
static_assert(2 * 128 * kRegSoftmax + 2 * 128 * kRegOther == 65536, "register split");

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_Q = 0;                               // NQT x (128 x 128 B), SW128 K-major
constexpr int DQ_KHI = 0, DQ_KLO = 16384, DQ_V0 = 32768, DQ_V1 = 40960;
constexpr int DEQ_BYTES = 49152;                       // K_hi, K_lo (128 x 128 B), V0, V1 (128 x 64 B)
constexpr int OFF_DEQ = NQT * 16384;
constexpr int OFF_DV = OFF_DEQ + ND * DEQ_BYTES;       // fp32 V scales [ND][64 key pairs][4]
constexpr int OFF_RAW = OFF_DV + ND * 1024;            // [NR][K raw | V raw]
constexpr int OFF_BAR = OFF_RAW + NR * 2 * RAWB;
// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_RAWFULL = 1;                 // NR
constexpr int B_RAWEMPTY = B_RAWFULL + NR;   // NR
constexpr int B_DEQFULL = B_RAWEMPTY + NR;   // ND
constexpr int B_DEQEMPTY = B_DEQFULL + ND;   // ND
constexpr int B_SFULL = B_DEQEMPTY + ND;     // NSB
constexpr int B_PFULL = B_SFULL + NSB;       // NQT
constexpr int B_PVDONE = B_PFULL + NQT;      // NQT
constexpr int B_DRAIN = B_PVDONE + NQT;
constexpr int NBAR = B_DRAIN + 1;
constexpr int OFF_CTL = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_CTL + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;           // alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_RAW % 16 == 0 && RAWB % 16 == 0, "bulk copy alignment");
static_assert(OFF_DEQ % 1024 == 0 && DEQ_BYTES % 1024 == 0, "swizzle atom alignment");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_O = 384;    // + 64 * tile

constexpr float kLog2e = 1.4426950408889634f;

// role ids recorded in the status word when a wait runs out
enum : uint32_t { R_SOFTMAX = 1, R_DEQUANT = 2, R_PRODUCER = 3, R_MMA = 4, R_DRAIN = 5 };

struct Ctl {
  uint32_t tmem_base;
  uint32_t abort;
};

// Warp-uniform bounded wait on an mbarrier phase.  All 32 lanes call it
// together.  Returns false when the CTA is aborting (honour_abort) or the
// budget ran out; in the latter case the first failure is recorded.  The budget
// is counted in SM cycles (the cycle counter is cheap to read, unlike the
// global nanosecond timer): budget_cycles = 2 x the nanosecond budget, which is
// the budget at 2 GHz and proportionally longer at lower clocks.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctl* ctl,
                                         uint64_t budget_cycles, uint32_t role, bool honour_abort) {
  if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
  const int lane = threadIdx.x & 31;
  const long long t0 = clock64();
  while (true) {
    const bool ok = mbar_try_wait_sleep(bar, parity, 100000u);   // sleep up to 0.1 ms per try
    if (__all_sync(0xFFFFFFFFu, ok)) return true;
    int stop = 0;
    if (lane == 0) {
      if (honour_abort && *reinterpret_cast<volatile uint32_t*>(&ctl->abort) != 0u) {
        stop = 1;
      } else if (static_cast<uint64_t>(clock64() - t0) > budget_cycles) {
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

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
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
  int T[NQT];             // key tiles each query tile needs (0 = inactive)
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

// Position of (query tile x, key tile t) in the QK issue sequence
// (t ascending, then x, skipping pairs with t >= T[x]); it selects the S buffer.
__device__ __forceinline__ int qk_seq(const Unit& u, int x, int t) {
  int k = 0;
#pragma unroll
  for (int y = 0; y < NQT; ++y) {
    k += min(t, u.T[y]);
    if (y < x && t < u.T[y]) ++k;
  }
  return k;
}

// ------------------------------------------------------------------ roles --

__device__ __forceinline__ void producer_role(const CUtensorMap* qmap, const ChunkArgs& a,
                                              const Unit& u, uint8_t* smem, uint32_t sbase,
                                              Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;   // cycles
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
    if (!wait_bar(bar(B_RAWEMPTY + sr), ((t / NR) & 1) ^ 1, ctl, budget, R_PRODUCER, true))
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
      wait_bar(bar(B_RAWFULL + s), (last_bulk[s] / NR) & 1, ctl, budget, R_DRAIN, false);
  }
  if (!skip_q) wait_bar(bar(B_QFULL), 0, ctl, budget, R_DRAIN, false);
}

__device__ __forceinline__ void dequant_role(const ChunkArgs& a, const Unit& u, uint8_t* smem,
                                             uint32_t sbase, Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;   // cycles
  const int k = threadIdx.x - 256;   // key row of the tile
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int ksw = k & 7;             // 128-byte swizzle phase of this K row
  const int vsw = (k >> 1) & 3;      // 64-byte swizzle phase of this V row
  for (int t = 0; t < u.T_all; ++t) {
    const int sr = t % NR, sd = t % ND;
    if (!wait_bar(bar(B_RAWFULL + sr), (t / NR) & 1, ctl, budget, R_DEQUANT, true)) break;
    if (!wait_bar(bar(B_DEQEMPTY + sd), ((t / ND) & 1) ^ 1, ctl, budget, R_DEQUANT, true))
      break;
    const int n_valid = static_cast<int>(i64min(BN, a.kv_len - static_cast<int64_t>(t) * BN));
    uint8_t* dq = smem + OFF_DEQ + sd * DEQ_BYTES;
    // V scales, interleaved per key pair: {d0[2p], d0[2p+1], d1[2p], d1[2p+1]}
    float* dvs = reinterpret_cast<float*>(smem + OFF_DV + sd * 1024) + (k >> 1) * 4 + (k & 1);
    uint4* khi_row = reinterpret_cast<uint4*>(dq + DQ_KHI + k * 128);
    uint4* klo_row = reinterpret_cast<uint4*>(dq + DQ_KLO + k * 128);
    if (k < n_valid) {
      const uint32_t* rk0 = reinterpret_cast<const uint32_t*>(smem + OFF_RAW + sr * 2 * RAWB + k * kRowBytes);
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        // block blk of the key row: bytes 34*blk .. 34*blk+33, inside words 8*blk .. 8*blk+8
        const uint32_t* rk = rk0 + 8 * blk;
        const uint32_t* rv = rk + RAWB / 4;
        uint8_t* v_row = dq + (blk ? DQ_V1 : DQ_V0) + (k >> 3) * 512 + (k & 7) * 64;
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = rk[i];
        const unsigned short dkb =
            blk == 0 ? static_cast<unsigned short>(w[0] & 0xFFFFu) : static_cast<unsigned short>(w[0] >> 16);
        const __half2 d2 = __half2half2(__ushort_as_half(dkb));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          // codes 8c .. 8c+7 of this block (block 0 codes start at byte 2, block 1 at byte 36)
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
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = rv[i];
        const unsigned short dvb =
            blk == 0 ? static_cast<unsigned short>(w[0] & 0xFFFFu) : static_cast<unsigned short>(w[0] >> 16);
        dvs[2 * blk] = __half2float(__ushort_as_half(dvb));
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
          *reinterpret_cast<uint4*>(v_row + 16 * (c ^ vsw)) = make_uint4(h2u(q0), h2u(q1), h2u(q2), h2u(q3));
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
      for (int blk = 0; blk < 2; ++blk) {
        uint8_t* v_row = dq + (blk ? DQ_V1 : DQ_V0) + (k >> 3) * 512 + (k & 7) * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(v_row + 16 * c) = z;
        dvs[2 * blk] = 0.0f;
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(bar(B_DEQFULL + sd));
    mbar_arrive(bar(B_RAWEMPTY + sr));
  }
}

__device__ __forceinline__ void mma_role(const ChunkArgs& a, const Unit& u, uint32_t sbase,
                                         uint32_t tmem, Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;   // cycles
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  constexpr uint32_t kIdescQK = idesc_f16_f32(128, BN, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, 32, 0, 1);

  auto issue_qk = [&](int x, int t, int buf) {
    const uint32_t dq = sbase + OFF_DEQ + (t % ND) * DEQ_BYTES;
    const uint32_t d_tmem = tmem + 128u * buf;
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
  // P' of 16 keys sits in 8 consecutive columns: keys 32c..32c+15 of block b at
  // columns 32c + 16b .. +7 and keys 32c+16..32c+31 at 32c + 16b + 8 .. +15.
  auto issue_pv = [&](int x, int t, int buf) {
    const uint32_t dq = sbase + OFF_DEQ + (t % ND) * DEQ_BYTES;
    const uint32_t p_tmem = tmem + 128u * buf;
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const uint32_t vb = dq + (blk ? DQ_V1 : DQ_V0);
        const uint64_t bd = smem_desc(vb + 1024 * kk, 512, 512, kSwizzle64);
        const uint32_t a_col = 32u * (kk >> 1) + 16u * blk + 8u * (kk & 1);
        mma_ts(tmem + T_O + 64 * x + 32 * blk, p_tmem + a_col, bd, kIdescPV, 1u);
      }
    }
  };

  // Event-driven issue: lane 0 polls the barriers without blocking and issues
  // whatever is ready, so one query tile's softmax never waits behind the other's.
  //   QK (in sequence order) once its key tile is dequantised (deq_full) and the
  //      S buffer's previous occupant has had its PV issued (MMAs issued by one
  //      thread execute in issue order, so that PV has read its P' first)
  //   PV_x(t) once tile x has written P'(t)              (p_full[x], phase t)
  //   stage r released (deq_empty) once every query tile has issued PV(r)
  bool ok = wait_bar(bar(B_QFULL), 0, ctl, budget, R_MMA, true);
  if (ok && lane == 0) {
    int pv_next[NQT];
#pragma unroll
    for (int x = 0; x < NQT; ++x) pv_next[x] = 0;
    int occ_x[NSB], occ_t[NSB];   // the (tile, key tile) whose S was last put in each buffer
#pragma unroll
    for (int b = 0; b < NSB; ++b) occ_x[b] = -1, occ_t[b] = 0;
    int qk_t = 0, qk_x = 0, qk_k = 0;   // next QK in sequence order
    auto qk_skip = [&]() {
      while (qk_t < u.T_all && qk_t >= u.T[qk_x]) {
        if (++qk_x == NQT) qk_x = 0, ++qk_t;
      }
    };
    qk_skip();
    int released = 0;
    long long last = clock64();
    int idle = 0;
    while (true) {
      bool progress = false;
      // QK: at most one per pass, in sequence order
      if (qk_t < u.T_all) {
        const int b = qk_k % NSB;
        bool free_buf = true;
#pragma unroll
        for (int bb = 0; bb < NSB; ++bb)
          if (bb == b && occ_x[bb] >= 0) {
#pragma unroll
            for (int y = 0; y < NQT; ++y)
              if (y == occ_x[bb]) free_buf = pv_next[y] > occ_t[bb];
          }
        if (free_buf && mbar_test_wait(bar(B_DEQFULL + qk_t % ND), (qk_t / ND) & 1)) {
          tc_fence_after();
          issue_qk(qk_x, qk_t, b);
          mma_commit(bar(B_SFULL + b));
#pragma unroll
          for (int bb = 0; bb < NSB; ++bb)
            if (bb == b) occ_x[bb] = qk_x, occ_t[bb] = qk_t;
          ++qk_k;
          if (++qk_x == NQT) qk_x = 0, ++qk_t;
          qk_skip();
          progress = true;
        }
      }
      // PV for whichever tile has written its P'
#pragma unroll
      for (int x = 0; x < NQT; ++x) {
        const int tp = pv_next[x];
        if (tp < u.T[x] && mbar_test_wait(bar(B_PFULL + x), tp & 1)) {
          tc_fence_after();
          issue_pv(x, tp, qk_seq(u, x, tp) % NSB);
          mma_commit(bar(B_PVDONE + x));
          pv_next[x] = tp + 1;
          progress = true;
        }
      }
      int lowest = u.T_all;
#pragma unroll
      for (int x = 0; x < NQT; ++x)
        if (pv_next[x] < u.T[x]) lowest = min(lowest, pv_next[x]);
      while (released < lowest) {
        mma_commit(bar(B_DEQEMPTY + released % ND));
        ++released;
        progress = true;
      }
      if (released >= u.T_all) break;   // every PV issued and every stage released
      if (progress) {
        idle = 0;
      } else if (++idle == 1) {
        last = clock64();   // start of this idle stretch
      } else if (idle > 8) {
        if (*reinterpret_cast<volatile uint32_t*>(&ctl->abort) != 0u) break;
        if (static_cast<uint64_t>(clock64() - last) > budget) {
          *reinterpret_cast<volatile uint32_t*>(&ctl->abort) = 1u;
          atomicCAS(&g_status, 0u, 1u | (R_MMA << 8));
          break;
        }
        __nanosleep(32);
      }
    }
  }
  __syncwarp();
  // Never leave with an MMA in flight.
  if (lane == 0) mma_commit(bar(B_DRAIN));
  __syncwarp();
  wait_bar(bar(B_DRAIN), 0, ctl, budget, R_DRAIN, false);
}

// Scores of chunk c (keys 32c .. 32c+31) above `li` are masked out.
__device__ __forceinline__ void mask_chunk(uint32_t (&s)[32], int c, int li) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (32 * c + j > li) s[j] = __float_as_uint(-INFINITY);
}

__device__ __forceinline__ void softmax_role(const ChunkArgs& a, const Unit& u, int x,
                                             uint8_t* smem, uint32_t sbase, uint32_t tmem,
                                             Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;   // cycles
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
  const uint32_t t_o = tmem + lane_off + T_O + 64 * x;

  float m_run = -INFINITY, l_run = 0.0f;
  if (active) {
    m_run = a.m[sidx];
    l_run = a.l[sidx];
  }
  // the O row enters TMEM in two 32-column halves
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t oh[32];
    if (active) {
      const float4* src = reinterpret_cast<const float4*>(a.o + sidx * kHeadDim) + 8 * half;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 p = src[i];
        oh[4 * i + 0] = __float_as_uint(p.x);
        oh[4 * i + 1] = __float_as_uint(p.y);
        oh[4 * i + 2] = __float_as_uint(p.z);
        oh[4 * i + 3] = __float_as_uint(p.w);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) oh[i] = 0u;
    }
    tmem_st32(t_o + 32 * half, oh);
  }
  tmem_wait_st();

  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  const int64_t q_first = a.q_pos0 + u.r0 + x * BM;   // position of the tile's first row
  bool ok = true;
  for (int t = 0; t < T; ++t) {
    const int sd = t % ND;
    const int kq = qk_seq(u, x, t);
    const uint32_t t_s = tmem + lane_off + 128u * (kq % NSB);
    if (!wait_bar(bar(B_SFULL + kq % NSB), (kq / NSB) & 1, ctl, budget, R_SOFTMAX, true) ||
        !wait_bar(bar(B_DEQFULL + sd), (t / ND) & 1, ctl, budget, R_SOFTMAX, true)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const int64_t k0 = static_cast<int64_t>(t) * BN;
    const bool need_mask = (k0 + BN > a.kv_len) || (a.causal && a.kv_start + k0 + BN - 1 > q_first);
    int li = BN - 1;
    if (need_mask) {
      int64_t lim = a.kv_len - 1 - k0;
      if (a.causal) lim = i64min(lim, pos - a.kv_start - k0);
      li = static_cast<int>(i64max(-1, i64min(lim, BN - 1)));
    }
    // pass 1: row max over the 128 scores, each 32-column chunk loaded while
    // the previous one is reduced (tcgen05.wait::ld waits for every load in
    // flight, so a load is issued only once the previous one is consumed)
    float pm[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pm[i] = -INFINITY;
    auto rowmax = [&](uint32_t (&s_)[32], int c) {
      if (need_mask) mask_chunk(s_, c, li);
#pragma unroll
      for (int p = 0; p < 16; ++p)
        pm[p & 7] = max3(pm[p & 7], __uint_as_float(s_[2 * p]), __uint_as_float(s_[2 * p + 1]));
    };
    {
      uint32_t sa[32], sb[32];
      tmem_ld32(t_s, sa);
      tmem_wait_ld(sa);
#pragma unroll 1
      for (int c = 0; c < 4; c += 2) {
        tmem_ld32(t_s + 32 * (c + 1), sb);
        rowmax(sa, c);
        tmem_wait_ld(sb);
        if (c + 2 < 4) tmem_ld32(t_s + 32 * (c + 2), sa);
        rowmax(sb, c + 1);
        if (c + 2 < 4) tmem_wait_ld(sa);
      }
    }
    const float mx = fmaxf(max3(pm[0], pm[1], pm[2]), max3(pm[3], pm[4], max3(pm[5], pm[6], pm[7])));
    const float m_new = fmaxf(m_run, mx * a.scale);
    float alpha = 1.0f, mlog = 0.0f;
    if (m_new != -INFINITY) {
      alpha = ex2_approx((m_run - m_new) * kLog2e);
      mlog = m_new * kLog2e;
    }
    const float2 nm2 = make_float2(-mlog, -mlog);
    const float4* dv = reinterpret_cast<const float4*>(smem + OFF_DV + sd * 1024);
    float2 rs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) rs[i] = make_float2(0.0f, 0.0f);
    // pass 2: weights of one 32-key chunk -> P'_0 at columns 32c..32c+15 and
    // P'_1 at 32c+16..32c+31, i.e. over the chunk's own S columns.  The next
    // chunk is loaded while one is processed (tcgen05.wait::ld waits for every
    // load in flight, so a load is only issued once the previous one is
    // consumed); the loop runs over chunk pairs so the two register buffers
    // keep static names.
    auto weights = [&](const uint32_t (&s_)[32], int c) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {        // 16 keys at a time
        uint32_t pa[8], pb[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = 16 * h + 2 * jj;
          const float2 sv = make_float2(__uint_as_float(s_[j]), __uint_as_float(s_[j + 1]));
          const float2 e = __ffma2_rn(sv, sl2, nm2);
          const float2 bt = make_float2(ex2_approx(e.x), ex2_approx(e.y));
          rs[jj & 3] = __fadd2_rn(rs[jj & 3], bt);
          const float4 d = dv[16 * c + 8 * h + jj];
          const float2 p0 = __fmul2_rn(bt, make_float2(d.x, d.y));
          const float2 p1 = __fmul2_rn(bt, make_float2(d.z, d.w));
          pa[jj] = pack_half2(p0.x, p0.y);
          pb[jj] = pack_half2(p1.x, p1.y);
        }
        tmem_st8(t_s + 32 * c + 8 * h, pa);
        tmem_st8(t_s + 32 * c + 16 + 8 * h, pb);
      }
    };
    {
      uint32_t sa[32], sb[32];
      tmem_ld32(t_s, sa);
      tmem_wait_ld(sa);
#pragma unroll 1
      for (int c = 0; c < 4; c += 2) {
        tmem_ld32(t_s + 32 * (c + 1), sb);
        if (need_mask) mask_chunk(sa, c, li);
        weights(sa, c);
        tmem_wait_ld(sb);
        if (c + 2 < 4) tmem_ld32(t_s + 32 * (c + 2), sa);
        if (need_mask) mask_chunk(sb, c + 1, li);
        weights(sb, c + 1);
        if (c + 2 < 4) tmem_wait_ld(sa);
      }
    }
    if (t > 0) {
      if (!wait_bar(bar(B_PVDONE + x), (t - 1) & 1, ctl, budget, R_SOFTMAX, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
    }
    if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
      const float2 al = make_float2(alpha, alpha);
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t oh[32];
        tmem_ld32(t_o + 32 * half, oh);
        tmem_wait_ld(oh);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 v = __fmul2_rn(make_float2(__uint_as_float(oh[i]), __uint_as_float(oh[i + 1])), al);
          oh[i] = __float_as_uint(v.x);
          oh[i + 1] = __float_as_uint(v.y);
        }
        tmem_st32(t_o + 32 * half, oh);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar(B_PFULL + x));
    const float2 r = __fadd2_rn(__fadd2_rn(rs[0], rs[1]), __fadd2_rn(rs[2], rs[3]));
    l_run = fmaf(l_run, alpha, r.x + r.y);   // same ops per tile with or without chunking
    m_run = m_new;
  }
  if (ok) {
    if (wait_bar(bar(B_PVDONE + x), (T - 1) & 1, ctl, budget, R_SOFTMAX, true)) {
      tc_fence_after();
      if (active) {
        a.m[sidx] = m_run;
        a.l[sidx] = l_run;
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t oh[32];
        tmem_ld32(t_o + 32 * half, oh);
        tmem_wait_ld(oh);
        if (active) {
          float4* dst = reinterpret_cast<float4*>(a.o + sidx * kHeadDim) + 8 * half;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(oh[4 * i]), __uint_as_float(oh[4 * i + 1]),
                                 __uint_as_float(oh[4 * i + 2]), __uint_as_float(oh[4 * i + 3]));
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

  // Register split: the softmax warpgroups hold half an S row plus the P'
  // fragments; the other warpgroups need far fewer registers.
  if (wg < 2) {
    reg_alloc<kRegSoftmax>();
    softmax_role(a, u, wg, smem, sbase, tmem, ctl);
  } else {
    reg_dealloc<kRegOther>();
    if (wg == 2) {
      dequant_role(a, u, smem, sbase, ctl);
    } else if (warp == 12) {
      producer_role(&qmap, a, u, smem, sbase, ctl);
    } else if (warp == 13) {
      mma_role(a, u, sbase, tmem, ctl);
    }
  }

  tc_fence_before();
  __syncthreads();
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
