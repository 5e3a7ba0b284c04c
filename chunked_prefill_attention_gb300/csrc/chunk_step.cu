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
// GB300 design (one CTA = one 128-row query tile of one (batch, head)):
//   warp 8      producer: TMA tensor load of the fp16 Q tile (128B swizzle), and
//               cp.async.bulk of the raw 68-byte-row K and V tiles (8704 B each,
//               contiguous in the head-major planes) into a 3-stage ring.
//   warps 4-7   dequant: one thread per key row.  K = d*q is split exactly into
//               K_hi = fp16(d*q) and K_lo = fp16(d*q - K_hi) (both exact, so
//               Q.K_hi + Q.K_lo reproduces Q.K from exact fp16 operands); V codes
//               are converted to fp16 exactly and the two V block scales are kept
//               aside as fp32.  Tiles are written in the tensor-core layouts:
//               K as K-major 128-byte swizzle, V as MN-major 64-byte swizzle.
//   warp 9      MMA issuer (one thread): S = Q K_hi^T + Q K_lo^T into TMEM
//               (M=128, N=128, 2 x 4 MMAs with K=16); O_b += P'_b V_b for the two
//               32-channel V blocks (M=128, N=32, A = P'_b read from TMEM).
//               S is double-buffered in TMEM so QK of tile t+1 overlaps the
//               softmax of tile t.  Completion is signalled with tcgen05.commit.
//   warps 0-3   softmax: thread i owns query row i (TMEM lane i), loads its S row
//               with tcgen05.ld, masks, takes the row max, forms beta with ex2,
//               folds the V block scale into the fp16 weights P'_b = fp16(beta*d_b)
//               (so the V codes stay exact), writes P' over its S row, rescales its
//               O row in TMEM when the max moved, and keeps m and l in registers.
//               It loads (m, l, O) from HBM before the first tile and stores them
//               back after the last.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,320); 512 allocated.
// Every mbarrier wait is bounded by a wall-clock budget; a wait that runs out
// records the failing role in a per-device status word, and every role then
// leaves its loop, waits (again bounded) for its own copies / MMAs in flight,
// and the CTA frees its TMEM and exits.

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace q8a {

__device__ uint32_t g_status;

namespace {

constexpr int BM = 128;                // query rows per CTA
constexpr int BN = 128;                // keys per tile
constexpr int RAWB = BN * kRowBytes;   // raw bytes of one K (or V) tile: 8704
constexpr int NR = 3;                  // raw ring stages
constexpr int ND = 2;                  // dequantised ring stages
constexpr int kThreads = 320;

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_Q = 0;                            // 128 x 128 B, SW128 K-major
constexpr int DEQ_BYTES = 49152;
constexpr int DQ_KHI = 0, DQ_KLO = 16384, DQ_V0 = 32768, DQ_V1 = 40960;
constexpr int OFF_DEQ = 16384;
constexpr int OFF_DV = OFF_DEQ + ND * DEQ_BYTES;    // fp32 V scales [ND][2][128]
constexpr int OFF_RAW = OFF_DV + ND * 1024;         // [NR][K raw | V raw]
constexpr int OFF_BAR = OFF_RAW + NR * 2 * RAWB;
// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_RAWFULL = 1;                 // NR
constexpr int B_RAWEMPTY = B_RAWFULL + NR;   // NR
constexpr int B_DEQFULL = B_RAWEMPTY + NR;   // ND
constexpr int B_DEQEMPTY = B_DEQFULL + ND;   // ND
constexpr int B_SFULL = B_DEQEMPTY + ND;     // 2
constexpr int B_PFULL = B_SFULL + 2;
constexpr int B_PVDONE = B_PFULL + 1;
constexpr int B_DRAIN = B_PVDONE + 1;
constexpr int NBAR = B_DRAIN + 1;
constexpr int OFF_CTL = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_CTL + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;        // alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_RAW % 16 == 0 && RAWB % 16 == 0, "bulk copy alignment");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_S0 = 0, T_S1 = 128, T_O = 256;

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

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ float sbyte(uint32_t w, int i) {
  return static_cast<float>(static_cast<int8_t>((w >> (8 * i)) & 0xFFu));
}

// Per-CTA work description.
struct Unit {
  int64_t bh, b, h, r0;   // (batch*heads index), query tile start row
  int T;                  // KV tiles to process (0 = nothing)
};

__device__ __forceinline__ Unit make_unit(const ChunkArgs& a) {
  Unit u;
  const int64_t idx = blockIdx.x;
  u.bh = idx / a.n_qtiles;
  const int64_t qt = a.tile0 + (a.n_qtiles - 1 - (idx % a.n_qtiles));   // heavy tiles first
  u.b = u.bh / a.heads;
  u.h = u.bh % a.heads;
  u.r0 = qt * BM;
  const int64_t r_last = i64min(u.r0 + BM - 1, a.n_q - 1);
  int64_t n_vis = a.kv_len;
  if (a.causal) n_vis = i64min(n_vis, a.q_pos0 + r_last - a.kv_start + 1);
  u.T = n_vis > 0 ? static_cast<int>((n_vis + BN - 1) / BN) : 0;
  return u;
}

// ------------------------------------------------------------------ roles --

__device__ void producer_role(const CUtensorMap* qmap, const ChunkArgs& a, const Unit& u,
                              uint8_t* smem, uint32_t sbase, Ctl* ctl) {
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const bool skip_q = (a.inject == 1) && (blockIdx.x == 0);
  if (lane == 0) {
    prefetch_tensormap(qmap);
    if (!skip_q) {
      mbar_arrive_expect_tx(bar(B_QFULL), BM * 128);
      tma_load_3d(sbase + OFF_Q, qmap, bar(B_QFULL), static_cast<int32_t>(u.h * kHeadDim),
                  static_cast<int32_t>(u.r0), static_cast<int32_t>(u.b));
    }
  }
  int last_bulk[NR];
#pragma unroll
  for (int s = 0; s < NR; ++s) last_bulk[s] = -1;

  const uint8_t* kp = a.k8 + u.bh * a.plane_stride;
  const uint8_t* vp = a.v8 + u.bh * a.plane_stride;
  for (int t = 0; t < u.T; ++t) {
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
      last_bulk[sr] = t;
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
    }
  }
  // Never leave with a copy in flight: wait (bounded, even when aborting) for the
  // last bulk copy issued into each stage, and for the Q tile.
#pragma unroll
  for (int s = 0; s < NR; ++s) {
    if (last_bulk[s] >= 0)
      wait_bar(bar(B_RAWFULL + s), (last_bulk[s] / NR) & 1, ctl, a.timeout_ns, R_DRAIN, false);
  }
  if (!skip_q) wait_bar(bar(B_QFULL), 0, ctl, a.timeout_ns, R_DRAIN, false);
}

__device__ void dequant_role(const ChunkArgs& a, const Unit& u, uint8_t* smem, uint32_t sbase,
                             Ctl* ctl) {
  const int k = threadIdx.x - 128;   // key row of the tile owned by this thread
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  for (int t = 0; t < u.T; ++t) {
    const int sr = t % NR, sd = t % ND;
    if (!wait_bar(bar(B_RAWFULL + sr), (t / NR) & 1, ctl, a.timeout_ns, R_DEQUANT, true)) break;
    if (!wait_bar(bar(B_DEQEMPTY + sd), ((t / ND) & 1) ^ 1, ctl, a.timeout_ns, R_DEQUANT, true))
      break;
    const int n_valid = static_cast<int>(i64min(BN, a.kv_len - static_cast<int64_t>(t) * BN));
    uint8_t* dq = smem + OFF_DEQ + sd * DEQ_BYTES;
    float* dvs = reinterpret_cast<float*>(smem + OFF_DV + sd * 1024);
    uint4* khi_row = reinterpret_cast<uint4*>(dq + DQ_KHI + k * 128);
    uint4* klo_row = reinterpret_cast<uint4*>(dq + DQ_KLO + k * 128);
    // V, MN-major 64-byte swizzle: 8-key atoms of 512 B, 64 B per key, 16-byte
    // chunk c stored at c ^ ((k >> 1) & 3)
    uint8_t* v0_row = dq + DQ_V0 + (k >> 3) * 512 + (k & 7) * 64;
    uint8_t* v1_row = dq + DQ_V1 + (k >> 3) * 512 + (k & 7) * 64;
    const int vsw = (k >> 1) & 3;
    if (k < n_valid) {
      const uint32_t* rk = reinterpret_cast<const uint32_t*>(smem + OFF_RAW + sr * 2 * RAWB + k * kRowBytes);
      const uint32_t* rv = rk + RAWB / 4;
      uint32_t w[17];
#pragma unroll
      for (int i = 0; i < 17; ++i) w[i] = rk[i];
      const float dk0 = __half2float(__ushort_as_half(static_cast<unsigned short>(w[0] & 0xFFFFu)));
      const float dk1 = __half2float(__ushort_as_half(static_cast<unsigned short>(w[8] >> 16)));
      // K: 8 chunks of 8 channels; chunk c < 4 from block 0 (bytes 2+8c ..), else block 1
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t c0, c1;
        if (c < 4) {
          c0 = __byte_perm(w[2 * c], w[2 * c + 1], 0x5432);
          c1 = __byte_perm(w[2 * c + 1], w[2 * c + 2], 0x5432);
        } else {
          c0 = w[9 + 2 * (c - 4)];
          c1 = w[10 + 2 * (c - 4)];
        }
        const float d = (c < 4) ? dk0 : dk1;
        float x[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[i] = d * sbyte(c0, i);        // exact in fp32 (11 x 8 significant bits)
          x[4 + i] = d * sbyte(c1, i);
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half h0 = __float2half_rn(x[2 * i]);
          const __half h1 = __float2half_rn(x[2 * i + 1]);
          const __half l0 = __float2half_rn(x[2 * i] - __half2float(h0));
          const __half l1 = __float2half_rn(x[2 * i + 1] - __half2float(h1));
          hi[i] = static_cast<uint32_t>(__half_as_ushort(h0)) |
                  (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
          lo[i] = static_cast<uint32_t>(__half_as_ushort(l0)) |
                  (static_cast<uint32_t>(__half_as_ushort(l1)) << 16);
        }
        const int pc = c ^ (k & 7);     // 128-byte swizzle within the 8-row atom
        khi_row[pc] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        klo_row[pc] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      // V codes -> fp16 (exact), scales aside
      uint32_t vw[17];
#pragma unroll
      for (int i = 0; i < 17; ++i) vw[i] = rv[i];
      dvs[k] = __half2float(__ushort_as_half(static_cast<unsigned short>(vw[0] & 0xFFFFu)));
      dvs[128 + k] = __half2float(__ushort_as_half(static_cast<unsigned short>(vw[8] >> 16)));
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t c0, c1;
        if (c < 4) {
          c0 = __byte_perm(vw[2 * c], vw[2 * c + 1], 0x5432);
          c1 = __byte_perm(vw[2 * c + 1], vw[2 * c + 2], 0x5432);
        } else {
          c0 = vw[9 + 2 * (c - 4)];
          c1 = vw[10 + 2 * (c - 4)];
        }
        uint32_t hv[4];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          hv[i] = pack_half2(sbyte(c0, 2 * i), sbyte(c0, 2 * i + 1));
          hv[2 + i] = pack_half2(sbyte(c1, 2 * i), sbyte(c1, 2 * i + 1));
        }
        uint8_t* vrow = (c < 4) ? v0_row : v1_row;
        const int cc = c & 3;
        *reinterpret_cast<uint4*>(vrow + 16 * (cc ^ vsw)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
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
      dvs[k] = 0.0f;
      dvs[128 + k] = 0.0f;
    }
    fence_proxy_async_smem();
    mbar_arrive(bar(B_DEQFULL + sd));
    mbar_arrive(bar(B_RAWEMPTY + sr));
  }
}

__device__ void mma_role(const ChunkArgs& a, const Unit& u, uint32_t sbase, uint32_t tmem,
                         Ctl* ctl) {
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  constexpr uint32_t kIdescQK = idesc_f16_f32(128, 128, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, 32, 0, 1);

  auto issue_qk = [&](int t) {
    const uint32_t dq = sbase + OFF_DEQ + (t % ND) * DEQ_BYTES;
    const uint32_t d_tmem = tmem + ((t & 1) ? T_S1 : T_S0);
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const uint32_t kb = dq + (part ? DQ_KLO : DQ_KHI);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = smem_desc(sbase + OFF_Q + 32 * kk, 1024, 1024, kSwizzle128);
        const uint64_t bd = smem_desc(kb + 32 * kk, 1024, 1024, kSwizzle128);
        mma_ss(d_tmem, ad, bd, kIdescQK, (part | kk) != 0 ? 1u : 0u);
      }
    }
  };
  auto issue_pv = [&](int t) {
    const uint32_t dq = sbase + OFF_DEQ + (t % ND) * DEQ_BYTES;
    const uint32_t p_tmem = tmem + ((t & 1) ? T_S1 : T_S0);
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const uint32_t vb = dq + (blk ? DQ_V1 : DQ_V0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t bd = smem_desc(vb + 1024 * kk, 512, 512, kSwizzle64);
        mma_ts(tmem + T_O + 32 * blk, p_tmem + 64 * blk + 8 * kk, bd, kIdescPV, 1u);
      }
    }
  };

  bool ok = wait_bar(bar(B_QFULL), 0, ctl, a.timeout_ns, R_MMA, true);
  if (ok) ok = wait_bar(bar(B_DEQFULL + 0), 0, ctl, a.timeout_ns, R_MMA, true);
  if (ok) {
    if (lane == 0) {
      tc_fence_after();
      issue_qk(0);
      mma_commit(bar(B_SFULL + 0));
    }
    __syncwarp();
    for (int t = 0; t < u.T; ++t) {
      if (t + 1 < u.T) {
        if (!wait_bar(bar(B_DEQFULL + (t + 1) % ND), ((t + 1) / ND) & 1, ctl, a.timeout_ns, R_MMA,
                      true))
          break;
        // S buffer (t+1)&1 was last read (as P') by PV(t-1)
        if (t >= 1 && !wait_bar(bar(B_PVDONE), (t - 1) & 1, ctl, a.timeout_ns, R_MMA, true)) break;
        if (lane == 0) {
          tc_fence_after();
          issue_qk(t + 1);
          mma_commit(bar(B_SFULL + ((t + 1) & 1)));
        }
        __syncwarp();
      }
      if (!wait_bar(bar(B_PFULL), t & 1, ctl, a.timeout_ns, R_MMA, true)) break;
      if (lane == 0) {
        tc_fence_after();
        issue_pv(t);
        mma_commit(bar(B_PVDONE));
        mma_commit(bar(B_DEQEMPTY + t % ND));
      }
      __syncwarp();
    }
  }
  // Never leave with an MMA in flight.
  if (lane == 0) mma_commit(bar(B_DRAIN));
  __syncwarp();
  wait_bar(bar(B_DRAIN), 0, ctl, a.timeout_ns, R_DRAIN, false);
}

__device__ void softmax_role(const ChunkArgs& a, const Unit& u, uint8_t* smem, uint32_t sbase,
                             uint32_t tmem, Ctl* ctl) {
  const int row = threadIdx.x;        // 0..127 == TMEM lane
  const int warp = row >> 5;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };

  const int64_t rg = u.r0 + row;
  const int64_t pos = a.q_pos0 + rg;
  const bool active = rg < a.n_q && (!a.causal || pos >= a.kv_start);
  const int64_t sidx = u.bh * a.n_q + rg;

  float m_run = -INFINITY, l_run = 0.0f;
  {
    uint32_t oa[32], ob[32];
    if (active) {
      m_run = a.m[sidx];
      l_run = a.l[sidx];
      const float4* src = reinterpret_cast<const float4*>(a.o + sidx * kHeadDim);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 x = src[i];
        oa[4 * i + 0] = __float_as_uint(x.x);
        oa[4 * i + 1] = __float_as_uint(x.y);
        oa[4 * i + 2] = __float_as_uint(x.z);
        oa[4 * i + 3] = __float_as_uint(x.w);
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
    tmem_st32(tmem + lane_off + T_O, oa);
    tmem_st32(tmem + lane_off + T_O + 32, ob);
    tmem_wait_st();
  }

  const float sl2 = a.scale_log2;
  bool ok = true;
  for (int t = 0; t < u.T; ++t) {
    const int sd = t % ND;
    const uint32_t s_tmem = tmem + lane_off + ((t & 1) ? T_S1 : T_S0);
    if (!wait_bar(bar(B_SFULL + (t & 1)), (t >> 1) & 1, ctl, a.timeout_ns, R_SOFTMAX, true) ||
        !wait_bar(bar(B_DEQFULL + sd), (t / ND) & 1, ctl, a.timeout_ns, R_SOFTMAX, true)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t s[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + 32 * c, s[c]);
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_wait_ld(s[c]);

    const int64_t k0 = static_cast<int64_t>(t) * BN;
    const bool need_mask = (k0 + BN > a.kv_len) ||
                           (a.causal && a.kv_start + k0 + BN - 1 > a.q_pos0 + u.r0);
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
      for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(s[c][j]));
    const float m_new = fmaxf(m_run, mx * a.scale);
    float alpha = 1.0f, mlog = 0.0f;
    if (m_new != -INFINITY) {
      alpha = ex2_approx((m_run - m_new) * kLog2e);
      mlog = m_new * kLog2e;
    }
    const float2* dv0 = reinterpret_cast<const float2*>(smem + OFF_DV + sd * 1024);
    const float2* dv1 = dv0 + 64;
    float rowsum = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t pa[16], pb[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const float b0 = ex2_approx(fmaf(__uint_as_float(s[c][2 * jj]), sl2, -mlog));
        const float b1 = ex2_approx(fmaf(__uint_as_float(s[c][2 * jj + 1]), sl2, -mlog));
        rowsum += b0 + b1;
        const float2 d0 = dv0[16 * c + jj];
        const float2 d1 = dv1[16 * c + jj];
        pa[jj] = pack_half2(b0 * d0.x, b1 * d0.y);
        pb[jj] = pack_half2(b0 * d1.x, b1 * d1.y);
      }
      tmem_st16(s_tmem + 16 * c, pa);
      tmem_st16(s_tmem + 64 + 16 * c, pb);
    }
    if (t > 0) {
      if (!wait_bar(bar(B_PVDONE), (t - 1) & 1, ctl, a.timeout_ns, R_SOFTMAX, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
    }
    if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
      uint32_t oa[32], ob[32];
      tmem_ld32(tmem + lane_off + T_O, oa);
      tmem_ld32(tmem + lane_off + T_O + 32, ob);
      tmem_wait_ld(oa);
      tmem_wait_ld(ob);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        oa[i] = __float_as_uint(__uint_as_float(oa[i]) * alpha);
        ob[i] = __float_as_uint(__uint_as_float(ob[i]) * alpha);
      }
      tmem_st32(tmem + lane_off + T_O, oa);
      tmem_st32(tmem + lane_off + T_O + 32, ob);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar(B_PFULL));
    l_run = l_run * alpha + rowsum;
    m_run = m_new;
  }
  if (ok && u.T > 0) {
    if (wait_bar(bar(B_PVDONE), (u.T - 1) & 1, ctl, a.timeout_ns, R_SOFTMAX, true)) {
      tc_fence_after();
      uint32_t oa[32], ob[32];
      tmem_ld32(tmem + lane_off + T_O, oa);
      tmem_ld32(tmem + lane_off + T_O + 32, ob);
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

  const Unit u = make_unit(a);
  if (u.T == 0) return;   // uniform over the CTA: no visible key for this tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t count = 1;
      if (i >= B_RAWEMPTY && i < B_RAWEMPTY + NR) count = 128;   // dequant threads
      if (i >= B_DEQFULL && i < B_DEQFULL + ND) count = 128;     // dequant threads
      if (i == B_PFULL) count = 128;                             // softmax threads
      mbar_init(sbase + OFF_BAR + 8u * i, count);
    }
    ctl->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(sbase + OFF_CTL, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp < 4) {
    softmax_role(a, u, smem, sbase, tmem, ctl);
  } else if (warp < 8) {
    dequant_role(a, u, smem, sbase, ctl);
  } else if (warp == 8) {
    producer_role(&qmap, a, u, smem, sbase, ctl);
  } else {
    mma_role(a, u, sbase, tmem, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
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
  const int64_t blocks = static_cast<int64_t>(args.n_qtiles) * args.bh;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  chunk_step_kernel<<<static_cast<unsigned>(blocks), kThreads, SMEM_BYTES, stream>>>(qmap, args);
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
