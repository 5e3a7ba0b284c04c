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
//   WG0, WG1   softmax of tile A / tile B.  Thread i owns query row i of its
//              tile (TMEM lane i).  Per key tile it loads its whole 128-score S
//              row from TMEM into registers, masks diagonal and tail tiles,
//              takes the row max, forms beta = ex2(S*c - m*log2e) with packed
//              fp32x2 arithmetic against the reference m, sums beta in fp32
//              (with the tile max's weight as fp16 rounds it) and writes
//              P = fp16(beta) over the first 64 columns of its S row, in two
//              halves (keys 0-63, then 64-127) announced on separate barriers
//              so that the first half of PV runs while the second half is
//              computed.  The reference m moves to the tile max only when that
//              exceeds it by more than 8 ln 2 (weights stay below 2^8); a warp
//              rescales its O rows in TMEM, before the first half is
//              announced, only when the reference of one of its rows moved.
//   WG2        dequant, one thread per key row.  K = d*q and V = d*q are each
//              split exactly into an fp16 high part fp16(d*q) and an fp16
//              residual fp16(d*q - high) (half2 multiply / fma on codes
//              converted by the exponent-bias trick), so every tensor-core
//              operand is exact.  The four 128 x 64 fp16 tiles (K_hi, K_lo,
//              V_hi, V_lo) are written with the 128-byte swizzle, one key per
//              128-byte row.  The K and V halves of a stage are filled and
//              released on separate barriers: K is free once its QKs are done,
//              before the softmax of that key tile starts.
//   WG3        warp 12: producer -- TMA tensor loads of the two fp16 Q tiles and
//              cp.async.bulk of the raw 68-byte-row K/V tiles (8704 B each,
//              contiguous in the head-major planes) into a 2-stage ring;
//              warp 13: MMA issuer (the whole warp runs the issue loop, so the
//              descriptors stay warp-uniform; one elected lane issues).
// MMAs (M=128, K=16, N=128 throughout: N=128 is the narrowest shape that runs
// at the tensor pipe's full rate on this part):
//   S_X  = Q_X K_hi^T + Q_X K_lo^T          8 instructions, both operands in smem
//   O_X += P_X [V_hi | V_lo]                8 instructions, P read from TMEM,
//          the two 64-column halves of O_X accumulate P.V_hi and P.V_lo and
//          are added when the state is written back.
// Issue order (ping-pong): PV_A(t), QK_A(t+1), PV_B(t), QK_B(t+1), ... so the
// tensor pipe works on one tile while the other tile's softmax runs.
// Paired mode (one 128-row query tile, no causal mask, e.g. burst
// verification): both pipelines take the same rows, A the even and B the odd
// key tiles, and A merges B's state at the end, so the ping-pong still has two
// chains to interleave.  Grouped-query attention only changes the K/V plane a
// CTA streams: query head h reads plane h / (heads / kv_heads).
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
// Every mbarrier wait is bounded by a budget; a wait that runs out records the
// failing role in a per-device status word, every role then leaves its loop,
// waits (again bounded) for its own copies / MMAs in flight, and the CTA frees
// its TMEM and exits.

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
constexpr int ND = 2;                  // dequantised ring stages
constexpr int kThreads = 512;
constexpr int kRegSoftmax = 184;       // setmaxnreg split: 2 x 128 x 184 + 2 x 128 x 72 = 65536
constexpr int kRegOther = 72;
static_assert(2 * 128 * kRegSoftmax + 2 * 128 * kRegOther == 65536, "register split");

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_Q = 0;                               // NQT x (128 x 128 B), SW128
constexpr int DQ_KHI = 0, DQ_KLO = 16384, DQ_VHI = 32768, DQ_VLO = 49152;
constexpr int DEQ_BYTES = 65536;                       // four 128 x 128 B tiles
constexpr int OFF_DEQ = NQT * 16384;
constexpr int OFF_RAW = OFF_DEQ + ND * DEQ_BYTES;      // [NR][K raw | V raw]
constexpr int OFF_BAR = OFF_RAW + NR * 2 * RAWB;
// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_RAWFULL = 1;                 // NR
constexpr int B_RAWEMPTY = B_RAWFULL + NR;   // NR
// K and V of a dequantised stage are filled and released separately: the K
// half is free once the QKs reading it have completed (which is early: the
// softmax of that key tile has not started yet), the V half once its PVs have.
constexpr int B_KFULL = B_RAWEMPTY + NR;     // ND
constexpr int B_KEMPTY = B_KFULL + ND;       // ND
constexpr int B_VFULL = B_KEMPTY + ND;       // ND
constexpr int B_VEMPTY = B_VFULL + ND;       // ND
constexpr int B_SFULL = B_VEMPTY + ND;       // NQT
constexpr int B_PFULL = B_SFULL + NQT;       // 2 x NQT: P_x keys 0-63, then keys 64-127
constexpr int B_ODONE = B_PFULL + 2 * NQT;   // NQT
constexpr int B_MERGE = B_ODONE + NQT;       // paired mode: tile B's final (m, l) published
constexpr int B_DRAIN = B_MERGE + 1;
constexpr int NBAR = B_DRAIN + 1;
constexpr int OFF_CTL = (OFF_BAR + NBAR * 8 + 15) / 16 * 16;
constexpr int CTL_BYTES = 32;                // struct Ctl, padded
constexpr int OFF_XCH = OFF_CTL + CTL_BYTES;  // paired mode: 128 x float4 {m, l, ok, -} of tile B
constexpr int SMEM_USED = OFF_XCH + BM * 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;           // alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_RAW % 16 == 0 && RAWB % 16 == 0, "bulk copy alignment");
static_assert(OFF_DEQ % 1024 == 0 && DEQ_BYTES % 1024 == 0, "swizzle atom alignment");
static_assert(OFF_BAR % 8 == 0 && OFF_XCH % 16 == 0, "mbarrier and 16-byte exchange-slot alignment");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_S = 0;      // + 128 * tile
constexpr uint32_t T_O = 256;    // + 128 * tile; high half at +0, residual half at +64

constexpr float kLog2e = 1.4426950408889634f;
// The softmax reference m moves only when a tile's max exceeds it by more than
// 8 ln 2, so the weights stay below 2^8 and O is rescaled only then.
constexpr float kLazyNat = 5.545177444479562f;

// l sums the fp32 weights beta, P holds them rounded to fp16.  For the tile's
// largest score (raw score mx) this returns fp16(beta) - beta, which l adds, so
// that a row dominated by one key divides that key's term by exactly the
// weight P gave it.  0 when every key of the tile is masked.
__device__ __forceinline__ float p_max_correction(float mx, float scale_log2, float mlog) {
  if (mx == -INFINITY) return 0.0f;
  const float bm = ex2_approx(fmaf(mx, scale_log2, -mlog));   // as the P loop forms it
  return __half2float(__float2half_rn(bm)) - bm;
}

// role ids recorded in the status word when a wait runs out
enum : uint32_t { R_SOFTMAX = 1, R_DEQUANT = 2, R_PRODUCER = 3, R_MMA = 4, R_DRAIN = 5 };

struct Ctl {
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(Ctl) <= CTL_BYTES, "control block");

__device__ __forceinline__ bool budget_ran_out(Ctl* ctl, long long t0, uint64_t budget_cycles,
                                               uint32_t role) {
  if (static_cast<uint64_t>(clock64() - t0) > budget_cycles) {
    *reinterpret_cast<volatile uint32_t*>(&ctl->abort) = 1u;
    atomicCAS(&g_status, 0u, 1u | (role << 8));
    return true;
  }
  return false;
}

// A CTA whose wait ran out copies the status word (the first failure of the
// device) into the host-mapped word, which q8a_status reads without any
// synchronisation.  Called once per CTA after its roles have stopped, so the
// waits themselves only set the abort flag and the device word.
__device__ __forceinline__ void publish_failure(uint32_t* host_word) {
  const uint32_t code = *reinterpret_cast<volatile uint32_t*>(&g_status);
  *reinterpret_cast<volatile uint32_t*>(host_word) = code ? code : 1u;
  __threadfence_system();
}

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
      } else if (budget_ran_out(ctl, t0, budget_cycles, role)) {
        stop = 2;
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

// tcgen05.ld 32x32b.x32 into registers r[O .. O+31] of a 128-register row.
template <int O>
__device__ __forceinline__ void tmem_ld32_at(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : Q8A_R8(r, O + 0), Q8A_R8(r, O + 8), Q8A_R8(r, O + 16), Q8A_R8(r, O + 24)
      : "r"(taddr));
}
// Ties r[O .. O+31] to a tcgen05.wait::ld (the first such wait does the waiting).
template <int O>
__device__ __forceinline__ void tmem_wait_ld_at(uint32_t (&r)[128]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : Q8A_M8(r, O + 0), Q8A_M8(r, O + 8), Q8A_M8(r, O + 16), Q8A_M8(r, O + 24)::"memory");
}
template <int O>
__device__ __forceinline__ void tmem_st32_at(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      Q8A_W8(r, O + 0), Q8A_W8(r, O + 8), Q8A_W8(r, O + 16), Q8A_W8(r, O + 24)
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

// The order of a launch's CTAs over (b, h) units and query units.  The (b, h)
// units are taken in groups of `group` (ChunkArgs::head_group); within a group
// the CTAs run the heaviest query units first, the group's (b, h) fastest.  So
// the longest CTAs of a group start together and the launch ends on the
// lightest ones (a near-even finish across the SMs), while the K/V planes read
// at any one time are those of one group, few enough to stay in L2 between the
// group's CTAs.  Every idx < units * n_bh gets a distinct (bh, qu).
__device__ __forceinline__ void cta_order(int64_t idx, int64_t units, int64_t n_bh, int64_t group, int64_t& bh,
                                          int64_t& qu) {
  const int64_t full = n_bh / group;   // complete groups
  const int64_t g = idx / (units * group);
  const int64_t gs = g < full ? group : n_bh - full * group;   // heads in this group
  const int64_t w = idx - g * units * group;
  bh = g * group + w % gs;
  qu = units - 1 - w / gs;
}

// The key range and state this CTA works on: the whole chunk and the state,
// or, in the split form, one key range and its partial state.
struct Range {
  int64_t kv_len, kv_start;
  const uint8_t* k8;
  const uint8_t* v8;
  float* m;
  float* l;
  float* o;
  bool fresh;   // start from the empty state instead of reading m, l, o
};

__device__ __forceinline__ Range make_range(const ChunkArgs& a) {
  Range r;
  r.kv_len = a.kv_len;
  r.kv_start = a.kv_start;
  r.k8 = a.k8;
  r.v8 = a.v8;
  r.m = a.m;
  r.l = a.l;
  r.o = a.o;
  r.fresh = false;
  if (a.split_keys > 0) {
    const int64_t off = static_cast<int64_t>(blockIdx.y) * a.split_keys;
    // state rows (batch, query head, query row); with packing bh counts K/V heads
    const int64_t rows = a.pack ? static_cast<int64_t>(a.bh / a.kv_heads) * a.heads * a.n_q
                                : static_cast<int64_t>(a.bh) * a.n_q;
    r.kv_len = i64min(a.split_keys, a.kv_len - off);
    r.kv_start = a.kv_start + off;
    r.k8 = a.k8 + off * kRowBytes;
    r.v8 = a.v8 + off * kRowBytes;
    r.m = a.part_m + blockIdx.y * rows;
    r.l = a.part_l + blockIdx.y * rows;
    r.o = a.part_o + blockIdx.y * rows * kHeadDim;
    r.fresh = true;
  }
  return r;
}

// Per-CTA work description.
//
// Paired mode (a.pair: one 128-row query tile per (b, h), no causal mask, as in
// burst verification): both softmax pipelines work on the same query rows, tile
// A on the even key tiles of the range and tile B on the odd ones, each with its
// own running state; tile A merges B's state into its own at the end.  The two
// pipelines then overlap exactly as two query tiles do in prefill, instead of
// one pipeline waiting out its own softmax -> PV -> QK chain.
struct Unit {
  int64_t bh, b, h, r0;   // (batch*heads index), first row of tile A
  int T[NQT];             // key tiles each query tile processes (0 = inactive)
  int T_all;              // key tiles streamed through the CTA
};

// Query row offset of tile x from u.r0, and the key tile of tile x's j-th step.
__device__ __forceinline__ int64_t tile_row0(const ChunkArgs& a, int x) {
  return a.pair ? 0 : static_cast<int64_t>(x) * BM;
}
__device__ __forceinline__ int key_tile(const ChunkArgs& a, int x, int j) {
  return a.pair ? 2 * j + x : j;
}

__device__ __forceinline__ Unit make_unit(const ChunkArgs& a, const Range& kr) {
  Unit u;
  int64_t bh, qu;   // n_qtiles counts 256-row units here
  cta_order(blockIdx.x, a.n_qtiles, a.bh, a.head_group, bh, qu);
  u.bh = bh;
  // u.h: the query head, or with packing the K/V head of the unit
  const int32_t nh = a.pack ? a.kv_heads : a.heads;
  u.b = u.bh / nh;
  u.h = u.bh % nh;
  u.r0 = static_cast<int64_t>(a.tile0) * BM + qu * (NQT * BM);
  u.T_all = 0;
  if (a.pair) {
    const int tiles = kr.kv_len > 0 ? static_cast<int>((kr.kv_len + BN - 1) / BN) : 0;
    u.T[0] = (tiles + 1) / 2;
    u.T[1] = tiles / 2;
    u.T_all = tiles;
    return u;
  }
  const int64_t n_rows = a.pack ? a.n_q * a.pack : a.n_q;   // rows of the tile space
#pragma unroll
  for (int x = 0; x < NQT; ++x) {
    const int64_t rx = u.r0 + x * BM;
    u.T[x] = 0;
    if (rx < n_rows) {
      const int64_t r_last = i64min(rx + BM - 1, n_rows - 1);
      const int64_t last_pos = a.q_pos0 + (a.pack ? r_last / a.pack : r_last);
      int64_t n_vis = kr.kv_len;
      if (a.causal) n_vis = i64min(n_vis, last_pos - kr.kv_start + 1);
      u.T[x] = n_vis > 0 ? static_cast<int>((n_vis + BN - 1) / BN) : 0;
    }
    u.T_all = max(u.T_all, u.T[x]);
  }
  return u;
}

// ------------------------------------------------------------------ roles --

// kKeep: the pipelined prefill's form (ChunkArgs::l2_keep_kv), a separate
// instantiation so that the other launches run exactly the plain code.
template <bool kKeep>
__device__ __forceinline__ void producer_role(const CUtensorMap* qmap, const ChunkArgs& a,
                                              const Range& kr, const Unit& u, uint8_t* smem,
                                              uint32_t sbase, Ctl* ctl) {
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
        if (u.T[x] > 0) {
          if (a.pack)   // box {64 channels, pack heads, 128 / pack query rows}
            tma_load_3d(sbase + OFF_Q + x * 16384, qmap, bar(B_QFULL), 0,
                        static_cast<int32_t>(u.h * a.pack),
                        static_cast<int32_t>(u.b * a.n_q + (u.r0 + tile_row0(a, x)) / a.pack));
          else if (kKeep)   // Q is read once: evict-first, the chunk's K/V stay in L2
            tma_load_3d_hint(sbase + OFF_Q + x * 16384, qmap, bar(B_QFULL),
                             static_cast<int32_t>(u.h * kHeadDim), static_cast<int32_t>(u.r0 + tile_row0(a, x)),
                             static_cast<int32_t>(u.b), l2_evict_first_policy());
          else
            tma_load_3d(sbase + OFF_Q + x * 16384, qmap, bar(B_QFULL),
                        static_cast<int32_t>(u.h * kHeadDim), static_cast<int32_t>(u.r0 + tile_row0(a, x)),
                        static_cast<int32_t>(u.b));
        }
    }
  }
  int last_bulk[NR];
#pragma unroll
  for (int s = 0; s < NR; ++s) last_bulk[s] = -1;

  // K/V plane of this query head (grouped-query attention: heads / kv_heads
  // query heads share one plane)
  const int64_t kv_plane = a.pack ? u.b * a.kv_heads + u.h : u.b * a.kv_heads + u.h / (a.heads / a.kv_heads);
  const uint8_t* kp = kr.k8 + kv_plane * a.plane_stride;
  const uint8_t* vp = kr.v8 + kv_plane * a.plane_stride;
  for (int t = 0; t < u.T_all; ++t) {
    const int sr = t % NR;
    if (!wait_bar(bar(B_RAWEMPTY + sr), ((t / NR) & 1) ^ 1, ctl, budget, R_PRODUCER, true))
      break;
    const int64_t k0 = static_cast<int64_t>(t) * BN;
    const int n = static_cast<int>(i64min(BN, kr.kv_len - k0));
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

// One 34-byte block of one key row (codes in words w[0..8] of the raw row,
// block `blk`) -> 4 high and 4 residual 16-byte chunks of the swizzled tiles.
__device__ __forceinline__ void dequant_block(const uint32_t (&w)[9], int blk, uint8_t* hi_row,
                                              uint8_t* lo_row, int sw) {
  const unsigned short db =
      blk == 0 ? static_cast<unsigned short>(w[0] & 0xFFFFu) : static_cast<unsigned short>(w[0] >> 16);
  const __half2 d2 = __half2half2(__ushort_as_half(db));
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
    const int pc = ((4 * blk + c) ^ sw) * 16;
    *reinterpret_cast<uint4*>(hi_row + pc) = make_uint4(h2u(h0), h2u(h1), h2u(h2), h2u(h3));
    *reinterpret_cast<uint4*>(lo_row + pc) = make_uint4(h2u(l0), h2u(l1), h2u(l2), h2u(l3));
  }
}

__device__ __forceinline__ void dequant_role(const ChunkArgs& a, const Range& kr, const Unit& u,
                                             uint8_t* smem, uint32_t sbase, Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;   // cycles
  const int k = threadIdx.x - 256;   // key row of the tile
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int sw = k & 7;              // 128-byte swizzle phase of this row
  const int row_off = (k >> 3) * 1024 + (k & 7) * 128;
  for (int t = 0; t < u.T_all; ++t) {
    const int sr = t % NR, sd = t % ND;
    const uint32_t fill = (t / ND) & 1;
    if (!wait_bar(bar(B_RAWFULL + sr), (t / NR) & 1, ctl, budget, R_DEQUANT, true)) break;
    const int n_valid = static_cast<int>(i64min(BN, kr.kv_len - static_cast<int64_t>(t) * BN));
    uint8_t* dq = smem + OFF_DEQ + sd * DEQ_BYTES + row_off;
    bool stop = false;
#pragma unroll 1
    for (int tensor = 0; tensor < 2; ++tensor) {   // K, then V
      if (!wait_bar(bar((tensor ? B_VEMPTY : B_KEMPTY) + sd), fill ^ 1, ctl, budget, R_DEQUANT,
                    true)) {
        stop = true;
        break;
      }
      uint8_t* hi_row = dq + (tensor ? DQ_VHI : DQ_KHI);
      uint8_t* lo_row = dq + (tensor ? DQ_VLO : DQ_KLO);
      if (k < n_valid) {
        const uint32_t* raw = reinterpret_cast<const uint32_t*>(
            smem + OFF_RAW + sr * 2 * RAWB + tensor * RAWB + k * kRowBytes);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          uint32_t w[9];
#pragma unroll
          for (int i = 0; i < 9; ++i) w[i] = raw[8 * blk + i];
          dequant_block(w, blk, hi_row, lo_row, sw);
        }
      } else {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(hi_row + 16 * c) = z;
          *reinterpret_cast<uint4*>(lo_row + 16 * c) = z;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar((tensor ? B_VFULL : B_KFULL) + sd));
    }
    if (stop) break;
    mbar_arrive(bar(B_RAWEMPTY + sr));
  }
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// The whole warp runs the issue loop, so every descriptor and TMEM address is
// warp-uniform and stays in uniform registers; one elected lane issues the
// MMAs and commits (always the same lane: commits track its own MMAs).
__device__ __forceinline__ void mma_role(const ChunkArgs& a, const Unit& u, uint32_t sbase,
                                         uint32_t tmem, Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;   // cycles
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  constexpr uint32_t kIdescQK = idesc_f16_f32(128, BN, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, 128, 0, 1);
  const bool leader = elect_one();

  // Descriptor start addresses advance in 16-byte units in the low bits (no
  // carry: shared addresses stay below 256 KB).
  //   S_x = Q_x K_hi^T + Q_x K_lo^T: K-major operands, 4 k-steps of 16 channels
  //   (32 bytes inside the 128-byte swizzled rows).
  //   O_x += P_x [V_hi | V_lo]: V tiles MN-major (channels contiguous); the two
  //   64-channel halves of N are 16 KB apart (leading byte offset) and each
  //   k-step covers 16 keys = two 8-row swizzle atoms (stride byte offset 1 KB,
  //   2 KB per k-step).  P of keys 16kk .. 16kk+15 sits in TMEM columns
  //   8kk .. 8kk+7 of S_x.
  const uint64_t qdesc0 = smem_desc(sbase + OFF_Q, 1024, 1024, kSwizzle128);
  const uint64_t kdesc0 = smem_desc(sbase + OFF_DEQ + DQ_KHI, 1024, 1024, kSwizzle128);
  const uint64_t vdesc0 = smem_desc(sbase + OFF_DEQ + DQ_VHI, DQ_VLO - DQ_VHI, 1024, kSwizzle128);
  // stage sd of the dequantised ring
  auto issue_qk = [&](int x, int sd) {
    const uint64_t qd = qdesc0 + static_cast<uint64_t>(x * (16384 >> 4));
    const uint64_t kd = kdesc0 + static_cast<uint64_t>(sd * (DEQ_BYTES >> 4));
    const uint32_t d = tmem + T_S + 128u * x;
    if (leader) {
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(d, qd + 2 * kk, kd + part * (16384 >> 4) + 2 * kk, kIdescQK, (part | kk) != 0 ? 1u : 0u);
    }
  };
  // half h covers keys 64h .. 64h+63 (k-steps 4h .. 4h+3)
  auto issue_pv = [&](int x, int sd, int h) {
    const uint64_t vd = vdesc0 + static_cast<uint64_t>(sd * (DEQ_BYTES >> 4));
    const uint32_t o = tmem + T_O + 128u * x;
    const uint32_t p = tmem + T_S + 128u * x;
    if (leader) {
#pragma unroll
      for (int kk = 4 * h; kk < 4 * h + 4; ++kk) mma_ts(o, p + 8u * kk, vd + 128 * kk, kIdescPV, 1u);
    }
  };
  auto commit = [&](int b) {
    if (leader) mma_commit(bar(b));
  };

  // Tile x's j-th key tile sits in stage kt % ND of the ring, filled for the
  // (kt / ND)-th time.  In prefill both tiles read every key tile, so a
  // stage half is released after tile B's MMA on it; in paired mode each key
  // tile has one reader.
  const bool pair = a.pair != 0;
  auto stage = [&](int x, int j) { return key_tile(a, x, j) % ND; };
  auto fill = [&](int x, int j) { return static_cast<uint32_t>((key_tile(a, x, j) / ND) & 1); };

  bool ok = wait_bar(bar(B_QFULL), 0, ctl, budget, R_MMA, true);
  if (ok) {
#pragma unroll
    for (int x = 0; x < NQT; ++x)
      if (ok && u.T[x] > 0) {
        ok = wait_bar(bar(B_KFULL + stage(x, 0)), fill(x, 0), ctl, budget, R_MMA, true);
        if (!ok) break;
        tc_fence_after();
        issue_qk(x, stage(x, 0));
        commit(B_SFULL + x);
        if (pair) commit(B_KEMPTY + stage(x, 0));
      }
    if (ok && !pair) commit(B_KEMPTY + 0);   // every reader of K(0) issued
  }
  const int steps = pair ? u.T[0] : u.T_all;
  for (int j = 0; ok && j < steps; ++j) {
#pragma unroll
    for (int x = 0; x < NQT; ++x) {
      if (j < u.T[x]) {
        const int sd = stage(x, j);
        if (!wait_bar(bar(B_VFULL + sd), fill(x, j), ctl, budget, R_MMA, true) ||
            !wait_bar(bar(B_PFULL + 2 * x), j & 1, ctl, budget, R_MMA, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(x, sd, 0);
        if (!wait_bar(bar(B_PFULL + 2 * x + 1), j & 1, ctl, budget, R_MMA, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(x, sd, 1);
        if (j == u.T[x] - 1) commit(B_ODONE + x);
        if (pair) commit(B_VEMPTY + sd);
      }
      if (!pair && x == NQT - 1) commit(B_VEMPTY + j % ND);   // every reader of V(j) issued
      if (j + 1 < u.T[x]) {
        const int sd = stage(x, j + 1);
        if (!wait_bar(bar(B_KFULL + sd), fill(x, j + 1), ctl, budget, R_MMA, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_qk(x, sd);
        commit(B_SFULL + x);
        if (pair) commit(B_KEMPTY + sd);
      }
      if (!pair && x == NQT - 1 && j + 1 < u.T_all) commit(B_KEMPTY + (j + 1) % ND);
    }
  }
  // Never leave with an MMA in flight.
  commit(B_DRAIN);
  __syncwarp();
  wait_bar(bar(B_DRAIN), 0, ctl, budget, R_DRAIN, false);
}

// Paired mode: fold tile B's final state (m_b, l_b; O at TMEM address t_ob)
// into tile A's (m_a, l_a; O at t_oa) and write the result -- the chunk
// recurrence applied to two partial states over disjoint keys.  The weight of
// the state holding the larger reference m is exactly 1.  O is the sum of each
// tile's high and residual halves.
__device__ __forceinline__ void merge_pair_out(const Range& kr, int64_t sidx, bool active,
                                               float m_a, float l_a, float m_b, float l_b,
                                               uint32_t t_oa, uint32_t t_ob) {
  const float m = fmaxf(m_a, m_b);
  const float wa = (m_a == m) ? 1.0f : (m_a == -INFINITY ? 0.0f : ex2_approx((m_a - m) * kLog2e));
  const float wb = (m_b == m) ? 1.0f : (m_b == -INFINITY ? 0.0f : ex2_approx((m_b - m) * kLog2e));
  if (active) {
    kr.m[sidx] = m;
    kr.l[sidx] = fmaf(wa, l_a, wb * l_b);
  }
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint32_t ah[32], al[32], bh[32], bl[32];
    tmem_ld32(t_oa + 32 * half, ah);
    tmem_ld32(t_oa + 64 + 32 * half, al);
    tmem_ld32(t_ob + 32 * half, bh);
    tmem_ld32(t_ob + 64 + 32 * half, bl);
    tmem_wait_ld(ah);
    tmem_wait_ld(al);
    tmem_wait_ld(bh);
    tmem_wait_ld(bl);
    if (active) {
      float4* dst = reinterpret_cast<float4*>(kr.o + sidx * kHeadDim) + 8 * half;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 4 * i + e;
          const float oa = __uint_as_float(ah[c]) + __uint_as_float(al[c]);
          const float ob = __uint_as_float(bh[c]) + __uint_as_float(bl[c]);
          v[e] = fmaf(wa, oa, wb * ob);
        }
        dst[i] = make_float4(v[0], v[1], v[2], v[3]);
      }
    }
  }
}

template <bool kKeep>
__device__ __forceinline__ void softmax_role(const ChunkArgs& a, const Range& kr, const Unit& u, int x,
                                             uint8_t* smem, uint32_t sbase, uint32_t tmem, Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;   // cycles
  const int row = threadIdx.x & 127;       // TMEM lane
  const int wq = (threadIdx.x >> 5) & 3;   // warp's lane quarter
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int T = u.T[x];
  if (T == 0) return;

  // this thread's row of the tile space; with packing a (query row, query
  // head) pair of the unit's K/V group
  const int64_t pr = u.r0 + tile_row0(a, x) + row;
  const int64_t rg = a.pack ? pr / a.pack : pr;   // query row
  const int64_t pos = a.q_pos0 + rg;
  const bool active = rg < a.n_q && (!a.causal || pos >= kr.kv_start);
  const int64_t sidx = a.pack ? (u.b * a.heads + u.h * a.pack + pr % a.pack) * a.n_q + rg : u.bh * a.n_q + rg;
  const uint32_t t_s = tmem + lane_off + T_S + 128u * x;
  const uint32_t t_o = tmem + lane_off + T_O + 128u * x;

  // in paired mode tile B starts from the empty state and tile A merges it in
  const bool fresh = kr.fresh || (a.pair && x == 1);
  const bool pair_merge = a.pair && u.T[1] > 0;
  float m_run = -INFINITY, l_run = 0.0f;
  if (active && !fresh) {
    if (kKeep) {   // the state is read once: evict-first, the chunk's K/V stay in L2
      const uint64_t pol = l2_evict_first_policy();
      m_run = ld_hint(kr.m + sidx, pol);
      l_run = ld_hint(kr.l + sidx, pol);
    } else {
      m_run = kr.m[sidx];
      l_run = kr.l[sidx];
    }
  }
  {
    // the O row enters TMEM as the high half; the residual half starts at 0
    uint32_t oh[64];
    if (kKeep && active && !fresh) {
      const uint64_t pol = l2_evict_first_policy();
      const float* src = kr.o + sidx * kHeadDim;   // 32-byte aligned (checked on the host)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t w[8];
        ld8_hint(src + 8 * i, w, pol);
#pragma unroll
        for (int e = 0; e < 8; ++e) oh[8 * i + e] = w[e];
      }
    } else if (active && !fresh) {
      const float4* src = reinterpret_cast<const float4*>(kr.o + sidx * kHeadDim);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 p = src[i];
        oh[4 * i + 0] = __float_as_uint(p.x);
        oh[4 * i + 1] = __float_as_uint(p.y);
        oh[4 * i + 2] = __float_as_uint(p.z);
        oh[4 * i + 3] = __float_as_uint(p.w);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) oh[i] = 0u;
    }
    tmem_st32_at<0>(t_o, oh);
    tmem_st32_at<32>(t_o + 32, oh);
#pragma unroll
    for (int i = 0; i < 64; ++i) oh[i] = 0u;
    tmem_st32_at<0>(t_o + 64, oh);
    tmem_st32_at<32>(t_o + 96, oh);
    tmem_wait_st();
  }

  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  // position of the tile's first row
  const int64_t q_first = a.q_pos0 + (a.pack ? (u.r0 + tile_row0(a, x)) / a.pack : u.r0 + tile_row0(a, x));
  bool ok = true;
#pragma unroll 1
  for (int t = 0; t < T; ++t) {
    if (!wait_bar(bar(B_SFULL + x), t & 1, ctl, budget, R_SOFTMAX, true)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t s[128];
    tmem_ld32_at<0>(t_s, s);
    tmem_ld32_at<32>(t_s + 32, s);
    tmem_ld32_at<64>(t_s + 64, s);
    tmem_ld32_at<96>(t_s + 96, s);
    tmem_wait_ld_at<0>(s);
    tmem_wait_ld_at<32>(s);
    tmem_wait_ld_at<64>(s);
    tmem_wait_ld_at<96>(s);

    const int64_t k0 = static_cast<int64_t>(key_tile(a, x, t)) * BN;
    const bool need_mask = (k0 + BN > kr.kv_len) || (a.causal && kr.kv_start + k0 + BN - 1 > q_first);
    if (__builtin_expect(need_mask, 0)) {
      int64_t lim = kr.kv_len - 1 - k0;
      if (a.causal) lim = i64min(lim, pos - kr.kv_start - k0);
      const int li = static_cast<int>(i64max(-1, i64min(lim, BN - 1)));
#pragma unroll
      for (int j = 0; j < 128; ++j)
        if (j > li) s[j] = __float_as_uint(-INFINITY);
    }
    float pm[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pm[i] = -INFINITY;
#pragma unroll
    for (int p = 0; p < 64; ++p)
      pm[p & 7] = max3(pm[p & 7], __uint_as_float(s[2 * p]), __uint_as_float(s[2 * p + 1]));
    const float mx = fmaxf(max3(pm[0], pm[1], pm[2]), max3(pm[3], pm[4], max3(pm[5], pm[6], pm[7])));
    const float t_nat = mx * a.scale;   // -inf when every key of the tile is masked
    float alpha = 1.0f;
    const bool resc = t_nat > m_run + kLazyNat;   // the reference moves
    if (resc) {
      alpha = (m_run == -INFINITY) ? 0.0f : ex2_approx((m_run - t_nat) * kLog2e);
      m_run = t_nat;
    }
    const float mlog = (m_run == -INFINITY) ? 0.0f : m_run * kLog2e;
    const float2 nm2 = make_float2(-mlog, -mlog);
    float2 rs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) rs[i] = make_float2(0.0f, 0.0f);
    // P for keys 0-63 (TMEM columns 0-31), then keys 64-127 (columns 32-63);
    // each half is announced on its own barrier so that the first half of
    // PV_x(t) runs while the second half is being computed.
    uint32_t p[64];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float2 sv = make_float2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
      const float2 e = __ffma2_rn(sv, sl2, nm2);
      const float2 bt = make_float2(ex2_approx(e.x), ex2_approx(e.y));
      rs[i & 3] = __fadd2_rn(rs[i & 3], bt);
      p[i] = pack_half2(bt.x, bt.y);
    }
    tmem_st32_at<0>(t_s, p);
    // PV_x(t-1) has completed (QK_x(t), issued after it, has), so O is stable;
    // it is rescaled before the first half of PV_x(t) accumulates into it,
    // 64 columns (the high then the residual half) per round.
    if (__any_sync(0xFFFFFFFFu, resc)) {
      const float2 al = make_float2(alpha, alpha);
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t o[64];
        tmem_ld32(t_o + 64 * hh, *reinterpret_cast<uint32_t (*)[32]>(&o[0]));
        tmem_ld32(t_o + 64 * hh + 32, *reinterpret_cast<uint32_t (*)[32]>(&o[32]));
        tmem_wait_ld(*reinterpret_cast<uint32_t (*)[32]>(&o[0]));
        tmem_wait_ld(*reinterpret_cast<uint32_t (*)[32]>(&o[32]));
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), al);
          o[i] = __float_as_uint(v.x);
          o[i + 1] = __float_as_uint(v.y);
        }
        tmem_st32_at<0>(t_o + 64 * hh, o);
        tmem_st32_at<32>(t_o + 64 * hh + 32, o);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar(B_PFULL + 2 * x));
#pragma unroll
    for (int i = 32; i < 64; ++i) {
      const float2 sv = make_float2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
      const float2 e = __ffma2_rn(sv, sl2, nm2);
      const float2 bt = make_float2(ex2_approx(e.x), ex2_approx(e.y));
      rs[i & 3] = __fadd2_rn(rs[i & 3], bt);
      p[i] = pack_half2(bt.x, bt.y);
    }
    tmem_st32_at<32>(t_s + 32, p);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar(B_PFULL + 2 * x + 1));
    const float2 r = __fadd2_rn(__fadd2_rn(rs[0], rs[1]), __fadd2_rn(rs[2], rs[3]));
    // same ops per tile with or without chunking
    l_run = fmaf(l_run, alpha, (r.x + r.y) + p_max_correction(mx, a.scale_log2, mlog));
  }
  float4* xch = reinterpret_cast<float4*>(smem + OFF_XCH) + row;
  if (pair_merge && x == 1) {
    // publish (m, l) for tile A, which reads this tile's O from TMEM itself
    *xch = make_float4(m_run, l_run, ok ? 1.0f : 0.0f, 0.0f);
    mbar_arrive(bar(B_MERGE));
    return;
  }
  if (ok) {
    if (wait_bar(bar(B_ODONE + x), 0, ctl, budget, R_SOFTMAX, true)) {
      tc_fence_after();
      if (pair_merge) {
        if (!wait_bar(bar(B_MERGE), 0, ctl, budget, R_SOFTMAX, true) ||
            !wait_bar(bar(B_ODONE + 1), 0, ctl, budget, R_SOFTMAX, true))
          return;
        tc_fence_after();
        const float4 pb = *xch;
        if (pb.z == 0.0f) return;   // tile B gave up; the failure is already recorded
        merge_pair_out(kr, sidx, active, m_run, l_run, pb.x, pb.y, t_o, t_o + 128u);
        return;
      }
      if (kKeep && active) {
        const uint64_t pol = l2_evict_first_policy();
        st_hint(kr.m + sidx, m_run, pol);
        st_hint(kr.l + sidx, l_run, pol);
      } else if (active) {
        kr.m[sidx] = m_run;
        kr.l[sidx] = l_run;
      }
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t oh[32], ol[32];
        tmem_ld32(t_o + 32 * half, oh);
        tmem_ld32(t_o + 64 + 32 * half, ol);
        tmem_wait_ld(oh);
        tmem_wait_ld(ol);
        if (kKeep && active) {
          const uint64_t pol = l2_evict_first_policy();
          float* dst = kr.o + sidx * kHeadDim + 32 * half;   // whole 32-byte sectors
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(oh[8 * i + e]) + __uint_as_float(ol[8 * i + e]);
            st8_hint(dst + 8 * i, v, pol);
          }
        } else if (active) {
          float4* dst = reinterpret_cast<float4*>(kr.o + sidx * kHeadDim) + 8 * half;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              v[e] = __uint_as_float(oh[4 * i + e]) + __uint_as_float(ol[4 * i + e]);
            dst[i] = make_float4(v[0], v[1], v[2], v[3]);
          }
        }
      }
    }
  }
}

template <bool kKeep>
__global__ void __launch_bounds__(kThreads, 1)
chunk_step_kernel(const __grid_constant__ CUtensorMap qmap, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();
  pdl_wait();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + OFF_CTL);
  const int warp = threadIdx.x >> 5;
  const int wg = warp >> 2;

  const Range kr = make_range(a);
  const Unit u = make_unit(a, kr);
  if (u.T_all == 0) return;   // uniform over the CTA: no visible key for these rows

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t count = 1;
      if (i >= B_RAWEMPTY && i < B_RAWEMPTY + NR) count = 128;   // dequant threads
      if (i >= B_KFULL && i < B_KFULL + ND) count = 128;         // dequant threads
      if (i >= B_VFULL && i < B_VFULL + ND) count = 128;         // dequant threads
      if (i == B_MERGE) count = 128;                             // softmax threads of tile B
      if (i >= B_PFULL && i < B_PFULL + 2 * NQT) count = 128;    // softmax threads of a tile
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

  // Register split: the softmax warpgroups hold a whole S row plus the P
  // fragments; the other warpgroups need far fewer registers.
  if (wg < 2) {
    reg_alloc<kRegSoftmax>();
    softmax_role<kKeep>(a, kr, u, wg, smem, sbase, tmem, ctl);
  } else {
    reg_dealloc<kRegOther>();
    if (wg == 2) {
      dequant_role(a, kr, u, smem, sbase, ctl);
    } else if (warp == 12) {
      producer_role<kKeep>(&qmap, a, kr, u, smem, sbase, ctl);
    } else if (warp == 13) {
      mma_role(a, u, sbase, tmem, ctl);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && a.host_status && *reinterpret_cast<volatile uint32_t*>(&ctl->abort))
    publish_failure(a.host_status);
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}


// ---------------------------------------------------------------------------
// head_dim 128.  A 136-byte Q8_0 row (four blocks) and an O row of 128 fp32
// channels do not fit the two-query-tile layout above (two 32 KB Q tiles and a
// 128 KB dequantised 128-key stage leave no room for the raw ring, and two O
// accumulators with residual halves would need 512 TMEM columns alone).  So a
// CTA takes one 128-row query tile and both softmax pipelines work on its rows
// (the paired arrangement above, here with or without the causal mask):
// pipeline A folds the even 64-key tiles, pipeline B the odd ones, each into
// its own running state, and A merges B's state at the end with the chunk
// recurrence.  The two pipelines interleave on the tensor pipe as the two query
// tiles do above.
//   QK_x: M = 128, N = 64 keys, 16 MMAs of K = 16 over Q.K_hi and Q.K_lo.
//   PV_x: M = 128, N = 128 channels, 8 MMAs (P.V_hi and P.V_lo, 4 k-steps each)
//         accumulating into the same 128 columns of O_x.
// TMEM columns: S_A [0,64), S_B [64,128), O_A [128,256), O_B [256,384).
// Shared memory: Q 32 KB (two 64-channel swizzle-atom columns), two
// dequantised stages of 64 KB (stage x holds pipeline x's key tile: K_hi, K_lo,
// V_hi, V_lo, each two 8 KB atom columns of 64 keys x 128 B), a two-stage raw
// ring of 2 x 8,704 B.  Dequantisation: thread k < 64 converts K row k, thread
// 64 + k V row k, so K and V of a tile are converted at once.
namespace d128 {

constexpr int D = 128;
constexpr int BM = 128;
constexpr int BN = 64;
constexpr int ROWB = 136;              // four 34-byte Q8_0 blocks
constexpr int RAWB = BN * ROWB;        // 8704
constexpr int NR = 2;
constexpr int kThreads = 512;
constexpr int kRegSoftmax = 136;   // a 64-score S row; the other warpgroups keep 120
constexpr int kRegOther = 120;
static_assert(2 * 128 * kRegSoftmax + 2 * 128 * kRegOther == 65536, "register split");

constexpr int TILE = 16384;                       // one 64-key x 128-channel fp16 tile
constexpr int DQ_KHI = 0, DQ_KLO = TILE, DQ_VHI = 2 * TILE, DQ_VLO = 3 * TILE;
constexpr int DEQ_BYTES = 4 * TILE;
constexpr int ATOMC = 8192;                       // one 64-channel atom column of a tile
constexpr int OFF_Q = 0;                          // 2 atom columns x (128 rows x 128 B)
constexpr int OFF_DEQ = 32768;
constexpr int OFF_RAW = OFF_DEQ + 2 * DEQ_BYTES;  // [NR][K raw | V raw]
constexpr int OFF_BAR = OFF_RAW + NR * 2 * RAWB;
constexpr int B_QFULL = 0;
constexpr int B_RAWFULL = 1;                 // NR
constexpr int B_RAWEMPTY = B_RAWFULL + NR;   // NR
constexpr int B_KFULL = B_RAWEMPTY + NR;     // 2 (stage = pipeline)
constexpr int B_KEMPTY = B_KFULL + 2;
constexpr int B_VFULL = B_KEMPTY + 2;
constexpr int B_VEMPTY = B_VFULL + 2;
constexpr int B_SFULL = B_VEMPTY + 2;
constexpr int B_PFULL = B_SFULL + 2;
constexpr int B_ODONE = B_PFULL + 2;
constexpr int B_MERGE = B_ODONE + 2;
constexpr int B_DRAIN = B_MERGE + 1;
constexpr int NBAR = B_DRAIN + 1;
constexpr int OFF_CTL = (OFF_BAR + NBAR * 8 + 15) / 16 * 16;
constexpr int OFF_XCH = OFF_CTL + CTL_BYTES;      // 128 x float4 {m, l, ok, -} of pipeline B
constexpr int SMEM_USED = OFF_XCH + BM * 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_RAW % 16 == 0 && RAWB % 16 == 0, "bulk copy alignment");
static_assert(OFF_DEQ % 1024 == 0 && TILE % 1024 == 0 && ATOMC % 1024 == 0, "swizzle atom alignment");

constexpr uint32_t T_S = 0;      // + 64 * pipeline
constexpr uint32_t T_O = 128;    // + 128 * pipeline

struct Unit {
  int64_t bh, b, h, r0;
  int T[2];      // key tiles of each pipeline
  int T_all;
};

// The chunk, or in the split form this CTA's key range and its partial state
// (as at head_dim 64, with 136-byte rows and 128-channel O rows).
__device__ __forceinline__ Range make_range(const ChunkArgs& a) {
  Range r;
  r.kv_len = a.kv_len;
  r.kv_start = a.kv_start;
  r.k8 = a.k8;
  r.v8 = a.v8;
  r.m = a.m;
  r.l = a.l;
  r.o = a.o;
  r.fresh = false;
  if (a.split_keys > 0) {
    const int64_t off = static_cast<int64_t>(blockIdx.y) * a.split_keys;
    const int64_t rows = static_cast<int64_t>(a.bh) * a.n_q;
    r.kv_len = i64min(a.split_keys, a.kv_len - off);
    r.kv_start = a.kv_start + off;
    r.k8 = a.k8 + off * ROWB;
    r.v8 = a.v8 + off * ROWB;
    r.m = a.part_m + blockIdx.y * rows;
    r.l = a.part_l + blockIdx.y * rows;
    r.o = a.part_o + blockIdx.y * rows * D;
    r.fresh = true;
  }
  return r;
}

__device__ __forceinline__ Unit make_unit(const ChunkArgs& a, const Range& kr) {
  Unit u;
  int64_t bh, qt;
  cta_order(blockIdx.x, a.n_qtiles, a.bh, a.head_group, bh, qt);
  u.bh = bh;
  u.b = u.bh / a.heads;
  u.h = u.bh % a.heads;
  u.r0 = (static_cast<int64_t>(a.tile0) + qt) * BM;
  int64_t n_vis = kr.kv_len;
  if (a.causal) {
    const int64_t r_last = i64min(u.r0 + BM - 1, a.n_q - 1);
    n_vis = i64min(n_vis, a.q_pos0 + r_last - kr.kv_start + 1);
  }
  const int tiles = n_vis > 0 ? static_cast<int>((n_vis + BN - 1) / BN) : 0;
  u.T[0] = (tiles + 1) / 2;
  u.T[1] = tiles / 2;
  u.T_all = tiles;
  return u;
}

__device__ __forceinline__ void producer(const CUtensorMap* qmap, const ChunkArgs& a, const Range& kr,
                                         const Unit& u, uint8_t* smem, uint32_t sbase, Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const bool skip_q = (a.inject == 1) && (blockIdx.x == 0);
  if (lane == 0) {
    prefetch_tensormap(qmap);
    if (!skip_q) {
      mbar_arrive_expect_tx(bar(B_QFULL), BM * D * 2);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tma_load_3d(sbase + OFF_Q + c * 16384, qmap, bar(B_QFULL),
                    static_cast<int32_t>(u.h * D + 64 * c), static_cast<int32_t>(u.r0),
                    static_cast<int32_t>(u.b));
    }
  }
  int last_bulk[NR];
#pragma unroll
  for (int s = 0; s < NR; ++s) last_bulk[s] = -1;
  const int64_t kv_plane = u.b * a.kv_heads + u.h / (a.heads / a.kv_heads);
  const uint8_t* kp = kr.k8 + kv_plane * a.plane_stride;
  const uint8_t* vp = kr.v8 + kv_plane * a.plane_stride;
  for (int t = 0; t < u.T_all; ++t) {
    const int sr = t % NR;
    if (!wait_bar(bar(B_RAWEMPTY + sr), ((t / NR) & 1) ^ 1, ctl, budget, R_PRODUCER, true)) break;
    const int64_t k0 = static_cast<int64_t>(t) * BN;
    const int n = static_cast<int>(i64min(BN, kr.kv_len - k0));
    const uint32_t bytes = static_cast<uint32_t>(n) * ROWB;
    const uint32_t dk = sbase + OFF_RAW + sr * 2 * RAWB;
    if ((bytes & 15u) == 0u) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_RAWFULL + sr), 2u * bytes);
        bulk_load(dk, kp + k0 * ROWB, bytes, bar(B_RAWFULL + sr));
        bulk_load(dk + RAWB, vp + k0 * ROWB, bytes, bar(B_RAWFULL + sr));
      }
#pragma unroll
      for (int s = 0; s < NR; ++s)
        if (s == sr) last_bulk[s] = t;
    } else {
      // ragged tail whose byte count is not a multiple of 16: plain 4-byte copies
      const uint32_t* sk = reinterpret_cast<const uint32_t*>(kp + k0 * ROWB);
      const uint32_t* sv = reinterpret_cast<const uint32_t*>(vp + k0 * ROWB);
      uint32_t* wk = reinterpret_cast<uint32_t*>(smem + OFF_RAW + sr * 2 * RAWB);
      uint32_t* wv = wk + RAWB / 4;
      const int words = n * (ROWB / 4);
      for (int w = lane; w < words; w += 32) {
        wk[w] = __ldg(sk + w);
        wv[w] = __ldg(sv + w);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_RAWFULL + sr));
#pragma unroll
      for (int s = 0; s < NR; ++s)
        if (s == sr) last_bulk[s] = -1;
    }
  }
#pragma unroll
  for (int s = 0; s < NR; ++s)
    if (last_bulk[s] >= 0) wait_bar(bar(B_RAWFULL + s), (last_bulk[s] / NR) & 1, ctl, budget, R_DRAIN, false);
  if (!skip_q) wait_bar(bar(B_QFULL), 0, ctl, budget, R_DRAIN, false);
}

// Thread k < 64: K row k of each tile; thread 64 + k: V row k.  Block b of a
// 136-byte row (channels 32b .. 32b+31) lands in atom column b / 2, 16-byte
// chunks 4 (b % 2) .. 4 (b % 2) + 3 of the key's 128-byte row, swizzled.
__device__ __forceinline__ void dequant(const ChunkArgs& a, const Range& kr, const Unit& u, uint8_t* smem,
                                        uint32_t sbase, Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;
  const int tid = threadIdx.x - 256;
  const int tensor = tid >> 6;        // 0: K, 1: V
  const int k = tid & 63;             // key row of the tile
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int sw = k & 7;
  for (int t = 0; t < u.T_all; ++t) {
    const int sr = t % NR;
    const int sd = t & 1;                              // the pipeline reading key tile t
    const uint32_t fill = static_cast<uint32_t>((t >> 1) & 1);
    if (!wait_bar(bar(B_RAWFULL + sr), (t / NR) & 1, ctl, budget, R_DEQUANT, true)) break;
    if (!wait_bar(bar((tensor ? B_VEMPTY : B_KEMPTY) + sd), fill ^ 1, ctl, budget, R_DEQUANT, true)) break;
    const int n_valid = static_cast<int>(i64min(BN, kr.kv_len - static_cast<int64_t>(t) * BN));
    uint8_t* hi = smem + OFF_DEQ + sd * DEQ_BYTES + (tensor ? DQ_VHI : DQ_KHI) + k * 128;
    uint8_t* lo = smem + OFF_DEQ + sd * DEQ_BYTES + (tensor ? DQ_VLO : DQ_KLO) + k * 128;
    if (k < n_valid) {
      const uint32_t* raw = reinterpret_cast<const uint32_t*>(
          smem + OFF_RAW + sr * 2 * RAWB + tensor * RAWB + k * ROWB);
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        // 9-word window: even blocks start word-aligned (scale in the low half of
        // word 0), odd blocks 2 bytes into a word (scale in its high half)
        const int w0 = 17 * (blk >> 1) + 8 * (blk & 1);
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = raw[w0 + i];
        dequant_block(w, blk & 1, hi + (blk >> 1) * ATOMC, lo + (blk >> 1) * ATOMC, sw);
      }
    } else {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          *reinterpret_cast<uint4*>(hi + c * ATOMC + 16 * j) = z;
          *reinterpret_cast<uint4*>(lo + c * ATOMC + 16 * j) = z;
        }
    }
    fence_proxy_async_smem();
    mbar_arrive(bar((tensor ? B_VFULL : B_KFULL) + sd));
    mbar_arrive(bar(B_RAWEMPTY + sr));
  }
}

__device__ __forceinline__ void mma(const ChunkArgs& a, const Unit& u, uint32_t sbase, uint32_t tmem,
                                    Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  constexpr uint32_t kIdescQK = idesc_f16_f32(128, BN, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, D, 0, 1);
  const bool leader = elect_one();
  // Q and K tiles K-major in two 64-channel atom columns (16 KB apart for Q,
  // 8 KB for K); k-step kk covers channels 16kk .. 16kk+15.  V tiles MN-major:
  // the two 64-channel halves of N are 8 KB apart (leading byte offset), each
  // k-step covers 16 keys = two 8-row swizzle atoms (2 KB).  P of keys
  // 16kk .. 16kk+15 sits in TMEM columns 8kk .. 8kk+7 of S_x.
  const uint64_t qdesc0 = smem_desc(sbase + OFF_Q, 1024, 1024, kSwizzle128);
  const uint64_t kdesc0 = smem_desc(sbase + OFF_DEQ + DQ_KHI, 1024, 1024, kSwizzle128);
  const uint64_t vdesc0 = smem_desc(sbase + OFF_DEQ + DQ_VHI, ATOMC, 1024, kSwizzle128);
  auto issue_qk = [&](int x) {
    const uint32_t d = tmem + T_S + 64u * x;
    const uint64_t kd = kdesc0 + static_cast<uint64_t>(x * (DEQ_BYTES >> 4));
    if (leader) {
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t qa = qdesc0 + static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          const uint64_t kb = kd + static_cast<uint64_t>((part * TILE + (kk >> 2) * ATOMC + (kk & 3) * 32) >> 4);
          mma_ss(d, qa, kb, kIdescQK, (part | kk) != 0 ? 1u : 0u);
        }
    }
  };
  auto issue_pv = [&](int x) {
    const uint32_t o = tmem + T_O + 128u * x;
    const uint32_t p = tmem + T_S + 64u * x;
    const uint64_t vd = vdesc0 + static_cast<uint64_t>(x * (DEQ_BYTES >> 4));
    if (leader) {
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(o, p + 8u * kk, vd + static_cast<uint64_t>((part * TILE + kk * 2048) >> 4), kIdescPV, 1u);
    }
  };
  auto commit = [&](int b) {
    if (leader) mma_commit(bar(b));
  };
  bool ok = wait_bar(bar(B_QFULL), 0, ctl, budget, R_MMA, true);
  if (ok) {
#pragma unroll
    for (int x = 0; x < 2; ++x)
      if (ok && u.T[x] > 0) {
        ok = wait_bar(bar(B_KFULL + x), 0, ctl, budget, R_MMA, true);
        if (!ok) break;
        tc_fence_after();
        issue_qk(x);
        commit(B_SFULL + x);
        commit(B_KEMPTY + x);
      }
  }
  for (int j = 0; ok && j < u.T[0]; ++j) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      if (j >= u.T[x]) continue;
      const uint32_t par = static_cast<uint32_t>(j & 1);
      if (!wait_bar(bar(B_VFULL + x), par, ctl, budget, R_MMA, true) ||
          !wait_bar(bar(B_PFULL + x), par, ctl, budget, R_MMA, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv(x);
      if (j == u.T[x] - 1) commit(B_ODONE + x);
      commit(B_VEMPTY + x);
      if (j + 1 < u.T[x]) {
        if (!wait_bar(bar(B_KFULL + x), par ^ 1, ctl, budget, R_MMA, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_qk(x);
        commit(B_SFULL + x);
        commit(B_KEMPTY + x);
      }
    }
  }
  commit(B_DRAIN);
  __syncwarp();
  wait_bar(bar(B_DRAIN), 0, ctl, budget, R_DRAIN, false);
}

template <int O>
__device__ __forceinline__ void ld32_at(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : Q8A_R8(r, O + 0), Q8A_R8(r, O + 8), Q8A_R8(r, O + 16), Q8A_R8(r, O + 24)
      : "r"(taddr));
}
template <int O>
__device__ __forceinline__ void wait_ld_at(uint32_t (&r)[64]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : Q8A_M8(r, O + 0), Q8A_M8(r, O + 8), Q8A_M8(r, O + 16), Q8A_M8(r, O + 24)::"memory");
}

// Rescale (or read) the 128 O columns of this thread's row in TMEM, 64 at a time.
__device__ __forceinline__ void scale_o(uint32_t t_o, float alpha) {
  const float2 al = make_float2(alpha, alpha);
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t o[64];
    ld32_at<0>(t_o + 64 * hh, o);
    ld32_at<32>(t_o + 64 * hh + 32, o);
    wait_ld_at<0>(o);
    wait_ld_at<32>(o);
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
      const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), al);
      o[i] = __float_as_uint(v.x);
      o[i + 1] = __float_as_uint(v.y);
    }
    tmem_st32_at<0>(t_o + 64 * hh, o);
    tmem_st32_at<32>(t_o + 64 * hh + 32, o);
  }
}

__device__ __forceinline__ void softmax(const ChunkArgs& a, const Range& kr, const Unit& u, int x,
                                        uint8_t* smem, uint32_t sbase, uint32_t tmem, Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;
  const int row = threadIdx.x & 127;
  const int wq = (threadIdx.x >> 5) & 3;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int T = u.T[x];
  if (T == 0) return;
  const int64_t rg = u.r0 + row;
  const int64_t pos = a.q_pos0 + rg;
  const bool active = rg < a.n_q && (!a.causal || pos >= kr.kv_start);
  const int64_t sidx = u.bh * a.n_q + rg;
  const uint32_t t_s = tmem + lane_off + T_S + 64u * x;
  const uint32_t t_o = tmem + lane_off + T_O + 128u * x;
  // pipeline B starts empty and A merges it in at the end; in the split form
  // both start empty (the partial state of this key range)
  const bool fresh = kr.fresh || x == 1;
  const bool pair_merge = u.T[1] > 0;
  float m_run = -INFINITY, l_run = 0.0f;
  if (active && !fresh) {
    m_run = kr.m[sidx];
    l_run = kr.l[sidx];
  }
  {
    uint32_t oh[64];
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      if (active && !fresh) {
        const float4* src = reinterpret_cast<const float4*>(kr.o + sidx * D + 64 * hh);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 p = src[i];
          oh[4 * i + 0] = __float_as_uint(p.x);
          oh[4 * i + 1] = __float_as_uint(p.y);
          oh[4 * i + 2] = __float_as_uint(p.z);
          oh[4 * i + 3] = __float_as_uint(p.w);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) oh[i] = 0u;
      }
      tmem_st32_at<0>(t_o + 64 * hh, oh);
      tmem_st32_at<32>(t_o + 64 * hh + 32, oh);
    }
    tmem_wait_st();
  }
  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  const int64_t q_first = a.q_pos0 + u.r0;
  bool ok = true;
#pragma unroll 1
  for (int t = 0; t < T; ++t) {
    if (!wait_bar(bar(B_SFULL + x), t & 1, ctl, budget, R_SOFTMAX, true)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t s[64];
    ld32_at<0>(t_s, s);
    ld32_at<32>(t_s + 32, s);
    wait_ld_at<0>(s);
    wait_ld_at<32>(s);
    const int64_t k0 = static_cast<int64_t>(2 * t + x) * BN;
    const bool need_mask = (k0 + BN > kr.kv_len) || (a.causal && kr.kv_start + k0 + BN - 1 > q_first);
    if (__builtin_expect(need_mask, 0)) {
      int64_t lim = kr.kv_len - 1 - k0;
      if (a.causal) lim = i64min(lim, pos - kr.kv_start - k0);
      const int li = static_cast<int>(i64max(-1, i64min(lim, BN - 1)));
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (j > li) s[j] = __float_as_uint(-INFINITY);
    }
    float pm[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pm[i] = -INFINITY;
#pragma unroll
    for (int p = 0; p < 32; ++p)
      pm[p & 3] = max3(pm[p & 3], __uint_as_float(s[2 * p]), __uint_as_float(s[2 * p + 1]));
    const float mx = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
    const float t_nat = mx * a.scale;
    float alpha = 1.0f;
    const bool resc = t_nat > m_run + kLazyNat;   // the reference moves
    if (resc) {
      alpha = (m_run == -INFINITY) ? 0.0f : ex2_approx((m_run - t_nat) * kLog2e);
      m_run = t_nat;
    }
    const float mlog = (m_run == -INFINITY) ? 0.0f : m_run * kLog2e;
    const float2 nm2 = make_float2(-mlog, -mlog);
    float2 rs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) rs[i] = make_float2(0.0f, 0.0f);
    uint32_t p[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float2 sv = make_float2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
      const float2 e = __ffma2_rn(sv, sl2, nm2);
      const float2 bt = make_float2(ex2_approx(e.x), ex2_approx(e.y));
      rs[i & 3] = __fadd2_rn(rs[i & 3], bt);
      p[i] = pack_half2(bt.x, bt.y);
    }
    tmem_st32(t_s, p);
    // PV_x(t-1) has completed (QK_x(t), issued after it, has): O is stable
    if (__any_sync(0xFFFFFFFFu, resc)) scale_o(t_o, alpha);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar(B_PFULL + x));
    const float2 r = __fadd2_rn(__fadd2_rn(rs[0], rs[1]), __fadd2_rn(rs[2], rs[3]));
    l_run = fmaf(l_run, alpha, (r.x + r.y) + p_max_correction(mx, a.scale_log2, mlog));
  }
  float4* xch = reinterpret_cast<float4*>(smem + OFF_XCH) + row;
  if (pair_merge && x == 1) {
    *xch = make_float4(m_run, l_run, ok ? 1.0f : 0.0f, 0.0f);
    mbar_arrive(bar(B_MERGE));
    return;
  }
  if (!ok) return;
  if (!wait_bar(bar(B_ODONE + x), 0, ctl, budget, R_SOFTMAX, true)) return;
  tc_fence_after();
  float m_b = -INFINITY, l_b = 0.0f;
  if (pair_merge) {
    if (!wait_bar(bar(B_MERGE), 0, ctl, budget, R_SOFTMAX, true) ||
        !wait_bar(bar(B_ODONE + 1), 0, ctl, budget, R_SOFTMAX, true))
      return;
    tc_fence_after();
    const float4 pb = *xch;
    if (pb.z == 0.0f) return;   // pipeline B gave up; the failure is already recorded
    m_b = pb.x;
    l_b = pb.y;
  }
  // the chunk recurrence over the two partial states (B's weight is 0 when
  // it holds no key); the weight of the larger reference is exactly 1
  const float m = fmaxf(m_run, m_b);
  const float wa = (m_run == m) ? 1.0f : (m_run == -INFINITY ? 0.0f : ex2_approx((m_run - m) * kLog2e));
  const float wb = (m_b == m) ? 1.0f : (m_b == -INFINITY ? 0.0f : ex2_approx((m_b - m) * kLog2e));
  if (active) {
    kr.m[sidx] = m;
    kr.l[sidx] = pair_merge ? fmaf(wa, l_run, wb * l_b) : l_run;
  }
#pragma unroll 1
  for (int q = 0; q < 4; ++q) {   // 32 channels at a time
    uint32_t oa[32], ob[32];
    tmem_ld32(t_o + 32 * q, oa);
    if (pair_merge) tmem_ld32(t_o + 128 + 32 * q, ob);
    tmem_wait_ld(oa);
    if (pair_merge) tmem_wait_ld(ob);
    if (active) {
      float4* dst = reinterpret_cast<float4*>(kr.o + sidx * D + 32 * q);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 4 * i + e;
          v[e] = pair_merge ? fmaf(wa, __uint_as_float(oa[c]), wb * __uint_as_float(ob[c]))
                            : __uint_as_float(oa[c]);
        }
        dst[i] = make_float4(v[0], v[1], v[2], v[3]);
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_step_d128_kernel(const __grid_constant__ CUtensorMap qmap, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();
  pdl_wait();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + OFF_CTL);
  const int warp = threadIdx.x >> 5;
  const int wg = warp >> 2;
  const Range kr = d128::make_range(a);
  const Unit u = d128::make_unit(a, kr);
  if (u.T_all == 0) return;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t count = 1;
      if (i >= B_RAWEMPTY && i < B_RAWEMPTY + NR) count = 128;   // every dequant thread
      if (i >= B_KFULL && i < B_KFULL + 2) count = 64;           // the K threads
      if (i >= B_VFULL && i < B_VFULL + 2) count = 64;           // the V threads
      if (i >= B_PFULL && i < B_PFULL + 2) count = 128;          // softmax threads of a pipeline
      if (i == B_MERGE) count = 128;                             // softmax threads of pipeline B
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
    softmax(a, kr, u, wg, smem, sbase, tmem, ctl);
  } else {
    reg_dealloc<kRegOther>();
    if (wg == 2) {
      dequant(a, kr, u, smem, sbase, ctl);
    } else if (warp == 12) {
      producer(&qmap, a, kr, u, smem, sbase, ctl);
    } else if (warp == 13) {
      mma(a, u, sbase, tmem, ctl);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && a.host_status && *reinterpret_cast<volatile uint32_t*>(&ctl->abort))
    publish_failure(a.host_status);
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace d128

// ---------------------------------------------------------------------------
// head_dim 128, two query tiles per CTA.  The paired kernel above dequantises
// every 64-key tile for one 128-row query tile; here the CTA's two softmax
// pipelines take two query tiles (rows r0 .. r0+127 and r0+128 .. r0+255) and
// both fold every key tile, so each dequantised tile serves 256 query rows, as
// in the head_dim 64 kernel.  The room comes from keeping Q in TMEM: each
// softmax thread stores its query row there once (column c holds channels 2c
// and 2c+1, the layout of an A operand), QK_x reads it as A, and shared memory
// holds only the dequantised ring and the raw ring.
//   QK_x: M = 128, N = 64 keys, 16 MMAs of K = 16 (Q.K_hi, Q.K_lo), A in TMEM.
//   PV_x: M = 128, N = 128 channels, 8 MMAs (P.V_hi, P.V_lo) into O_x.
// TMEM columns: S_A [0,64), S_B [64,128), O_A [128,256), O_B [256,384),
// Q_A [384,448), Q_B [448,512).
// Shared memory: two dequantised stages of 64 KB (K_hi, K_lo, V_hi, V_lo of one
// key tile, each two 8 KB atom columns of 64 keys x 128 B) and a two-stage raw
// ring of 2 x 8,704 B.  The MMA order and the stage releases follow the head_dim
// 64 kernel: PV_A(t), QK_A(t+1), PV_B(t), QK_B(t+1); a stage half is released
// once both tiles' MMAs on it are issued.
namespace d128x2 {

constexpr int D = 128;
constexpr int BM = 128;
constexpr int NQT = 2;
constexpr int BN = 64;
constexpr int ROWB = 136;
constexpr int RAWB = BN * ROWB;        // 8704
constexpr int NR = 2;
constexpr int ND = 2;
constexpr int kThreads = 512;
constexpr int kRegSoftmax = 136;
constexpr int kRegOther = 120;
static_assert(2 * 128 * kRegSoftmax + 2 * 128 * kRegOther == 65536, "register split");

constexpr int TILE = 16384;                       // one 64-key x 128-channel fp16 tile
constexpr int DQ_KHI = 0, DQ_KLO = TILE, DQ_VHI = 2 * TILE, DQ_VLO = 3 * TILE;
constexpr int DEQ_BYTES = 4 * TILE;
constexpr int ATOMC = 8192;                       // one 64-channel atom column of a tile
constexpr int OFF_DEQ = 0;
constexpr int OFF_RAW = OFF_DEQ + ND * DEQ_BYTES;  // [NR][K raw | V raw]
constexpr int OFF_BAR = OFF_RAW + NR * 2 * RAWB;
constexpr int B_QFULL = 0;                   // NQT: Q_x is in TMEM
constexpr int B_RAWFULL = B_QFULL + NQT;     // NR
constexpr int B_RAWEMPTY = B_RAWFULL + NR;   // NR
constexpr int B_KFULL = B_RAWEMPTY + NR;     // ND
constexpr int B_KEMPTY = B_KFULL + ND;       // ND
constexpr int B_VFULL = B_KEMPTY + ND;       // ND
constexpr int B_VEMPTY = B_VFULL + ND;       // ND
constexpr int B_SFULL = B_VEMPTY + ND;       // NQT
constexpr int B_PFULL = B_SFULL + NQT;       // NQT
constexpr int B_ODONE = B_PFULL + NQT;       // NQT
constexpr int B_DRAIN = B_ODONE + NQT;
constexpr int NBAR = B_DRAIN + 1;
constexpr int OFF_CTL = (OFF_BAR + NBAR * 8 + 15) / 16 * 16;
constexpr int SMEM_USED = OFF_CTL + CTL_BYTES;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_RAW % 16 == 0 && RAWB % 16 == 0, "bulk copy alignment");
static_assert(OFF_DEQ % 1024 == 0 && TILE % 1024 == 0 && ATOMC % 1024 == 0, "swizzle atom alignment");
static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");

constexpr uint32_t T_S = 0;      // + 64 * tile
constexpr uint32_t T_O = 128;    // + 128 * tile
constexpr uint32_t T_Q = 384;    // + 64 * tile

struct Unit {
  int64_t bh, b, h, r0;   // (batch*heads index), first row of tile A
  int T[NQT];             // key tiles each query tile folds (0 = inactive)
  int T_all;              // key tiles streamed through the CTA
};

// a.n_qtiles counts 128-row query tiles from a.tile0; a CTA takes two of them,
// and a tile past the count is inactive even when its rows exist (a launch may
// cover a range of query tiles)
__device__ __forceinline__ Unit make_unit(const ChunkArgs& a) {
  Unit u;
  const int64_t units = (static_cast<int64_t>(a.n_qtiles) + 1) / 2;
  int64_t bh, qu;
  cta_order(blockIdx.x, units, a.bh, a.head_group, bh, qu);
  u.bh = bh;
  u.b = u.bh / a.heads;
  u.h = u.bh % a.heads;
  u.r0 = (static_cast<int64_t>(a.tile0) + 2 * qu) * BM;
  u.T_all = 0;
#pragma unroll
  for (int x = 0; x < NQT; ++x) {
    const int64_t rx = u.r0 + x * BM;
    u.T[x] = 0;
    if (2 * qu + x < a.n_qtiles && rx < a.n_q) {
      const int64_t r_last = i64min(rx + BM - 1, a.n_q - 1);
      int64_t n_vis = a.kv_len;
      if (a.causal) n_vis = i64min(n_vis, a.q_pos0 + r_last - a.kv_start + 1);
      u.T[x] = n_vis > 0 ? static_cast<int>((n_vis + BN - 1) / BN) : 0;
    }
    u.T_all = max(u.T_all, u.T[x]);
  }
  return u;
}

__device__ __forceinline__ void producer(const ChunkArgs& a, const Unit& u, uint8_t* smem, uint32_t sbase,
                                         Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  int last_bulk[NR];
#pragma unroll
  for (int s = 0; s < NR; ++s) last_bulk[s] = -1;
  const int64_t kv_plane = u.b * a.kv_heads + u.h / (a.heads / a.kv_heads);
  const uint8_t* kp = a.k8 + kv_plane * a.plane_stride;
  const uint8_t* vp = a.v8 + kv_plane * a.plane_stride;
  for (int t = 0; t < u.T_all; ++t) {
    const int sr = t % NR;
    if (!wait_bar(bar(B_RAWEMPTY + sr), ((t / NR) & 1) ^ 1, ctl, budget, R_PRODUCER, true)) break;
    const int64_t k0 = static_cast<int64_t>(t) * BN;
    const int n = static_cast<int>(i64min(BN, a.kv_len - k0));
    const uint32_t bytes = static_cast<uint32_t>(n) * ROWB;
    const uint32_t dk = sbase + OFF_RAW + sr * 2 * RAWB;
    if ((bytes & 15u) == 0u) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_RAWFULL + sr), 2u * bytes);
        bulk_load(dk, kp + k0 * ROWB, bytes, bar(B_RAWFULL + sr));
        bulk_load(dk + RAWB, vp + k0 * ROWB, bytes, bar(B_RAWFULL + sr));
      }
#pragma unroll
      for (int s = 0; s < NR; ++s)
        if (s == sr) last_bulk[s] = t;
    } else {
      // ragged tail whose byte count is not a multiple of 16: plain 4-byte copies
      const uint32_t* sk = reinterpret_cast<const uint32_t*>(kp + k0 * ROWB);
      const uint32_t* sv = reinterpret_cast<const uint32_t*>(vp + k0 * ROWB);
      uint32_t* wk = reinterpret_cast<uint32_t*>(smem + OFF_RAW + sr * 2 * RAWB);
      uint32_t* wv = wk + RAWB / 4;
      const int words = n * (ROWB / 4);
      for (int w = lane; w < words; w += 32) {
        wk[w] = __ldg(sk + w);
        wv[w] = __ldg(sv + w);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_RAWFULL + sr));
#pragma unroll
      for (int s = 0; s < NR; ++s)
        if (s == sr) last_bulk[s] = -1;
    }
  }
#pragma unroll
  for (int s = 0; s < NR; ++s)
    if (last_bulk[s] >= 0) wait_bar(bar(B_RAWFULL + s), (last_bulk[s] / NR) & 1, ctl, budget, R_DRAIN, false);
}

// Thread k < 64: K row k of each key tile; thread 64 + k: V row k.
__device__ __forceinline__ void dequant(const ChunkArgs& a, const Unit& u, uint8_t* smem, uint32_t sbase,
                                        Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;
  const int tid = threadIdx.x - 256;
  const int tensor = tid >> 6;        // 0: K, 1: V
  const int k = tid & 63;             // key row of the tile
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int sw = k & 7;
  for (int t = 0; t < u.T_all; ++t) {
    const int sr = t % NR;
    const int sd = t % ND;
    const uint32_t fill = static_cast<uint32_t>((t / ND) & 1);
    if (!wait_bar(bar(B_RAWFULL + sr), (t / NR) & 1, ctl, budget, R_DEQUANT, true)) break;
    if (!wait_bar(bar((tensor ? B_VEMPTY : B_KEMPTY) + sd), fill ^ 1, ctl, budget, R_DEQUANT, true)) break;
    const int n_valid = static_cast<int>(i64min(BN, a.kv_len - static_cast<int64_t>(t) * BN));
    uint8_t* hi = smem + OFF_DEQ + sd * DEQ_BYTES + (tensor ? DQ_VHI : DQ_KHI) + k * 128;
    uint8_t* lo = smem + OFF_DEQ + sd * DEQ_BYTES + (tensor ? DQ_VLO : DQ_KLO) + k * 128;
    if (k < n_valid) {
      const uint32_t* raw = reinterpret_cast<const uint32_t*>(
          smem + OFF_RAW + sr * 2 * RAWB + tensor * RAWB + k * ROWB);
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        // 9-word window: even blocks start word-aligned (scale in the low half of
        // word 0), odd blocks 2 bytes into a word (scale in its high half)
        const int w0 = 17 * (blk >> 1) + 8 * (blk & 1);
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = raw[w0 + i];
        dequant_block(w, blk & 1, hi + (blk >> 1) * ATOMC, lo + (blk >> 1) * ATOMC, sw);
      }
    } else {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          *reinterpret_cast<uint4*>(hi + c * ATOMC + 16 * j) = z;
          *reinterpret_cast<uint4*>(lo + c * ATOMC + 16 * j) = z;
        }
    }
    fence_proxy_async_smem();
    mbar_arrive(bar((tensor ? B_VFULL : B_KFULL) + sd));
    mbar_arrive(bar(B_RAWEMPTY + sr));
  }
}

__device__ __forceinline__ void mma(const ChunkArgs& a, const Unit& u, uint32_t sbase, uint32_t tmem,
                                    Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  constexpr uint32_t kIdescQK = idesc_f16_f32(128, BN, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, D, 0, 1);
  const bool leader = elect_one();
  // K tiles K-major in two 64-channel atom columns 8 KB apart (k-step kk covers
  // channels 16kk .. 16kk+15); Q_x in TMEM, 8 columns per k-step.  V tiles
  // MN-major: the two 64-channel halves of N are 8 KB apart (leading byte
  // offset), each k-step covers 16 keys = two 8-row swizzle atoms (2 KB).  P of
  // keys 16kk .. 16kk+15 sits in TMEM columns 8kk .. 8kk+7 of S_x.
  const uint64_t kdesc0 = smem_desc(sbase + OFF_DEQ + DQ_KHI, 1024, 1024, kSwizzle128);
  const uint64_t vdesc0 = smem_desc(sbase + OFF_DEQ + DQ_VHI, ATOMC, 1024, kSwizzle128);
  auto issue_qk = [&](int x, int sd) {
    const uint32_t d = tmem + T_S + 64u * x;
    const uint32_t qa = tmem + T_Q + 64u * x;
    const uint64_t kd = kdesc0 + static_cast<uint64_t>(sd * (DEQ_BYTES >> 4));
    if (leader) {
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t kb = kd + static_cast<uint64_t>((part * TILE + (kk >> 2) * ATOMC + (kk & 3) * 32) >> 4);
          mma_ts(d, qa + 8u * kk, kb, kIdescQK, (part | kk) != 0 ? 1u : 0u);
        }
    }
  };
  auto issue_pv = [&](int x, int sd) {
    const uint32_t o = tmem + T_O + 128u * x;
    const uint32_t p = tmem + T_S + 64u * x;
    const uint64_t vd = vdesc0 + static_cast<uint64_t>(sd * (DEQ_BYTES >> 4));
    if (leader) {
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(o, p + 8u * kk, vd + static_cast<uint64_t>((part * TILE + kk * 2048) >> 4), kIdescPV, 1u);
    }
  };
  auto commit = [&](int b) {
    if (leader) mma_commit(bar(b));
  };
  // Key tile j sits in stage j % ND, filled for the (j / ND)-th time; both
  // query tiles read it, so a stage half is released after tile B's MMA on it.
  bool ok = true;
#pragma unroll
  for (int x = 0; x < NQT; ++x)
    if (ok && u.T[x] > 0) {
      ok = wait_bar(bar(B_QFULL + x), 0, ctl, budget, R_MMA, true) &&
           wait_bar(bar(B_KFULL + 0), 0, ctl, budget, R_MMA, true);
      if (!ok) break;
      tc_fence_after();
      issue_qk(x, 0);
      commit(B_SFULL + x);
    }
  if (ok) commit(B_KEMPTY + 0);   // every reader of K(0) issued
  for (int j = 0; ok && j < u.T_all; ++j) {
#pragma unroll
    for (int x = 0; x < NQT; ++x) {
      if (j < u.T[x]) {
        const int sd = j % ND;
        if (!wait_bar(bar(B_VFULL + sd), static_cast<uint32_t>((j / ND) & 1), ctl, budget, R_MMA, true) ||
            !wait_bar(bar(B_PFULL + x), static_cast<uint32_t>(j & 1), ctl, budget, R_MMA, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(x, sd);
        if (j == u.T[x] - 1) commit(B_ODONE + x);
      }
      if (x == NQT - 1) commit(B_VEMPTY + j % ND);   // every reader of V(j) issued
      if (j + 1 < u.T[x]) {
        const int sd = (j + 1) % ND;
        if (!wait_bar(bar(B_KFULL + sd), static_cast<uint32_t>(((j + 1) / ND) & 1), ctl, budget, R_MMA, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_qk(x, sd);
        commit(B_SFULL + x);
      }
      if (x == NQT - 1 && j + 1 < u.T_all) commit(B_KEMPTY + (j + 1) % ND);
    }
  }
  // never leave with an MMA in flight
  commit(B_DRAIN);
  __syncwarp();
  wait_bar(bar(B_DRAIN), 0, ctl, budget, R_DRAIN, false);
}

__device__ __forceinline__ void softmax(const ChunkArgs& a, const Unit& u, int x, uint32_t sbase,
                                        uint32_t tmem, Ctl* ctl) {
  const uint64_t budget = 2 * a.timeout_ns;
  const int row = threadIdx.x & 127;
  const int wq = (threadIdx.x >> 5) & 3;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int T = u.T[x];
  if (T == 0) return;
  const int64_t rg = u.r0 + static_cast<int64_t>(x) * BM + row;
  const int64_t pos = a.q_pos0 + rg;
  const bool active = rg < a.n_q && (!a.causal || pos >= a.kv_start);
  const int64_t sidx = u.bh * a.n_q + rg;
  const uint32_t t_s = tmem + lane_off + T_S + 64u * x;
  const uint32_t t_o = tmem + lane_off + T_O + 128u * x;
  const uint32_t t_q = tmem + lane_off + T_Q + 64u * x;
  {
    // this row of Q into TMEM, the A operand of QK_x: column c holds channels
    // 2c (low half) and 2c + 1; rows past n_q are zero
    uint32_t qv[64];
    if (rg < a.n_q) {
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((u.b * a.n_q + rg) * a.heads + u.h) * static_cast<int64_t>(D * 2));
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint4 w = src[i];
        qv[4 * i + 0] = w.x;
        qv[4 * i + 1] = w.y;
        qv[4 * i + 2] = w.z;
        qv[4 * i + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) qv[i] = 0u;
    }
    tmem_st32_at<0>(t_q, qv);
    tmem_st32_at<32>(t_q + 32, qv);
  }
  float m_run = -INFINITY, l_run = 0.0f;
  if (active) {
    m_run = a.m[sidx];
    l_run = a.l[sidx];
  }
  {
    uint32_t oh[64];
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      if (active) {
        const float4* src = reinterpret_cast<const float4*>(a.o + sidx * D + 64 * hh);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 p = src[i];
          oh[4 * i + 0] = __float_as_uint(p.x);
          oh[4 * i + 1] = __float_as_uint(p.y);
          oh[4 * i + 2] = __float_as_uint(p.z);
          oh[4 * i + 3] = __float_as_uint(p.w);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) oh[i] = 0u;
      }
      tmem_st32_at<0>(t_o + 64 * hh, oh);
      tmem_st32_at<32>(t_o + 64 * hh + 32, oh);
    }
  }
  tmem_wait_st();
  tc_fence_before();
  // test hook: the first CTA's tile A never announces its Q, so the waits on it run out
  if (!(a.inject == 1 && blockIdx.x == 0 && x == 0)) mbar_arrive(bar(B_QFULL + x));

  const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
  const int64_t q_first = a.q_pos0 + u.r0 + static_cast<int64_t>(x) * BM;
  bool ok = true;
#pragma unroll 1
  for (int t = 0; t < T; ++t) {
    if (!wait_bar(bar(B_SFULL + x), t & 1, ctl, budget, R_SOFTMAX, true)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t s[64];
    d128::ld32_at<0>(t_s, s);
    d128::ld32_at<32>(t_s + 32, s);
    d128::wait_ld_at<0>(s);
    d128::wait_ld_at<32>(s);
    const int64_t k0 = static_cast<int64_t>(t) * BN;
    const bool need_mask = (k0 + BN > a.kv_len) || (a.causal && a.kv_start + k0 + BN - 1 > q_first);
    if (__builtin_expect(need_mask, 0)) {
      int64_t lim = a.kv_len - 1 - k0;
      if (a.causal) lim = i64min(lim, pos - a.kv_start - k0);
      const int li = static_cast<int>(i64max(-1, i64min(lim, BN - 1)));
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (j > li) s[j] = __float_as_uint(-INFINITY);
    }
    float pm[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pm[i] = -INFINITY;
#pragma unroll
    for (int p = 0; p < 32; ++p)
      pm[p & 3] = max3(pm[p & 3], __uint_as_float(s[2 * p]), __uint_as_float(s[2 * p + 1]));
    const float mx = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
    const float t_nat = mx * a.scale;   // -inf when every key of the tile is masked
    float alpha = 1.0f;
    const bool resc = t_nat > m_run + kLazyNat;   // the reference moves
    if (resc) {
      alpha = (m_run == -INFINITY) ? 0.0f : ex2_approx((m_run - t_nat) * kLog2e);
      m_run = t_nat;
    }
    const float mlog = (m_run == -INFINITY) ? 0.0f : m_run * kLog2e;
    const float2 nm2 = make_float2(-mlog, -mlog);
    float2 rs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) rs[i] = make_float2(0.0f, 0.0f);
    uint32_t p[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float2 sv = make_float2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
      const float2 e = __ffma2_rn(sv, sl2, nm2);
      const float2 bt = make_float2(ex2_approx(e.x), ex2_approx(e.y));
      rs[i & 3] = __fadd2_rn(rs[i & 3], bt);
      p[i] = pack_half2(bt.x, bt.y);
    }
    tmem_st32(t_s, p);
    // PV_x(t-1) has completed (QK_x(t), issued after it, has): O is stable
    if (__any_sync(0xFFFFFFFFu, resc)) d128::scale_o(t_o, alpha);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar(B_PFULL + x));
    const float2 r = __fadd2_rn(__fadd2_rn(rs[0], rs[1]), __fadd2_rn(rs[2], rs[3]));
    l_run = fmaf(l_run, alpha, (r.x + r.y) + p_max_correction(mx, a.scale_log2, mlog));
  }
  if (!ok) return;
  if (!wait_bar(bar(B_ODONE + x), 0, ctl, budget, R_SOFTMAX, true)) return;
  tc_fence_after();
  if (active) {
    a.m[sidx] = m_run;
    a.l[sidx] = l_run;
  }
#pragma unroll 1
  for (int q = 0; q < 4; ++q) {   // 32 channels at a time
    uint32_t ov[32];
    tmem_ld32(t_o + 32 * q, ov);
    tmem_wait_ld(ov);
    if (active) {
      float4* dst = reinterpret_cast<float4*>(a.o + sidx * D + 32 * q);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]),
                             __uint_as_float(ov[4 * i + 2]), __uint_as_float(ov[4 * i + 3]));
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) chunk_step_d128x2_kernel(const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();
  pdl_wait();
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
      if (i >= B_QFULL && i < B_QFULL + NQT) count = 128;        // softmax threads of a tile
      if (i >= B_RAWEMPTY && i < B_RAWEMPTY + NR) count = 128;   // every dequant thread
      if (i >= B_KFULL && i < B_KFULL + ND) count = 64;          // the K threads
      if (i >= B_VFULL && i < B_VFULL + ND) count = 64;          // the V threads
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
    softmax(a, u, wg, sbase, tmem, ctl);
  } else {
    reg_dealloc<kRegOther>();
    if (wg == 2) {
      dequant(a, u, smem, sbase, ctl);
    } else if (warp == 12) {
      producer(a, u, smem, sbase, ctl);
    } else if (warp == 13) {
      mma(a, u, sbase, tmem, ctl);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && a.host_status && *reinterpret_cast<volatile uint32_t*>(&ctl->abort))
    publish_failure(a.host_status);
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace d128x2

}  // namespace

cudaError_t launch_chunk_step(const CUtensorMap& qmap, const ChunkArgs& args, cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    // The setmaxnreg split assumes every thread is launched with 65536 / 512
    // registers; with fewer, an increase could wait forever, so such a build is
    // refused before any launch.
    for (auto* fn : {chunk_step_kernel<false>, chunk_step_kernel<true>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (e != cudaSuccess) return e;
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return e;
      if (fa.numRegs * kThreads != 65536 || fa.maxThreadsPerBlock < kThreads) {
        set_launch_note("chunk_step_kernel has %d registers per thread and at most %d threads per "
                        "block; the register split needs %d and %d",
                        fa.numRegs, fa.maxThreadsPerBlock, 65536 / kThreads, kThreads);
        return cudaErrorInvalidConfiguration;
      }
    }
    configured_device = dev;
  }
  // the host counts 128-row query tiles; a CTA takes NQT of them
  ChunkArgs units = args;
  units.n_qtiles = (args.n_qtiles + NQT - 1) / NQT;
  const int64_t blocks = static_cast<int64_t>(units.n_qtiles) * units.bh;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const unsigned gy = args.split_keys > 0 ? static_cast<unsigned>(args.n_splits) : 1u;
  e = launch_kernel(args.l2_keep_kv ? chunk_step_kernel<true> : chunk_step_kernel<false>,
                    dim3(static_cast<unsigned>(blocks), gy), dim3(kThreads), SMEM_BYTES, stream, qmap, units);
  if (e != cudaSuccess)
    set_launch_note("chunk_step_kernel<<<(%lld, %u), %d, %d>>>", static_cast<long long>(blocks), gy,
                    kThreads, SMEM_BYTES);
  return e;
}

cudaError_t launch_chunk_step_d128(const CUtensorMap& qmap, const ChunkArgs& args, cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(d128::chunk_step_d128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             d128::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, d128::chunk_step_d128_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * d128::kThreads != 65536 || fa.maxThreadsPerBlock < d128::kThreads) {
      set_launch_note("chunk_step_d128_kernel has %d registers per thread and at most %d threads per "
                      "block; the register split needs %d and %d",
                      fa.numRegs, fa.maxThreadsPerBlock, 65536 / d128::kThreads, d128::kThreads);
      return cudaErrorInvalidConfiguration;
    }
    configured_device = dev;
  }
  if (args.n_qtiles >= 2 && args.split_keys == 0) {
    // two query tiles per CTA, Q in TMEM
    static thread_local int configured_x2 = -1;
    if (configured_x2 != dev) {
      e = cudaFuncSetAttribute(d128x2::chunk_step_d128x2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               d128x2::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, d128x2::chunk_step_d128x2_kernel);
      if (e != cudaSuccess) return e;
      if (fa.numRegs * d128x2::kThreads != 65536 || fa.maxThreadsPerBlock < d128x2::kThreads) {
        set_launch_note("chunk_step_d128x2_kernel has %d registers per thread and at most %d threads "
                        "per block; the register split needs %d and %d",
                        fa.numRegs, fa.maxThreadsPerBlock, 65536 / d128x2::kThreads, d128x2::kThreads);
        return cudaErrorInvalidConfiguration;
      }
      configured_x2 = dev;
    }
    const int64_t blocks = (static_cast<int64_t>(args.n_qtiles) + 1) / 2 * args.bh;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    e = launch_kernel(d128x2::chunk_step_d128x2_kernel, dim3(static_cast<unsigned>(blocks)), dim3(d128x2::kThreads),
                      d128x2::SMEM_BYTES, stream, args);
    if (e != cudaSuccess)
      set_launch_note("chunk_step_d128x2_kernel<<<%lld, %d, %d>>>", static_cast<long long>(blocks),
                      d128x2::kThreads, d128x2::SMEM_BYTES);
    return e;
  }
  // a single query tile, or the split form: one query tile per CTA, both
  // pipelines on its rows (paired); the split form adds a grid row per key range
  const int64_t blocks = static_cast<int64_t>(args.n_qtiles) * args.bh;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const unsigned gy = args.split_keys > 0 ? static_cast<unsigned>(args.n_splits) : 1u;
  e = launch_kernel(d128::chunk_step_d128_kernel, dim3(static_cast<unsigned>(blocks), gy), dim3(d128::kThreads),
                    d128::SMEM_BYTES, stream, qmap, args);
  if (e != cudaSuccess)
    set_launch_note("chunk_step_d128_kernel<<<%lld, %d, %d>>>", static_cast<long long>(blocks),
                    d128::kThreads, d128::SMEM_BYTES);
  return e;
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
