// FlashAttention-2 backward for bf16, head dim 32, 64, 96 or 128, on the sm_100-family
// tensor cores (tcgen05 MMA with accumulators in tensor memory, operands
// staged in shared memory by TMA).
//
// Loop order follows "CUDA 算子工程" ch.16 §16.2: one CTA owns a 128-row key
// block K_j, V_j (resident in shared memory) and walks the 128-row query
// blocks Q_i, dO_i.  dV_j and dK_j accumulate in tensor memory and are
// written once; dQ partials are added into the fp32 accumulator without
// waiting for the result (§16.3, scheme A').  Under the causal mask the walk starts
// at the diagonal block, so fully masked pairs are never loaded (§16.8 item 2).
//
// The scores are computed transposed, S^T = K_j Q_i^T, so that TMEM lane r is
// key row r: P^T and dS^T then sit with keys as the M dimension, which is
// what dV += P^T dO and dK += dS^T Q need, and P^T feeds the dV product
// straight from tensor memory.
//
// Warp roles (736 threads):
//   warps 0-15 compute.  Warp w owns TMEM lanes 32*(w%4) .. +31 (key rows for
//              S, dP, dV, dK) and column quarter w/4 of them (four warps per
//              SM sub-partition hide each other's latencies).
//              Per query block: P = exp2(S*scale*log2e - L*log2e) -> bf16
//              into TMEM; dS = P * (dP - D) -> bf16 into shared memory
//              (128-byte swizzle).  Epilogue: dV (w < 8) and scale * dK
//              (w >= 8), half the columns each.
//   warps 16-19 dQ drain, one per TMEM lane quarter (query rows of dQ):
//              TMEM -> shared memory -> bulk fp32 reductions into the
//              accumulator, off the compute warps' path.
//   warp 20    TMA producer: K, V once; Q (two stages, with its L and D rows)
//              and dO (one stage for d = 128, two for d = 64).
//   warp 21    TMEM allocator; issues dV(i) and S(i+1).
//   warp 22    issues dQ(i), dK(i) and dP(i+1).  Each MMA warp waits only on
//              its own chain's barriers, so one's waits overlap the other's
//              issue (one elected lane of each issues).
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128)     S^T; P^T (bf16) is written over it: query columns
//               [32g, 32g + 32) of S become P columns [32g, 32g + 16)
//   [128,256)   dP^T (d > 64: then the dQ tile of the same step over it)
//   [256,256+d) dV accumulator, [256+LD,256+LD+d) dK accumulator (LD = 64
//               for d <= 64, else 128)
//   [384,512)   d <= 64: a second S^T/P^T buffer for odd query blocks; dQ(i)
//               goes into the first d columns of S buffer i % 2 once dV(i)
//               has read P(i) there
//
// MMA issue order per query block i (software pipelined), per MMA warp:
//   warp 21:  dV(i)  S(i+1)
//   warp 22:  d > 64:   dQ(i)  dK(i)  dP(i+1)
//             d <= 64:  dP(i+1)  dQ(i)  dK(i)
// dQ goes before dK so that its drain starts early.  For d > 64, dP(i+1) is
// issued as soon as the drain warps have read dQ(i) out of the columns dP
// shares, so the tensor pipe computes dP(i+1) while the compute warps turn
// S(i+1) into P(i+1).  For d <= 64 (smaller products, so the hand-offs weigh
// more) dP(i+1) only waits until the compute warps have read dP(i) into
// registers, and dS is double-buffered in shared memory.
//
// Every wait is bounded; when one runs out the CTA records FA_ERR_TIMEOUT,
// drains its own TMA loads, MMAs and bulk reductions, frees tensor memory and
// exits.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "dq_layout.cuh"
#include "row_dot.cuh"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBlk = 128;  // Br = Bc = 128
constexpr int kComputeWarps = 16;               // 4 per TMEM lane quarter
constexpr int kDrainWarps = 4;                  // 1 per TMEM lane quarter
constexpr int kDrainWarp0 = kComputeWarps;      // warps 16-19
constexpr int kProducerWarp = kComputeWarps + kDrainWarps;
constexpr int kMmaWarp = kProducerWarp + 1;     // dV and S^T; TMEM allocator
constexpr int kMma2Warp = kMmaWarp + 1;         // dQ, dK and dP^T
constexpr int kThreads = 32 * (kComputeWarps + kDrainWarps + 3);
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kDrainThreads = 32 * kDrainWarps;
constexpr int kStagedUnits = 4;                 // dQ units per drain warp staged for one bulk reduction
constexpr int kHeadGroup = 4;  // heads whose key blocks interleave in the single-launch grid order
constexpr float kLog2e = 1.4426950408889634f;

// Barriers a block of head dim > 64 uses come first; the third Q and dO
// stages and the second S buffer's barriers of head dims <= 64 follow.
enum BarId {
  KV_FULL = 0,  // K, V landed
  QFULL0,       // Q stage (with its L, D rows) landed; 32 arrivals
  QFULL1,
  QEMPTY0,      // Q stage free again
  QEMPTY1,
  DOFULL0,      // dO stage landed
  DOFULL1,
  DOEMPTY0,     // dO stage free again (dV and dP commit)
  DOEMPTY1,
  S_FULL0,      // S^T(i) in TMEM buffer i % kSBufs (one barrier per buffer)
  S_FULL1,
  P_FULL,       // P^T(i) in TMEM (one per compute thread)
  DV_DONE0,     // dV(i) product done: P(i) read out of S buffer i % kSBufs
  DP_FULL,      // dP^T(i) in TMEM
  DS_FULL,      // dS^T(i) in shared memory (one per compute thread)
  DQ_FULL0,     // dQ(i) in TMEM (two S buffers: one barrier per buffer)
  DQ_EMPTY0,    // dQ(i) drained from TMEM (one per drain thread)
  ACC_FULL,     // every MMA done: dK, dV final
  QFULL2,
  QEMPTY2,
  DOFULL2,
  DOEMPTY2,
  S_READ0,      // two S buffers: S^T(i) read out of buffer i % 2 (one per compute thread)
  S_READ1,
  DV_DONE1,
  DP_READ,      // two S buffers: dP^T(i) read out of TMEM (one per compute thread)
  DS_EMPTY,     // two S buffers: dS(i) read by dK(i) and dQ(i)
  DQ_FULL1,
  DQ_EMPTY1,
  kNumBars
};

// Member s of the barrier set whose first member is `first` (stages, buffers).
__device__ __forceinline__ int bar_member(int first, int s) {
  switch (first) {
    case QFULL0: return s == 0 ? QFULL0 : s == 1 ? QFULL1 : QFULL2;
    case QEMPTY0: return s == 0 ? QEMPTY0 : s == 1 ? QEMPTY1 : QEMPTY2;
    case DOFULL0: return s == 0 ? DOFULL0 : s == 1 ? DOFULL1 : DOFULL2;
    case DOEMPTY0: return s == 0 ? DOEMPTY0 : s == 1 ? DOEMPTY1 : DOEMPTY2;
    case DV_DONE0: return s == 0 ? DV_DONE0 : DV_DONE1;
    case DQ_FULL0: return s == 0 ? DQ_FULL0 : DQ_FULL1;
    case DQ_EMPTY0: return s == 0 ? DQ_EMPTY0 : DQ_EMPTY1;
    default: return first + s;  // S_FULL0, S_READ0: consecutive
  }
}

// Stage and phase parity of item i (>= 0) of a ring of N stages, in unsigned
// arithmetic (a signed % or / costs several instructions in the per-block
// loops, and the compute warps are issue-bound).
template <int N>
__device__ __forceinline__ int ring_stage(int i) { return (int)((unsigned)i % (unsigned)N); }
template <int N>
__device__ __forceinline__ uint32_t ring_phase(int i) { return ((unsigned)i / (unsigned)N) & 1u; }

// Shared-memory and TMEM layout for tiles LD = 64 or 128 columns wide (head
// dims 32 and 64 use LD = 64, 96 and 128 use LD = 128; the TMA zero-fills the
// columns past d).
template <int LD>
struct Layout {
  // Two S^T buffers where the accumulators leave room (LD = 64).  Then S(i+1)
  // need not wait for dV(i) to read P(i); P(i) is packed into the lower 64
  // columns of its buffer, and dQ(i) goes into the upper 64 columns of the
  // other buffer once S(i+1) has been read out of it, so dP^T keeps its
  // columns to itself.  Q and dO get three stages each, so that no TMA load
  // sits inside the per-block chain of hand-offs.
  static constexpr int kSBufs = LD == 64 ? 2 : 1;
  static constexpr int kQStages = LD == 64 ? 3 : 2;
  static constexpr int kDoStages = LD == 64 ? 3 : 1;
  static constexpr int kChunk = kBlk * 128;     // 128 rows x 128 bytes (64 bf16 columns)
  static constexpr int kTile = kBlk * LD * 2;   // one Q / K / V / dO tile
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;                  // kQStages stages
  static constexpr int kdO = kQ + kQStages * kTile;      // kDoStages stages
  static constexpr int kdS = kdO + kDoStages * kTile;    // 128 x 128 bf16, two 64-column chunks
  // dQ staging for bulk reductions: one slot of kStagedUnits 2 KB units
  // (32 rows x 16 fp32 columns each) per drain warp
  static constexpr int kStage = kdS + 2 * kChunk;
  static constexpr int kStageBytes = kDrainWarps * kStagedUnits * 2048;
  static constexpr int kL = kStage + kStageBytes;        // kQStages x 128 fp32 (L * log2 e)
  static constexpr int kD = kL + kQStages * kBlk * 4;    // kQStages x 128 fp32
  static constexpr int kBar = kD + kQStages * kBlk * 4;
  static constexpr int kMisc = kBar + kNumBars * 8;      // TMEM base address, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr uint32_t kColS = 0, kColS1 = 384, kColdP = 128, kColdQ = 128;
  static constexpr uint32_t kColdV = 256, kColdK = 256 + LD;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kQStages <= 3 && kDoStages <= 3, "barrier slots");
  static_assert(kBytes <= 232448, "shared memory budget");
};

struct BwdParams {
  const float* L;
  const float* D;
  float* dq_accum;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  int32_t* status;
  uint64_t wait_ns;
  int B, H, N, Nk;      // query rows, key rows
  int n_tiles;          // ceil(N / 128): query blocks (and dQ accumulator tiles)
  int nk_tiles;         // ceil(Nk / 128): key blocks, one CTA each per head
  int offset;           // Nk - N: key j visible to query i iff j <= i + offset (causal)
  int64_t sb, sh, sn;   // Q-shaped strides
  int64_t ksb, ksh, ksn;  // K-shaped strides (dK, dV written with these)
  float scale;
  int causal;
  int64_t slice_elems;  // > 0: deterministic, key block kb stores into slice kb
  // non-null: [0] += (key block, query block) pairs executed, [1] += executed
  // pairs with no visible entry (tile-pair accounting; null in fa_bwd)
  unsigned long long* pair_count;
  int head_group;       // heads whose key blocks interleave in the grid order (bwd_sm103_kernel)
};

// Does query block qb (128 rows) hold a query that sees key k0?  Key j is
// visible to query i iff j <= i + offset under the causal mask.
__device__ __forceinline__ bool block_sees_key(int qb, int k0, int N, int offset, int causal) {
  const int last_q = min(qb * kBlk + kBlk - 1, N - 1);
  return !causal || k0 <= last_q + offset;
}

using ptx::warp_wait;
using ptx::warp_wait2;

// Bounded wait until *c >= target (acquire, GPU scope), polled by one thread.
__device__ __forceinline__ bool wait_counter(const int32_t* c, int target, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer();
  for (;;) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    if (v >= target) return true;
    if (ptx::globaltimer() - t0 > limit_ns) return false;
    __nanosleep(256);
  }
}

// The backward for one key block kb of head bh, run by a whole CTA.
// kRect: causal with N_k != N (the mask is offset from the diagonal); a
// separate instantiation so that the square case keeps its cheaper loop.
// ready (may be null): before any load, wait (bounded) until *ready >=
// ready_target, i.e. until D and the zeroed accumulator of this head have
// been published.  done (may be null): once every dQ contribution of this
// block has reached global memory, add 1 (release).
// kFused: run inside the single-launch backward (ready and done are used,
// D is read coherently since this launch writes it); otherwise both are null.
// kCount: tile-pair accounting into prm.pair_count (a separate instantiation,
// so that the kernels fa_bwd runs carry no counting code: a per-block branch
// in the MMA warp alone measured 2.6 % slower).
template <int HD, bool kDet, bool kRect, bool kFused, bool kCount>
__device__ __forceinline__ void bwd_block(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                          const CUtensorMap& tmdO, const CUtensorMap& tmdK, const CUtensorMap& tmdV,
                                          const BwdParams& prm, const int kb, const int bh,
                                          const int32_t* ready, int ready_target, int32_t* done) {
  constexpr int LD = HD <= 64 ? 64 : 128;
  using Ly = Layout<LD>;
  constexpr int kDoSt = Ly::kDoStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_addr(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(prm.status, 0, (int32_t)FA_ERR_DEVICE);
    return;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kMisc + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + Ly::kBar + 8 * i; };
  auto barm = [&](int first, int s) -> uint32_t { return bar(bar_member(first, s)); };

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(KV_FULL), 1);
    for (int st = 0; st < Ly::kQStages; ++st) {
      ptx::mbar_init(barm(QFULL0, st), 32);
      ptx::mbar_init(barm(QEMPTY0, st), 1);
    }
    for (int st = 0; st < kDoSt; ++st) {
      ptx::mbar_init(barm(DOFULL0, st), 1);
      ptx::mbar_init(barm(DOEMPTY0, st), 2);  // dP (second MMA warp) and dV (first) read the stage
    }
    for (int sb = 0; sb < 2; ++sb) {
      ptx::mbar_init(barm(S_FULL0, sb), 1);
      ptx::mbar_init(barm(S_READ0, sb), kComputeThreads);
      ptx::mbar_init(barm(DV_DONE0, sb), 1);
      ptx::mbar_init(barm(DQ_FULL0, sb), 1);
      ptx::mbar_init(barm(DQ_EMPTY0, sb), kDrainThreads);
    }
    ptx::mbar_init(bar(P_FULL), kComputeThreads);
    ptx::mbar_init(bar(DP_FULL), 1);
    ptx::mbar_init(bar(DP_READ), kComputeThreads);
    ptx::mbar_init(bar(DS_FULL), kComputeThreads);
    ptx::mbar_init(bar(DS_EMPTY), 1);
    ptx::mbar_init(bar(ACC_FULL), 2);  // one commit from each MMA warp
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(sbase + Ly::kMisc, Ly::kTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tm = __shfl_sync(0xffffffffu, *tmem_slot, 0);
  if (kFused) {
    if (threadIdx.x == 0) {
      if (!wait_counter(ready, ready_target, prm.wait_ns)) {
        *abort_flag = 1;
        atomicCAS(prm.status, 0, (int32_t)FA_ERR_TIMEOUT);
      }
      // the zeros were written by generic stores; the TMA's bulk reductions
      // (async proxy) must come after them
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncthreads();
    if (*abort_flag) {  // nothing was started: free tensor memory and leave
      if (warp == kMmaWarp) ptx::tmem_dealloc(tm, Ly::kTmemCols);
      return;
    }
  }

  const int b = bh / prm.H, h = bh % prm.H;
  const int k0 = kb * kBlk;
  // first query block holding a query that sees key k0: i >= k0 - offset
  // (every key block has one, the last query sees every key)
  const int q_first = !prm.causal ? 0 : !kRect ? kb : (k0 > prm.offset ? (k0 - prm.offset) / kBlk : 0);
  const int n_iter = prm.n_tiles - q_first;
  const ptx::Waiter W{abort_flag, prm.status, prm.wait_ns};

  const uint32_t sK = sbase + Ly::kK, sV = sbase + Ly::kV;
  constexpr int kSB = Ly::kSBufs;
  constexpr int kQSt = Ly::kQStages;
  const uint32_t sdS = sbase + Ly::kdS;
  // S^T buffer of query block i
  auto tS = [&](int i) -> uint32_t { return tm + (kSB == 2 && (i & 1) ? Ly::kColS1 : Ly::kColS); };
  // dQ(i): over dP^T with one S buffer; with two, the upper 64 columns of the
  // buffer that S(i+1) uses (after S(i+1) has been read out of it)
  auto tdQ = [&](int i) -> uint32_t { return kSB == 2 ? tS(i + 1) + 64 : tm + Ly::kColdQ; };
  auto sQ = [&](int st) -> uint32_t { return sbase + Ly::kQ + st * Ly::kTile; };
  auto sdO = [&](int st) -> uint32_t { return sbase + Ly::kdO + st * Ly::kTile; };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int q_issued = 0, do_issued = 0;
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmQ);
      ptx::prefetch_tensormap(&tmK);
      ptx::prefetch_tensormap(&tmV);
      ptx::prefetch_tensormap(&tmdO);
      ptx::mbar_arrive_expect_tx(bar(KV_FULL), 2 * Ly::kTile);
#pragma unroll
      for (int c = 0; c < LD / 64; ++c) {
        ptx::tma_load_4d(sK + c * Ly::kChunk, &tmK, bar(KV_FULL), c * 64, k0, h, b);
        ptx::tma_load_4d(sV + c * Ly::kChunk, &tmV, bar(KV_FULL), c * 64, k0, h, b);
      }
    }
    // L and D rows of the next query block are read into registers one block
    // ahead, so their global-load latency hides behind the stage waits.
    float lv[kBlk / 32], dv[kBlk / 32];
    auto fetch_rows = [&](int it) {
      const int q0 = (q_first + it) * kBlk;
#pragma unroll
      for (int u = 0; u < kBlk / 32; ++u) {
        const int q = q0 + lane + 32 * u;
        lv[u] = q < prm.N ? __ldg(prm.L + (int64_t)bh * prm.N + q) * kLog2e : INFINITY;
        // D may have been written earlier in this launch: read it at L2
        dv[u] = q < prm.N ? (kFused ? __ldcg(prm.D + (int64_t)bh * prm.N + q) : __ldg(prm.D + (int64_t)bh * prm.N + q))
                          : 0.f;
      }
    };
    fetch_rows(0);
    for (int i = 0; i < n_iter; ++i) {
      const int st = ring_stage<kQSt>(i);
      const int q0 = (q_first + i) * kBlk;
      if (i >= kQSt) {
        ok = warp_wait(barm(QEMPTY0, st), ring_phase<kQSt>(i - kQSt), W);
        if (!ok) break;
      }
      float* sL = reinterpret_cast<float*>(smem + Ly::kL) + st * kBlk;
      float* sD = reinterpret_cast<float*>(smem + Ly::kD) + st * kBlk;
#pragma unroll
      for (int u = 0; u < kBlk / 32; ++u) {
        sL[lane + 32 * u] = lv[u];
        sD[lane + 32 * u] = dv[u];
      }
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(barm(QFULL0, st), Ly::kTile);
#pragma unroll
        for (int c = 0; c < LD / 64; ++c)
          ptx::tma_load_4d(sQ(st) + c * Ly::kChunk, &tmQ, barm(QFULL0, st), c * 64, q0, h, b);
      } else {
        ptx::mbar_arrive(barm(QFULL0, st));
      }
      q_issued = i + 1;
      const int sd = ring_stage<kDoSt>(i);
      if (i >= kDoSt) {
        ok = warp_wait(barm(DOEMPTY0, sd), ring_phase<kDoSt>(i - kDoSt), W);
        if (!ok) break;
      }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(barm(DOFULL0, sd), Ly::kTile);
#pragma unroll
        for (int c = 0; c < LD / 64; ++c)
          ptx::tma_load_4d(sdO(sd) + c * Ly::kChunk, &tmdO, barm(DOFULL0, sd), c * 64, q0, h, b);
      }
      __syncwarp();
      do_issued = i + 1;
      if (i + 1 < n_iter) fetch_rows(i + 1);
    }
    if (!ok) {  // let every copy this CTA started land before the CTA exits
      ptx::wait_bounded(bar(KV_FULL), 0, W, false);
      for (int i = q_issued > kQSt ? q_issued - kQSt : 0; i < q_issued; ++i)
        ptx::wait_bounded(barm(QFULL0, ring_stage<kQSt>(i)), ring_phase<kQSt>(i), W, false);
      for (int i = do_issued > kDoSt ? do_issued - kDoSt : 0; i < do_issued; ++i)
        ptx::wait_bounded(barm(DOFULL0, ring_stage<kDoSt>(i)), ring_phase<kDoSt>(i), W, false);
    }
  } else if (warp == kMmaWarp || warp == kMma2Warp) {
    // ------------------------------------------------------------ MMA issue
    // Two warps issue, each running its own chain (disjoint accumulators and
    // operand buffers), so that one warp's barrier waits overlap the other's:
    //   first  (kMmaWarp):  dV(i) once P(i) is in TMEM, then S(i+1)
    //   second (kMma2Warp): dQ(i), dK(i) once dS(i) is in shared memory, then
    //                       dP(i+1) once the drain has read dQ(i) out of the
    //                       columns dP shares
    // A dO stage is released by both (dV and dP read it).  The whole warp
    // runs each loop and waits; one elected lane issues the MMAs and commits.
    // Every operand is warp-uniform (the TMEM base is broadcast from lane 0,
    // K steps are unrolled) so each tcgen05.mma issues at the tensor pipe's
    // own rate.
    constexpr uint32_t kIdS = ptx::idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
    constexpr uint32_t kIdKV = ptx::idesc_bf16_f32(128, HD, false, true);   // dV, dK
    constexpr uint32_t kIdQ = ptx::idesc_bf16_f32(128, HD, true, true);     // dQ
    // K-major operand: 16-element K step kk inside 64-column chunks
    auto kdesc = [&](uint32_t tile, int kk) -> uint64_t {
      return ptx::sdesc_sw128(tile + (kk >> 2) * Ly::kChunk + (kk & 3) * 32, 16, 1024);
    };
    // MN-major operand: 16-row K step kk; 64-column MN blocks one chunk apart
    auto mndesc = [&](uint32_t tile, int kk) -> uint64_t {
      return ptx::sdesc_sw128(tile + kk * 2048, Ly::kChunk, 1024);
    };
    const uint32_t tdP = tm + Ly::kColdP;
    const uint32_t tdV = tm + Ly::kColdV, tdK = tm + Ly::kColdK;
    // S^T(i) = K Q(i)^T into buffer i % kSB
    auto issue_S = [&](int i) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        ptx::mma_ss(tS(i), kdesc(sK, kk), kdesc(sQ(ring_stage<kQSt>(i)), kk), kIdS, kk > 0);
      ptx::tc_commit(barm(S_FULL0, (kSB == 2 ? (i & 1) : 0)));
    };
    // dP^T = V dO^T; the dO stage's dP reader is done at this commit
    auto issue_dP = [&](int sd) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) ptx::mma_ss(tdP, kdesc(sV, kk), kdesc(sdO(sd), kk), kIdS, kk > 0);
      ptx::tc_commit(bar(DP_FULL));
      ptx::tc_commit(barm(DOEMPTY0, sd));
    };
    // dK += dS^T Q (the last reader of Q(i): S(i) read it before P(i) existed)
    auto issue_dK = [&](int i) {
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)
        ptx::mma_ss(tdK, kdesc(sdS, kk), mndesc(sQ(ring_stage<kQSt>(i)), kk), kIdKV, (i | kk) != 0);
      ptx::tc_commit(barm(QEMPTY0, ring_stage<kQSt>(i)));
    };
    // dQ = dS K
    auto issue_dQ = [&](int i) {
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk) ptx::mma_ss(tdQ(i), mndesc(sdS, kk), mndesc(sK, kk), kIdQ, kk > 0);
      ptx::tc_commit(barm(DQ_FULL0, (kSB == 2 ? ((i + 1) & 1) : 0)));
    };
    // TMEM column of P^T for the 16-query K step kk of dV: with one S buffer
    // query columns [32g, 32g + 32) of S became P columns [32g, 32g + 16);
    // with two, compute warp g owned query columns [16g, 16g + 16) and
    // [64 + 16g, 64 + 16g + 16) and packed them into P columns [16g, 16g + 16)
    auto p_col = [](int kk) -> uint32_t {
      return kSB == 2 ? (kk & 3) * 16 + (kk >> 2) * 8 : (kk >> 1) * 32 + (kk & 1) * 8;
    };

    bool ok = warp_wait(bar(KV_FULL), 0, W);
    unsigned n_exec = 0, n_masked = 0;  // tile-pair accounting (pair_count)
    if (warp == kMmaWarp) {
      if (ok && (ok = warp_wait(bar(QFULL0), 0, W))) {
        ptx::tc_fence_after();
        if (ptx::elect_one()) issue_S(0);
        __syncwarp();
      }
      for (int i = 0; ok && i < n_iter; ++i) {
        const int sd = ring_stage<kDoSt>(i);
        const uint32_t qph = ring_phase<kQSt>(i + 1);  // phase of Q(i+1)
        if constexpr (kSB == 2) {
          // S^T(i+1) first, into buffer (i+1) % 2 as soon as its last readers
          // are done: dV(i-1) (P(i-1) in the lower columns) and the drain of
          // dQ(i-2) (upper columns).  It is then computed while the compute
          // warps still turn S(i) into P(i).
          if (i + 1 < n_iter) {
            ok = (i < 2 ? warp_wait(barm(QFULL0, ring_stage<kQSt>(i + 1)), qph, W)
                        : warp_wait2(barm(QFULL0, ring_stage<kQSt>(i + 1)), qph, barm(DQ_EMPTY0, ((i + 1) & 1)),
                                     ((i - 2) >> 1) & 1, W)) &&
                 (i < 1 || warp_wait(barm(DV_DONE0, ((i - 1) & 1)), ((i - 1) >> 1) & 1, W));
            if (!ok) break;
            ptx::tc_fence_after();
            if (ptx::elect_one()) issue_S(i + 1);
            __syncwarp();
          }
        }
        // dV += P^T dO   (A = P^T from TMEM) once P(i) is there and dO(i) has
        // landed (P(i) does not imply dO(i); the other MMA warp's dP(i)
        // waits for it too)
        if (!(ok = warp_wait2(bar(P_FULL), i & 1, barm(DOFULL0, sd), ring_phase<kDoSt>(i), W))) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kBlk / 16; ++kk)
            ptx::mma_ts(tdV, tS(i) + p_col(kk), mndesc(sdO(sd), kk), kIdKV, (i | kk) != 0);
          ptx::tc_commit(barm(DV_DONE0, (kSB == 2 ? (i & 1) : 0)));
          ptx::tc_commit(barm(DOEMPTY0, sd));
        }
        __syncwarp();
        if constexpr (kSB == 1) {
          // S^T(i+1) = K Q(i+1)^T once dV(i) has read P(i) out of the buffer
          if (i + 1 < n_iter) {
            if (!(ok = warp_wait2(barm(QFULL0, ring_stage<kQSt>(i + 1)), qph, bar(DV_DONE0), i & 1, W))) break;
            ptx::tc_fence_after();
            if (ptx::elect_one()) issue_S(i + 1);
            __syncwarp();
          }
        }
      }
    } else if constexpr (kSB == 2) {
      // dP(i+1) as soon as the compute warps have read dP(i) out of tensor
      // memory; dK(i) once dS(i) is in shared memory; dQ(i) once S(i+1) has
      // been read out of the buffer whose upper columns take it (for the last
      // block: once the dQ that was there before has been drained).  The
      // compute warps write dS(i+1) after DS_EMPTY, committed behind dQ(i).
      if (ok && (ok = warp_wait(bar(DOFULL0), 0, W))) {
        ptx::tc_fence_after();
        if (ptx::elect_one()) issue_dP(0);
        __syncwarp();
      }
      for (int i = 0; ok && i < n_iter; ++i) {
        if (i + 1 < n_iter) {
          const int sd1 = ring_stage<kDoSt>(i + 1);
          if (!(ok = warp_wait2(bar(DP_READ), i & 1, barm(DOFULL0, sd1), ring_phase<kDoSt>(i + 1), W))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) issue_dP(sd1);
          __syncwarp();
        }
        if (!(ok = warp_wait(bar(DS_FULL), i & 1, W))) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) issue_dK(i);
        __syncwarp();
        if (i + 1 < n_iter)
          ok = warp_wait(barm(S_READ0, ((i + 1) & 1)), ((i + 1) >> 1) & 1, W);
        else if (i >= 2)
          ok = warp_wait(barm(DQ_EMPTY0, ((i + 1) & 1)), ((i - 2) >> 1) & 1, W);
        if (!ok) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          issue_dQ(i);
          ptx::tc_commit(bar(DS_EMPTY));
        }
        __syncwarp();
        if constexpr (kCount) {
          ++n_exec;
          n_masked += block_sees_key(q_first + i, k0, prm.N, prm.offset, prm.causal) ? 0u : 1u;
        }
      }
    } else {
      if (ok && (ok = warp_wait(bar(DOFULL0), 0, W))) {
        ptx::tc_fence_after();
        if (ptx::elect_one()) issue_dP(0);
        __syncwarp();
      }
      for (int i = 0; ok && i < n_iter; ++i) {
        const uint32_t ph = i & 1;
        // dQ first so that its drain starts early.  The compute warps
        // overwrite dS only after DP_FULL of the next block, which completes
        // after this dK.
        if (!(ok = warp_wait(bar(DS_FULL), ph, W))) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          issue_dQ(i);
          issue_dK(i);
        }
        __syncwarp();
        if constexpr (kCount) {
          ++n_exec;
          n_masked += block_sees_key(q_first + i, k0, prm.N, prm.offset, prm.causal) ? 0u : 1u;
        }
        // dP(i+1) once dQ(i) has been drained out of the columns it shares
        // and dO(i+1) has landed
        if (i + 1 < n_iter) {
          const int sd1 = ring_stage<kDoSt>(i + 1);
          if (!(ok = warp_wait2(bar(DQ_EMPTY0), ph, barm(DOFULL0, sd1), ring_phase<kDoSt>(i + 1), W))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) issue_dP(sd1);
          __syncwarp();
        }
      }
    }
    const bool lead = ptx::elect_one();
    if (lead) ptx::tc_commit(bar(ACC_FULL));
    if (kCount && lead && warp == kMma2Warp) {
      atomicAdd(prm.pair_count, (unsigned long long)n_exec);
      atomicAdd(prm.pair_count + 1, (unsigned long long)n_masked);
    }
    __syncwarp();
    // nothing in flight at exit (the other MMA warp commits too, on its way out)
    if (!ok) ptx::wait_bounded(bar(ACC_FULL), 0, W, false);
  } else if (warp >= kDrainWarp0) {
    // ------------------------------------------------------------ dQ drain
    // One warp per TMEM lane quarter reads its 32 query rows of dQ(i) out of
    // tensor memory as soon as the MMA has produced them, frees the columns
    // for dP(i+1), then adds them to the fp32 accumulator as bulk reductions
    // by the TMA unit, staged through this warp's slot of kStagedUnits 2 KB
    // units: the first units straight from the tensor-memory loads, the rest
    // (d > 64) from registers once the first operation has read the slot.
    // Vector reductions straight from registers would queue in the
    // sub-partition's memory pipe ahead of the compute warps' shared-memory
    // traffic (measured 17 % slower at d = 128 and 4-6 % at d = 64).  The
    // compute warps never wait for this.
    const int qq = warp & 3;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    constexpr int kUnitsQ = HD / 16;                      // 16-column units of this lane quarter
    constexpr int kStaged = kUnitsQ < kStagedUnits ? kUnitsQ : kStagedUnits;
    constexpr int kHeld = kUnitsQ - kStaged;              // units held in registers for a second round
    constexpr bool det = kDet;                            // store into this key block's slice instead of adding
    const uint32_t slot = sbase + Ly::kStage + qq * (kStagedUnits * 2048);
    bool ok = true;
    for (int i = 0; i < n_iter; ++i) {
      const int db = kSB == 2 ? ((i + 1) & 1) : 0;  // with two S buffers: the buffer holding dQ(i)
      const uint32_t tQ = tdQ(i) + lane_off;
      if (!(ok = warp_wait(barm(DQ_FULL0, db), kSB == 2 ? (i >> 1) & 1 : i & 1, W))) break;
      ptx::tc_fence_after();
      float* dst = prm.dq_accum + (det ? kb * prm.slice_elems : 0) +
                   dq_unit_offset(bh, prm.n_tiles, q_first + i, qq, 0, HD);
      if (lane == 0) ptx::bulk_wait_read_all();
      __syncwarp();
      // staged units, 32 columns (two units) per TMEM load
#pragma unroll
      for (int u = 0; u < kStaged; u += 2) {
        uint32_t r[32];
        ptx::tmem_ld32(tQ + u * 16, r);
#pragma unroll
        for (int v = 0; v < 2; ++v)
#pragma unroll
          for (int g = 0; g < 4; ++g)
            ptx::st_shared_v4(slot + (u + v) * 2048 + g * 512 + lane * 16, r[v * 16 + 4 * g], r[v * 16 + 4 * g + 1],
                              r[v * 16 + 4 * g + 2], r[v * 16 + 4 * g + 3]);
      }
      uint32_t h[kHeld > 0 ? kHeld * 16 : 1];
      if constexpr (kHeld == 4) {
        ptx::tmem_ld64(tQ + kStaged * 16, tQ + kStaged * 16 + 32, *reinterpret_cast<uint32_t(*)[64]>(h));
      } else if constexpr (kHeld == 2) {
        ptx::tmem_ld32(tQ + kStaged * 16, *reinterpret_cast<uint32_t(*)[32]>(h));
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(barm(DQ_EMPTY0, db));  // the columns are free for dP(i+1) (or S(i+3))
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (det)
          ptx::bulk_store(dst, slot, kStaged * 2048);
        else
          ptx::bulk_reduce_add_f32(dst, slot, kStaged * 2048);
        ptx::bulk_commit();
      }
      if constexpr (kHeld > 0) {
        // second round through the same slot once the first has been read
        if (lane == 0) ptx::bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int u = 0; u < kHeld; ++u)
#pragma unroll
          for (int g = 0; g < 4; ++g)
            ptx::st_shared_v4(slot + u * 2048 + g * 512 + lane * 16, h[u * 16 + 4 * g], h[u * 16 + 4 * g + 1],
                              h[u * 16 + 4 * g + 2], h[u * 16 + 4 * g + 3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (det)
            ptx::bulk_store(dst + kStaged * kDqUnitFloats, slot, kHeld * 2048);
          else
            ptx::bulk_reduce_add_f32(dst + kStaged * kDqUnitFloats, slot, kHeld * 2048);
          ptx::bulk_commit();
        }
      }
    }
    // Shared memory is released at exit, so this warp's last operations must
    // have read their staging slots.  Their writes to global memory need not
    // be waited for (they are complete when the grid is), except in the
    // single-launch backward, which publishes them.
    if (lane == 0) {
      ptx::bulk_wait_read_all();
      if (kFused) {
        ptx::bulk_wait_all();
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute
    const int qq = warp & 3;               // TMEM lane quarter
    const int G = warp >> 2;               // column quarter
    const int t = qq * 32 + lane;          // TMEM lane
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const int kr = k0 + t;                 // key row of S, dP, dV, dK
    const bool key_ok = kr < prm.Nk;
    const int kd = kRect ? k0 - prm.offset : k0;  // key k0 + t visible to query q iff q - kd >= t
    const float sl2 = prm.scale * kLog2e;
    uint32_t pk[16];                       // P for this warp's 32 query columns, bf16 pairs
    bool ok = true;
    if constexpr (kSB == 1) {
      // one S buffer (d > 64)
      const int c0 = G * 32;               // query columns [c0, c0 + 32) of S, dP
      for (int i = 0; i < n_iter; ++i) {
        const int st = i & 1;
        const uint32_t ph = i & 1;
        const int q0 = (q_first + i) * kBlk;
        // ---- P(i)
        // S(i); L(i) rows
        if (!(ok = warp_wait2(bar(S_FULL0), ph, barm(QFULL0, st), (i >> 1) & 1, W))) break;
        const uint32_t tSi = tm + Ly::kColS;
        ptx::tc_fence_after();
        {
          uint32_t r[32];
          ptx::tmem_ld32(tSi + lane_off + c0, r);
          const uint32_t sLa = sbase + Ly::kL + st * kBlk * 4 + c0 * 4;
          // key k0 + t is visible to query q0 + col iff col >= t - rel; the
          // block needs the mask unless every entry passes (rel >= 127).
          // Square problems: rel = 0 on the diagonal block only.
          const int rel = kRect ? q0 - kd : 0;
          const bool diag = prm.causal && (kRect ? rel < kBlk - 1 : q0 == k0);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 l4 = ptx::ld_shared_f4(sLa + j * 4);
            float p0 = ptx::ex2(fmaf(__uint_as_float(r[j + 0]), sl2, -l4.x));
            float p1 = ptx::ex2(fmaf(__uint_as_float(r[j + 1]), sl2, -l4.y));
            float p2 = ptx::ex2(fmaf(__uint_as_float(r[j + 2]), sl2, -l4.z));
            float p3 = ptx::ex2(fmaf(__uint_as_float(r[j + 3]), sl2, -l4.w));
            if (diag) {
              const int col = c0 + j;
              const int lim = t - rel;  // masked iff col < lim
              p0 = col + 0 < lim ? 0.f : p0;
              p1 = col + 1 < lim ? 0.f : p1;
              p2 = col + 2 < lim ? 0.f : p2;
              p3 = col + 3 < lim ? 0.f : p3;
            }
            pk[j / 2] = ptx::pack_bf16x2(p0, p1);
            pk[j / 2 + 1] = ptx::pack_bf16x2(p2, p3);
          }
          if (!key_ok) {
#pragma unroll
            for (int k = 0; k < 16; ++k) pk[k] = 0u;
          }
          // P columns [c0, c0 + 16) lie over this warp's own S columns
          ptx::tmem_st16(tSi + lane_off + c0, &pk[0]);
          ptx::tmem_st_wait();
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(P_FULL));
        // ---- dS(i).  Written after DP_FULL(i), which completes after dK(i-1),
        // the last reader of dS(i-1).
        if (!(ok = warp_wait(bar(DP_FULL), ph, W))) break;
        ptx::tc_fence_after();
        {
          uint32_t r[32];
          ptx::tmem_ld32(tm + Ly::kColdP + lane_off + c0, r);
          const uint32_t sDa = sbase + Ly::kD + st * kBlk * 4 + c0 * 4;
          uint32_t ds[16];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            // dS = P * (dP - D): the difference in fp32 (dP and D nearly
            // cancel), then one bf16x2 product with the packed bf16 P
            const float4 d4 = ptx::ld_shared_f4(sDa + j * 4);
            const uint32_t g01 = ptx::pack_bf16x2(__uint_as_float(r[j + 0]) - d4.x, __uint_as_float(r[j + 1]) - d4.y);
            const uint32_t g23 = ptx::pack_bf16x2(__uint_as_float(r[j + 2]) - d4.z, __uint_as_float(r[j + 3]) - d4.w);
            ds[j / 2] = ptx::mul_bf16x2(pk[j / 2], g01);
            ds[j / 2 + 1] = ptx::mul_bf16x2(pk[j / 2 + 1], g23);
          }
          // row t of dS^T, query columns [c0, c0 + 32): chunk G / 2, 16-byte
          // pieces 4 * (G % 2) .. +3, 128-byte swizzle (piece XOR row % 8)
          const uint32_t row = sdS + (G >> 1) * Ly::kChunk + t * 128;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t piece = (uint32_t)((G & 1) * 4 + u);
            ptx::st_shared_v4(row + ((piece ^ (uint32_t)(t & 7)) << 4), ds[4 * u], ds[4 * u + 1], ds[4 * u + 2],
                              ds[4 * u + 3]);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(DS_FULL));
      }
    } else {
      // two S buffers (d <= 64)
      // Query columns of S and dP this warp owns: [cA, cA + 16) and
      // [cB, cB + 16), so that its P (16 packed columns) goes over its own
      // first 16 and the upper 64 columns of the buffer are free once S has
      // been read.  Element j of the 32 is column col(j).
      const int cA = 16 * G, cB = 64 + 16 * G;
      auto col = [&](int j) -> int { return j < 16 ? cA + j : cB + (j - 16); };
      auto ld_cols = [&](uint32_t base, uint32_t (&r)[32]) {
        ptx::tmem_ld16x2(base + lane_off + cA, base + lane_off + cB, r);
      };

      for (int i = 0; i < n_iter; ++i) {
        const int qs = ring_stage<kQSt>(i);  // Q stage (with the L and D rows)
        const int q0 = (q_first + i) * kBlk;
        // ---- P(i)
        // S(i); L(i) rows
        if (!(ok = warp_wait2(barm(S_FULL0, i & 1), (i >> 1) & 1, barm(QFULL0, qs), ring_phase<kQSt>(i), W))) break;
        const uint32_t tSi = tS(i);
        ptx::tc_fence_after();
        {
          uint32_t r[32];
          ld_cols(tSi, r);
          // the upper columns may take dQ(i-1) now
          ptx::tc_fence_before();
          ptx::mbar_arrive(barm(S_READ0, i & 1));
          // L of columns [cA, cA + 16) and [cB, cB + 16)
          const uint32_t sLa = sbase + Ly::kL + qs * kBlk * 4 + cA * 4, sLb = sLa + (cB - cA) * 4;
          // key k0 + t is visible to query q0 + c iff c >= t - rel; the
          // block needs the mask unless every entry passes (rel >= 127).
          // Square problems: rel = 0 on the diagonal block only.
          const int rel = kRect ? q0 - kd : 0;
          const bool diag = prm.causal && (kRect ? rel < kBlk - 1 : q0 == k0);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 l4 = ptx::ld_shared_f4(j < 16 ? sLa + j * 4 : sLb + (j - 16) * 4);
            float p0 = ptx::ex2(fmaf(__uint_as_float(r[j + 0]), sl2, -l4.x));
            float p1 = ptx::ex2(fmaf(__uint_as_float(r[j + 1]), sl2, -l4.y));
            float p2 = ptx::ex2(fmaf(__uint_as_float(r[j + 2]), sl2, -l4.z));
            float p3 = ptx::ex2(fmaf(__uint_as_float(r[j + 3]), sl2, -l4.w));
            if (diag) {
              const int c = col(j);
              const int lim = t - rel;  // masked iff c < lim
              p0 = c + 0 < lim ? 0.f : p0;
              p1 = c + 1 < lim ? 0.f : p1;
              p2 = c + 2 < lim ? 0.f : p2;
              p3 = c + 3 < lim ? 0.f : p3;
            }
            pk[j / 2] = ptx::pack_bf16x2(p0, p1);
            pk[j / 2 + 1] = ptx::pack_bf16x2(p2, p3);
          }
          if (!key_ok) {
#pragma unroll
            for (int k = 0; k < 16; ++k) pk[k] = 0u;
          }
          // P columns [cA, cA + 16) lie over this warp's own S columns
          ptx::tmem_st16(tSi + lane_off + cA, &pk[0]);
          ptx::tmem_st_wait();
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(P_FULL));
        // ---- dS(i).  dP(i) is released as soon as it is in registers, and
        // dS(i) waits for DS_EMPTY, which follows dK(i-1) and dQ(i-1).
        if (!(ok = warp_wait(bar(DP_FULL), i & 1, W))) break;
        ptx::tc_fence_after();
        {
          uint32_t r[32];
          ld_cols(tm + Ly::kColdP, r);
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(DP_READ));
          const uint32_t sDa = sbase + Ly::kD + qs * kBlk * 4 + cA * 4, sDb = sDa + (cB - cA) * 4;
          uint32_t ds[16];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            // dS = P * (dP - D): the difference in fp32 (dP and D nearly
            // cancel), then one bf16x2 product with the packed bf16 P
            const float4 d4 = ptx::ld_shared_f4(j < 16 ? sDa + j * 4 : sDb + (j - 16) * 4);
            const uint32_t g01 = ptx::pack_bf16x2(__uint_as_float(r[j + 0]) - d4.x, __uint_as_float(r[j + 1]) - d4.y);
            const uint32_t g23 = ptx::pack_bf16x2(__uint_as_float(r[j + 2]) - d4.z, __uint_as_float(r[j + 3]) - d4.w);
            ds[j / 2] = ptx::mul_bf16x2(pk[j / 2], g01);
            ds[j / 2 + 1] = ptx::mul_bf16x2(pk[j / 2 + 1], g23);
          }
          if (i >= 1 && !(ok = warp_wait(bar(DS_EMPTY), (i - 1) & 1, W))) break;
          // row t of dS^T: 16-byte pieces (8 query columns) of the 64-column
          // chunks, 128-byte swizzle (piece XOR row % 8).  ds[4u .. 4u + 3]
          // holds this warp's columns col(8u) .. +7: chunk u / 2, piece
          // 2G + u % 2.
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t chunk = (uint32_t)(u >> 1);
            const uint32_t piece = (uint32_t)(2 * G + (u & 1));
            ptx::st_shared_v4(sdS + chunk * Ly::kChunk + t * 128 + ((piece ^ (uint32_t)(t & 7)) << 4), ds[4 * u],
                              ds[4 * u + 1], ds[4 * u + 2], ds[4 * u + 3]);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(DS_FULL));
      }
    }
    // ---- epilogue: this lane's key row t of dV (warps G = 0, 1) or scale *
    // dK (G = 2, 3), half the columns each, into shared memory as the
    // 64-column, 128-byte-swizzled chunks of a TMA box: dV into the dS buffer,
    // dK into the first Q stage (their last readers, dK and dQ of the last
    // block, are done at ACC_FULL, and no Q load is left in flight).  Two TMA
    // stores then write whole lines (rows past N_k and columns past d are not
    // written).  Stores from registers, each lane its own row 16 bytes at a
    // time, took ~6 k cycles per CTA at d = 128; staging dK over the dQ
    // staging slots, which made it wait for the last dQ drain, cost 0.5-1.3 %.
    // Every compute warp reaches the named barrier below, also after a wait
    // ran out (which set the CTA's abort flag): the stores are then skipped.
    const bool isV = G < 2;
    if (ok && warp_wait(bar(ACC_FULL), 0, W)) {
      ptx::tc_fence_after();
      constexpr int kHalf = HD / 2;
      const int cc = (G & 1) * kHalf;
      const uint32_t src = tm + (isV ? Ly::kColdV : Ly::kColdK) + lane_off + cc;
      const uint32_t dst = isV ? sdS : sQ(0);
      const float mul = isV ? 1.f : prm.scale;
#pragma unroll 1
      for (int c = 0; c < kHalf; c += 16) {
        uint32_t v[16];
        ptx::tmem_ld16(src + c, v);
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // 8 columns (16 bytes) each
          const int col = cc + c + 8 * q;
          const uint32_t piece = (uint32_t)((col & 63) >> 3);
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = ptx::pack_bf16x2(__uint_as_float(v[8 * q + 2 * e]) * mul, __uint_as_float(v[8 * q + 2 * e + 1]) * mul);
          ptx::st_shared_v4(dst + (col >> 6) * Ly::kChunk + t * 128 + ((piece ^ (uint32_t)(t & 7)) << 4), w[0], w[1],
                            w[2], w[3]);
        }
      }
      ptx::fence_proxy_async_smem();
    }
    ptx::bar_sync(1, kComputeThreads);
    if (warp == 0 && lane == 0 && !*abort_flag) {
#pragma unroll
      for (int c = 0; c < LD / 64; ++c) {
        ptx::tma_store_4d(&tmdV, sdS + c * Ly::kChunk, c * 64, k0, h, b);
        ptx::tma_store_4d(&tmdK, sQ(0) + c * Ly::kChunk, c * 64, k0, h, b);
      }
      ptx::bulk_commit();
      // shared memory is released at exit: the stores must have read it
      // (and, in the single-launch backward, be complete)
      if (kFused)
        ptx::bulk_wait_all();
      else
        ptx::bulk_wait_read_all();
    }
    __syncwarp();
  }

  if (kFused) __threadfence();  // this thread's reductions and stores before the release
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tm, Ly::kTmemCols);
  }
  if (kFused && threadIdx.x == 0) {
    __threadfence();
    atomicAdd(done, 1);
  }
}

template <int HD, bool kDet, bool kRect, bool kCount>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                     const BwdParams prm) {
  // work item: key block kb of head (b, h).  Heads are taken in groups of
  // prm.head_group so the CTAs resident at any time share a few heads' Q, dO
  // and dQ accumulator in L2; inside a group the key blocks go round the
  // heads, key block 0 (the longest causal walk) first, so the short walks of
  // the last group fill the SMs at the end of the grid.
  const int hg = prm.head_group;
  const int bh_total = prm.B * prm.H;
  const int grp = blockIdx.x / (hg * prm.nk_tiles);
  const int gsize = min(hg, bh_total - grp * hg);
  const int r = blockIdx.x - grp * hg * prm.nk_tiles;
  bwd_block<HD, kDet, kRect, false, kCount>(tmQ, tmK, tmV, tmdO, tmdK, tmdV, prm, r / gsize, grp * hg + r % gsize,
                                            nullptr, 0, nullptr);
}

// ---------------------------------------------------------------------------
// Single-launch backward: preprocess (D, zeroed accumulator), the key blocks
// and convert as items of one grid.  Each CTA takes a ticket in the order
// CTAs start, and the ticket names its item; an item only waits for items
// with smaller tickets (started, so resident or finished), so no wait can
// depend on a CTA that has not been scheduled.  Order, with heads in groups
// of kHeadGroup:  P(0), then for each group k: P(k+1), B(k), C(k-1); last
// C(G-1).  P = D and the zeroed accumulator of kTilesPerItem 128-row query
// tiles, B = one key block (waits until every P of its head is done), C =
// the dQ conversion of kTilesPerItem query tiles (waits until every B of its
// head is done).
// ---------------------------------------------------------------------------
enum : int { kItemPre = 0, kItemBwd = 1, kItemCvt = 2 };
constexpr int kTilesPerItem = 8;  // query tiles per P and per C item

struct FusedParams {
  const __nv_bfloat16* O;
  const __nv_bfloat16* dO;
  __nv_bfloat16* dQ;
  float* D;
  // [0] ticket; [1, 1 + BH) P items done per head; [1 + BH, 1 + 2 BH) B items
  // done per head; zeroed before the launch
  int32_t* sync;
};

// Ticket t -> (role, bh, idx): idx is the item of query tiles (P, C; T items
// per head) or the key block (B; Tk per head).
__host__ __device__ inline void fused_item(int64_t t, int BH, int T, int Tk, int& role, int& bh, int& idx) {
  const int G = (BH + kHeadGroup - 1) / kHeadGroup;
  auto gs = [&](int g) { return BH - kHeadGroup * g < kHeadGroup ? BH - kHeadGroup * g : kHeadGroup; };
  auto sp = [&](int k) -> int64_t { return k + 1 < G ? (int64_t)gs(k + 1) * T : 0; };
  auto sb = [&](int k) -> int64_t { return (int64_t)gs(k) * Tk; };
  auto sc = [&](int k) -> int64_t { return k >= 1 ? (int64_t)gs(k - 1) * T : 0; };
  auto in_slot = [&](int k, int64_t o) {
    if (o < sp(k)) {
      role = kItemPre;
      bh = kHeadGroup * (k + 1) + (int)(o / T);
      idx = (int)(o % T);
      return;
    }
    o -= sp(k);
    if (o < sb(k)) {  // key blocks go round the heads of the group, block 0 first
      role = kItemBwd;
      bh = kHeadGroup * k + (int)(o % gs(k));
      idx = (int)(o / gs(k));
      return;
    }
    o -= sb(k);
    role = kItemCvt;
    bh = kHeadGroup * (k - 1) + (int)(o / T);
    idx = (int)(o % T);
  };
  const int64_t p0 = (int64_t)gs(0) * T;
  if (t < p0) {
    role = kItemPre;
    bh = (int)(t / T);
    idx = (int)(t % T);
    return;
  }
  t -= p0;
  int k = 0;
  // slots 1 .. full - 2 only involve full groups: one size, skipped by division
  const int full = BH / kHeadGroup;
  const int64_t s0 = sp(0) + sb(0) + sc(0);
  if (t < s0) return in_slot(0, t);
  t -= s0;
  k = 1;
  if (full >= 3) {
    const int64_t U = (int64_t)kHeadGroup * (2 * (int64_t)T + Tk);
    const int64_t nu = full - 2;
    if (t < nu * U) return in_slot(1 + (int)(t / U), t % U);
    t -= nu * U;
    k = full - 1;
  }
  for (; k < G; ++k) {
    const int64_t sk = sp(k) + sb(k) + sc(k);
    if (t < sk) return in_slot(k, t);
    t -= sk;
  }
  role = kItemCvt;  // C(G - 1)
  bh = kHeadGroup * (G - 1) + (int)(t / T);
  idx = (int)(t % T);
}

// P item: D for query rows [tile * 128, +128) of head bh (computed exactly as
// the preprocess kernel does, see row_dot.cuh), and the accumulator tile
// zeroed.
template <int HD>
__device__ __forceinline__ void pre_tile(const BwdParams& prm, const FusedParams& fp, int bh, int tile, bool zero) {
  using RD = RowDot<__nv_bfloat16, HD>;
  constexpr int kRowsPerStep = kComputeThreads / RD::kLanes;
  const int b = bh / prm.H, h = bh % prm.H;
  const int64_t head = (int64_t)b * prm.sb + (int64_t)h * prm.sh;
  if (threadIdx.x < kComputeThreads) {
    const int sub = threadIdx.x % RD::kLanes, row_in_step = threadIdx.x / RD::kLanes;
#pragma unroll
    for (int r0 = 0; r0 < kBlk; r0 += kRowsPerStep) {
      const int n = tile * kBlk + r0 + row_in_step;
      float acc = n < prm.N ? RD::partial(fp.O + head + (int64_t)n * prm.sn, fp.dO + head + (int64_t)n * prm.sn, sub)
                            : 0.f;
      acc = RD::reduce(acc);
      if (sub == 0 && n < prm.N) fp.D[(int64_t)bh * prm.N + n] = acc;
    }
  }
  if (zero) {
    float4* z = reinterpret_cast<float4*>(prm.dq_accum + ((int64_t)bh * prm.n_tiles + tile) * kBlk * HD);
    for (int k = threadIdx.x; k < kBlk * HD / 4; k += kThreads) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// P item: query tiles [item * kTilesPerItem, +kTilesPerItem) of head bh.
template <int HD>
__device__ __forceinline__ void pre_item(const BwdParams& prm, const FusedParams& fp, int bh, int item, bool zero) {
  const int t1 = min(prm.n_tiles, (item + 1) * kTilesPerItem);
  for (int tile = item * kTilesPerItem; tile < t1; ++tile) pre_tile<HD>(prm, fp, bh, tile, zero);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd(fp.sync + 1 + bh, 1);
}

// C item: dQ rows [tile * 128, +128) of head bh = bf16(scale * accumulator),
// once every key block of the head is done; the tile goes through shared
// memory to undo the unit-blocked layout.  Deterministic: the key blocks'
// slices are summed in increasing order (causal: those that reach the tile).
template <int HD, bool kDet>
__device__ __forceinline__ void cvt_tile(const BwdParams& prm, const FusedParams& fp, uint8_t* smem, int bh,
                                         int tile) {
  constexpr int kPitch = HD + 4;
  float* tile_s = reinterpret_cast<float*>(smem);
  const float4* src = reinterpret_cast<const float4*>(prm.dq_accum + ((int64_t)bh * prm.n_tiles + tile) * kBlk * HD);
  int last = 0;
  if (kDet) {
    last = prm.nk_tiles - 1;
    if (prm.causal) {
      const int64_t hi = (int64_t)tile * kBlk + kBlk - 1 + prm.offset;
      last = hi < 0 ? -1 : (hi / kBlk < last ? (int)(hi / kBlk) : last);
    }
  }
  const int64_t slice4 = prm.slice_elems / 4;
  // a tile is 4 x (HD / 16) units of [4 column groups][32 rows][4 columns]
  for (int k = threadIdx.x; k < kBlk * HD / 4; k += kThreads) {
    const int unit = k / 128, g = (k % 128) / 32, r = k % 32;
    const int row = (unit / (HD / 16)) * 32 + r, col = (unit % (HD / 16)) * 16 + g * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (last >= 0) v = __ldcg(src + k);
    for (int sl = 1; sl <= last; ++sl) {
      const float4 w = __ldcg(src + sl * slice4 + k);
      v.x += w.x;
      v.y += w.y;
      v.z += w.z;
      v.w += w.w;
    }
    *reinterpret_cast<float4*>(tile_s + row * kPitch + col) = v;
  }
  __syncthreads();
  const int b = bh / prm.H, h = bh % prm.H;
  __nv_bfloat16* out = fp.dQ + (int64_t)b * prm.sb + (int64_t)h * prm.sh;
  constexpr int kPerRow = HD / 8;  // 16-byte stores per row
  for (int k = threadIdx.x; k < kBlk * kPerRow; k += kThreads) {
    const int r = k / kPerRow, c = (k % kPerRow) * 8;
    const int n = tile * kBlk + r;
    if (n >= prm.N) continue;
    const float* v = tile_s + r * kPitch + c;
    uint4 u;
    u.x = ptx::pack_bf16x2(prm.scale * v[0], prm.scale * v[1]);
    u.y = ptx::pack_bf16x2(prm.scale * v[2], prm.scale * v[3]);
    u.z = ptx::pack_bf16x2(prm.scale * v[4], prm.scale * v[5]);
    u.w = ptx::pack_bf16x2(prm.scale * v[6], prm.scale * v[7]);
    *reinterpret_cast<uint4*>(out + (int64_t)n * prm.sn + c) = u;
  }
}

// C item: query tiles [item * kTilesPerItem, +kTilesPerItem) of head bh, once
// every key block of the head is done.
template <int HD, bool kDet>
__device__ __forceinline__ void cvt_item(const BwdParams& prm, const FusedParams& fp, uint8_t* smem, int bh,
                                         int item) {
  volatile int* flag = reinterpret_cast<volatile int*>(smem + kBlk * (HD + 4) * 4);
  const int BH = prm.B * prm.H;
  if (threadIdx.x == 0) {
    const bool ok = wait_counter(fp.sync + 1 + BH + bh, prm.nk_tiles, prm.wait_ns);
    if (!ok) atomicCAS(prm.status, 0, (int32_t)FA_ERR_TIMEOUT);
    *flag = ok;
  }
  __syncthreads();
  if (!*flag) return;
  const int t1 = min(prm.n_tiles, (item + 1) * kTilesPerItem);
  for (int tile = item * kTilesPerItem; tile < t1; ++tile) {
    cvt_tile<HD, kDet>(prm, fp, smem, bh, tile);
    __syncthreads();  // the shared tile is rewritten by the next one
  }
}

template <int HD, bool kDet, bool kRect>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                     const BwdParams prm, const FusedParams fp) {
  using Ly = Layout<(HD <= 64 ? 64 : 128)>;
  extern __shared__ __align__(1024) uint8_t smem[];
  volatile int32_t* slot = reinterpret_cast<volatile int32_t*>(smem + Ly::kMisc + 8);
  if (threadIdx.x == 0) *slot = atomicAdd(fp.sync, 1);
  __syncthreads();
  const int ticket = *slot;
  __syncthreads();  // the slot's bytes are free again before any role uses shared memory
  const int BH = prm.B * prm.H;
  int role, bh, idx;
  const int Ti = (prm.n_tiles + kTilesPerItem - 1) / kTilesPerItem;  // P and C items per head
  fused_item(ticket, BH, Ti, prm.nk_tiles, role, bh, idx);
  if (role == kItemBwd)
    bwd_block<HD, kDet, kRect, true, false>(tmQ, tmK, tmV, tmdO, tmdK, tmdV, prm, idx, bh, fp.sync + 1 + bh, Ti,
                                     fp.sync + 1 + BH + bh);
  else if (role == kItemPre)
    pre_item<HD>(prm, fp, bh, idx, !kDet);
  else
    cvt_item<HD, kDet>(prm, fp, smem, bh, idx);
}

template <int HD, bool kDet, bool kRect, bool kCount>
cudaError_t launch_hd(const fa_problem& p, const CUtensorMap* maps, const BwdParams& prm, cudaStream_t s) {
  using Ly = Layout<(HD <= 64 ? 64 : 128)>;
  cudaError_t e = cudaFuncSetAttribute(bwd_sm103_kernel<HD, kDet, kRect, kCount>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((int64_t)prm.nk_tiles * p.B * p.H));
  bwd_sm103_kernel<HD, kDet, kRect, kCount><<<grid, kThreads, Ly::kBytes, s>>>(maps[0], maps[1], maps[2], maps[3],
                                                                                maps[4], maps[5], prm);
  return cudaGetLastError();
}

template <int HD, bool kCount>
cudaError_t launch_d(const fa_problem& p, const CUtensorMap* maps, const BwdParams& prm, bool det, bool rect,
                     cudaStream_t s) {
  if (det)
    return rect ? launch_hd<HD, true, true, kCount>(p, maps, prm, s) : launch_hd<HD, true, false, kCount>(p, maps, prm, s);
  return rect ? launch_hd<HD, false, true, kCount>(p, maps, prm, s) : launch_hd<HD, false, false, kCount>(p, maps, prm, s);
}

template <int HD, bool kDet, bool kRect>
cudaError_t launch_fused_hd(const CUtensorMap* maps, const BwdParams& prm, const FusedParams& fp, int64_t items,
                            cudaStream_t s) {
  using Ly = Layout<(HD <= 64 ? 64 : 128)>;
  cudaError_t e = cudaFuncSetAttribute(bwd_fused_kernel<HD, kDet, kRect>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kBytes);
  if (e != cudaSuccess) return e;
  bwd_fused_kernel<HD, kDet, kRect><<<(unsigned)items, kThreads, Ly::kBytes, s>>>(maps[0], maps[1], maps[2], maps[3],
                                                                                maps[4], maps[5], prm, fp);
  return cudaGetLastError();
}

template <int HD>
cudaError_t launch_fused_d(const CUtensorMap* maps, const BwdParams& prm, const FusedParams& fp, int64_t items,
                           bool det, bool rect, cudaStream_t s) {
  if (det)
    return rect ? launch_fused_hd<HD, true, true>(maps, prm, fp, items, s)
                : launch_fused_hd<HD, true, false>(maps, prm, fp, items, s);
  return rect ? launch_fused_hd<HD, false, true>(maps, prm, fp, items, s)
              : launch_fused_hd<HD, false, false>(maps, prm, fp, items, s);
}

// Heads per group of the separate kernel's grid order.  Each key block of a
// head walks that head's Q and dO blocks and adds into its accumulator tiles,
// so the group's Q, dO and fp32 accumulator are what the resident CTAs
// re-read from L2; groups stay within kGroupL2Bytes of them (and at most
// kHeadGroup heads, which measured best while that fits).
constexpr int64_t kGroupL2Bytes = int64_t(48) << 20;
int head_group(const fa_problem& p) {
  const int64_t per_head = (int64_t)p.N * p.d * 2 * 2 + ceil_div(p.N, kBlk) * kBlk * p.d * 4;
  const int64_t g = kGroupL2Bytes / per_head;
  return g < 1 ? 1 : (g > kHeadGroup ? kHeadGroup : (int)g);
}

// Kernel parameters shared by the separate and the single-launch backward.
BwdParams bwd_params(const fa_problem& p, const float* L, const float* D, float* dq_accum, void* dK, void* dV,
                     int32_t* status, uint64_t wait_ns) {
  BwdParams prm;
  prm.pair_count = nullptr;
  prm.head_group = kHeadGroup;
  prm.L = L;
  prm.D = D;
  prm.dq_accum = dq_accum;
  prm.dK = (__nv_bfloat16*)dK;
  prm.dV = (__nv_bfloat16*)dV;
  prm.status = status;
  prm.wait_ns = wait_ns;
  prm.B = p.B;
  prm.H = p.H;
  prm.N = p.N;
  prm.Nk = p.N_k;
  prm.n_tiles = (int)ceil_div(p.N, kBlk);
  prm.nk_tiles = (int)ceil_div(p.N_k, kBlk);
  prm.offset = (int)causal_offset(p);
  prm.sb = p.stride_b;
  prm.sh = p.stride_h;
  prm.sn = p.stride_n;
  prm.ksb = p.kstride_b;
  prm.ksh = p.kstride_h;
  prm.ksn = p.kstride_n;
  prm.scale = p.scale;
  prm.causal = p.causal;
  prm.slice_elems = deterministic(p) ? dq_slice_elems(p) : 0;
  return prm;
}

// Maps and parameters of one fa_bwd launch, then the kernel for p's head dim.
template <bool kCount>
cudaError_t launch_bwd(const fa_problem& p, const void* Q, const void* K, const void* V, const void* dO,
                       const float* L, const float* D, float* dq_accum, void* dK, void* dV, int32_t* status,
                       uint64_t wait_ns, cudaStream_t s, unsigned long long* pair_count) {
  CUtensorMap maps[6];
  if (!make_bf16_tile_map(&maps[0], Q, p, false) || !make_bf16_tile_map(&maps[1], K, p, true) ||
      !make_bf16_tile_map(&maps[2], V, p, true) || !make_bf16_tile_map(&maps[3], dO, p, false) ||
      !make_bf16_tile_map(&maps[4], dK, p, true) || !make_bf16_tile_map(&maps[5], dV, p, true))
    return cudaErrorInvalidValue;
  BwdParams prm = bwd_params(p, L, D, dq_accum, dK, dV, status, wait_ns);
  prm.pair_count = pair_count;
  prm.head_group = head_group(p);
  const bool det = prm.slice_elems > 0;
  const bool rect = p.causal && prm.offset != 0;
  switch (p.d) {
    case 32: return launch_d<32, kCount>(p, maps, prm, det, rect, s);
    case 64: return launch_d<64, kCount>(p, maps, prm, det, rect, s);
    case 96: return launch_d<96, kCount>(p, maps, prm, det, rect, s);
    case 128: return launch_d<128, kCount>(p, maps, prm, det, rect, s);
  }
  return cudaErrorInvalidValue;
}
}  // namespace

#if FA_BWD_SM103_COUNTING
// Built by fa_bwd_sm103_count.cu: the counting instantiations only.
cudaError_t launch_bwd_sm103_count(const fa_problem& p, const void* Q, const void* K, const void* V,
                                   const void* dO, const float* L, const float* D, float* dq_accum, void* dK,
                                   void* dV, int32_t* status, uint64_t wait_ns, cudaStream_t s,
                                   unsigned long long* pair_count) {
  return launch_bwd<true>(p, Q, K, V, dO, L, D, dq_accum, dK, dV, status, wait_ns, s, pair_count);
}
#else
cudaError_t launch_bwd_sm103(const fa_problem& p, const void* Q, const void* K, const void* V, const void* dO,
                             const float* L, const float* D, float* dq_accum, void* dK, void* dV, int32_t* status,
                             uint64_t wait_ns, cudaStream_t s) {
  return launch_bwd<false>(p, Q, K, V, dO, L, D, dq_accum, dK, dV, status, wait_ns, s, nullptr);
}

int64_t fused_items(const fa_problem& p) {
  return (int64_t)p.B * p.H * (2 * ceil_div(ceil_div(p.N, kBlk), kTilesPerItem) + ceil_div(p.N_k, kBlk));
}

cudaError_t launch_bwd_fused_sm103(const fa_problem& p, const void* Q, const void* K, const void* V, const void* O,
                                   const void* dO, const float* L, float* D, float* dq_accum, int32_t* sync, void* dQ,
                                   void* dK, void* dV, int32_t* status, uint64_t wait_ns, cudaStream_t s) {
  const int64_t items = fused_items(p);
  if (items > 0x7fffffff) return cudaErrorInvalidValue;
  CUtensorMap maps[6];
  if (!make_bf16_tile_map(&maps[0], Q, p, false) || !make_bf16_tile_map(&maps[1], K, p, true) ||
      !make_bf16_tile_map(&maps[2], V, p, true) || !make_bf16_tile_map(&maps[3], dO, p, false) ||
      !make_bf16_tile_map(&maps[4], dK, p, true) || !make_bf16_tile_map(&maps[5], dV, p, true))
    return cudaErrorInvalidValue;
  const BwdParams prm = bwd_params(p, L, D, dq_accum, dK, dV, status, wait_ns);
  FusedParams fp;
  fp.O = (const __nv_bfloat16*)O;
  fp.dO = (const __nv_bfloat16*)dO;
  fp.dQ = (__nv_bfloat16*)dQ;
  fp.D = D;
  fp.sync = sync;
  cudaError_t e = cudaMemsetAsync(sync, 0, sizeof(int32_t) * (1 + 2 * (size_t)p.B * p.H), s);
  if (e != cudaSuccess) return e;
  const bool det = prm.slice_elems > 0;
  const bool rect = p.causal && prm.offset != 0;
  switch (p.d) {
    case 32: return launch_fused_d<32>(maps, prm, fp, items, det, rect, s);
    case 64: return launch_fused_d<64>(maps, prm, fp, items, det, rect, s);
    case 96: return launch_fused_d<96>(maps, prm, fp, items, det, rect, s);
    case 128: return launch_fused_d<128>(maps, prm, fp, items, det, rect, s);
  }
  return cudaErrorInvalidValue;
}

#endif  // FA_BWD_SM103_COUNTING

}  // namespace fa
