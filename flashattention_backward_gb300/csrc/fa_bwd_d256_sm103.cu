// FlashAttention-2 backward for bf16 at head dim 256 on the sm_100-family
// tensor cores (tcgen05 MMA, accumulators in tensor memory, TMA-staged
// operands).
//
// At d = 256 the dK and dV accumulators of a 128-row key block would fill all
// 512 tensor-memory columns, and a 128 x 256 bf16 tile of each of Q, K, V and
// dO is 256 KB of shared memory.  The work of a key block therefore goes to
// two CTAs, split by output columns: CTA (j, half) accumulates dV_j[:, half]
// and dK_j[:, half] (128 columns each) and adds dQ[:, half] into the fp32
// accumulator.  Each of the two recomputes the full S^T and dP^T, which
// contract over all 256 columns.  Query blocks are 64 rows, so one Q and one
// dO tile (32 KB each) fit beside the resident K_j and V_j (64 KB each).
//
// Loop order, scale placement and masking follow "CUDA 算子工程" ch.16
// (§16.2 key-block outer loop, §16.3 fp32 dQ accumulator with fire-and-forget
// reductions, §16.8 item 2 causal block skipping), as in the head-dim <= 128
// kernel.  The scores are transposed (TMEM lane = key row), P^T feeds
// dV += P^T dO from tensor memory, and dS^T goes to shared memory.
//
// dQ is produced for a 128-row query tile at a time: dQ = dS K_j[:, half] with
// the dS of two consecutive 64-row blocks stacked as the 128 rows of the A
// operand (two 64-query blocks of the MN-major layout), so its rows land in
// tensor-memory lanes in the accumulator's own tile order.  The walk over
// query blocks therefore starts on a 128-row tile boundary; a causal block
// that lies wholly before the diagonal is computed with P = 0.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,64) [64,128)    S^T of even / odd query blocks; P^T (bf16) over it
//   [128,192) [192,256) dP^T of even / odd blocks; the dQ tile of the two
//                      blocks over both once both dS are in shared memory
//   [256,384)          dV accumulator (this CTA's 128 columns)
//   [384,512)          dK accumulator
//
// Shared memory: K_j, V_j (4 chunks of 128 rows x 64 columns each), Q_i and
// dO_i (4 chunks of 64 rows x 64 columns each, one stage), dS^T of two
// blocks, L and D rows of two blocks, barriers.  The Q and dO chunks of the
// other CTA's column half are read only by S^T and dP^T, so they are freed
// (and the next block's loaded) as soon as those products finish; this CTA's
// own chunks are read again by dK += dS^T Q and dV += P^T dO.  S^T(i+1)
// contracts over the other half first, while the own half still loads.
//
// Warp roles (448 threads):
//   warps 0-7   compute: TMEM lane quarter w % 4, query columns
//               [32 (w / 4), +32).  P = exp2(S scale log2e - L log2e) -> bf16
//               into TMEM; dS = P (dP - D) -> bf16 into shared memory.
//               Epilogue: dV (w < 4), scale * dK (w >= 4).
//   warps 8-11  dQ drain, one per lane quarter: tensor memory -> registers ->
//               vector reductions into the accumulator.
//   warp 12     TMA producer (K, V once; Q, dO per block; L, D rows).
//   warp 13     TMEM allocator and MMA issuer (one elected lane issues).
//
// MMA issue order per query block i:
//   dV(i)  S(i+1)[other half]  dK(i)  [dQ(tile) after odd i]  S(i+1)[own half]  dP(i+1)
//
// Every wait is bounded; when one runs out the CTA records FA_ERR_TIMEOUT,
// waits for its own TMA loads and MMAs, frees tensor memory and exits.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "dq_layout.cuh"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kHD = 256;         // head dim served here
constexpr int kHalfD = 128;      // output columns per CTA
constexpr int kKeyRows = 128;    // key block (TMEM lanes)
constexpr int kQRows = 64;       // query block
constexpr int kComputeWarps = 8;
constexpr int kDrainWarp0 = kComputeWarps;      // warps 8-11
constexpr int kProducerWarp = kDrainWarp0 + 4;  // warp 12
constexpr int kMmaWarp = kProducerWarp + 1;     // warp 13
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kDrainThreads = 128;
constexpr int kHeadGroup = 4;  // heads whose key blocks interleave in the grid order
constexpr float kLog2e = 1.4426950408889634f;

enum BarId {
  KV_FULL = 0,  // K, V landed
  QO_FULL,      // Q(i): the other half's chunks landed
  QW_FULL,      // Q(i): this CTA's own chunks landed
  DOO_FULL,     // dO(i): other half landed
  DOW_FULL,     // dO(i): own half landed
  QO_EMPTY,     // S(i) done: Q other-half chunks free
  QW_EMPTY,     // dK(i) done: Q own chunks free
  DOO_EMPTY,    // dP(i) done: dO other-half chunks free
  DOW_EMPTY,    // dV(i) done: dO own chunks free
  LD_FULL0,     // L, D rows of an even / odd block written (32 producer lanes)
  LD_FULL1,
  S_FULL0,      // S^T of an even / odd block in TMEM
  S_FULL1,
  DV_DONE0,     // dV of an even / odd block done: its S/P columns reusable
  DV_DONE1,
  P_FULL,       // P^T(i) in TMEM (every compute thread)
  DP_FULL,      // dP^T(i) in TMEM
  DS_FULL,      // dS^T(i) in shared memory (every compute thread)
  DS_EMPTY,     // dK and dQ of a tile done: both dS^T slots reusable
  DQ_FULL,      // dQ of a tile in TMEM
  DQ_EMPTY,     // dQ drained from TMEM (every drain thread)
  ACC_FULL,     // every MMA done: dK, dV final
  kNumBars
};

struct Ly {
  static constexpr int kKChunk = kKeyRows * 128;  // 128 rows x 128 bytes
  static constexpr int kQChunk = kQRows * 128;    // 64 rows x 128 bytes
  static constexpr int kK = 0;
  static constexpr int kV = kK + 4 * kKChunk;
  static constexpr int kQ = kV + 4 * kKChunk;
  static constexpr int kdO = kQ + 4 * kQChunk;
  static constexpr int kdS = kdO + 4 * kQChunk;         // 2 slots of 128 keys x 64 queries bf16
  static constexpr int kdSSlot = kKeyRows * 128;
  static constexpr int kL = kdS + 2 * kdSSlot;          // 2 slots x 64 fp32 (L log2 e)
  static constexpr int kD = kL + 2 * kQRows * 4;        // 2 slots x 64 fp32
  static constexpr int kBar = kD + 2 * kQRows * 4;
  static constexpr int kMisc = kBar + kNumBars * 8;     // TMEM base address, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr uint32_t kColS0 = 0, kColS1 = 64, kColdP0 = 128, kColdP1 = 192, kColdQ = 128;
  static constexpr uint32_t kColdV = 256, kColdK = 384;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kBytes <= 232448, "shared memory budget");
};

struct D256Params {
  const float* L;
  const float* D;
  float* dq_accum;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  int32_t* status;
  uint64_t wait_ns;
  int B, H, N, Nk;
  int n_tiles;          // ceil(N / 128): dQ accumulator tiles
  int nk_tiles;         // ceil(Nk / 128): key blocks
  int offset;           // Nk - N: key j visible to query i iff j <= i + offset (causal)
  int64_t ksb, ksh, ksn;  // K-shaped strides (dK, dV written with these)
  float scale;
  int causal;
  int64_t slice_elems;  // > 0: deterministic, key block kb stores into slice kb
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const ptx::Waiter& w) {
  return __all_sync(0xffffffffu, ptx::wait_bounded(bar, parity, w, true));
}
__device__ __forceinline__ bool warp_wait2(uint32_t a, uint32_t pa, uint32_t b, uint32_t pb, const ptx::Waiter& w) {
  const bool done = (ptx::mbar_try_wait(a, pa) & ptx::mbar_try_wait(b, pb)) != 0;
  if (__all_sync(0xffffffffu, done)) return true;
  return __all_sync(0xffffffffu, ptx::wait_bounded(a, pa, w, true) && ptx::wait_bounded(b, pb, w, true));
}

// 128 fp32 columns of this thread's TMEM lane -> bf16 in global memory.
__device__ __forceinline__ void store_row128(uint32_t taddr, bool valid, __nv_bfloat16* dst, float mul) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    ptx::tmem_ld32(taddr + c * 32, r);
    if (valid) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint4 v;
        v.x = ptx::pack_bf16x2(__uint_as_float(r[8 * u + 0]) * mul, __uint_as_float(r[8 * u + 1]) * mul);
        v.y = ptx::pack_bf16x2(__uint_as_float(r[8 * u + 2]) * mul, __uint_as_float(r[8 * u + 3]) * mul);
        v.z = ptx::pack_bf16x2(__uint_as_float(r[8 * u + 4]) * mul, __uint_as_float(r[8 * u + 5]) * mul);
        v.w = ptx::pack_bf16x2(__uint_as_float(r[8 * u + 6]) * mul, __uint_as_float(r[8 * u + 7]) * mul);
        *reinterpret_cast<uint4*>(dst + c * 32 + u * 8) = v;
      }
    }
  }
}

// 32 fp32 columns (two 16-column units) of one query row into the dQ
// accumulator: unit u, column group g at float offset u * 512 + g * 128 + row * 4.
template <bool kDet>
__device__ __forceinline__ void drain32(float* unit0, int lane, const uint32_t (&r)[32]) {
#pragma unroll
  for (int v = 0; v < 2; ++v)
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float* p = unit0 + v * kDqUnitFloats + g * 128 + lane * 4;
      const float a = __uint_as_float(r[16 * v + 4 * g]), b = __uint_as_float(r[16 * v + 4 * g + 1]);
      const float c = __uint_as_float(r[16 * v + 4 * g + 2]), d = __uint_as_float(r[16 * v + 4 * g + 3]);
      if (kDet)
        ptx::st_global_v4(p, a, b, c, d);
      else
        ptx::red_add_v4(p, a, b, c, d);
    }
}

template <bool kDet>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_d256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const D256Params prm) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_addr(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(prm.status, 0, (int32_t)FA_ERR_DEVICE);
    return;
  }
  // Work item: (head, key block, column half).  Heads go in groups of
  // kHeadGroup; inside a group key block 0 (the longest causal walk) comes
  // first, and the two halves of a key block are neighbours in the grid, so
  // they run at the same time and share their loads in L2.
  const int bh_total = prm.B * prm.H;
  const int per_group = kHeadGroup * prm.nk_tiles * 2;
  const int grp = blockIdx.x / per_group;
  const int gsize = min(kHeadGroup, bh_total - grp * kHeadGroup);
  const int rr = blockIdx.x - grp * per_group;
  const int kb = rr / (2 * gsize);
  const int bh = grp * kHeadGroup + (rr % (2 * gsize)) / 2;
  const int hf = rr & 1;  // this CTA's column half
  const int b = bh / prm.H, hh = bh % prm.H;

  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kMisc + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + Ly::kBar + 8 * i; };

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(KV_FULL), 1);
    ptx::mbar_init(bar(QO_FULL), 1);
    ptx::mbar_init(bar(QW_FULL), 1);
    ptx::mbar_init(bar(DOO_FULL), 1);
    ptx::mbar_init(bar(DOW_FULL), 1);
    ptx::mbar_init(bar(QO_EMPTY), 1);
    ptx::mbar_init(bar(QW_EMPTY), 1);
    ptx::mbar_init(bar(DOO_EMPTY), 1);
    ptx::mbar_init(bar(DOW_EMPTY), 1);
    ptx::mbar_init(bar(LD_FULL0), 32);
    ptx::mbar_init(bar(LD_FULL1), 32);
    ptx::mbar_init(bar(S_FULL0), 1);
    ptx::mbar_init(bar(S_FULL1), 1);
    ptx::mbar_init(bar(DV_DONE0), 1);
    ptx::mbar_init(bar(DV_DONE1), 1);
    ptx::mbar_init(bar(P_FULL), kComputeThreads);
    ptx::mbar_init(bar(DP_FULL), 1);
    ptx::mbar_init(bar(DS_FULL), kComputeThreads);
    ptx::mbar_init(bar(DS_EMPTY), 1);
    ptx::mbar_init(bar(DQ_FULL), 1);
    ptx::mbar_init(bar(DQ_EMPTY), kDrainThreads);
    ptx::mbar_init(bar(ACC_FULL), 1);
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

  const int k0 = kb * kKeyRows;
  // first 128-row query tile holding a query that sees key k0 (i >= k0 - offset)
  const int tile_first = !prm.causal ? 0 : (k0 > prm.offset ? (k0 - prm.offset) / kKeyRows : 0);
  const int blk_first = 2 * tile_first;               // in 64-row query blocks
  const int n_iter = 2 * (prm.n_tiles - tile_first);  // even: whole tiles
  const int64_t khead = (int64_t)b * prm.ksb + (int64_t)hh * prm.ksh;
  const ptx::Waiter W{abort_flag, prm.status, prm.wait_ns};
  const int own = 2 * hf, other = 2 * (1 - hf);  // first 64-column chunk of each half

  const uint32_t sK = sbase + Ly::kK, sV = sbase + Ly::kV, sQ = sbase + Ly::kQ, sdO = sbase + Ly::kdO;
  const uint32_t sdS = sbase + Ly::kdS;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int n_qo = 0, n_qw = 0, n_doo = 0, n_dow = 0;  // loads issued per barrier
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmQ);
      ptx::prefetch_tensormap(&tmK);
      ptx::prefetch_tensormap(&tmV);
      ptx::prefetch_tensormap(&tmdO);
      ptx::mbar_arrive_expect_tx(bar(KV_FULL), 8 * Ly::kKChunk);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        ptx::tma_load_4d(sK + c * Ly::kKChunk, &tmK, bar(KV_FULL), c * 64, k0, hh, b);
        ptx::tma_load_4d(sV + c * Ly::kKChunk, &tmV, bar(KV_FULL), c * 64, k0, hh, b);
      }
    }
    // L and D rows of the next block are read into registers one block
    // ahead, so their global-load latency hides behind the stage waits.
    float lv[2], dv[2];
    auto fetch_rows = [&](int it) {
      const int q0 = (blk_first + it) * kQRows;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = q0 + lane + 32 * u;
        lv[u] = q < prm.N ? __ldg(prm.L + (int64_t)bh * prm.N + q) * kLog2e : INFINITY;
        dv[u] = q < prm.N ? __ldg(prm.D + (int64_t)bh * prm.N + q) : 0.f;
      }
    };
    auto load_half = [&](const CUtensorMap* map, uint32_t tile, int c, uint32_t full, int q0) {
      ptx::mbar_arrive_expect_tx(full, 2 * Ly::kQChunk);
      ptx::tma_load_4d(tile + c * Ly::kQChunk, map, full, c * 64, q0, hh, b);
      ptx::tma_load_4d(tile + (c + 1) * Ly::kQChunk, map, full, (c + 1) * 64, q0, hh, b);
    };
    fetch_rows(0);
    for (int i = 0; i < n_iter; ++i) {
      const int q0 = (blk_first + i) * kQRows;
      const uint32_t pp = (i - 1) & 1;  // phase of the previous block's release
      // L, D rows into slot i & 1 (its last reader, dS(i-2), finished before
      // S(i-1) was issued, i.e. before QO_EMPTY(i-1))
      if (i >= 1 && !(ok = warp_wait(bar(QO_EMPTY), pp, W))) break;
      float* sL = reinterpret_cast<float*>(smem + Ly::kL) + (i & 1) * kQRows;
      float* sD = reinterpret_cast<float*>(smem + Ly::kD) + (i & 1) * kQRows;
      sL[lane] = lv[0];
      sL[lane + 32] = lv[1];
      sD[lane] = dv[0];
      sD[lane + 32] = dv[1];
      ptx::mbar_arrive(bar(LD_FULL0 + (i & 1)));
      if (lane == 0) load_half(&tmQ, sQ, other, bar(QO_FULL), q0);
      n_qo = i + 1;
      if (i >= 1 && !(ok = warp_wait(bar(DOO_EMPTY), pp, W))) break;
      if (lane == 0) load_half(&tmdO, sdO, other, bar(DOO_FULL), q0);
      n_doo = i + 1;
      if (i >= 1 && !(ok = warp_wait(bar(DOW_EMPTY), pp, W))) break;
      if (lane == 0) load_half(&tmdO, sdO, own, bar(DOW_FULL), q0);
      n_dow = i + 1;
      if (i >= 1 && !(ok = warp_wait(bar(QW_EMPTY), pp, W))) break;
      if (lane == 0) load_half(&tmQ, sQ, own, bar(QW_FULL), q0);
      n_qw = i + 1;
      __syncwarp();
      if (i + 1 < n_iter) fetch_rows(i + 1);
    }
    if (!ok) {  // let every copy this CTA started land before the CTA exits
      ptx::wait_bounded(bar(KV_FULL), 0, W, false);
      // one stage: only the last load on each barrier can still be in flight
      if (n_qo) ptx::wait_bounded(bar(QO_FULL), (n_qo - 1) & 1, W, false);
      if (n_qw) ptx::wait_bounded(bar(QW_FULL), (n_qw - 1) & 1, W, false);
      if (n_doo) ptx::wait_bounded(bar(DOO_FULL), (n_doo - 1) & 1, W, false);
      if (n_dow) ptx::wait_bounded(bar(DOW_FULL), (n_dow - 1) & 1, W, false);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t kIdS = ptx::idesc_bf16_f32(128, kQRows, false, false);  // S^T, dP^T
    constexpr uint32_t kIdKV = ptx::idesc_bf16_f32(128, kHalfD, false, true);  // dV, dK
    constexpr uint32_t kIdQ = ptx::idesc_bf16_f32(128, kHalfD, true, true);    // dQ
    // K-major operand, 16-element K step kk inside 64-column chunks
    auto kdesc = [&](uint32_t tile, uint32_t chunk, int kk) -> uint64_t {
      return ptx::sdesc_sw128(tile + (kk >> 2) * chunk + (kk & 3) * 32, 16, 1024);
    };
    // MN-major operand, 16-row K step kk; 64-column MN blocks `chunk` apart
    auto mndesc = [&](uint32_t tile, uint32_t chunk, int kk) -> uint64_t {
      return ptx::sdesc_sw128(tile + kk * 2048, chunk, 1024);
    };
    auto tS = [&](int i) -> uint32_t { return tm + ((i & 1) ? Ly::kColS1 : Ly::kColS0); };
    auto tdP = [&](int i) -> uint32_t { return tm + ((i & 1) ? Ly::kColdP1 : Ly::kColdP0); };
    const uint32_t tdQ = tm + Ly::kColdQ, tdV = tm + Ly::kColdV, tdK = tm + Ly::kColdK;
    // 16-column K steps of one 128-column half of S^T = K Q^T or dP^T = V dO^T
    auto issue_half = [&](uint32_t d, uint32_t a_tile, uint32_t b_tile, int c, bool first) {
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int kk = 4 * c + s;
        ptx::mma_ss(d, kdesc(a_tile, Ly::kKChunk, kk), kdesc(b_tile, Ly::kQChunk, kk), kIdS, !(first && s == 0));
      }
    };

    bool ok = warp_wait(bar(KV_FULL), 0, W) && warp_wait(bar(QO_FULL), 0, W);
    if (ok) {
      ptx::tc_fence_after();
      if (ptx::elect_one()) issue_half(tS(0), sK, sQ, other, true);
      __syncwarp();
      ok = warp_wait(bar(QW_FULL), 0, W);
    }
    if (ok) {
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        issue_half(tS(0), sK, sQ, own, false);
        ptx::tc_commit(bar(S_FULL0));
        ptx::tc_commit(bar(QO_EMPTY));
      }
      __syncwarp();
      ok = warp_wait(bar(DOO_FULL), 0, W);
    }
    if (ok) {
      ptx::tc_fence_after();
      if (ptx::elect_one()) issue_half(tdP(0), sV, sdO, other, true);
      __syncwarp();
      ok = warp_wait(bar(DOW_FULL), 0, W);
    }
    if (ok) {
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        issue_half(tdP(0), sV, sdO, own, false);
        ptx::tc_commit(bar(DP_FULL));
        ptx::tc_commit(bar(DOO_EMPTY));
      }
      __syncwarp();
    }
    for (int i = 0; ok && i < n_iter; ++i) {
      const uint32_t ph = i & 1;
      const uint32_t ph1 = (i + 1) & 1;
      const bool more = i + 1 < n_iter;
      // dV += P^T dO[:, own]  (A = P^T from TMEM: 16-query K steps 2g, 2g+1 in
      // columns [32g, 32g + 16) of the S buffer)
      if (!(ok = warp_wait(bar(P_FULL), ph, W))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kQRows / 16; ++kk)
          ptx::mma_ts(tdV, tS(i) + (kk >> 1) * 32 + (kk & 1) * 8, mndesc(sdO + own * Ly::kQChunk, Ly::kQChunk, kk),
                      kIdKV, (i | kk) != 0);
        ptx::tc_commit(bar(DV_DONE0 + (i & 1)));
        ptx::tc_commit(bar(DOW_EMPTY));
      }
      __syncwarp();
      // S^T(i+1), other half, once its Q chunks have landed and the S buffer's
      // last reader dV(i-1) is done
      if (more) {
        ok = i >= 1 ? warp_wait2(bar(QO_FULL), ph1, bar(DV_DONE0 + ((i + 1) & 1)), ((i - 1) >> 1) & 1, W)
                    : warp_wait(bar(QO_FULL), ph1, W);
        if (!ok) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) issue_half(tS(i + 1), sK, sQ, other, true);
        __syncwarp();
      }
      // dK += dS^T Q[:, own]; after an odd block, dQ of the tile:
      // dQ = [dS(i-1); dS(i)] K[:, own] (A: the two dS^T slots as the two
      // 64-query MN blocks)
      if (!(ok = warp_wait(bar(DS_FULL), ph, W))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        const uint32_t slot = sdS + (i & 1) * Ly::kdSSlot;
#pragma unroll
        for (int kk = 0; kk < kQRows / 16; ++kk)
          ptx::mma_ss(tdK, kdesc(slot, Ly::kdSSlot, kk), mndesc(sQ + own * Ly::kQChunk, Ly::kQChunk, kk), kIdKV,
                      (i | kk) != 0);
        ptx::tc_commit(bar(QW_EMPTY));
        if (i & 1) {
#pragma unroll
          for (int kk = 0; kk < kKeyRows / 16; ++kk)
            ptx::mma_ss(tdQ, mndesc(sdS, Ly::kdSSlot, kk), mndesc(sK + own * Ly::kKChunk, Ly::kKChunk, kk), kIdQ,
                        kk > 0);
          ptx::tc_commit(bar(DQ_FULL));
          ptx::tc_commit(bar(DS_EMPTY));
        }
      }
      __syncwarp();
      if (!more) break;
      // S^T(i+1), own half
      if (!(ok = warp_wait(bar(QW_FULL), ph1, W))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        issue_half(tS(i + 1), sK, sQ, own, false);
        ptx::tc_commit(bar(S_FULL0 + ((i + 1) & 1)));
        ptx::tc_commit(bar(QO_EMPTY));
      }
      __syncwarp();
      // dP^T(i+1); an even block's columns held the dQ tile just drained
      ok = (i & 1) ? warp_wait2(bar(DQ_EMPTY), (i >> 1) & 1, bar(DOO_FULL), ph1, W)
                   : warp_wait(bar(DOO_FULL), ph1, W);
      if (!ok) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) issue_half(tdP(i + 1), sV, sdO, other, true);
      __syncwarp();
      if (!(ok = warp_wait(bar(DOW_FULL), ph1, W))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        issue_half(tdP(i + 1), sV, sdO, own, false);
        ptx::tc_commit(bar(DP_FULL));
        ptx::tc_commit(bar(DOO_EMPTY));
      }
      __syncwarp();
    }
    if (ptx::elect_one()) ptx::tc_commit(bar(ACC_FULL));
    __syncwarp();
    if (!ok) ptx::wait_bounded(bar(ACC_FULL), 0, W, false);  // nothing in flight at exit
  } else if (warp >= kDrainWarp0) {
    // ------------------------------------------------------------ dQ drain
    // One warp per TMEM lane quarter (32 query rows of the tile): this CTA's
    // 128 columns are eight 16-column units, contiguous in the accumulator.
    const int qq = warp & 3;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const uint32_t src = tm + Ly::kColdQ + lane_off;
    for (int t = 0; t < n_iter / 2; ++t) {
      if (!warp_wait(bar(DQ_FULL), t & 1, W)) break;
      ptx::tc_fence_after();
      float* dst = prm.dq_accum + (kDet ? kb * prm.slice_elems : 0) +
                   dq_unit_offset(bh, prm.n_tiles, tile_first + t, qq, hf * (kHalfD / 16), kHD);
      uint32_t r[64];
      ptx::tmem_ld64(src, src + 32, r);
      drain32<kDet>(dst, lane, *reinterpret_cast<const uint32_t(*)[32]>(&r[0]));
      drain32<kDet>(dst + 2 * kDqUnitFloats, lane, *reinterpret_cast<const uint32_t(*)[32]>(&r[32]));
      ptx::tmem_ld64(src + 64, src + 96, r);
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(DQ_EMPTY));  // the columns are free for dP
      drain32<kDet>(dst + 4 * kDqUnitFloats, lane, *reinterpret_cast<const uint32_t(*)[32]>(&r[0]));
      drain32<kDet>(dst + 6 * kDqUnitFloats, lane, *reinterpret_cast<const uint32_t(*)[32]>(&r[32]));
    }
  } else {
    // ------------------------------------------------------------ compute
    const int qq = warp & 3;               // TMEM lane quarter
    const int G = warp >> 2;               // query column half of the block
    const int t = qq * 32 + lane;          // TMEM lane = key row
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const int kr = k0 + t;
    const bool key_ok = kr < prm.Nk;
    const int kd = k0 - prm.offset;        // key k0 + t visible to query q iff q - kd >= t
    const float sl2 = prm.scale * kLog2e;
    const int c0 = G * 32;                 // query columns [c0, c0 + 32)
    uint32_t pk[16];                       // P for those columns, bf16 pairs

    bool ok = true;
    for (int i = 0; i < n_iter; ++i) {
      const uint32_t ph = i & 1;
      const int q0 = (blk_first + i) * kQRows;
      // ---- P(i)
      if (!(ok = warp_wait2(bar(S_FULL0 + (i & 1)), (i >> 1) & 1, bar(LD_FULL0 + (i & 1)), (i >> 1) & 1, W)))
        break;
      const uint32_t tSi = tm + ((i & 1) ? Ly::kColS1 : Ly::kColS0);
      ptx::tc_fence_after();
      {
        uint32_t r[32];
        ptx::tmem_ld32(tSi + lane_off + c0, r);
        const uint32_t sLa = sbase + Ly::kL + (i & 1) * kQRows * 4 + c0 * 4;
        // key k0 + t is visible to query q0 + col iff col >= t - rel; the
        // block needs the mask unless every entry passes (rel >= 127)
        const int rel = q0 - kd;
        const bool diag = prm.causal && rel < kKeyRows - 1;
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
      // ---- dS(i) into slot i & 1, once dK and dQ of the previous tile have
      // read both slots (checked at the first block of each tile)
      ok = ((i & 1) == 0 && i >= 2) ? warp_wait2(bar(DP_FULL), ph, bar(DS_EMPTY), ((i >> 1) - 1) & 1, W)
                                    : warp_wait(bar(DP_FULL), ph, W);
      if (!ok) break;
      ptx::tc_fence_after();
      {
        uint32_t r[32];
        ptx::tmem_ld32(tm + ((i & 1) ? Ly::kColdP1 : Ly::kColdP0) + lane_off + c0, r);
        const uint32_t sDa = sbase + Ly::kD + (i & 1) * kQRows * 4 + c0 * 4;
        uint32_t ds[16];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          // dS = P * (dP - D): the difference in fp32, then one bf16x2
          // product with the packed bf16 P
          const float4 d4 = ptx::ld_shared_f4(sDa + j * 4);
          const uint32_t g01 = ptx::pack_bf16x2(__uint_as_float(r[j + 0]) - d4.x, __uint_as_float(r[j + 1]) - d4.y);
          const uint32_t g23 = ptx::pack_bf16x2(__uint_as_float(r[j + 2]) - d4.z, __uint_as_float(r[j + 3]) - d4.w);
          ds[j / 2] = ptx::mul_bf16x2(pk[j / 2], g01);
          ds[j / 2 + 1] = ptx::mul_bf16x2(pk[j / 2 + 1], g23);
        }
        // row t of dS^T (64 queries = 128 bytes), 16-byte pieces 4G .. 4G+3,
        // 128-byte swizzle (piece XOR row % 8)
        const uint32_t row = sdS + (i & 1) * Ly::kdSSlot + t * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t piece = (uint32_t)(G * 4 + u);
          ptx::st_shared_v4(row + ((piece ^ (uint32_t)(t & 7)) << 4), ds[4 * u], ds[4 * u + 1], ds[4 * u + 2],
                            ds[4 * u + 3]);
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(DS_FULL));
    }
    if (ok && warp_wait(bar(ACC_FULL), 0, W)) {
      ptx::tc_fence_after();
      const int64_t off = khead + (int64_t)kr * prm.ksn + hf * kHalfD;
      if (G == 0)
        store_row128(tm + Ly::kColdV + lane_off, key_ok, prm.dV + off, 1.0f);
      else
        store_row128(tm + Ly::kColdK + lane_off, key_ok, prm.dK + off, prm.scale);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tm, Ly::kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [B, H, rows, 256] bf16 (Q-shaped: kv = false, K-shaped: kv = true) as a
// 4-D TMA map with boxes of 64 columns x box_rows rows, 128-byte swizzle;
// rows past the end read as zeros.
bool make_map(CUtensorMap* m, const void* base, const fa_problem& p, bool kv, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const int64_t rows = kv ? p.N_k : p.N;
  const int64_t sn = kv ? p.kstride_n : p.stride_n, sh = kv ? p.kstride_h : p.stride_h;
  const int64_t sb = kv ? p.kstride_b : p.stride_b;
  cuuint64_t dims[4] = {(cuuint64_t)p.d, (cuuint64_t)rows, (cuuint64_t)p.H, (cuuint64_t)p.B};
  cuuint64_t strides[3] = {(cuuint64_t)sn * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool kDet>
cudaError_t launch_t(const CUtensorMap* maps, const D256Params& prm, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(bwd_d256_kernel<kDet>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = (int64_t)prm.nk_tiles * prm.B * prm.H * 2;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  bwd_d256_kernel<kDet><<<(unsigned)grid, kThreads, Ly::kBytes, s>>>(maps[0], maps[1], maps[2], maps[3], prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_d256_sm103(const fa_problem& p, const void* Q, const void* K, const void* V, const void* dO,
                                  const float* L, const float* D, float* dq_accum, void* dK, void* dV,
                                  int32_t* status, uint64_t wait_ns, cudaStream_t s) {
  if (p.d != kHD || p.dtype != FA_BF16) return cudaErrorInvalidValue;
  CUtensorMap maps[4];
  if (!make_map(&maps[0], Q, p, false, kQRows) || !make_map(&maps[1], K, p, true, kKeyRows) ||
      !make_map(&maps[2], V, p, true, kKeyRows) || !make_map(&maps[3], dO, p, false, kQRows))
    return cudaErrorInvalidValue;
  D256Params prm;
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
  prm.n_tiles = (int)ceil_div(p.N, kKeyRows);
  prm.nk_tiles = (int)ceil_div(p.N_k, kKeyRows);
  prm.offset = (int)causal_offset(p);
  prm.ksb = p.kstride_b;
  prm.ksh = p.kstride_h;
  prm.ksn = p.kstride_n;
  prm.scale = p.scale;
  prm.causal = p.causal;
  prm.slice_elems = deterministic(p) ? dq_slice_elems(p) : 0;
  return prm.slice_elems > 0 ? launch_t<true>(maps, prm, s) : launch_t<false>(maps, prm, s);
}

}  // namespace fa
