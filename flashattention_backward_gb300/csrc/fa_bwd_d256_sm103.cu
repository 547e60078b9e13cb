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
// dQ is produced transposed per query block, dQ^T = K_j[:, half]^T dS^T
// (M = the 128 columns of the half, N = 64 queries), into the tensor-memory
// columns of the block's dP^T once dS has been formed from it.  The drain
// warps turn each 4 x 4 piece (4 columns of 4 query rows) around with two
// rounds of lane shuffles inside groups of four lanes, so that every lane
// holds 4 consecutive columns of one query row, and add them into the
// accumulator with vector reductions.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,64) [64,128)    S^T of even / odd query blocks; P^T (bf16) over it
//   [128,192) [192,256) dP^T of even / odd blocks; then dQ^T of that block
//   [256,384)          dV accumulator (this CTA's 128 columns)
//   [384,512)          dK accumulator
//
// Shared memory: K_j, V_j (4 chunks of 128 rows x 64 columns each); Q in
// three regions of two 64 x 64 chunks (a half of the columns of one block
// each); dO_i (4 chunks of 64 x 64, one stage); dS^T (128 keys x 64
// queries); L and D rows of two blocks; barriers.  Block i keeps the other
// CTA's half of Q (read only by S^T) in region i % 3 and its own half (read
// again by dK += dS^T Q) in region (i + 2) % 3, so both halves of Q(i+1) go
// into regions freed by S^T(i) and by dK(i-1), and S^T(i+1) can be issued
// before dS(i) is ready.  dO's halves are freed by dP^T(i) and dV(i), both
// early in the block.
//
// Warp roles (448 threads):
//   warps 0-7   compute: TMEM lane quarter w % 4, query columns
//               [32 (w / 4), +32).  P = exp2(S scale log2e - L log2e) -> bf16
//               into TMEM; dS = P (dP - D) -> bf16 into shared memory.
//               Epilogue: dV (w < 4), scale * dK (w >= 4).
//   warps 8-11  dQ drain, one per lane quarter (32 of the half's columns).
//   warp 12     TMA producer (K, V once; Q, dO per block; L, D rows).
//   warp 13     TMEM allocator and MMA issuer (one elected lane issues).
//
// MMA issue order per query block i:
//   dV(i)  S(i+1)  dK(i)  dQ^T(i)  dP(i+1)
//
// Every wait is bounded; when one runs out the CTA records FA_ERR_TIMEOUT,
// waits for its own TMA loads and MMAs, frees tensor memory and exits.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

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
  Q_FULL,       // Q(i) landed (both halves)
  DOO_FULL,     // dO(i): the other half's chunks landed
  DOW_FULL,     // dO(i): this CTA's own chunks landed
  DOO_EMPTY,    // dP(i) done: dO other-half chunks free
  DOW_EMPTY,    // dV(i) done: dO own chunks free
  QREG_FREE0,   // Q region r released (by S(i) for i % 3 == r, by dK(i)
  QREG_FREE1,   //   for (i + 2) % 3 == r)
  QREG_FREE2,
  LD_FULL0,     // L, D rows of an even / odd block written (32 producer lanes)
  LD_FULL1,
  S_FULL0,      // S^T of an even / odd block in TMEM
  S_FULL1,
  DV_DONE0,     // dV of an even / odd block done: its S/P columns reusable
  DV_DONE1,
  P_FULL,       // P^T(i) in TMEM (every compute thread)
  DP_FULL,      // dP^T(i) in TMEM
  DS_FULL,      // dS^T(i) in shared memory (every compute thread)
  DS_EMPTY,     // dK(i) and dQ^T(i) done: the dS^T buffer is reusable
  DQ_FULL,      // dQ^T(i) in TMEM
  DQ_EMPTY,     // dQ^T(i) drained from TMEM (every drain thread)
  ACC_FULL,     // every MMA done: dK, dV final
  kNumBars
};

struct Ly {
  static constexpr int kKChunk = kKeyRows * 128;  // 128 rows x 128 bytes
  static constexpr int kQChunk = kQRows * 128;    // 64 rows x 128 bytes
  static constexpr int kQRegion = 2 * kQChunk;    // half of a Q block's columns
  static constexpr int kK = 0;
  static constexpr int kV = kK + 4 * kKChunk;
  static constexpr int kQ = kV + 4 * kKChunk;           // 3 regions
  static constexpr int kdO = kQ + 3 * kQRegion;
  static constexpr int kdS = kdO + 4 * kQChunk;         // 128 keys x 64 queries bf16
  static constexpr int kdSBytes = kKeyRows * 128;
  static constexpr int kL = kdS + kdSBytes;             // 2 slots x 64 fp32 (L log2 e)
  static constexpr int kD = kL + 2 * kQRows * 4;        // 2 slots x 64 fp32
  static constexpr int kBar = kD + 2 * kQRows * 4;
  static constexpr int kMisc = kBar + kNumBars * 8;     // TMEM base address, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr uint32_t kColS0 = 0, kColS1 = 64, kColdP0 = 128, kColdP1 = 192;
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
  // non-null: [0] += (key block, 64-row query block) pairs executed, [1] +=
  // executed pairs with no visible entry; counted by the column-half-0 CTA
  unsigned long long* pair_count;
};

using ptx::warp_wait;
using ptx::warp_wait2;

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

// Transpose of a 4 x 4 piece held by four lanes (lane b of the group holds
// x[k] = piece[k][b]): afterwards lane b holds x[j] = piece[b][j].  Two
// rounds of exchanges with the partner lane b ^ 2, then b ^ 1, each moving
// the two entries that belong to the partner's half.
__device__ __forceinline__ void quad_transpose(float (&x)[4], int b) {
  const bool hi2 = (b & 2) != 0;
  float a0 = hi2 ? x[0] : x[2], a1 = hi2 ? x[1] : x[3];
  a0 = __shfl_xor_sync(0xffffffffu, a0, 2);
  a1 = __shfl_xor_sync(0xffffffffu, a1, 2);
  if (hi2) {
    x[0] = a0;
    x[1] = a1;
  } else {
    x[2] = a0;
    x[3] = a1;
  }
  const bool hi1 = (b & 1) != 0;
  a0 = hi1 ? x[0] : x[1];
  a1 = hi1 ? x[2] : x[3];
  a0 = __shfl_xor_sync(0xffffffffu, a0, 1);
  a1 = __shfl_xor_sync(0xffffffffu, a1, 1);
  if (hi1) {
    x[0] = a0;
    x[2] = a1;
  } else {
    x[1] = a0;
    x[3] = a1;
  }
}

// kCount: tile-pair accounting into prm.pair_count (instantiated apart, so
// that the kernel fa_bwd runs carries no counting code).
template <bool kDet, bool kCount>
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
    ptx::mbar_init(bar(Q_FULL), 1);
    ptx::mbar_init(bar(DOO_FULL), 1);
    ptx::mbar_init(bar(DOW_FULL), 1);
    ptx::mbar_init(bar(DOO_EMPTY), 1);
    ptx::mbar_init(bar(DOW_EMPTY), 1);
    ptx::mbar_init(bar(QREG_FREE0), 1);
    ptx::mbar_init(bar(QREG_FREE1), 1);
    ptx::mbar_init(bar(QREG_FREE2), 1);
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
  // first 64-row query block holding a query that sees key k0
  // (i >= k0 - offset; every key block has one, the last query sees every key)
  const int blk_first = !prm.causal ? 0 : (k0 > prm.offset ? (k0 - prm.offset) / kQRows : 0);
  const int n_iter = (prm.N + kQRows - 1) / kQRows - blk_first;
  const int64_t khead = (int64_t)b * prm.ksb + (int64_t)hh * prm.ksh;
  const ptx::Waiter W{abort_flag, prm.status, prm.wait_ns};
  const int own = 2 * hf, other = 2 * (1 - hf);  // first 64-column chunk of each half

  const uint32_t sK = sbase + Ly::kK, sV = sbase + Ly::kV, sQ = sbase + Ly::kQ, sdO = sbase + Ly::kdO;
  const uint32_t sdS = sbase + Ly::kdS;
  // Q regions of block i: the other half in i % 3, this CTA's half in (i + 2) % 3
  auto q_other = [&](int i) -> int { return i % 3; };
  auto q_own = [&](int i) -> int { return (i + 2) % 3; };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int n_q = 0, n_doo = 0, n_dow = 0;  // loads issued per barrier
    int reg_loads0 = 0, reg_loads1 = 0, reg_loads2 = 0;  // loads into each Q region so far
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
    // two 64 x 64 chunks (columns c, c + 1) of a 64-row block
    auto load2 = [&](const CUtensorMap* map, uint32_t dst, int c, uint32_t full, int q0) {
      ptx::tma_load_4d(dst, map, full, c * 64, q0, hh, b);
      ptx::tma_load_4d(dst + Ly::kQChunk, map, full, (c + 1) * 64, q0, hh, b);
    };
    // a Q region may be refilled once its previous contents' reader is done
    auto region_free = [&](int r) -> bool {
      int n;
      if (r == 0)
        n = reg_loads0++;
      else if (r == 1)
        n = reg_loads1++;
      else
        n = reg_loads2++;
      return n == 0 || warp_wait(bar(QREG_FREE0 + r), (n - 1) & 1, W);
    };
    fetch_rows(0);
    for (int i = 0; i < n_iter; ++i) {
      const int q0 = (blk_first + i) * kQRows;
      const uint32_t pp = (i - 1) & 1;  // phase of the previous block's release
      // Q(i): both regions free (their last readers were dK(i-2) and S(i-1),
      // which also means dS(i-2) is done with L, D slot i & 1)
      if (!(ok = region_free(q_other(i)) && region_free(q_own(i)))) break;
      float* sL = reinterpret_cast<float*>(smem + Ly::kL) + (i & 1) * kQRows;
      float* sD = reinterpret_cast<float*>(smem + Ly::kD) + (i & 1) * kQRows;
      sL[lane] = lv[0];
      sL[lane + 32] = lv[1];
      sD[lane] = dv[0];
      sD[lane + 32] = dv[1];
      ptx::mbar_arrive(bar(LD_FULL0 + (i & 1)));
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(Q_FULL), 4 * Ly::kQChunk);
        load2(&tmQ, sQ + q_other(i) * Ly::kQRegion, other, bar(Q_FULL), q0);
        load2(&tmQ, sQ + q_own(i) * Ly::kQRegion, own, bar(Q_FULL), q0);
      }
      n_q = i + 1;
      if (i >= 1 && !(ok = warp_wait(bar(DOO_EMPTY), pp, W))) break;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(DOO_FULL), 2 * Ly::kQChunk);
        load2(&tmdO, sdO + other * Ly::kQChunk, other, bar(DOO_FULL), q0);
      }
      n_doo = i + 1;
      if (i >= 1 && !(ok = warp_wait(bar(DOW_EMPTY), pp, W))) break;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(DOW_FULL), 2 * Ly::kQChunk);
        load2(&tmdO, sdO + own * Ly::kQChunk, own, bar(DOW_FULL), q0);
      }
      n_dow = i + 1;
      __syncwarp();
      if (i + 1 < n_iter) fetch_rows(i + 1);
    }
    if (!ok) {  // let every copy this CTA started land before the CTA exits
      ptx::wait_bounded(bar(KV_FULL), 0, W, false);
      // each barrier's earlier loads were consumed before the next was issued
      if (n_q) ptx::wait_bounded(bar(Q_FULL), (n_q - 1) & 1, W, false);
      if (n_doo) ptx::wait_bounded(bar(DOO_FULL), (n_doo - 1) & 1, W, false);
      if (n_dow) ptx::wait_bounded(bar(DOW_FULL), (n_dow - 1) & 1, W, false);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t kIdS = ptx::idesc_bf16_f32(128, kQRows, false, false);  // S^T, dP^T
    constexpr uint32_t kIdKV = ptx::idesc_bf16_f32(128, kHalfD, false, true);  // dV, dK
    constexpr uint32_t kIdQ = ptx::idesc_bf16_f32(128, kQRows, true, true);    // dQ^T
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
    const uint32_t tdV = tm + Ly::kColdV, tdK = tm + Ly::kColdK;
    // S^T(i) = K Q(i)^T, 16 K steps over the 256 columns; the Q chunk of
    // column block c sits in the region of its half
    auto issue_S = [&](int i) {
      const uint32_t qo = sQ + q_other(i) * Ly::kQRegion, qw = sQ + q_own(i) * Ly::kQRegion;
#pragma unroll
      for (int kk = 0; kk < kHD / 16; ++kk) {
        const int c = kk >> 2;
        const uint32_t qb = (c >> 1) == hf ? qw : qo;
        ptx::mma_ss(tS(i), kdesc(sK, Ly::kKChunk, kk), kdesc(qb + (c & 1) * Ly::kQChunk, 0, kk & 3), kIdS, kk > 0);
      }
      ptx::tc_commit(bar(S_FULL0 + (i & 1)));
      ptx::tc_commit(bar(QREG_FREE0 + q_other(i)));
    };
    // dP^T(i) = V dO(i)^T, in two halves (each as soon as its chunks landed)
    auto issue_dP_half = [&](int i, int c, bool first) {
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int kk = 4 * c + s;
        ptx::mma_ss(tdP(i), kdesc(sV, Ly::kKChunk, kk), kdesc(sdO, Ly::kQChunk, kk), kIdS, !(first && s == 0));
      }
    };

    bool ok = warp_wait(bar(KV_FULL), 0, W) && warp_wait(bar(Q_FULL), 0, W);
    if (ok) {
      ptx::tc_fence_after();
      if (ptx::elect_one()) issue_S(0);
      __syncwarp();
      ok = warp_wait(bar(DOO_FULL), 0, W);
    }
    if (ok) {
      ptx::tc_fence_after();
      if (ptx::elect_one()) issue_dP_half(0, other, true);
      __syncwarp();
      ok = warp_wait(bar(DOW_FULL), 0, W);
    }
    if (ok) {
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        issue_dP_half(0, own, false);
        ptx::tc_commit(bar(DP_FULL));
        ptx::tc_commit(bar(DOO_EMPTY));
      }
      __syncwarp();
    }
    unsigned n_exec = 0, n_masked = 0;  // tile-pair accounting (pair_count)
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
      // S^T(i+1) once Q(i+1) has landed and the S buffer's last reader dV(i-1)
      // is done, so that it is ready when the compute warps finish dS(i)
      if (more) {
        ok = i >= 1 ? warp_wait2(bar(Q_FULL), ph1, bar(DV_DONE0 + ((i + 1) & 1)), ((i - 1) >> 1) & 1, W)
                    : warp_wait(bar(Q_FULL), ph1, W);
        if (!ok) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) issue_S(i + 1);
        __syncwarp();
      }
      // dK += dS^T Q[:, own]; then dQ^T = K[:, own]^T dS^T into the columns
      // of dP^T(i) (read by the compute warps before DS_FULL), once the drain
      // has emptied the other dP^T buffer for dP(i+1)
      if (!(ok = warp_wait(bar(DS_FULL), ph, W))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        const uint32_t qw = sQ + q_own(i) * Ly::kQRegion;
#pragma unroll
        for (int kk = 0; kk < kQRows / 16; ++kk)
          ptx::mma_ss(tdK, kdesc(sdS, 0, kk), mndesc(qw, Ly::kQChunk, kk), kIdKV, (i | kk) != 0);
        ptx::tc_commit(bar(QREG_FREE0 + q_own(i)));
      }
      __syncwarp();
      if (i >= 1 && !(ok = warp_wait(bar(DQ_EMPTY), (i - 1) & 1, W))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kKeyRows / 16; ++kk)
          ptx::mma_ss(tdP(i), mndesc(sK + own * Ly::kKChunk, Ly::kKChunk, kk), mndesc(sdS, Ly::kdSBytes, kk), kIdQ,
                      kk > 0);
        ptx::tc_commit(bar(DQ_FULL));
        ptx::tc_commit(bar(DS_EMPTY));
      }
      __syncwarp();
      if constexpr (kCount) {
        const int last_q = min((blk_first + i) * kQRows + kQRows - 1, prm.N - 1);
        ++n_exec;
        n_masked += !prm.causal || k0 <= last_q + prm.offset ? 0u : 1u;
      }
      if (!more) break;
      // dP^T(i+1), each half of the columns as soon as its dO chunks landed
      if (!(ok = warp_wait(bar(DOO_FULL), ph1, W))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) issue_dP_half(i + 1, other, true);
      __syncwarp();
      if (!(ok = warp_wait(bar(DOW_FULL), ph1, W))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        issue_dP_half(i + 1, own, false);
        ptx::tc_commit(bar(DP_FULL));
        ptx::tc_commit(bar(DOO_EMPTY));
      }
      __syncwarp();
    }
    const bool lead = ptx::elect_one();
    if (lead) ptx::tc_commit(bar(ACC_FULL));
    if (kCount && lead && hf == 0) {
      atomicAdd(prm.pair_count, (unsigned long long)n_exec);
      atomicAdd(prm.pair_count + 1, (unsigned long long)n_masked);
    }
    __syncwarp();
    if (!ok) ptx::wait_bounded(bar(ACC_FULL), 0, W, false);  // nothing in flight at exit
  } else if (warp >= kDrainWarp0) {
    // ------------------------------------------------------------ dQ drain
    // Warp qq holds TMEM lanes 32 qq .. +31, i.e. columns hf*128 + 32 qq + lane
    // of dQ, for the 64 query rows of the block (TMEM columns).  Lane 4a + b
    // transposes with its group so that it holds columns 4a .. 4a + 3 of
    // query rows 4m + b, one 16-byte piece of the accumulator layout each.
    const int qq = warp & 3;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const int ga = lane >> 2, gb = lane & 3;
    const int cb = hf * (kHalfD / 16) + 2 * qq + (ga >> 2);  // 16-column block
    const int cg = ga & 3;                                    // 4-column group in it
    for (int i = 0; i < n_iter; ++i) {
      if (!warp_wait(bar(DQ_FULL), i & 1, W)) break;
      ptx::tc_fence_after();
      uint32_t r[64];
      ptx::tmem_ld64(tm + ((i & 1) ? Ly::kColdP1 : Ly::kColdP0) + lane_off,
                     tm + ((i & 1) ? Ly::kColdP1 : Ly::kColdP0) + lane_off + 32, r);
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(DQ_EMPTY));  // the columns are free for dP(i+2)
      const int blk = blk_first + i;    // 64-row block: tile blk / 2, rows 64 (blk % 2) + ...
      float* base = prm.dq_accum + (kDet ? kb * prm.slice_elems : 0) +
                    dq_unit_offset(bh, prm.n_tiles, blk >> 1, 0, cb, kHD) + cg * 128;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        float x[4] = {__uint_as_float(r[4 * m]), __uint_as_float(r[4 * m + 1]), __uint_as_float(r[4 * m + 2]),
                      __uint_as_float(r[4 * m + 3])};
        quad_transpose(x, gb);
        const int row = (blk & 1) * kQRows + 4 * m + gb;  // query row inside the 128-row tile
        float* p = base + (int64_t)(row >> 5) * (kHD / 16) * kDqUnitFloats + (row & 31) * 4;
        if (kDet)
          ptx::st_global_v4(p, x[0], x[1], x[2], x[3]);
        else
          ptx::red_add_v4(p, x[0], x[1], x[2], x[3]);
      }
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
      // ---- dS(i), once dK(i-1) and dQ^T(i-1) have read the buffer
      ok = i >= 1 ? warp_wait2(bar(DP_FULL), ph, bar(DS_EMPTY), ph ^ 1, W) : warp_wait(bar(DP_FULL), ph, W);
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
        const uint32_t row = sdS + t * 128;
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

template <bool kDet, bool kCount>
cudaError_t launch_t(const CUtensorMap* maps, const D256Params& prm, cudaStream_t s) {
  cudaError_t e =
      cudaFuncSetAttribute(bwd_d256_kernel<kDet, kCount>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = (int64_t)prm.nk_tiles * prm.B * prm.H * 2;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  bwd_d256_kernel<kDet, kCount><<<(unsigned)grid, kThreads, Ly::kBytes, s>>>(maps[0], maps[1], maps[2], maps[3],
                                                                             prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_d256_sm103(const fa_problem& p, const void* Q, const void* K, const void* V, const void* dO,
                                  const float* L, const float* D, float* dq_accum, void* dK, void* dV,
                                  int32_t* status, uint64_t wait_ns, cudaStream_t s,
                                  unsigned long long* pair_count) {
  if (p.d != kHD || p.dtype != FA_BF16) return cudaErrorInvalidValue;
  CUtensorMap maps[4];
  if (!make_bf16_tile_map_rows(&maps[0], Q, p, false, kQRows) ||
      !make_bf16_tile_map_rows(&maps[1], K, p, true, kKeyRows) ||
      !make_bf16_tile_map_rows(&maps[2], V, p, true, kKeyRows) ||
      !make_bf16_tile_map_rows(&maps[3], dO, p, false, kQRows))
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
  prm.pair_count = pair_count;
  if (pair_count) return prm.slice_elems > 0 ? launch_t<true, true>(maps, prm, s) : launch_t<false, true>(maps, prm, s);
  return prm.slice_elems > 0 ? launch_t<true, false>(maps, prm, s) : launch_t<false, false>(maps, prm, s);
}

}  // namespace fa
