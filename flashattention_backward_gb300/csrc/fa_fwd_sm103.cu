// Forward pass (companion of the backward) for bf16, head dim 32, 64, 96, 128 or
// 256, on the sm_100-family tensor cores.  Online softmax over key blocks of
// 128 keys (64 at d = 256)
// (1point3acres FlashAttention write-up, online-softmax paragraphs; "CUDA
// 算子工程" ch.16 §16.4 for L = m + log l):
//   m' = max(m, rowmax(S_b)),  alpha = exp(m - m'),  l' = alpha l + sum(p_b),
//   O' = alpha O + p_b V_b,    O = O' / l,  L = m + log l.
//
// One CTA owns a 128-row query block (resident in shared memory) and walks
// the key blocks it can see (all, or up to the diagonal under the causal
// mask).  S_b = Q K_b^T goes to one of three TMEM buffers; P_b (bf16) is
// written over S_b and feeds O += P_b V_b straight from TMEM; O accumulates
// in TMEM.  With three buffers S_b can be computed while the softmax warps
// still work on P_{b-1} and P_{b-2}; S_b and O += P_b V_b are issued by two
// warps, each waiting only for its own inputs.
// K lives in three shared-memory stages (two at d = 256), each freed as soon
// as its S block is done; V in three at d = 96, 128 (two otherwise), each
// freed when its O += P V is done.
// At d = 256 the 64-key blocks keep a 64 KB Q tile and two stages each of K
// and V (32 KB a tile) inside shared memory, and O takes tensor-memory
// columns 256-511 beside three 64-column S buffers.
//
// The exponent base m is only moved when a row maximum grows by more than
// 2^8 (in exp2 units): otherwise P = exp2(S - m) <= 256 stays well inside
// fp32 and bf16, and O, l keep the old base, so O in TMEM is rescaled only
// on those rare steps.  The final O / l and L = m + log l are exact for any
// base.
//
// Warp roles (640 threads; 352 at d = 256):
//   warps 0-15 softmax (0-7 at d = 256).  Warp w owns query rows
//              32*(w%4) .. +31 (its TMEM lane quarter) and 32 key columns of
//              each block (column group w/4).  The warps of a lane quarter
//              exchange row maxima through a dead column of their S slices in
//              tensor memory, and the final row sums through shared memory.
//              Epilogue (the first two warps of each lane quarter): O columns
//              [d/2 * (w/4), +d/2) and L.
//   then       TMA producer of Q (once) and K; TMEM allocator and issuer of
//              the S products; TMA producer of V; issuer of O += P V (one
//              elected lane in each MMA warp; at d = 256 the allocator's warp
//              issues both).
//
// Every wait is bounded (same mechanism as the backward kernel).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {


namespace {

constexpr int kBlk = 128;
constexpr int kKStages = 3;  // K tiles in shared memory
constexpr int kVStages = 3;  // V tiles in shared memory (at most; two at d <= 64 and d = 256)
constexpr int kSBufs = 3;    // S/P buffers in TMEM
constexpr int kHeadGroup = 4;  // heads whose query blocks interleave in the grid order
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum BarId {
  Q_FULL = 0,
  K_FULL0,                         // K stage landed (kKStages)
  K_EMPTY0 = K_FULL0 + kKStages,   // K stage read by its S block
  V_FULL0 = K_EMPTY0 + kKStages,   // V stage landed (kVStages)
  V_EMPTY0 = V_FULL0 + kVStages,   // V stage read by its O += P V
  S_READY0 = V_EMPTY0 + kVStages,  // S_b may be issued: K_b forwarded by its producer and
                                   // buffer b % 3 read by O += P_{b-3} V_{b-3} (2 arrivals)
  S_FULL0 = S_READY0 + kSBufs,     // S_b in TMEM buffer b % 3
  P_FULL0 = S_FULL0 + kSBufs,      // P_b in buffer b % 3 and V_b forwarded (softmax threads + 1)
  O_DONE0 = P_FULL0 + kSBufs,      // O += P_b V_b (and every MMA before it) done, on
                                   // barrier b % 3.  The softmax warps ask about block b-1
                                   // only after S_b, which is issued only once O += P_{b-3}
                                   // V_{b-3} (and every earlier product of that chain) is
                                   // done, so the parity always names the current phase
  DRAIN = O_DONE0 + kSBufs,        // every MMA of both MMA warps done (waited only when a
                                   // CTA gives up)
  kNumBars
};

// Tiles LD = 64, 128 or 256 columns wide: head dims 32 and 64 use LD = 64, 96
// and 128 use LD = 128, 256 uses LD = 256; the TMA zero-fills the columns
// past d.  Key blocks are BK rows: 128, or 64 at LD = 256.
template <int LD>
struct FwdLayout {
  // softmax warps: four per TMEM lane quarter, each on 32 key columns of a
  // block (two at d = 256, whose blocks have 64 keys)
  static constexpr int kGroups = LD == 256 ? 2 : 4;     // softmax warps per lane quarter
  static constexpr int kSmWarps = 4 * kGroups;
  static constexpr int kSmThreads = 32 * kSmWarps;
  // MMA issue split over two warps (S products; O += P V products) at
  // d <= 128; at d = 256 the split measured 13 % slower and one warp issues both
  static constexpr bool kSplitMma = LD != 256;
  static constexpr int kProdK = kSmWarps;               // TMA producer of Q and K
  static constexpr int kMma = kSmWarps + 1;             // TMEM allocator; issues the S products
  static constexpr int kProdV = kSmWarps + 2;           // TMA producer of V
  static constexpr int kMmaPV = kSplitMma ? kSmWarps + 3 : kMma;  // issues the O += P V products
  static constexpr int kThreads = 32 * (kSmWarps + (kSplitMma ? 4 : 3));
  static constexpr int BK = LD == 256 ? 64 : 128;       // keys per block
  // Three stages each of K and V at d = 96, 128: with two V stages V_b waited
  // for O += P_{b-2} V_{b-2}, and with two K stages K_b for S_{b-2}, so a TMA
  // load sat in the per-block chain (measured: 1×32×8192×128 causal 1314-1320
  // TFLOPS against 1158-1162 with two V stages, 930 with two K stages).  At
  // d <= 64 a third V stage would leave room for one CTA per SM instead of
  // two (measured slower).  d = 256 has room for five 64-key tiles: three K
  // and two V measured 1131 TFLOPS on 1×16×8192×256 causal, against 1056 with
  // two of each and 1020 with two K and three V.
  static constexpr int kKSt = kKStages;                 // K stages
  static constexpr int kVSt = LD == 128 ? kVStages : 2;  // V stages
  static constexpr int kQChunk = kBlk * 128;            // 128 rows x 64 columns
  static constexpr int kKVChunk = BK * 128;             // BK rows x 64 columns
  static constexpr int kQTile = kBlk * LD * 2;
  static constexpr int kKVTile = BK * LD * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQTile;                // kKSt tiles
  static constexpr int kV = kK + kKSt * kKVTile;        // kVSt tiles
  static constexpr int kX = kV + kVSt * kKVTile;        // row-sum exchange: [kGroups][128] fp32
  static constexpr int kBar = kX + kGroups * kBlk * 4;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr uint32_t kColO = LD == 256 ? 256 : kSBufs * BK;  // S/P buffers at 0, BK, 2 BK
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSBufs * BK <= kColO && kColO + LD <= kTmemCols, "tensor memory budget");
  static_assert(kBytes <= 232448, "shared memory budget");
};

struct FwdParams {
  __nv_bfloat16* O;
  float* L;
  int32_t* status;
  uint64_t wait_ns;
  int B, H, N;
  int n_tiles;
  int64_t sb, sh, sn;
  float scale;
  int causal;
  int Nk;            // key rows
  int offset;        // Nk - N: key j visible to query i iff j <= i + offset (causal)
};

using ptx::warp_wait;

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Arrive on named barrier `id` without waiting.
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

constexpr int fwd_ld(int hd) { return hd <= 64 ? 64 : (hd <= 128 ? 128 : 256); }

template <int HD>
__global__ void __launch_bounds__(FwdLayout<fwd_ld(HD)>::kThreads, 1)
    fwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const FwdParams prm) {
  constexpr int LD = fwd_ld(HD);
  using Ly = FwdLayout<LD>;
  constexpr int BK = Ly::BK;       // keys per block
  constexpr int NG = Ly::kGroups;  // softmax warps per lane quarter
  constexpr int KC = BK / NG;      // key columns per softmax warp (32)
  constexpr int kKSt = Ly::kKSt;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_addr(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(prm.status, 0, (int32_t)FA_ERR_DEVICE);
    return;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kMisc + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + Ly::kBar + 8 * i; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i)
      ptx::mbar_init(bar(i), (i >= P_FULL0 && i < P_FULL0 + kSBufs)     ? Ly::kSmThreads + 1
                             : (i >= S_READY0 && i < S_READY0 + kSBufs) ? 2
                             : i == DRAIN                               ? (Ly::kSplitMma ? 2 : 1)
                                                                        : 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == Ly::kMma) {
    ptx::tmem_alloc(sbase + Ly::kMisc, Ly::kTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tm = __shfl_sync(0xffffffffu, *tmem_slot, 0);

  // work item: query block qt of head (b, h).  Heads are taken in groups of
  // kHeadGroup (K, V of a few heads shared in L2); inside a group the query
  // blocks go round the heads, the last (longest causal walk) first, so the
  // short walks of the last group fill the SMs at the end of the grid.
  const int bh_total = prm.B * prm.H;
  const int grp = blockIdx.x / (kHeadGroup * prm.n_tiles);
  const int gsize = min(kHeadGroup, bh_total - grp * kHeadGroup);
  const int r = blockIdx.x - grp * kHeadGroup * prm.n_tiles;
  const int bh = grp * kHeadGroup + r % gsize;
  const int qt = prm.n_tiles - 1 - r / gsize;
  const int b = bh / prm.H, h = bh % prm.H;
  const int q0 = qt * kBlk;
  // key blocks this query block sees: all, or (causal) up to the last key its
  // last row sees; none if even that row sees no key
  const int nk_blocks = (prm.Nk + BK - 1) / BK;
  int n_blk = nk_blocks;
  if (prm.causal) {
    const int hi = min(q0 + kBlk - 1, prm.N - 1) + prm.offset;
    n_blk = hi < 0 ? 0 : min(nk_blocks, hi / BK + 1);
  }
  const ptx::Waiter W{abort_flag, prm.status, prm.wait_ns};
  const uint32_t sQ = sbase + Ly::kQ;
  auto sK = [&](int st) -> uint32_t { return sbase + Ly::kK + st * Ly::kKVTile; };
  auto sV = [&](int st) -> uint32_t { return sbase + Ly::kV + st * Ly::kKVTile; };

  if (warp == Ly::kProdK || warp == Ly::kProdV) {
    // ------------------------------------------------------------ producers
    // K producer: Q once, then K_b into stage b % kKSt once S_{b-kKSt} has
    // read it; V producer: V_b into stage b % 2 once O += P_{b-2} V_{b-2} has
    // read it.
    // Each producer waits for its own copies and forwards their completion
    // (K_b to S_READY, V_b to P_FULL), so the MMA warp waits on two
    // barriers per block.  Forwarding block b-1 after issuing block b keeps
    // one copy in flight while the previous one is confirmed.
    const bool isK = warp == Ly::kProdK;
    const int nst = isK ? kKSt : Ly::kVSt;
    const int full0 = isK ? K_FULL0 : V_FULL0, empty0 = isK ? K_EMPTY0 : V_EMPTY0;
    const CUtensorMap* map = isK ? &tmK : &tmV;
    auto forward = [&](int j) -> bool {
      if (!warp_wait(bar(full0 + j % nst), (j / nst) & 1, W)) return false;
      if (lane == 0) {
        if (isK) {
          ptx::mbar_arrive(bar(S_READY0 + j % kSBufs));
          if (j < kSBufs) ptx::mbar_arrive(bar(S_READY0 + j));  // no earlier reader of the buffer
        } else {
          ptx::mbar_arrive(bar(P_FULL0 + j % kSBufs));
        }
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    int issued = 0, forwarded = 0;
    if (lane == 0) {
      ptx::prefetch_tensormap(map);
      if (isK && n_blk > 0) {
        ptx::prefetch_tensormap(&tmQ);
        ptx::mbar_arrive_expect_tx(bar(Q_FULL), Ly::kQTile);
#pragma unroll
        for (int c = 0; c < LD / 64; ++c) ptx::tma_load_4d(sQ + c * Ly::kQChunk, &tmQ, bar(Q_FULL), c * 64, q0, h, b);
      }
    }
    for (int j = 0; j < n_blk; ++j) {
      const int st = j % nst;
      if (j >= nst && !(ok = warp_wait(bar(empty0 + st), ((j - nst) / nst) & 1, W))) break;
      if (lane == 0) {
        const uint32_t dst = isK ? sK(st) : sV(st);
        ptx::mbar_arrive_expect_tx(bar(full0 + st), Ly::kKVTile);
#pragma unroll
        for (int c = 0; c < LD / 64; ++c)
          ptx::tma_load_4d(dst + c * Ly::kKVChunk, map, bar(full0 + st), c * 64, j * BK, h, b);
      }
      __syncwarp();
      issued = j + 1;
      if (j >= 1) {
        if (!(ok = forward(j - 1))) break;
        forwarded = j;
      }
    }
    if (ok && issued > 0) {
      if ((ok = forward(issued - 1))) forwarded = issued;
    }
    if (!ok) {
      // shared memory must not be released under copies still in flight
      if (isK && n_blk > 0) ptx::wait_bounded(bar(Q_FULL), 0, W, false);
      for (int j = forwarded; j < issued; ++j) ptx::wait_bounded(bar(full0 + j % nst), (j / nst) & 1, W, false);
    }
  } else if (warp == Ly::kMma || warp == Ly::kMmaPV) {
    // ------------------------------------------------------------ MMA issue
    // At d <= 128 two warps run two independent chains: one issues S_j as
    // soon as K_j has landed and O += P_{j-3} V_{j-3} has read its buffer; the
    // other issues O += P_j V_j as soon as P_j is in its buffer and V_j has
    // landed.  With one warp issuing both, S_{j+2} waited behind the wait for
    // P_j (or, issued first, for O += P_{j-1} V_{j-1} to complete), and the
    // softmax warps waited for their S block every block (clock64 stamps).
    constexpr uint32_t kIdS = ptx::idesc_bf16_f32(128, BK, false, false);  // S = Q K^T
    constexpr uint32_t kIdO = ptx::idesc_bf16_f32(128, HD, false, true);   // O += P V
    auto kdesc = [&](uint32_t tile, uint32_t chunk, int kk) -> uint64_t {
      return ptx::sdesc_sw128(tile + (kk >> 2) * chunk + (kk & 3) * 32, 16, 1024);
    };
    auto mndesc = [&](uint32_t tile, int kk) -> uint64_t {
      return ptx::sdesc_sw128(tile + kk * 2048, Ly::kKVChunk, 1024);
    };
    const uint32_t tO = tm + Ly::kColO;
    // S_j into buffer j % 3 once K_j has landed and (j >= 3) O += P_{j-3} V_{j-3}
    // has read the buffer
    auto issue_S = [&](int j) -> bool {
      const int sb = j % kSBufs, ks = j % kKSt;
      if (!warp_wait(bar(S_READY0 + sb), (j / kSBufs) & 1, W)) return false;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        const uint32_t tS = tm + sb * BK;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          ptx::mma_ss(tS, kdesc(sQ, Ly::kQChunk, kk), kdesc(sK(ks), Ly::kKVChunk, kk), kIdS, kk > 0);
        ptx::tc_commit(bar(S_FULL0 + sb));
        ptx::tc_commit(bar(K_EMPTY0 + ks));
      }
      __syncwarp();
      return true;
    };
    // O += P_j V_j  (A = P_j from TMEM: the 16-key steps of softmax warp g
    // of a lane quarter in columns [g KC, g KC + KC/2)) once P_j and V_j are there
    auto issue_PV = [&](int j) -> bool {
      const int sb = j % kSBufs, vs = j % Ly::kVSt;
      if (!warp_wait(bar(P_FULL0 + sb), (j / kSBufs) & 1, W)) return false;  // P_j and V_j
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        const uint32_t tP = tm + sb * BK;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          ptx::mma_ts(tO, tP + (kk / (KC / 16)) * KC + (kk % (KC / 16)) * 8, mndesc(sV(vs), kk), kIdO, (j | kk) != 0);
        ptx::tc_commit(bar(S_READY0 + sb));  // buffer free for S_{j+3}
        ptx::tc_commit(bar(O_DONE0 + sb));
        ptx::tc_commit(bar(V_EMPTY0 + vs));
      }
      __syncwarp();
      return true;
    };
    bool ok = n_blk == 0 || (Ly::kSplitMma && warp == Ly::kMmaPV) || warp_wait(bar(Q_FULL), 0, W);
    if constexpr (Ly::kSplitMma) {
      if (warp == Ly::kMma)
        for (int j = 0; ok && j < n_blk; ++j) ok = issue_S(j);
      else
        for (int j = 0; ok && j < n_blk; ++j) ok = issue_PV(j);
    } else {
      // one warp: S_0, S_1, then per block S_{j+2} first (it waits only for
      // O += P_{j-1} V_{j-1}, so the score block two ahead is in flight while
      // the softmax warps finish P_j) and O += P_j V_j
      if (ok && n_blk > 0) ok = issue_S(0);
      if (ok && n_blk > 1) ok = issue_S(1);
      for (int j = 0; ok && j < n_blk; ++j) ok = (j + 2 >= n_blk || issue_S(j + 2)) && issue_PV(j);
    }
    // the softmax warps wait for the last O_DONE; on an abort make sure no
    // MMA is still in flight before tensor memory is freed
    if (ptx::elect_one()) ptx::tc_commit(bar(DRAIN));
    __syncwarp();
    if (!ok) ptx::wait_bounded(bar(DRAIN), 0, W, false);
  } else {
    // ------------------------------------------------------------ softmax
    const int qq = warp & 3, G = warp >> 2;
    const int t = qq * 32 + lane;          // query row in the block == TMEM lane
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const int qrow = q0 + t;
    const int c0 = G * KC;                 // key columns [c0, c0 + KC) of each block
    const float sl2 = prm.scale * kLog2e;
    float* xchg = reinterpret_cast<float*>(smem + Ly::kX);
    float m_run = -INFINITY;               // exponent base (log2 units)
    float l_part = 0.f;                    // this warp's part of the row sum
    // Every softmax warp meets its lane quarter's named barrier n_blk + 1
    // times (once per block, once in the epilogue).  A warp whose wait runs
    // out leaves the loop and makes up the rest with non-blocking arrivals,
    // so that no warp of its quarter blocks there for good.
    int met = n_blk + 1;                   // barrier meetings done when leaving the loop early
    bool ok = true;
    for (int j = 0; j < n_blk; ++j) {
      const int sb = j % kSBufs;       // TMEM buffer of S_j / P_j
      const uint32_t tS = tm + sb * BK;
      if (!(ok = warp_wait(bar(S_FULL0 + sb), (j / kSBufs) & 1, W))) {
        met = j;
        break;
      }
      ptx::tc_fence_after();
      uint32_t r[KC];
      if constexpr (KC == 64)
        ptx::tmem_ld64(tS + lane_off + c0, tS + lane_off + c0 + 32, *reinterpret_cast<uint32_t(*)[64]>(r));
      else
        ptx::tmem_ld32(tS + lane_off + c0, *reinterpret_cast<uint32_t(*)[32]>(r));
      const int k0 = j * BK + c0;
      if ((prm.causal && j * BK + BK - 1 > q0 + prm.offset) || (j * BK + BK > prm.Nk)) {
        // columns c >= lim of this warp's KC are masked (past N_k, or later
        // than the query's last visible key under the causal mask)
        int lim = prm.Nk - k0;
        if (prm.causal) lim = min(lim, qrow + prm.offset - k0 + 1);
#pragma unroll
        for (int c = 0; c < KC; ++c) r[c] = c < lim ? r[c] : __float_as_uint(-INFINITY);
      }
      // row maximum of the raw scores (scale > 0 commutes with max), four
      // independent chains
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < KC; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(r[c]));
      float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
      // row maximum over the lane quarter's warps, exchanged through tensor
      // memory (a shared-memory load would queue behind the score MMAs'
      // operand reads): each warp parks its maximum in the last column of its
      // own S slice, which is dead once loaded and which P does not overwrite
      ptx::tmem_st1(tS + lane_off + c0 + KC - 1, __float_as_uint(mx));
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      named_bar_sync(1 + qq, 32 * NG);
      ptx::tc_fence_after();
      if constexpr (NG == 2) {
        mx = fmaxf(mx, __uint_as_float(ptx::tmem_ld1(tS + lane_off + (c0 ^ KC) + KC - 1)));
      } else {
        uint32_t o3[3];
        ptx::tmem_ld1x3(tS + lane_off + ((G + 1) % NG) * KC + KC - 1, tS + lane_off + ((G + 2) % NG) * KC + KC - 1,
                        tS + lane_off + ((G + 3) % NG) * KC + KC - 1, o3);
        mx = fmaxf(fmaxf(mx, __uint_as_float(o3[0])), fmaxf(__uint_as_float(o3[1]), __uint_as_float(o3[2])));
      }
      float m_new = m_run;
      bool rescale = false;
      if (j == 0 || mx > m_run + kRescaleThreshold) {
        m_new = fmaxf(m_run, mx);
        rescale = j > 0;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O and l move to the new base: O *= 2^(m - m').  O's columns belong
        // to the first two warps of the lane quarter, half each.
        const float alpha = rescale ? ptx::ex2(m_run - m_new) : 1.f;
        l_part *= alpha;
        if (G < 2) {
          if (!(ok = warp_wait(bar(O_DONE0 + (j - 1) % kSBufs), ((j - 1) / kSBufs) & 1, W))) {
            met = j + 1;
            break;
          }
          ptx::tc_fence_after();
          constexpr int kOC = HD / 2;  // this warp's O columns, in 16-column pieces
#pragma unroll
          for (int c = 0; c < kOC; c += 16) {
            uint32_t o[16];
            ptx::tmem_ld16(tm + Ly::kColO + lane_off + G * kOC + c, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st16(tm + Ly::kColO + lane_off + G * kOC + c, o);
          }
          ptx::tmem_st_wait();
        }
      }
      m_run = m_new;
      const float mb = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pk[KC / 2];
#pragma unroll
      for (int c = 0; c < KC; c += 2) {
        const float p0 = ptx::ex2(fmaf(__uint_as_float(r[c]), sl2, -mb));
        const float p1 = ptx::ex2(fmaf(__uint_as_float(r[c + 1]), sl2, -mb));
        l_part += p0 + p1;
        pk[c / 2] = ptx::pack_bf16x2(p0, p1);
      }
      // P columns [c0, c0 + KC/2) lie over this warp's own S columns
#pragma unroll
      for (int u = 0; u < KC / 32; ++u) ptx::tmem_st16(tS + lane_off + c0 + 16 * u, &pk[16 * u]);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(P_FULL0 + sb));
    }
    for (int k = met; k < n_blk + 1; ++k) named_bar_arrive(1 + qq, 32 * NG);
    // epilogue: O / l and L.  O goes into the Q tile (dead once the last S
    // has been computed, which O += P V of the last block implies) as the
    // 64-column, 128-byte-swizzled chunks of a TMA box, and one TMA store
    // writes it (whole lines; rows past N are not written).  Stores from
    // registers, each lane its own row 16 bytes at a time, are uncoalesced.
    if (ok) {
      xchg[G * kBlk + t] = l_part;
      named_bar_sync(1 + qq, 32 * NG);
      float l = 0.f;
#pragma unroll
      for (int g = 0; g < NG; ++g) l += xchg[g * kBlk + t];
      // A row that sees no key (l = 0; every row of a block with n_blk = 0,
      // whose O in tensor memory was never written) stores O = 0, L = +inf.
      // O's columns and L belong to the first two warps of the lane quarter
      if (G < 2 && (n_blk == 0 || warp_wait(bar(O_DONE0 + (n_blk - 1) % kSBufs), ((n_blk - 1) / kSBufs) & 1, W))) {
        ptx::tc_fence_after();
        const bool empty = !(l > 0.f);
        const float inv = empty ? 0.f : 1.f / l;
        constexpr int kOC = HD / 2;
#pragma unroll 1
        for (int c = 0; c < kOC; c += 16) {
          uint32_t o[16];
          if (n_blk > 0) ptx::tmem_ld16(tm + Ly::kColO + lane_off + G * kOC + c, o);
#pragma unroll
          for (int q = 0; q < 2; ++q) {  // 8 columns (16 bytes) each
            const int col = G * kOC + c + 8 * q;
            const uint32_t piece = (uint32_t)((col & 63) >> 3);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = empty ? 0u : ptx::pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * inv,
                                                  __uint_as_float(o[8 * q + 2 * e + 1]) * inv);
            ptx::st_shared_v4(sQ + (col >> 6) * Ly::kQChunk + t * 128 + ((piece ^ (uint32_t)(t & 7)) << 4), w[0],
                              w[1], w[2], w[3]);
          }
        }
        ptx::fence_proxy_async_smem();
        if (G == 0 && qrow < prm.N)
          prm.L[(int64_t)bh * prm.N + qrow] = empty ? INFINITY : (m_run + log2f(l)) * kLn2;
      }
    }
    // every O warp reaches this barrier (also after a wait ran out, which
    // set the CTA's abort flag: the store is then skipped)
    if (G < 2) {
      named_bar_sync(5, 32 * 8);
      if (warp == 0 && lane == 0 && !*abort_flag) {
#pragma unroll
        for (int c = 0; c < LD / 64; ++c) ptx::tma_store_4d(&tmO, sQ + c * Ly::kQChunk, c * 64, q0, h, b);
        ptx::bulk_commit();
        ptx::bulk_wait_read_all();  // shared memory is released at exit
      }
      __syncwarp();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == Ly::kMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tm, Ly::kTmemCols);
  }
}

template <int HD>
cudaError_t launch_fwd_hd(const fa_problem& p, const CUtensorMap* maps, const FwdParams& prm, cudaStream_t s) {
  using Ly = FwdLayout<fwd_ld(HD)>;
  cudaError_t e = cudaFuncSetAttribute(fwd_sm103_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((int64_t)prm.n_tiles * p.B * p.H));
  fwd_sm103_kernel<HD><<<grid, Ly::kThreads, Ly::kBytes, s>>>(maps[0], maps[1], maps[2], maps[3], prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_sm103(const fa_problem& p, const void* Q, const void* K, const void* V, void* O, float* L,
                             int32_t* status, uint64_t wait_ns, cudaStream_t s) {
  CUtensorMap maps[4];
  const int bk = p.d == 256 ? 64 : kBlk;  // key block rows
  if (!make_bf16_tile_map(&maps[0], Q, p, false) || !make_bf16_tile_map_rows(&maps[1], K, p, true, bk) ||
      !make_bf16_tile_map_rows(&maps[2], V, p, true, bk) || !make_bf16_tile_map(&maps[3], O, p, false))
    return cudaErrorInvalidValue;
  FwdParams prm;
  prm.O = (__nv_bfloat16*)O;
  prm.L = L;
  prm.status = status;
  prm.wait_ns = wait_ns;
  prm.B = p.B;
  prm.H = p.H;
  prm.N = p.N;
  prm.n_tiles = (int)ceil_div(p.N, kBlk);
  prm.Nk = p.N_k;
  prm.offset = (int)causal_offset(p);
  prm.sb = p.stride_b;
  prm.sh = p.stride_h;
  prm.sn = p.stride_n;
  prm.scale = p.scale;
  prm.causal = p.causal;
  switch (p.d) {
    case 32: return launch_fwd_hd<32>(p, maps, prm, s);
    case 64: return launch_fwd_hd<64>(p, maps, prm, s);
    case 96: return launch_fwd_hd<96>(p, maps, prm, s);
    case 128: return launch_fwd_hd<128>(p, maps, prm, s);
    case 256: return launch_fwd_hd<256>(p, maps, prm, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
