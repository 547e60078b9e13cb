// CUDA-core (FFMA) kernels for float32 problems (tensor cores have no fp32
// mode that keeps float32 accuracy, and the fp32 workload is a small
// correctness problem); all arithmetic is fp32:
//  * the forward pass (online softmax), 64 x 64 tiles;
//  * the backward pass, 64 x 64 tiles (32 x 32 at d = 256, to fit shared
//    memory).
// 256 threads arranged 16 x 16; thread (ty, tx) owns rows ty + 16a and
// columns tx + 16b of a tile, so the lanes that share a row sit in one
// half-warp and reduce with 4 shuffles.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "dq_layout.cuh"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kT = 64;          // rows per tile (query and key)
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ void from_f(float* p, float v) { *p = v; }

// Copy a ROWS x HD tile of rows [row0, row0 + ROWS) into shared memory as fp32
// with row pitch `pitch`; rows >= N are zero.
template <typename T, int HD, int ROWS = kT>
__device__ __forceinline__ void load_tile(float* dst, int pitch, const T* src, int64_t sn, int row0, int N) {
  for (int k = threadIdx.x; k < ROWS * HD; k += kThreads) {
    const int r = k / HD, c = k % HD;
    const int n = row0 + r;
    dst[r * pitch + c] = n < N ? to_f(src[(int64_t)n * sn + c]) : 0.f;
  }
}

__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int m = 8; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int m = 8; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// ----------------------------------------------------------------------------
// Forward.  One block per (b, h, 64-row query tile); loop over key tiles with
// running max m (log2 domain), running sum l and rescale alpha = 2^(m - m').
// ----------------------------------------------------------------------------
template <typename T, int HD>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                            const T* __restrict__ V, T* __restrict__ O,
                                                            float* __restrict__ L, int H, int N, int64_t sb,
                                                            int64_t sh, int64_t sn, float scale, int causal,
                                                            int Nk, int64_t ksb, int64_t ksh, int64_t ksn) {
  // Q, O: N rows with strides (sb, sh, sn); K, V: Nk rows with (ksb, ksh,
  // ksn).  Causal: key j visible to query i iff j <= i + Nk - N.
  constexpr int kPQ = HD + 1, kPV = HD, kPP = kT + 1;
  constexpr int kCols = HD / 16;
  extern __shared__ float smem[];
  float* sQ = smem;
  float* sK = sQ + kT * kPQ;
  float* sV = sK + kT * kPQ;
  float* sP = sV + kT * kPV;

  const int tiles = (N + kT - 1) / kT;
  const int k_tiles = (Nk + kT - 1) / kT;
  const int offset = Nk - N;
  const int qt = blockIdx.x % tiles;
  const int bh = blockIdx.x / tiles;
  const int b = bh / H, h = bh % H;
  const int64_t head = (int64_t)b * sb + (int64_t)h * sh;
  const int64_t khead = (int64_t)b * ksb + (int64_t)h * ksh;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int q0 = qt * kT;
  const float sl2 = scale * kLog2e;

  load_tile<T, HD>(sQ, kPQ, Q + head, sn, q0, N);

  float m[4], l[4], acc[4][kCols];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m[a] = -INFINITY;
    l[a] = 0.f;
#pragma unroll
    for (int u = 0; u < kCols; ++u) acc[a][u] = 0.f;
  }

  int kt_end = k_tiles;
  if (causal) {  // up to the last key the tile's last row sees
    const int hi = min(q0 + kT - 1, N - 1) + offset;
    kt_end = hi < 0 ? 0 : min(k_tiles, hi / kT + 1);
  }
  for (int kt = 0; kt < kt_end; ++kt) {
    const int k0 = kt * kT;
    __syncthreads();  // previous tile's sK/sV/sP reads are done
    load_tile<T, HD>(sK, kPQ, K + khead, ksn, k0, Nk);
    load_tile<T, HD>(sV, kPV, V + khead, ksn, k0, Nk);
    __syncthreads();

    float s[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) s[a][bb] = 0.f;
#pragma unroll 4
    for (int c = 0; c < HD; ++c) {
      float qv[4], kv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) qv[a] = sQ[(ty + 16 * a) * kPQ + c];
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) kv[bb] = sK[(tx + 16 * bb) * kPQ + c];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) s[a][bb] = fmaf(qv[a], kv[bb], s[a][bb]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = q0 + ty + 16 * a;
      float rmax = -INFINITY;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int j = k0 + tx + 16 * bb;
        const bool masked = (j >= Nk) || (causal && j > i + offset);
        s[a][bb] = masked ? -INFINITY : s[a][bb] * sl2;
        rmax = fmaxf(rmax, s[a][bb]);
      }
      rmax = half_warp_max(rmax);
      const float m_new = fmaxf(m[a], rmax);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ptx::ex2(m[a] - m_use);
      float rsum = 0.f;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const float p = ptx::ex2(s[a][bb] - m_use);
        rsum += p;
        sP[(ty + 16 * a) * kPP + tx + 16 * bb] = p;
      }
      rsum = half_warp_sum(rsum);
      l[a] = l[a] * alpha + rsum;
      m[a] = m_new;
#pragma unroll
      for (int u = 0; u < kCols; ++u) acc[a][u] *= alpha;
    }
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < kT; ++j) {
      float pv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) pv[a] = sP[(ty + 16 * a) * kPP + j];
#pragma unroll
      for (int u = 0; u < kCols; ++u) {
        const float v = sV[j * kPV + tx + 16 * u];
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a][u] = fmaf(pv[a], v, acc[a][u]);
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = q0 + ty + 16 * a;
    if (i >= N) continue;
    const bool empty = !(l[a] > 0.f);  // no visible key: O = 0, L = +inf
    const float inv = empty ? 0.f : 1.f / l[a];
    T* orow = O + head + (int64_t)i * sn;
#pragma unroll
    for (int u = 0; u < kCols; ++u) from_f(orow + tx + 16 * u, empty ? 0.f : acc[a][u] * inv);
    if (tx == 0) L[(int64_t)bh * N + i] = empty ? INFINITY : (m[a] + log2f(l[a])) * kLn2;
  }
}

// ----------------------------------------------------------------------------
// Backward.  One block per (b, h, KT-key block); inner loop over query tiles
// of KT rows.  dV and dK accumulate in registers; dQ partials go to the fp32
// accumulator with atomicAdd (unit-blocked layout of include/fa.h).
// ----------------------------------------------------------------------------
template <typename T, int HD, int KT>
__global__ void __launch_bounds__(kThreads) bwd_simt_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V, const T* __restrict__ dO,
    const float* __restrict__ Lg, const float* __restrict__ Dg, float* __restrict__ dq_accum, T* __restrict__ dK,
    T* __restrict__ dV, int H, int N, int64_t sb, int64_t sh, int64_t sn, float scale, int causal,
    int64_t slice_elems, int Nk, int64_t ksb, int64_t ksh, int64_t ksn, unsigned long long* pair_count) {
  // slice_elems > 0 (deterministic): this key block's dQ contributions are
  // stored into its own slice of the accumulator instead of added.
  // Q, dO: N rows with strides (sb, sh, sn); K, V, dK, dV: Nk rows with
  // (ksb, ksh, ksn).  Causal: key j visible to query i iff j <= i + Nk - N.
  constexpr int kP = HD + 1, kPP = KT + 1;
  constexpr int kR = KT / 16;   // rows (and columns) of a tile per thread
  constexpr int kCols = HD / 16;
  extern __shared__ float smem[];
  float* sK = smem;
  float* sV = sK + KT * kP;
  float* sQ = sV + KT * kP;
  float* sdO = sQ + KT * kP;
  float* sP = sdO + KT * kP;   // [query][key]
  float* sdS = sP + KT * kPP;  // [query][key]
  float* sL = sdS + KT * kPP;  // L * log2(e), +inf for rows >= N
  float* sD = sL + KT;

  const int tiles = (N + KT - 1) / KT;       // query tiles
  const int k_tiles = (Nk + KT - 1) / KT;    // key blocks, one per block of threads
  const int offset = Nk - N;
  const int kb = blockIdx.x % k_tiles;
  const int bh = blockIdx.x / k_tiles;
  const int b = bh / H, h = bh % H;
  const int64_t head = (int64_t)b * sb + (int64_t)h * sh;
  const int64_t khead = (int64_t)b * ksb + (int64_t)h * ksh;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int k0 = kb * KT;
  const float sl2 = scale * kLog2e;
  const int acc_tiles = (N + kTileRows - 1) / kTileRows;

  load_tile<T, HD, KT>(sK, kP, K + khead, ksn, k0, Nk);
  load_tile<T, HD, KT>(sV, kP, V + khead, ksn, k0, Nk);

  float dv[kR][kCols], dk[kR][kCols];
#pragma unroll
  for (int a = 0; a < kR; ++a)
#pragma unroll
    for (int u = 0; u < kCols; ++u) dv[a][u] = dk[a][u] = 0.f;

  // first query tile holding a query that sees key k0: i >= k0 - offset
  const int qt_first = causal && k0 > offset ? (k0 - offset) / KT : 0;
  unsigned n_exec = 0, n_masked = 0;  // tile-pair accounting (pair_count)
  for (int qt = qt_first; qt < tiles; ++qt) {
    const int q0 = qt * KT;
    if (pair_count) {
      ++n_exec;
      n_masked += !causal || k0 <= min(q0 + KT - 1, N - 1) + offset ? 0u : 1u;
    }
    __syncthreads();
    load_tile<T, HD, KT>(sQ, kP, Q + head, sn, q0, N);
    load_tile<T, HD, KT>(sdO, kP, dO + head, sn, q0, N);
    if (threadIdx.x < KT) {
      const int i = q0 + threadIdx.x;
      sL[threadIdx.x] = i < N ? Lg[(int64_t)bh * N + i] * kLog2e : INFINITY;
      sD[threadIdx.x] = i < N ? Dg[(int64_t)bh * N + i] : 0.f;
    }
    __syncthreads();
    // S, P and dP, dS for the (query a, key bb) entries this thread owns
    float s[kR][kR], dp[kR][kR];
#pragma unroll
    for (int a = 0; a < kR; ++a)
#pragma unroll
      for (int bb = 0; bb < kR; ++bb) s[a][bb] = dp[a][bb] = 0.f;
#pragma unroll 2
    for (int c = 0; c < HD; ++c) {
      float qv[kR], gv[kR], kv[kR], vv[kR];
#pragma unroll
      for (int a = 0; a < kR; ++a) {
        qv[a] = sQ[(ty + 16 * a) * kP + c];
        gv[a] = sdO[(ty + 16 * a) * kP + c];
      }
#pragma unroll
      for (int bb = 0; bb < kR; ++bb) {
        kv[bb] = sK[(tx + 16 * bb) * kP + c];
        vv[bb] = sV[(tx + 16 * bb) * kP + c];
      }
#pragma unroll
      for (int a = 0; a < kR; ++a)
#pragma unroll
        for (int bb = 0; bb < kR; ++bb) {
          s[a][bb] = fmaf(qv[a], kv[bb], s[a][bb]);
          dp[a][bb] = fmaf(gv[a], vv[bb], dp[a][bb]);
        }
    }
#pragma unroll
    for (int a = 0; a < kR; ++a) {
      const int il = ty + 16 * a, i = q0 + il;
#pragma unroll
      for (int bb = 0; bb < kR; ++bb) {
        const int jl = tx + 16 * bb, j = k0 + jl;
        const bool masked = (j >= Nk) || (causal && j > i + offset);
        const float p = masked ? 0.f : ptx::ex2(fmaf(s[a][bb], sl2, -sL[il]));
        sP[il * kPP + jl] = p;
        sdS[il * kPP + jl] = p * (dp[a][bb] - sD[il]);
      }
    }
    __syncthreads();
    // dV[j] += sum_i P[i][j] dO[i];  dK[j] += sum_i dS[i][j] Q[i]
#pragma unroll 2
    for (int i = 0; i < KT; ++i) {
      float pv[kR], sv[kR];
#pragma unroll
      for (int a = 0; a < kR; ++a) {
        pv[a] = sP[i * kPP + ty + 16 * a];
        sv[a] = sdS[i * kPP + ty + 16 * a];
      }
#pragma unroll
      for (int u = 0; u < kCols; ++u) {
        const float g = sdO[i * kP + tx + 16 * u];
        const float q = sQ[i * kP + tx + 16 * u];
#pragma unroll
        for (int a = 0; a < kR; ++a) {
          dv[a][u] = fmaf(pv[a], g, dv[a][u]);
          dk[a][u] = fmaf(sv[a], q, dk[a][u]);
        }
      }
    }
    // dQ[i] partial = sum_j dS[i][j] K[j]
    float dq[kR][kCols];
#pragma unroll
    for (int a = 0; a < kR; ++a)
#pragma unroll
      for (int u = 0; u < kCols; ++u) dq[a][u] = 0.f;
#pragma unroll 2
    for (int j = 0; j < KT; ++j) {
      float sv[kR];
#pragma unroll
      for (int a = 0; a < kR; ++a) sv[a] = sdS[(ty + 16 * a) * kPP + j];
#pragma unroll
      for (int u = 0; u < kCols; ++u) {
        const float kv = sK[j * kP + tx + 16 * u];
#pragma unroll
        for (int a = 0; a < kR; ++a) dq[a][u] = fmaf(sv[a], kv, dq[a][u]);
      }
    }
#pragma unroll
    for (int a = 0; a < kR; ++a) {
      const int i = q0 + ty + 16 * a;
      if (i >= N) continue;
#pragma unroll
      for (int u = 0; u < kCols; ++u) {
        const int c = tx + 16 * u;
        if (slice_elems > 0)
          dq_accum[kb * slice_elems + dq_accum_index(bh, acc_tiles, i, c, HD)] = dq[a][u];
        else
          atomicAdd(dq_accum + dq_accum_index(bh, acc_tiles, i, c, HD), dq[a][u]);
      }
    }
  }
  if (pair_count && threadIdx.x == 0) {
    atomicAdd(pair_count, (unsigned long long)n_exec);
    atomicAdd(pair_count + 1, (unsigned long long)n_masked);
  }
#pragma unroll
  for (int a = 0; a < kR; ++a) {
    const int j = k0 + ty + 16 * a;
    if (j >= Nk) continue;
#pragma unroll
    for (int u = 0; u < kCols; ++u) {
      const int c = tx + 16 * u;
      from_f(dV + khead + (int64_t)j * ksn + c, dv[a][u]);
      from_f(dK + khead + (int64_t)j * ksn + c, scale * dk[a][u]);
    }
  }
}

template <typename Kern>
cudaError_t set_smem(Kern k, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int HD>
cudaError_t launch_fwd_t(const fa_problem& p, const T* Q, const T* K, const T* V, T* O, float* L, cudaStream_t s) {
  const size_t sm = sizeof(float) * (size_t)(2 * kT * (HD + 1) + kT * HD + kT * (kT + 1));
  cudaError_t e = set_smem(fwd_simt_kernel<T, HD>, sm);
  if (e != cudaSuccess) return e;
  const int tiles = (p.N + kT - 1) / kT;
  const dim3 grid((unsigned)((int64_t)p.B * p.H * tiles));
  fwd_simt_kernel<T, HD><<<grid, kThreads, sm, s>>>(Q, K, V, O, L, p.H, p.N, p.stride_b, p.stride_h, p.stride_n,
                                                   p.scale, p.causal, p.N_k, p.kstride_b, p.kstride_h,
                                                   p.kstride_n);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fwd_dt(const fa_problem& p, const void* Q, const void* K, const void* V, void* O, float* L,
                          cudaStream_t s) {
  const T* q = (const T*)Q;
  const T* k = (const T*)K;
  const T* v = (const T*)V;
  T* o = (T*)O;
  switch (p.d) {
    case 16: return launch_fwd_t<T, 16>(p, q, k, v, o, L, s);
    case 32: return launch_fwd_t<T, 32>(p, q, k, v, o, L, s);
    case 64: return launch_fwd_t<T, 64>(p, q, k, v, o, L, s);
    case 96: return launch_fwd_t<T, 96>(p, q, k, v, o, L, s);
    case 128: return launch_fwd_t<T, 128>(p, q, k, v, o, L, s);
    case 256: return launch_fwd_t<T, 256>(p, q, k, v, o, L, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T, int HD>
cudaError_t launch_bwd_t(const fa_problem& p, const void* Q, const void* K, const void* V, const void* dO,
                         const float* L, const float* D, float* acc, void* dK, void* dV, cudaStream_t s,
                         unsigned long long* pc) {
  constexpr int KT = HD == 256 ? 32 : kT;
  const size_t sm = sizeof(float) * (size_t)(4 * KT * (HD + 1) + 2 * KT * (KT + 1) + 2 * KT);
  cudaError_t e = set_smem(bwd_simt_kernel<T, HD, KT>, sm);
  if (e != cudaSuccess) return e;
  const int k_tiles = (p.N_k + KT - 1) / KT;
  const dim3 grid((unsigned)((int64_t)p.B * p.H * k_tiles));
  bwd_simt_kernel<T, HD, KT><<<grid, kThreads, sm, s>>>(
      (const T*)Q, (const T*)K, (const T*)V, (const T*)dO, L, D, acc, (T*)dK, (T*)dV, p.H, p.N, p.stride_b,
      p.stride_h, p.stride_n, p.scale, p.causal, deterministic(p) ? dq_slice_elems(p) : 0, p.N_k, p.kstride_b,
      p.kstride_h, p.kstride_n, pc);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_dt(const fa_problem& p, const void* Q, const void* K, const void* V, const void* dO,
                          const float* L, const float* D, float* acc, void* dK, void* dV, cudaStream_t s,
                          unsigned long long* pc) {
  switch (p.d) {
    case 16: return launch_bwd_t<T, 16>(p, Q, K, V, dO, L, D, acc, dK, dV, s, pc);
    case 32: return launch_bwd_t<T, 32>(p, Q, K, V, dO, L, D, acc, dK, dV, s, pc);
    case 64: return launch_bwd_t<T, 64>(p, Q, K, V, dO, L, D, acc, dK, dV, s, pc);
    case 96: return launch_bwd_t<T, 96>(p, Q, K, V, dO, L, D, acc, dK, dV, s, pc);
    case 128: return launch_bwd_t<T, 128>(p, Q, K, V, dO, L, D, acc, dK, dV, s, pc);
    case 256: return launch_bwd_t<T, 256>(p, Q, K, V, dO, L, D, acc, dK, dV, s, pc);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

// fp32 only: every bf16 head dim has tensor-core kernels.
cudaError_t launch_fwd_simt(const fa_problem& p, const void* Q, const void* K, const void* V, void* O, float* L,
                            cudaStream_t s) {
  if (p.dtype == FA_BF16) return cudaErrorInvalidValue;
  return launch_fwd_dt<float>(p, Q, K, V, O, L, s);
}

cudaError_t launch_bwd_simt(const fa_problem& p, const void* Q, const void* K, const void* V, const void* dO,
                            const float* L, const float* D, float* acc, void* dK, void* dV, cudaStream_t s,
                            unsigned long long* pair_count) {
  if (p.dtype == FA_BF16) return cudaErrorInvalidValue;
  return launch_bwd_dt<float>(p, Q, K, V, dO, L, D, acc, dK, dV, s, pair_count);
}

}  // namespace fa
