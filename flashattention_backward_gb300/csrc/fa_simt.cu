// CUDA-core (FFMA) kernels for float32 problems (tensor cores have no fp32
// mode that keeps float32 accuracy, and the fp32 workload is a small
// correctness problem):
//  * the forward pass (online softmax);
//  * the backward pass.
// Both use 64 x 64 tiles and 256 threads arranged 16 x 16; thread (ty, tx)
// owns rows ty + 16a and columns tx + 16b of a tile, so the lanes that share
// a row sit in one half-warp and reduce with 4 shuffles.

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

// Copy a kT x HD tile of rows [row0, row0 + kT) into shared memory as fp32
// with row pitch `pitch`; rows >= N are zero.
template <typename T, int HD>
__device__ __forceinline__ void load_tile(float* dst, int pitch, const T* src, int64_t sn, int row0, int N) {
  for (int k = threadIdx.x; k < kT * HD; k += kThreads) {
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
                                                            int64_t sh, int64_t sn, float scale, int causal) {
  constexpr int kPQ = HD + 1, kPV = HD, kPP = kT + 1;
  constexpr int kCols = HD / 16;
  extern __shared__ float smem[];
  float* sQ = smem;
  float* sK = sQ + kT * kPQ;
  float* sV = sK + kT * kPQ;
  float* sP = sV + kT * kPV;

  const int tiles = (N + kT - 1) / kT;
  const int qt = blockIdx.x % tiles;
  const int bh = blockIdx.x / tiles;
  const int b = bh / H, h = bh % H;
  const int64_t head = (int64_t)b * sb + (int64_t)h * sh;
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

  const int kt_end = causal ? qt + 1 : tiles;
  for (int kt = 0; kt < kt_end; ++kt) {
    const int k0 = kt * kT;
    __syncthreads();  // previous tile's sK/sV/sP reads are done
    load_tile<T, HD>(sK, kPQ, K + head, sn, k0, N);
    load_tile<T, HD>(sV, kPV, V + head, sn, k0, N);
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
        const bool masked = (j >= N) || (causal && j > i);
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
    const float inv = 1.f / l[a];
    T* orow = O + head + (int64_t)i * sn;
#pragma unroll
    for (int u = 0; u < kCols; ++u) from_f(orow + tx + 16 * u, acc[a][u] * inv);
    if (tx == 0) L[(int64_t)bh * N + i] = (m[a] + log2f(l[a])) * kLn2;
  }
}

// ----------------------------------------------------------------------------
// fp32 backward.  One block per (b, h, 64-key block); inner loop over query
// tiles.  dV and dK accumulate in registers; dQ partials go to the fp32
// accumulator with atomicAdd (unit-blocked layout of include/fa.h).
// ----------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(kThreads) bwd_simt_fp32_kernel(
    const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
    const float* __restrict__ dO, const float* __restrict__ Lg, const float* __restrict__ Dg,
    float* __restrict__ dq_accum, float* __restrict__ dK, float* __restrict__ dV, int H, int N, int64_t sb,
    int64_t sh, int64_t sn, float scale, int causal, int64_t slice_elems) {
  // slice_elems > 0 (deterministic): this key block's dQ contributions are
  // stored into its own slice of the accumulator instead of added.
  constexpr int kP = HD + 1, kPP = kT + 1;
  constexpr int kCols = HD / 16;
  extern __shared__ float smem[];
  float* sK = smem;
  float* sV = sK + kT * kP;
  float* sQ = sV + kT * kP;
  float* sdO = sQ + kT * kP;
  float* sP = sdO + kT * kP;   // [query][key]
  float* sdS = sP + kT * kPP;  // [query][key]
  float* sL = sdS + kT * kPP;  // L * log2(e), +inf for rows >= N
  float* sD = sL + kT;

  const int tiles = (N + kT - 1) / kT;
  const int kb = blockIdx.x % tiles;
  const int bh = blockIdx.x / tiles;
  const int b = bh / H, h = bh % H;
  const int64_t head = (int64_t)b * sb + (int64_t)h * sh;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int k0 = kb * kT;
  const float sl2 = scale * kLog2e;
  const int acc_tiles = (N + kTileRows - 1) / kTileRows;

  load_tile<float, HD>(sK, kP, K + head, sn, k0, N);
  load_tile<float, HD>(sV, kP, V + head, sn, k0, N);

  float dv[4][kCols], dk[4][kCols];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int u = 0; u < kCols; ++u) dv[a][u] = dk[a][u] = 0.f;

  for (int qt = causal ? kb : 0; qt < tiles; ++qt) {
    const int q0 = qt * kT;
    __syncthreads();
    load_tile<float, HD>(sQ, kP, Q + head, sn, q0, N);
    load_tile<float, HD>(sdO, kP, dO + head, sn, q0, N);
    if (threadIdx.x < kT) {
      const int i = q0 + threadIdx.x;
      sL[threadIdx.x] = i < N ? Lg[(int64_t)bh * N + i] * kLog2e : INFINITY;
      sD[threadIdx.x] = i < N ? Dg[(int64_t)bh * N + i] : 0.f;
    }
    __syncthreads();
    // S, P and dP, dS for the (query a, key bb) entries this thread owns
    float s[4][4], dp[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) s[a][bb] = dp[a][bb] = 0.f;
#pragma unroll 2
    for (int c = 0; c < HD; ++c) {
      float qv[4], gv[4], kv[4], vv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        qv[a] = sQ[(ty + 16 * a) * kP + c];
        gv[a] = sdO[(ty + 16 * a) * kP + c];
      }
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        kv[bb] = sK[(tx + 16 * bb) * kP + c];
        vv[bb] = sV[(tx + 16 * bb) * kP + c];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          s[a][bb] = fmaf(qv[a], kv[bb], s[a][bb]);
          dp[a][bb] = fmaf(gv[a], vv[bb], dp[a][bb]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int il = ty + 16 * a, i = q0 + il;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int jl = tx + 16 * bb, j = k0 + jl;
        const bool masked = (j >= N) || (causal && j > i);
        const float p = masked ? 0.f : ptx::ex2(fmaf(s[a][bb], sl2, -sL[il]));
        sP[il * kPP + jl] = p;
        sdS[il * kPP + jl] = p * (dp[a][bb] - sD[il]);
      }
    }
    __syncthreads();
    // dV[j] += sum_i P[i][j] dO[i];  dK[j] += sum_i dS[i][j] Q[i]
#pragma unroll 2
    for (int i = 0; i < kT; ++i) {
      float pv[4], sv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        pv[a] = sP[i * kPP + ty + 16 * a];
        sv[a] = sdS[i * kPP + ty + 16 * a];
      }
#pragma unroll
      for (int u = 0; u < kCols; ++u) {
        const float g = sdO[i * kP + tx + 16 * u];
        const float q = sQ[i * kP + tx + 16 * u];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          dv[a][u] = fmaf(pv[a], g, dv[a][u]);
          dk[a][u] = fmaf(sv[a], q, dk[a][u]);
        }
      }
    }
    // dQ[i] partial = sum_j dS[i][j] K[j]
    float dq[4][kCols];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int u = 0; u < kCols; ++u) dq[a][u] = 0.f;
#pragma unroll 2
    for (int j = 0; j < kT; ++j) {
      float sv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) sv[a] = sdS[(ty + 16 * a) * kPP + j];
#pragma unroll
      for (int u = 0; u < kCols; ++u) {
        const float kv = sK[j * kP + tx + 16 * u];
#pragma unroll
        for (int a = 0; a < 4; ++a) dq[a][u] = fmaf(sv[a], kv, dq[a][u]);
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
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
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int j = k0 + ty + 16 * a;
    if (j >= N) continue;
#pragma unroll
    for (int u = 0; u < kCols; ++u) {
      const int c = tx + 16 * u;
      dV[head + (int64_t)j * sn + c] = dv[a][u];
      dK[head + (int64_t)j * sn + c] = scale * dk[a][u];
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
                                                   p.scale, p.causal);
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
    case 128: return launch_fwd_t<T, 128>(p, q, k, v, o, L, s);
  }
  return cudaErrorInvalidValue;
}

template <int HD>
cudaError_t launch_bwd_fp32_t(const fa_problem& p, const float* Q, const float* K, const float* V, const float* dO,
                              const float* L, const float* D, float* acc, float* dK, float* dV, cudaStream_t s) {
  const size_t sm = sizeof(float) * (size_t)(4 * kT * (HD + 1) + 2 * kT * (kT + 1) + 2 * kT);
  cudaError_t e = set_smem(bwd_simt_fp32_kernel<HD>, sm);
  if (e != cudaSuccess) return e;
  const int tiles = (p.N + kT - 1) / kT;
  const dim3 grid((unsigned)((int64_t)p.B * p.H * tiles));
  bwd_simt_fp32_kernel<HD><<<grid, kThreads, sm, s>>>(Q, K, V, dO, L, D, acc, dK, dV, p.H, p.N, p.stride_b,
                                                      p.stride_h, p.stride_n, p.scale, p.causal,
                                                      deterministic(p) ? dq_slice_elems(p) : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const fa_problem& p, const void* Q, const void* K, const void* V, void* O, float* L,
                            cudaStream_t s) {
  return launch_fwd_dt<float>(p, Q, K, V, O, L, s);
}

cudaError_t launch_bwd_simt_fp32(const fa_problem& p, const float* Q, const float* K, const float* V,
                                 const float* dO, const float* L, const float* D, float* acc, float* dK, float* dV,
                                 cudaStream_t s) {
  switch (p.d) {
    case 16: return launch_bwd_fp32_t<16>(p, Q, K, V, dO, L, D, acc, dK, dV, s);
    case 32: return launch_bwd_fp32_t<32>(p, Q, K, V, dO, L, D, acc, dK, dV, s);
    case 64: return launch_bwd_fp32_t<64>(p, Q, K, V, dO, L, D, acc, dK, dV, s);
    case 128: return launch_bwd_fp32_t<128>(p, Q, K, V, dO, L, D, acc, dK, dV, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
