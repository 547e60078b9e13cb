// Host side of libfa: argument validation, the per-device status word, and
// the two bandwidth-bound kernels of the backward pass (preprocess and
// convert).  Entry points are declared in include/fa.h.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "dq_layout.cuh"
#include "row_dot.cuh"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// ----------------------------------------------------------------------------
// Device status word: one int per device, in a file-scope __device__ variable.
// Host code must not hand the symbol itself to a kernel (on the host it only
// names a shadow); its device address is looked up once per device.
// ----------------------------------------------------------------------------
__device__ int32_t g_status_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_status_ptr[kMaxDevices] = {nullptr};
std::atomic<uint64_t> g_wait_ns{2000000000ull};
}  // namespace

int32_t* device_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int32_t*>(p);
  }
  return g_status_ptr[dev];
}

uint64_t wait_limit_ns() { return g_wait_ns.load(); }

// ----------------------------------------------------------------------------
// Preprocess: D = rowsum(O * dO) in fp32 and zero the dQ accumulator.
// One block of 256 threads per (b, h, 128-row tile).  Each thread reads 16
// bytes of O and of dO per step; the lanes that share a row reduce with warp
// shuffles.  The same block then zeroes that tile of the accumulator
// (128 * d floats, float4 stores).  Pure HBM streaming.
// ----------------------------------------------------------------------------
template <typename T, int HD>
__global__ void __launch_bounds__(256) preprocess_kernel(const T* __restrict__ O, const T* __restrict__ dO,
                                                         float* __restrict__ D, float* __restrict__ dq_accum,
                                                         int H, int N, int64_t sb, int64_t sh, int64_t sn,
                                                         int tiles_per_head, int zero_slices,
                                                         int64_t slice_elems) {
  using RD = RowDot<T, HD>;
  constexpr int kRowsPerStep = 256 / RD::kLanes;
  constexpr int kSteps = kTileRows / kRowsPerStep;
  const int tile = blockIdx.x % tiles_per_head;
  const int bh = blockIdx.x / tiles_per_head;
  const int b = bh / H, h = bh % H;
  const int sub = threadIdx.x % RD::kLanes;
  const int row_in_step = threadIdx.x / RD::kLanes;
  const int64_t head_off = (int64_t)b * sb + (int64_t)h * sh;

  float acc[kSteps];
#pragma unroll
  for (int s = 0; s < kSteps; ++s) {
    const int n = tile * kTileRows + s * kRowsPerStep + row_in_step;
    acc[s] = n < N ? RD::partial(O + head_off + (int64_t)n * sn, dO + head_off + (int64_t)n * sn, sub) : 0.f;
  }
#pragma unroll
  for (int s = 0; s < kSteps; ++s) {
    acc[s] = RD::reduce(acc[s]);
    const int n = tile * kTileRows + s * kRowsPerStep + row_in_step;
    if (sub == 0 && n < N) D[(int64_t)bh * N + n] = acc[s];
  }
  // zero this tile of the accumulator (128 * HD floats) in each slice
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < zero_slices; ++s) {
    float4* z = reinterpret_cast<float4*>(dq_accum + s * slice_elems +
                                          ((int64_t)bh * tiles_per_head + tile) * (int64_t)kTileRows * HD);
#pragma unroll 4
    for (int k = threadIdx.x; k < kTileRows * HD / 4; k += 256) z[k] = zero;
  }
}

template <typename T>
static cudaError_t launch_preprocess_t(const fa_problem& p, const T* O, const T* dO, float* D, float* acc,
                                       cudaStream_t s) {
  const int tiles = (int)ceil_div(p.N, kTileRows);
  const dim3 grid((unsigned)((int64_t)p.B * p.H * tiles));
  // Deterministic, tensor-core kernels: every slice element the convert reads
  // is written by the backward kernel, so nothing needs zeroing.  The
  // CUDA-core kernel's 64- or 32-row key blocks leave parts of some slices
  // untouched; zero them all.
  const int zero_slices = !deterministic(p) ? 1 : (tensor_core(p) ? 0 : (int)dq_slices(p));
  const int64_t slice_elems = dq_slice_elems(p);
#define FA_PRE_CASE(HDV)                                                                                    \
  case HDV:                                                                                                 \
    preprocess_kernel<T, HDV><<<grid, 256, 0, s>>>(O, dO, D, acc, p.H, p.N, p.stride_b, p.stride_h,        \
                                                   p.stride_n, tiles, zero_slices, slice_elems);            \
    break;
  switch (p.d) {
    FA_PRE_CASE(16)
    FA_PRE_CASE(32)
    FA_PRE_CASE(64)
    FA_PRE_CASE(96)
    FA_PRE_CASE(128)
    FA_PRE_CASE(256)
    default:
      return cudaErrorInvalidValue;
  }
#undef FA_PRE_CASE
  return cudaGetLastError();
}

cudaError_t launch_preprocess(const fa_problem& p, const void* O, const void* dO, float* D, float* dq_accum,
                              cudaStream_t s) {
  if (p.dtype == FA_BF16)
    return launch_preprocess_t<__nv_bfloat16>(p, (const __nv_bfloat16*)O, (const __nv_bfloat16*)dO, D,
                                              dq_accum, s);
  return launch_preprocess_t<float>(p, (const float*)O, (const float*)dO, D, dq_accum, s);
}

// ----------------------------------------------------------------------------
// Convert: dQ = T(scale * dq_accum), undoing the unit-blocked layout without a
// trip through shared memory.  A "piece" is 16 columns of one query row: the
// row's 16 floats of one 2 KB unit, i.e. one float4 in each of the unit's 4
// column-group planes.  The 32 lanes of a warp take the 32 rows of one unit,
// so each of its four loads reads one whole 512-byte plane; a lane then writes
// its row's 16 columns (32 bytes in bf16) with one 256-bit store when the
// output is 32-byte aligned (two 128-bit stores otherwise).  Measured on the
// 1×32×8192×128 accumulator: 5.1 TB/s with the lanes of a warp spread over a
// row's column blocks (64-byte runs), 5.4 TB/s with a row per lane, 5.9 TB/s
// with the 256-bit store.  Each thread handles kPieces pieces and issues all
// their loads before its first store.
// ----------------------------------------------------------------------------
constexpr int kConvThreads = 256;
constexpr int kConvPieces = 2;

template <bool kWide>
__device__ __forceinline__ void store_piece(float* dst, const float4 (&v)[4], float scale) {
#pragma unroll
  for (int g = 0; g < 4; g += 2) {
    const float4 x = v[g], y = v[g + 1];
    if (kWide) {
      ptx::st_global_v8(dst + 4 * g, __float_as_uint(scale * x.x), __float_as_uint(scale * x.y),
                        __float_as_uint(scale * x.z), __float_as_uint(scale * x.w), __float_as_uint(scale * y.x),
                        __float_as_uint(scale * y.y), __float_as_uint(scale * y.z), __float_as_uint(scale * y.w));
    } else {
      reinterpret_cast<float4*>(dst)[g] = make_float4(scale * x.x, scale * x.y, scale * x.z, scale * x.w);
      reinterpret_cast<float4*>(dst)[g + 1] = make_float4(scale * y.x, scale * y.y, scale * y.z, scale * y.w);
    }
  }
}
template <bool kWide>
__device__ __forceinline__ void store_piece(__nv_bfloat16* dst, const float4 (&v)[4], float scale) {
  uint32_t w[8];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    w[2 * g] = ptx::pack_bf16x2(scale * v[g].x, scale * v[g].y);
    w[2 * g + 1] = ptx::pack_bf16x2(scale * v[g].z, scale * v[g].w);
  }
  if (kWide) {
    ptx::st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
  } else {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <typename T, int HD, bool kSlices, bool kWide>
__global__ void __launch_bounds__(kConvThreads) convert_dq_kernel(const float* __restrict__ acc, T* __restrict__ dQ,
                                                                  int H, int N, int64_t sb, int64_t sh, int64_t sn,
                                                                  int tiles_per_head, float scale, int slices,
                                                                  int64_t slice_elems, int causal, int kb_rows,
                                                                  int64_t offset, int64_t pieces) {
  constexpr int kCb = HD / 16;  // 16-column blocks (units) per row
  float4 v[kConvPieces][4];
  int64_t out_off[kConvPieces];
  bool live[kConvPieces];
#pragma unroll
  for (int j = 0; j < kConvPieces; ++j) {
    const int64_t gp = ((int64_t)blockIdx.x * kConvPieces + j) * kConvThreads + threadIdx.x;
    // piece gp is row gp % 32 of unit gp / 32 = (bt * 4 + rt / 32) * kCb + cb
    const int64_t unit = gp / 32;
    const int cb = (int)(unit % kCb);
    const int64_t ug = unit / kCb;
    const int rt = (int)(ug % 4) * 32 + (int)(gp % 32);  // row within the 128-row tile
    const int64_t bt = ug / 4;                            // bh * T + tile
    const int tile = (int)(bt % tiles_per_head);
    const int64_t bh = bt / tiles_per_head;
    const int n = tile * kTileRows + rt;
    live[j] = gp < pieces && n < N;
    const int b = (int)(bh / H), h = (int)(bh % H);
    out_off[j] = (int64_t)b * sb + (int64_t)h * sh + (int64_t)n * sn + cb * 16;
    // the row's float4 in plane g of its unit is at + g * 128 floats
    const float4* src = reinterpret_cast<const float4*>(acc + unit * 512 + (gp % 32) * 4);
    // Key blocks that touch this query tile: all, or (causal) those starting
    // at or before the last key its last row sees (row + offset); none when
    // that is negative.  Their slices are summed in increasing order.
    int last = kSlices ? slices - 1 : 0;
    if (kSlices && causal) {
      const int64_t hi = (int64_t)tile * kTileRows + kTileRows - 1 + offset;
      last = hi < 0 ? -1 : (hi / kb_rows < last ? (int)(hi / kb_rows) : last);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) v[j][g] = live[j] && last >= 0 ? __ldg(src + g * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (kSlices && live[j]) {
      const int64_t slice4 = slice_elems / 4;
      for (int sl = 1; sl <= last; ++sl)
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float4 w = __ldg(src + sl * slice4 + g * 32);
          v[j][g].x += w.x;
          v[j][g].y += w.y;
          v[j][g].z += w.z;
          v[j][g].w += w.w;
        }
    }
  }
#pragma unroll
  for (int j = 0; j < kConvPieces; ++j)
    if (live[j]) store_piece<kWide>(dQ + out_off[j], v[j], scale);
}

template <typename T>
static cudaError_t launch_convert_t(const fa_problem& p, const float* acc, T* dQ, cudaStream_t s) {
  const int tiles = (int)ceil_div(p.N, kTileRows);
  const int64_t pieces = (int64_t)p.B * p.H * tiles * kTileRows * (p.d / 16);
  const dim3 grid((unsigned)ceil_div(pieces, kConvThreads * kConvPieces));
  // a piece's 16 columns start 32-byte aligned when the base and every stride are
  const int64_t es = (int64_t)sizeof(T);
  const bool wide = (uintptr_t)dQ % 32 == 0 && (p.stride_b * es) % 32 == 0 && (p.stride_h * es) % 32 == 0 &&
                    (p.stride_n * es) % 32 == 0;
#define FA_CONV_CASE(HDV)                                                                                  \
  case HDV: {                                                                                              \
    auto kern = deterministic(p) ? (wide ? convert_dq_kernel<T, HDV, true, true>                           \
                                         : convert_dq_kernel<T, HDV, true, false>)                         \
                                 : (wide ? convert_dq_kernel<T, HDV, false, true>                          \
                                         : convert_dq_kernel<T, HDV, false, false>);                       \
    kern<<<grid, kConvThreads, 0, s>>>(acc, dQ, p.H, p.N, p.stride_b, p.stride_h, p.stride_n, tiles,       \
                                       p.scale, (int)dq_slices(p), dq_slice_elems(p), p.causal,            \
                                       key_block_rows(p), causal_offset(p), pieces);                       \
    break;                                                                                                 \
  }
  switch (p.d) {
    FA_CONV_CASE(16)
    FA_CONV_CASE(32)
    FA_CONV_CASE(64)
    FA_CONV_CASE(96)
    FA_CONV_CASE(128)
    FA_CONV_CASE(256)
    default:
      return cudaErrorInvalidValue;
  }
#undef FA_CONV_CASE
  return cudaGetLastError();
}

cudaError_t launch_convert_dq(const fa_problem& p, const float* acc, void* dQ, cudaStream_t s) {
  if (p.dtype == FA_BF16) return launch_convert_t<__nv_bfloat16>(p, acc, (__nv_bfloat16*)dQ, s);
  return launch_convert_t<float>(p, acc, (float*)dQ, s);
}

// ----------------------------------------------------------------------------
// Failure-detection self test: one warp waits on an mbarrier that nothing
// arrives at, with the bounded wait used by the tensor-core kernels.
// ----------------------------------------------------------------------------
__global__ void selftest_wait_kernel(int32_t* status, uint64_t wait_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bar), 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  ptx::Waiter w{&abort_flag, status, wait_ns};
  // phase 0 never completes: nobody arrives
  (void)ptx::wait_bounded(ptx::smem_addr(&bar), 0, w, true);
  __syncthreads();
}

cudaError_t launch_selftest_wait(int32_t* status, uint64_t wait_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, wait_ns);
  return cudaGetLastError();
}

}  // namespace fa

// ============================================================================
// Public C ABI
// ============================================================================
namespace {

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status validate_normalized(const fa_problem* p) {
  if (p->B < 1 || p->H < 1 || p->N < 1 || p->N_k < 1 || p->d < 1) return FA_ERR_INVALID_ARG;
  if (p->reserved != 0) return FA_ERR_INVALID_ARG;
  if (p->flags & ~(int32_t)FA_FLAG_DETERMINISTIC) return FA_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return FA_ERR_INVALID_ARG;
  if (!(p->scale == p->scale) || p->scale <= 0.f || p->scale > 1e30f) return FA_ERR_INVALID_ARG;
  if (p->dtype != FA_BF16 && p->dtype != FA_FP32) return FA_ERR_INVALID_ARG;
  if (p->N > (1 << 24) || p->N_k > (1 << 24) || (int64_t)p->B * p->H > (1 << 24)) return FA_ERR_UNSUPPORTED;
  // every kernel launches a 1-D grid of at most B * H * ceil(rows / 32) * 2 CTAs
  const int64_t rows = p->N > p->N_k ? p->N : p->N_k;
  if ((int64_t)p->B * p->H * ((rows + 31) / 32) * 2 > INT32_MAX) return FA_ERR_UNSUPPORTED;
  const int64_t es = p->dtype == FA_BF16 ? 2 : 4;
  if (p->stride_n < p->d || p->stride_h < 1 || p->stride_b < 1) return FA_ERR_INVALID_ARG;
  if ((p->stride_n * es) % 16 || (p->stride_h * es) % 16 || (p->stride_b * es) % 16) return FA_ERR_INVALID_ARG;
  if (p->kstride_n < p->d || p->kstride_h < 1 || p->kstride_b < 1) return FA_ERR_INVALID_ARG;
  if ((p->kstride_n * es) % 16 || (p->kstride_h * es) % 16 || (p->kstride_b * es) % 16) return FA_ERR_INVALID_ARG;
  if (p->dtype == FA_BF16) {
    if (p->d != 32 && p->d != 64 && p->d != 96 && p->d != 128 && p->d != 256) return FA_ERR_UNSUPPORTED;
  } else {
    if (p->d != 16 && p->d != 32 && p->d != 64 && p->d != 96 && p->d != 128 && p->d != 256)
      return FA_ERR_UNSUPPORTED;
  }
  return FA_OK;
}

// Validates *in and writes its normalised form (N_k = 0: self-attention,
// N_k = N with the Q strides) to *out.
fa_status normalize(const fa_problem* in, fa_problem* out) {
  if (!in) return FA_ERR_INVALID_ARG;
  if (in->N_k < 0) return FA_ERR_INVALID_ARG;
  *out = *in;
  if (in->N_k == 0) {
    out->N_k = in->N;
    out->kstride_b = in->stride_b;
    out->kstride_h = in->stride_h;
    out->kstride_n = in->stride_n;
  }
  return validate_normalized(out);
}

fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace

namespace fa {
bool normalize_problem(const fa_problem* in, fa_problem* out) { return normalize(in, out) == FA_OK; }
}  // namespace fa

extern "C" {

size_t fa_dq_accum_elems(const fa_problem* p) {
  fa_problem pn;
  if (normalize(p, &pn) != FA_OK) return 0;
  return (size_t)(fa::dq_slices(pn) * fa::dq_slice_elems(pn));
}

fa_status fa_fwd(const fa_problem* p, const void* Q, const void* K, const void* V, void* O, float* L,
                 void* stream) {
  fa::NvtxRange range("fa_fwd");
  fa_problem pn;
  fa_status st = normalize(p, &pn);
  if (st != FA_OK) return st;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(L)) return FA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (!fa::tensor_core(pn)) return from_cuda(fa::launch_fwd_simt(pn, Q, K, V, O, L, s));
  int32_t* status = fa::device_status_word();
  if (!status) return FA_ERR_CUDA;
  return from_cuda(fa::launch_fwd_sm103(pn, Q, K, V, O, L, status, fa::wait_limit_ns(), s));
}

fa_status fa_bwd_preprocess(const fa_problem* p, const void* O, const void* dO, float* D, float* dQ_accum,
                            void* stream) {
  fa::NvtxRange range("fa_bwd_preprocess");
  fa_problem pn;
  fa_status st = normalize(p, &pn);
  if (st != FA_OK) return st;
  if (!aligned16(O) || !aligned16(dO) || !aligned16(D) || !aligned16(dQ_accum)) return FA_ERR_INVALID_ARG;
  return from_cuda(fa::launch_preprocess(pn, O, dO, D, dQ_accum, (cudaStream_t)stream));
}

fa_status fa_bwd(const fa_problem* p, const void* Q, const void* K, const void* V, const void* dO, const float* L,
                 const float* D, float* dQ_accum, void* dK, void* dV, void* stream) {
  fa::NvtxRange range("fa_bwd");
  fa_problem pn;
  fa_status st = normalize(p, &pn);
  if (st != FA_OK) return st;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dO) || !aligned16(L) || !aligned16(D) ||
      !aligned16(dQ_accum) || !aligned16(dK) || !aligned16(dV))
    return FA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (!fa::tensor_core(pn))
    return from_cuda(fa::launch_bwd_simt(pn, Q, K, V, dO, L, D, dQ_accum, dK, dV, s));
  int32_t* status = fa::device_status_word();
  if (!status) return FA_ERR_CUDA;
  if (pn.d == 256)
    return from_cuda(
        fa::launch_bwd_d256_sm103(pn, Q, K, V, dO, L, D, dQ_accum, dK, dV, status, fa::wait_limit_ns(), s));
  return from_cuda(fa::launch_bwd_sm103(pn, Q, K, V, dO, L, D, dQ_accum, dK, dV, status, fa::wait_limit_ns(), s));
}

fa_status fa_bwd_tile_pair_count(const fa_problem* p, const void* Q, const void* K, const void* V, const void* dO,
                                 const float* L, const float* D, float* dQ_accum, void* dK, void* dV,
                                 unsigned long long* counts, int32_t* key_rows, int32_t* query_rows, void* stream) {
  fa::NvtxRange range("fa_bwd_tile_pair_count");
  fa_problem pn;
  fa_status st = normalize(p, &pn);
  if (st != FA_OK) return st;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dO) || !aligned16(L) || !aligned16(D) ||
      !aligned16(dQ_accum) || !aligned16(dK) || !aligned16(dV) || !counts ||
      (reinterpret_cast<uintptr_t>(counts) & 7u) || !key_rows || !query_rows)
    return FA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (!fa::tensor_core(pn)) {
    *key_rows = *query_rows = fa::key_block_rows(pn);
    return from_cuda(fa::launch_bwd_simt(pn, Q, K, V, dO, L, D, dQ_accum, dK, dV, s, counts));
  }
  int32_t* status = fa::device_status_word();
  if (!status) return FA_ERR_CUDA;
  *key_rows = 128;
  if (pn.d == 256) {
    *query_rows = 64;
    return from_cuda(fa::launch_bwd_d256_sm103(pn, Q, K, V, dO, L, D, dQ_accum, dK, dV, status, fa::wait_limit_ns(),
                                               s, counts));
  }
  *query_rows = 128;
  return from_cuda(
      fa::launch_bwd_sm103_count(pn, Q, K, V, dO, L, D, dQ_accum, dK, dV, status, fa::wait_limit_ns(), s, counts));
}

fa_status fa_convert_dq(const fa_problem* p, const float* dQ_accum, void* dQ, void* stream) {
  fa::NvtxRange range("fa_convert_dq");
  fa_problem pn;
  fa_status st = normalize(p, &pn);
  if (st != FA_OK) return st;
  if (!aligned16(dQ_accum) || !aligned16(dQ)) return FA_ERR_INVALID_ARG;
  return from_cuda(fa::launch_convert_dq(pn, dQ_accum, dQ, (cudaStream_t)stream));
}

fa_status fa_backward(const fa_problem* p, const void* Q, const void* K, const void* V, const void* O,
                      const void* dO, const float* L, float* D, float* dQ_accum, void* dQ, void* dK, void* dV,
                      void* stream) {
  fa::NvtxRange range("fa_backward");
  fa_problem pn;
  fa_status st = normalize(p, &pn);
  if (st != FA_OK) return st;
  if (!aligned16(dQ)) return FA_ERR_INVALID_ARG;
  st = fa_bwd_preprocess(p, O, dO, D, dQ_accum, stream);
  if (st != FA_OK) return st;
  st = fa_bwd(p, Q, K, V, dO, L, D, dQ_accum, dK, dV, stream);
  if (st != FA_OK) return st;
  return fa_convert_dq(p, dQ_accum, dQ, stream);
}

size_t fa_backward_fused_sync_elems(const fa_problem* p) {
  fa_problem pn;
  if (normalize(p, &pn) != FA_OK || !fa::fused_supported(pn)) return 0;
  return 1 + 2 * (size_t)pn.B * pn.H;
}

fa_status fa_backward_fused(const fa_problem* p, const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* L, float* D, float* dQ_accum, int32_t* sync, void* dQ,
                            void* dK, void* dV, void* stream) {
  fa::NvtxRange range("fa_backward_fused");
  fa_problem pn;
  fa_status st = normalize(p, &pn);
  if (st != FA_OK) return st;
  if (!fa::fused_supported(pn)) return FA_ERR_UNSUPPORTED;
  if (fa::fused_items(pn) > 0x7fffffff) return FA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(L) ||
      !aligned16(D) || !aligned16(dQ_accum) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV) || !sync ||
      (reinterpret_cast<uintptr_t>(sync) & 3u))
    return FA_ERR_INVALID_ARG;
  int32_t* status = fa::device_status_word();
  if (!status) return FA_ERR_CUDA;
  return from_cuda(fa::launch_bwd_fused_sm103(pn, Q, K, V, O, dO, L, D, dQ_accum, sync, dQ, dK, dV, status,
                                              fa::wait_limit_ns(), (cudaStream_t)stream));
}

fa_status fa_get_device_status(void* stream, int32_t* code) {
  if (!code) return FA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FA_ERR_CUDA;
  int32_t* word = fa::device_status_word();
  if (!word) return FA_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  const int32_t zero = 0;
  if (cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  *code = v;
  return FA_OK;
}

void fa_set_wait_limit_ns(uint64_t ns) { fa::g_wait_ns.store(ns == 0 ? 1 : ns); }

fa_status fa_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  int32_t* status = fa::device_status_word();
  if (!status) return FA_ERR_CUDA;
  return from_cuda(fa::launch_selftest_wait(status, limit_ns, (cudaStream_t)stream));
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported problem";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device wait timed out";
    case FA_ERR_DEVICE: return "device self check failed";
  }
  return "unknown status";
}

int32_t fa_version(void) { return 100; }

}  // extern "C"
