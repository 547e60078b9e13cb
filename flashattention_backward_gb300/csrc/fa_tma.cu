// TMA tensor maps for the tensor-core kernels.  cuTensorMapEncodeTiled is a
// driver entry point, resolved once at run time through the runtime so that
// the library itself does not link libcuda.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

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

}  // namespace

bool make_bf16_tile_map_rows(CUtensorMap* m, const void* base, const fa_problem& p, bool kv, int box_rows) {
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

bool make_bf16_tile_map(CUtensorMap* m, const void* base, const fa_problem& p, bool kv) {
  return make_bf16_tile_map_rows(m, base, p, kv, kTileRows);
}

}  // namespace fa
