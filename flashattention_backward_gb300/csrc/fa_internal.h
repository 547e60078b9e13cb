// Internal declarations shared by the translation units of libfa.
// Nothing here is part of the public ABI (include/fa.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

// NVTX range around a public entry point, so that Nsight Systems and
// Nsight Compute timelines show each fa_* call; without a tool attached a
// push/pop pair costs a few nanoseconds.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Query/key tile height used by the dQ accumulator layout and by the
// tensor-core kernels.
constexpr int kTileRows = 128;

// Device status word codes are the fa_status values.
struct DeviceStatus {
  int32_t* word;  // device address of this device's status word
};

// Resolved once per device by the API layer.
int32_t* device_status_word();

// Wait limit (ns) used by every bounded wait in device code.
uint64_t wait_limit_ns();

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
// floor(a / b) for b > 0 and any sign of a
inline int64_t floor_div(int64_t a, int64_t b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Every launcher below takes a problem normalised by the API layer: N_k > 0
// and the kstride fields set (N_k = 0 in a caller's fa_problem means N_k = N
// with the Q strides).  Causal offset: key j is visible to query i iff
// j <= i + causal_offset(p).
bool normalize_problem(const fa_problem* in, fa_problem* out);  // false: invalid or unsupported
inline int64_t causal_offset(const fa_problem& p) { return (int64_t)p.N_k - p.N; }

inline bool deterministic(const fa_problem& p) { return (p.flags & FA_FLAG_DETERMINISTIC) != 0; }
// bf16 runs on the tensor-core kernels (at d = 256 the backward splits each
// key block over two CTAs, one per half of the output columns); fp32 on the
// CUDA-core kernels.  The single-launch backward exists for d <= 128.
inline bool tensor_core(const fa_problem& p) { return p.dtype == FA_BF16; }
inline bool fused_supported(const fa_problem& p) { return p.dtype == FA_BF16 && p.d <= 128; }
// Key-block height of the backward kernel that serves p (tensor-core
// kernels: 128; CUDA-core kernel: 64, or 32 at d = 256).
inline int key_block_rows(const fa_problem& p) { return tensor_core(p) ? 128 : (p.d == 256 ? 32 : 64); }
// dQ accumulator slices: one per key block in deterministic mode, else one.
inline int64_t dq_slices(const fa_problem& p) {
  return deterministic(p) ? ceil_div(p.N_k, key_block_rows(p)) : 1;
}
// Floats in one slice: B * H * ceil(N/128) * 128 * d.
inline int64_t dq_slice_elems(const fa_problem& p) {
  return (int64_t)p.B * p.H * ceil_div(p.N, 128) * 128 * p.d;
}

// A Q-shaped [B, H, N, d] (kv = false) or K-shaped [B, H, N_k, d] (kv = true)
// bf16 tensor of p as a 4-D TMA map: boxes of 64 columns x box_rows rows,
// 128-byte swizzle, rows past the end and columns past d read as zeros.
// False if the map cannot be encoded (or the driver entry point is missing).
bool make_bf16_tile_map_rows(CUtensorMap* m, const void* base, const fa_problem& p, bool kv, int box_rows);
// The same with 128-row boxes (the tiles of the head-dim <= 128 kernels).
bool make_bf16_tile_map(CUtensorMap* m, const void* base, const fa_problem& p, bool kv);

// ---- launchers (return a cudaError_t from the launch) -------------------
cudaError_t launch_preprocess(const fa_problem& p, const void* O, const void* dO, float* D,
                              float* dq_accum, cudaStream_t s);
cudaError_t launch_convert_dq(const fa_problem& p, const float* dq_accum, void* dQ, cudaStream_t s);
// CUDA-core forward and backward for fp32 problems (exact fp32 arithmetic).
cudaError_t launch_fwd_simt(const fa_problem& p, const void* Q, const void* K, const void* V,
                            void* O, float* L, cudaStream_t s);
// pair_count (optional, two device words): the backward kernels add the
// (key block, query block) pairs they execute to [0] and those among them
// with no visible entry to [1] (tile-pair accounting).
cudaError_t launch_bwd_simt(const fa_problem& p, const void* Q, const void* K, const void* V,
                            const void* dO, const float* L, const float* D, float* dq_accum,
                            void* dK, void* dV, cudaStream_t s, unsigned long long* pair_count = nullptr);
// tcgen05 / TMEM / TMA backward for bf16, d in {32, 64, 96, 128}.  Returns
// cudaErrorInvalidValue if a tensor map cannot be encoded.
cudaError_t launch_bwd_sm103(const fa_problem& p, const void* Q, const void* K, const void* V,
                             const void* dO, const float* L, const float* D, float* dq_accum,
                             void* dK, void* dV, int32_t* status, uint64_t wait_ns, cudaStream_t s);
// The same with tile-pair accounting into pair_count (instantiations of their
// own, built in fa_bwd_sm103_count.cu).
cudaError_t launch_bwd_sm103_count(const fa_problem& p, const void* Q, const void* K, const void* V,
                                   const void* dO, const float* L, const float* D, float* dq_accum,
                                   void* dK, void* dV, int32_t* status, uint64_t wait_ns, cudaStream_t s,
                                   unsigned long long* pair_count);
// tcgen05 / TMEM / TMA backward for bf16 at d = 256: two CTAs per key block,
// each accumulating dK and dV for 128 of the 256 columns.
cudaError_t launch_bwd_d256_sm103(const fa_problem& p, const void* Q, const void* K, const void* V,
                                  const void* dO, const float* L, const float* D, float* dq_accum,
                                  void* dK, void* dV, int32_t* status, uint64_t wait_ns, cudaStream_t s,
                                  unsigned long long* pair_count = nullptr);
// The whole backward (preprocess, tcgen05 backward, convert) in one launch
// of the tcgen05 kernel for bf16, d in {32, 64, 96, 128}; sync holds
// 1 + 2 B H int32 (zeroed by the launcher).
int64_t fused_items(const fa_problem& p);
cudaError_t launch_bwd_fused_sm103(const fa_problem& p, const void* Q, const void* K, const void* V, const void* O,
                                   const void* dO, const float* L, float* D, float* dq_accum, int32_t* sync,
                                   void* dQ, void* dK, void* dV, int32_t* status, uint64_t wait_ns, cudaStream_t s);
// tcgen05 forward for bf16, d in {32, 64, 96, 128, 256}.
cudaError_t launch_fwd_sm103(const fa_problem& p, const void* Q, const void* K, const void* V, void* O, float* L,
                             int32_t* status, uint64_t wait_ns, cudaStream_t s);
cudaError_t launch_selftest_wait(int32_t* status, uint64_t wait_ns, cudaStream_t s);

}  // namespace fa
