// D_i = sum_c O_ic * dO_ic for one row (CUDA 算子工程 ch.16 §16.1 identity,
// §16.8 item 1), computed the same way by the preprocess kernel and by the
// single-launch backward so that both give bitwise the same D: a row is read
// as 16-byte vectors, lane `sub` of the kLanes lanes that share the row takes
// vectors sub, sub + kLanes, ... in order, and the lanes then reduce with an
// XOR shuffle tree.  Products and sums are written out with explicit fmaf so
// that no contraction choice of the compiler changes the rounding.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace fa {

template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int kElems = 4;
  __device__ static __forceinline__ float dot(const uint4& a, const uint4& b) {
    float s = __uint_as_float(a.x) * __uint_as_float(b.x);
    s = fmaf(__uint_as_float(a.y), __uint_as_float(b.y), s);
    s = fmaf(__uint_as_float(a.z), __uint_as_float(b.z), s);
    return fmaf(__uint_as_float(a.w), __uint_as_float(b.w), s);
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ static __forceinline__ float dot2(uint32_t a, uint32_t b, float s) {
    s = fmaf(__uint_as_float(a << 16), __uint_as_float(b << 16), s);
    return fmaf(__uint_as_float(a & 0xffff0000u), __uint_as_float(b & 0xffff0000u), s);
  }
  __device__ static __forceinline__ float dot(const uint4& a, const uint4& b) {
    return dot2(a.w, b.w, dot2(a.z, b.z, dot2(a.y, b.y, dot2(a.x, b.x, 0.f))));
  }
};

template <typename T, int HD>
struct RowDot {
  static constexpr int kVecs = HD / Vec16<T>::kElems;  // 16-byte vectors per row: 2 .. 64
  // lanes per row: a power of two (lanes past kVecs idle), at most 32
  static constexpr int kLanes = kVecs <= 2 ? 2 : kVecs <= 4 ? 4 : kVecs <= 8 ? 8 : kVecs <= 16 ? 16 : 32;
  static constexpr int kPerLane = (kVecs + kLanes - 1) / kLanes;
  // this lane's part of the row (o, g point at the row's first element)
  __device__ static __forceinline__ float partial(const T* o, const T* g, int sub) {
    float acc = 0.f;
#pragma unroll
    for (int v = 0; v < kPerLane; ++v) {
      const int vec = sub + v * kLanes;
      if (vec < kVecs) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(o) + vec);
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(g) + vec);
        acc += Vec16<T>::dot(a, b);
      }
    }
    return acc;
  }
  // sum over the kLanes lanes of a row (aligned groups of kLanes lanes)
  __device__ static __forceinline__ float reduce(float acc) {
#pragma unroll
    for (int m = kLanes / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    return acc;
  }
};

}  // namespace fa
