// Layout of the fp32 dQ accumulator (documented in include/fa.h).
//
// Per (b, h) the query rows form tiles of 128 (the last one padded).  Inside
// a tile, rows split into 4 quarters of 32 and columns into blocks of 16;
// each (quarter, block) pair is one 2 KB unit laid out [4 column groups of 4]
// [32 rows][4 columns].  A unit is what one warp of the tensor-core backward
// stages in shared memory and hands to one bulk reduction.
#pragma once

#include <stdint.h>

namespace fa {

constexpr int kDqUnitFloats = 32 * 16;  // 2 KB

// Float offset of unit (quarter qq, column block cb) of query tile `tile`.
__host__ __device__ __forceinline__ int64_t dq_unit_offset(int64_t bh, int n_tiles, int tile, int qq, int cb,
                                                           int d) {
  return (((bh * n_tiles + tile) * 4 + qq) * (d / 16) + cb) * kDqUnitFloats;
}

// Float offset of element (query row n, column c) of head bh.
__host__ __device__ __forceinline__ int64_t dq_accum_index(int64_t bh, int n_tiles, int n, int c, int d) {
  const int r = n % 128;
  return dq_unit_offset(bh, n_tiles, n / 128, r / 32, c / 16, d) + ((c % 16) / 4) * 128 + (r % 32) * 4 + (c % 4);
}

}  // namespace fa
