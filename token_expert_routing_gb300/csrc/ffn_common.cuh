// Row-group -> tile mapping shared by the grouped-FFN kernels.
#pragma once

#include "common.cuh"

namespace semmoe {

struct GroupTile {
  int group;   // physical bucket, -1 = tile past the last one
  int expert;  // expert of that bucket
  int row0;    // first row of the tile
  int rows;    // valid rows in the tile (<= BM)
};

// Block-cooperative (every thread must call; n_groups <= blockDim.x):
// m-tile `tile` of the concatenation of ceil(rows_g / BM) tiles per group g,
// groups in physical order, rows [offsets[g], offsets[g+1]).  offsets == nullptr
// means one group of rows [0, P) on expert 0.  scan[] needs blockDim.x ints.
// Returns the result to every thread.  Bad offsets/experts set `err_bits`.
__device__ inline GroupTile group_tile_block(const int32_t* __restrict__ offsets,
                                             const int32_t* __restrict__ phys_to_expert, int n_groups,
                                             int P, int E, int BM, int tile, int* scan, GroupTile* out,
                                             int* err_bits) {
  const int g = threadIdx.x;
  int lo = 0, hi = 0;
  if (g < n_groups) {
    if (offsets != nullptr) {
      lo = offsets[g];
      hi = offsets[g + 1];
      if (lo < 0 || hi < lo || hi > P) { atomicOr(err_bits, SEMMOE_DEVERR_PAIRS); lo = hi = 0; }
    } else {
      lo = 0;
      hi = P;
    }
  }
  const int mine = (hi - lo + BM - 1) / BM;
  scan[threadIdx.x] = mine;
  if (threadIdx.x == 0) *out = GroupTile{-1, 0, 0, 0};
  __syncthreads();
  for (int d = 1; d < (int)blockDim.x; d <<= 1) {  // inclusive Hillis-Steele scan
    int v = threadIdx.x >= (unsigned)d ? scan[threadIdx.x - d] : 0;
    __syncthreads();
    scan[threadIdx.x] += v;
    __syncthreads();
  }
  const int incl = scan[threadIdx.x], excl = incl - mine;
  if (g < n_groups && tile >= excl && tile < incl) {
    int e = phys_to_expert != nullptr ? phys_to_expert[g] : 0;
    if (e < 0 || e >= E) {
      atomicOr(err_bits, SEMMOE_DEVERR_EXPERT);
    } else {
      int row0 = lo + (tile - excl) * BM;
      int rows = hi - row0 < BM ? hi - row0 : BM;
      *out = GroupTile{g, e, row0, rows};
    }
  }
  __syncthreads();
  return *out;
}

}  // namespace semmoe
