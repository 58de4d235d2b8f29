// tmap.h -- host-side construction of the TMA tensor maps the attention
// kernels use, and device helpers shared by the forward and backward kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "internal.h"
#include "sm100.cuh"

namespace ulysses {

// 4-D map over a head-sharded activation [P*B][S][heads][D] (bf16): dims
// innermost first {D, heads, S, P*B}; a box is 64 elements of D (one
// 128-byte swizzle row) x 1 head x `box_rows` positions x 1.  Rows past S
// read as zero, so a tile never reads into the next batch or rank.
inline bool make_act_map(const TmaEncoder &enc, CUtensorMap *m, const void *base, int D, int heads,
                         int S, int PB, int box_rows) {
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)S, (cuuint64_t)PB};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2,
                                 (cuuint64_t)S * heads * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc.encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 2-D map over a row-major bf16 matrix [rows][cols] (cols contiguous): a box
// is 64 columns (one 128-byte swizzle row) x `box_rows` rows; rows past the
// end read as zero.
inline bool make_mat_map(const TmaEncoder &enc, CUtensorMap *m, const void *base, long long cols, long long rows,
                         int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc.encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over a float array of `rows` rows of S values, `ld` floats apart
// (ld >= S, a multiple of 4): box of `box` positions of one row; positions
// past S read as zero.
inline bool make_row_map(const TmaEncoder &enc, CUtensorMap *m, const void *base, int S, int ld, int rows,
                         int box) {
  const cuuint64_t dims[2] = {(cuuint64_t)S, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  const cuuint32_t boxd[2] = {(cuuint32_t)box, 1};
  const cuuint32_t estr[2] = {1, 1};
  return enc.encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides,
                    boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

namespace dev {

// A bounded wait whose outcome is the same for every lane of the warp (the
// tcgen05.ld/st that follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          const volatile uint32_t *gst) {
  const bool ok = sm100::mbar_wait_bounded(bar, parity, abort_flag, gst);
  return __all_sync(0xffffffffu, ok);
}

// CTA order over n_heads heads x n_tiles tiles: heads in consecutive groups of
// `group_heads`, and within a group the tiles by rank (rank 0, the longest,
// first), the group's heads interleaved.  A group's K/V (or Q/dO) tiles then
// stay in L2 while its CTAs run, instead of every head's streaming through at
// once; longest-first keeps the tail short.
struct HeadTile {
  int head, rank;
};
__device__ __forceinline__ HeadTile grouped_order(int b, int n_heads, int n_tiles, int group_heads) {
  const int g = b / (group_heads * n_tiles);
  const int hg = min(group_heads, n_heads - g * group_heads);
  const int r = b - g * group_heads * n_tiles;
  return {g * group_heads + r % hg, r / hg};
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

}  // namespace dev
}  // namespace ulysses
