// Pieces of the chunk preparation (A1 cumulative log-decay, A4 in-block pairwise scores)
// shared by the CUDA-core preparation kernel (chunk_fwd.cu) and the tensor-core one
// (chunk_prep_tc.cu).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

// (i, j) of pair p in the lower triangle (diagonal included), row-major order
__device__ __forceinline__ void tri_index(int p, int& i, int& j) {
  int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
  while (r * (r + 1) / 2 > p) --r;
  while ((r + 1) * (r + 2) / 2 <= p) ++r;
  i = r;
  j = p - r * (r + 1) / 2;
}

// In-block pairwise scores (A4) for the blocks flagged unsafe: 4 lanes per (i, j) pair,
// each summing a quarter of the channels, reduced with two xor shuffles. Writes
// scale * sum q k E into the Aqk staging tile and beta_i * sum k k E (i > j) into Akk
// (at [i][j], or at [j][i] when AKK_T: the tensor-core preparation keeps Akk transposed).
template <class T, int DK, int NTHR, bool AKK_T = false>
__device__ __noinline__ void prep_pairwise(bool unsafe1, bool unsafe2, const T* q, const T* k, size_t row0,
                                           size_t rs, FTile<C, DK> Gs, Tile<T, C, C> Tst, FTile<C, C, 4> Akk,
                                           const float* beta_s, float scale, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  for (int blk = 0; blk < 2; ++blk) {
    if (!(blk == 0 ? unsafe1 : unsafe2)) continue;
    const int bs = blk * BLK;
    constexpr int NPAIR = BLK * (BLK + 1) / 2;
    for (int base = 0; base < NPAIR; base += 8 * (NTHR / 32)) {
      const int p = base + warp * 8 + (lane >> 2), quarter = lane & 3;
      const bool valid = p < NPAIR;
      int i = 0, j = 0;
      float sq = 0.f, sk = 0.f;
      if (valid) {
        tri_index(p, i, j);
        const T* qi = q + (row0 + (size_t)(bs + i) * rs) * DK;
        const T* ki = k + (row0 + (size_t)(bs + i) * rs) * DK;
        const T* kj = k + (row0 + (size_t)(bs + j) * rs) * DK;
        for (int c = quarter * (DK / 4); c < (quarter + 1) * (DK / 4); ++c) {
          const float e = __expf(Gs.at(bs + i, c) - Gs.at(bs + j, c));
          const float kje = to_f32(kj[c]) * e;
          sq = fmaf(to_f32(qi[c]), kje, sq);
          sk = fmaf(to_f32(ki[c]), kje, sk);
        }
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sk += __shfl_xor_sync(0xffffffffu, sk, 1);
      sq += __shfl_xor_sync(0xffffffffu, sq, 2);
      sk += __shfl_xor_sync(0xffffffffu, sk, 2);
      if (valid && quarter == 0) {
        Tst.at(bs + i, bs + j) = from_f32<T>(scale * sq);
        if (i > j) {
          if (AKK_T) Akk.at(bs + j, bs + i) = beta_s[bs + i] * sk;
          else Akk.at(bs + i, bs + j) = beta_s[bs + i] * sk;
        }
      }
    }
  }
}

// A1: inclusive cumulative log-decay per channel in fp32, G[r][c] = sum_{s<=r} g[s][c]:
// lanes 2c and 2c + 1 take channel c, one 32-row block each in registers; the second
// block adds the first block's total (from its partner lane). graw: the chunk's raw
// per-channel g [C][DK] (row-major), gsc: one decay per token (PC false).
template <class T, int DK, int NTHR, bool PC>
__device__ __forceinline__ void prep_cumsum(FTile<C, DK> Gs, const T* graw, const float* gsc, int tid) {
  static_assert((2 * DK) % 32 == 0, "whole warps per pass");
  const int lane = tid & 31;
  for (int u = tid; u < 2 * DK; u += NTHR) {
    const int c = u >> 1, hb = u & 1, r0 = hb * BLK;
    float v[BLK];
#pragma unroll
    for (int i = 0; i < BLK; ++i) v[i] = PC ? to_f32(graw[(r0 + i) * DK + c]) : gsc[r0 + i];
#pragma unroll
    for (int i = 1; i < BLK; ++i) v[i] += v[i - 1];
    const float base = __shfl_sync(0xffffffffu, v[BLK - 1], lane & ~1);
#pragma unroll
    for (int i = 0; i < BLK; ++i) Gs.at(r0 + i, c) = hb ? v[i] + base : v[i];
  }
}

}  // namespace
}  // namespace gdn
