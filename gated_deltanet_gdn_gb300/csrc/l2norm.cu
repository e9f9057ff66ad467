// Optional q/k L2 normalisation for the chunked path ("gated-deltanet" kernel card,
// sections Usage and Correctness: use_qk_l2norm): every (token, head) row of q and of
// k is divided by sqrt(sum of squares + 1e-6) before the rule sees it.
//
// The chunked forward normalises once, into the residual buffer (the normalised rows
// and their inverse norms), and every chunk kernel of the forward and the backward
// reads those rows in place of q and k. The backward's dq and dk are then taken back
// through the normalisation in place: with r the inverse norm and x-hat = r x,
// dx = r (dx-hat - x-hat <x-hat, dx-hat>). One warp per row; the norm is the shared
// warp_row_inv_norm, the same arithmetic the recurrent kernels use.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int NORM_THREADS = 256;

template <class T, int DK>
__global__ void __launch_bounds__(NORM_THREADS) l2norm_rows_kernel(const T* q, const T* k, T* qn, T* kn,
                                                                   float* qinv, float* kinv, size_t rows) {
  const int lane = threadIdx.x & 31;
  const size_t w = (size_t)blockIdx.x * (NORM_THREADS / 32) + (threadIdx.x >> 5);  // (row, tensor)
  const size_t row = w >> 1;
  if (row >= rows) return;
  const bool isk = (w & 1) != 0;
  const T* x = (isk ? k : q) + row * DK;
  T* y = (isk ? kn : qn) + row * DK;
  constexpr int V = DK / 32;  // consecutive elements per lane
  const float inv = warp_row_inv_norm<DK>(x, lane);
  float xv[V];
  load_vec<V>(x + V * lane, xv);
#pragma unroll
  for (int j = 0; j < V; j += 2) store2(y + V * lane + j, xv[j] * inv, xv[j + 1] * inv);
  if (lane == 0) (isk ? kinv : qinv)[row] = inv;
}

template <class T, int DK>
__global__ void __launch_bounds__(NORM_THREADS) l2norm_bwd_kernel(T* dq, T* dk, const T* qn, const T* kn,
                                                                  const float* qinv, const float* kinv,
                                                                  size_t rows) {
  const int lane = threadIdx.x & 31;
  const size_t w = (size_t)blockIdx.x * (NORM_THREADS / 32) + (threadIdx.x >> 5);
  const size_t row = w >> 1;
  if (row >= rows) return;
  const bool isk = (w & 1) != 0;
  T* dx = (isk ? dk : dq) + row * DK;
  const T* xh = (isk ? kn : qn) + row * DK;
  const float r = (isk ? kinv : qinv)[row];
  constexpr int V = DK / 32;  // consecutive elements per lane
  float g[V], xv[V], dot = 0.f;
  load_vec<V>(dx + V * lane, g);
  load_vec<V>(xh + V * lane, xv);
#pragma unroll
  for (int j = 0; j < V; ++j) dot = fmaf(xv[j], g[j], dot);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
#pragma unroll
  for (int j = 0; j < V; j += 2) store2(dx + V * lane + j, r * (g[j] - xv[j] * dot), r * (g[j + 1] - xv[j + 1] * dot));
}

template <class T, int DK>
cudaError_t rows_t(const void* q, const void* k, void* qn, void* kn, float* qinv, float* kinv, size_t rows,
                   cudaStream_t s) {
  const size_t blocks = (2 * rows + NORM_THREADS / 32 - 1) / (NORM_THREADS / 32);
  prof_mark(K_L2NORM, s, true);
  l2norm_rows_kernel<T, DK><<<(unsigned)blocks, NORM_THREADS, 0, s>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<T*>(qn), static_cast<T*>(kn), qinv, kinv, rows);
  prof_mark(K_L2NORM, s, false);
  return cudaGetLastError();
}

template <class T, int DK>
cudaError_t bwd_t(void* dq, void* dk, const void* qn, const void* kn, const float* qinv, const float* kinv,
                  size_t rows, cudaStream_t s) {
  const size_t blocks = (2 * rows + NORM_THREADS / 32 - 1) / (NORM_THREADS / 32);
  prof_mark(K_L2NORM_BWD, s, true);
  l2norm_bwd_kernel<T, DK><<<(unsigned)blocks, NORM_THREADS, 0, s>>>(
      static_cast<T*>(dq), static_cast<T*>(dk), static_cast<const T*>(qn), static_cast<const T*>(kn), qinv, kinv,
      rows);
  prof_mark(K_L2NORM_BWD, s, false);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_l2norm_rows(const void* q, const void* k, void* qn, void* kn, float* qinv, float* kinv,
                               size_t rows, int DK, int bf16_in, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (bf16_in) return DK == 64 ? rows_t<bf16, 64>(q, k, qn, kn, qinv, kinv, rows, s)
                               : rows_t<bf16, 128>(q, k, qn, kn, qinv, kinv, rows, s);
  return DK == 64 ? rows_t<float, 64>(q, k, qn, kn, qinv, kinv, rows, s)
                  : rows_t<float, 128>(q, k, qn, kn, qinv, kinv, rows, s);
}

cudaError_t launch_l2norm_bwd(void* dq, void* dk, const void* qn, const void* kn, const float* qinv,
                              const float* kinv, size_t rows, int DK, int bf16_in, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (bf16_in) return DK == 64 ? bwd_t<bf16, 64>(dq, dk, qn, kn, qinv, kinv, rows, s)
                               : bwd_t<bf16, 128>(dq, dk, qn, kn, qinv, kinv, rows, s);
  return DK == 64 ? bwd_t<float, 64>(dq, dk, qn, kn, qinv, kinv, rows, s)
                  : bwd_t<float, 128>(dq, dk, qn, kn, qinv, kinv, rows, s);
}

}  // namespace gdn
