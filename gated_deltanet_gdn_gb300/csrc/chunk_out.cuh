// Chunk outputs of the chunked forward, O = (scale Q-hat) S0 + (scale Aqk) U, for one
// 64-token chunk and head from the records the preparation and the forward scan stored
// (chunked WY form; see the header of chunk_fwd.cu). Used by chunk_out_kernel
// (chunk_fwd.cu) and by the output CTAs that run beside the tensor-core forward scan
// (chunk_scan_tc.cu).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int OUT_THREADS = 256;

template <class T, int DK, int DV>
struct OutLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int QH = 0;                         // [C][DK]
  static constexpr int AQ = a1k(QH + C * DK * ES);     // [C][C]
  static constexpr int S0 = a1k(AQ + C * C * ES);      // S0^T [DV][DK]
  static constexpr int U = a1k(S0 + DK * DV * ES);     // U^T [DV][C], then the output tile
  static constexpr int BYTES = a1k(U + C * DV * ES);
};

// The products and the store of one chunk's outputs from its four record tiles already in
// shared memory at sm (OutLayout). Threads 0..OUT_THREADS-1 call it; sync() is a barrier
// over exactly them. Ends after a sync(): the tiles may be refilled right after.
template <class T, int DK, int DV, class Sync>
__device__ __forceinline__ void out_compute_store(const ChunkFwdArgs& a, int n, int bh, uint8_t* sm, int tid,
                                                  Sync sync) {
  typedef OutLayout<T, DK, DV> L;
  const int lane = tid & 31, warp = tid >> 5;
  const int b = bh / a.H, h = bh % a.H;
  constexpr int EPC = 16 / (int)sizeof(T);
  Tile<T, C, DK> Qs{reinterpret_cast<T*>(sm + L::QH)};
  Tile<T, C, C> As{reinterpret_cast<T*>(sm + L::AQ)};
  Tile<T, DV, DK> S0s{reinterpret_cast<T*>(sm + L::S0)};
  Tile<T, DV, C> Us{reinterpret_cast<T*>(sm + L::U)};
  const int m0 = 16 * (warp & 3), n0 = (warp >> 2) * (DV / 2);
  constexpr int NW = DV / 16;
  float o[1][NW][4];
  zero(o);
  Gemm<T>::template runk<1, NW, 0, DK>(o, aview<false>(Qs), bview<false>(S0s), m0, n0, lane);
  Gemm<T>::template runk<1, NW, 0, C>(o, aview<false>(As), bview<false>(Us), m0, n0, lane);
  sync();  // U consumed: stage the output tile in its place
  Tile<T, C, DV> Os{reinterpret_cast<T*>(sm + L::U)};
#pragma unroll
  for (int nt = 0; nt < NW; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      Os.at(m0 + frag_row(lane, e), n0 + 8 * nt + frag_col(lane, e)) = from_f32<T>(o[0][nt][e]);
  fence_proxy_async();  // the tile may next be refilled by bulk copies (async proxy)
  sync();
  T* out = static_cast<T*>(a.out);
  const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
  for (int i = tid; i < C * DV / EPC; i += OUT_THREADS) {
    const int r = i / (DV / EPC), c0 = (i % (DV / EPC)) * EPC;
    copy16(out + (row0 + (size_t)r * a.H) * DV + c0, Os.ptr(r, c0));
  }
  sync();
}

// One chunk's outputs by a CTA of OUT_THREADS threads: the records by cp.async, then
// out_compute_store. sm: 1024-byte aligned shared memory of at least OutLayout::BYTES.
template <class T, int DK, int DV>
__device__ __forceinline__ void out_unit(const ChunkFwdArgs& a, int n, int bh, uint8_t* sm, int tid) {
  typedef OutLayout<T, DK, DV> L;
  const int N = a.T / C;
  const size_t ch = (size_t)bh * N + n;
  constexpr int EPC = 16 / (int)sizeof(T);
  {
    const T* s1 = static_cast<const T*>(a.res.qh) + ch * (C * DK);
    for (int i = tid; i < C * DK / EPC; i += OUT_THREADS) cp_async16(reinterpret_cast<T*>(sm + L::QH) + i * EPC, s1 + i * EPC);
    const T* s2 = static_cast<const T*>(a.res.aqk) + ch * (C * C);
    for (int i = tid; i < C * C / EPC; i += OUT_THREADS) cp_async16(reinterpret_cast<T*>(sm + L::AQ) + i * EPC, s2 + i * EPC);
    const T* s3 = static_cast<const T*>(a.res.state) + ch * (DK * DV);
    for (int i = tid; i < DK * DV / EPC; i += OUT_THREADS) cp_async16(reinterpret_cast<T*>(sm + L::S0) + i * EPC, s3 + i * EPC);
    const T* s4 = static_cast<const T*>(a.res.u) + ch * (C * DV);
    for (int i = tid; i < C * DV / EPC; i += OUT_THREADS) cp_async16(reinterpret_cast<T*>(sm + L::U) + i * EPC, s4 + i * EPC);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  out_compute_store<T, DK, DV>(a, n, bh, sm, tid, [] { __syncthreads(); });
}

}  // namespace
}  // namespace gdn
