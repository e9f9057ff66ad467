// Chunk outputs of the chunked forward, O = (scale Q-hat) S0 + (scale Aqk) U, for 64 rows
// of one chunk (a 64-token chunk, or either block of a 128-token chunk) and head from the
// records the preparation and the forward scan stored (chunked WY form; see the header of
// chunk_fwd.cu). Used by chunk_out_kernel (chunk_fwd.cu) and by the output CTAs that run
// beside the tensor-core forward scan (chunk_scan_tc.cu).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int OUT_THREADS = 256;

// CC: chunk length (C, or C2 for 128-token chunks); the tile holds 64 rows of the chunk
template <class T, int DK, int DV, int CC = C>
struct OutLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int QH = 0;                         // [C][DK]: the rows' Q-hat
  static constexpr int AQ = a1k(QH + C * DK * ES);     // [C][CC]: the rows' Aqk
  static constexpr int S0 = a1k(AQ + C * CC * ES);     // S0^T [DV][DK]
  static constexpr int U = a1k(S0 + DK * DV * ES);     // U^T [DV][CC], then the output tile
  static constexpr int BYTES = a1k(U + CC * DV * ES);
};

// The products and the store of 64 output rows (rows C hh .. of chunk n) from the four
// record tiles already in shared memory at sm (OutLayout). Threads 0..OUT_THREADS-1 call
// it; sync() is a barrier over exactly them. Ends after a sync(): the tiles may be
// refilled right after.
template <class T, int DK, int DV, int CC = C, class Sync>
__device__ __forceinline__ void out_compute_store(const ChunkFwdArgs& a, int n, int bh, uint8_t* sm, int tid,
                                                  Sync sync, int hh = 0) {
  typedef OutLayout<T, DK, DV, CC> L;
  const int lane = tid & 31, warp = tid >> 5;
  const int b = bh / a.H, h = bh % a.H;
  constexpr int EPC = 16 / (int)sizeof(T);
  Tile<T, C, DK> Qs{reinterpret_cast<T*>(sm + L::QH)};
  Tile<T, C, CC> As{reinterpret_cast<T*>(sm + L::AQ)};
  Tile<T, DV, DK> S0s{reinterpret_cast<T*>(sm + L::S0)};
  Tile<T, DV, CC> Us{reinterpret_cast<T*>(sm + L::U)};
  const int m0 = 16 * (warp & 3), n0 = (warp >> 2) * (DV / 2);
  constexpr int NW = DV / 16;
  float o[1][NW][4];
  zero(o);
  Gemm<T>::template runk<1, NW, 0, DK>(o, aview<false>(Qs), bview<false>(S0s), m0, n0, lane);
  if (hh == 0)  // the first block's rows see only the first block's tokens
    Gemm<T>::template runk<1, NW, 0, C>(o, aview<false>(As), bview<false>(Us), m0, n0, lane);
  else
    Gemm<T>::template runk<1, NW, 0, CC>(o, aview<false>(As), bview<false>(Us), m0, n0, lane);
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
  const size_t row0 = ((size_t)b * a.T + (size_t)n * CC + (size_t)C * hh) * a.H + h;
  for (int i = tid; i < C * DV / EPC; i += OUT_THREADS) {
    const int r = i / (DV / EPC), c0 = (i % (DV / EPC)) * EPC;
    copy16(out + (row0 + (size_t)r * a.H) * DV + c0, Os.ptr(r, c0));
  }
  sync();
}

// Rows C hh .. C hh + C - 1 (unit x = chunk n * (CC / C) + hh) of one chunk's outputs by a
// CTA of OUT_THREADS threads: the records by cp.async, then out_compute_store. The Q-hat
// and Aqk records [CC][.] are panel-major images (Sw) whose rows C hh .. are one
// contiguous run per panel, with the swizzle of rows 0..C-1 (it depends on the row mod 8).
// sm: 1024-byte aligned shared memory of at least OutLayout::BYTES.
template <class T, int DK, int DV, int CC = C>
__device__ __forceinline__ void out_unit(const ChunkFwdArgs& a, const void* qh, const void* aqk, const void* state,
                                         const void* u, int x, int bh, uint8_t* sm, int tid) {
  typedef OutLayout<T, DK, DV, CC> L;
  const int N = a.T / CC, n = x / (CC / C), hh = x % (CC / C);
  const size_t ch = (size_t)bh * N + n;
  constexpr int EPC = 16 / (int)sizeof(T);
  {
    constexpr int PQ = Sw<T, CC, DK>::PW, PA = Sw<T, CC, CC>::PW;
    const T* s1 = static_cast<const T*>(qh) + ch * (CC * DK) + (size_t)C * hh * PQ;
    for (int i = tid; i < C * DK / EPC; i += OUT_THREADS) {
      const int e = i * EPC, p = e / (C * PQ);
      cp_async16(reinterpret_cast<T*>(sm + L::QH) + e, s1 + (size_t)p * (CC - C) * PQ + e);
    }
    const T* s2 = static_cast<const T*>(aqk) + ch * (CC * CC) + (size_t)C * hh * PA;
    for (int i = tid; i < C * CC / EPC; i += OUT_THREADS) {
      const int e = i * EPC, p = e / (C * PA);
      cp_async16(reinterpret_cast<T*>(sm + L::AQ) + e, s2 + (size_t)p * (CC - C) * PA + e);
    }
    const T* s3 = static_cast<const T*>(state) + ch * (DK * DV);
    for (int i = tid; i < DK * DV / EPC; i += OUT_THREADS) cp_async16(reinterpret_cast<T*>(sm + L::S0) + i * EPC, s3 + i * EPC);
    const T* s4 = static_cast<const T*>(u) + ch * (CC * DV);
    for (int i = tid; i < CC * DV / EPC; i += OUT_THREADS) cp_async16(reinterpret_cast<T*>(sm + L::U) + i * EPC, s4 + i * EPC);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  out_compute_store<T, DK, DV, CC>(a, n, bh, sm, tid, [] { __syncthreads(); }, hh);
}

}  // namespace
}  // namespace gdn
