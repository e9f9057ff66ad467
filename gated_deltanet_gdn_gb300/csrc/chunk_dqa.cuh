// The chunk products of the backward that need only forward records and dO:
//   dQ-hat = scale dO S0^T  and  dAqk = scale (dO U^T) masked j <= t
// (chunked WY backward, see chunk_bwd.cu), as a kernel of their own after the CUDA-core
// reverse scan (Dk = 64, or fp32 operands; with bf16 at Dk = Dv = 128 the fused
// tensor-core kernel of chunk_bwd_tc.cu computes them with the other chunk products).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int DQA_THREADS = 256;
constexpr int DQA_CG = DQA_THREADS / 128;  // column groups (4 row groups of warps each)

// The DQA_THREADS threads of the kernel synchronise on named barrier 2.
__device__ __forceinline__ void dqa_sync() { asm volatile("bar.sync 2, 256;\n" ::: "memory"); }

template <class T, int DK, int DV>
struct DqaLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int DO = 0;                        // dO    [C][DV]
  static constexpr int U = a1k(DO + C * DV * ES);     // U^T   [DV][C]
  static constexpr int S0 = a1k(U + C * DV * ES);     // S0^T  [DV][DK], as 64-channel panels
  static constexpr int BYTES = a1k(S0 + DV * DK * ES);
};

// Chunk-heads unit0, unit0 + stride, ... Called by threads 0 .. DQA_THREADS - 1 of a CTA;
// sm is its 1024-byte aligned shared memory.
template <class T, int DK, int DV>
__device__ __forceinline__ void dqa_units(const ChunkBwdArgs& a, uint8_t* sm, int unit0, int stride, int tid) {
  typedef DqaLayout<T, DK, DV> L;
  constexpr int NPAN = DK / 64;
  constexpr int EPC = 16 / (int)sizeof(T);
  const int lane = tid & 31, warp = tid >> 5;
  const int N = a.T / C, units = N * a.B * a.H;
#pragma unroll 1
  for (int unit = unit0; unit < units; unit += stride) {
    const int n = unit % N, bh = unit / N, b = bh / a.H, h = bh % a.H;
    const size_t ch = (size_t)bh * N + n;
    Tile<T, C, DV> dOs{reinterpret_cast<T*>(sm + L::DO)};
    Tile<T, DV, C> Us{reinterpret_cast<T*>(sm + L::U)};  // U^T
    const T* dout = static_cast<const T*>(a.dout);
    const T* s0rec = static_cast<const T*>(a.res.state) + ch * (DK * DV);
    const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
    const size_t rs = a.H;
    {  // group 0: dO and U^T (dAqk); group 1: the S0^T record (dQ-hat)
      const T* su = static_cast<const T*>(a.res.u) + ch * (C * DV);
      for (int i = tid; i < C * DV / EPC; i += DQA_THREADS) {
        const int r = i / (DV / EPC), c0 = (i % (DV / EPC)) * EPC;
        cp_async16(Us.p + i * EPC, su + i * EPC);
        cp_async16(dOs.ptr(r, c0), dout + (row0 + r * rs) * DV + c0);
      }
      cp_async_commit();
      T* s0 = reinterpret_cast<T*>(sm + L::S0);
      for (int i = tid; i < DV * DK / EPC; i += DQA_THREADS) cp_async16(s0 + i * EPC, s0rec + i * EPC);
      cp_async_commit();
    }
    cp_async_wait<1>();
    dqa_sync();
    // warp w: rows 16 (w % 4) .. + 15 and column group w / 4 of every product
    const int m0 = 16 * (warp & 3), hf = warp >> 2;
    {
      constexpr int NCC = C / (8 * DQA_CG);
      const int c0 = hf * (C / DQA_CG);
      float aq[1][NCC][4];
      zero(aq);
      if (!(m0 < BLK && c0 >= BLK))  // block-1 rows see no block-2 columns
        Gemm<T>::template runk<1, NCC, 0, DV>(aq, aview<false>(dOs), bview<true>(Us), m0, c0, lane);
      T* da = static_cast<T*>(a.ws.daqk) + ch * (C * C);
#pragma unroll
      for (int nt = 0; nt < NCC; ++nt)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int r = m0 + frag_row(lane, e), j = c0 + 8 * nt + frag_col(lane, e);
          store2(da + Sw<T, C, C>::off(r, j), j <= r ? a.scale * aq[0][nt][e] : 0.f,
                 j + 1 <= r ? a.scale * aq[0][nt][e + 1] : 0.f);
        }
    }
    cp_async_wait<0>();
    dqa_sync();
    constexpr int NH = 64 / (8 * DQA_CG);
    const int n0 = hf * (64 / DQA_CG);
    T* dst = static_cast<T*>(a.ws.dqh) + ch * (C * DK);
#pragma unroll 1
    for (int p = 0; p < NPAN; ++p) {
      Tile<T, DV, 64> S0p{reinterpret_cast<T*>(sm + L::S0) + (size_t)p * DV * 64};
      float acc[1][NH][4];
      zero(acc);
      Gemm<T>::template runk<1, NH, 0, DV>(acc, aview<false>(dOs), bview<true>(S0p), m0, n0, lane);
#pragma unroll
      for (int nt = 0; nt < NH; ++nt)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int r = m0 + frag_row(lane, e), c = 64 * p + n0 + 8 * nt + frag_col(lane, e);
          store2(dst + Sw<T, C, DK>::off(r, c), a.scale * acc[0][nt][e], a.scale * acc[0][nt][e + 1]);
        }
    }
    dqa_sync();  // the tiles are refilled for the next unit
  }
}

}  // namespace
}  // namespace gdn
