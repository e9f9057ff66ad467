// 128-token chunks of the chunked forward (GDN_FLAG_CHUNK128): each chunk is two
// consecutive 64-token blocks, the chunk of KernelConfig's bt = 2 bc (atomic-ops 0.1.0,
// section API). The preparation kernels form every block's records exactly as for a
// 64-token chunk (chunk_fwd.cu, chunk_prep_tc.cu): scale Aqk, -W, U'^T, scale Q-hat,
// K-tilde and gam, each relative to the block's own start. Taking the block boundary b
// (the last token of block 1) as the reference, the 128-token chunk's records follow
// from the two blocks' records alone:
//   M       = (-W2) K-tilde1^T                       (64 x 64)  = -T22 A21
//   Aqk21   = (scale Q-hat2) K-tilde1^T               (64 x 64)  the cross-block scores
//   -W      = [ -W1 ; (-W2) diag(gam1) + M (-W1) ]
//   U'^T    = [ U'1^T , U'2^T + U'1^T M^T ]
//   Q-hat   = [ Q-hat1 ; Q-hat2 diag(gam1) ],   K-tilde = [ K-tilde1 diag(gam2) ; K-tilde2 ]
//   gam     = gam1 gam2,   Aqk = [[Aqk1, 0], [Aqk21, Aqk2]]
// A21 is the cross-block tile of diag(beta) (k k^T weighted by exp(G_i - G_j)), and
// M (-W1), M U'1 apply the off-diagonal block T21 = -T22 A21 T11 of the 128-token WY
// inverse to beta Gam k and beta v (T11, T22 are the blocks' own inverses). Q-hat2 carries
// exp(G_i - G_b) <= 1 and K-tilde1 exp(G_b - G_j) <= 1, so the cross-block tiles are the
// factored 64-query x 64-key product of the marin.community note "factoring GDN-2 decay
// on TPU" (section Approach), and no factor can leave the fp32 range whatever the decay
// spread. The state scan and the outputs then run over the 128-token chunks
// (chunk_fwd.cu, CC = C2).
//
// chunk_merge128_kernel: grid (T / 128, B*H), 256 threads (8 warps), one chunk-head each.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int MERGE_THREADS = 256;

template <class T, int DK, int DV>
struct MergeLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int W1 = 0;                       // -W of block 1 [C][DK]
  static constexpr int W2 = a1k(W1 + C * DK * ES);   // -W of block 2, then the chunk's rows 64..127
  static constexpr int Q2 = a1k(W2 + C * DK * ES);   // scale Q-hat of block 2 [C][DK]
  static constexpr int K1 = a1k(Q2 + C * DK * ES);   // K-tilde of block 1 [C][DK]
  static constexpr int U1 = a1k(K1 + C * DK * ES);   // U'^T of block 1 [DV][C]
  static constexpr int U2 = a1k(U1 + DV * C * ES);   // U'^T of block 2, then the chunk's columns 64..127
  static constexpr int M = a1k(U2 + DV * C * ES);    // M = (-W2) K-tilde1^T [C][C]
  static constexpr int G1 = a1k(M + C * C * ES);     // gam of blocks 1 and 2, fp32 [2][DK]
  static constexpr int BYTES = G1 + 2 * DK * 4;
};

// Copies the ROWS x COLS record image src (Sw<T, ROWS, COLS>, global or shared memory) into
// the DR x DC record image dst at rows r0.., columns c0.. (c0 a multiple of 16 bytes of
// elements), 16 bytes at a time; with colscale (shared memory) each element of source
// column c is multiplied by colscale[c] (fp32) and rounded once. Every load of a thread is
// issued before its first store, so a copy from global memory waits out one round trip.
template <class T, int ROWS, int COLS, int DR, int DC>
__device__ __forceinline__ void place(T* __restrict__ dst, const T* __restrict__ src, int r0, int c0,
                                      const float* colscale, int tid) {
  constexpr int EPC = 16 / (int)sizeof(T);
  constexpr int NCH = ROWS * COLS / EPC;
  static_assert(NCH % MERGE_THREADS == 0, "whole passes");
  constexpr int NIT = NCH / MERGE_THREADS;
  uint4 v[NIT];
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int i = tid + it * MERGE_THREADS, r = i / (COLS / EPC), c = (i % (COLS / EPC)) * EPC;
    v[it] = *reinterpret_cast<const uint4*>(src + Sw<T, ROWS, COLS>::off(r, c));
  }
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int i = tid + it * MERGE_THREADS, r = i / (COLS / EPC), c = (i % (COLS / EPC)) * EPC;
    if (colscale) {
      __align__(16) T x[EPC];
      *reinterpret_cast<uint4*>(x) = v[it];
#pragma unroll
      for (int e = 0; e < EPC; ++e) x[e] = from_f32<T>(to_f32(x[e]) * colscale[c + e]);
      v[it] = *reinterpret_cast<const uint4*>(x);
    }
    *reinterpret_cast<uint4*>(dst + Sw<T, DR, DC>::off(r + r0, c + c0)) = v[it];
  }
}

template <class T, int DK, int DV>
__global__ void __launch_bounds__(MERGE_THREADS) chunk_merge128_kernel(ChunkFwdArgs a) {
  pdl_wait();  // the blocks' records come from the preparation launched just before
  pdl_trigger();
  typedef MergeLayout<T, DK, DV> L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m = blockIdx.x, bh = blockIdx.y;
  const int N = a.T / C, N2 = a.T / C2;
  const size_t c1 = (size_t)bh * N + 2 * m, c2 = c1 + 1, cm = (size_t)bh * N2 + m;
  constexpr int EPC = 16 / (int)sizeof(T);
  const ResidualPtrs& r = a.res;
  const Residual128Ptrs& o = a.res2;
  const T* w1g = static_cast<const T*>(r.wneg) + c1 * (C * DK);
  const T* w2g = static_cast<const T*>(r.wneg) + c2 * (C * DK);
  const T* q1g = static_cast<const T*>(r.qh) + c1 * (C * DK);
  const T* q2g = static_cast<const T*>(r.qh) + c2 * (C * DK);
  const T* k1g = static_cast<const T*>(r.kt) + c1 * (C * DK);
  const T* k2g = static_cast<const T*>(r.kt) + c2 * (C * DK);
  const T* u1g = static_cast<const T*>(r.up) + c1 * (C * DV);
  const T* u2g = static_cast<const T*>(r.up) + c2 * (C * DV);
  const T* a1g = static_cast<const T*>(r.aqk) + c1 * (C * C);
  const T* a2g = static_cast<const T*>(r.aqk) + c2 * (C * C);
  const float* g1g = r.gam + c1 * DK;
  const float* g2g = r.gam + c2 * DK;
  T* wo = static_cast<T*>(o.wneg) + cm * (C2 * DK);
  T* qo = static_cast<T*>(o.qh) + cm * (C2 * DK);
  T* ko = static_cast<T*>(o.kt) + cm * (C2 * DK);
  T* uo = static_cast<T*>(o.up) + cm * (C2 * DV);
  T* ao = static_cast<T*>(o.aqk) + cm * (C2 * C2);

  Tile<T, C, DK> W1s{reinterpret_cast<T*>(sm + L::W1)};
  Tile<T, C, DK> W2s{reinterpret_cast<T*>(sm + L::W2)};
  Tile<T, C, DK> Q2s{reinterpret_cast<T*>(sm + L::Q2)};
  Tile<T, C, DK> K1s{reinterpret_cast<T*>(sm + L::K1)};
  Tile<T, DV, C> U1s{reinterpret_cast<T*>(sm + L::U1)};
  Tile<T, DV, C> U2s{reinterpret_cast<T*>(sm + L::U2)};
  Tile<T, C, C> Ms{reinterpret_cast<T*>(sm + L::M)};
  float* g1s = reinterpret_cast<float*>(sm + L::G1);
  float* g2s = g1s + DK;

  // the six operand records, byte images of the shared tiles
  for (int i = tid; i < C * DK / EPC; i += MERGE_THREADS) {
    cp_async16(W1s.p + i * EPC, w1g + i * EPC);
    cp_async16(W2s.p + i * EPC, w2g + i * EPC);
    cp_async16(Q2s.p + i * EPC, q2g + i * EPC);
    cp_async16(K1s.p + i * EPC, k1g + i * EPC);
  }
  for (int i = tid; i < DV * C / EPC; i += MERGE_THREADS) {
    cp_async16(U1s.p + i * EPC, u1g + i * EPC);
    cp_async16(U2s.p + i * EPC, u2g + i * EPC);
  }
  cp_async_commit();
  for (int c = tid; c < DK; c += MERGE_THREADS) {
    const float x = g1g[c], y = g2g[c];
    g1s[c] = x;
    g2s[c] = y;
    o.gam[cm * DK + c] = x * y;
  }
  // records that pass through unchanged and are not operands: global to global while the
  // operand tiles arrive
  place<T, C, DK, C2, DK>(qo, q1g, 0, 0, nullptr, tid);
  place<T, C, DK, C2, DK>(ko, k2g, C, 0, nullptr, tid);
  place<T, C, C, C2, C2>(ao, a1g, 0, 0, nullptr, tid);
  place<T, C, C, C2, C2>(ao, a2g, C, C, nullptr, tid);
  for (int i = tid; i < C * C / EPC; i += MERGE_THREADS) {  // block 1 never sees block 2
    const int rr = i / (C / EPC), cc = (i % (C / EPC)) * EPC;
    *reinterpret_cast<uint4*>(ao + Sw<T, C2, C2>::off(rr, C + cc)) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_wait<0>();
  __syncthreads();
  // the operands that also pass through, unchanged or rescaled, from shared memory
  place<T, C, DK, C2, DK>(wo, W1s.p, 0, 0, nullptr, tid);
  place<T, C, DK, C2, DK>(qo, Q2s.p, C, 0, g1s, tid);
  place<T, C, DK, C2, DK>(ko, K1s.p, 0, 0, g2s, tid);
  place<T, DV, C, DV, C2>(uo, U1s.p, 0, 0, nullptr, tid);

  // M = (-W2) K-tilde1^T and the cross-block scores (scale Q-hat2) K-tilde1^T:
  // warp w takes rows 16 (w & 3) .. + 15 and key columns 32 (w >> 2) .. + 31 of both
  {
    const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
    float am[1][4][4], aq[1][4][4];
    zero(am);
    zero(aq);
    Gemm<T>::template runk<1, 4, 0, DK>(am, aview<false>(W2s), bview<false>(K1s), m0, n0, lane);
    Gemm<T>::template runk<1, 4, 0, DK>(aq, aview<false>(Q2s), bview<false>(K1s), m0, n0, lane);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int rr = m0 + frag_row(lane, e), j = n0 + 8 * nt + frag_col(lane, e);
        Ms.at(rr, j) = from_f32<T>(am[0][nt][e]);
        Ms.at(rr, j + 1) = from_f32<T>(am[0][nt][e + 1]);
        store2(ao + Sw<T, C2, C2>::off(C + rr, j), aq[0][nt][e], aq[0][nt][e + 1]);
      }
  }
  __syncthreads();  // M complete; W2 and U2 are next read only element by element, in place

  // rows 64..127 of -W: (-W2) diag(gam1) + M (-W1); warp w: rows 16 (w & 3), columns
  // (w >> 2) Dk/2 .. + Dk/2 - 1
  {
    constexpr int NW = DK / 16;
    const int m0 = 16 * (warp & 3), n0 = (warp >> 2) * (DK / 2);
    float acc[1][NW][4];
    zero(acc);
    Gemm<T>::template runk<1, NW, 0, C>(acc, aview<false>(Ms), bview<true>(W1s), m0, n0, lane);
#pragma unroll
    for (int nt = 0; nt < NW; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rr = m0 + frag_row(lane, e), c = n0 + 8 * nt + frag_col(lane, e);
        W2s.at(rr, c) = from_f32<T>(fmaf(to_f32(W2s.at(rr, c)), g1s[c], acc[0][nt][e]));
      }
  }
  // columns 64..127 of U'^T: U'2^T + U'1^T M^T; warp w: value rows 16 MT (w & 3) ..,
  // token columns 32 (w >> 2) .. + 31
  {
    constexpr int MT = DV / 64;
    const int m0 = 16 * MT * (warp & 3), n0 = 32 * (warp >> 2);
    float acc[MT][4][4];
    zero(acc);
    Gemm<T>::template runk<MT, 4, 0, C>(acc, aview<false>(U1s), bview<false>(Ms), m0, n0, lane);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = m0 + 16 * mt + frag_row(lane, e), t = n0 + 8 * nt + frag_col(lane, e);
          U2s.at(v, t) = from_f32<T>(to_f32(U2s.at(v, t)) + acc[mt][nt][e]);
        }
  }
  __syncthreads();
  place<T, C, DK, C2, DK>(wo, W2s.p, C, 0, nullptr, tid);
  place<T, DV, C, DV, C2>(uo, U2s.p, 0, C, nullptr, tid);
}

template <class T, int DK, int DV>
cudaError_t launch_merge_t(const ChunkFwdArgs& a, cudaStream_t s) {
  const int bytes = MergeLayout<T, DK, DV>::BYTES + 1024;
  auto kern = chunk_merge128_kernel<T, DK, DV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  prof_mark(K_MERGE, s, true);
  e = launch_pdl(kern, dim3(a.T / C2, a.B * a.H), dim3(MERGE_THREADS), bytes, s, a);
  prof_mark(K_MERGE, s, false);
  return e;
}

template <class T>
cudaError_t launch_merge_dims(const ChunkFwdArgs& a, cudaStream_t s) {
  if (a.DK == 64) return a.DV == 64 ? launch_merge_t<T, 64, 64>(a, s) : launch_merge_t<T, 64, 128>(a, s);
  return a.DV == 64 ? launch_merge_t<T, 128, 64>(a, s) : launch_merge_t<T, 128, 128>(a, s);
}

}  // namespace

cudaError_t launch_chunk_merge128(const ChunkFwdArgs& a, cudaStream_t s) {
  if (a.T < C2 || a.B * a.H == 0) return cudaSuccess;
  return a.bf16 ? launch_merge_dims<bf16>(a, s) : launch_merge_dims<float>(a, s);
}

}  // namespace gdn
