// Chunk preparation of the chunked forward on the 5th-generation tensor cores (bf16
// operands, Dk = Dv = 128): steps A1-A5 of one 64-token chunk and head at a time.
//
//   A1  G = cumsum(g) per key channel (fp32), gam = exp(G_C)
//   A2  the scan records scale Gam q and exp(G_C - G) k, and the row-scaled operands of
//       the boundary-split decay factorisation (marin.community note "factoring GDN-2
//       decay on TPU", section Approach) about the last token b of the first block:
//       q exp(G - G_b), k exp(G - G_b) (query side), k exp(G_b - G) (key side)
//   A3  the scores, one tcgen05.mma sequence with the two query-side tiles stacked to
//       M = 128:  [q e1 ; k e1] (k e2)^T  -> rows 0..63: Aqk, rows 64..127: Akk
//   A4  blocks whose decay spread would push the row factors out of range (or every
//       block, with GDN_FLAG_PAIRWISE_WITHIN_BLOCK) get their in-block scores pairwise on
//       CUDA cores (chunk_prep.cuh), as the note's kernel does for every in-block pair
//   A5  T = (I + Akk)^-1: the two 32 x 32 diagonal blocks by forward substitution in fp32
//       registers (a lane per column), then the off-diagonal block -T22 A21 T11 as two
//       tcgen05 products over 64 x 64 tiles restricted to the 32 k-steps that carry the
//       blocks (rows and columns outside them land in tensor memory that is never read,
//       so no zero blocks are written). With Tb = T diag(beta):
//       W = Tb (Gam k) (M = tokens, N = key channels) and U'^T = v^T Tb^T (M = value
//       columns, N = tokens), so neither k nor v is scaled by beta on the CUDA cores
// (the ai4snews "Gated DeltaNet" topic page, FlyWheel item, recasts triangular inversion
// as matrix products; atomic-ops 0.1.0, section Features, names the stages chunk scores,
// WY block solve, recompute). One decay per head (g [B,T,H]) uses the mask form: the
// scores are the raw products times exp(G_t - G_j) <= 1.
//
// The records it writes are those of the CUDA-core preparation (chunk_fwd.cu): the same
// layouts, so the scans and the backward read either. 256 threads, two persistent CTAs
// per SM, each taking every (2 x SMs)-th chunk: q, k, g and v arrive by TMA and the T,
// -W and U'^T records leave by bulk copies from shared memory (one thread issues them).
// Thread 0 issues every MMA; accumulators in tensor memory (192 columns).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "chunk_prep.cuh"
#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int PT = 128;  // Dk = Dv
constexpr int PTC_THREADS = 256;
constexpr uint32_t PTC_TMEM_COLS = 256;
// TMEM columns: the scores, then W (128 columns); level product 1; level product 2,
// then U'^T (64 columns)
constexpr int TP_S = 0, TP_X = 64, TP_T21 = 128, TP_W = 0, TP_U = 128;

typedef FTile<C, C, 4> AkkTile;  // fp32 Akk, transposed: at(j, i) = Akk[i][j] (padded rows)

struct PtcLayout {
  static constexpr int G = 0;                    // fp32 [C][Dk] cumulative log-decay
  static constexpr int K = G + C * PT * 4;       // k -> Gam k
  static constexpr int XS = K + C * PT * 2;      // [q e1 ; k e1] [2C][Dk] (q by TMA); later Akk fp32, XT
  static constexpr int TST = XS + 2 * C * PT * 2;  // [C][C]: scale Aqk staging, then T
  static constexpr int Y = TST + C * C * 2;      // raw g (row-major), then k e2; later v (TMA)
  static constexpr int BETA = Y + C * PT * 2;    // float [C] beta, float [C] scalar g
  static constexpr int BAR = BETA + 2 * C * 4;   // MMA completion, q/k/g landed, v landed
  static constexpr int TSLOT = BAR + 3 * 8;
  static constexpr int BYTES = TSLOT + 8;
  // the inverse's operand tiles, in the cumulative-decay region once the in-block pairwise
  // scores (the last reader of G) are done: Tb = T diag(beta) [C][C] (TBB) and the A21
  // operand AT [C][C] (A21 at rows C/2.., columns ..C/2); XT = A21 T11 [C][C] behind
  // Akk. The M = 128 products over TST, TBB and AT read the 64 rows behind each (Y, AT
  // and the rest of G) as rows whose results land in tensor-memory lanes never read.
  static constexpr int TBB = G + C * C * 2;
  static constexpr int AT = G + 2 * C * C * 2;
  static constexpr int XT = XS + a1k(AkkTile::BYTES);
  static constexpr uint32_t TX_QK = (uint32_t)(2 * C * PT * 2);
  static constexpr uint32_t TX_G = (uint32_t)(C * PT * 2);
  static constexpr uint32_t TX_V = (uint32_t)(C * PT * 2);
};
static_assert(PtcLayout::AT + 2 * C * C * 2 <= PtcLayout::K, "inverse tiles and the rows read behind them fit in G");
static_assert(PtcLayout::TST + 2 * C * C * 2 <= PtcLayout::BETA, "the rows read behind T are Y's");
static_assert(PtcLayout::XT + C * C * 2 <= PtcLayout::Y, "A21 T11 fits behind Akk");
static_assert(PtcLayout::K % 1024 == 0 && PtcLayout::XS % 1024 == 0 && PtcLayout::Y % 1024 == 0 &&
                  PtcLayout::TST % 1024 == 0 && PtcLayout::TBB % 1024 == 0 && PtcLayout::AT % 1024 == 0,
              "TMA and UMMA tiles on 1024-byte boundaries");
static_assert(2 * (PtcLayout::BYTES + 1024) <= 227 * 1024, "two CTAs per SM");

__device__ __forceinline__ uint32_t pack2(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
}
__device__ __forceinline__ void unpack8(float (&x)[8], const uint4 u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
    x[2 * e] = __low2float(h);
    x[2 * e + 1] = __high2float(h);
  }
}
// Packed fp32 pairs (f32x2 arithmetic): one instruction does the fp32 operation on both
// halves, each rounded as the scalar one.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ void ld8f(float (&x)[8], const float* p) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <bool PC>
__global__ void __launch_bounds__(PTC_THREADS, 2)
    chunk_prep_tc_kernel(ChunkFwdArgs a, const __grid_constant__ CUtensorMap q_map,
                         const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                         const __grid_constant__ CUtensorMap g_map) {
  pdl_wait();
  pdl_trigger();
  typedef PtcLayout L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  FTile<C, PT> Gs{reinterpret_cast<float*>(sm + L::G)};
  Tile<bf16, C, PT> Ks{reinterpret_cast<bf16*>(sm + L::K)};
  Tile<bf16, 2 * C, PT> XS{reinterpret_cast<bf16*>(sm + L::XS)};
  Tile<bf16, C, PT> Ys{reinterpret_cast<bf16*>(sm + L::Y)};
  Tile<bf16, C, C> Tst{reinterpret_cast<bf16*>(sm + L::TST)};
  float* beta_s = reinterpret_cast<float*>(sm + L::BETA);
  float* gsc = beta_s + C;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* bar_ld = bar + 1;
  uint64_t* bar_v = bar + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::TSLOT);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = a.T / C, units = N * a.B * a.H;
  const size_t rs = a.H;
  const bf16* q = static_cast<const bf16*>(a.q);
  const bf16* k = static_cast<const bf16*>(a.k);
  const bf16* g = static_cast<const bf16*>(a.g);
  const bf16* beta = static_cast<const bf16*>(a.beta);

  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(bar_ld, 1);
    mbar_init(bar_v, 1);
    fence_mbar_init();
  }
  // the forward scan's per-(batch, head) chunk counters start at zero (read only after
  // this kernel has completed)
  if (blockIdx.x == 0 && a.res.progress)
    for (int i = tid; i < a.B * a.H; i += PTC_THREADS) a.res.progress[i * PROGRESS_STRIDE] = 0u;
  if (warp == 0) {
    tmem_alloc(tslot, PTC_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's TMEM lane quarter
  const int rowl = 32 * (warp & 3) + lane, half = warp >> 2;
  uint32_t phase = 0, ldphase = 0;
  auto mma_done = [&]() {
    mbar_wait(bar, phase, a.err);
    phase ^= 1u;
    tc_fence_after();
  };
  const bf16* graw = reinterpret_cast<const bf16*>(sm + L::Y);

  // Persistent: unit u = (bh, chunk n), u = bh N + n, strided by the grid.
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int n = u % N, bh = u / N, b = bh / a.H, h = bh % a.H;
    const size_t ch = (size_t)u;
    const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
    const int tok = b * a.T + n * C;
    // ---- loads: q -> the upper half of XS, k -> K, per-channel g (row-major) -> Y
    if (tid == 0) {
      bulk_wait_read0();  // the previous chunk's T, -W and U'^T records have left TST, K and Y
      mbar_arrive_expect_tx(bar_ld, L::TX_QK + (PC ? L::TX_G : 0u));
      tma_load_3d(sm + L::XS, &q_map, 0, h, tok, bar_ld);
      tma_load_3d(sm + L::XS + 2 * C * 128, &q_map, 64, h, tok, bar_ld);
      tma_load_3d(sm + L::K, &k_map, 0, h, tok, bar_ld);
      tma_load_3d(sm + L::K + C * 128, &k_map, 64, h, tok, bar_ld);
      if (PC) tma_load_3d(sm + L::Y, &g_map, 0, h, tok, bar_ld);
    }
    if (tid < C) {
      beta_s[tid] = to_f32(beta[row0 + tid * rs]);
      if (!PC) gsc[tid] = to_f32(g[row0 + tid * rs]);
    }
    mbar_wait(bar_ld, ldphase, a.err);
    __syncthreads();

    // ---- A1
    prep_cumsum<bf16, PT, PTC_THREADS, PC>(Gs, graw, gsc, tid);
    __syncthreads();
    const bool force = (a.flags & FLAG_PAIRWISE) != 0;
    const bool mask_form = !PC && !force;
    bool u1 = false, u2 = false;
    if (PC)
      for (int c = tid; c < PT; c += PTC_THREADS) {
        u1 |= !(Gs.at(0, c) - Gs.at(BLK - 1, c) <= SAFE_SPREAD);
        u2 |= !(Gs.at(BLK - 1, c) - Gs.at(C - 1, c) <= SAFE_SPREAD);
      }
    const bool unsafe1 = __syncthreads_or(u1 || force) != 0;
    const bool unsafe2 = __syncthreads_or(u2 || force) != 0;

    // ---- A2: one pass. Thread: key channels cc .. cc + 7 of rows rb + 16 j, j < 4 (rows
    // of one swizzle phase, so every tile offset is the first row's plus j 16 rows).
    bf16* qh_g = static_cast<bf16*>(a.res.qh) + ch * (C * PT);
    bf16* kt_g = static_cast<bf16*>(a.res.kt) + ch * (C * PT);
    {
      const int cc = (lane & 15) * 8, rb = 2 * warp + (lane >> 4);
      const bool fast = !mask_form && !(unsafe1 || unsafe2);  // every factor in range
      float Gb[8], GC[8], eGb[8], eCb[8];
      ld8f(Gb, &Gs.at(BLK - 1, cc));
      ld8f(GC, &Gs.at(C - 1, cc));
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        eGb[e] = fast ? __expf(Gb[e]) : 0.f;
        eCb[e] = fast ? __expf(GC[e] - Gb[e]) : 0.f;
      }
      const int o1 = Sw<bf16, C, PT>::off(rb, cc);       // K, Y and the records
      const int oq = Sw<bf16, 2 * C, PT>::off(rb, cc);   // XS, query rows; key rows C below
      constexpr int RSTEP = 16 * (PT / 2);               // 16 rows of a 64-column panel
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = rb + 16 * j;
        const bool dead_q = !mask_form && j < 2 && unsafe1;   // query-side factor may overflow
        const bool dead_k = !mask_form && j >= 2 && unsafe2;  // key-side factor may overflow
        float qv[8], kv[8], G[8], o1v[8], o2v[8], xq[8], xk[8], yk[8], gk[8];
        unpack8(qv, *reinterpret_cast<const uint4*>(XS.p + oq + j * RSTEP));
        unpack8(kv, *reinterpret_cast<const uint4*>(Ks.p + o1 + j * RSTEP));
        ld8f(G, &Gs.at(r, cc));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float e1, e2, gm, kd;
          if (mask_form) {
            e1 = e2 = 1.f;
            gm = __expf(G[e]);
            kd = __expf(GC[e] - G[e]);
          } else {
            e1 = dead_q ? 0.f : __expf(G[e] - Gb[e]);
            e2 = dead_k ? 0.f : __expf(Gb[e] - G[e]);
            gm = fast ? eGb[e] * e1 : __expf(G[e]);
            kd = fast ? eCb[e] * e2 : __expf(GC[e] - G[e]);
          }
          o1v[e] = a.scale * gm * qv[e];
          o2v[e] = kd * kv[e];
          xq[e] = qv[e] * e1;
          xk[e] = kv[e] * e1;
          yk[e] = kv[e] * e2;
          gk[e] = gm * kv[e];
        }
        *reinterpret_cast<uint4*>(qh_g + o1 + j * RSTEP) = pack8(o1v);
        *reinterpret_cast<uint4*>(kt_g + o1 + j * RSTEP) = pack8(o2v);
        *reinterpret_cast<uint4*>(XS.p + oq + j * RSTEP) = pack8(xq);
        *reinterpret_cast<uint4*>(XS.p + oq + C * (PT / 2) + j * RSTEP) = pack8(xk);
        *reinterpret_cast<uint4*>(Ys.p + o1 + j * RSTEP) = pack8(yk);
        *reinterpret_cast<uint4*>(Ks.p + o1 + j * RSTEP) = pack8(gk);
      }
    }
    for (int c = tid; c < PT; c += PTC_THREADS) a.res.gam[ch * PT + c] = __expf(Gs.at(C - 1, c));
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- A3: [q e1 ; k e1] (k e2)^T (M = 2C, N = C, K = Dk)
    constexpr uint32_t id_s = umma_idesc_bf16(128, C, false, false);
    if (tid == 0) {
      tc_fence_after();
      const uint64_t dA = desc_kmajor(XS.p), dB = desc_kmajor(Ys.p);
#pragma unroll
      for (int ks = 0; ks < PT / 16; ++ks)
        umma_bf16(tm + TP_S, kstep_kmajor(dA, ks, 2 * C * 128), kstep_kmajor(dB, ks, C * 128), id_s, ks > 0);
      umma_commit(bar);
    }
    mma_done();
    // scores epilogue. Thread: row t' = rowl of [Aqk ; Akk], key columns 32 half .. + 31.
    AkkTile Akk{reinterpret_cast<float*>(sm + L::XS)};  // XS was read by the finished product
    {
      float d[32];
      tmem_ld32(tl + TP_S + 32 * half, d);
      const int tp = rowl, t = tp & (C - 1);
      const float Gt = Gs.at(t, 0);
      if (tp < C) {
        float o[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * half + jj;
          const float dec = mask_form && j < t ? __expf(Gt - Gs.at(j, 0)) : 1.f;
          o[jj] = j <= t ? a.scale * d[jj] * dec : 0.f;
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 pk;
          pk.x = pack2(o[8 * q4 + 0], o[8 * q4 + 1]);
          pk.y = pack2(o[8 * q4 + 2], o[8 * q4 + 3]);
          pk.z = pack2(o[8 * q4 + 4], o[8 * q4 + 5]);
          pk.w = pack2(o[8 * q4 + 6], o[8 * q4 + 7]);
          *reinterpret_cast<uint4*>(Tst.ptr(t, 32 * half + 8 * q4)) = pk;
        }
      }
      tc_fence_before();
      __syncthreads();  // every thread has read the scores: XS becomes the fp32 Akk
      if (tp >= C) {
        const float br = beta_s[t];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * half + jj;
          const float dec = mask_form && j < t ? __expf(Gt - Gs.at(j, 0)) : 1.f;
          Akk.at(j, t) = j < t ? br * d[jj] * dec : 0.f;  // transposed: lanes write one row
        }
      }
    }
    __syncthreads();
    if (unsafe1 || unsafe2) {
      prep_pairwise<bf16, PT, PTC_THREADS, true>(unsafe1, unsafe2, q, k, row0, rs, Gs, Tst, Akk, beta_s,
                                           a.scale, tid);
      __syncthreads();
    }
    {  // the scaled Aqk record
      bf16* dst = static_cast<bf16*>(a.res.aqk) + ch * (C * C);
      for (int i = tid; i < C * C / 8; i += PTC_THREADS) copy16(dst + i * 8, Tst.p + i * 8);
    }
    __syncthreads();  // Tst now takes T

    // ---- A5: diagonal blocks. Warps 0 and 1: block o = 32 warp, lane = column j; the
    // others write the zero upper-right blocks of T and Tb and copy A21 into AT.
    Tile<bf16, C, C> Tb{reinterpret_cast<bf16*>(sm + L::TBB)};     // T diag(beta)
    Tile<bf16, C, C> AT{reinterpret_cast<bf16*>(sm + L::AT)};      // A21 at rows C/2.., cols ..C/2
    Tile<bf16, C, C> XT{reinterpret_cast<bf16*>(sm + L::XT)};      // A21 T11 at rows C/2.., cols ..C/2
    if (warp < 2) {
      // Column j of the block's inverse, right-looking in groups of four rows:
      // acc[i] = sum over finished rows kk of A[i][kk] T[kk][j]; a group's four entries
      // T[i][j] = -acc[i] (1 on the diagonal, 0 above) follow from the rows before them
      // inside the group, then every later row takes the group's four terms at once. The
      // accumulators of rows 2p and 2p + 1 form one packed fp32 pair (fma.rn.f32x2: each
      // half is the scalar fmaf, in the same order), fed by 16-byte loads of Akk^T that
      // hold one column of four consecutive rows.
      const int o = BLK * warp, j = lane;
      float t[BLK];
      uint64_t acc2[BLK / 2];
#pragma unroll
      for (int p2 = 0; p2 < BLK / 2; ++p2) acc2[p2] = f2_pack(0.f, 0.f);
#pragma unroll
      for (int mg = 0; mg < BLK / 4; ++mg) {
        const int m = 4 * mg;
        float am[4];
        f2_unpack(acc2[m / 2], am[0], am[1]);
        f2_unpack(acc2[m / 2 + 1], am[2], am[3]);
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          const int i = m + ii;
          float x = am[ii];
#pragma unroll
          for (int kk = 0; kk < ii; ++kk) x = fmaf(Akk.at(o + m + kk, o + i), t[m + kk], x);
          t[i] = i == j ? 1.f : (i > j ? -x : 0.f);
        }
        uint64_t tt[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) tt[q] = f2_pack(t[m + q], t[m + q]);
#pragma unroll
        for (int i = m + 4; i < BLK; i += 4) {  // rows i .. i + 3: two packed pairs
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 a4 = *reinterpret_cast<const float4*>(&Akk.at(o + m + q, o + i));
            acc2[i / 2] = f2_fma(f2_pack(a4.x, a4.y), tt[q], acc2[i / 2]);
            acc2[i / 2 + 1] = f2_fma(f2_pack(a4.z, a4.w), tt[q], acc2[i / 2 + 1]);
          }
        }
      }
      const float bj = beta_s[o + j];
#pragma unroll
      for (int i = 0; i < BLK; ++i) {
        Tst.at(o + i, o + j) = __float2bfloat16_rn(t[i]);
        Tb.at(o + i, o + j) = __float2bfloat16_rn(t[i] * bj);
      }
    } else {
      // v is needed from the W / U' products on: it streams into Y (read by the finished
      // score products), issued by a warp that has time while warps 0 and 1 substitute
      if (tid == PTC_THREADS - 32) {
        mbar_arrive_expect_tx(bar_v, L::TX_V);
        tma_load_3d(sm + L::Y, &v_map, 0, h, tok, bar_v);
        tma_load_3d(sm + L::Y + C * 128, &v_map, 64, h, tok, bar_v);
      }
      // 16-byte pieces: 0..127 the zero blocks (T, Tb: 32 rows x 4 pieces each), 128..255
      // A21 (32 rows x 4 pieces of 8 columns)
      for (int i = tid - 64; i < 256; i += PTC_THREADS - 64) {
        const int r = (i & 127) >> 2, c = 8 * (i & 3);
        if (i < 128) {
          *reinterpret_cast<uint4*>(Tst.ptr(r, BLK + c)) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(Tb.ptr(r, BLK + c)) = make_uint4(0u, 0u, 0u, 0u);
        } else {
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = Akk.at(c + e, BLK + r);
          *reinterpret_cast<uint4*>(AT.ptr(BLK + r, c)) = pack8(x);
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    // A21 T11 = (AT T)[C/2.., ..C/2]: M = 2C, N = C, K restricted to the first C/2
    // (A21's columns, T11's rows); other rows and columns of the result are not read
    constexpr uint32_t id_l = umma_idesc_bf16(128, C, false, true);
    if (tid == 0) {
      tc_fence_after();
      const uint64_t dA = desc_kmajor(AT.p), dB = desc_mnmajor(Tst.p, C * 128);
#pragma unroll
      for (int ks = 0; ks < BLK / 16; ++ks)
        umma_bf16(tm + TP_X, kstep_kmajor(dA, ks, C * 128), kstep_mnmajor(dB, ks), id_l, ks > 0);
      umma_commit(bar);
    }
    mma_done();
    if (warp == 1) {  // TMEM lanes 32..63: rows of block 2; columns 0..31
      float x[32];
      tmem_ld32(tl + TP_X, x);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = x[8 * c8 + e];
        *reinterpret_cast<uint4*>(XT.ptr(BLK + lane, 8 * c8)) = pack8(y);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    // T21 = -T22 (A21 T11) = -(T XT)[C/2.., ..C/2]: K restricted to the last C/2 (T22's
    // columns, the rows of A21 T11)
    if (tid == 0) {
      tc_fence_after();
      const uint64_t dA = desc_kmajor(Tst.p), dB = desc_mnmajor(XT.p, C * 128);
#pragma unroll
      for (int ks = BLK / 16; ks < C / 16; ++ks)
        umma_bf16(tm + TP_T21, kstep_kmajor(dA, ks, C * 128), kstep_mnmajor(dB, ks), id_l, ks > BLK / 16);
      umma_commit(bar);
    }
    mma_done();
    if (warp == 1) {
      float x[32];
      tmem_ld32(tl + TP_T21, x);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        float y[8], yb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          y[e] = -x[8 * c8 + e];
          yb[e] = y[e] * beta_s[8 * c8 + e];
        }
        *reinterpret_cast<uint4*>(Tst.ptr(BLK + lane, 8 * c8)) = pack8(y);
        *reinterpret_cast<uint4*>(Tb.ptr(BLK + lane, 8 * c8)) = pack8(yb);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    // W = Tb (Gam k) (M = C padded to 128, N = Dk, K = C) and U'^T = v^T Tb^T (M = Dv,
    // N = C, K = C); the T record leaves by a bulk copy meanwhile
    constexpr uint32_t id_w = umma_idesc_bf16(128, PT, false, true);
    constexpr uint32_t id_u = umma_idesc_bf16(128, C, true, false);
    if (tid == 0) {
      bulk_s2g(static_cast<bf16*>(a.res.tmat) + ch * (C * C), Tst.p, (uint32_t)(C * C * 2));
      bulk_commit();
      tc_fence_after();
      const uint64_t dTb = desc_kmajor(Tb.p);
      const uint64_t dK = desc_mnmajor(Ks.p, C * 128), dV = desc_mnmajor(Ys.p, C * 128);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        umma_bf16(tm + TP_W, kstep_kmajor(dTb, ks, C * 128), kstep_mnmajor(dK, ks), id_w, ks > 0);
      mbar_wait(bar_v, ldphase, a.err);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        umma_bf16(tm + TP_U, kstep_mnmajor(dV, ks), kstep_kmajor(dTb, ks, C * 128), id_u, ks > 0);
      umma_commit(bar);
    }
    mma_done();
    ldphase ^= 1u;
    {  // -W [C][Dk] staged over K (Gam k, read by the finished product): warps of lane
       // quarters 0 and 1 (lane = token), key channels 64 half .. + 63
      if ((warp & 3) < 2) {
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          float w[32];
          tmem_ld32(tl + TP_W + 64 * half + 32 * c2, w);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = -w[8 * q4 + e];
            *reinterpret_cast<uint4*>(Ks.ptr(rowl, 64 * half + 32 * c2 + 8 * q4)) = pack8(x);
          }
        }
      }
      // U'^T [Dv][C] staged over Y (v, read by the finished product): lane = value column
      // rowl, tokens 32 half .. + 31
      Tile<bf16, PT, C> Ust{reinterpret_cast<bf16*>(sm + L::Y)};
      float uu[32];
      tmem_ld32(tl + TP_U + 32 * half, uu);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = uu[8 * q4 + e];
        *reinterpret_cast<uint4*>(Ust.ptr(rowl, 32 * half + 8 * q4)) = pack8(x);
      }
    }
    // every thread is done with this unit's tiles and tensor memory; the staged records
    // leave by bulk copies (waited for before the next loads into K and Y)
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      bulk_s2g(static_cast<bf16*>(a.res.wneg) + ch * (C * PT), Ks.p, (uint32_t)(C * PT * 2));
      bulk_s2g(static_cast<bf16*>(a.res.up) + ch * (C * PT), sm + L::Y, (uint32_t)(C * PT * 2));
      bulk_commit();
    }
  }
  // In normal operation every load and MMA has completed (each was waited for); after a
  // failed wait they may not have, and none may be in flight when tensor memory is freed
  // or the CTA retires. The last T record has left shared memory.
  if (tid == 0) {
    if ((int)blockIdx.x < units) {
      mbar_drain(bar_ld, ldphase ^ 1u);
      mbar_drain(bar_v, ldphase ^ 1u);
    }
    umma_commit(bar);
    mbar_drain(bar, phase);
    bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, PTC_TMEM_COLS);
}

}  // namespace

bool prep_tc_applies(int bf16_operands, int DK, int DV) { return bf16_operands && DK == PT && DV == PT; }

cudaError_t launch_chunk_prep_tc(const ChunkFwdArgs& a, cudaStream_t s) {
  const long long units = (long long)(a.T / C) * a.B * a.H;
  if (units == 0) return cudaSuccess;
  if ((long long)a.B * a.T > 0x7fffffffLL) return cudaErrorInvalidValue;  // TMA token coordinate
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
  if (!encode) return cudaErrorNotSupported;
  // q, k, v [B*T][H][128] bf16: 64 channels x 1 head x 64 tokens per box, 128-byte
  // swizzle (the UMMA operand layout); per-channel g: 128 channels per box, row-major
  const cuuint64_t dims[3] = {(cuuint64_t)PT, (cuuint64_t)a.H, (cuuint64_t)a.B * a.T};
  const cuuint64_t strides[2] = {(cuuint64_t)PT * 2, (cuuint64_t)a.H * PT * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
  const cuuint32_t gbox[3] = {PT, 1, (cuuint32_t)C};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap qm, km, vm, gm;
  auto enc = [&](CUtensorMap* m, const void* p, const cuuint32_t* bx, CUtensorMapSwizzle sw) {
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p), dims, strides, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  if (!enc(&qm, a.q, box, CU_TENSOR_MAP_SWIZZLE_128B) || !enc(&km, a.k, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !enc(&vm, a.v, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (a.per_channel) {
    if (!enc(&gm, a.g, gbox, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
  } else {
    gm = qm;  // not read: one decay per token arrives by plain loads
  }
  const int bytes = PtcLayout::BYTES + 1024;
  auto kern = a.per_channel ? chunk_prep_tc_kernel<true> : chunk_prep_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int grid = units < 2LL * nsm ? (int)units : 2 * nsm;  // two resident CTAs per SM
  prof_mark(K_PREP_TC, s, true);
  e = launch_pdl(kern, dim3(grid), dim3(PTC_THREADS), bytes, s, a, qm, km, vm, gm);
  prof_mark(K_PREP_TC, s, false);
  return e;
}

}  // namespace gdn
