// Chunk preparation of the chunked forward on the 5th-generation tensor cores (bf16
// operands, Dk = Dv = 128): steps A1-A5 of one 64-token chunk and head per CTA.
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
//       tcgen05 products of block-sparse 64 x 64 operands; then W^T = (beta Gam k)^T T^T
//       and U'^T = (beta v)^T T^T, M = 128 (key channels / value columns)
// (the ai4snews "Gated DeltaNet" topic page, FlyWheel item, recasts triangular inversion
// as matrix products; atomic-ops 0.1.0, section Features, names the stages chunk scores,
// WY block solve, recompute). One decay per head (g [B,T,H]) uses the mask form: the
// scores are the raw products times exp(G_t - G_j) <= 1.
//
// The records it writes are those of the CUDA-core preparation (chunk_fwd.cu): the same
// layouts and roundings, so the scans and the backward read either. 256 threads, two
// CTAs per SM; thread 0 issues every MMA; accumulators in tensor memory (192 columns).
#include "chunk_prep.cuh"
#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int PT = 128;              // Dk = Dv
constexpr int PTC_THREADS = 256;
constexpr uint32_t PTC_TMEM_COLS = 256;
// TMEM columns: scores, then W^T; level product 1, then U'^T; level product 2
constexpr int TP_S = 0, TP_X = 64, TP_T21 = 128, TP_W = 0, TP_U = 64;

typedef FTile<C, C, 4> AkkTile;  // fp32 Akk (padded rows)

struct PtcLayout {
  static constexpr int G = 0;                          // fp32 [C][Dk] cumulative log-decay
  static constexpr int K = G + C * PT * 4;             // k -> beta Gam k; later -W staging
  static constexpr int XS = K + C * PT * 2;            // [q e1 ; k e1] [2C][Dk]; later Akk fp32, XT
  static constexpr int Y = XS + 2 * C * PT * 2;        // raw g, then k e2; later v -> beta v, U'^T staging
  static constexpr int TST = Y + C * PT * 2;           // [C][C]: scale Aqk staging, then T
  static constexpr int BETA = TST + C * C * 2;         // float [C] beta, float [C] scalar g
  static constexpr int BAR = BETA + 2 * C * 4;
  static constexpr int TSLOT = BAR + 8;
  static constexpr int BYTES = TSLOT + 8;
  // the inverse's operand tiles, in the cumulative-decay region once the in-block pairwise
  // scores (the last reader of G) are done: TB = blockdiag(T11, T22) [2C][C] (rows C.. unused)
  // and AT = A21 block [2C][C]; XT = A21 T11 [C][C] behind Akk
  static constexpr int TB = G;
  static constexpr int AT = G + 2 * C * C * 2;
  static constexpr int XT = XS + a1k(AkkTile::BYTES);
};
static_assert(PtcLayout::AT + 2 * C * C * 2 <= PtcLayout::K, "inverse tiles fit in the G region");
static_assert(PtcLayout::XT + C * C * 2 <= PtcLayout::Y, "A21 T11 fits behind Akk");
static_assert(2 * (PtcLayout::BYTES + 1024) <= 227 * 1024, "two CTAs per SM");

__device__ __forceinline__ uint32_t pack2(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <bool PC>
__global__ void __launch_bounds__(PTC_THREADS, 2) chunk_prep_tc_kernel(ChunkFwdArgs a) {
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
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::TSLOT);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  const int N = a.T / C;
  const size_t ch = (size_t)bh * N + n;
  const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
  const size_t rs = a.H;
  constexpr int EPC = 8;
  constexpr int CPR = PT / EPC;  // 16-byte chunks per row
  const bf16* q = static_cast<const bf16*>(a.q);
  const bf16* k = static_cast<const bf16*>(a.k);
  const bf16* v = static_cast<const bf16*>(a.v);
  const bf16* g = static_cast<const bf16*>(a.g);
  const bf16* beta = static_cast<const bf16*>(a.beta);

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, PTC_TMEM_COLS);
    tmem_relinquish();
  }
  // ---- loads: k -> K, q -> the upper half of XS, per-channel g (raw, row-major) -> Y
  bf16* graw = reinterpret_cast<bf16*>(sm + L::Y);
  for (int i = tid; i < C * CPR; i += PTC_THREADS) {
    const int r = i / CPR, c = (i % CPR) * EPC;
    const size_t gi = (row0 + r * rs) * PT + c;
    cp_async16(Ks.ptr(r, c), k + gi);
    cp_async16(XS.ptr(r, c), q + gi);
    if (PC) cp_async16(graw + r * PT + c, g + gi);
  }
  cp_async_commit();
  if (tid < C) {
    beta_s[tid] = to_f32(beta[row0 + tid * rs]);
    if (!PC) gsc[tid] = to_f32(g[row0 + tid * rs]);
  }
  cp_async_wait<0>();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's TMEM lane quarter
  const int rowl = 32 * (warp & 3) + lane, half = warp >> 2;
  uint32_t phase = 0;
  auto mma_done = [&]() {
    mbar_wait(bar, phase, a.err);
    phase ^= 1u;
    tc_fence_after();
  };

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

  // ---- A2: one pass, each thread always on the same four channels
  bf16* qh_g = static_cast<bf16*>(a.res.qh) + ch * (C * PT);
  bf16* kt_g = static_cast<bf16*>(a.res.kt) + ch * (C * PT);
  {
    const int cc = (tid % (PT / 4)) * 4;
    const bool fast = !mask_form && !(unsafe1 || unsafe2);  // every factor in range
    float Gb[4], GC[4], eGb[4], eCb[4];
    ld4(Gb, &Gs.at(BLK - 1, cc));
    ld4(GC, &Gs.at(C - 1, cc));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      eGb[e] = fast ? __expf(Gb[e]) : 0.f;
      eCb[e] = fast ? __expf(GC[e] - Gb[e]) : 0.f;
    }
#pragma unroll 2
    for (int i = tid; i < C * (PT / 4); i += PTC_THREADS) {
      const int r = i / (PT / 4);
      const bool dead_q = !mask_form && r < BLK && unsafe1;   // query-side factor may overflow
      const bool dead_k = !mask_form && r >= BLK && unsafe2;  // key-side factor may overflow
      float qv[4], kv[4], G[4], o1[4], o2[4], xq[4], xk[4], yk[4], bk[4];
      ld4(qv, XS.ptr(r, cc));
      ld4(kv, Ks.ptr(r, cc));
      ld4(G, &Gs.at(r, cc));
      const float br = beta_s[r];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
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
        o1[e] = a.scale * gm * qv[e];
        o2[e] = kd * kv[e];
        xq[e] = qv[e] * e1;
        xk[e] = kv[e] * e1;
        yk[e] = kv[e] * e2;
        bk[e] = br * gm * kv[e];
      }
      const int off = Sw<bf16, C, PT>::off(r, cc);
      st4(qh_g + off, o1);
      st4(kt_g + off, o2);
      st4(XS.ptr(r, cc), xq);
      st4(XS.ptr(C + r, cc), xk);
      st4(Ys.ptr(r, cc), yk);
      st4(Ks.ptr(r, cc), bk);
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
  // v is needed from A5 on: it streams in now, into Y (read by the score products, done)
  Tile<bf16, C, PT> Vs{reinterpret_cast<bf16*>(sm + L::Y)};
  for (int i = tid; i < C * CPR; i += PTC_THREADS) {
    const int r = i / CPR, c = (i % CPR) * EPC;
    cp_async16(Vs.ptr(r, c), v + (row0 + r * rs) * PT + c);
  }
  cp_async_commit();
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
        uint4 u;
        u.x = pack2(o[8 * q4 + 0], o[8 * q4 + 1]);
        u.y = pack2(o[8 * q4 + 2], o[8 * q4 + 3]);
        u.z = pack2(o[8 * q4 + 4], o[8 * q4 + 5]);
        u.w = pack2(o[8 * q4 + 6], o[8 * q4 + 7]);
        *reinterpret_cast<uint4*>(Tst.ptr(t, 32 * half + 8 * q4)) = u;
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
        Akk.at(t, j) = j < t ? br * d[jj] * dec : 0.f;
      }
    }
  }
  __syncthreads();
  if (unsafe1 || unsafe2) {
    prep_pairwise<bf16, PT, PTC_THREADS>(unsafe1, unsafe2, q, k, row0, rs, Gs, Tst, Akk, beta_s, a.scale, tid);
    __syncthreads();
  }
  {  // the scaled Aqk record
    bf16* dst = static_cast<bf16*>(a.res.aqk) + ch * (C * C);
    for (int i = tid; i < C * C / EPC; i += PTC_THREADS) copy16(dst + i * EPC, Tst.p + i * EPC);
  }
  __syncthreads();  // Tst now takes T

  // ---- A5: diagonal blocks. Warps 0 and 1: block o = 32 warp, lane = column j; the
  // others write the zero blocks of T, TB and the A21 operand AT.
  Tile<bf16, 2 * C, C> TB{reinterpret_cast<bf16*>(sm + L::TB)};  // blockdiag(T11, T22)
  Tile<bf16, 2 * C, C> AT{reinterpret_cast<bf16*>(sm + L::AT)};  // A21 at rows C/2.., cols ..C/2
  Tile<bf16, C, C> XT{reinterpret_cast<bf16*>(sm + L::XT)};      // A21 T11 at rows C/2..
  if (warp < 2) {
    const int o = BLK * warp, j = lane;
    float t[BLK];
#pragma unroll
    for (int i = 0; i < BLK; ++i) t[i] = i == j ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < BLK; ++i) {  // T[i][j] = -sum_{kk<i} A[i][kk] T[kk][j], four partial sums
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < i; ++kk) acc[kk & 3] = fmaf(Akk.at(o + i, o + kk), t[kk], acc[kk & 3]);
      if (i > j) t[i] = -((acc[0] + acc[1]) + (acc[2] + acc[3]));
    }
#pragma unroll
    for (int i = 0; i < BLK; ++i) {
      const bf16 x = __float2bfloat16_rn(t[i]);
      Tst.at(o + i, o + j) = x;
      TB.at(o + i, o + j) = x;
    }
  } else {
    for (int i = tid - 64; i < BLK * BLK; i += PTC_THREADS - 64) {
      const int r = i / BLK, c = i % BLK;
      const bf16 z = __float2bfloat16_rn(0.f);
      Tst.at(r, BLK + c) = z;                  // T is lower triangular
      TB.at(r, BLK + c) = z;                   // TB is block diagonal
      TB.at(BLK + r, c) = z;
      AT.at(r, c) = z;                         // AT holds only A21
      AT.at(r, BLK + c) = z;
      AT.at(BLK + r, c) = __float2bfloat16_rn(Akk.at(BLK + r, c));
      AT.at(BLK + r, BLK + c) = z;
      XT.at(r, c) = z;                         // rows of XT above A21 T11 are zero
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  // A21 T11 = (AT TB)[C/2.., ..C/2] (M = 2C, N = C, K = C); rows C.. of AT are not used
  constexpr uint32_t id_l = umma_idesc_bf16(128, C, false, true);
  if (tid == 0) {
    tc_fence_after();
    const uint64_t dA = desc_kmajor(AT.p), dB = desc_mnmajor(TB.p, 2 * C * 128);
#pragma unroll
    for (int ks = 0; ks < C / 16; ++ks)
      umma_bf16(tm + TP_X, kstep_kmajor(dA, ks, 2 * C * 128), kstep_mnmajor(dB, ks), id_l, ks > 0);
    umma_commit(bar);
  }
  mma_done();
  if (warp == 1) {  // TMEM lanes 32..63: rows of block 2; columns 0..31
    float x[32];
    tmem_ld32(tl + TP_X, x);
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) XT.at(BLK + lane, jj) = __float2bfloat16_rn(x[jj]);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  // T21 = -T22 (A21 T11) = -(TB XT)[C/2.., ..C/2]
  if (tid == 0) {
    tc_fence_after();
    const uint64_t dA = desc_kmajor(TB.p), dB = desc_mnmajor(XT.p, C * 128);
#pragma unroll
    for (int ks = 0; ks < C / 16; ++ks)
      umma_bf16(tm + TP_T21, kstep_kmajor(dA, ks, 2 * C * 128), kstep_mnmajor(dB, ks), id_l, ks > 0);
    umma_commit(bar);
  }
  mma_done();
  if (warp == 1) {
    float x[32];
    tmem_ld32(tl + TP_T21, x);
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) Tst.at(BLK + lane, jj) = __float2bfloat16_rn(-x[jj]);
  }
  cp_async_wait<0>();  // v
  __syncthreads();
  {  // the T record; beta v in place
    bf16* dst = static_cast<bf16*>(a.res.tmat) + ch * (C * C);
    for (int i = tid; i < C * C / EPC; i += PTC_THREADS) copy16(dst + i * EPC, Tst.p + i * EPC);
    for (int i = tid; i < C * CPR; i += PTC_THREADS) {
      const int r = i / CPR, c0 = (i % CPR) * EPC;
      __align__(16) bf16 vv[EPC];
      copy16(vv, Vs.ptr(r, c0));
#pragma unroll
      for (int e = 0; e < EPC; ++e) vv[e] = __float2bfloat16_rn(beta_s[r] * __bfloat162float(vv[e]));
      copy16(Vs.ptr(r, c0), vv);
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  // W^T = (beta Gam k)^T T^T and U'^T = (beta v)^T T^T (M = Dk or Dv, N = C, K = C)
  constexpr uint32_t id_w = umma_idesc_bf16(128, C, true, false);
  if (tid == 0) {
    tc_fence_after();
    const uint64_t dT = desc_kmajor(Tst.p);
    const uint64_t dK = desc_mnmajor(Ks.p, C * 128), dV = desc_mnmajor(Vs.p, C * 128);
#pragma unroll
    for (int ks = 0; ks < C / 16; ++ks)
      umma_bf16(tm + TP_W, kstep_mnmajor(dK, ks), kstep_kmajor(dT, ks, C * 128), id_w, ks > 0);
#pragma unroll
    for (int ks = 0; ks < C / 16; ++ks)
      umma_bf16(tm + TP_U, kstep_mnmajor(dV, ks), kstep_kmajor(dT, ks, C * 128), id_w, ks > 0);
    umma_commit(bar);
  }
  mma_done();
  // -W [C][Dk] staged over K, U'^T [Dv][C] staged over V (both read by the finished
  // products). Thread: lane = key channel / value column rowl, tokens 32 half .. + 31.
  Tile<bf16, C, PT> Wst{reinterpret_cast<bf16*>(sm + L::K)};
  Tile<bf16, PT, C> Ust{reinterpret_cast<bf16*>(sm + L::Y)};
  {
    float w[32];
    tmem_ld32(tl + TP_W + 32 * half, w);
    float u[32];
    tmem_ld32(tl + TP_U + 32 * half, u);
    tc_fence_before();
    __syncthreads();  // every product has been read before the staging tiles are written
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) Wst.at(32 * half + jj, rowl) = __float2bfloat16_rn(-w[jj]);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint4 pk;
      pk.x = pack2(u[8 * q4 + 0], u[8 * q4 + 1]);
      pk.y = pack2(u[8 * q4 + 2], u[8 * q4 + 3]);
      pk.z = pack2(u[8 * q4 + 4], u[8 * q4 + 5]);
      pk.w = pack2(u[8 * q4 + 6], u[8 * q4 + 7]);
      *reinterpret_cast<uint4*>(Ust.ptr(rowl, 32 * half + 8 * q4)) = pk;
    }
  }
  __syncthreads();
  {
    bf16* dw = static_cast<bf16*>(a.res.wneg) + ch * (C * PT);
    for (int i = tid; i < C * PT / EPC; i += PTC_THREADS) copy16(dw + i * EPC, Wst.p + i * EPC);
    bf16* du = static_cast<bf16*>(a.res.up) + ch * (C * PT);
    for (int i = tid; i < C * PT / EPC; i += PTC_THREADS) copy16(du + i * EPC, Ust.p + i * EPC);
  }
  if (tid == 0) {  // every MMA has completed (waited above); nothing is in flight
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, PTC_TMEM_COLS);
}

}  // namespace

bool prep_tc_applies(int bf16_operands, int DK, int DV) { return bf16_operands && DK == PT && DV == PT; }

cudaError_t launch_chunk_prep_tc(const ChunkFwdArgs& a, cudaStream_t s) {
  const int N = a.T / C, BH = a.B * a.H;
  if (N == 0 || BH == 0) return cudaSuccess;
  const int bytes = PtcLayout::BYTES + 1024;
  auto kern = a.per_channel ? chunk_prep_tc_kernel<true> : chunk_prep_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  prof_mark(K_PREP_TC, s, true);
  e = launch_pdl(kern, dim3(N, BH), dim3(PTC_THREADS), bytes, s, a);
  prof_mark(K_PREP_TC, s, false);
  return e;
}

}  // namespace gdn
