// Chunked forward of the gated delta rule: chunk-parallel preparation + sequential scan.
//
// Per chunk of C = 64 tokens (two 32-token blocks) and incoming state S0:
//   G = cumsum(g) per key channel, Gam = exp(G), gam = Gam[C-1]
//   Aqk[t,j] = sum_c q_tc k_jc exp(G_tc - G_jc) (j <= t),  Akk = diag(beta) (same, j < t, k for q)
//   T = (I + Akk)^-1,  W = T diag(beta)(Gam * k),  U' = T diag(beta) V
//   U = U' - W S0,  O = scale (Gam*q) S0 + scale Aqk U,  S1 = diag(gam) S0 + (exp(G_C - G) * k)^T U
// This is the WY/UT chunked form of the token recurrence; atomic-ops 0.1.0 (section
// Features) names the same four forward stages: chunk scores, WY block solve, recompute,
// inter-chunk scan.
//
// Scores use the boundary-split decay factorisation of the marin.community note
// "factoring GDN-2 decay on TPU" (section Approach): each query row and key row is
// scaled by its decay relative to the last token of the first block, so the cross-block
// tile is one tensor-core product with every factor <= 1. Rows of the first block use
// the chunk start as reference and rows of the second block reuse the boundary, so the
// in-block tiles are products too; their key factors are >= 1 and stay below
// exp(SAFE_SPREAD) whenever the block's decay spread does. A block whose spread is
// larger (or every block, with GDN_FLAG_PAIRWISE_WITHIN_BLOCK) gets its in-block
// scores from the direct pairwise sum on CUDA cores instead (four lanes per pair,
// reduced with warp shuffles), which is what the note's kernel does in every block.
//
// Kernels
//   chunk_prep_kernel      grid (chunks, B*H), 256 threads: A1-A5, writes the residual
//                          records (scaled Aqk, T, -W, U', scaled Q-hat, K-tilde, gam)
//   chunk_scan_fwd_kernel  grid (Dv/64, B*H), 256 threads: A6, fp32 state slice in
//                          registers; chunk records arrive by cp.async.bulk on mbarriers
//   chunk_out_kernel       grid (chunks, B*H), 256 threads: outputs from stored states
#include "chunk_out.cuh"
#include "chunk_prep.cuh"
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int PREP_THREADS = 256;
constexpr int SCAN_THREADS = 256;
// In-place inverse of the unit lower triangular L = I + A. On entry M holds A (strictly
// lower, zeros on and above the diagonal); on exit it holds T = L^-1 with its unit
// diagonal and zero upper part stored explicitly. Doubling: if T11, T22 invert the
// diagonal blocks of size s, the inverse of the 2s block is [[T11, 0], [-T22 A21 T11, T22]].
// The 16 x 16 diagonal blocks are inverted by forward substitution (a lane per column,
// in registers), and the 32 and 64 levels run on tensor cores with
// the three-term TF32 split (about 21 significant bits, far below the bf16 operand error).
typedef FTile<C, C, 4> MTile;        // padded rows: fragment loads are conflict free
typedef FTile<BLK, BLK, 4> XTile;

template <int NTHR>
__device__ void unit_lower_inverse64(MTile M, XTile X, int tid) {
  static_assert(NTHR == 256, "tensor-core levels assume 8 warps");
  const int warp = tid >> 5, lane = tid & 31;
  // 16 x 16 diagonal blocks by forward substitution: each lane of warps 0 and 1 keeps one
  // column of one block's inverse in registers, T[i][j] = -sum_{k<i} A[i][k] T[k][j]
  if (warp < 2) {
    const int o = 16 * (2 * warp + (lane >> 4)), j = lane & 15;
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = i == j ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int kk = 0; kk < i; ++kk) acc = fmaf(M.at(o + i, o + kk), t[kk], acc);
      if (i > j) t[i] = -acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) M.at(o + i, o + j) = t[i];
  }
  __syncthreads();
  // s = 16: two blocks (rows/cols offset o = 0, 32); warps 0..3: block w >> 1, columns 8 (w & 1)
  if (warp < 4) {
    const int o = (warp >> 1) * 32, n0 = (warp & 1) * 8;
    float acc[1][1][4];
    zero(acc);
    Gemm<float>::runk<1, 1, 0, 16>(acc, aview<false>(M, o + 16, o), bview<true>(M, o, o), 0, n0, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) X.at((warp >> 1) * 16 + frag_row(lane, e), n0 + frag_col(lane, e)) = acc[0][0][e];
  }
  __syncthreads();
  if (warp < 4) {
    const int o = (warp >> 1) * 32, n0 = (warp & 1) * 8;
    float acc[1][1][4];
    zero(acc);
    Gemm<float>::runk<1, 1, 0, 16>(acc, aview<false>(M, o + 16, o + 16), bview<true>(X, (warp >> 1) * 16, 0), 0, n0,
                                   lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) M.at(o + 16 + frag_row(lane, e), o + n0 + frag_col(lane, e)) = -acc[0][0][e];
  }
  __syncthreads();
  // s = 32: one block; warp w: rows 16 (w & 1), columns 8 (w >> 1)
  {
    const int m0 = 16 * (warp & 1), n0 = 8 * (warp >> 1);
    float acc[1][1][4];
    zero(acc);
    Gemm<float>::runk<1, 1, 0, 32>(acc, aview<false>(M, 32, 0), bview<true>(M, 0, 0), m0, n0, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) X.at(m0 + frag_row(lane, e), n0 + frag_col(lane, e)) = acc[0][0][e];
    __syncthreads();
    zero(acc);
    Gemm<float>::runk<1, 1, 0, 32>(acc, aview<false>(M, 32, 32), bview<true>(X, 0, 0), m0, n0, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) M.at(32 + m0 + frag_row(lane, e), n0 + frag_col(lane, e)) = -acc[0][0][e];
  }
  __syncthreads();
}

template <class T, int DK, int DV>
struct PrepLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int MX = DK > DV ? DK : DV;
  static constexpr int RK = C * MX * ES;
  static constexpr int RX = C * MX * ES > MTile::BYTES ? C * MX * ES : MTile::BYTES;
  static constexpr int RY = C * MX * ES > XTile::BYTES ? C * MX * ES : XTile::BYTES;
  static constexpr int G = 0;                         // float [C][DK] cumulative log-decay
  static constexpr int K = a1k(G + C * DK * 4);       // k, then beta Gam k in place
  static constexpr int X = a1k(K + RK);               // q, then q e1; then Akk / T (fp32); then beta v
  static constexpr int X2 = a1k(X + RX);              // k e1 (query side of Akk); then -W staging
  static constexpr int Y = a1k(X2 + RK);              // raw g; k e2 (key side); inverse scratch; U' staging
  static constexpr int TST = a1k(Y + RY);             // [C][C]: scale*Aqk staging, then T
  static constexpr int BETA = a1k(TST + C * C * ES);  // float [C] beta, float [C] scalar decay
  static constexpr int BYTES = BETA + 2 * C * 4;
};

template <class T, int DK, int DV, bool PC>
__global__ void __launch_bounds__(PREP_THREADS) chunk_prep_kernel(ChunkFwdArgs a) {
  pdl_wait();
  pdl_trigger();
  typedef PrepLayout<T, DK, DV> L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  FTile<C, DK> Gs{reinterpret_cast<float*>(sm + L::G)};
  Tile<T, C, DK> ks{reinterpret_cast<T*>(sm + L::K)};
  Tile<T, C, DK> Xs{reinterpret_cast<T*>(sm + L::X)};
  Tile<T, C, DK> Ys{reinterpret_cast<T*>(sm + L::Y)};
  Tile<T, C, C> Tst{reinterpret_cast<T*>(sm + L::TST)};
  float* beta_s = reinterpret_cast<float*>(sm + L::BETA);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  const int N = a.T / C;
  const size_t ch = (size_t)bh * N + n;
  const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
  const size_t rs = a.H;
  constexpr int EPC = 16 / (int)sizeof(T);
  constexpr int CPR = DK / EPC;  // 16-byte chunks per row
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* g = static_cast<const T*>(a.g);
  const T* beta = static_cast<const T*>(a.beta);

  // ---- asynchronous loads: k -> K, q -> X, per-channel g (raw) -> Y
  T* graw = reinterpret_cast<T*>(sm + L::Y);
  for (int i = tid; i < C * CPR; i += PREP_THREADS) {
    const int r = i / CPR, c = (i % CPR) * EPC;
    const size_t gi = (row0 + r * rs) * DK + c;
    cp_async16(ks.ptr(r, c), k + gi);
    cp_async16(Xs.ptr(r, c), q + gi);
    if (PC) cp_async16(graw + r * DK + c, g + gi);
  }
  cp_async_commit();
  float* gsc = reinterpret_cast<float*>(sm + L::BETA) + C;  // scalar decay per token
  if (tid < C) {
    beta_s[tid] = to_f32(beta[row0 + tid * rs]);
    if (!PC) gsc[tid] = to_f32(g[row0 + tid * rs]);
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- A1: inclusive cumulative log-decay per channel (fp32)
  prep_cumsum<T, DK, PREP_THREADS, PC>(Gs, graw, gsc, tid);
  __syncthreads();
  // Reference point for every row: the boundary b = last token of the first block.
  // Factor ranges: block 1 queries exp(G_t - G_b) <= exp(G_0 - G_b); block 2 keys
  // exp(G_b - G_j) <= exp(G_b - G_C-1). Each must stay inside the fp32/bf16 range.
  // With one decay per head (PC false) the scores are the raw products times the C x C
  // factor exp(G_t - G_j) <= 1, which never leaves the fp32 range: no range check (the
  // mask form; GDN_FLAG_PAIRWISE_WITHIN_BLOCK still makes every in-block tile pairwise).
  const bool force = (a.flags & 1) != 0;
  bool u1 = false, u2 = false;
  if (PC)
    for (int c = tid; c < DK; c += PREP_THREADS) {
      u1 |= !(Gs.at(0, c) - Gs.at(BLK - 1, c) <= SAFE_SPREAD);
      u2 |= !(Gs.at(BLK - 1, c) - Gs.at(C - 1, c) <= SAFE_SPREAD);
    }
  const bool unsafe1 = __syncthreads_or(u1 || force) != 0;
  const bool unsafe2 = __syncthreads_or(u2 || force) != 0;

  // ---- A2, one pass with four exponentials per element: the scan records (scale Q-hat,
  // K-tilde), the row-scaled score operands about the block boundary b (q e1 and k e1 on
  // the query side, k e2 on the key side; e1 = exp(G - G_b), e2 = exp(G_b - G)) and
  // beta Gam k for W, written over k
  Tile<T, C, DK> X2s{reinterpret_cast<T*>(sm + L::X2)};
  T* qh_g = static_cast<T*>(a.res.qh) + ch * (C * DK);
  T* kt_g = static_cast<T*>(a.res.kt) + ch * (C * DK);
  // Each thread always takes the same four channels. When both blocks are safe (spreads
  // <= SAFE_SPREAD, so exp(G_b), exp(G_C - G_b), e1 and e2 are all in fp32 range),
  // Gam = exp(G_b) e1 and exp(G_C - G) = exp(G_C - G_b) e2 save two exponentials per
  // element (the pass is compiled for that case); otherwise every factor is its own
  // exponential.
  static_assert(PREP_THREADS % (DK / 4) == 0, "fixed channels per thread");
  auto a2_pass = [&](auto fast_tag) {
    constexpr bool FAST = decltype(fast_tag)::value;
    const int cc = (tid % (DK / 4)) * 4;
    float Gb[4], GC[4], eGb[4], eCb[4];
    ld4(Gb, &Gs.at(BLK - 1, cc));
    ld4(GC, &Gs.at(C - 1, cc));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      eGb[e] = FAST ? __expf(Gb[e]) : 0.f;
      eCb[e] = FAST ? __expf(GC[e] - Gb[e]) : 0.f;
    }
#pragma unroll 2
    for (int i = tid; i < C * (DK / 4); i += PREP_THREADS) {
      const int r = i / (DK / 4), c0 = cc;
      const bool dead_q = !FAST && r < BLK && unsafe1;  // query rows whose factor may overflow
      const bool dead_k = !FAST && r >= BLK && unsafe2;  // key rows whose factor may overflow
      float qv[4], kv[4], G[4], o1[4], o2[4], xq[4], xk[4], yk[4], bk[4];
      ld4(qv, Xs.ptr(r, c0));
      ld4(kv, ks.ptr(r, c0));
      ld4(G, &Gs.at(r, c0));
      const float br = beta_s[r];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float e1 = dead_q ? 0.f : __expf(G[e] - Gb[e]);
        const float e2 = dead_k ? 0.f : __expf(Gb[e] - G[e]);
        const float gm = FAST ? eGb[e] * e1 : __expf(G[e]);
        const float kd = FAST ? eCb[e] * e2 : __expf(GC[e] - G[e]);
        o1[e] = a.scale * gm * qv[e];
        o2[e] = kd * kv[e];
        xq[e] = qv[e] * e1;
        xk[e] = kv[e] * e1;
        yk[e] = kv[e] * e2;
        bk[e] = br * gm * kv[e];
      }
      const int off = Sw<T, C, DK>::off(r, c0);
      st4(qh_g + off, o1);
      st4(kt_g + off, o2);
      st4(Xs.ptr(r, c0), xq);
      st4(X2s.ptr(r, c0), xk);
      st4(Ys.ptr(r, c0), yk);
      st4(ks.ptr(r, c0), bk);
    }
  };
  // one decay per head: the score operands are q and k themselves (the decay enters the
  // scores as a C x C factor), and Gam, exp(G_C - G) are one exponential per row
  auto a2_scalar = [&]() {
    for (int i = tid; i < C * (DK / 4); i += PREP_THREADS) {
      const int r = i / (DK / 4), c0 = (i % (DK / 4)) * 4;
      const float Gr = Gs.at(r, 0);
      const float gm = __expf(Gr), kd = __expf(Gs.at(C - 1, 0) - Gr), br = beta_s[r];
      float qv[4], kv[4], o1[4], o2[4], bk[4];
      ld4(qv, Xs.ptr(r, c0));
      ld4(kv, ks.ptr(r, c0));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o1[e] = a.scale * gm * qv[e];
        o2[e] = kd * kv[e];
        bk[e] = br * gm * kv[e];
      }
      const int off = Sw<T, C, DK>::off(r, c0);
      st4(qh_g + off, o1);
      st4(kt_g + off, o2);
      st4(X2s.ptr(r, c0), kv);
      st4(Ys.ptr(r, c0), kv);
      st4(ks.ptr(r, c0), bk);
    }
  };
  if (!PC && !force)
    a2_scalar();
  else if (!(unsafe1 || unsafe2))
    a2_pass(BoolTag<true>{});
  else
    a2_pass(BoolTag<false>{});
  for (int c = tid; c < DK; c += PREP_THREADS) a.res.gam[ch * DK + c] = __expf(Gs.at(C - 1, c));
  __syncthreads();

  // ---- A3: scores. Warp w: rows 16 (w & 3) .. +15, key columns 32 (w >> 2) .. +31.
  // Block-1 rows never see block-2 keys; unsafe blocks leave their in-block tile to A4.
  const int rg = warp & 3, hf = warp >> 2, m0 = 16 * rg, n0 = 32 * hf;
  const bool skip = (m0 < BLK) && (hf == 1 || unsafe1);
  float aq[1][4][4], ak[1][4][4];
  zero(aq);
  zero(ak);
  if (!skip) {
    Gemm<T>::template runk<1, 4, 0, DK>(aq, aview<false>(Xs), bview<false>(Ys), m0, n0, lane);
    Gemm<T>::template runk<1, 4, 0, DK>(ak, aview<false>(X2s), bview<false>(Ys), m0, n0, lane);
  }
  __syncthreads();  // every warp is done reading X: it becomes the fp32 Akk
  MTile Akk{reinterpret_cast<float*>(sm + L::X)};
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = m0 + frag_row(lane, e), j = n0 + 8 * nt + frag_col(lane, e);
      // one decay per head (mask form): exp(G_r - G_j) on the raw products
      const float dec = PC || force || j > r ? 1.f : __expf(Gs.at(r, 0) - Gs.at(j, 0));
      Tst.at(r, j) = from_f32<T>(j <= r ? a.scale * aq[0][nt][e] * dec : 0.f);
      Akk.at(r, j) = j < r ? beta_s[r] * ak[0][nt][e] * dec : 0.f;
    }
  __syncthreads();
  if (unsafe1 || unsafe2) {
    prep_pairwise<T, DK, PREP_THREADS>(unsafe1, unsafe2, q, k, row0, rs, Gs, Tst, Akk, beta_s, a.scale, tid);
    __syncthreads();
  }

  // ---- scaled Aqk record; A5: T = (I + Akk)^-1 (inverse scratch in Y)
  {
    T* dst = static_cast<T*>(a.res.aqk) + ch * (C * C);
    for (int i = tid; i < C * C / EPC; i += PREP_THREADS) copy16(dst + i * EPC, Tst.p + i * EPC);
  }
  unit_lower_inverse64<PREP_THREADS>(Akk, XTile{reinterpret_cast<float*>(sm + L::Y)}, tid);
  for (int i = tid; i < C * C; i += PREP_THREADS) {
    const int r = i / C, c = i % C;
    Tst.at(r, c) = from_f32<T>(r >= c ? Akk.at(r, c) : 0.f);
  }
  __syncthreads();  // T in Tst; X (fp32 T) free: v arrives there
  Tile<T, C, DV> Vs{reinterpret_cast<T*>(sm + L::X)};
  constexpr int CPRV = DV / EPC;
  for (int i = tid; i < C * CPRV; i += PREP_THREADS) {
    const int r = i / CPRV, c = (i % CPRV) * EPC;
    cp_async16(Vs.ptr(r, c), v + (row0 + r * rs) * DV + c);
  }
  cp_async_commit();
  {
    T* dst = static_cast<T*>(a.res.tmat) + ch * (C * C);
    for (int i = tid; i < C * C / EPC; i += PREP_THREADS) copy16(dst + i * EPC, Tst.p + i * EPC);
  }
  // -W = -T (beta Gam k), staged in X2
  {
    constexpr int NW = DK / 16;
    float accw[1][NW][4];
    zero(accw);
    Gemm<T>::template runk<1, NW, 0, C>(accw, aview<false>(Tst), bview<true>(ks), m0, hf * (DK / 2), lane);
    cp_async_wait<0>();
    __syncthreads();  // v has landed
    Tile<T, C, DK> wst{reinterpret_cast<T*>(sm + L::X2)};
#pragma unroll
    for (int nt = 0; nt < NW; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        wst.at(m0 + frag_row(lane, e), hf * (DK / 2) + 8 * nt + frag_col(lane, e)) = from_f32<T>(-accw[0][nt][e]);
  }
  for (int i = tid; i < C * CPRV; i += PREP_THREADS) {  // beta v in place
    const int r = i / CPRV, c0 = (i % CPRV) * EPC;
    __align__(16) T vv[EPC];
    copy16(vv, Vs.ptr(r, c0));
#pragma unroll
    for (int e = 0; e < EPC; ++e) vv[e] = from_f32<T>(beta_s[r] * to_f32(vv[e]));
    copy16(Vs.ptr(r, c0), vv);
  }
  __syncthreads();  // beta v complete; U' is staged in Y
  {
    constexpr int NU = DV / 16;
    float accu[1][NU][4];
    zero(accu);
    Gemm<T>::template runk<1, NU, 0, C>(accu, aview<false>(Tst), bview<true>(Vs), m0, hf * (DV / 2), lane);
    T* ust = reinterpret_cast<T*>(sm + L::Y);
#pragma unroll
    for (int nt = 0; nt < NU; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + frag_row(lane, e), c = hf * (DV / 2) + 8 * nt + frag_col(lane, e);
        ust[Sw<T, DV, C>::off(c, r)] = from_f32<T>(accu[0][nt][e]);  // U'^T [Dv][C]
      }
  }
  __syncthreads();
  {
    T* dw = static_cast<T*>(a.res.wneg) + ch * (C * DK);
    const T* sw = reinterpret_cast<const T*>(sm + L::X2);
    for (int i = tid; i < C * DK / EPC; i += PREP_THREADS) copy16(dw + i * EPC, sw + i * EPC);
    T* du = static_cast<T*>(a.res.up) + ch * (C * DV);
    const T* su = reinterpret_cast<const T*>(sm + L::Y);
    for (int i = tid; i < C * DV / EPC; i += PREP_THREADS) copy16(du + i * EPC, su + i * EPC);
  }
}

// ------------------------------------------------------------------ state scan
// Only the recurrence is sequential: U = U' + (-W) S and S <- diag(gam) S + K-tilde^T U.
// The outputs O = (scale Q-hat) S + (scale Aqk) U need no sequential order and are
// produced afterwards by chunk_out_kernel from the states and U this scan stores.
// CC: chunk length, C or C2 (128-token chunks, whose records chunk_merge.cu forms)
template <class T, int DK, int CC = C>
struct ScanLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int W = 0;                         // -W        [CC][DK]
  static constexpr int KT = W + CC * DK * ES;         // K-tilde   [CC][DK]
  static constexpr int UP = KT + CC * DK * ES;        // U'^T rows of this slice [NTS][CC]
  static constexpr int GAM = UP + CC * NTS * ES;      // float [DK]
  static constexpr int STAGE = a1k(GAM + DK * 4);
  static constexpr int STAGES = ES == 2 ? (CC == C ? 4 : 2) : 1;
  static constexpr int SS = STAGES * STAGE;           // state operand, transposed [NTS][DK]
  static constexpr int US = a1k(SS + DK * NTS * ES);  // U, transposed [NTS][CC]
  static constexpr int BAR = a1k(US + CC * NTS * ES);
  static constexpr int BYTES = BAR + 64;
  static constexpr uint32_t TX = (uint32_t)(2 * CC * DK * ES + CC * NTS * ES + DK * 4);
};

// The records a scan or output kernel over CC-token chunks reads and writes.
struct ChunkRecs {
  void *aqk, *wneg, *up, *qh, *kt;
  const float* gam;
  void *state, *u;
};
template <int CC>
__device__ __forceinline__ ChunkRecs chunk_recs(const ChunkFwdArgs& a) {
  if (CC == C) return ChunkRecs{a.res.aqk, a.res.wneg, a.res.up, a.res.qh, a.res.kt, a.res.gam, a.res.state, a.res.u};
  return ChunkRecs{a.res2.aqk, a.res2.wneg, a.res2.up, a.res2.qh, a.res2.kt, a.res2.gam, a.res2.state, a.res2.u};
}

// One CTA per (batch*head, NTS = 64 value columns), 8 warps. Warp w owns state rows
// (w & 3) * Dk/4 .. + Dk/4 and columns 32 (w >> 2) .. + 31 of the slice, and rows
// (w & 3) * CC/4 .. + CC/4 of U. The state and U records are stored transposed (value
// rows): S^T [Dv][Dk] and U^T [Dv][CC]; this CTA writes their rows tile * NTS .. + NTS - 1.
template <class T, int DK, int DV, int CC = C>
__global__ void __launch_bounds__(SCAN_THREADS) chunk_scan_fwd_kernel(ChunkFwdArgs a) {
  typedef ScanLayout<T, DK, CC> L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, bh = blockIdx.y;
  const int N = a.T / CC;
  const ChunkRecs R = chunk_recs<CC>(a);
  constexpr int MTS = DK / 64;    // m16 tiles of state rows per warp
  constexpr int MU = CC / 64;     // m16 tiles of U rows per warp
  const int rg = warp & 3, cg = warp >> 2;
  const int srow = rg * 16 * MTS, col0 = 32 * cg, urow = rg * 16 * MU;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  Tile<T, NTS, DK> Ss{reinterpret_cast<T*>(sm + L::SS)};  // S^T rows of this slice
  Tile<T, NTS, CC> Us{reinterpret_cast<T*>(sm + L::US)};  // U^T rows of this slice

  float S[MTS][4][4];
  const size_t sb = (size_t)bh * DK * DV;
#pragma unroll
  for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = srow + 16 * mt + frag_row(lane, e);
        const int c = tile * NTS + col0 + 8 * nt + frag_col(lane, e);
        S[mt][nt][e] = a.h0 ? a.h0[sb + (size_t)r * DV + c] : 0.f;
      }

  if (tid == 0) {
    for (int s = 0; s < L::STAGES; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto issue = [&](int n) {
    const int s = n % L::STAGES;
    uint8_t* st = sm + s * L::STAGE;
    const size_t ch = (size_t)bh * N + n;
    mbar_arrive_expect_tx(&bars[s], L::TX);
    bulk_g2s(st + L::W, static_cast<const T*>(R.wneg) + ch * (CC * DK), CC * DK * sizeof(T), &bars[s]);
    bulk_g2s(st + L::KT, static_cast<const T*>(R.kt) + ch * (CC * DK), CC * DK * sizeof(T), &bars[s]);
    {  // rows tile * NTS .. + NTS - 1 of U'^T: one piece per column panel
      constexpr int PW = Sw<T, DV, CC>::PW;
      const T* src = static_cast<const T*>(R.up) + ch * (CC * DV);
      for (int p = 0; p < CC / PW; ++p)
        bulk_g2s(st + L::UP + p * NTS * PW * sizeof(T), src + (size_t)p * DV * PW + (size_t)tile * NTS * PW,
                 NTS * PW * sizeof(T), &bars[s]);
    }
    bulk_g2s(st + L::GAM, R.gam + ch * DK, DK * 4, &bars[s]);
  };
  if (tid == 0)
    for (int n = 0; n < L::STAGES - 1 && n < N; ++n) issue(n);

  for (int n = 0; n < N; ++n) {
    const int s = n % L::STAGES;
    const uint32_t par = (uint32_t)(n / L::STAGES) & 1u;
    // refill the stage freed at the end of the previous step
    if (tid == 0 && n + L::STAGES - 1 < N) issue(n + L::STAGES - 1);
    uint8_t* st = sm + s * L::STAGE;
    Tile<T, CC, DK> Wt{reinterpret_cast<T*>(st + L::W)};
    Tile<T, CC, DK> Kt{reinterpret_cast<T*>(st + L::KT)};
    Tile<T, NTS, CC> Up{reinterpret_cast<T*>(st + L::UP)};  // this slice's rows of U'^T
    const float* gam = reinterpret_cast<const float*>(st + L::GAM);
    const size_t ch = (size_t)bh * N + n;

#pragma unroll
    for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          Ss.at(col0 + 8 * nt + frag_col(lane, e), srow + 16 * mt + frag_row(lane, e)) = from_f32<T>(S[mt][nt][e]);
    fence_proxy_async();  // the state copy is read by the bulk store below
    mbar_wait(&bars[s], par, a.err);
    __syncthreads();
    if (tid == 0) {  // residual: chunk-start state
      store_row_block<T, DV, DK>(static_cast<T*>(R.state) + ch * (DK * DV), Ss.p, tile * NTS, NTS);
      bulk_commit();
    }
    float ws[MU][4][4];
    zero(ws);
    Gemm<T>::template runk<MU, 4, 0, DK>(ws, aview<false>(Wt), bview<false>(Ss), urow, col0, lane);
#pragma unroll
    for (int mt = 0; mt < MU; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = urow + 16 * mt + frag_row(lane, e), c = col0 + 8 * nt + frag_col(lane, e);
          Us.at(c, r) = from_f32<T>(to_f32(Up.at(c, r)) + ws[mt][nt][e]);
        }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {  // residual: U
      store_row_block<T, DV, CC>(static_cast<T*>(R.u) + ch * (CC * DV), Us.p, tile * NTS, NTS);
      bulk_commit();
    }
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) S[mt][nt][e] *= gam[srow + 16 * mt + frag_row(lane, e)];
    Gemm<T>::template runk<MTS, 4, 0, CC>(S, aview<true>(Kt), bview<false>(Us), srow, col0, lane);
    if (tid == 0) bulk_wait_read0();  // the bulk stores have read Ss and Us before they are rewritten
    __syncthreads();
  }
  if (tid == 0) {  // every load landed and the residual stores complete before the CTA retires
    drain_ring(bars, L::STAGES, N);
    bulk_wait0();
  }
  if (a.h_final) {
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = srow + 16 * mt + frag_row(lane, e);
          const int c = tile * NTS + col0 + 8 * nt + frag_col(lane, e);
          a.h_final[sb + (size_t)r * DV + c] = S[mt][nt][e];
        }
  }
}

// ------------------------------------------------------------------ outputs
// O = (scale Q-hat) S0 + (scale Aqk) U per chunk, from the scan's chunk-start states and U
// (out_unit, chunk_out.cuh); one CTA per 64 rows of a chunk.
template <class T, int DK, int DV, int CC = C>
__global__ void __launch_bounds__(OUT_THREADS) chunk_out_kernel(ChunkFwdArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const ChunkRecs R = chunk_recs<CC>(a);
  out_unit<T, DK, DV, CC>(a, R.qh, R.aqk, R.state, R.u, blockIdx.x, blockIdx.y, align1024(smem_raw), threadIdx.x);
}

// 128-token chunks: the 64-token blocks' records from the preparation, merged
// (chunk_merge.cu), then the scan and the outputs over the 128-token chunks.
template <class T, int DK, int DV>
cudaError_t launch_fwd128_rest(const ChunkFwdArgs& a, cudaStream_t s) {
  const int BH = a.B * a.H;
  cudaError_t e = launch_chunk_merge128(a, s);
  if (e != cudaSuccess) return e;
  {
    const int bytes = ScanLayout<T, DK, C2>::BYTES + 1024;
    auto kern = chunk_scan_fwd_kernel<T, DK, DV, C2>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
      return e;
    prof_mark(K_SCAN_FWD, s, true);
    kern<<<dim3(DV / NTS, BH), SCAN_THREADS, bytes, s>>>(a);
    prof_mark(K_SCAN_FWD, s, false);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.T == 0) return cudaSuccess;
  const int bytes = OutLayout<T, DK, DV, C2>::BYTES + 1024;
  auto kern = chunk_out_kernel<T, DK, DV, C2>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) return e;
  prof_mark(K_OUT, s, true);
  e = launch_pdl(kern, dim3(a.T / C, BH), dim3(OUT_THREADS), bytes, s, a);
  prof_mark(K_OUT, s, false);
  return e;
}

template <class T, int DK, int DV>
cudaError_t launch_fwd_t(const ChunkFwdArgs& a, cudaStream_t s) {
  const int N = a.T / C, BH = a.B * a.H;
  cudaError_t e;
  if (prep_tc_applies(a.bf16, DK, DV)) {
    if ((e = launch_chunk_prep_tc(a, s)) != cudaSuccess) return e;
  } else {
    const int bytes = PrepLayout<T, DK, DV>::BYTES + 1024;
    auto kern = a.per_channel ? chunk_prep_kernel<T, DK, DV, true> : chunk_prep_kernel<T, DK, DV, false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (N > 0) {
      prof_mark(K_PREP, s, true);
      if ((e = launch_pdl(kern, dim3(N, BH), dim3(PREP_THREADS), bytes, s, a)) != cudaSuccess) return e;
      prof_mark(K_PREP, s, false);
    }
  }
  if (a.flags & FLAG_CHUNK128) return launch_fwd128_rest<T, DK, DV>(a, s);
  bool outputs_done = false;
  if (scan_tc_applies(a.bf16, DK, DV)) {
    if ((e = launch_scan_fwd_tc(a, s, &outputs_done)) != cudaSuccess) return e;
  } else {
    const int bytes = ScanLayout<T, DK>::BYTES + 1024;
    auto kern = chunk_scan_fwd_kernel<T, DK, DV>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    prof_mark(K_SCAN_FWD, s, true);
    kern<<<dim3(DV / NTS, BH), SCAN_THREADS, bytes, s>>>(a);
    prof_mark(K_SCAN_FWD, s, false);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (N > 0 && !outputs_done) {
    const int bytes = OutLayout<T, DK, DV>::BYTES + 1024;
    auto kern = chunk_out_kernel<T, DK, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    prof_mark(K_OUT, s, true);
    if ((e = launch_pdl(kern, dim3(N, BH), dim3(OUT_THREADS), bytes, s, a)) != cudaSuccess) return e;
    prof_mark(K_OUT, s, false);
  }
  return cudaSuccess;
}

template <class T>
cudaError_t launch_fwd_dims(const ChunkFwdArgs& a, cudaStream_t s) {
  if (a.DK == 64) return a.DV == 64 ? launch_fwd_t<T, 64, 64>(a, s) : launch_fwd_t<T, 64, 128>(a, s);
  return a.DV == 64 ? launch_fwd_t<T, 128, 64>(a, s) : launch_fwd_t<T, 128, 128>(a, s);
}

}  // namespace

cudaError_t launch_chunk_fwd(const ChunkFwdArgs& a, cudaStream_t s) {
  if (a.B * a.H == 0) return cudaSuccess;
  return a.bf16 ? launch_fwd_dims<bf16>(a, s) : launch_fwd_dims<float>(a, s);
}

}  // namespace gdn
