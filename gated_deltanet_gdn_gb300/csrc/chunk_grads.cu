// Chunk-parallel gradients of the chunked gated delta rule backward (bf16 or fp32
// operands, fp32 arithmetic).
//
// One CTA per (64-channel group, chunk, batch*head). Inputs: q, k, g, beta of the
// chunk and the state products dQ-hat, dBk, dK-tilde, dAqk, dAkk, dgam written by
// chunk_dstate_kernel (chunk_bwd.cu). Decay-weighted scores
//   P[t,j] = sum_c x_tc y_jc exp(G_tc - G_jc)
// have the gradients dx = (dP (*) E) y, dy = (dP^T (*) E) x and dG = x dx - y dy.
// Both products run on tensor cores with the rows scaled about one reference point,
// the last token b of the first block (the boundary-split factorisation of the
// marin.community note "factoring GDN-2 decay on TPU", section Approach): key rows
// by exp(G_b - G_j), query rows by exp(G_t - G_b). A block whose decay spread would
// push those factors out of range takes its in-block part from the pairwise sums.
//   Aqk family: x = q, dP = dAqk (diagonal handled apart: its dG terms cancel)
//   Akk family: x = k, dP = diag(beta) dAkk; sum_c k dx' gives the score part of dbeta
// dG further collects dQ-hat * Q-hat + beta dBk * K-hat - dK-tilde * K-tilde, and at
// the last row the K-tilde column sums and dgam * gam; dg is its reverse cumulative
// sum. dbeta and scalar-decay dg need sums over all channels: each CTA writes its
// channel group's partials and chunk_bwd_finalize_kernel adds them in a fixed order.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int GR_THREADS = 256;
constexpr int HC = 64;  // channels per CTA (one 128-byte panel of a bf16 C x Dk record, two of fp32)

template <class T>
struct GrLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int GLD = HC + 8;                  // padded fp32 row
  static constexpr int G = 0;                         // float [C][GLD]
  static constexpr int Q = a1k(G + C * GLD * 4);      // q     [C][HC]
  static constexpr int K = a1k(Q + C * HC * ES);      // k     [C][HC]
  static constexpr int X = a1k(K + C * HC * ES);      // query-side rows q e1
  static constexpr int XB = X + C * HC * ES;          // query-side rows beta k e1
  static constexpr int Y = a1k(XB + C * HC * ES);     // key-side rows k e2
  static constexpr int DQH = a1k(Y + C * HC * ES);    // dQ-hat   [C][HC]
  static constexpr int DBK = a1k(DQH + C * HC * ES);  // dBk      [C][HC]
  static constexpr int DKT = a1k(DBK + C * HC * ES);  // dK-tilde [C][HC]
  static constexpr int DAQ = a1k(DKT + C * HC * ES);  // dAqk [C][C]
  static constexpr int DAK = a1k(DAQ + C * C * ES);   // dAkk [C][C]
  static constexpr int BETA = a1k(DAK + C * C * ES);  // float [C]
  static constexpr int DIAG = BETA + C * 4;           // float [C] diagonal of dAqk
  static constexpr int DBS = DIAG + C * 4;            // float [2][C] dbeta partials
  static constexpr int COLS = DBS + 2 * C * 4;        // float [4][HC] K-tilde column partials
  static constexpr int GCOL = COLS + 4 * HC * 4;      // float [HC] dgam * gam
  static constexpr int GSC = GCOL + HC * 4;           // float [C] scalar decay per token
  static constexpr int BYTES = GSC + C * 4;
  static constexpr int DG = X;                        // float [C][HC] dG staging over X and XB
  static_assert(2 * C * HC * ES >= C * HC * 4 && XB - X == C * HC * ES, "dG staging spans X and XB");
};

template <class T>
using HTile = Tile<T, C, HC>;

// sum over j in [j0, j1] of dP(r, j) y(j, c) exp(G(r,c) - G(j,c)) (in-block x side)
template <class T>
__device__ __noinline__ float pw_dx(const Tile<T, C, C>* dP, const HTile<T>* ys, const float* G, int r, int c,
                                    int j0, int j1) {
  constexpr int LD = GrLayout<T>::GLD;
  const float Gr = G[r * LD + c];
  float s = 0.f;
  for (int j = j0; j <= j1; ++j)
    s = fmaf(to_f32(dP->at(r, j)) * to_f32(ys->at(j, c)), __expf(Gr - G[j * LD + c]), s);
  return s;
}
// sum over t in [t0, t1] of dP(t, j) w_t x(t, c) exp(G(t,c) - G(j,c)) (in-block y side)
template <class T>
__device__ __noinline__ float pw_dy(const Tile<T, C, C>* dP, const HTile<T>* xs, const float* w, const float* G,
                                    int j, int c, int t0, int t1) {
  constexpr int LD = GrLayout<T>::GLD;
  const float Gj = G[j * LD + c];
  float s = 0.f;
  for (int t = t0; t <= t1; ++t) {
    const float wt = w ? w[t] : 1.f;
    s = fmaf(to_f32(dP->at(t, j)) * wt * to_f32(xs->at(t, c)), __expf(G[t * LD + c] - Gj), s);
  }
  return s;
}

// bf16: two CTAs per SM; fp32 tiles take one SM's shared memory, so all registers are free
template <class T, bool PC>
__global__ void __launch_bounds__(GR_THREADS, sizeof(T) == 2 ? 2 : 1) chunk_grads_kernel(ChunkBwdArgs a) {
  pdl_wait();
  pdl_trigger();
  typedef GrLayout<T> L;
  typedef HTile<T> HT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = blockIdx.x, n = blockIdx.y, bh = blockIdx.z, b = bh / a.H, h = bh % a.H;
  const int N = a.T / C, DK = a.DK, NGRP = DK / HC;
  const size_t ch = (size_t)bh * N + n;
  const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
  const size_t rs = a.H;
  const int cbase = grp * HC;  // first channel of this CTA
  constexpr int EPC = 16 / (int)sizeof(T);
  float* Gp = reinterpret_cast<float*>(sm + L::G);
  auto Gat = [&](int r, int c) -> float& { return Gp[r * L::GLD + c]; };
  HT Qs{reinterpret_cast<T*>(sm + L::Q)};
  HT Ks{reinterpret_cast<T*>(sm + L::K)};
  HT Xs{reinterpret_cast<T*>(sm + L::X)};
  HT Ys{reinterpret_cast<T*>(sm + L::Y)};
  HT dQh{reinterpret_cast<T*>(sm + L::DQH)};
  HT dBk{reinterpret_cast<T*>(sm + L::DBK)};
  HT dKt{reinterpret_cast<T*>(sm + L::DKT)};
  Tile<T, C, C> dAq{reinterpret_cast<T*>(sm + L::DAQ)};
  Tile<T, C, C> dAk{reinterpret_cast<T*>(sm + L::DAK)};
  float* beta_s = reinterpret_cast<float*>(sm + L::BETA);
  float* diag_s = reinterpret_cast<float*>(sm + L::DIAG);
  float* db_s = reinterpret_cast<float*>(sm + L::DBS);
  float* cols_s = reinterpret_cast<float*>(sm + L::COLS);
  float* gcol_s = reinterpret_cast<float*>(sm + L::GCOL);
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* g = static_cast<const T*>(a.g);
  const T* beta = static_cast<const T*>(a.beta);

  // ---- asynchronous loads in two groups: what the cumulative decay, the row-scaled
  // operands and the score products need (per-channel g lands raw in X first), then the
  // state-product tiles that only the epilogue reads, which arrive during those phases
  T* graw = reinterpret_cast<T*>(sm + L::X);
  for (int i = tid; i < C * HC / EPC; i += GR_THREADS) {
    const int r = i / (HC / EPC), c = (i % (HC / EPC)) * EPC;
    const size_t gi = (row0 + r * rs) * DK + cbase + c;
    cp_async16(Qs.ptr(r, c), q + gi);
    cp_async16(Ks.ptr(r, c), k + gi);
    if (PC) cp_async16(graw + r * HC + c, g + gi);
  }
  {
    if (tid < HC / 4) cp_async16(gcol_s + 4 * tid, a.ws.dgam + ch * DK + cbase + 4 * tid);  // dgam, scaled below
    const T* sa = static_cast<const T*>(a.ws.daqk) + ch * (C * C);
    const T* sk = static_cast<const T*>(a.ws.dakk) + ch * (C * C);
    for (int i = tid; i < C * C / EPC; i += GR_THREADS) {
      cp_async16(dAq.p + i * EPC, sa + i * EPC);
      cp_async16(dAk.p + i * EPC, sk + i * EPC);
    }
  }
  cp_async_commit();
  {
    // the C x Dk records are column panels of 128 bytes: this CTA's 64 columns are contiguous
    const size_t pan = ch * (C * (size_t)DK) + (size_t)grp * C * HC;
    const T* s1 = static_cast<const T*>(a.ws.dqh) + pan;
    const T* s2 = static_cast<const T*>(a.ws.dbk) + pan;
    const T* s3 = static_cast<const T*>(a.ws.dkt) + pan;
    for (int i = tid; i < C * HC / EPC; i += GR_THREADS) {
      cp_async16(dQh.p + i * EPC, s1 + i * EPC);
      cp_async16(dBk.p + i * EPC, s2 + i * EPC);
      cp_async16(dKt.p + i * EPC, s3 + i * EPC);
    }
  }
  cp_async_commit();
  float* gsc = reinterpret_cast<float*>(sm + L::GSC);
  if (tid < C) {
    beta_s[tid] = to_f32(beta[row0 + tid * rs]);
    if (!PC) gsc[tid] = to_f32(g[row0 + tid * rs]);
  }
  cp_async_wait<1>();
  __syncthreads();
  if (tid < C) {  // the diagonal of dAqk only feeds dq and dk (its dG terms cancel exactly)
    diag_s[tid] = to_f32(dAq.at(tid, tid));
    dAq.at(tid, tid) = from_f32<T>(0.f);
  }
  // cumulative log-decay (fp32): lanes 2c and 2c + 1 take channel c, one 32-row block
  // each in registers; the second block adds the first block's total (from its partner)
  static_assert(2 * HC <= GR_THREADS, "two threads per channel");
  if (tid < 2 * HC) {
    const int c = tid >> 1, hb = tid & 1, r0 = hb * BLK;
    float v[BLK];
#pragma unroll
    for (int i = 0; i < BLK; ++i) v[i] = PC ? to_f32(graw[(r0 + i) * HC + c]) : gsc[r0 + i];
#pragma unroll
    for (int i = 1; i < BLK; ++i) v[i] += v[i - 1];
    const float base = __shfl_sync(0xffffffffu, v[BLK - 1], lane & ~1);
#pragma unroll
    for (int i = 0; i < BLK; ++i) Gat(r0 + i, c) = hb ? v[i] + base : v[i];
  }
  __syncthreads();
  // One decay per head (PC false) without the pairwise flag: the mask form. The score
  // gradients are (dP (*) E) y and (dP (*) E)^T x with E[t][j] = exp(G_t - G_j) <= 1,
  // applied to the dP tiles, and the operands are q, beta k and k themselves.
  const bool force = (a.flags & 1) != 0;
  const bool mask_form = !PC && !force;
  bool u1 = false, u2 = false;
  for (int c = tid; c < HC; c += GR_THREADS) {
    if (PC) {
      u1 |= !(Gat(0, c) - Gat(BLK - 1, c) <= SAFE_SPREAD);
      u2 |= !(Gat(BLK - 1, c) - Gat(C - 1, c) <= SAFE_SPREAD);
    }
    gcol_s[c] *= __expf(Gat(C - 1, c));  // dgam * gam
  }
  if (!PC && tid < C) gsc[tid] = Gat(tid, 0);  // one decay per head: G per token, read by the mask form
  auto gsc_cum = [&](int r) { return gsc[r]; };
  const bool unsafe1 = __syncthreads_or(u1 || force) != 0;
  const bool unsafe2 = __syncthreads_or(u2 || force) != 0;

  // row-scaled operands, one pass: X = q e1, XB = beta k e1 (query side), Y = k e2 (key side),
  // with e1 = exp(G - G_b), e2 = exp(G_b - G) about the block boundary b
  HT XBs{reinterpret_cast<T*>(sm + L::XB)};
  static_assert(C * (HC / 4) % GR_THREADS == 0, "whole passes");
#pragma unroll
  for (int i = tid; i < C * (HC / 4); i += GR_THREADS) {
    const int r = i / (HC / 4), c0 = (i % (HC / 4)) * 4;
    float kv[4], qv[4], G[4], Gb[4], xq[4], xb[4], yk[4];
    ld4(kv, Ks.ptr(r, c0));
    ld4(qv, Qs.ptr(r, c0));
    ld4(G, &Gat(r, c0));
    ld4(Gb, &Gat(BLK - 1, c0));
    const bool dead_x = r < BLK && unsafe1, dead_y = r >= BLK && unsafe2;
    const float br = beta_s[r];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float d = G[e] - Gb[e];
      const float e1 = mask_form ? 1.f : dead_x ? 0.f : __expf(d);
      const float e2 = mask_form ? 1.f : dead_y ? 0.f : __expf(-d);
      xq[e] = qv[e] * e1;
      xb[e] = br * kv[e] * e1;
      yk[e] = kv[e] * e2;
    }
    st4(Xs.ptr(r, c0), xq);
    st4(XBs.ptr(r, c0), xb);
    st4(Ys.ptr(r, c0), yk);
  }
  if (mask_form) {  // dP (*) E on both score tiles (strictly lower part; the diagonal has E = 1)
    for (int i = tid; i < C * C / 2; i += GR_THREADS) {
      const int t = i / (C / 2), j = 2 * (i % (C / 2));
      if (j < t) {
        const float Gt = Gat(t, 0);
        const float e0 = __expf(Gt - gsc_cum(j)), e1 = j + 1 < t ? __expf(Gt - gsc_cum(j + 1)) : 0.f;
        const float2 fq = ld2(dAq.ptr(t, j)), fk = ld2(dAk.ptr(t, j));
        store2(dAq.ptr(t, j), fq.x * e0, j + 1 < t ? fq.y * e1 : fq.y);
        store2(dAk.ptr(t, j), fk.x * e0, j + 1 < t ? fk.y * e1 : fk.y);
      }
    }
  }
  __syncthreads();

  // warp w: rows m0 .. m0 + 15, channels c0 .. c0 + 31 of this group
  const int m0 = 16 * (warp & 3), cq = warp >> 2, c0 = 32 * cq;
  const bool blk1 = m0 < BLK;
  const bool pw_rows = blk1 ? unsafe1 : unsafe2;  // in-block part of these rows is pairwise
  // x side: dP Y over key columns [0, BLK) for block-1 rows, [0, C) otherwise;
  // y side: dP^T X over query rows [0, C) for block-1 rows, [BLK, C) otherwise
  float axB[1][4][4], ayB[1][4][4], axA[1][4][4], ayA[1][4][4];
  zero(axB);
  zero(ayB);
  zero(axA);
  zero(ayA);
  if (blk1) {
    if (!unsafe1) {
      Gemm<T>::template runk<1, 4, 0, BLK>(axB, aview<false>(dAk), bview<true>(Ys), m0, c0, lane);
      Gemm<T>::template runk<1, 4, 0, BLK>(axA, aview<false>(dAq), bview<true>(Ys), m0, c0, lane);
    }
    Gemm<T>::template runk<1, 4, 0, C>(ayB, aview<true>(dAk), bview<true>(XBs), m0, c0, lane);
    Gemm<T>::template runk<1, 4, 0, C>(ayA, aview<true>(dAq), bview<true>(Xs), m0, c0, lane);
  } else {
    Gemm<T>::template runk<1, 4, 0, C>(axB, aview<false>(dAk), bview<true>(Ys), m0, c0, lane);
    Gemm<T>::template runk<1, 4, 0, C>(axA, aview<false>(dAq), bview<true>(Ys), m0, c0, lane);
    if (!unsafe2) {
      Gemm<T>::template runk<1, 4, BLK, C>(ayB, aview<true>(dAk), bview<true>(XBs), m0, c0, lane);
      Gemm<T>::template runk<1, 4, BLK, C>(ayA, aview<true>(dAq), bview<true>(Xs), m0, c0, lane);
    }
  }

  cp_async_wait<0>();  // the state-product tiles
  __syncthreads();  // every warp is done reading X and XB: dG is staged there
  // one epilogue per element pair: every gradient term of (r, c) and (r, c + 1)
  float* dGs = reinterpret_cast<float*>(sm + L::DG);
  float dbp[2] = {0.f, 0.f}, colp[4][2];
  // FAST (both blocks safe): no pairwise rows, and Gam = exp(G_b) e1, exp(G_C - G) =
  // exp(G_C - G_b) e2 with every factor in fp32 range, two exponentials per element fewer
  auto epilogue = [&](auto fast_tag, auto mask_tag) {
    constexpr bool FAST = decltype(fast_tag)::value;
    constexpr bool MASK = decltype(mask_tag)::value;  // scalar decay: E already in dP
    const int bs = blk1 ? 0 : BLK;
    const bool skip_x = !FAST && blk1 && unsafe1, skip_y = !FAST && !blk1 && unsafe2;
    float rgm[2] = {0.f, 0.f}, rkd[2] = {0.f, 0.f};  // MASK: Gam and exp(G_C - G) of this thread's two rows
    if (MASK)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const float Gr = Gat(m0 + frag_row(lane, 2 * h2), 0);
        rgm[h2] = __expf(Gr);
        rkd[h2] = __expf(Gat(C - 1, 0) - Gr);
      }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int c = c0 + 8 * nt + 2 * (lane & 3);
      const float2 gb = *reinterpret_cast<const float2*>(&Gat(BLK - 1, c));
      const float2 gc = *reinterpret_cast<const float2*>(&Gat(C - 1, c));
      float eb[2] = {0.f, 0.f}, ecb[2] = {0.f, 0.f};
      if (FAST && !MASK) {
        eb[0] = __expf(gb.x);
        eb[1] = __expf(gb.y);
        ecb[0] = __expf(gc.x - gb.x);
        ecb[1] = __expf(gc.y - gb.y);
      }
      colp[nt][0] = colp[nt][1] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int r = m0 + frag_row(lane, e);
        const float2 G2 = *reinterpret_cast<const float2*>(&Gat(r, c));
        const float2 k2 = ld2(Ks.ptr(r, c)), q2 = ld2(Qs.ptr(r, c)), h2 = ld2(dQh.ptr(r, c));
        const float2 b2 = ld2(dBk.ptr(r, c)), t2 = ld2(dKt.ptr(r, c));
        const float br = beta_s[r], dg = diag_s[r];
        float oq[2], ok[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float G = u ? G2.y : G2.x, Gb = u ? gb.y : gb.x, GC = u ? gc.y : gc.x;
          const float kf = u ? k2.y : k2.x, qf = u ? q2.y : q2.x;
          const float dqh = u ? h2.y : h2.x, dbk = u ? b2.y : b2.x, dkt = u ? t2.y : t2.x;
          const float e1 = MASK ? 1.f : __expf(G - Gb), e2 = MASK ? 1.f : __expf(Gb - G);
          const float gm = MASK ? rgm[e >> 1] : FAST ? eb[u] * e1 : __expf(G);
          const float kd = MASK ? rkd[e >> 1] : FAST ? ecb[u] * e2 : __expf(GC - G);
          float dxb = skip_x ? 0.f : axB[0][nt][e + u] * e1;  // Akk family, dP = dAkk
          float dyb = skip_y ? 0.f : ayB[0][nt][e + u] * e2;
          float dxa = skip_x ? 0.f : axA[0][nt][e + u] * e1;  // Aqk family
          float dya = skip_y ? 0.f : ayA[0][nt][e + u] * e2;
          if (!FAST && pw_rows) {
            dxb += pw_dx(&dAk, &Ks, Gp, r, c + u, bs, r);
            dyb += pw_dy(&dAk, &Ks, beta_s, Gp, r, c + u, r, bs + BLK - 1);
            dxa += pw_dx(&dAq, &Ks, Gp, r, c + u, bs, r);
            dya += pw_dy(&dAq, &Qs, nullptr, Gp, r, c + u, r, bs + BLK - 1);
          }
          const float khat = gm * kf, ktil = kd * kf, dkh = br * dbk;
          oq[u] = dqh * gm + dxa + dg * kf;
          ok[u] = br * dxb + dyb + dya + dg * qf + dkh * gm + dkt * kd;
          dGs[r * HC + c + u] = kf * (br * dxb - dyb - dya) + qf * (dxa + dqh * gm) + dkh * khat - dkt * ktil;
          dbp[e >> 1] += kf * dxb + dbk * khat;
          colp[nt][u] += dkt * ktil;
        }
        // staged over this thread's own dQ-hat / dBk elements, stored row-wise below
        store2(dQh.ptr(r, c), oq[0], oq[1]);
        store2(dBk.ptr(r, c), ok[0], ok[1]);
      }
    }
  };
  if (mask_form)
    epilogue(BoolTag<true>{}, BoolTag<true>{});
  else if (!(unsafe1 || unsafe2))
    epilogue(BoolTag<true>{}, BoolTag<false>{});
  else
    epilogue(BoolTag<false>{}, BoolTag<false>{});
  // column sums over this warp's 16 rows (lanes sharing a column differ in bits 2..4)
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float x = colp[nt][u];
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      x += __shfl_xor_sync(0xffffffffu, x, 8);
      x += __shfl_xor_sync(0xffffffffu, x, 16);
      if (lane < 4) cols_s[(warp & 3) * HC + c0 + 8 * nt + 2 * lane + u] = x;
    }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    dbp[i] += __shfl_xor_sync(0xffffffffu, dbp[i], 1);
    dbp[i] += __shfl_xor_sync(0xffffffffu, dbp[i], 2);
  }
  if ((lane & 3) == 0) {
    db_s[cq * C + m0 + (lane >> 2)] = dbp[0];
    db_s[cq * C + m0 + (lane >> 2) + 8] = dbp[1];
  }
  __syncthreads();  // dG, column and dbeta partials, dq and dk tiles complete
  if (tid < C) a.ws.dbpart[(ch * 2 + grp) * C + tid] = db_s[tid] + db_s[C + tid];
  {
    T* dq = static_cast<T*>(a.dq);
    T* dk = static_cast<T*>(a.dk);
    for (int i = tid; i < C * HC / EPC; i += GR_THREADS) {
      const int r = i / (HC / EPC), cc = (i % (HC / EPC)) * EPC;
      const size_t gi = (row0 + r * rs) * DK + cbase + cc;
      copy16(dq + gi, dQh.ptr(r, cc));
      copy16(dk + gi, dBk.ptr(r, cc));
    }
  }
  // reverse cumulative sum per channel; the last row also gets the K-tilde column sum and
  // dgam * gam (both are derivatives with respect to G at the chunk's last token). Lanes
  // 2c and 2c + 1 take channel c, one 32-row block each; the first block adds the
  // second block's total (from its partner)
  if (tid < 2 * HC) {
    const int c = tid >> 1, hi = tid & 1, r0 = hi * BLK;
    float v[BLK];
#pragma unroll
    for (int i = 0; i < BLK; ++i) v[i] = dGs[(r0 + i) * HC + c];
    float s = hi ? (cols_s[c] + cols_s[HC + c] + cols_s[2 * HC + c] + cols_s[3 * HC + c] + gcol_s[c]) : 0.f;
#pragma unroll
    for (int i = BLK - 1; i >= 0; --i) {
      s += v[i];
      v[i] = s;
    }
    const float top = __shfl_sync(0xffffffffu, v[0], lane | 1);  // rows >= BLK summed (with the extras)
#pragma unroll
    for (int i = 0; i < BLK; ++i) dGs[(r0 + i) * HC + c] = hi ? v[i] : v[i] + top;
  }
  __syncthreads();
  T* dg = static_cast<T*>(a.dg);
  if (PC) {
    for (int i = tid; i < C * HC / EPC; i += GR_THREADS) {
      const int r = i / (HC / EPC), cc = (i % (HC / EPC)) * EPC;
      __align__(16) T o[EPC];
#pragma unroll
      for (int e = 0; e < EPC; ++e) o[e] = from_f32<T>(dGs[r * HC + cc + e]);
      copy16(dg + (row0 + r * rs) * DK + cbase + cc, o);
    }
  } else {
    for (int r = warp; r < C; r += GR_THREADS / 32) {
      float s = dGs[r * HC + lane] + dGs[r * HC + lane + 32];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (lane == 0) a.ws.dgpart[(ch * 2 + grp) * C + r] = s;
    }
  }
  (void)NGRP;
}

// dbeta = dbeta_v + the channel groups' partials (and scalar-decay dg), fixed order.
template <class T, bool PC>
__global__ void chunk_bwd_finalize_kernel(ChunkBwdArgs a) {
  pdl_wait();
  pdl_trigger();
  const size_t total = (size_t)a.B * a.H * a.T;
  const int N = a.T / C, NGRP = a.DK / HC;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i % C);
    const size_t ch = i / C;  // (bh, n) record
    const int n = (int)(ch % N);
    const int bh = (int)(ch / N), b = bh / a.H, h = bh % a.H;
    const size_t row = ((size_t)b * a.T + (size_t)n * C + t) * a.H + h;
    float db = a.ws.dbv[ch * C + t] + a.ws.dbpart[(ch * 2) * C + t];
    if (NGRP > 1) db += a.ws.dbpart[(ch * 2 + 1) * C + t];
    static_cast<T*>(a.dbeta)[row] = from_f32<T>(db);
    if (!PC) {
      float s = a.ws.dgpart[(ch * 2) * C + t];
      if (NGRP > 1) s += a.ws.dgpart[(ch * 2 + 1) * C + t];
      static_cast<T*>(a.dg)[row] = from_f32<T>(s);
    }
  }
}

template <class T>
cudaError_t launch_grads_t(const ChunkBwdArgs& a, cudaStream_t s) {
  const int N = a.T / C, BH = a.B * a.H;
  const int bytes = GrLayout<T>::BYTES + 1024;
  auto kern = a.per_channel ? chunk_grads_kernel<T, true> : chunk_grads_kernel<T, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  prof_mark(K_GRADS, s, true);
  if ((e = launch_pdl(kern, dim3(a.DK / HC, N, BH), dim3(GR_THREADS), bytes, s, a)) != cudaSuccess) return e;
  prof_mark(K_GRADS, s, false);
  const size_t total = (size_t)BH * a.T;
  const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  prof_mark(K_FINALIZE, s, true);
  e = launch_pdl(a.per_channel ? chunk_bwd_finalize_kernel<T, true> : chunk_bwd_finalize_kernel<T, false>,
                 dim3(blocks), dim3(256), 0, s, a);
  prof_mark(K_FINALIZE, s, false);
  return e;
}

}  // namespace

cudaError_t launch_chunk_grads(const ChunkBwdArgs& a, cudaStream_t s) {
  if (a.B * a.H == 0 || a.T == 0) return cudaSuccess;
  return a.bf16 ? launch_grads_t<bf16>(a, s) : launch_grads_t<float>(a, s);
}

}  // namespace gdn
