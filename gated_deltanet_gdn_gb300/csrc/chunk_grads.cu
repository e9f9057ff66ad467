// Chunk-parallel gradients of the chunked gated delta rule backward (bf16 operands).
//
// One CTA per (chunk, batch, head). Inputs: q, k, v, g, beta of the chunk, the WY
// inverse T saved by the forward, and the reverse scan's dU plus the state products
// dW, dQ-hat, dK-tilde, dAqk, dgam (chunk_bwd.cu). The algebra is listed at the top of
// chunk_bwd.cu. Score gradients reuse the forward's row-scaled tiles (boundary-split
// factorisation, marin.community note "factoring GDN-2 decay on TPU", section
// Approach); blocks whose decay spread leaves the safe range take the pairwise sums.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int GR_THREADS = 256;

// ------------------------------------------------------------------ chunk gradients
template <int DK, int DV>
struct GrLayout {
  static constexpr int MX = DK > DV ? DK : DV;
  static constexpr int G = 0;                        // float [C][DK]
  static constexpr int Q = a1k(G + C * DK * 4);      // q
  static constexpr int K = a1k(Q + C * DK * 2);      // k
  static constexpr int V = a1k(K + C * DK * 2);      // v
  static constexpr int TM = a1k(V + C * DV * 2);     // T
  static constexpr int DW = a1k(TM + C * C * 2);     // dW, later x-side scaled k
  static constexpr int DU = a1k(DW + C * DK * 2);    // dU (NT slices), later Y1   [C][MX]
  static constexpr int BUF = a1k(DU + C * MX * 2);   // Bk, Bv, later Y2   [C][MX]
  static constexpr int DT = a1k(BUF + C * MX * 2);   // dT, X = T^T dT; later Pkk (fp32), Xq
  static constexpr int XS = DT + C * C * 2;
  static constexpr int DPKK = a1k(XS + C * C * 2);   // beta * dAkk
  static constexpr int DAQK = a1k(DPKK + C * C * 2); // dAqk (scaled, masked)
  static constexpr int BETA = a1k(DAQK + C * C * 2); // float [C]
  static constexpr int DB = BETA + C * 4;            // float [2][C] dbeta halves
  static constexpr int DIAG = DB + 2 * C * 4;        // float [C] diagonal of dAqk
  static constexpr int BYTES = DIAG + C * 4;
  static_assert(BUF - DW >= C * DK * 4, "dG staging spans the dW and dU regions");
};

template <int DK, int DV, bool PC>
__global__ void __launch_bounds__(GR_THREADS) chunk_grads_kernel(ChunkBwdArgs a) {
  typedef bf16 T;
  typedef GrLayout<DK, DV> L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  const int N = a.T / C;
  const size_t ch = (size_t)bh * N + n;
  const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
  const size_t rs = a.H;
  constexpr int EPC = 8;
  FTile<C, DK> Gs{reinterpret_cast<float*>(sm + L::G)};
  Tile<T, C, DK> Qs{reinterpret_cast<T*>(sm + L::Q)};
  Tile<T, C, DK> Ks{reinterpret_cast<T*>(sm + L::K)};
  Tile<T, C, DV> Vs{reinterpret_cast<T*>(sm + L::V)};
  Tile<T, C, C> Ts{reinterpret_cast<T*>(sm + L::TM)};
  Tile<T, C, DK> dWs{reinterpret_cast<T*>(sm + L::DW)};
  TTile<T, C, DV, NT> dUs{reinterpret_cast<T*>(sm + L::DU)};
  Tile<T, C, C> dTs{reinterpret_cast<T*>(sm + L::DT)};
  Tile<T, C, C> Xs{reinterpret_cast<T*>(sm + L::XS)};
  Tile<T, C, C> dPs{reinterpret_cast<T*>(sm + L::DPKK)};
  Tile<T, C, C> dAs{reinterpret_cast<T*>(sm + L::DAQK)};
  float* beta_s = reinterpret_cast<float*>(sm + L::BETA);
  float* db_s = reinterpret_cast<float*>(sm + L::DB);
  float* diag_s = reinterpret_cast<float*>(sm + L::DIAG);
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* g = static_cast<const T*>(a.g);
  const T* beta = static_cast<const T*>(a.beta);

  // ---- loads
  for (int i = tid; i < C * DK / EPC; i += GR_THREADS) {
    const int r = i / (DK / EPC), c = (i % (DK / EPC)) * EPC;
    const size_t gi = (row0 + r * rs) * DK + c;
    cp_async16(Qs.ptr(r, c), q + gi);
    cp_async16(Ks.ptr(r, c), k + gi);
  }
  for (int i = tid; i < C * DV / EPC; i += GR_THREADS) {
    const int r = i / (DV / EPC), c = (i % (DV / EPC)) * EPC;
    cp_async16(Vs.ptr(r, c), v + (row0 + r * rs) * DV + c);
  }
  {
    const T* st = static_cast<const T*>(a.res.tmat) + ch * (C * C);
    const T* sa = static_cast<const T*>(a.ws.daqk) + ch * (C * C);
    for (int i = tid; i < C * C / EPC; i += GR_THREADS) {
      cp_async16(Ts.p + i * EPC, st + i * EPC);
      cp_async16(dAs.p + i * EPC, sa + i * EPC);
    }
    const T* sw = static_cast<const T*>(a.ws.dw) + ch * (C * DK);
    for (int i = tid; i < C * DK / EPC; i += GR_THREADS) cp_async16(dWs.p + i * EPC, sw + i * EPC);
    const T* su = static_cast<const T*>(a.ws.du) + ch * (C * DV);
    for (int i = tid; i < C * DV / EPC; i += GR_THREADS) cp_async16(dUs.p + i * EPC, su + i * EPC);
  }
  cp_async_commit();
  if (PC) {
    for (int i = tid; i < C * DK / EPC; i += GR_THREADS) {
      const int r = i / (DK / EPC), c = (i % (DK / EPC)) * EPC;
      __align__(16) T gv[EPC];
      copy16(gv, g + (row0 + r * rs) * DK + c);
#pragma unroll
      for (int e = 0; e < EPC; ++e) Gs.at(r, c + e) = to_f32(gv[e]);
    }
  } else {
    for (int i = tid; i < C * DK; i += GR_THREADS) Gs.at(i / DK, i % DK) = to_f32(g[row0 + (i / DK) * rs]);
  }
  if (tid < C) beta_s[tid] = to_f32(beta[row0 + tid * rs]);
  cp_async_wait<0>();
  __syncthreads();
  // The diagonal of dAqk (decay factor 1) only feeds dq and dk: its two dG terms
  // q_t dP_tt k_t and k_t dP_tt q_t cancel exactly, so it is taken out of the
  // row-scaled products (where bf16 rounding would leave a residual) and added back below.
  if (tid < C) {
    diag_s[tid] = to_f32(dAs.at(tid, tid));
    dAs.at(tid, tid) = from_f32<T>(0.f);
  }
  for (int c = tid; c < DK; c += GR_THREADS) {
    float s = 0.f;
    for (int r = 0; r < C; ++r) {
      s += Gs.at(r, c);
      Gs.at(r, c) = s;
    }
  }
  __syncthreads();
  const bool force = (a.flags & 1) != 0;
  bool u1 = false, u2 = false;
  for (int c = tid; c < DK; c += GR_THREADS) {
    u1 |= !(-Gs.at(BLK - 1, c) <= SAFE_SPREAD);
    u2 |= !(Gs.at(BLK - 1, c) - Gs.at(C - 1, c) <= SAFE_SPREAD);
  }
  const bool unsafe1 = __syncthreads_or(u1 || force) != 0;
  const bool unsafe2 = __syncthreads_or(u2 || force) != 0;

  // warp partition: rows m0 .. m0 + 15, column half hf
  const int m0 = 16 * (warp & 3), hf = warp >> 2;
  constexpr int NWK = DK / 16, NWV = DV / 16;  // n8 tiles per warp for C x DK / C x DV outputs
  const int ck0 = hf * (DK / 2), cv0 = hf * (DV / 2), cc0 = hf * 32;
  float db[2] = {0.f, 0.f};  // dbeta partials for rows m0 + g and m0 + g + 8

  // ---- Bk = beta Gam k
  Tile<T, C, DK> Bk{reinterpret_cast<T*>(sm + L::BUF)};
  Tile<T, C, DV> Bv{reinterpret_cast<T*>(sm + L::BUF)};
  for (int i = tid; i < C * DK; i += GR_THREADS) {
    const int r = i / DK, c = i % DK;
    Bk.at(r, c) = from_f32<T>(beta_s[r] * __expf(Gs.at(r, c)) * to_f32(Ks.at(r, c)));
  }
  __syncthreads();
  float dT[1][4][4];
  zero(dT);
  Gemm<T>::template run<1, 4>(dT, aview<false>(dWs), bview<false>(Bk), m0, cc0, 0, DK, lane);
  __syncthreads();
  for (int i = tid; i < C * DV; i += GR_THREADS) {
    const int r = i / DV, c = i % DV;
    Bv.at(r, c) = from_f32<T>(beta_s[r] * to_f32(Vs.at(r, c)));
  }
  __syncthreads();
  Gemm<T>::template run<1, 4>(dT, aview<false>(dUs), bview<false>(Bv), m0, cc0, 0, DV, lane);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      dTs.at(m0 + frag_row(lane, e), cc0 + 8 * nt + frag_col(lane, e)) = from_f32<T>(dT[0][nt][e]);

  // ---- dv = beta (T^T dU)
  {
    float acc[1][NWV][4];
    zero(acc);
    Gemm<T>::template run<1, NWV>(acc, aview<true>(Ts), bview<true>(dUs), m0, cv0, 0, C, lane);
    T* dv = static_cast<T*>(a.dv);
#pragma unroll
    for (int nt = 0; nt < NWV; ++nt)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int r = m0 + frag_row(lane, e), c = cv0 + 8 * nt + frag_col(lane, e);
        db[e >> 1] += acc[0][nt][e] * to_f32(Vs.at(r, c)) + acc[0][nt][e + 1] * to_f32(Vs.at(r, c + 1));
        store2(dv + (row0 + r * rs) * DV + c, beta_s[r] * acc[0][nt][e], beta_s[r] * acc[0][nt][e + 1]);
      }
  }
  // ---- dBk = T^T dW: dK-hat = beta dBk; dk += dK-hat Gam; dG += dK-hat K-hat
  float dq_acc[NWK][4], dk_acc[NWK][4], dG_acc[NWK][4];
  {
    float acc[1][NWK][4];
    zero(acc);
    Gemm<T>::template run<1, NWK>(acc, aview<true>(Ts), bview<true>(dWs), m0, ck0, 0, C, lane);
#pragma unroll
    for (int nt = 0; nt < NWK; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + frag_row(lane, e), c = ck0 + 8 * nt + frag_col(lane, e);
        const float gm = __expf(Gs.at(r, c));
        const float khat = gm * to_f32(Ks.at(r, c));
        db[e >> 1] += acc[0][nt][e] * khat;
        const float dkh = beta_s[r] * acc[0][nt][e];
        dq_acc[nt][e] = 0.f;
        dk_acc[nt][e] = dkh * gm;
        dG_acc[nt][e] = dkh * khat;
      }
  }
  __syncthreads();  // dT complete; dW and dU no longer needed after this point except dUs reads done
  // ---- X = T^T dT ; dAkk = -(X T^T) masked strict
  {
    float acc[1][4][4];
    zero(acc);
    Gemm<T>::template run<1, 4>(acc, aview<true>(Ts), bview<true>(dTs), m0, cc0, 0, C, lane);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        Xs.at(m0 + frag_row(lane, e), cc0 + 8 * nt + frag_col(lane, e)) = from_f32<T>(acc[0][nt][e]);
  }
  // x-side scaled keys (into dW), Y1 (into dU), Y2 (into BUF)
  Tile<T, C, DK> Xk{reinterpret_cast<T*>(sm + L::DW)};
  Tile<T, BLK, DK> Y1{reinterpret_cast<T*>(sm + L::DU)};
  Tile<T, C, DK> Y2{reinterpret_cast<T*>(sm + L::BUF)};
  __syncthreads();
  float dAkk[1][4][4];
  zero(dAkk);
  Gemm<T>::template run<1, 4>(dAkk, aview<false>(Xs), bview<false>(Ts), m0, cc0, 0, C, lane);
  for (int i = tid; i < C * DK; i += GR_THREADS) {
    const int r = i / DK, c = i % DK;
    const float G = Gs.at(r, c), Gb = Gs.at(BLK - 1, c), kf = to_f32(Ks.at(r, c));
    Xk.at(r, c) = from_f32<T>(kf * __expf(r < BLK ? G : G - Gb));
    Y2.at(r, c) = from_f32<T>((r < BLK || !unsafe2) ? kf * __expf(Gb - G) : 0.f);
    if (r < BLK) Y1.at(r, c) = from_f32<T>(unsafe1 ? 0.f : kf * __expf(-G));
  }
  __syncthreads();  // X consumed; DT/XS region becomes Pkk
  FTile<C, C> Pk{reinterpret_cast<float*>(sm + L::DT)};
  {
    float acc[1][4][4];
    zero(acc);
    const bool blk1 = m0 < BLK;
    if (!(blk1 && (unsafe1 || hf == 1))) {
      if (blk1) Gemm<T>::template run<1, 4>(acc, aview<false>(Xk), bview<false>(Y1), m0, 0, 0, DK, lane);
      else Gemm<T>::template run<1, 4>(acc, aview<false>(Xk), bview<false>(Y2), m0, cc0, 0, DK, lane);
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + frag_row(lane, e), j = cc0 + 8 * nt + frag_col(lane, e);
        Pk.at(r, j) = j < r ? acc[0][nt][e] : 0.f;
      }
  }
  __syncthreads();
  if (unsafe1 || unsafe2) {  // pairwise in-block scores, four lanes per pair
    for (int blk = 0; blk < 2; ++blk) {
      if (!(blk == 0 ? unsafe1 : unsafe2)) continue;
      const int bs = blk * BLK;
      constexpr int NPAIR = BLK * (BLK - 1) / 2;  // strict triangle
      for (int base = 0; base < NPAIR; base += 8 * (GR_THREADS / 32)) {
        const int p = base + warp * 8 + (lane >> 2), quarter = lane & 3;
        const bool valid = p < NPAIR;
        int i = 1, j = 0;
        float sk = 0.f;
        if (valid) {
          int r = (int)((sqrtf(8.f * p + 1.f) + 1.f) * 0.5f);  // strict: p = i(i-1)/2 + j
          while (r * (r - 1) / 2 > p) --r;
          while ((r + 1) * r / 2 <= p) ++r;
          i = r;
          j = p - r * (r - 1) / 2;
          for (int c = quarter * (DK / 4); c < (quarter + 1) * (DK / 4); ++c)
            sk = fmaf(to_f32(Ks.at(bs + i, c)), to_f32(Ks.at(bs + j, c)) * __expf(Gs.at(bs + i, c) - Gs.at(bs + j, c)), sk);
        }
        sk += __shfl_xor_sync(0xffffffffu, sk, 1);
        sk += __shfl_xor_sync(0xffffffffu, sk, 2);
        if (valid && quarter == 0) Pk.at(bs + i, bs + j) = sk;
      }
    }
    __syncthreads();
  }
  // dbeta += rowsum(dAkk * Pkk); dPkk = beta dAkk
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = m0 + frag_row(lane, e), j = cc0 + 8 * nt + frag_col(lane, e);
      const float d = j < r ? -dAkk[0][nt][e] : 0.f;
      db[e >> 1] += d * Pk.at(r, j);
      dPs.at(r, j) = from_f32<T>(beta_s[r] * d);
    }
  __syncthreads();  // Pkk consumed: DT/XS region becomes the query-side scaled q
  Tile<T, C, DK> Xq{reinterpret_cast<T*>(sm + L::DT)};
  for (int i = tid; i < C * DK; i += GR_THREADS) {
    const int r = i / DK, c = i % DK;
    const float G = Gs.at(r, c);
    Xq.at(r, c) = from_f32<T>(to_f32(Qs.at(r, c)) * __expf(r < BLK ? G : G - Gs.at(BLK - 1, c)));
  }
  __syncthreads();

  // ---- score backward. x side: dx_t = f_t * sum_j dP[t,j] Y_j ; y side: dy_j = sum over
  // query blocks of f'_j * sum_t dP[t,j] X_t (row-scaled tiles as in the forward).
  auto score_bwd = [&](const Tile<T, C, C>& dP, const Tile<T, C, DK>& Xx, bool x_is_q, bool strict) {
    float acc[1][NWK][4];
    // dx
    zero(acc);
    const bool blk1 = m0 < BLK;
    if (blk1) {
      if (!unsafe1) Gemm<T>::template run<1, NWK>(acc, aview<false>(dP), bview<true>(Y1), m0, ck0, 0, BLK, lane);
    } else {
      Gemm<T>::template run<1, NWK>(acc, aview<false>(dP), bview<true>(Y2), m0, ck0, 0, C, lane);
    }
#pragma unroll
    for (int nt = 0; nt < NWK; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + frag_row(lane, e), c = ck0 + 8 * nt + frag_col(lane, e);
        const float G = Gs.at(r, c);
        float dx = acc[0][nt][e] * __expf(blk1 ? G : G - Gs.at(BLK - 1, c));
        if (blk1 ? unsafe1 : unsafe2) {  // in-block part, pairwise
          const int bs = blk1 ? 0 : BLK, jmax = strict ? r - 1 : r;
#pragma unroll 1
          for (int j = bs; j <= jmax; ++j)
            dx = fmaf(to_f32(dP.at(r, j)) * to_f32(Ks.at(j, c)), __expf(G - Gs.at(j, c)), dx);
        }
        const float xv = to_f32(x_is_q ? Qs.at(r, c) : Ks.at(r, c));
        if (x_is_q) dq_acc[nt][e] += dx; else dk_acc[nt][e] += dx;
        dG_acc[nt][e] += xv * dx;
      }
    // dy: part from second-block queries (t in 32..63), then first-block queries (t < 32)
    zero(acc);
    if (!(m0 >= BLK && unsafe2))
      Gemm<T>::template run<1, NWK>(acc, aview<true>(dP), bview<true>(Xx), m0, ck0, BLK, C, lane);
    float acc1[1][NWK][4];
    zero(acc1);
    if (m0 < BLK && !unsafe1)
      Gemm<T>::template run<1, NWK>(acc1, aview<true>(dP), bview<true>(Xx), m0, ck0, 0, BLK, lane);
#pragma unroll
    for (int nt = 0; nt < NWK; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = m0 + frag_row(lane, e), c = ck0 + 8 * nt + frag_col(lane, e);
        const float G = Gs.at(j, c), Gb = Gs.at(BLK - 1, c);
        float dy = 0.f;
        if (!(j >= BLK && unsafe2)) dy = acc[0][nt][e] * __expf(Gb - G);
        if (j < BLK && !unsafe1) dy = fmaf(acc1[0][nt][e], __expf(-G), dy);
        const bool up = j < BLK ? unsafe1 : unsafe2;
        if (up) {
          const int be = j < BLK ? BLK : C, tmin = strict ? j + 1 : j;
#pragma unroll 1
          for (int t = tmin; t < be; ++t) {
            const float xv = to_f32(x_is_q ? Qs.at(t, c) : Ks.at(t, c));
            dy = fmaf(to_f32(dP.at(t, j)) * xv, __expf(Gs.at(t, c) - G), dy);
          }
        }
        dk_acc[nt][e] += dy;
        dG_acc[nt][e] -= to_f32(Ks.at(j, c)) * dy;
      }
  };
  score_bwd(dAs, Xq, true, false);
  score_bwd(dPs, Xk, false, true);
#pragma unroll
  for (int nt = 0; nt < NWK; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = m0 + frag_row(lane, e), c = ck0 + 8 * nt + frag_col(lane, e);
      dq_acc[nt][e] = fmaf(diag_s[r], to_f32(Ks.at(r, c)), dq_acc[nt][e]);
      dk_acc[nt][e] = fmaf(diag_s[r], to_f32(Qs.at(r, c)), dk_acc[nt][e]);
    }

  // ---- elementwise terms of Q-hat and K-tilde
  {
    const T* dqh = static_cast<const T*>(a.ws.dqh) + ch * (C * DK);
    const T* dkt = static_cast<const T*>(a.ws.dkt) + ch * (C * DK);
#pragma unroll
    for (int nt = 0; nt < NWK; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + frag_row(lane, e), c = ck0 + 8 * nt + frag_col(lane, e);
        const int off = Sw<T, C, DK>::off(r, c);
        const float G = Gs.at(r, c), GC = Gs.at(C - 1, c);
        const float gm = __expf(G), kdec = __expf(GC - G);
        const float a1 = to_f32(dqh[off]), a2 = to_f32(dkt[off]);
        const float kf = to_f32(Ks.at(r, c));
        dq_acc[nt][e] += a1 * gm;
        dk_acc[nt][e] += a2 * kdec;
        dG_acc[nt][e] += a1 * gm * to_f32(Qs.at(r, c)) - a2 * kdec * kf;
      }
  }
  // ---- dq, dk out; dbeta reduce
  {
    T* dq = static_cast<T*>(a.dq);
    T* dk = static_cast<T*>(a.dk);
#pragma unroll
    for (int nt = 0; nt < NWK; ++nt)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int r = m0 + frag_row(lane, e), c = ck0 + 8 * nt + frag_col(lane, e);
        const size_t gi = (row0 + r * rs) * DK + c;
        store2(dq + gi, dq_acc[nt][e], dq_acc[nt][e + 1]);
        store2(dk + gi, dk_acc[nt][e], dk_acc[nt][e + 1]);
      }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      db[i] += __shfl_xor_sync(0xffffffffu, db[i], 1);
      db[i] += __shfl_xor_sync(0xffffffffu, db[i], 2);
    }
    if ((lane & 3) == 0) {
      db_s[hf * C + m0 + (lane >> 2)] = db[0];
      db_s[hf * C + m0 + (lane >> 2) + 8] = db[1];
    }
  }
  __syncthreads();  // all score tiles consumed: dW/dU region becomes the dG staging
  FTile<C, DK> dGs{reinterpret_cast<float*>(sm + L::DW)};
#pragma unroll
  for (int nt = 0; nt < NWK; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      dGs.at(m0 + frag_row(lane, e), ck0 + 8 * nt + frag_col(lane, e)) = dG_acc[nt][e];
  if (tid < C) {
    T* dbeta = static_cast<T*>(a.dbeta);
    dbeta[row0 + tid * rs] = from_f32<T>(db_s[tid] + db_s[C + tid]);
  }
  __syncthreads();
  // reverse cumulative sum per channel; the last row also collects the K-tilde column
  // sums and dgam * gam (both depend on G at the chunk's last token)
  for (int c = tid; c < DK; c += GR_THREADS) {
    const T* dkt = static_cast<const T*>(a.ws.dkt) + ch * (C * DK);
    const float GC = Gs.at(C - 1, c);
    float extra = static_cast<const float*>(a.ws.dgam)[ch * DK + c] * __expf(GC);
    for (int t = 0; t < C; ++t)
      extra = fmaf(to_f32(dkt[Sw<T, C, DK>::off(t, c)]), __expf(GC - Gs.at(t, c)) * to_f32(Ks.at(t, c)), extra);
    float s = extra;
    for (int t = C - 1; t >= 0; --t) {
      s += dGs.at(t, c);
      dGs.at(t, c) = s;
    }
  }
  __syncthreads();
  T* dg = static_cast<T*>(a.dg);
  if (PC) {
    for (int i = tid; i < C * DK / 2; i += GR_THREADS) {
      const int r = i / (DK / 2), c = (i % (DK / 2)) * 2;
      store2(dg + (row0 + r * rs) * DK + c, dGs.at(r, c), dGs.at(r, c + 1));
    }
  } else {
    for (int r = warp; r < C; r += GR_THREADS / 32) {
      float s = 0.f;
      for (int c = lane; c < DK; c += 32) s += dGs.at(r, c);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (lane == 0) dg[row0 + r * rs] = from_f32<T>(s);
    }
  }
}


template <int DK, int DV>
cudaError_t launch_grads_t(const ChunkBwdArgs& a, cudaStream_t s) {
  const int N = a.T / C, BH = a.B * a.H;
  const int bytes = GrLayout<DK, DV>::BYTES + 1024;
  auto kern = a.per_channel ? chunk_grads_kernel<DK, DV, true> : chunk_grads_kernel<DK, DV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  prof_mark(K_GRADS, s, true);
  kern<<<dim3(N, BH), GR_THREADS, bytes, s>>>(a);
  prof_mark(K_GRADS, s, false);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_grads(const ChunkBwdArgs& a, cudaStream_t s) {
  if (a.B * a.H == 0 || a.T == 0) return cudaSuccess;
  return a.DK == 64 ? launch_grads_t<64, 64>(a, s) : launch_grads_t<128, 128>(a, s);
}

}  // namespace gdn
