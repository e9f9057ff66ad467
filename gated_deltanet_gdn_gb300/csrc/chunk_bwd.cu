// Chunked backward of the gated delta rule (bf16 operands, fp32 state and accumulation).
//
// Hand-derived from the chunked forward (see chunk_fwd.cu). With dS1 the gradient of the
// state leaving a chunk and dO the output gradient of its tokens:
//   reverse scan   dU  = scale Aqk^T dO + K-tilde dS1
//                  dS0 = diag(gam) dS1 + scale Q-hat^T dO - W^T dU
//   chunk products dQ-hat = scale dO S0^T, dW = -dU S0^T, dK-tilde = U dS1^T,
//                  dAqk = scale (dO U^T) masked j <= t, dgam = rowsum(dS1 * S0)
//   chunk grads    dT = dW Bk^T + dU Bv^T (Bk = diag(beta) Gam*k, Bv = diag(beta) V),
//                  dBk = T^T dW, dBv = T^T dU, dAkk = -(T^T dT T^T) masked j < t,
//                  dbeta = rowsum(dBk * K-hat) + rowsum(dBv * V) + rowsum(dAkk * Pkk),
//                  decay-weighted scores P[t,j] = sum_c x_tc y_jc exp(G_tc - G_jc) give
//                  dx = (dP (*) E) y, dy = (dP^T (*) E) x and dG = x dx - y dy,
//                  and dg is the reverse cumulative sum of dG inside the chunk.
// atomic-ops 0.1.0 (sections Features and Limitations) describes a backward made of
// stage kernels that reuse forward residuals, with the pairwise-decay score backward
// as one of them; the staging here is this library's own.
//
// Kernels
//   chunk_scan_bwd_kernel   grid (Dv/64, B*H), 256 threads, sequential over chunks in
//                           reverse: dS in registers, writes dU and dS1 per chunk, dh0
//   chunk_dstate_kernel     grid (chunks, B*H), 128 threads: the four products with the
//                           chunk states (contractions over Dv) and dgam
//   chunk_grads_kernel      (chunk_grads.cu) everything else
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int RSCAN_THREADS = 256;
constexpr int DST_THREADS = 256;


// ------------------------------------------------------------------ reverse state scan
// One CTA per (batch*head, NTS = 64 value columns), 8 warps; warp w owns gradient rows
// (w & 3) * Dk/4 .. + Dk/4 and columns 32 (w >> 2) .. + 31 of the slice.
template <int DK>
struct RScanLayout {
  static constexpr int ES = 2;
  static constexpr int W = 0;                      // -W          [C][DK]
  static constexpr int QH = W + C * DK * ES;       // scale Q-hat [C][DK]
  static constexpr int KT = QH + C * DK * ES;      // K-tilde     [C][DK]
  static constexpr int AQK = KT + C * DK * ES;     // scale Aqk   [C][C]
  static constexpr int GAM = AQK + C * C * ES;     // float [DK]
  static constexpr int DO = a1k(GAM + DK * 4);     // dO slice    [C][NTS]
  static constexpr int STAGE = a1k(DO + C * NTS * ES);
  static constexpr int DSS = 2 * STAGE;            // dS operand, transposed [NTS][DK]
  static constexpr int DUS = a1k(DSS + DK * NTS * ES);  // dU, transposed  [NTS][C]
  static constexpr int BAR = a1k(DUS + C * NTS * ES);
  static constexpr int BYTES = BAR + 64;
  static constexpr uint32_t TX = (uint32_t)(3 * C * DK * ES + C * C * ES + DK * 4);
};

template <int DK, int DV>
__global__ void __launch_bounds__(RSCAN_THREADS) chunk_scan_bwd_kernel(ChunkBwdArgs a) {
  typedef bf16 T;
  typedef RScanLayout<DK> L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  const int N = a.T / C;
  constexpr int NTILE = DV / NT, MTS = DK / 64, EPC = 8;
  const int rg = warp & 3, cg = warp >> 2;
  const int srow = rg * 16 * MTS, col0 = 32 * cg;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  Tile<T, NTS, DK> dSs{reinterpret_cast<T*>(sm + L::DSS)};  // dS^T rows of this slice
  Tile<T, NTS, C> dUs{reinterpret_cast<T*>(sm + L::DUS)};   // dU^T rows of this slice
  const T* dout = static_cast<const T*>(a.dout);

  float dS[MTS][4][4];
  const size_t sb = (size_t)bh * DK * DV;
#pragma unroll
  for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = srow + 16 * mt + frag_row(lane, e);
        const int c = tile * NTS + col0 + 8 * nt + frag_col(lane, e);
        dS[mt][nt][e] = a.dh_final ? a.dh_final[sb + (size_t)r * DV + c] : 0.f;
      }
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto issue = [&](int n, int s) {  // all threads: dO via cp.async; thread 0: records via bulk
    uint8_t* st = sm + s * L::STAGE;
    const size_t ch = (size_t)bh * N + n;
    if (tid == 0) {
      mbar_arrive_expect_tx(&bars[s], L::TX);
      bulk_g2s(st + L::W, static_cast<const T*>(a.res.wneg) + ch * (C * DK), C * DK * 2, &bars[s]);
      bulk_g2s(st + L::QH, static_cast<const T*>(a.res.qh) + ch * (C * DK), C * DK * 2, &bars[s]);
      bulk_g2s(st + L::KT, static_cast<const T*>(a.res.kt) + ch * (C * DK), C * DK * 2, &bars[s]);
      bulk_g2s(st + L::AQK, static_cast<const T*>(a.res.aqk) + ch * (C * C), C * C * 2, &bars[s]);
      bulk_g2s(st + L::GAM, a.res.gam + ch * DK, DK * 4, &bars[s]);
    }
    Tile<T, C, NTS> dOt{reinterpret_cast<T*>(st + L::DO)};
    const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
    for (int i = tid; i < C * NTS / EPC; i += RSCAN_THREADS) {
      const int r = i / (NTS / EPC), c0 = (i % (NTS / EPC)) * EPC;
      cp_async16(dOt.ptr(r, c0), dout + (row0 + (size_t)r * a.H) * DV + tile * NTS + c0);
    }
    cp_async_commit();
  };
  if (N > 0) issue(N - 1, 0);

  for (int it = 0; it < N; ++it) {
    const int n = N - 1 - it, s = it & 1;
    const uint32_t par = (uint32_t)(it >> 1) & 1u;
    const bool more = it + 1 < N;
    if (more) issue(n - 1, s ^ 1);
    uint8_t* st = sm + s * L::STAGE;
    Tile<T, C, DK> Wt{reinterpret_cast<T*>(st + L::W)};
    Tile<T, C, DK> Qt{reinterpret_cast<T*>(st + L::QH)};
    Tile<T, C, DK> Kt{reinterpret_cast<T*>(st + L::KT)};
    Tile<T, C, C> At{reinterpret_cast<T*>(st + L::AQK)};
    Tile<T, C, NTS> dOt{reinterpret_cast<T*>(st + L::DO)};
    const float* gam = reinterpret_cast<const float*>(st + L::GAM);
    const size_t ch = (size_t)bh * N + n;

#pragma unroll
    for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dSs.at(col0 + 8 * nt + frag_col(lane, e), srow + 16 * mt + frag_row(lane, e)) = from_f32<T>(dS[mt][nt][e]);
    fence_proxy_async();  // read by the bulk store below
    if (more) cp_async_wait<1>(); else cp_async_wait<0>();
    mbar_wait(&bars[s], par, a.err);
    __syncthreads();
    if (tid == 0) {  // gradient of the state leaving chunk n
      store_row_block<T, DV, DK>(static_cast<T*>(a.ws.dstate) + ch * (DK * DV), dSs.p, tile * NTS, NTS);
      bulk_commit();
    }
    float du[1][4][4];
    zero(du);
    Gemm<T>::template runk<1, 4, 0, C>(du, aview<true>(At), bview<true>(dOt), 16 * rg, col0, lane);
    Gemm<T>::template runk<1, 4, 0, DK>(du, aview<false>(Kt), bview<false>(dSs), 16 * rg, col0, lane);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        dUs.at(col0 + 8 * nt + frag_col(lane, e), 16 * rg + frag_row(lane, e)) = from_f32<T>(du[0][nt][e]);
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
      store_row_block<T, DV, C>(static_cast<T*>(a.ws.du) + ch * (C * DV), dUs.p, tile * NTS, NTS);
      bulk_commit();
    }
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dS[mt][nt][e] *= gam[srow + 16 * mt + frag_row(lane, e)];
    Gemm<T>::template runk<MTS, 4, 0, C>(dS, aview<true>(Qt), bview<true>(dOt), srow, col0, lane);
    Gemm<T>::template runk<MTS, 4, 0, C>(dS, aview<true>(Wt), bview<false>(dUs), srow, col0, lane);
    if (tid == 0) bulk_wait_read0();  // the bulk stores have read dSs and dUs before they are rewritten
    __syncthreads();
  }
  if (tid == 0) bulk_wait0();  // residual stores complete before the CTA retires
  if (a.dh0) {
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = srow + 16 * mt + frag_row(lane, e);
          const int c = tile * NTS + col0 + 8 * nt + frag_col(lane, e);
          a.dh0[sb + (size_t)r * DV + c] = dS[mt][nt][e];
        }
  }
}

// ------------------------------------------------------------------ state products
// Per chunk: everything that contracts over the value columns. With Y = T^T dU:
//   dv = beta Y, dbeta_v = rowsum(Y * V), dQ-hat = scale dO S0^T, dBk = -Y S0^T,
//   dK-tilde = U dS1^T, dAqk = scale dO U^T (j <= t), dAkk = -Y U^T (j < t),
//   dgam = rowsum(dS1 * S0).
template <int DK, int DV>
struct DstLayout {
  static constexpr int TM = 0;                       // T    [C][C]
  static constexpr int DO = a1k(TM + C * C * 2);     // dO   [C][DV]
  static constexpr int V = a1k(DO + C * DV * 2);     // v    [C][DV]
  static constexpr int U = a1k(V + C * DV * 2);      // U^T   [DV][C]
  static constexpr int DU = a1k(U + C * DV * 2);     // dU^T  [DV][C], then Y [C][DV]
  static constexpr int S0 = a1k(DU + C * DV * 2);    // S0^T  [DV][DK]
  static constexpr int DS1 = a1k(S0 + DK * DV * 2);  // dS1^T [DV][DK]
  static constexpr int OQH = a1k(DS1 + DK * DV * 2);  // output records staged as tiles:
  static constexpr int OBK = OQH + C * DK * 2;         //   dQ-hat, dBk, dK-tilde [C][DK]
  static constexpr int OKT = OBK + C * DK * 2;
  static constexpr int OAQ = OKT + C * DK * 2;         //   dAqk, dAkk [C][C]
  static constexpr int OAK = OAQ + C * C * 2;
  static constexpr int BETA = OAK + C * C * 2;
  static constexpr int DB = BETA + C * 4;            // float [2][C]
  static constexpr int GQ = DB + 2 * C * 4;          // float [quarters][DK] dgam partials
  static constexpr int BYTES = GQ + (DST_THREADS / (DK / 2)) * DK * 4;
};

template <int DK, int DV>
__global__ void __launch_bounds__(DST_THREADS) chunk_dstate_kernel(ChunkBwdArgs a) {
  typedef bf16 T;
  typedef DstLayout<DK, DV> L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  const int N = a.T / C;
  const size_t ch = (size_t)bh * N + n;
  constexpr int EPC = 8;
  Tile<T, C, C> Ts{reinterpret_cast<T*>(sm + L::TM)};
  Tile<T, C, DV> dOs{reinterpret_cast<T*>(sm + L::DO)};
  Tile<T, C, DV> Vs{reinterpret_cast<T*>(sm + L::V)};
  Tile<T, DV, C> Us{reinterpret_cast<T*>(sm + L::U)};       // U^T
  Tile<T, DV, C> dUs{reinterpret_cast<T*>(sm + L::DU)};      // dU^T
  Tile<T, DV, DK> S0s{reinterpret_cast<T*>(sm + L::S0)};     // S0^T
  Tile<T, DV, DK> dS1s{reinterpret_cast<T*>(sm + L::DS1)};   // dS1^T
  float* beta_s = reinterpret_cast<float*>(sm + L::BETA);
  float* db_s = reinterpret_cast<float*>(sm + L::DB);
  const T* dout = static_cast<const T*>(a.dout);
  const T* v = static_cast<const T*>(a.v);
  const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
  const size_t rs = a.H;
  for (int i = tid; i < C * DV / EPC; i += DST_THREADS) {
    const int r = i / (DV / EPC), c0 = (i % (DV / EPC)) * EPC;
    cp_async16(dOs.ptr(r, c0), dout + (row0 + r * rs) * DV + c0);
    cp_async16(Vs.ptr(r, c0), v + (row0 + r * rs) * DV + c0);
  }
  {
    const T* st = static_cast<const T*>(a.res.tmat) + ch * (C * C);
    for (int i = tid; i < C * C / EPC; i += DST_THREADS) cp_async16(Ts.p + i * EPC, st + i * EPC);
    const T* su = static_cast<const T*>(a.res.u) + ch * (C * DV);
    const T* sdu = static_cast<const T*>(a.ws.du) + ch * (C * DV);
    for (int i = tid; i < C * DV / EPC; i += DST_THREADS) {
      cp_async16(Us.p + i * EPC, su + i * EPC);
      cp_async16(dUs.p + i * EPC, sdu + i * EPC);
    }
    const T* ss = static_cast<const T*>(a.res.state) + ch * (DK * DV);
    const T* sds = static_cast<const T*>(a.ws.dstate) + ch * (DK * DV);
    for (int i = tid; i < DK * DV / EPC; i += DST_THREADS) {
      cp_async16(S0s.p + i * EPC, ss + i * EPC);
      cp_async16(dS1s.p + i * EPC, sds + i * EPC);
    }
  }
  cp_async_commit();
  if (tid < C) beta_s[tid] = to_f32(static_cast<const T*>(a.beta)[row0 + tid * rs]);
  cp_async_wait<0>();
  __syncthreads();

  const int m0 = 16 * (warp & 3), hf = warp >> 2;
  // Y = T^T dU; dv = beta Y; dbeta_v = rowsum(Y * V)
  constexpr int NWV = DV / 16;
  float y[1][NWV][4];
  zero(y);
  Gemm<T>::template runk<1, NWV, 0, C>(y, aview<true>(Ts), bview<false>(dUs), m0, hf * (DV / 2), lane);
  {
    float db[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < NWV; ++nt)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int r = m0 + frag_row(lane, e), c = hf * (DV / 2) + 8 * nt + frag_col(lane, e);
        db[e >> 1] += y[0][nt][e] * to_f32(Vs.at(r, c)) + y[0][nt][e + 1] * to_f32(Vs.at(r, c + 1));
        // dv staged over this thread's own v elements, stored row-wise below
        store2(Vs.ptr(r, c), beta_s[r] * y[0][nt][e], beta_s[r] * y[0][nt][e + 1]);
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
  __syncthreads();  // dU consumed: Y takes its place
  Tile<T, C, DV> Ys{reinterpret_cast<T*>(sm + L::DU)};
#pragma unroll
  for (int nt = 0; nt < NWV; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      Ys.at(m0 + frag_row(lane, e), hf * (DV / 2) + 8 * nt + frag_col(lane, e)) = from_f32<T>(y[0][nt][e]);
  if (tid < C) a.ws.dbv[ch * C + tid] = db_s[tid] + db_s[C + tid];
  {
    T* dv = static_cast<T*>(a.dv);
    for (int i = tid; i < C * DV / EPC; i += DST_THREADS) {
      const int r = i / (DV / EPC), c0 = (i % (DV / EPC)) * EPC;
      copy16(dv + (row0 + r * rs) * DV + c0, Vs.ptr(r, c0));
    }
  }
  {  // dgam_c = sum_v dS1[c][v] S0[c][v]: thread (channel pair, quarter of v), then the quarters
    constexpr int NQ = DST_THREADS / (DK / 2), VQ = DV / NQ;
    const int c = 2 * (tid % (DK / 2)), vq = tid / (DK / 2);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 8
    for (int v2 = vq * VQ; v2 < (vq + 1) * VQ; ++v2) {
      const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(dS1s.ptr(v2, c));
      const __nv_bfloat162 z = *reinterpret_cast<const __nv_bfloat162*>(S0s.ptr(v2, c));
      acc0 = fmaf(__low2float(x), __low2float(z), acc0);
      acc1 = fmaf(__high2float(x), __high2float(z), acc1);
    }
    float* part = reinterpret_cast<float*>(sm + L::GQ);
    part[vq * DK + c] = acc0;
    part[vq * DK + c + 1] = acc1;
  }
  __syncthreads();
  for (int c = tid; c < DK; c += DST_THREADS) {
    constexpr int NQ = DST_THREADS / (DK / 2);
    const float* part = reinterpret_cast<const float*>(sm + L::GQ);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < NQ; ++i) acc += part[i * DK + c];
    a.ws.dgam[ch * DK + c] = acc;
  }

  // C x DK products: warp rows m0, columns hf * DK / 2 .. + DK / 2
  constexpr int NH = DK / 16;
  const int n0 = hf * (DK / 2);
  auto store_cdk = [&](int region, const float (&acc)[1][NH][4], float mul) {
    T* dst = reinterpret_cast<T*>(sm + region);
#pragma unroll
    for (int nt = 0; nt < NH; ++nt)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int r = m0 + frag_row(lane, e), c = n0 + 8 * nt + frag_col(lane, e);
        store2(dst + Sw<T, C, DK>::off(r, c), mul * acc[0][nt][e], mul * acc[0][nt][e + 1]);
      }
  };
  {
    float acc[1][NH][4];
    zero(acc);
    Gemm<T>::template runk<1, NH, 0, DV>(acc, aview<false>(dOs), bview<true>(S0s), m0, n0, lane);
    store_cdk(L::OQH, acc, a.scale);
    zero(acc);
    Gemm<T>::template runk<1, NH, 0, DV>(acc, aview<false>(Ys), bview<true>(S0s), m0, n0, lane);
    store_cdk(L::OBK, acc, -1.f);
    zero(acc);
    Gemm<T>::template runk<1, NH, 0, DV>(acc, aview<true>(Us), bview<true>(dS1s), m0, n0, lane);
    store_cdk(L::OKT, acc, 1.f);
  }
  // C x C products: warp rows m0, columns 32 hf .. +31 (block-1 rows see no block-2 columns)
  {
    const int c0 = 32 * hf;
    const bool dead = m0 < BLK && hf == 1;
    float aq[1][4][4], ak[1][4][4];
    zero(aq);
    zero(ak);
    if (!dead) {
      Gemm<T>::template runk<1, 4, 0, DV>(aq, aview<false>(dOs), bview<true>(Us), m0, c0, lane);
      Gemm<T>::template runk<1, 4, 0, DV>(ak, aview<false>(Ys), bview<true>(Us), m0, c0, lane);
    }
    T* da = reinterpret_cast<T*>(sm + L::OAQ);
    T* dk = reinterpret_cast<T*>(sm + L::OAK);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int r = m0 + frag_row(lane, e), j = c0 + 8 * nt + frag_col(lane, e);
        const int off = Sw<T, C, C>::off(r, j);
        store2(da + off, j <= r ? a.scale * aq[0][nt][e] : 0.f, j + 1 <= r ? a.scale * aq[0][nt][e + 1] : 0.f);
        store2(dk + off, j < r ? -ak[0][nt][e] : 0.f, j + 1 < r ? -ak[0][nt][e + 1] : 0.f);
      }
  }
  fence_proxy_async();  // the staged records are read by the bulk copies below
  __syncthreads();
  if (tid == 0) {
    bulk_s2g(static_cast<T*>(a.ws.dqh) + ch * (C * DK), sm + L::OQH, C * DK * 2);
    bulk_s2g(static_cast<T*>(a.ws.dbk) + ch * (C * DK), sm + L::OBK, C * DK * 2);
    bulk_s2g(static_cast<T*>(a.ws.dkt) + ch * (C * DK), sm + L::OKT, C * DK * 2);
    bulk_s2g(static_cast<T*>(a.ws.daqk) + ch * (C * C), sm + L::OAQ, C * C * 2);
    bulk_s2g(static_cast<T*>(a.ws.dakk) + ch * (C * C), sm + L::OAK, C * C * 2);
    bulk_commit();
    bulk_wait_read0();  // the staged tiles are read before the CTA releases its shared memory
  }
}

template <int DK, int DV>
cudaError_t launch_bwd_t(const ChunkBwdArgs& a, cudaStream_t s) {
  const int N = a.T / C, BH = a.B * a.H;
  cudaError_t e;
  if (scan_tc_applies(1, DK, DV)) {
    if ((e = launch_scan_bwd_tc(a, s)) != cudaSuccess) return e;
  } else {
    const int bytes = RScanLayout<DK>::BYTES + 1024;
    auto kern = chunk_scan_bwd_kernel<DK, DV>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) return e;
    prof_mark(K_SCAN_BWD, s, true);
    kern<<<dim3(DV / NTS, BH), RSCAN_THREADS, bytes, s>>>(a);
    prof_mark(K_SCAN_BWD, s, false);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (N == 0) return cudaSuccess;
  {
    const int bytes = DstLayout<DK, DV>::BYTES + 1024;
    auto kern = chunk_dstate_kernel<DK, DV>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) return e;
    prof_mark(K_DSTATE, s, true);
    kern<<<dim3(N, BH), DST_THREADS, bytes, s>>>(a);
    prof_mark(K_DSTATE, s, false);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return launch_chunk_grads(a, s);
}

}  // namespace

cudaError_t launch_chunk_bwd(const ChunkBwdArgs& a, cudaStream_t s) {
  if (a.B * a.H == 0) return cudaSuccess;
  return a.DK == 64 ? launch_bwd_t<64, 64>(a, s) : launch_bwd_t<128, 128>(a, s);
}

}  // namespace gdn
