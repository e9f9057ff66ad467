// Chunked backward of the gated delta rule (bf16 or fp32 operands, fp32 state and
// accumulation).
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
// Kernels of the CUDA-core path (Dk = 64, or fp32 operands; bf16 with Dk = Dv = 128 runs
// chunk_bwd_tc.cu instead), launched in this order on the caller's stream:
//   chunk_scan_bwd_kernel   grid (Dv/64, B*H), 256 threads, sequential over chunks in
//                           reverse: dS in registers, writes dU and dS1 per chunk, dh0
//   chunk_dqa_kernel        one CTA per chunk-head, 256 threads: dQ-hat and dAqk, the
//                           products that need only forward records and dO
//   chunk_dstate_kernel     grid (chunks, B*H), 256 threads: the products with dU and dS1
//                           (contractions over Dv) and dgam
//   chunk_grads_kernel      (chunk_grads.cu) everything else
#include "chunk_dqa.cuh"
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int RSCAN_THREADS = 256;
constexpr int DST_THREADS = 256;
constexpr int DST_CG = DST_THREADS / 128;  // column groups of the state-products warps (4 row groups each)


// ------------------------------------------------------------------ reverse state scan
// One CTA per (batch*head, NTS = 64 value columns), 8 warps; warp w owns gradient rows
// (w & 3) * Dk/4 .. + Dk/4 and columns 32 (w >> 2) .. + 31 of the slice. bf16 records
// are double-buffered (the next chunk loads during this one); fp32 records take twice
// the room, so one stage, loaded at the top of its step.
template <class T, int DK>
struct RScanLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int STAGES = ES == 2 ? 2 : 1;
  static constexpr int W = 0;                      // -W          [C][DK]
  static constexpr int QH = W + C * DK * ES;       // scale Q-hat [C][DK]
  static constexpr int KT = QH + C * DK * ES;      // K-tilde     [C][DK]
  static constexpr int AQK = KT + C * DK * ES;     // scale Aqk   [C][C]
  static constexpr int GAM = AQK + C * C * ES;     // float [DK]
  static constexpr int DO = a1k(GAM + DK * 4);     // dO slice    [C][NTS]
  static constexpr int STAGE = a1k(DO + C * NTS * ES);
  static constexpr int DSS = STAGES * STAGE;       // dS operand, transposed [NTS][DK]
  static constexpr int DUS = a1k(DSS + DK * NTS * ES);  // dU, transposed  [NTS][C]
  static constexpr int BAR = a1k(DUS + C * NTS * ES);
  static constexpr int BYTES = BAR + 64;
  static constexpr uint32_t TX = (uint32_t)(3 * C * DK * ES + C * C * ES + DK * 4);
};

template <class T, int DK, int DV>
__global__ void __launch_bounds__(RSCAN_THREADS) chunk_scan_bwd_kernel(ChunkBwdArgs a) {
  typedef RScanLayout<T, DK> L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  const int N = a.T / C;
  constexpr int MTS = DK / 64, EPC = 16 / (int)sizeof(T), STAGES = L::STAGES;
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
    for (int i = 0; i < STAGES; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto issue = [&](int n, int s) {  // all threads: dO via cp.async; thread 0: records via bulk
    uint8_t* st = sm + s * L::STAGE;
    const size_t ch = (size_t)bh * N + n;
    if (tid == 0) {
      mbar_arrive_expect_tx(&bars[s], L::TX);
      bulk_g2s(st + L::W, static_cast<const T*>(a.res.wneg) + ch * (C * DK), C * DK * L::ES, &bars[s]);
      bulk_g2s(st + L::QH, static_cast<const T*>(a.res.qh) + ch * (C * DK), C * DK * L::ES, &bars[s]);
      bulk_g2s(st + L::KT, static_cast<const T*>(a.res.kt) + ch * (C * DK), C * DK * L::ES, &bars[s]);
      bulk_g2s(st + L::AQK, static_cast<const T*>(a.res.aqk) + ch * (C * C), C * C * L::ES, &bars[s]);
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
  // step it works on chunk N - 1 - it in stage it % STAGES; its loads were issued
  // STAGES - 1 steps earlier
  for (int i = 0; i < STAGES - 1 && i < N; ++i) issue(N - 1 - i, i);

  for (int it = 0; it < N; ++it) {
    const int n = N - 1 - it, s = it % STAGES;
    const uint32_t par = (uint32_t)(it / STAGES) & 1u;
    const bool more = STAGES > 1 && it + 1 < N;  // a later chunk's dO group is in flight
    if (it + STAGES - 1 < N) issue(n - (STAGES - 1), (it + STAGES - 1) % STAGES);
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
  cp_async_wait<0>();
  if (tid == 0) {  // every load landed and the residual stores complete before the CTA retires
    drain_ring(bars, STAGES, N);
    bulk_wait0();
  }
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
// Per chunk: everything that contracts over the value columns. Without the reverse
// scan's results (chunk_dqa_kernel): dQ-hat = scale dO S0^T, dAqk = scale dO U^T
// (j <= t). With Y = T^T dU (chunk_dstate_kernel): dv = beta Y, dbeta_v = rowsum(Y * V),
// dBk = -Y S0^T, dK-tilde = U dS1^T, dAkk = -Y U^T (j < t), dgam = rowsum(dS1 * S0).
// The products without the reverse scan's results, after the CUDA-core scan (the
// tensor-core scan runs them as extra CTAs of its own launch).
template <class T, int DK, int DV>
__global__ void __launch_bounds__(DQA_THREADS, sizeof(T) == 2 ? 2 : 1) chunk_dqa_kernel(ChunkBwdArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  dqa_units<T, DK, DV>(a, align1024(smem_raw), blockIdx.x, gridDim.x, threadIdx.x);
}

template <class T, int DK, int DV>
struct DstLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int TM = 0;                        // T     [C][C]
  static constexpr int V = a1k(TM + C * C * ES);      // v     [C][DV], then dv; then S0^T panel 1
  static constexpr int U = a1k(V + C * DV * ES);      // U^T   [DV][C]
  static constexpr int DU = a1k(U + C * DV * ES);     // dU^T  [DV][C], then Y [C][DV]
  static constexpr int S0P = a1k(DU + C * DV * ES);   // S0^T  [DV][64], one 64-channel panel
  static constexpr int DSP = a1k(S0P + DV * 64 * ES); // dS1^T [DV][64], one 64-channel panel
  static constexpr int BETA = a1k(DSP + DV * 64 * ES);
  static constexpr int DB = BETA + C * 4;            // float [DST_CG][C]
  static constexpr int GQ = DB + DST_CG * C * 4;     // float [DST_THREADS / 32][DK] dgam partials
  static constexpr int BYTES = GQ + (DST_THREADS / 32) * DK * 4;
};

// Two CTAs per SM with bf16 records (one with fp32): while one computes, the other's
// loads are in flight. The state and state-gradient records are taken one 64-channel
// panel at a time; the second S0^T panel is prefetched into v's buffer as soon as dv has
// left it.
template <class T, int DK, int DV>
__global__ void __launch_bounds__(DST_THREADS, sizeof(T) == 2 ? 2 : 1) chunk_dstate_kernel(ChunkBwdArgs a) {
  pdl_wait();
  pdl_trigger();
  typedef DstLayout<T, DK, DV> L;
  constexpr int NPAN = DK / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  const int N = a.T / C;
  const size_t ch = (size_t)bh * N + n;
  constexpr int EPC = 16 / (int)sizeof(T);
  Tile<T, C, C> Ts{reinterpret_cast<T*>(sm + L::TM)};
  Tile<T, C, DV> Vs{reinterpret_cast<T*>(sm + L::V)};
  Tile<T, DV, C> Us{reinterpret_cast<T*>(sm + L::U)};    // U^T
  Tile<T, DV, C> dUs{reinterpret_cast<T*>(sm + L::DU)};  // dU^T
  float* beta_s = reinterpret_cast<float*>(sm + L::BETA);
  float* db_s = reinterpret_cast<float*>(sm + L::DB);
  float* gq = reinterpret_cast<float*>(sm + L::GQ);
  const T* v = static_cast<const T*>(a.v);
  const T* s0rec = static_cast<const T*>(a.res.state) + ch * (DK * DV);
  const T* ds1rec = static_cast<const T*>(a.ws.dstate) + ch * (DK * DV);
  const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
  const size_t rs = a.H;
  auto load_panel = [&](T* dst, const T* rec, int p) {  // columns 64p .. 64p + 63 of an S^T record
    const T* src = rec + (size_t)p * DV * 64;
    for (int i = tid; i < DV * 64 / EPC; i += DST_THREADS) cp_async16(dst + i * EPC, src + i * EPC);
  };
  // group 0: what Y, dv and dbeta_v need
  {
    const T* st = static_cast<const T*>(a.res.tmat) + ch * (C * C);
    for (int i = tid; i < C * C / EPC; i += DST_THREADS) cp_async16(Ts.p + i * EPC, st + i * EPC);
    const T* sdu = static_cast<const T*>(a.ws.du) + ch * (C * DV);
    for (int i = tid; i < C * DV / EPC; i += DST_THREADS) {
      const int r = i / (DV / EPC), c0 = (i % (DV / EPC)) * EPC;
      cp_async16(dUs.p + i * EPC, sdu + i * EPC);
      cp_async16(Vs.ptr(r, c0), v + (row0 + r * rs) * DV + c0);
    }
  }
  cp_async_commit();
  // group 1: the products with U, S0 and dS1 (first channel panel)
  {
    const T* su = static_cast<const T*>(a.res.u) + ch * (C * DV);
    for (int i = tid; i < C * DV / EPC; i += DST_THREADS) cp_async16(Us.p + i * EPC, su + i * EPC);
    load_panel(reinterpret_cast<T*>(sm + L::S0P), s0rec, 0);
    load_panel(reinterpret_cast<T*>(sm + L::DSP), ds1rec, 0);
  }
  cp_async_commit();
  if (tid < C) beta_s[tid] = to_f32(static_cast<const T*>(a.beta)[row0 + tid * rs]);
  cp_async_wait<1>();
  __syncthreads();

  // warp w: rows 16 (w % 4) .. + 15 and column group w / 4 of every product
  const int m0 = 16 * (warp & 3), hf = warp >> 2;
  // Y = T^T dU; dv = beta Y; dbeta_v = rowsum(Y * V)
  constexpr int NWV = DV / (8 * DST_CG);
  float y[1][NWV][4];
  zero(y);
  Gemm<T>::template runk<1, NWV, 0, C>(y, aview<true>(Ts), bview<false>(dUs), m0, hf * (DV / DST_CG), lane);
  {
    float db[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < NWV; ++nt)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int r = m0 + frag_row(lane, e), c = hf * (DV / DST_CG) + 8 * nt + frag_col(lane, e);
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
  __syncthreads();  // dU consumed: Y takes its place; dv complete
  Tile<T, C, DV> Ys{reinterpret_cast<T*>(sm + L::DU)};
#pragma unroll
  for (int nt = 0; nt < NWV; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      Ys.at(m0 + frag_row(lane, e), hf * (DV / DST_CG) + 8 * nt + frag_col(lane, e)) = from_f32<T>(y[0][nt][e]);
  if (tid < C) {
    float sdb = 0.f;
#pragma unroll
    for (int i = 0; i < DST_CG; ++i) sdb += db_s[i * C + tid];
    a.ws.dbv[ch * C + tid] = sdb;
  }
  {
    T* dv = static_cast<T*>(a.dv);
    for (int i = tid; i < C * DV / EPC; i += DST_THREADS) {
      const int r = i / (DV / EPC), c0 = (i % (DV / EPC)) * EPC;
      copy16(dv + (row0 + r * rs) * DV + c0, Vs.ptr(r, c0));
    }
  }
  __syncthreads();  // v's buffer free: prefetch the second S0^T panel there
  if (NPAN > 1) {
    load_panel(reinterpret_cast<T*>(sm + L::V), s0rec, 1);
    cp_async_commit();
    cp_async_wait<1>();  // group 1 (first panels, U) complete
  } else {
    cp_async_wait<0>();
  }
  __syncthreads();

  // dAkk: warp rows m0, columns hf * C / DST_CG .. (block-1 rows see no block-2 columns);
  // stored straight into the record (swizzled tile image)
  {
    constexpr int NCC = C / (8 * DST_CG);
    const int c0 = hf * (C / DST_CG);
    float ak[1][NCC][4];
    zero(ak);
    if (!(m0 < BLK && c0 >= BLK))
      Gemm<T>::template runk<1, NCC, 0, DV>(ak, aview<false>(Ys), bview<true>(Us), m0, c0, lane);
    T* dk = static_cast<T*>(a.ws.dakk) + ch * (C * C);
#pragma unroll
    for (int nt = 0; nt < NCC; ++nt)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int r = m0 + frag_row(lane, e), j = c0 + 8 * nt + frag_col(lane, e);
        store2(dk + Sw<T, C, C>::off(r, j), j < r ? -ak[0][nt][e] : 0.f, j + 1 < r ? -ak[0][nt][e + 1] : 0.f);
      }
  }

  // C x 64 products per channel panel: warp rows m0, columns hf * 64 / DST_CG ..
  constexpr int NH = 64 / (8 * DST_CG);
  const int n0 = hf * (64 / DST_CG);
  auto store_cdk = [&](void* base, int p, const float (&acc)[1][NH][4], float mul) {
    T* dst = static_cast<T*>(base) + ch * (C * DK);
#pragma unroll
    for (int nt = 0; nt < NH; ++nt)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int r = m0 + frag_row(lane, e), c = 64 * p + n0 + 8 * nt + frag_col(lane, e);
        store2(dst + Sw<T, C, DK>::off(r, c), mul * acc[0][nt][e], mul * acc[0][nt][e + 1]);
      }
  };
  // dgam over one panel: thread (channel pair, 1/16 of the value rows), partials in gq
  auto dgam_part = [&](Tile<T, DV, 64> s0, Tile<T, DV, 64> ds1, int p) {
    constexpr int NQ = DST_THREADS / 32, VQ = DV / NQ;
    const int c = 2 * (tid % 32), vq = tid / 32;
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int v2 = vq * VQ; v2 < (vq + 1) * VQ; ++v2) {
      const float2 x = ld2(ds1.ptr(v2, c)), z = ld2(s0.ptr(v2, c));
      acc0 = fmaf(x.x, z.x, acc0);
      acc1 = fmaf(x.y, z.y, acc1);
    }
    gq[vq * DK + 64 * p + c] = acc0;
    gq[vq * DK + 64 * p + c + 1] = acc1;
  };
#pragma unroll 1
  // per panel: the products with dS1^T first, so that the next dS1^T panel streams in
  // behind this panel's products with S0^T
  for (int p = 0; p < NPAN; ++p) {
    Tile<T, DV, 64> S0p{reinterpret_cast<T*>(sm + (p == 0 ? L::S0P : L::V))};
    Tile<T, DV, 64> dS1p{reinterpret_cast<T*>(sm + L::DSP)};
    float acc[1][NH][4];
    if (p > 0) {
      cp_async_wait<0>();  // this dS1^T panel
      __syncthreads();
    }
    zero(acc);
    Gemm<T>::template runk<1, NH, 0, DV>(acc, aview<true>(Us), bview<true>(dS1p), m0, n0, lane);
    store_cdk(a.ws.dkt, p, acc, 1.f);
    dgam_part(S0p, dS1p, p);
    if (p + 1 < NPAN) {
      __syncthreads();  // this dS1^T panel is consumed: the next one loads in its place
      load_panel(reinterpret_cast<T*>(sm + L::DSP), ds1rec, p + 1);
      cp_async_commit();
    }
    zero(acc);
    Gemm<T>::template runk<1, NH, 0, DV>(acc, aview<false>(Ys), bview<true>(S0p), m0, n0, lane);
    store_cdk(a.ws.dbk, p, acc, -1.f);
  }
  __syncthreads();
  for (int c = tid; c < DK; c += DST_THREADS) {
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < DST_THREADS / 32; ++i) acc += gq[i * DK + c];
    a.ws.dgam[ch * DK + c] = acc;
  }
}

template <class T, int DK, int DV>
cudaError_t launch_bwd_t(const ChunkBwdArgs& a, cudaStream_t s) {
  const int N = a.T / C, BH = a.B * a.H;
  const int bf16_ops = sizeof(T) == 2;
  cudaError_t e;
  // bf16 with Dk = Dv = 128: the tensor-core reverse scan and one fused tensor-core kernel
  // for every chunk product and gradient (chunk_bwd_tc.cu), in one launch where they fit
  // side by side. Otherwise (Dk = 64, or fp32 operands): the CUDA-core scan, then the
  // products that need no scan result (chunk_dqa.cuh), the state products, the score
  // gradients and the channel-group sums.
  if (scan_tc_applies(bf16_ops, DK, DV) && bwd_tc_applies(DK, DV)) return launch_chunk_bwd_tc(a, s);
  {
    const int bytes = RScanLayout<T, DK>::BYTES + 1024;
    auto kern = chunk_scan_bwd_kernel<T, DK, DV>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) return e;
    prof_mark(K_SCAN_BWD, s, true);
    kern<<<dim3(DV / NTS, BH), RSCAN_THREADS, bytes, s>>>(a);
    prof_mark(K_SCAN_BWD, s, false);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (N == 0) return cudaSuccess;
  {
    const int bytes = DqaLayout<T, DK, DV>::BYTES + 1024;
    auto kern = chunk_dqa_kernel<T, DK, DV>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) return e;
    prof_mark(K_DQA, s, true);
    if ((e = launch_pdl(kern, dim3(N * BH), dim3(DQA_THREADS), bytes, s, a)) != cudaSuccess) return e;
    prof_mark(K_DQA, s, false);
  }
  {
    const int bytes = DstLayout<T, DK, DV>::BYTES + 1024;
    auto kern = chunk_dstate_kernel<T, DK, DV>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) return e;
    prof_mark(K_DSTATE, s, true);
    if ((e = launch_pdl(kern, dim3(N, BH), dim3(DST_THREADS), bytes, s, a)) != cudaSuccess) return e;
    prof_mark(K_DSTATE, s, false);
  }
  return launch_chunk_grads(a, s);
}

template <class T>
cudaError_t launch_bwd_dims(const ChunkBwdArgs& a, cudaStream_t s) {
  if (a.DK == 64) return a.DV == 64 ? launch_bwd_t<T, 64, 64>(a, s) : launch_bwd_t<T, 64, 128>(a, s);
  return a.DV == 64 ? launch_bwd_t<T, 128, 64>(a, s) : launch_bwd_t<T, 128, 128>(a, s);
}

}  // namespace

cudaError_t launch_chunk_bwd(const ChunkBwdArgs& a, cudaStream_t s) {
  if (a.B * a.H == 0) return cudaSuccess;
  return a.bf16 ? launch_bwd_dims<bf16>(a, s) : launch_bwd_dims<float>(a, s);
}

}  // namespace gdn
