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
// With 128-token chunks (GDN_FLAG_CHUNK128) the reverse scan runs over them and
// chunk_mid128_kernel forms the 64-token blocks' records before the chunk products.
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
// CC: chunk length. With CC = C2 (128-token chunks, bf16 operands only: one stage of
// 128-token records fills the shared memory) the scan reads the 128-token records, stores
// the gradient of the state leaving each 128-token chunk as the dS1 record of its second
// 64-token block and no dU (chunk_mid128_kernel forms the 64-token blocks' dU and the
// first block's dS1 from it).
template <class T, int DK, int CC = C>
struct RScanLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int STAGES = ES == 2 && CC == C ? 2 : 1;
  static constexpr int W = 0;                       // -W          [CC][DK]
  static constexpr int QH = W + CC * DK * ES;       // scale Q-hat [CC][DK]
  static constexpr int KT = QH + CC * DK * ES;      // K-tilde     [CC][DK]
  static constexpr int AQK = KT + CC * DK * ES;     // scale Aqk   [CC][CC]
  static constexpr int GAM = AQK + CC * CC * ES;    // float [DK]
  static constexpr int DO = a1k(GAM + DK * 4);      // dO slice    [CC][NTS]
  static constexpr int STAGE = a1k(DO + CC * NTS * ES);
  static constexpr int DSS = STAGES * STAGE;        // dS operand, transposed [NTS][DK]
  static constexpr int DUS = a1k(DSS + DK * NTS * ES);  // dU, transposed  [NTS][CC]
  static constexpr int BAR = a1k(DUS + CC * NTS * ES);
  static constexpr int BYTES = BAR + 64;
  static constexpr uint32_t TX = (uint32_t)(3 * CC * DK * ES + CC * CC * ES + DK * 4);
};

template <class T, int DK, int DV, int CC = C>
__global__ void __launch_bounds__(RSCAN_THREADS) chunk_scan_bwd_kernel(ChunkBwdArgs a) {
  typedef RScanLayout<T, DK, CC> L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  const int N = a.T / CC;
  constexpr int MTS = DK / 64, EPC = 16 / (int)sizeof(T), STAGES = L::STAGES;
  constexpr int MU = CC / 64;  // m16 tiles of dU rows per warp
  const int rg = warp & 3, cg = warp >> 2;
  const int srow = rg * 16 * MTS, col0 = 32 * cg, urow = rg * 16 * MU;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  Tile<T, NTS, DK> dSs{reinterpret_cast<T*>(sm + L::DSS)};  // dS^T rows of this slice
  Tile<T, NTS, CC> dUs{reinterpret_cast<T*>(sm + L::DUS)};  // dU^T rows of this slice
  const T* dout = static_cast<const T*>(a.dout);
  // the CC-token records: the 64-token ones, or those of the 128-token chunks
  const void* rw = CC == C ? a.res.wneg : a.res2.wneg;
  const void* rq = CC == C ? a.res.qh : a.res2.qh;
  const void* rk = CC == C ? a.res.kt : a.res2.kt;
  const void* ra = CC == C ? a.res.aqk : a.res2.aqk;
  const float* rg_ = CC == C ? a.res.gam : a.res2.gam;

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
      bulk_g2s(st + L::W, static_cast<const T*>(rw) + ch * (CC * DK), CC * DK * L::ES, &bars[s]);
      bulk_g2s(st + L::QH, static_cast<const T*>(rq) + ch * (CC * DK), CC * DK * L::ES, &bars[s]);
      bulk_g2s(st + L::KT, static_cast<const T*>(rk) + ch * (CC * DK), CC * DK * L::ES, &bars[s]);
      bulk_g2s(st + L::AQK, static_cast<const T*>(ra) + ch * (CC * CC), CC * CC * L::ES, &bars[s]);
      bulk_g2s(st + L::GAM, rg_ + ch * DK, DK * 4, &bars[s]);
    }
    Tile<T, CC, NTS> dOt{reinterpret_cast<T*>(st + L::DO)};
    const size_t row0 = ((size_t)b * a.T + (size_t)n * CC) * a.H + h;
    for (int i = tid; i < CC * NTS / EPC; i += RSCAN_THREADS) {
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
    Tile<T, CC, DK> Wt{reinterpret_cast<T*>(st + L::W)};
    Tile<T, CC, DK> Qt{reinterpret_cast<T*>(st + L::QH)};
    Tile<T, CC, DK> Kt{reinterpret_cast<T*>(st + L::KT)};
    Tile<T, CC, CC> At{reinterpret_cast<T*>(st + L::AQK)};
    Tile<T, CC, NTS> dOt{reinterpret_cast<T*>(st + L::DO)};
    const float* gam = reinterpret_cast<const float*>(st + L::GAM);
    const size_t ch = (size_t)bh * N + n;
    // the 64-token record that takes this chunk's dS1: the chunk itself, or the second
    // block of the 128-token chunk
    const size_t chd = CC == C ? ch : (size_t)bh * (a.T / C) + 2 * (size_t)n + 1;

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
      store_row_block<T, DV, DK>(static_cast<T*>(a.ws.dstate) + chd * (DK * DV), dSs.p, tile * NTS, NTS);
      bulk_commit();
    }
    float du[MU][4][4];
    zero(du);
    Gemm<T>::template runk<MU, 4, 0, CC>(du, aview<true>(At), bview<true>(dOt), urow, col0, lane);
    Gemm<T>::template runk<MU, 4, 0, DK>(du, aview<false>(Kt), bview<false>(dSs), urow, col0, lane);
#pragma unroll
    for (int mt = 0; mt < MU; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dUs.at(col0 + 8 * nt + frag_col(lane, e), urow + 16 * mt + frag_row(lane, e)) = from_f32<T>(du[mt][nt][e]);
    fence_proxy_async();
    __syncthreads();
    if (CC == C && tid == 0) {
      store_row_block<T, DV, C>(static_cast<T*>(a.ws.du) + ch * (C * DV), dUs.p, tile * NTS, NTS);
      bulk_commit();
    }
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dS[mt][nt][e] *= gam[srow + 16 * mt + frag_row(lane, e)];
    Gemm<T>::template runk<MTS, 4, 0, CC>(dS, aview<true>(Qt), bview<true>(dOt), srow, col0, lane);
    Gemm<T>::template runk<MTS, 4, 0, CC>(dS, aview<true>(Wt), bview<false>(dUs), srow, col0, lane);
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

// ------------------------------------------------------------------ 128-token chunks
// The backward over 128-token chunks (FLAG_CHUNK128, bf16 operands). The reverse scan runs
// over the 128-token chunks, half the sequential steps, and stores the gradient of the
// state leaving each 128-token chunk (dS_end) as the dS1 record of its second 64-token
// block. Per 128-token chunk this kernel then forms, from the two blocks' own records
// (block 1 and block 2, each relative to its own start, as the preparation wrote them),
// what the 64-token chunk products read: one reverse step and one forward step of the
// 64-token recurrence across the block boundary,
//   dU2   = scale Aqk2^T dO2 + K-tilde2 dS_end                  (block 2's dU)
//   dSmid = diag(gam2) dS_end + scale Q-hat2^T dO2 - W2^T dU2    (block 1's dS1)
//   dU1   = scale Aqk1^T dO1 + K-tilde1 dSmid                    (block 1's dU)
//   Smid  = diag(gam1) S + K-tilde1^T U1                         (block 2's chunk-start state)
// with S the 128-token chunk's start state and U1, U2 the halves of its U (the 64-token
// deltas are the 128-token ones). All in value-major form, as the records are stored.
// One CTA of 256 threads per 128-token chunk-head.
constexpr int MID_THREADS = 256;

template <class T, int DK, int DV>
struct MidLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int DO1 = 0;                        // dO of block 1 [C][DV]
  static constexpr int A1 = a1k(DO1 + C * DV * ES);    // scale Aqk of block 1 [C][C]
  static constexpr int K1 = a1k(A1 + C * C * ES);      // K-tilde of block 1 [C][DK]
  static constexpr int DS = a1k(K1 + C * DK * ES);     // dS_end^T [DV][DK], then dSmid^T
  static constexpr int U1 = a1k(DS + DV * DK * ES);    // U1^T [DV][C]
  static constexpr int DU2 = a1k(U1 + DV * C * ES);    // dU2^T [DV][C]
  static constexpr int GAM = a1k(DU2 + DV * C * ES);   // float gam1 [DK], gam2 [DK]
  // read only until dSmid is formed; then S^T [DV][DK] (from DO2) and Smid^T (from Q2)
  static constexpr int DO2 = a1k(GAM + 2 * DK * 4);    // dO of block 2
  static constexpr int A2 = a1k(DO2 + C * DV * ES);    // scale Aqk of block 2
  static constexpr int K2 = a1k(A2 + C * C * ES);      // K-tilde of block 2
  static constexpr int Q2 = a1k(K2 + C * DK * ES);     // scale Q-hat of block 2 [C][DK]
  static constexpr int W2 = a1k(Q2 + C * DK * ES);     // -W of block 2
  static constexpr int BYTES = a1k(W2 + C * DK * ES);
  static constexpr int S0 = DO2, SMID = Q2;
  static_assert(Q2 - DO2 >= DV * DK * ES && BYTES - Q2 >= DV * DK * ES, "state tiles fit the freed space");
};

template <class T, int DK, int DV>
__global__ void __launch_bounds__(MID_THREADS) chunk_mid128_kernel(ChunkBwdArgs a) {
  pdl_wait();  // dS_end comes from the reverse scan launched just before
  pdl_trigger();
  typedef MidLayout<T, DK, DV> L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  const int N = a.T / C, N2 = a.T / C2;
  const size_t c1 = (size_t)bh * N + 2 * m, c2 = c1 + 1, cm = (size_t)bh * N2 + m;
  constexpr int EPC = 16 / (int)sizeof(T);
  Tile<T, C, DV> dO1s{reinterpret_cast<T*>(sm + L::DO1)};
  Tile<T, C, DV> dO2s{reinterpret_cast<T*>(sm + L::DO2)};
  Tile<T, C, C> A1s{reinterpret_cast<T*>(sm + L::A1)};
  Tile<T, C, C> A2s{reinterpret_cast<T*>(sm + L::A2)};
  Tile<T, C, DK> Q2s{reinterpret_cast<T*>(sm + L::Q2)};
  Tile<T, C, DK> W2s{reinterpret_cast<T*>(sm + L::W2)};
  Tile<T, C, DK> K1s{reinterpret_cast<T*>(sm + L::K1)};
  Tile<T, C, DK> K2s{reinterpret_cast<T*>(sm + L::K2)};
  Tile<T, DV, DK> dSs{reinterpret_cast<T*>(sm + L::DS)};
  Tile<T, DV, C> U1s{reinterpret_cast<T*>(sm + L::U1)};
  Tile<T, DV, C> dU2s{reinterpret_cast<T*>(sm + L::DU2)};
  float* g1s = reinterpret_cast<float*>(sm + L::GAM);
  float* g2s = g1s + DK;

  const T* dout = static_cast<const T*>(a.dout);
  const size_t row0 = ((size_t)b * a.T + (size_t)m * C2) * a.H + h;
  for (int i = tid; i < C * DV / EPC; i += MID_THREADS) {
    const int r = i / (DV / EPC), c0 = (i % (DV / EPC)) * EPC;
    cp_async16(dO1s.ptr(r, c0), dout + (row0 + (size_t)r * a.H) * DV + c0);
    cp_async16(dO2s.ptr(r, c0), dout + (row0 + (size_t)(C + r) * a.H) * DV + c0);
  }
  auto rec = [&](T* dst, const void* base, size_t ch, int elems) {
    const T* src = static_cast<const T*>(base) + ch * elems;
    for (int i = tid; i < elems / EPC; i += MID_THREADS) cp_async16(dst + i * EPC, src + i * EPC);
  };
  rec(A1s.p, a.res.aqk, c1, C * C);
  rec(A2s.p, a.res.aqk, c2, C * C);
  rec(Q2s.p, a.res.qh, c2, C * DK);
  rec(W2s.p, a.res.wneg, c2, C * DK);
  rec(K1s.p, a.res.kt, c1, C * DK);
  rec(K2s.p, a.res.kt, c2, C * DK);
  rec(dSs.p, a.ws.dstate, c2, DV * DK);
  {  // U1^T: the first C columns of the 128-token U^T image are its first DV x C elements
    const T* src = static_cast<const T*>(a.res2.u) + cm * (C2 * DV);
    for (int i = tid; i < DV * C / EPC; i += MID_THREADS) cp_async16(U1s.p + i * EPC, src + i * EPC);
  }
  cp_async_commit();
  for (int c = tid; c < DK; c += MID_THREADS) {
    g1s[c] = a.res.gam[c1 * DK + c];
    g2s[c] = a.res.gam[c2 * DK + c];
  }
  {  // block 2's U: the second half of the 128-token U^T image, global to global, every
     // load of a thread before its first store
    const T* src = static_cast<const T*>(a.res2.u) + cm * (C2 * DV) + (size_t)DV * C;
    T* dst = static_cast<T*>(a.res.u) + c2 * (C * DV);
    constexpr int NIT = DV * C / EPC / MID_THREADS;
    static_assert(DV * C / EPC % MID_THREADS == 0, "whole passes");
    uint4 v[NIT];
#pragma unroll
    for (int it = 0; it < NIT; ++it) v[it] = *reinterpret_cast<const uint4*>(src + (tid + it * MID_THREADS) * EPC);
#pragma unroll
    for (int it = 0; it < NIT; ++it) *reinterpret_cast<uint4*>(dst + (tid + it * MID_THREADS) * EPC) = v[it];
  }
  cp_async_wait<0>();
  __syncthreads();

  // warp w: value rows 16 MT (w & 3) .., columns (w >> 2) N / 2 .. of a [DV][N] result
  constexpr int MT = DV / 64, NC = C / 16, NK = DK / 16;
  const int m0 = 16 * MT * (warp & 3), hf = warp >> 2;
  {  // dU2^T = dO2^T (scale Aqk2) + dS_end^T K-tilde2^T
    float acc[MT][NC][4];
    zero(acc);
    Gemm<T>::template runk<MT, NC, 0, C>(acc, aview<true>(dO2s), bview<true>(A2s), m0, hf * (C / 2), lane);
    Gemm<T>::template runk<MT, NC, 0, DK>(acc, aview<false>(dSs), bview<false>(K2s), m0, hf * (C / 2), lane);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NC; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dU2s.at(m0 + 16 * mt + frag_row(lane, e), hf * (C / 2) + 8 * nt + frag_col(lane, e)) =
              from_f32<T>(acc[mt][nt][e]);
  }
  __syncthreads();  // dU2 complete; dS_end is next read only element by element, in place
  {  // dSmid^T = dS_end^T diag(gam2) + dO2^T (scale Q-hat2) + dU2^T (-W2)
    float acc[MT][NK][4];
    zero(acc);
    Gemm<T>::template runk<MT, NK, 0, C>(acc, aview<true>(dO2s), bview<true>(Q2s), m0, hf * (DK / 2), lane);
    Gemm<T>::template runk<MT, NK, 0, C>(acc, aview<false>(dU2s), bview<true>(W2s), m0, hf * (DK / 2), lane);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NK; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = m0 + 16 * mt + frag_row(lane, e), c = hf * (DK / 2) + 8 * nt + frag_col(lane, e);
          dSs.at(v, c) = from_f32<T>(fmaf(to_f32(dSs.at(v, c)), g2s[c], acc[mt][nt][e]));
        }
  }
  __syncthreads();  // dO2, Aqk2, K-tilde2, Q-hat2 and -W2 are dead: S^T arrives in their place
  Tile<T, DV, DK> S0s{reinterpret_cast<T*>(sm + L::S0)};
  Tile<T, DV, DK> Sms{reinterpret_cast<T*>(sm + L::SMID)};
  rec(S0s.p, a.res2.state, cm, DV * DK);
  cp_async_commit();
  {  // records: block 2's dU, block 1's dS1 and U
    T* du2 = static_cast<T*>(a.ws.du) + c2 * (C * DV);
    T* ds1 = static_cast<T*>(a.ws.dstate) + c1 * (DK * DV);
    T* u1 = static_cast<T*>(a.res.u) + c1 * (C * DV);
    for (int i = tid; i < DV * C / EPC; i += MID_THREADS) {
      copy16(du2 + i * EPC, dU2s.p + i * EPC);
      copy16(u1 + i * EPC, U1s.p + i * EPC);
    }
    for (int i = tid; i < DV * DK / EPC; i += MID_THREADS) copy16(ds1 + i * EPC, dSs.p + i * EPC);
  }
  {  // dU1^T = dO1^T (scale Aqk1) + dSmid^T K-tilde1^T, straight to its record
    float acc[MT][NC][4];
    zero(acc);
    Gemm<T>::template runk<MT, NC, 0, C>(acc, aview<true>(dO1s), bview<true>(A1s), m0, hf * (C / 2), lane);
    Gemm<T>::template runk<MT, NC, 0, DK>(acc, aview<false>(dSs), bview<false>(K1s), m0, hf * (C / 2), lane);
    T* du1 = static_cast<T*>(a.ws.du) + c1 * (C * DV);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NC; ++nt)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int v = m0 + 16 * mt + frag_row(lane, e), t = hf * (C / 2) + 8 * nt + frag_col(lane, e);
          store2(du1 + Sw<T, DV, C>::off(v, t), acc[mt][nt][e], acc[mt][nt][e + 1]);
        }
  }
  {  // Smid^T = S^T diag(gam1) + U1^T K-tilde1, staged; block 1's state is S itself
    float acc[MT][NK][4];
    zero(acc);
    Gemm<T>::template runk<MT, NK, 0, C>(acc, aview<false>(U1s), bview<true>(K1s), m0, hf * (DK / 2), lane);
    cp_async_wait<0>();
    __syncthreads();  // S^T has landed
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NK; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = m0 + 16 * mt + frag_row(lane, e), c = hf * (DK / 2) + 8 * nt + frag_col(lane, e);
          Sms.at(v, c) = from_f32<T>(fmaf(to_f32(S0s.at(v, c)), g1s[c], acc[mt][nt][e]));
        }
  }
  __syncthreads();
  T* st1 = static_cast<T*>(a.res.state) + c1 * (DK * DV);
  T* st2 = static_cast<T*>(a.res.state) + c2 * (DK * DV);
  for (int i = tid; i < DV * DK / EPC; i += MID_THREADS) {
    copy16(st1 + i * EPC, S0s.p + i * EPC);
    copy16(st2 + i * EPC, Sms.p + i * EPC);
  }
}

// The reverse scan over 128-token chunks, then the 64-token blocks' records (bf16 only).
template <class T, int DK, int DV>
cudaError_t launch_rscan128(const ChunkBwdArgs& a, cudaStream_t s) {
  if constexpr (sizeof(T) != 2) {
    return cudaErrorNotSupported;  // one stage of fp32 128-token records exceeds the shared memory
  } else {
    const int BH = a.B * a.H;
    cudaError_t e;
    {
      const int bytes = RScanLayout<T, DK, C2>::BYTES + 1024;
      auto kern = chunk_scan_bwd_kernel<T, DK, DV, C2>;
      if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
        return e;
      prof_mark(K_SCAN_BWD, s, true);
      kern<<<dim3(DV / NTS, BH), RSCAN_THREADS, bytes, s>>>(a);
      prof_mark(K_SCAN_BWD, s, false);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.T < C2) return cudaSuccess;
    const int bytes = MidLayout<T, DK, DV>::BYTES + 1024;
    auto kern = chunk_mid128_kernel<T, DK, DV>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) return e;
    prof_mark(K_MID, s, true);
    e = launch_pdl(kern, dim3(a.T / C2, BH), dim3(MID_THREADS), bytes, s, a);
    prof_mark(K_MID, s, false);
    return e;
  }
}

template <class T, int DK, int DV>
cudaError_t launch_bwd_t(const ChunkBwdArgs& a, cudaStream_t s) {
  const int N = a.T / C, BH = a.B * a.H;
  const int bf16_ops = sizeof(T) == 2;
  const bool c128 = (a.flags & FLAG_CHUNK128) != 0;
  cudaError_t e;
  // bf16 with Dk = Dv = 128: the tensor-core reverse scan and one fused tensor-core kernel
  // for every chunk product and gradient (chunk_bwd_tc.cu), in one launch where they fit
  // side by side. Otherwise (Dk = 64, or fp32 operands): the CUDA-core scan, then the
  // products that need no scan result (chunk_dqa.cuh), the state products, the score
  // gradients and the channel-group sums. With 128-token chunks the scan runs over them
  // and chunk_mid128_kernel forms the 64-token blocks' records; the chunk products follow.
  const bool tc = scan_tc_applies(bf16_ops, DK, DV) && bwd_tc_applies(DK, DV);
  if (c128) {
    if ((e = launch_rscan128<T, DK, DV>(a, s)) != cudaSuccess) return e;
    if (tc) return launch_chunk_bwd_tc(a, s, true);
  } else if (tc) {
    return launch_chunk_bwd_tc(a, s);
  } else {
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
