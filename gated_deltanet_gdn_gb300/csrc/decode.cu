// Single-token decode step of the gated delta rule (T = 1): the state of every
// (batch, head) is read once and written once, so the step is a stream over the
// fp32 states and the kernel is shaped to keep HBM busy.
//
// "gated-deltanet" kernel card, section Method: per token a decay, a read S^T k, a
// delta beta (v - S^T k), a rank-one write k d^T and a read S^T q. This kernel does
// exactly the arithmetic of recurrent_kernel (recurrent.cu) for one token, in the same
// order, so a sequence decoded one token per call equals one prefill call bitwise:
// per value column, 16 partial sums over the key rows c = p (mod 16), each an fmaf
// chain over ascending rows, combined by the same balanced tree as recurrent_kernel's
// 16-lane butterfly (((x0 + x1) + (x2 + x3)) + ...).
//
// GB300 layout: persistent CTAs (one per SM), each taking heads j = blockIdx.x,
// blockIdx.x + gridDim.x, ... A producer warp streams a head's whole state (64 KiB at
// Dk = Dv = 128, one cp.async.bulk) and its token row into a three-stage ring and, once
// the compute warps have updated the state in place, stores it back with a bulk copy;
// two heads' states are in flight while a third is computed. Compute thread (w, l)
// takes value columns 4 cg .. 4 cg + 3 and key rows part + 16 i with
// cg = 8 (w mod Dv/32) + l mod 8 and part = 4 (w div Dv/32) + l div 8, so a quarter
// warp reads one 128-byte state row segment (no bank conflicts) and the first two
// butterfly levels are lane shuffles (xor 8, 16), the last two a shared-memory exchange.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

template <class T, int DK, int DV>
struct DecLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int STATE = 0;                      // fp32 [DK][DV]
  static constexpr int Q = STATE + DK * DV * 4;        // token row q [DK]
  static constexpr int K = Q + DK * ES;                // k [DK]
  static constexpr int V = K + DK * ES;                // v [DV]
  static constexpr int G = V + DV * ES;                // per-channel g [DK]
  static constexpr int STAGE = a1k(G + DK * ES);
  static constexpr int STAGES = 3;
  static constexpr int RED = STAGES * STAGE;           // float [2][4][DV]: pv and ov partials
  static constexpr int A = RED + 2 * 4 * DV * 4;       // float [DK] exp(g)
  static constexpr int NINV = A + DK * 4;              // float [2]: q, k inverse norms
  static constexpr int BAR = NINV + 16;                // full[STAGES], computed[STAGES]
  static constexpr int BYTES = BAR + 16 * STAGES;
  static constexpr int COMPUTE = DV / 4 * 16;          // threads: 4 columns x 16 row parts each
  static constexpr int THREADS = COMPUTE + 32;         // + the producer warp
};

__device__ __forceinline__ void decode_sync(int n) { asm volatile("bar.sync 1, %0;\n" ::"r"(n) : "memory"); }

template <class T, int DK, int DV, bool PC>
__global__ void __launch_bounds__(DecLayout<T, DK, DV>::THREADS, 1) decode_kernel(RecurrentArgs p) {
  typedef DecLayout<T, DK, DV> L;
  constexpr int RPT = DK / 16;      // key rows per thread
  constexpr int WPR = DV / 32;      // warps per row-part quarter
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* computed = full + L::STAGES;
  float* red = reinterpret_cast<float*>(sm + L::RED);
  float* aexp = reinterpret_cast<float*>(sm + L::A);
  float* ninv = reinterpret_cast<float*>(sm + L::NINV);
  const int nunits = (BH - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // heads of this CTA

  if (tid == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&computed[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);
  const T* g = static_cast<const T*>(p.g);
  const T* beta = static_cast<const T*>(p.beta);
  constexpr uint32_t SB = (uint32_t)(DK * DV * 4);

  if (warp == L::COMPUTE / 32) {  // ---- producer
    if (lane == 0) {
      auto store_back = [&](int m) {  // the updated state of this CTA's m-th head
        const int s = m % L::STAGES, j = (int)blockIdx.x + m * (int)gridDim.x;
        mbar_wait(&computed[s], (uint32_t)(m / L::STAGES) & 1u, p.err);
        bulk_s2g(p.h_final + (size_t)j * DK * DV, sm + s * L::STAGE + L::STATE, SB);
        bulk_commit();
      };
      for (int m = 0; m < nunits; ++m) {
        const int s = m % L::STAGES, j = (int)blockIdx.x + m * (int)gridDim.x;
        if (m >= L::STAGES) {
          store_back(m - L::STAGES);
          bulk_wait_read0();  // the stage's old state has left shared memory
        }
        uint8_t* st = sm + s * L::STAGE;
        const size_t row = (size_t)(j / p.H) * p.H + (j % p.H);  // token 0 of (b, h): (b * T + 0) * H + h
        const uint32_t tx = (p.h0 ? SB : 0u) + (uint32_t)((2 * DK + DV + (PC ? DK : 0)) * sizeof(T));
        mbar_arrive_expect_tx(&full[s], tx);
        if (p.h0) bulk_g2s(st + L::STATE, p.h0 + (size_t)j * DK * DV, SB, &full[s]);
        bulk_g2s(st + L::Q, q + row * DK, DK * sizeof(T), &full[s]);
        bulk_g2s(st + L::K, k + row * DK, DK * sizeof(T), &full[s]);
        bulk_g2s(st + L::V, v + row * DV, DV * sizeof(T), &full[s]);
        if (PC) bulk_g2s(st + L::G, g + row * DK, DK * sizeof(T), &full[s]);
      }
      for (int m = nunits > L::STAGES ? nunits - L::STAGES : 0; m < nunits; ++m) store_back(m);
      drain_ring(full, L::STAGES, nunits);
      bulk_wait0();
    }
    return;
  }

  // ---- compute warps
  const int cg = 8 * (warp % WPR) + (lane & 7);   // column group: columns 4 cg .. 4 cg + 3
  const int ph = warp / WPR, pl = lane >> 3;      // row part = 4 ph + pl
  const int part = 4 * ph + pl;
#pragma unroll 1
  for (int m = 0; m < nunits; ++m) {
    const int s = m % L::STAGES, j = (int)blockIdx.x + m * (int)gridDim.x;
    const size_t row = (size_t)(j / p.H) * p.H + (j % p.H);
    uint8_t* st = sm + s * L::STAGE;
    float* S_sm = reinterpret_cast<float*>(st + L::STATE);
    const T* qs = reinterpret_cast<const T*>(st + L::Q);
    const T* ks = reinterpret_cast<const T*>(st + L::K);
    const T* vs = reinterpret_cast<const T*>(st + L::V);
    const float bt = to_f32(beta[row]);
    const float as = PC ? 1.f : expf(to_f32(g[row]));
    mbar_wait(&full[s], (uint32_t)(m / L::STAGES) & 1u, p.err);
    if (PC || p.qk_norm) {
      if (PC) {
        const T* gs = reinterpret_cast<const T*>(st + L::G);
        for (int c = tid; c < DK; c += L::COMPUTE) aexp[c] = expf(to_f32(gs[c]));
      }
      if (p.qk_norm && warp < 2) {  // warp 0: the q row, warp 1: the k row
        const float inv = warp_row_inv_norm<DK>(warp ? ks : qs, lane);
        if (lane == 0) ninv[warp] = inv;
      }
      decode_sync(L::COMPUTE);
    }
    const float nq = p.qk_norm ? ninv[0] : 1.f, nk = p.qk_norm ? ninv[1] : 1.f;
    float S[RPT][4];
    float pv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = part + 16 * i;
      if (p.h0) {
        const float4 x = *reinterpret_cast<const float4*>(S_sm + r * DV + 4 * cg);
        S[i][0] = x.x; S[i][1] = x.y; S[i][2] = x.z; S[i][3] = x.w;
      } else {
        S[i][0] = S[i][1] = S[i][2] = S[i][3] = 0.f;
      }
      const float a = PC ? aexp[r] : as;
      const float kr = to_f32(ks[r]) * nk;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        S[i][e] *= a;
        pv[e] = fmaf(S[i][e], kr, pv[e]);
      }
    }
    // row parts xor 1 and xor 2 are lanes xor 8 and xor 16; parts xor 4 and xor 8 are
    // the four warps ph = 0..3, combined as (s0 + s1) + (s2 + s3)
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1)
#pragma unroll
      for (int e = 0; e < 4; ++e) pv[e] += __shfl_xor_sync(0xffffffffu, pv[e], off);
    if (pl == 0) *reinterpret_cast<float4*>(red + ph * DV + 4 * cg) = make_float4(pv[0], pv[1], pv[2], pv[3]);
    decode_sync(L::COMPUTE);
    float d[4];
    {
      const float4 r0 = *reinterpret_cast<const float4*>(red + 0 * DV + 4 * cg);
      const float4 r1 = *reinterpret_cast<const float4*>(red + 1 * DV + 4 * cg);
      const float4 r2 = *reinterpret_cast<const float4*>(red + 2 * DV + 4 * cg);
      const float4 r3 = *reinterpret_cast<const float4*>(red + 3 * DV + 4 * cg);
      const float t[4] = {(r0.x + r1.x) + (r2.x + r3.x), (r0.y + r1.y) + (r2.y + r3.y),
                          (r0.z + r1.z) + (r2.z + r3.z), (r0.w + r1.w) + (r2.w + r3.w)};
#pragma unroll
      for (int e = 0; e < 4; ++e) d[e] = bt * (to_f32(vs[4 * cg + e]) - t[e]);
    }
    float ov[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = part + 16 * i;
      const float kr = to_f32(ks[r]) * nk;
      const float qr = to_f32(qs[r]) * nq;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        S[i][e] = fmaf(kr, d[e], S[i][e]);
        ov[e] = fmaf(S[i][e], qr, ov[e]);
      }
      *reinterpret_cast<float4*>(S_sm + r * DV + 4 * cg) = make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
    }
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1)
#pragma unroll
      for (int e = 0; e < 4; ++e) ov[e] += __shfl_xor_sync(0xffffffffu, ov[e], off);
    float* red2 = red + 4 * DV;
    if (pl == 0) *reinterpret_cast<float4*>(red2 + ph * DV + 4 * cg) = make_float4(ov[0], ov[1], ov[2], ov[3]);
    fence_proxy_async();  // the updated state is read by the producer's bulk store
    decode_sync(L::COMPUTE);
    if (tid < DV / 4) {  // one thread per column group writes the output
      const int c4 = 4 * tid;
      const float4 r0 = *reinterpret_cast<const float4*>(red2 + 0 * DV + c4);
      const float4 r1 = *reinterpret_cast<const float4*>(red2 + 1 * DV + c4);
      const float4 r2 = *reinterpret_cast<const float4*>(red2 + 2 * DV + c4);
      const float4 r3 = *reinterpret_cast<const float4*>(red2 + 3 * DV + c4);
      const float o[4] = {(r0.x + r1.x) + (r2.x + r3.x), (r0.y + r1.y) + (r2.y + r3.y),
                          (r0.z + r1.z) + (r2.z + r3.z), (r0.w + r1.w) + (r2.w + r3.w)};
      T* out = static_cast<T*>(p.out) + row * DV + c4;
      if (sizeof(T) == 4) {
        *reinterpret_cast<float4*>(out) = make_float4(p.scale * o[0], p.scale * o[1], p.scale * o[2], p.scale * o[3]);
      } else {
        __align__(8) T tmp[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) tmp[e] = from_f32<T>(p.scale * o[e]);
        *reinterpret_cast<uint2*>(out) = *reinterpret_cast<const uint2*>(tmp);
      }
    }
    if (tid == 0) mbar_arrive(&computed[s]);
    decode_sync(L::COMPUTE);  // the reduction buffers are reused by the next head
  }
}

int sm_count() {
  static int n[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev];
}

template <class T, int DK, int DV>
cudaError_t launch_dec_t(const RecurrentArgs& a, cudaStream_t s) {
  typedef DecLayout<T, DK, DV> L;
  const int bytes = L::BYTES + 1024;
  auto kern = a.per_channel ? decode_kernel<T, DK, DV, true> : decode_kernel<T, DK, DV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  const int nsm = sm_count();
  const int BH = a.B * a.H;
  const int grid = nsm > 0 && BH > nsm ? nsm : BH;
  prof_mark(K_DECODE, s, true);
  kern<<<grid, L::THREADS, bytes, s>>>(a);
  prof_mark(K_DECODE, s, false);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const RecurrentArgs& a, cudaStream_t s) {
  if (a.bf16) {
    if (a.DK == 128) return a.DV == 128 ? launch_dec_t<bf16, 128, 128>(a, s) : launch_dec_t<bf16, 128, 64>(a, s);
    return a.DV == 128 ? launch_dec_t<bf16, 64, 128>(a, s) : launch_dec_t<bf16, 64, 64>(a, s);
  }
  if (a.DK == 128) return a.DV == 128 ? launch_dec_t<float, 128, 128>(a, s) : launch_dec_t<float, 128, 64>(a, s);
  return a.DV == 128 ? launch_dec_t<float, 64, 128>(a, s) : launch_dec_t<float, 64, 64>(a, s);
}

}  // namespace gdn
