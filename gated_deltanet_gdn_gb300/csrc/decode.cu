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
// GB300 layout: persistent CTAs, each taking work units u = blockIdx.x,
// blockIdx.x + gridDim.x, ... A unit is NC value columns of one (batch, head) state:
//  * NC = Dv (batches with at least as many heads as SMs): a whole head, its state
//    (64 KiB at Dk = Dv = 128) moved by one cp.async.bulk each way, one CTA per SM;
//  * NC = 32 (fewer heads than SMs, e.g. B2 H48): a 32-column slice of a head, moved by
//    2-D TMA tensor copies (box 32 columns x Dk rows of the [B*H*Dk, Dv] fp32 state),
//    so B*H*Dv/32 CTAs share the SMs instead of B*H. The delta rule never mixes value
//    columns, so a slice needs only its own columns plus the whole q, k, g rows.
// A producer warp streams each unit's state and token row into a three-stage ring and,
// once the compute warps have updated the state in place, stores it back; two units'
// states are in flight while a third is computed. Compute thread (w, l) takes columns
// 4 cg .. 4 cg + 3 of the unit and key rows part + 16 i with cg = 8 (w mod NC/32) + l mod 8
// and part = 4 (w div NC/32) + l div 8, so a quarter warp reads one 128-byte state row
// segment (no bank conflicts) and the first two butterfly levels are lane shuffles
// (xor 8, 16), the last two a shared-memory exchange. The arithmetic of a column does not
// depend on NC: both unit widths give the same bits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

template <class T, int DK, int NC>
struct DecLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int STATE = 0;                      // fp32 [DK][NC]
  static constexpr int Q = STATE + DK * NC * 4;        // token row q [DK]
  static constexpr int K = Q + DK * ES;                // k [DK]
  static constexpr int V = K + DK * ES;                // v, the unit's NC columns
  static constexpr int G = V + NC * ES;                // per-channel g [DK]
  static constexpr int STAGE = a1k(G + DK * ES);
  static constexpr int STAGES = 3;
  static constexpr int RED = STAGES * STAGE;           // float [2][4][NC]: pv and ov partials
  static constexpr int A = RED + 2 * 4 * NC * 4;       // float [DK] exp(g)
  static constexpr int NINV = A + DK * 4;              // float [2]: q, k inverse norms
  static constexpr int BAR = NINV + 16;                // full[STAGES], computed[STAGES]
  static constexpr int BYTES = BAR + 16 * STAGES;
  static constexpr int COMPUTE = NC / 4 * 16;          // threads: 4 columns x 16 row parts each
  static constexpr int THREADS = COMPUTE + 32;         // + the producer warp
};

// 2-D tensor copies of a state slice (box NC columns x DK rows), global <-> shared.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}

__device__ __forceinline__ void decode_sync(int n) { asm volatile("bar.sync 1, %0;\n" ::"r"(n) : "memory"); }

// h0_map, hf_map: the [B*H*DK, DV] fp32 h0 and h_final as 2-D tensors, box NC x DK
// (used only when NC < DV; h0_map only when h0 is not NULL).
template <class T, int DK, int DV, int NC, bool PC>
__global__ void __launch_bounds__(DecLayout<T, DK, NC>::THREADS, 1)
    decode_kernel(RecurrentArgs p, const __grid_constant__ CUtensorMap h0_map,
                  const __grid_constant__ CUtensorMap hf_map) {
  typedef DecLayout<T, DK, NC> L;
  constexpr int RPT = DK / 16;      // key rows per thread
  constexpr int WPR = NC / 32;      // warps per row-part quarter
  constexpr int NS = DV / NC;       // units per head
  constexpr bool SLICE = NC < DV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H * NS;  // units
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* computed = full + L::STAGES;
  float* red = reinterpret_cast<float*>(sm + L::RED);
  float* aexp = reinterpret_cast<float*>(sm + L::A);
  float* ninv = reinterpret_cast<float*>(sm + L::NINV);
  const int nunits = (BH - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // units of this CTA

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
  constexpr uint32_t SB = (uint32_t)(DK * NC * 4);

  if (warp == L::COMPUTE / 32) {  // ---- producer
    if (lane == 0) {
      auto store_back = [&](int m) {  // the updated state of this CTA's m-th unit
        const int s = m % L::STAGES, u = (int)blockIdx.x + m * (int)gridDim.x, j = u / NS, sl = u % NS;
        mbar_wait(&computed[s], (uint32_t)(m / L::STAGES) & 1u, p.err);
        if (SLICE)
          tma_store_2d(&hf_map, sl * NC, j * DK, sm + s * L::STAGE + L::STATE);
        else
          bulk_s2g(p.h_final + (size_t)j * DK * DV, sm + s * L::STAGE + L::STATE, SB);
        bulk_commit();
      };
      for (int m = 0; m < nunits; ++m) {
        const int s = m % L::STAGES, u = (int)blockIdx.x + m * (int)gridDim.x, j = u / NS, sl = u % NS;
        if (m >= L::STAGES) {
          store_back(m - L::STAGES);
          bulk_wait_read0();  // the stage's old state has left shared memory
        }
        uint8_t* st = sm + s * L::STAGE;
        const size_t row = (size_t)(j / p.H) * p.H + (j % p.H);  // token 0 of (b, h): (b * T + 0) * H + h
        const uint32_t tx = (p.h0 ? SB : 0u) + (uint32_t)((2 * DK + NC + (PC ? DK : 0)) * sizeof(T));
        mbar_arrive_expect_tx(&full[s], tx);
        if (p.h0) {
          if (SLICE)
            tma_load_2d(st + L::STATE, &h0_map, sl * NC, j * DK, &full[s]);
          else
            bulk_g2s(st + L::STATE, p.h0 + (size_t)j * DK * DV, SB, &full[s]);
        }
        bulk_g2s(st + L::Q, q + row * DK, DK * sizeof(T), &full[s]);
        bulk_g2s(st + L::K, k + row * DK, DK * sizeof(T), &full[s]);
        bulk_g2s(st + L::V, v + row * DV + sl * NC, NC * sizeof(T), &full[s]);
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
    const int s = m % L::STAGES, u = (int)blockIdx.x + m * (int)gridDim.x, j = u / NS, sl = u % NS;
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
        const float4 x = *reinterpret_cast<const float4*>(S_sm + r * NC + 4 * cg);
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
    if (pl == 0) *reinterpret_cast<float4*>(red + ph * NC + 4 * cg) = make_float4(pv[0], pv[1], pv[2], pv[3]);
    decode_sync(L::COMPUTE);
    float d[4];
    {
      const float4 r0 = *reinterpret_cast<const float4*>(red + 0 * NC + 4 * cg);
      const float4 r1 = *reinterpret_cast<const float4*>(red + 1 * NC + 4 * cg);
      const float4 r2 = *reinterpret_cast<const float4*>(red + 2 * NC + 4 * cg);
      const float4 r3 = *reinterpret_cast<const float4*>(red + 3 * NC + 4 * cg);
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
      *reinterpret_cast<float4*>(S_sm + r * NC + 4 * cg) = make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
    }
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1)
#pragma unroll
      for (int e = 0; e < 4; ++e) ov[e] += __shfl_xor_sync(0xffffffffu, ov[e], off);
    float* red2 = red + 4 * NC;
    if (pl == 0) *reinterpret_cast<float4*>(red2 + ph * NC + 4 * cg) = make_float4(ov[0], ov[1], ov[2], ov[3]);
    fence_proxy_async();  // the updated state is read by the producer's bulk store
    decode_sync(L::COMPUTE);
    if (tid < NC / 4) {  // one thread per column group writes the output
      const int c4 = 4 * tid;
      const float4 r0 = *reinterpret_cast<const float4*>(red2 + 0 * NC + c4);
      const float4 r1 = *reinterpret_cast<const float4*>(red2 + 1 * NC + c4);
      const float4 r2 = *reinterpret_cast<const float4*>(red2 + 2 * NC + c4);
      const float4 r3 = *reinterpret_cast<const float4*>(red2 + 3 * NC + c4);
      const float o[4] = {(r0.x + r1.x) + (r2.x + r3.x), (r0.y + r1.y) + (r2.y + r3.y),
                          (r0.z + r1.z) + (r2.z + r3.z), (r0.w + r1.w) + (r2.w + r3.w)};
      T* out = static_cast<T*>(p.out) + row * DV + sl * NC + c4;
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

// [B*H*DK, DV] fp32 state as a 2-D tensor map with box NC columns x DK rows.
template <int DK, int DV, int NC>
bool state_map(CUtensorMap* map, const float* base, int BH) {
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
  if (!encode) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)DV, (cuuint64_t)BH * DK};
  const cuuint64_t strides[1] = {(cuuint64_t)DV * 4};
  const cuuint32_t box[2] = {(cuuint32_t)NC, (cuuint32_t)DK};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class T, int DK, int DV, int NC>
cudaError_t launch_dec_nc(const RecurrentArgs& a, cudaStream_t s, int grid) {
  typedef DecLayout<T, DK, NC> L;
  const int bytes = L::BYTES + 1024;
  auto kern = a.per_channel ? decode_kernel<T, DK, DV, NC, true> : decode_kernel<T, DK, DV, NC, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  CUtensorMap h0_map{}, hf_map{};
  if (NC < DV) {
    if (!state_map<DK, DV, NC>(&hf_map, a.h_final, a.B * a.H)) return cudaErrorInvalidValue;
    if (a.h0 && !state_map<DK, DV, NC>(&h0_map, a.h0, a.B * a.H)) return cudaErrorInvalidValue;
  }
  prof_mark(K_DECODE, s, true);
  kern<<<grid, L::THREADS, bytes, s>>>(a, h0_map, hf_map);
  prof_mark(K_DECODE, s, false);
  return cudaGetLastError();
}

// Whole heads when there are at least as many as SMs (one persistent CTA per SM);
// otherwise 32-column slices, one CTA per slice, so that every SM takes part.
template <class T, int DK, int DV>
cudaError_t launch_dec_t(const RecurrentArgs& a, cudaStream_t s) {
  const int nsm = sm_count();
  const int BH = a.B * a.H;
  if (nsm > 0 && BH >= nsm) return launch_dec_nc<T, DK, DV, DV>(a, s, nsm);
  return launch_dec_nc<T, DK, DV, 32>(a, s, BH * (DV / 32));
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
