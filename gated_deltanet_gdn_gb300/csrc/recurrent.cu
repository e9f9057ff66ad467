// Token-recurrent gated delta rule (prefill and decode are the same kernel).
//
// "gated-deltanet" kernel card, section Method: per token a decay, a read, a delta
// scaled by the write gate, a rank-one write and a read with the query; the state is
// the whole cost, so it is read from memory once and written once per call.
//
// GB300 layout: one CTA owns a (batch, head, 32-column value slice) of the fp32 state.
// The delta rule never mixes value columns (each column of S evolves with the same
// k, g, beta and its own v), so slicing Dv multiplies the number of CTAs by Dv / 32
// without any exchange. Inside a CTA, 16 threads share a group of 4 value columns and
// each holds Dk / 16 key rows of those columns in registers; the two Dk reductions per
// token (S^T k and S^T q) are 16-lane butterfly shuffles in a fixed order, so a
// sequence split into several calls gives bit-identical results. Token inputs are
// staged through shared memory in batches of TB tokens with cp.async double buffering.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int REC_COLS = 32;                 // value columns per CTA
constexpr int REC_VEC = 4;                   // value columns per thread
constexpr int REC_TPC = 16;                  // threads sharing a column group
constexpr int REC_THREADS = (REC_COLS / REC_VEC) * REC_TPC;  // 128
// Tokens per staged batch (TB): 16, in dynamic shared memory (about 61 KB at Dk = 128 fp32,
// three CTAs per SM); a batch boundary costs one wait and one barrier.

template <class T, int DK, int TB>
struct RecSmem {
  T q[2][TB][DK];
  T k[2][TB][DK];
  T v[2][TB][REC_COLS];
  T graw[2][TB][DK];  // per-channel g (scalar g uses gs)
  float a[TB][DK];    // exp(g) of the batch being computed
  float gs[2][TB];    // scalar decay: exp(g) per token
  float beta[2][TB];
  float inv[2][TB];   // q/k L2 normalisation: inverse norms of the batch's q and k rows
};

// Packed fp32 pairs (Blackwell f32x2 arithmetic): one instruction does the fp32 operation
// on both halves with the same rounding as the scalar one, so the state update below is
// element for element the scalar arithmetic of decode_kernel, in half the instructions.
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
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// QK: q/k L2 normalisation (GDN_FLAG_QK_L2NORM) is compiled in only when asked for, so
// the plain per-token chain carries no extra multiplies.
template <class T, int DK, bool PC, int TB, bool QK>
__global__ void __launch_bounds__(REC_THREADS) recurrent_kernel(RecurrentArgs p) {
  constexpr int RPT = DK / REC_TPC;  // key rows per thread
  extern __shared__ __align__(16) uint8_t rec_smem[];
  RecSmem<T, DK, TB>& sm = *reinterpret_cast<RecSmem<T, DK, TB>*>(rec_smem);
  const int tid = threadIdx.x;
  const int cg = tid / REC_TPC;    // column group 0..7
  const int part = tid % REC_TPC;  // row interleave 0..15
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int col0 = blockIdx.x * REC_COLS + cg * REC_VEC;
  const int DV = p.DV, H = p.H, T_ = p.T;

  // state slice: rows part + 16 i, columns col0 .. col0 + 3, as two packed pairs per row
  static_assert(REC_VEC == 4, "two packed pairs per row");
  uint64_t S[RPT][2];
  const size_t sbase = (size_t)bh * DK * DV;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = part + REC_TPC * i;
    if (p.h0) {
      const float4 x = *reinterpret_cast<const float4*>(p.h0 + sbase + (size_t)r * DV + col0);
      S[i][0] = f2_pack(x.x, x.y);
      S[i][1] = f2_pack(x.z, x.w);
    } else {
      S[i][0] = S[i][1] = f2_pack(0.f, 0.f);
    }
  }

  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);
  const T* g = static_cast<const T*>(p.g);
  const T* beta = static_cast<const T*>(p.beta);
  constexpr int EPC = 16 / (int)sizeof(T);  // elements per 16-byte copy

  auto stage = [&](int buf, int t0) {
    const int nt = min(TB, T_ - t0);
    // q, k (and per-channel g): rows of DK elements
    constexpr int CPR = DK / EPC;  // copies per row
    for (int i = tid; i < nt * CPR; i += REC_THREADS) {
      const int tt = i / CPR, c = (i % CPR) * EPC;
      const size_t row = ((size_t)b * T_ + t0 + tt) * H + h;
      cp_async16(&sm.q[buf][tt][c], q + row * DK + c);
      cp_async16(&sm.k[buf][tt][c], k + row * DK + c);
      if (PC) cp_async16(&sm.graw[buf][tt][c], g + row * DK + c);
    }
    constexpr int VPR = REC_COLS / EPC;
    for (int i = tid; i < nt * VPR; i += REC_THREADS) {
      const int tt = i / VPR, c = (i % VPR) * EPC;
      const size_t row = ((size_t)b * T_ + t0 + tt) * H + h;
      cp_async16(&sm.v[buf][tt][c], v + row * DV + blockIdx.x * REC_COLS + c);
    }
    if (tid < nt) {
      const size_t row = ((size_t)b * T_ + t0 + tid) * H + h;
      sm.beta[buf][tid] = to_f32(beta[row]);
      if (!PC) sm.gs[buf][tid] = expf(to_f32(g[row]));  // the decay factor, off the token chain
    }
    cp_async_commit();
  };

  // The loop is software-pipelined by one token: token t's output partials are reduced in
  // the same butterfly as token t + 1's S^T k, and written then.
  float ovp[REC_VEC] = {0.f, 0.f, 0.f, 0.f};
  size_t rowp = 0;
  bool pend = false;
  auto write_out = [&](size_t row, const float (&ov)[REC_VEC]) {
    if (part != 0) return;
    T* o = static_cast<T*>(p.out) + row * DV + col0;
    if (sizeof(T) == 4) {
      *reinterpret_cast<float4*>(o) = make_float4(p.scale * ov[0], p.scale * ov[1], p.scale * ov[2], p.scale * ov[3]);
    } else {
      __align__(8) T tmp[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) tmp[j] = from_f32<T>(p.scale * ov[j]);
      *reinterpret_cast<uint2*>(o) = *reinterpret_cast<const uint2*>(tmp);
    }
  };

  const int nbatch = (T_ + TB - 1) / TB;
  if (nbatch > 0) stage(0, 0);
  for (int bi = 0; bi < nbatch; ++bi) {
    const int buf = bi & 1, t0 = bi * TB, nt = min(TB, T_ - t0);
    cp_async_wait<0>();
    __syncthreads();  // batch bi visible; everyone finished batch bi-1 (its buffer is free)
    if (bi + 1 < nbatch) stage(buf ^ 1, t0 + TB);
    if (PC || QK) {
      if (PC)
        for (int i = tid; i < nt * DK; i += REC_THREADS) {
          const int tt = i / DK, c = i % DK;
          sm.a[tt][c] = expf(to_f32(sm.graw[buf][tt][c]));
        }
      if (QK) {  // one warp per q or k row of the batch
        const int warp = tid >> 5, lane = tid & 31;
        for (int rr = warp; rr < 2 * nt; rr += REC_THREADS / 32) {
          const float inv = warp_row_inv_norm<DK>((rr & 1) ? sm.k[buf][rr >> 1] : sm.q[buf][rr >> 1], lane);
          if (lane == 0) sm.inv[rr & 1][rr >> 1] = inv;
        }
      }
      __syncthreads();
    }
    for (int tt = 0; tt < nt; ++tt) {
      const float bt = sm.beta[buf][tt];
      const float as = PC ? 1.f : sm.gs[buf][tt];
      const float nq = QK ? sm.inv[0][tt] : 1.f, nk = QK ? sm.inv[1][tt] : 1.f;
      uint64_t pv2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int r = part + REC_TPC * i;
        const float a = PC ? sm.a[tt][r] : as;
        const float kr = to_f32(sm.k[buf][tt][r]) * nk;
        const uint64_t a2 = f2_pack(a, a), k2 = f2_pack(kr, kr);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          S[i][h2] = f2_mul(S[i][h2], a2);
          pv2[h2] = f2_fma(S[i][h2], k2, pv2[h2]);
        }
      }
      float pv[REC_VEC];
      f2_unpack(pv2[0], pv[0], pv[1]);
      f2_unpack(pv2[1], pv[2], pv[3]);
      // one butterfly for this token's S^T k and the previous token's output partials:
      // the two reductions are independent, and each keeps its own order (xor 1, 2, 4, 8)
#pragma unroll
      for (int off = 1; off < REC_TPC; off <<= 1)
#pragma unroll
        for (int j = 0; j < REC_VEC; ++j) {
          pv[j] += __shfl_xor_sync(0xffffffffu, pv[j], off);
          ovp[j] += __shfl_xor_sync(0xffffffffu, ovp[j], off);
        }
      if (pend) write_out(rowp, ovp);
      float d[REC_VEC];
#pragma unroll
      for (int j = 0; j < REC_VEC; ++j) d[j] = bt * (to_f32(sm.v[buf][tt][cg * REC_VEC + j]) - pv[j]);
      const uint64_t d2[2] = {f2_pack(d[0], d[1]), f2_pack(d[2], d[3])};
      uint64_t ov2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int r = part + REC_TPC * i;
        const float kr = to_f32(sm.k[buf][tt][r]) * nk;
        const float qr = to_f32(sm.q[buf][tt][r]) * nq;
        const uint64_t k2 = f2_pack(kr, kr), q2 = f2_pack(qr, qr);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          S[i][h2] = f2_fma(k2, d2[h2], S[i][h2]);
          ov2[h2] = f2_fma(S[i][h2], q2, ov2[h2]);
        }
      }
      f2_unpack(ov2[0], ovp[0], ovp[1]);
      f2_unpack(ov2[1], ovp[2], ovp[3]);
      rowp = ((size_t)b * T_ + t0 + tt) * H + h;
      pend = true;
    }
  }
  if (pend) {  // the last token's output
#pragma unroll
    for (int off = 1; off < REC_TPC; off <<= 1)
#pragma unroll
      for (int j = 0; j < REC_VEC; ++j) ovp[j] += __shfl_xor_sync(0xffffffffu, ovp[j], off);
    write_out(rowp, ovp);
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = part + REC_TPC * i;
    float4 x;
    f2_unpack(S[i][0], x.x, x.y);
    f2_unpack(S[i][1], x.z, x.w);
    *reinterpret_cast<float4*>(p.h_final + sbase + (size_t)r * DV + col0) = x;
  }
}

template <class T, int DK, int TB, bool PC, bool QK>
cudaError_t launch_rec_one(const RecurrentArgs& a, cudaStream_t s) {
  auto kern = recurrent_kernel<T, DK, PC, TB, QK>;
  const int bytes = (int)sizeof(RecSmem<T, DK, TB>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  kern<<<dim3(a.DV / REC_COLS, a.B * a.H), REC_THREADS, bytes, s>>>(a);
  return cudaGetLastError();
}

template <class T, int DK, int TB>
cudaError_t launch_rec_tb(const RecurrentArgs& a, cudaStream_t s) {
  if (a.qk_norm)
    return a.per_channel ? launch_rec_one<T, DK, TB, true, true>(a, s) : launch_rec_one<T, DK, TB, false, true>(a, s);
  return a.per_channel ? launch_rec_one<T, DK, TB, true, false>(a, s) : launch_rec_one<T, DK, TB, false, false>(a, s);
}

template <class T, int DK>
cudaError_t launch_rec_t(const RecurrentArgs& a, cudaStream_t s) {
  prof_mark(K_RECURRENT, s, true);
  const cudaError_t e = launch_rec_tb<T, DK, 16>(a, s);  // single-token calls go to decode_kernel (decode.cu)
  prof_mark(K_RECURRENT, s, false);
  return e;
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentArgs& a, cudaStream_t s) {
  if (a.B * a.H == 0) return cudaSuccess;
  if (a.T == 1) return launch_decode(a, s);  // same arithmetic, shaped for one token
  if (a.bf16) return a.DK == 64 ? launch_rec_t<bf16, 64>(a, s) : launch_rec_t<bf16, 128>(a, s);
  return a.DK == 64 ? launch_rec_t<float, 64>(a, s) : launch_rec_t<float, 128>(a, s);
}

}  // namespace gdn
