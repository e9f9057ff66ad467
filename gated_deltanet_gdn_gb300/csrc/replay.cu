// Decode with the state held as a checkpoint plus a buffer of recent tokens, after the
// ReplaySSM summary on the ai4snews "Gated DeltaNet" topic page (item "SSM decoding
// stops writing state every step"): the checkpoint is read every step but written only
// when the buffer is full, and every step's output is computed directly from the
// checkpoint and the buffered tokens.
//
// The algebra is the gated delta rule ("gated-deltanet" kernel card, section Method)
// unrolled from the checkpoint S_c. With G_j = sum of the log-decays of buffered tokens
// 0..j (per key channel, counted from the checkpoint) and d_j = beta_j (v_j - S'_j^T k_j)
// the delta of token j, the state after token n is
//     S_n = diag(exp(G_n)) S_c + sum_{j<=n} diag(exp(G_n - G_j)) k_j d_j^T,
// so the new token n needs only reads of S_c:
//     d_n = beta_n (v_n - S_c^T (exp(G_n) k_n) - sum_{j<n} a_j d_j),
//     o_n = scale (S_c^T (exp(G_n) q_n) + sum_{j<n} b_j d_j + (q_n . k_n) d_n),
//     a_j = sum_c k_nc k_jc exp(G_nc - G_jc),  b_j = sum_c q_nc k_jc exp(G_nc - G_jc).
// Every exponent is <= 0 (G only falls along the buffer), so no factor can overflow,
// whatever the decay. A buffer slot holds (k_j, G_j, d_j) in fp32. When a step finds
// the buffer full (fill == L) it first folds it into the checkpoint,
//     S_c <- diag(exp(G_{L-1})) S_c + sum_j diag(exp(G_{L-1} - G_j)) k_j d_j^T,
// writes S_c back, and then processes its token against the new checkpoint as slot 0.
// Rolling back r <= fill tokens (speculative decoding) is lowering fill by r.
//
// GB300 layout: persistent CTAs like decode_kernel; a producer warp streams each head's
// checkpoint (one cp.async.bulk of Dk*Dv*4 bytes), its filled slots and its token row
// into a two-stage ring. The checkpoint region of a stage is released as soon as the
// compute threads hold the state in registers (mbarrier `sfree`), the rest once the
// head is done (`computed`), so the next head's checkpoint streams in during the
// head's pairwise and output phases. Compute thread (w, l) holds the state elements of
// value columns 4 cg .. 4 cg + 3 and key rows part + 16 i, as in decode_kernel.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr unsigned ERR_REPLAY_FILL = 2u;  // a fill count outside [0, L]

template <class T, int DK, int DV>
struct RepLayout {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int SLOTF = 2 * DK + DV;              // floats per slot: k, G, d
  static constexpr int SLOTB = SLOTF * 4;
  static constexpr int STATE = 0;                        // fp32 [DK][DV] checkpoint
  static constexpr int SLOTS = STATE + DK * DV * 4;      // [REPLAY_MAX_TOKENS][SLOTF]
  static constexpr int Q = SLOTS + REPLAY_MAX_TOKENS * SLOTB;
  static constexpr int K = Q + DK * ES;
  static constexpr int V = K + DK * ES;
  static constexpr int G = V + DV * ES;
  static constexpr int STAGE = a1k(G + DK * ES);
  static constexpr int STAGES = 2;
  static constexpr int RED = STAGES * STAGE;             // float [2][4][DV]: x and y partials
  static constexpr int KN = RED + 2 * 4 * DV * 4;        // float [DK] k of the new token (normalised)
  static constexpr int QN = KN + DK * 4;                 // float [DK] q of the new token
  static constexpr int GN = QN + DK * 4;                 // float [DK] G_n
  static constexpr int EN = GN + DK * 4;                 // float [DK] exp(G_n)
  static constexpr int EF = EN + DK * 4;                 // float [DK] exp(G_{L-1}) for a fold
  static constexpr int AB = EF + DK * 4;                 // float [2][REPLAY_MAX_TOKENS + 1]: a_j, b_j
  static constexpr int NINV = AB + (2 * (REPLAY_MAX_TOKENS + 1) * 4 + 15) / 16 * 16;
  static constexpr int BAR = NINV + 16;                  // full, sfree, computed [STAGES] each
  static constexpr int BYTES = BAR + 8 * 3 * STAGES;
  static constexpr int COMPUTE = DV / 4 * 16;
  static constexpr int THREADS = COMPUTE + 32;
};

__device__ __forceinline__ void rep_sync(int n) { asm volatile("bar.sync 1, %0;\n" ::"r"(n) : "memory"); }

// Slots of the head's buffer in use at the start of the step: fill clamped to [0, L].
__device__ __forceinline__ int read_fill(const int* fill, int j, int L, unsigned* err, bool report) {
  int n = fill[j];
  if (n < 0 || n > L) {
    if (report && err) atomicOr(err, ERR_REPLAY_FILL);
    n = n < 0 ? 0 : L;
  }
  return n;
}

// Fold coefficients of n filled slots, in place: k_j <- k_j * exp(G_{n-1} - G_j), and
// ef = exp(G_{n-1}). replay_state_kernel and a full step of replay_decode_kernel use
// this and fold_row4 below, so a materialised state equals the checkpoint that the
// next step writes, bitwise.
template <int DK, int SLOTF>
__device__ __forceinline__ void fold_coefficients(float* slots, float* ef, int n, int tid, int nthreads) {
  const float* Gl = slots + (n - 1) * SLOTF + DK;
  for (int idx = tid; idx < n * DK; idx += nthreads) {
    const int j = idx / DK, c = idx - j * DK;
    slots[j * SLOTF + c] *= expf(Gl[c] - slots[j * SLOTF + DK + c]);
  }
  for (int c = tid; c < DK; c += nthreads) ef[c] = expf(Gl[c]);
}

// s = ef[r] s + sum_j coef_j[r] d_j[4 cg .. 4 cg + 3], j ascending (fmaf chain).
template <int DK, int SLOTF>
__device__ __forceinline__ void fold_row4(float (&s)[4], int r, int cg, const float* slots, const float* ef, int n) {
  const float e = ef[r];
#pragma unroll
  for (int x = 0; x < 4; ++x) s[x] *= e;
  for (int j = 0; j < n; ++j) {
    const float c = slots[j * SLOTF + r];
    const float4 d = *reinterpret_cast<const float4*>(slots + j * SLOTF + 2 * DK + 4 * cg);
    s[0] = fmaf(c, d.x, s[0]);
    s[1] = fmaf(c, d.y, s[1]);
    s[2] = fmaf(c, d.z, s[2]);
    s[3] = fmaf(c, d.w, s[3]);
  }
}

template <class T, int DK, int DV, bool PC>
__global__ void __launch_bounds__(RepLayout<T, DK, DV>::THREADS, 1) replay_decode_kernel(ReplayArgs p) {
  typedef RepLayout<T, DK, DV> L;
  constexpr int RPT = DK / 16;
  constexpr int WPR = DV / 32;
  constexpr int NW = L::COMPUTE / 32;
  constexpr int SLOTF = L::SLOTF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* sfree = full + L::STAGES;
  uint64_t* computed = sfree + L::STAGES;
  float* red = reinterpret_cast<float*>(sm + L::RED);
  float* kn_s = reinterpret_cast<float*>(sm + L::KN);
  float* qn_s = reinterpret_cast<float*>(sm + L::QN);
  float* gn_s = reinterpret_cast<float*>(sm + L::GN);
  float* en_s = reinterpret_cast<float*>(sm + L::EN);
  float* ef_s = reinterpret_cast<float*>(sm + L::EF);
  float* a_s = reinterpret_cast<float*>(sm + L::AB);
  float* b_s = a_s + REPLAY_MAX_TOKENS + 1;
  float* ninv = reinterpret_cast<float*>(sm + L::NINV);
  const int nunits = (BH - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int Lc = p.L;

  if (tid == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfree[s], L::COMPUTE);
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
  float* buf = p.buffer;
  constexpr uint32_t SB = (uint32_t)(DK * DV * 4);

  if (warp == NW) {  // ---- producer
    if (lane == 0) {
      for (int m = 0; m < nunits; ++m) {
        const int s = m % L::STAGES, j = (int)blockIdx.x + m * (int)gridDim.x;
        const uint32_t par = (uint32_t)((m - L::STAGES) / L::STAGES) & 1u;
        uint8_t* st = sm + s * L::STAGE;
        const int n = read_fill(p.fill, j, Lc, p.err, false);
        const uint32_t tx = SB + (uint32_t)n * L::SLOTB + (uint32_t)((2 * DK + DV + (PC ? DK : 0)) * sizeof(T));
        if (m >= L::STAGES) mbar_wait(&sfree[s], par, p.err);
        mbar_arrive_expect_tx(&full[s], tx);
        bulk_g2s(st + L::STATE, p.ckpt + (size_t)j * DK * DV, SB, &full[s]);
        if (m >= L::STAGES) mbar_wait(&computed[s], par, p.err);
        if (n) bulk_g2s(st + L::SLOTS, buf + (size_t)j * Lc * SLOTF, (uint32_t)n * L::SLOTB, &full[s]);
        bulk_g2s(st + L::Q, q + (size_t)j * DK, DK * sizeof(T), &full[s]);
        bulk_g2s(st + L::K, k + (size_t)j * DK, DK * sizeof(T), &full[s]);
        bulk_g2s(st + L::V, v + (size_t)j * DV, DV * sizeof(T), &full[s]);
        if (PC) bulk_g2s(st + L::G, g + (size_t)j * DK, DK * sizeof(T), &full[s]);
      }
    }
    return;
  }

  // ---- compute warps
  const int cg = 8 * (warp % WPR) + (lane & 7);
  const int ph = warp / WPR, pl = lane >> 3;
  const int part = 4 * ph + pl;
#pragma unroll 1
  for (int m = 0; m < nunits; ++m) {
    const int s = m % L::STAGES, j = (int)blockIdx.x + m * (int)gridDim.x;  // j = b * H + h: the token row
    uint8_t* st = sm + s * L::STAGE;
    float* S_sm = reinterpret_cast<float*>(st + L::STATE);
    float* slots = reinterpret_cast<float*>(st + L::SLOTS);
    const T* qs = reinterpret_cast<const T*>(st + L::Q);
    const T* ks = reinterpret_cast<const T*>(st + L::K);
    const T* vs = reinterpret_cast<const T*>(st + L::V);
    const int n = read_fill(p.fill, j, Lc, p.err, tid == 0);
    const bool fold = n == Lc;
    const int nb = fold ? 0 : n;  // buffered tokens before this one, after an optional fold
    const float bt = to_f32(beta[j]);
    const float gsc = PC ? 0.f : to_f32(g[j]);
    float* slot_out = buf + ((size_t)j * Lc + nb) * SLOTF;
    mbar_wait(&full[s], (uint32_t)(m / L::STAGES) & 1u, p.err);

    // phase 0: fold coefficients, inverse norms
    if (fold) fold_coefficients<DK, SLOTF>(slots, ef_s, Lc, tid, L::COMPUTE);
    if (p.qk_norm && warp < 2) {
      const float inv = warp_row_inv_norm<DK>(warp ? ks : qs, lane);
      if (lane == 0) ninv[warp] = inv;
    }
    if (fold || p.qk_norm) rep_sync(L::COMPUTE);
    // phase 0b: the new token's per-channel rows; its k and G go to the buffer slot
    {
      const float nq = p.qk_norm ? ninv[0] : 1.f, nk = p.qk_norm ? ninv[1] : 1.f;
      for (int c = tid; c < DK; c += L::COMPUTE) {
        const float kc = to_f32(ks[c]) * nk, qc = to_f32(qs[c]) * nq;
        const float gp = nb > 0 ? slots[(nb - 1) * SLOTF + DK + c] : 0.f;
        const float gc = gp + (PC ? to_f32(reinterpret_cast<const T*>(st + L::G)[c]) : gsc);
        kn_s[c] = kc;
        qn_s[c] = qc;
        gn_s[c] = gc;
        en_s[c] = expf(gc);
        slot_out[c] = kc;
        slot_out[DK + c] = gc;
      }
    }
    rep_sync(L::COMPUTE);

    // phase 1: the checkpoint (folded if the buffer was full) and its two reads
    float S[RPT][4];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float4 x = *reinterpret_cast<const float4*>(S_sm + (part + 16 * i) * DV + 4 * cg);
      S[i][0] = x.x; S[i][1] = x.y; S[i][2] = x.z; S[i][3] = x.w;
    }
    mbar_arrive(&sfree[s]);
    if (fold) {
      float* ck = p.ckpt + (size_t)j * DK * DV;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int r = part + 16 * i;
        fold_row4<DK, SLOTF>(S[i], r, cg, slots, ef_s, Lc);
        *reinterpret_cast<float4*>(ck + r * DV + 4 * cg) = make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
      }
    }
    float xv[4] = {0.f, 0.f, 0.f, 0.f}, yv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = part + 16 * i;
      const float kh = en_s[r] * kn_s[r], qh = en_s[r] * qn_s[r];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xv[e] = fmaf(S[i][e], kh, xv[e]);
        yv[e] = fmaf(S[i][e], qh, yv[e]);
      }
    }
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xv[e] += __shfl_xor_sync(0xffffffffu, xv[e], off);
        yv[e] += __shfl_xor_sync(0xffffffffu, yv[e], off);
      }
    if (pl == 0) {
      *reinterpret_cast<float4*>(red + ph * DV + 4 * cg) = make_float4(xv[0], xv[1], xv[2], xv[3]);
      *reinterpret_cast<float4*>(red + (4 + ph) * DV + 4 * cg) = make_float4(yv[0], yv[1], yv[2], yv[3]);
    }
    // pairwise scores of the new token with the buffered ones (job nb: q_n . k_n)
    for (int jj = warp; jj <= nb; jj += NW) {
      float a = 0.f, b = 0.f;
      if (jj < nb) {
        const float* sl = slots + jj * SLOTF;
        for (int c = lane; c < DK; c += 32) {
          const float t = expf(gn_s[c] - sl[DK + c]) * sl[c];
          a = fmaf(kn_s[c], t, a);
          b = fmaf(qn_s[c], t, b);
        }
      } else {
        for (int c = lane; c < DK; c += 32) b = fmaf(qn_s[c], kn_s[c], b);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
      }
      if (lane == 0) {
        a_s[jj] = a;
        b_s[jj] = b;
      }
    }
    rep_sync(L::COMPUTE);

    // phase 2: delta and output per value column
    if (tid < DV) {
      const int c = tid;
      const float x = (red[0 * DV + c] + red[1 * DV + c]) + (red[2 * DV + c] + red[3 * DV + c]);
      const float y = (red[4 * DV + c] + red[5 * DV + c]) + (red[6 * DV + c] + red[7 * DV + c]);
      float acc = 0.f, acco = 0.f;
      for (int jj = 0; jj < nb; ++jj) {
        const float dj = slots[jj * SLOTF + 2 * DK + c];
        acc = fmaf(a_s[jj], dj, acc);
        acco = fmaf(b_s[jj], dj, acco);
      }
      const float dn = bt * ((to_f32(vs[c]) - x) - acc);
      const float o = p.scale * (y + fmaf(b_s[nb], dn, acco));
      static_cast<T*>(p.out)[(size_t)j * DV + c] = from_f32<T>(o);
      slot_out[2 * DK + c] = dn;
    }
    if (tid == 0) p.fill[j] = nb + 1;
    rep_sync(L::COMPUTE);  // slots and reduction buffers are reused by the next head
    if (tid == 0) mbar_arrive(&computed[s]);
  }
}

// The state a buffer stands for: h_out = the fold of fill slots into the checkpoint.
// One CTA per (batch, head); h_out may be the checkpoint itself (element-wise in place).
template <int DK, int DV>
__global__ void __launch_bounds__(256) replay_state_kernel(ReplayStateArgs p) {
  constexpr int SLOTF = 2 * DK + DV;
  __shared__ __align__(16) float slots[REPLAY_MAX_TOKENS * SLOTF];
  __shared__ float ef[DK];
  const int j = blockIdx.x, tid = threadIdx.x;
  const int n = read_fill(p.fill, j, p.L, p.err, tid == 0);
  const float* src = p.buffer + (size_t)j * p.L * SLOTF;
  for (int i = tid; i < n * SLOTF / 4; i += 256)
    reinterpret_cast<float4*>(slots)[i] = reinterpret_cast<const float4*>(src)[i];
  __syncthreads();
  if (n > 0) {
    fold_coefficients<DK, SLOTF>(slots, ef, n, tid, 256);
    __syncthreads();
  }
  const float* ck = p.ckpt + (size_t)j * DK * DV;
  float* h = p.h_out + (size_t)j * DK * DV;
  for (int idx = tid; idx < DK * DV / 4; idx += 256) {
    const int r = idx / (DV / 4), cg = idx - r * (DV / 4);
    const float4 x = *reinterpret_cast<const float4*>(ck + r * DV + 4 * cg);
    float s4[4] = {x.x, x.y, x.z, x.w};
    if (n > 0) fold_row4<DK, SLOTF>(s4, r, cg, slots, ef, n);
    *reinterpret_cast<float4*>(h + r * DV + 4 * cg) = make_float4(s4[0], s4[1], s4[2], s4[3]);
  }
}

template <class T, int DK, int DV>
cudaError_t launch_rep_t(const ReplayArgs& a, cudaStream_t s) {
  typedef RepLayout<T, DK, DV> L;
  const int bytes = L::BYTES + 1024;
  auto kern = a.per_channel ? replay_decode_kernel<T, DK, DV, true> : replay_decode_kernel<T, DK, DV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int BH = a.B * a.H;
  const int grid = nsm > 0 && BH > nsm ? nsm : BH;
  prof_mark(K_REPLAY, s, true);
  kern<<<grid, L::THREADS, bytes, s>>>(a);
  prof_mark(K_REPLAY, s, false);
  return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t launch_rep_state_t(const ReplayStateArgs& a, cudaStream_t s) {
  prof_mark(K_REPLAY_STATE, s, true);
  replay_state_kernel<DK, DV><<<a.B * a.H, 256, 0, s>>>(a);
  prof_mark(K_REPLAY_STATE, s, false);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_replay_decode(const ReplayArgs& a, cudaStream_t s) {
  if (a.bf16) {
    if (a.DK == 128) return a.DV == 128 ? launch_rep_t<bf16, 128, 128>(a, s) : launch_rep_t<bf16, 128, 64>(a, s);
    return a.DV == 128 ? launch_rep_t<bf16, 64, 128>(a, s) : launch_rep_t<bf16, 64, 64>(a, s);
  }
  if (a.DK == 128) return a.DV == 128 ? launch_rep_t<float, 128, 128>(a, s) : launch_rep_t<float, 128, 64>(a, s);
  return a.DV == 128 ? launch_rep_t<float, 64, 128>(a, s) : launch_rep_t<float, 64, 64>(a, s);
}

cudaError_t launch_replay_state(const ReplayStateArgs& a, cudaStream_t s) {
  if (a.DK == 128) return a.DV == 128 ? launch_rep_state_t<128, 128>(a, s) : launch_rep_state_t<128, 64>(a, s);
  return a.DV == 128 ? launch_rep_state_t<64, 128>(a, s) : launch_rep_state_t<64, 64>(a, s);
}

}  // namespace gdn
