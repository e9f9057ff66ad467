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
// GB300 layout: persistent CTAs like decode_kernel. One producer thread feeds two rings:
// the checkpoints (two stages of Dk*Dv*4 bytes, one cp.async.bulk each, released as
// soon as the state warps hold the state in registers) and the per-head data (four
// stages: a header with the fill count and gates, the filled slots, the token row,
// released when the head is done, so that a head's slots arrive and its prep work is
// done while the heads before it are computed). Four prep warps compute the next head's channel
// values and pairwise scores while the state warps compute the current head's reads of
// the checkpoint. State thread (w, l) holds the state elements of value columns
// 4 cg .. 4 cg + 3 and key rows part + 16 i, as in decode_kernel.
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
  static constexpr int SB = DK * DV * 4;                 // one fp32 checkpoint
  static constexpr int SSTAGES = 2;                      // checkpoint ring
  // the per-head ring: header, buffer slots, token rows
  static constexpr int A_SLOTS = 0;                      // [REPLAY_MAX_TOKENS][SLOTF]
  static constexpr int A_Q = A_SLOTS + REPLAY_MAX_TOKENS * SLOTB;
  static constexpr int A_K = A_Q + DK * ES;
  static constexpr int A_V = A_K + DK * ES;
  static constexpr int A_G = A_V + DV * ES;
  static constexpr int A_HDR = A_G + DK * ES;            // int fill, float beta, float g (scalar decay)
  static constexpr int ASTAGE = A_HDR + 16;
  static constexpr int ASTAGES = 4;
  static constexpr int AUX = SSTAGES * SB;
  static constexpr int RED = AUX + ASTAGES * ASTAGE;     // float [2][4][DV]: x and y partials
  // per-head values the prep warps hand to the state warps, two buffers (head parity)
  static constexpr int P_KQ = 0;                         // float2 [DK]: exp(G_n) k_n, exp(G_n) q_n
  static constexpr int P_AB = P_KQ + DK * 8;             // float [2][REPLAY_MAX_TOKENS + 1]: a_j, b_j
  static constexpr int P_NINV = P_AB + (2 * (REPLAY_MAX_TOKENS + 1) * 4 + 15) / 16 * 16;  // float [2]
  static constexpr int PBUF = P_NINV + 16;
  static constexpr int PREPB = RED + 2 * 4 * DV * 4;
  // full_s, sfree [2]; full_a, afree [4]; prepdone, prepfree [2]
  static constexpr int BAR = PREPB + 2 * PBUF;
  static constexpr int BYTES = BAR + 8 * (2 * SSTAGES + 2 * ASTAGES + 4);
  static constexpr int COMPUTE = DV / 4 * 16;            // state warps
  static constexpr int PREP = 128;                       // prep warps
  static constexpr int THREADS = COMPUTE + PREP + 32;    // + the producer warp
  static_assert(BYTES <= 232448, "replay stages exceed the 227 KiB of shared memory per block");
  static_assert(ASTAGE % 16 == 0 && PBUF % 16 == 0, "bulk copy destinations must be 16-byte aligned");
};

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void rep_sync(int n) { asm volatile("bar.sync 1, %0;\n" ::"r"(n) : "memory"); }
__device__ __forceinline__ void prep_sync(int n) { asm volatile("bar.sync 2, %0;\n" ::"r"(n) : "memory"); }

// Slots of the head's buffer in use at the start of the step: fill clamped to [0, L].
__device__ __forceinline__ int read_fill(const int* fill, int j, int L, unsigned* err, bool report) {
  int n = fill[j];
  if (n < 0 || n > L) {
    if (report && err) atomicOr(err, ERR_REPLAY_FILL);
    n = n < 0 ? 0 : L;
  }
  return n;
}

// Fold coefficients of n filled slots, in place: k_j <- k_j * exp(G_{n-1} - G_j).
// replay_state_kernel and a full step of replay_decode_kernel use this and the row
// folds below, so a materialised state equals the checkpoint that the next step
// writes, bitwise.
template <int DK, int SLOTF>
__device__ __forceinline__ void fold_coefficients(float* slots, int n, int tid, int nthreads) {
  const float* Gl = slots + (n - 1) * SLOTF + DK;
  for (int idx = tid; idx < n * DK; idx += nthreads) {
    const int j = idx / DK, c = idx - j * DK;
    slots[j * SLOTF + c] *= expf(Gl[c] - slots[j * SLOTF + DK + c]);
  }
}

// s = exp(G_{n-1}[r]) s + sum_j coef_j[r] d_j[4 cg .. 4 cg + 3], j ascending (fmaf chain).
template <int DK, int SLOTF>
__device__ __forceinline__ void fold_row4(float (&s)[4], int r, int cg, const float* slots, int n) {
  const float e = expf(slots[(n - 1) * SLOTF + DK + r]);
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

// The fold of n slots into the thread's state rows part + 16 i (columns 4 cg ..):
// per element the same operations as fold_row4 (scale by exp(G_{n-1}), then an fmaf
// chain over ascending j), with the delta row loaded once per j for all rows.
template <int DK, int SLOTF, int RPT>
__device__ __forceinline__ void fold_rows(float (&S)[RPT][4], int part, int cg, const float* slots, int n) {
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const float e = expf(slots[(n - 1) * SLOTF + DK + part + 16 * i]);
#pragma unroll
    for (int x = 0; x < 4; ++x) S[i][x] *= e;
  }
  for (int j = 0; j < n; ++j) {
    const float4 d = *reinterpret_cast<const float4*>(slots + j * SLOTF + 2 * DK + 4 * cg);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float c = slots[j * SLOTF + part + 16 * i];
      S[i][0] = fmaf(c, d.x, S[i][0]);
      S[i][1] = fmaf(c, d.y, S[i][1]);
      S[i][2] = fmaf(c, d.z, S[i][2]);
      S[i][3] = fmaf(c, d.w, S[i][3]);
    }
  }
}

template <class T, int DK, int DV, bool PC>
__global__ void __launch_bounds__(RepLayout<T, DK, DV>::THREADS, 1) replay_decode_kernel(ReplayArgs p) {
  typedef RepLayout<T, DK, DV> L;
  constexpr int RPT = DK / 16;
  constexpr int WPR = DV / 32;
  constexpr int NSW = L::COMPUTE / 32;  // state warps
  constexpr int NPW = L::PREP / 32;     // prep warps
  constexpr int SLOTF = L::SLOTF;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;  // 16-byte alignment is all the bulk copies need
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  uint64_t* full_s = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* sfree = full_s + L::SSTAGES;
  uint64_t* full_a = sfree + L::SSTAGES;
  uint64_t* afree = full_a + L::ASTAGES;
  uint64_t* prepdone = afree + L::ASTAGES;
  uint64_t* prepfree = prepdone + 2;
  float* red = reinterpret_cast<float*>(sm + L::RED);
  const int nunits = (BH - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int Lc = p.L;

  if (tid == 0) {
    for (int i = 0; i < L::SSTAGES; ++i) {
      mbar_init(&full_s[i], 1);
      mbar_init(&sfree[i], L::COMPUTE);
    }
    for (int i = 0; i < L::ASTAGES; ++i) {
      mbar_init(&full_a[i], 1);
      mbar_init(&afree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&prepdone[i], L::PREP);
      mbar_init(&prepfree[i], L::COMPUTE);
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

  if (warp == NSW + NPW) {  // ---- producer
    if (lane == 0) {
      // One thread feeds both rings, each as far ahead as its free stages allow: it polls
      // (never blocks on) the two release barriers and issues whichever load is ready.
      // The head's fill count and gates travel in the per-head ring's header, so the
      // other warps start a head without a global load; they are read one head ahead.
      int ms = 0, ma = 0;  // next head to load into the checkpoint ring / per-head ring
      int n_next = nunits > 0 ? p.fill[blockIdx.x] : 0;
      T b_next = nunits > 0 ? beta[blockIdx.x] : T(0.f), g_next = (!PC && nunits > 0) ? g[blockIdx.x] : T(0.f);
      uint32_t idle = 0;
      while (ms < nunits || ma < nunits) {
        bool moved = false;
        if (ms < nunits) {
          const int ss = ms % L::SSTAGES;
          if (ms < L::SSTAGES || mbar_test(&sfree[ss], (uint32_t)((ms - L::SSTAGES) / L::SSTAGES) & 1u)) {
            const int j = (int)blockIdx.x + ms * (int)gridDim.x;
            mbar_arrive_expect_tx(&full_s[ss], (uint32_t)L::SB);
            bulk_g2s(sm + ss * L::SB, p.ckpt + (size_t)j * DK * DV, (uint32_t)L::SB, &full_s[ss]);
            ++ms;
            moved = true;
          }
        }
        if (ma < nunits) {
          const int sa = ma % L::ASTAGES;
          if (ma < L::ASTAGES || mbar_test(&afree[sa], (uint32_t)((ma - L::ASTAGES) / L::ASTAGES) & 1u)) {
            const int j = (int)blockIdx.x + ma * (int)gridDim.x;
            uint8_t* ax = sm + L::AUX + sa * L::ASTAGE;
            int n = n_next;
            const float bt = to_f32(b_next);
            const float gsc = PC ? 0.f : to_f32(g_next);
            if (ma + 1 < nunits) {
              const int jn = j + (int)gridDim.x;
              n_next = p.fill[jn];
              b_next = beta[jn];
              if (!PC) g_next = g[jn];
            }
            if (n < 0 || n > Lc) {  // clamped; reported in the error word
              if (p.err) atomicOr(p.err, ERR_REPLAY_FILL);
              n = n < 0 ? 0 : Lc;
            }
            int* hdr = reinterpret_cast<int*>(ax + L::A_HDR);
            hdr[0] = n;
            reinterpret_cast<float*>(hdr)[1] = bt;
            reinterpret_cast<float*>(hdr)[2] = gsc;
            mbar_arrive_expect_tx(&full_a[sa], (uint32_t)n * L::SLOTB +
                                                   (uint32_t)((2 * DK + DV + (PC ? DK : 0)) * sizeof(T)));
            if (n) bulk_g2s(ax + L::A_SLOTS, buf + (size_t)j * Lc * SLOTF, (uint32_t)n * L::SLOTB, &full_a[sa]);
            bulk_g2s(ax + L::A_Q, q + (size_t)j * DK, DK * sizeof(T), &full_a[sa]);
            bulk_g2s(ax + L::A_K, k + (size_t)j * DK, DK * sizeof(T), &full_a[sa]);
            bulk_g2s(ax + L::A_V, v + (size_t)j * DV, DV * sizeof(T), &full_a[sa]);
            if (PC) bulk_g2s(ax + L::A_G, g + (size_t)j * DK, DK * sizeof(T), &full_a[sa]);
            ++ma;
            moved = true;
          }
        }
        if (moved) {
          idle = 0;
        } else if (++idle == (1u << 24)) {  // the consumers stopped releasing stages
          if (p.err) atomicOr(p.err, ERR_WAIT_TIMEOUT);
          break;
        }
      }
      drain_ring(full_s, L::SSTAGES, ms);
      drain_ring(full_a, L::ASTAGES, ma);
    }
    return;
  }

  if (warp >= NSW) {  // ---- prep warps: per-channel values, pairwise scores, fold coefficients
    const int pt = tid - L::COMPUTE, pw = warp - NSW;
#pragma unroll 1
    for (int m = 0; m < nunits; ++m) {
      const int sa = m % L::ASTAGES, P = m & 1, j = (int)blockIdx.x + m * (int)gridDim.x;
      uint8_t* ax = sm + L::AUX + sa * L::ASTAGE;
      float* slots = reinterpret_cast<float*>(ax + L::A_SLOTS);
      const T* qs = reinterpret_cast<const T*>(ax + L::A_Q);
      const T* ks = reinterpret_cast<const T*>(ax + L::A_K);
      const T* gs = reinterpret_cast<const T*>(ax + L::A_G);
      uint8_t* pb = sm + L::PREPB + P * L::PBUF;
      float2* kq = reinterpret_cast<float2*>(pb + L::P_KQ);
      float* a_s = reinterpret_cast<float*>(pb + L::P_AB);
      float* b_s = a_s + REPLAY_MAX_TOKENS + 1;
      float* ninv = reinterpret_cast<float*>(pb + L::P_NINV);
      mbar_wait(&full_a[sa], (uint32_t)(m / L::ASTAGES) & 1u, p.err);
      if (m >= 2) mbar_wait(&prepfree[P], (uint32_t)((m - 2) / 2) & 1u, p.err);
      const int* hdr = reinterpret_cast<const int*>(ax + L::A_HDR);
      const int n = hdr[0];
      const float gsc = reinterpret_cast<const float*>(hdr)[2];
      const bool fold = n == Lc;
      const int nb = fold ? 0 : n;
      if (fold) fold_coefficients<DK, SLOTF>(slots, Lc, pt, L::PREP);
      if (p.qk_norm && pw < 2) {
        const float inv = warp_row_inv_norm<DK>(pw ? ks : qs, lane);
        if (lane == 0) ninv[pw] = inv;
      }
      if (fold || p.qk_norm) prep_sync(L::PREP);
      const float nq = p.qk_norm ? ninv[0] : 1.f, nk = p.qk_norm ? ninv[1] : 1.f;
      // the new token's channel values: k, q (normalised), G_n = G_{n-1} + g_n
      auto chan = [&](int c, float& kc, float& qc, float& gc) {
        kc = to_f32(ks[c]) * nk;
        qc = to_f32(qs[c]) * nq;
        gc = (nb > 0 ? slots[(nb - 1) * SLOTF + DK + c] : 0.f) + (PC ? to_f32(gs[c]) : gsc);
      };
      float* slot_out = buf + ((size_t)j * Lc + nb) * SLOTF;
      for (int c = pt; c < DK; c += L::PREP) {
        float kc, qc, gc;
        chan(c, kc, qc, gc);
        const float e = expf(gc);
        kq[c] = make_float2(e * kc, e * qc);
        slot_out[c] = kc;
        slot_out[DK + c] = gc;
      }
      // pairwise scores of the new token with the buffered ones; job nb is q_n . k_n.
      // Lane l holds channels l, l + 32, ...
      constexpr int CPL = DK / 32;
      float kl[CPL], ql[CPL], gl[CPL];
#pragma unroll
      for (int i = 0; i < CPL; ++i) chan(lane + 32 * i, kl[i], ql[i], gl[i]);
      for (int jj = pw; jj <= nb; jj += NPW) {
        float a = 0.f, b = 0.f;
        const float* sl = slots + jj * SLOTF;
        if (jj < nb) {
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            const float t = expf(gl[i] - sl[DK + c]) * sl[c];
            a = fmaf(kl[i], t, a);
            b = fmaf(ql[i], t, b);
          }
        } else {
#pragma unroll
          for (int i = 0; i < CPL; ++i) b = fmaf(ql[i], kl[i], b);
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
      mbar_arrive(&prepdone[P]);
    }
    return;
  }

  // ---- state warps
  const int cg = 8 * (warp % WPR) + (lane & 7);
  const int ph = warp / WPR, pl = lane >> 3;
  const int part = 4 * ph + pl;
#pragma unroll 1
  for (int m = 0; m < nunits; ++m) {
    const int ss = m % L::SSTAGES, sa = m % L::ASTAGES, P = m & 1, j = (int)blockIdx.x + m * (int)gridDim.x;
    const float* S_sm = reinterpret_cast<const float*>(sm + ss * L::SB);
    const uint8_t* ax = sm + L::AUX + sa * L::ASTAGE;
    const float* slots = reinterpret_cast<const float*>(ax + L::A_SLOTS);
    const T* vs = reinterpret_cast<const T*>(ax + L::A_V);
    const uint8_t* pb = sm + L::PREPB + P * L::PBUF;
    const float2* kq = reinterpret_cast<const float2*>(pb + L::P_KQ);
    const float* a_s = reinterpret_cast<const float*>(pb + L::P_AB);
    const float* b_s = a_s + REPLAY_MAX_TOKENS + 1;
    mbar_wait(&full_s[ss], (uint32_t)(m / L::SSTAGES) & 1u, p.err);
    float S[RPT][4];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float4 x = *reinterpret_cast<const float4*>(S_sm + (part + 16 * i) * DV + 4 * cg);
      S[i][0] = x.x; S[i][1] = x.y; S[i][2] = x.z; S[i][3] = x.w;
    }
    mbar_arrive(&sfree[ss]);
    mbar_wait(&full_a[sa], (uint32_t)(m / L::ASTAGES) & 1u, p.err);
    const int* hdr = reinterpret_cast<const int*>(ax + L::A_HDR);
    const int n = hdr[0];
    const float bt = reinterpret_cast<const float*>(hdr)[1];
    const bool fold = n == Lc;
    const int nb = fold ? 0 : n;  // buffered tokens before this one, after an optional fold
    mbar_wait(&prepdone[P], (uint32_t)(m / 2) & 1u, p.err);

    // the checkpoint (folded if the buffer was full), its two reads, and the buffered
    // deltas' terms: part p < nb adds a_p d_p and b_p d_p to its partial sums
    if (fold) {
      fold_rows<DK, SLOTF>(S, part, cg, slots, Lc);
      float* ck = p.ckpt + (size_t)j * DK * DV;
#pragma unroll
      for (int i = 0; i < RPT; ++i)
        *reinterpret_cast<float4*>(ck + (part + 16 * i) * DV + 4 * cg) = make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
    }
    float xv[4] = {0.f, 0.f, 0.f, 0.f}, yv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float2 h = kq[part + 16 * i];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xv[e] = fmaf(S[i][e], h.x, xv[e]);
        yv[e] = fmaf(S[i][e], h.y, yv[e]);
      }
    }
    if (part < nb) {
      const float4 d = *reinterpret_cast<const float4*>(slots + part * SLOTF + 2 * DK + 4 * cg);
      const float a = a_s[part], b = b_s[part];
      const float dd[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xv[e] = fmaf(a, dd[e], xv[e]);
        yv[e] = fmaf(b, dd[e], yv[e]);
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
    rep_sync(L::COMPUTE);

    // delta and output per value column
    if (tid < DV) {
      const int c = tid;
      const float x = (red[0 * DV + c] + red[1 * DV + c]) + (red[2 * DV + c] + red[3 * DV + c]);
      const float y = (red[4 * DV + c] + red[5 * DV + c]) + (red[6 * DV + c] + red[7 * DV + c]);
      const float dn = bt * (to_f32(vs[c]) - x);
      const float o = p.scale * fmaf(b_s[nb], dn, y);
      static_cast<T*>(p.out)[(size_t)j * DV + c] = from_f32<T>(o);
      buf[((size_t)j * Lc + nb) * SLOTF + 2 * DK + c] = dn;
    }
    if (tid == 0) p.fill[j] = nb + 1;
    mbar_arrive(&prepfree[P]);
    rep_sync(L::COMPUTE);  // slots, token rows and reduction buffers are free for the next head
    if (tid == 0) mbar_arrive(&afree[sa]);
  }
}

// The state a buffer stands for: h_out = the fold of fill slots into the checkpoint.
// One CTA per (batch, head); h_out may be the checkpoint itself (element-wise in place).
template <int DK, int DV>
__global__ void __launch_bounds__(256) replay_state_kernel(ReplayStateArgs p) {
  constexpr int SLOTF = 2 * DK + DV;
  __shared__ __align__(16) float slots[REPLAY_MAX_TOKENS * SLOTF];
  const int j = blockIdx.x, tid = threadIdx.x;
  const int n = read_fill(p.fill, j, p.L, p.err, tid == 0);
  const float* src = p.buffer + (size_t)j * p.L * SLOTF;
  for (int i = tid; i < n * SLOTF / 4; i += 256)
    reinterpret_cast<float4*>(slots)[i] = reinterpret_cast<const float4*>(src)[i];
  __syncthreads();
  if (n > 0) {
    fold_coefficients<DK, SLOTF>(slots, n, tid, 256);
    __syncthreads();
  }
  const float* ck = p.ckpt + (size_t)j * DK * DV;
  float* h = p.h_out + (size_t)j * DK * DV;
  for (int idx = tid; idx < DK * DV / 4; idx += 256) {
    const int r = idx / (DV / 4), cg = idx - r * (DV / 4);
    const float4 x = *reinterpret_cast<const float4*>(ck + r * DV + 4 * cg);
    float s4[4] = {x.x, x.y, x.z, x.w};
    if (n > 0) fold_row4<DK, SLOTF>(s4, r, cg, slots, n);
    *reinterpret_cast<float4*>(h + r * DV + 4 * cg) = make_float4(s4[0], s4[1], s4[2], s4[3]);
  }
}

template <class T, int DK, int DV>
cudaError_t launch_rep_t(const ReplayArgs& a, cudaStream_t s) {
  typedef RepLayout<T, DK, DV> L;
  const int bytes = L::BYTES;
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
