// Float64 token-serial oracle for the gated delta rule.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path (the CUDA library and
// its Python binding) may load, link or call this file; only the test suite,
// the package smoke check and the benchmark's CPU-baseline leg use it.
//
// What it computes (per batch b and head h, independently):
//
//   S <- diag(exp(g_t)) S            per-key-channel decay (scalar g: one factor)
//   p  = S^T k_t                     what the state predicts for key k_t
//   d  = beta_t (v_t - p)            the delta, scaled by the write gate
//   S <- S + k_t d^T                 rank-one write
//   o_t = scale * S^T q_t            read with the query, after the write
//
// Sources: "gated-deltanet" kernel card (hf kernels hub), section Method: the
// per-token order decay -> read -> delta -> write -> read; marin.community
// note "factoring GDN-2 decay on TPU", section Background: one decay rate per
// channel, cumulative log-decay per channel. The output scale is the one the
// atomic-ops API passes as `scale` (d_head ** -0.5 in its quick start).
//
// The reverse pass below is derived by hand from the forward, one token at a
// time in reverse order, recomputing the states of each 64-token segment from
// a checkpoint taken at the segment start (memory stays O(T/64 * Dk * Dv)).
//
// Layouts (row-major, contiguous, float64):
//   q, k        [B, T, H, Dk]
//   v, out      [B, T, H, Dv]
//   g           [B, T, H, Dk] (g_per_channel = 1) or [B, T, H] (= 0)
//   beta        [B, T, H]
//   h0, h_final [B, H, Dk, Dv]   (h0 may be NULL: zero state)
//
// Every (b, h) pair is independent; pairs are spread over std::thread workers.

#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstring>
#include <thread>
#include <vector>

namespace {

struct Geometry {
  int B, T, H, Dk, Dv, g_per_channel;
  size_t qk_index(int b, int t, int h, int c) const {
    return (((size_t)b * T + t) * H + h) * Dk + c;
  }
  size_t v_index(int b, int t, int h, int c) const {
    return (((size_t)b * T + t) * H + h) * Dv + c;
  }
  size_t gate_index(int b, int t, int h) const { return ((size_t)b * T + t) * H + h; }
  size_t state_offset(int b, int h) const { return ((size_t)b * H + h) * Dk * Dv; }
  // log-decay of key channel c at token t
  double g_at(const double* g, int b, int t, int h, int c) const {
    return g_per_channel ? g[qk_index(b, t, h, c)] : g[gate_index(b, t, h)];
  }
};

template <class F>
void parallel_over_heads(int B, int H, int nthreads, F&& work) {
  const int pairs = B * H;
  if (nthreads <= 0) nthreads = (int)std::thread::hardware_concurrency();
  if (nthreads <= 0) nthreads = 1;
  if (nthreads > pairs) nthreads = pairs;
  std::atomic<int> next{0};
  auto worker = [&]() {
    for (;;) {
      int p = next.fetch_add(1);
      if (p >= pairs) break;
      work(p / H, p % H);
    }
  };
  if (nthreads <= 1) {
    worker();
    return;
  }
  std::vector<std::thread> pool;
  for (int i = 0; i < nthreads; ++i) pool.emplace_back(worker);
  for (auto& th : pool) th.join();
}

// One token of the forward recurrence on state S (Dk x Dv, row = key channel).
// Writes the output row into o (may be NULL) and the delta into d_out / p_out
// when those are given (the reverse pass needs them).
void forward_token(const Geometry& G, double* S, const double* q, const double* k,
                   const double* v, const double* g, const double* beta, double scale,
                   int b, int t, int h, double* o, double* p_out, double* d_out,
                   std::vector<double>& p) {
  const int Dk = G.Dk, Dv = G.Dv;
  // decay: S <- diag(exp(g_t)) S
  for (int c = 0; c < Dk; ++c) {
    const double a = std::exp(G.g_at(g, b, t, h, c));
    double* row = S + (size_t)c * Dv;
    for (int j = 0; j < Dv; ++j) row[j] *= a;
  }
  // read: p = S^T k
  for (int j = 0; j < Dv; ++j) p[j] = 0.0;
  for (int c = 0; c < Dk; ++c) {
    const double kc = k[G.qk_index(b, t, h, c)];
    const double* row = S + (size_t)c * Dv;
    for (int j = 0; j < Dv; ++j) p[j] += row[j] * kc;
  }
  // delta and rank-one write
  const double bt = beta[G.gate_index(b, t, h)];
  for (int j = 0; j < Dv; ++j) {
    const double dj = bt * (v[G.v_index(b, t, h, j)] - p[j]);
    if (p_out) p_out[j] = p[j];
    if (d_out) d_out[j] = dj;
    p[j] = dj;  // p now holds d
  }
  for (int c = 0; c < Dk; ++c) {
    const double kc = k[G.qk_index(b, t, h, c)];
    double* row = S + (size_t)c * Dv;
    for (int j = 0; j < Dv; ++j) row[j] += kc * p[j];
  }
  // read after the write: o = scale * S^T q
  if (o) {
    for (int j = 0; j < Dv; ++j) o[j] = 0.0;
    for (int c = 0; c < Dk; ++c) {
      const double qc = q[G.qk_index(b, t, h, c)];
      const double* row = S + (size_t)c * Dv;
      for (int j = 0; j < Dv; ++j) o[j] += row[j] * qc;
    }
    for (int j = 0; j < Dv; ++j) o[j] *= scale;
  }
}

bool valid_geometry(int B, int T, int H, int Dk, int Dv) {
  return B >= 0 && T >= 0 && H >= 0 && Dk > 0 && Dv > 0;
}

}  // namespace

extern "C" {

// Forward. Returns 0 on success, 1 on invalid geometry or a NULL required pointer.
int oracle_fwd(int B, int T, int H, int Dk, int Dv, int g_per_channel, const double* q,
               const double* k, const double* v, const double* g, const double* beta,
               const double* h0, double scale, double* out, double* h_final, int nthreads) {
  if (!valid_geometry(B, T, H, Dk, Dv)) return 1;
  if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return 1;
  if (!h_final) return 1;
  const Geometry G{B, T, H, Dk, Dv, g_per_channel};
  parallel_over_heads(B, H, nthreads, [&](int b, int h) {
    std::vector<double> S((size_t)Dk * Dv, 0.0), p(Dv), o(Dv);
    if (h0) std::memcpy(S.data(), h0 + G.state_offset(b, h), sizeof(double) * Dk * Dv);
    for (int t = 0; t < T; ++t) {
      forward_token(G, S.data(), q, k, v, g, beta, scale, b, t, h, o.data(), nullptr, nullptr, p);
      for (int j = 0; j < Dv; ++j) out[G.v_index(b, t, h, j)] = o[j];
    }
    std::memcpy(h_final + G.state_offset(b, h), S.data(), sizeof(double) * Dk * Dv);
  });
  return 0;
}

// Reverse pass. dout and dh_final are the upstream gradients of out and h_final
// (dh_final may be NULL: zero). Writes dq, dk, dv, dg (same shape as g), dbeta
// and dh0 (may be NULL). h0 may be NULL (zero state).
int oracle_bwd(int B, int T, int H, int Dk, int Dv, int g_per_channel, const double* q,
               const double* k, const double* v, const double* g, const double* beta,
               const double* h0, double scale, const double* dout, const double* dh_final,
               double* dq, double* dk, double* dv, double* dg, double* dbeta, double* dh0,
               int nthreads) {
  if (!valid_geometry(B, T, H, Dk, Dv)) return 1;
  if (T > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg || !dbeta))
    return 1;
  const Geometry G{B, T, H, Dk, Dv, g_per_channel};
  const int SEG = 64;  // checkpoint spacing in tokens
  parallel_over_heads(B, H, nthreads, [&](int b, int h) {
    const size_t SZ = (size_t)Dk * Dv;
    const int nseg = (T + SEG - 1) / SEG;
    // checkpoints: the state entering each segment
    std::vector<double> ckpt((size_t)nseg * SZ), S(SZ, 0.0), p(Dv);
    if (h0) std::memcpy(S.data(), h0 + G.state_offset(b, h), sizeof(double) * SZ);
    for (int t = 0; t < T; ++t) {
      if (t % SEG == 0) std::memcpy(&ckpt[(size_t)(t / SEG) * SZ], S.data(), sizeof(double) * SZ);
      forward_token(G, S.data(), q, k, v, g, beta, scale, b, t, h, nullptr, nullptr, nullptr, p);
    }
    // per segment: states after each token, and the per-token p and d
    std::vector<double> seg_states((size_t)(SEG + 1) * SZ), seg_p((size_t)SEG * Dv),
        seg_d((size_t)SEG * Dv);
    std::vector<double> dS(SZ, 0.0), dd(Dv), dp(Dv);
    if (dh_final) std::memcpy(dS.data(), dh_final + G.state_offset(b, h), sizeof(double) * SZ);
    for (int s = nseg - 1; s >= 0; --s) {
      const int t0 = s * SEG, t1 = std::min(T, t0 + SEG);
      // recompute: seg_states[i] = state after token t0 + i - 1 (i = 0: entering state)
      std::memcpy(seg_states.data(), &ckpt[(size_t)s * SZ], sizeof(double) * SZ);
      for (int t = t0; t < t1; ++t) {
        const int i = t - t0;
        std::memcpy(&seg_states[(size_t)(i + 1) * SZ], &seg_states[(size_t)i * SZ],
                    sizeof(double) * SZ);
        forward_token(G, &seg_states[(size_t)(i + 1) * SZ], q, k, v, g, beta, scale, b, t, h,
                      nullptr, &seg_p[(size_t)i * Dv], &seg_d[(size_t)i * Dv], p);
      }
      for (int t = t1 - 1; t >= t0; --t) {
        const int i = t - t0;
        const double* S_prev = &seg_states[(size_t)i * SZ];    // S_{t-1}
        const double* S_t = &seg_states[(size_t)(i + 1) * SZ];  // S_t
        const double* pt = &seg_p[(size_t)i * Dv];
        const double* d_t = &seg_d[(size_t)i * Dv];
        const double bt = beta[G.gate_index(b, t, h)];
        // o_t = scale S_t^T q_t
        for (int c = 0; c < Dk; ++c) {
          const double qc = q[G.qk_index(b, t, h, c)];
          double* row = &dS[(size_t)c * Dv];
          const double* srow = S_t + (size_t)c * Dv;
          double acc = 0.0;
          for (int j = 0; j < Dv; ++j) {
            const double doj = dout[G.v_index(b, t, h, j)];
            row[j] += scale * qc * doj;
            acc += srow[j] * doj;
          }
          dq[G.qk_index(b, t, h, c)] = scale * acc;
        }
        // S_t = S' + k d^T
        for (int j = 0; j < Dv; ++j) dd[j] = 0.0;
        for (int c = 0; c < Dk; ++c) {
          const double kc = k[G.qk_index(b, t, h, c)];
          const double* row = &dS[(size_t)c * Dv];
          double acc = 0.0;
          for (int j = 0; j < Dv; ++j) {
            dd[j] += row[j] * kc;
            acc += row[j] * d_t[j];
          }
          dk[G.qk_index(b, t, h, c)] = acc;
        }
        // d = beta (v - p)
        double dbeta_t = 0.0;
        for (int j = 0; j < Dv; ++j) {
          dbeta_t += dd[j] * (v[G.v_index(b, t, h, j)] - pt[j]);
          dv[G.v_index(b, t, h, j)] = bt * dd[j];
          dp[j] = -bt * dd[j];
        }
        dbeta[G.gate_index(b, t, h)] = dbeta_t;
        // p = S'^T k with S' = diag(a) S_{t-1};  dS' = dS + k dp^T
        double dg_scalar = 0.0;
        for (int c = 0; c < Dk; ++c) {
          const double a = std::exp(G.g_at(g, b, t, h, c));
          const double kc = k[G.qk_index(b, t, h, c)];
          const double* prow = S_prev + (size_t)c * Dv;
          double* row = &dS[(size_t)c * Dv];
          double acc_k = 0.0, acc_g = 0.0;
          for (int j = 0; j < Dv; ++j) {
            const double sp = a * prow[j];
            acc_k += sp * dp[j];
            const double dsp = row[j] + kc * dp[j];
            acc_g += dsp * sp;
            row[j] = a * dsp;  // becomes dS_{t-1}
          }
          dk[G.qk_index(b, t, h, c)] += acc_k;
          if (g_per_channel)
            dg[G.qk_index(b, t, h, c)] = acc_g;
          else
            dg_scalar += acc_g;
        }
        if (!g_per_channel) dg[G.gate_index(b, t, h)] = dg_scalar;
      }
    }
    if (dh0) std::memcpy(dh0 + G.state_offset(b, h), dS.data(), sizeof(double) * SZ);
  });
  return 0;
}

}  // extern "C"
