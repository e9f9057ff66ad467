// C ABI of the gated delta rule library: argument validation, buffer layouts and
// dispatch to the kernels. Declared in include/gdn.h.
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/gdn.h"
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

// Error word written by kernels that gave up on a bounded wait (bit values in common.cuh).
__device__ unsigned g_device_error;

constexpr int MAX_DEVICES = 64;
unsigned* g_err_ptr[MAX_DEVICES];
std::mutex g_err_mutex;

// Device address of the error word on the current device (resolved once per device,
// with that device current).
unsigned* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mutex);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_err_ptr[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// One thread first waits, with the kernels' own bounded cross-CTA counter wait
// (wait_counter, as the forward's output CTAs wait on the scan), for a counter that
// nothing raises, giving up after max_tries polls: the error word gets ERR_WAIT_TIMEOUT.
// Then it waits on an mbarrier that nothing ever arrives on, giving up after max_tries
// tries exactly as the kernels' own bounded waits do, and runs SELFTEST_LATER_WAITS of
// the kernels' own waits (mbar_wait) on the same barrier, which must give up soon after
// WAIT_BAIL_TRIES tries because the error word is set. The kernel returns normally. With
// `cycles` non-NULL it records the clock cycles of the first mbarrier wait, of the later
// ones together, and of the counter wait (0 had it succeeded).
constexpr int SELFTEST_LATER_WAITS = 4;
__device__ unsigned g_selftest_counter = 0;  // never raised
__global__ void wait_timeout_selftest_kernel(unsigned* err, unsigned max_tries, unsigned long long* cycles) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  const long long c0 = clock64();
  const bool counter_ok = wait_counter(&g_selftest_counter, 1u, err, max_tries);
  const long long c1 = clock64();
  const long long t0 = clock64();
  for (unsigned i = 0; i < max_tries; ++i)
    if (mbar_try_wait(&bar, 0u)) return;
  atomicOr(err, ERR_WAIT_TIMEOUT);
  __threadfence();
  const long long t1 = clock64();
  for (int w = 0; w < SELFTEST_LATER_WAITS; ++w) (void)mbar_wait(&bar, 0u, err);
  const long long t2 = clock64();
  if (cycles) {
    cycles[0] = (unsigned long long)(t1 - t0);
    cycles[1] = (unsigned long long)(t2 - t1);
    cycles[2] = counter_ok ? 0ull : (unsigned long long)(c1 - c0);
  }
}

// Common dims checks. Returns GDN_OK or the status to report.
int check_dims(const gdn_dims* d, bool chunked) {
  if (!d) return GDN_ERR_INVALID_ARG;
  if (d->B < 0 || d->T < 0 || d->H < 0) return GDN_ERR_INVALID_ARG;
  if (d->dtype != GDN_F32 && d->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if ((d->Dk != 64 && d->Dk != 128) || (d->Dv != 64 && d->Dv != 128)) return GDN_ERR_UNSUPPORTED;
  if ((long long)d->B * d->H > 65535) return GDN_ERR_UNSUPPORTED;  // grid y limit
  if (d->flags & ~(GDN_FLAG_PAIRWISE_WITHIN_BLOCK | GDN_FLAG_QK_L2NORM | GDN_FLAG_CHUNK128))
    return GDN_ERR_INVALID_ARG;
  if (chunked && d->T % ((d->flags & GDN_FLAG_CHUNK128) ? GDN_CHUNK128 : GDN_CHUNK) != 0) return GDN_ERR_SHAPE;
  return GDN_OK;
}

int esize(const gdn_dims* d) { return d->dtype == GDN_BF16 ? 2 : 4; }

// Required tensor: non-NULL and 16-byte aligned when the call has work.
bool tensor_ok(const void* p, bool has_work) { return !has_work || (p && aligned(p, 16)); }
bool optional_ok(const void* p) { return !p || aligned(p, 16); }
// [B,T,H] gates: element alignment only.
bool gate_ok(const void* p, bool has_work, int es) { return !has_work || (p && aligned(p, es)); }

bool qk_norm(const gdn_dims* d) { return (d->flags & GDN_FLAG_QK_L2NORM) != 0; }
bool chunk128(const gdn_dims* d) { return (d->flags & GDN_FLAG_CHUNK128) != 0; }

ResidualLayout residual_layout_of(const gdn_dims* d) {
  return residual_layout(d->B, d->T, d->H, d->Dk, d->Dv, esize(d), qk_norm(d), chunk128(d));
}

Residual128Ptrs residual128_ptrs(const gdn_dims* d, void* base) {
  const ResidualLayout L = residual_layout_of(d);
  char* b = static_cast<char*>(base);
  Residual128Ptrs r;
  r.aqk = b + L.aqk2;
  r.wneg = b + L.wneg2;
  r.up = b + L.up2;
  r.qh = b + L.qh2;
  r.kt = b + L.kt2;
  r.gam = reinterpret_cast<float*>(b + L.gam2);
  r.state = b + L.state2;
  r.u = b + L.u2;
  return r;
}

ResidualPtrs residual_ptrs(const gdn_dims* d, void* base) {
  const ResidualLayout L = residual_layout_of(d);
  char* b = static_cast<char*>(base);
  ResidualPtrs r;
  r.aqk = b + L.aqk;
  r.tmat = b + L.tmat;
  r.wneg = b + L.wneg;
  r.up = b + L.up;
  r.qh = b + L.qh;
  r.kt = b + L.kt;
  r.gam = reinterpret_cast<float*>(b + L.gam);
  r.state = b + L.state;
  r.u = b + L.u;
  r.progress = reinterpret_cast<unsigned*>(b + L.progress);
  if (qk_norm(d)) {
    r.qn = b + L.qn;
    r.kn = b + L.kn;
    r.qinv = reinterpret_cast<float*>(b + L.qinv);
    r.kinv = reinterpret_cast<float*>(b + L.kinv);
  }
  return r;
}

BwdWorkspacePtrs workspace_ptrs(const gdn_dims* d, void* base) {
  const BwdWorkspaceLayout L = bwd_workspace_layout(d->B, d->T, d->H, d->Dk, d->Dv, esize(d));
  char* b = static_cast<char*>(base);
  BwdWorkspacePtrs w;
  w.du = b + L.du;
  w.dstate = b + L.dstate;
  w.dqh = b + L.dqh;
  w.dbk = b + L.dbk;
  w.dkt = b + L.dkt;
  w.daqk = b + L.daqk;
  w.dakk = b + L.dakk;
  w.dgam = reinterpret_cast<float*>(b + L.dgam);
  w.dbv = reinterpret_cast<float*>(b + L.dbv);
  w.dbpart = reinterpret_cast<float*>(b + L.dbpart);
  w.dgpart = reinterpret_cast<float*>(b + L.dgpart);
  w.sync = reinterpret_cast<unsigned*>(b + L.sync);
  w.sync_bytes = L.sync_bytes;
  return w;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// Per-launch timing: a pool of event pairs, recorded around each kernel launch while on.
struct ProfRec {
  int id;
  cudaEvent_t a, b;
};
std::mutex g_prof_mutex;
std::vector<ProfRec> g_prof;
size_t g_prof_used = 0;
bool g_prof_on = false;
bool g_prof_failed = false;

const char* kKernelNames[K_COUNT] = {"chunk_prep_kernel",    "chunk_scan_fwd_kernel",
                                     "chunk_scan_bwd_kernel", "chunk_dstate_kernel",
                                     "chunk_grads_kernel",    "recurrent_kernel",
                                     "chunk_bwd_finalize_kernel", "chunk_out_kernel",
                                     "chunk_scan_fwd_tc_kernel", "chunk_scan_bwd_tc_kernel",
                                     "decode_kernel", "l2norm_rows_kernel", "l2norm_bwd_kernel",
                                     "replay_decode_kernel", "replay_state_kernel", "chunk_dqa_kernel",
                                     "chunk_bwd_tc_kernel", "chunk_prep_tc_kernel",
                                     "chunk_bwd_sync_zero_kernel", "chunk_merge128_kernel",
                                     "chunk_mid128_kernel"};

}  // namespace

void prof_mark(KernelId id, cudaStream_t s, bool begin) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  if (begin) {
    if (g_prof_used == g_prof.size()) {
      ProfRec r{};
      if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) {
        g_prof_failed = true;
        return;
      }
      g_prof.push_back(r);
    }
    g_prof[g_prof_used].id = (int)id;
    if (cudaEventRecord(g_prof[g_prof_used].a, s) != cudaSuccess) g_prof_failed = true;
  } else {
    if (g_prof_used >= g_prof.size()) return;
    if (cudaEventRecord(g_prof[g_prof_used].b, s) != cudaSuccess) g_prof_failed = true;
    ++g_prof_used;
  }
}

}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_chunk_residual_bytes(const gdn_dims* d) {
  if (check_dims(d, true) != GDN_OK) return 0;
  return residual_layout_of(d).total;
}

size_t gdn_chunk_bwd_workspace_bytes(const gdn_dims* d) {
  if (check_dims(d, true) != GDN_OK) return 0;
  if (chunk128(d) && d->dtype != GDN_BF16) return 0;  // 128-token backward: bf16 operands only
  return bwd_workspace_layout(d->B, d->T, d->H, d->Dk, d->Dv, esize(d)).total;
}

int gdn_chunk_fwd(const gdn_dims* d, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, const float* h0, float scale, void* out, float* h_final,
                  void* residuals, void* stream) {
  int st = check_dims(d, true);
  if (st != GDN_OK) return st;
  if (!std::isfinite(scale)) return GDN_ERR_INVALID_ARG;
  const bool work = (long long)d->B * d->H * d->T > 0;
  const int es = esize(d);
  if (!tensor_ok(q, work) || !tensor_ok(k, work) || !tensor_ok(v, work) || !tensor_ok(out, work))
    return GDN_ERR_INVALID_ARG;
  if (d->g_per_channel ? !tensor_ok(g, work) : !gate_ok(g, work, es)) return GDN_ERR_INVALID_ARG;
  if (!gate_ok(beta, work, es)) return GDN_ERR_INVALID_ARG;
  if (!optional_ok(h0) || !optional_ok(h_final)) return GDN_ERR_INVALID_ARG;
  if (work && (!residuals || !aligned(residuals, 256))) return GDN_ERR_INVALID_ARG;
  if ((long long)d->B * d->H == 0) return GDN_OK;
  ChunkFwdArgs a{};
  a.B = d->B; a.T = d->T; a.H = d->H; a.DK = d->Dk; a.DV = d->Dv;
  a.per_channel = d->g_per_channel ? 1 : 0;
  a.bf16 = d->dtype == GDN_BF16;
  a.flags = d->flags;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.scale = scale;
  a.out = out; a.h_final = h_final;
  if (residuals) {
    a.res = residual_ptrs(d, residuals);
    if (chunk128(d)) a.res2 = residual128_ptrs(d, residuals);
  }
  a.err = device_error_word();
  if (!a.err) return GDN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (qk_norm(d) && work) {  // every chunk kernel reads the normalised rows
    const cudaError_t e = launch_l2norm_rows(q, k, a.res.qn, a.res.kn, a.res.qinv, a.res.kinv,
                                             (size_t)d->B * d->T * d->H, d->Dk, a.bf16, s);
    if (e != cudaSuccess) return launch_status(e);
    a.q = a.res.qn;
    a.k = a.res.kn;
  }
  return launch_status(launch_chunk_fwd(a, s));
}

int gdn_chunk_bwd(const gdn_dims* d, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, const float* h0, float scale, const void* residuals,
                  const void* dout, const float* dh_final, void* dq, void* dk, void* dv, void* dg,
                  void* dbeta, float* dh0, void* workspace, void* stream) {
  int st = check_dims(d, true);
  if (st != GDN_OK) return st;
  // 128-token chunks: bf16 operands only (one stage of fp32 128-token records would not
  // fit the reverse scan's shared memory)
  if (chunk128(d) && d->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return GDN_ERR_INVALID_ARG;
  const bool work = (long long)d->B * d->H * d->T > 0;
  const int es = esize(d);
  (void)h0;  // the chunk-start states in the residuals already carry h0
  if (!tensor_ok(q, work) || !tensor_ok(k, work) || !tensor_ok(v, work) || !tensor_ok(dout, work) ||
      !tensor_ok(dq, work) || !tensor_ok(dk, work) || !tensor_ok(dv, work))
    return GDN_ERR_INVALID_ARG;
  if (d->g_per_channel ? (!tensor_ok(g, work) || !tensor_ok(dg, work))
                       : (!gate_ok(g, work, es) || !gate_ok(dg, work, es)))
    return GDN_ERR_INVALID_ARG;
  if (!gate_ok(beta, work, es) || !gate_ok(dbeta, work, es)) return GDN_ERR_INVALID_ARG;
  if (!optional_ok(dh_final) || !optional_ok(dh0)) return GDN_ERR_INVALID_ARG;
  if (work && (!residuals || !aligned(residuals, 256) || !workspace || !aligned(workspace, 256)))
    return GDN_ERR_INVALID_ARG;
  if ((long long)d->B * d->H == 0) return GDN_OK;
  ChunkBwdArgs a{};
  a.B = d->B; a.T = d->T; a.H = d->H; a.DK = d->Dk; a.DV = d->Dv;
  a.per_channel = d->g_per_channel ? 1 : 0;
  a.bf16 = d->dtype == GDN_BF16;
  a.flags = d->flags;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
  if (residuals) {
    a.res = residual_ptrs(d, const_cast<void*>(residuals));
    if (chunk128(d)) a.res2 = residual128_ptrs(d, const_cast<void*>(residuals));
  }
  a.dout = dout; a.dh_final = dh_final;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
  if (workspace) a.ws = workspace_ptrs(d, workspace);
  a.err = device_error_word();
  if (!a.err) return GDN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool norm = qk_norm(d) && work;
  if (norm) {  // the gradients come out with respect to the normalised rows first
    a.q = a.res.qn;
    a.k = a.res.kn;
  }
  cudaError_t e = launch_chunk_bwd(a, s);
  if (e == cudaSuccess && norm)
    e = launch_l2norm_bwd(dq, dk, a.res.qn, a.res.kn, a.res.qinv, a.res.kinv, (size_t)d->B * d->T * d->H, d->Dk,
                          a.bf16, s);
  return launch_status(e);
}

int gdn_recurrent(const gdn_dims* d, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, const float* h0, float scale, void* out, float* h_final,
                  void* stream) {
  int st = check_dims(d, false);
  if (st != GDN_OK) return st;
  if (!std::isfinite(scale)) return GDN_ERR_INVALID_ARG;
  const bool work = (long long)d->B * d->H * d->T > 0;
  const bool heads = (long long)d->B * d->H > 0;
  const int es = esize(d);
  if (!tensor_ok(q, work) || !tensor_ok(k, work) || !tensor_ok(v, work) || !tensor_ok(out, work))
    return GDN_ERR_INVALID_ARG;
  if (d->g_per_channel ? !tensor_ok(g, work) : !gate_ok(g, work, es)) return GDN_ERR_INVALID_ARG;
  if (!gate_ok(beta, work, es)) return GDN_ERR_INVALID_ARG;
  if (!optional_ok(h0) || !tensor_ok(h_final, heads)) return GDN_ERR_INVALID_ARG;
  if (!heads) return GDN_OK;
  RecurrentArgs a{};
  a.B = d->B; a.T = d->T; a.H = d->H; a.DK = d->Dk; a.DV = d->Dv;
  a.per_channel = d->g_per_channel ? 1 : 0;
  a.bf16 = d->dtype == GDN_BF16;
  a.qk_norm = qk_norm(d) ? 1 : 0;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.scale = scale;
  a.out = out; a.h_final = h_final;
  a.err = device_error_word();
  if (!a.err) return GDN_ERR_CUDA;
  return launch_status(launch_recurrent(a, static_cast<cudaStream_t>(stream)));
}

size_t gdn_replay_buffer_bytes(const gdn_dims* d, int L) {
  if (check_dims(d, false) != GDN_OK || L < 1 || L > GDN_REPLAY_MAX_TOKENS) return 0;
  return (size_t)d->B * d->H * L * (2 * d->Dk + d->Dv) * sizeof(float);
}

int gdn_replay_decode(const gdn_dims* d, int L, const void* q, const void* k, const void* v,
                      const void* g, const void* beta, float scale, float* ckpt, void* buffer,
                      int* fill, void* out, void* stream) {
  int st = check_dims(d, false);
  if (st != GDN_OK) return st;
  if (L < 1 || L > GDN_REPLAY_MAX_TOKENS || !std::isfinite(scale)) return GDN_ERR_INVALID_ARG;
  if (d->T != 1) return GDN_ERR_SHAPE;
  const bool work = (long long)d->B * d->H > 0;
  const int es = esize(d);
  if (!tensor_ok(q, work) || !tensor_ok(k, work) || !tensor_ok(v, work) || !tensor_ok(out, work))
    return GDN_ERR_INVALID_ARG;
  if (d->g_per_channel ? !tensor_ok(g, work) : !gate_ok(g, work, es)) return GDN_ERR_INVALID_ARG;
  if (!gate_ok(beta, work, es)) return GDN_ERR_INVALID_ARG;
  if (!tensor_ok(ckpt, work) || !tensor_ok(buffer, work) || !gate_ok(fill, work, 4)) return GDN_ERR_INVALID_ARG;
  if (!work) return GDN_OK;
  ReplayArgs a{};
  a.B = d->B; a.H = d->H; a.DK = d->Dk; a.DV = d->Dv; a.L = L;
  a.per_channel = d->g_per_channel ? 1 : 0;
  a.bf16 = d->dtype == GDN_BF16;
  a.qk_norm = qk_norm(d) ? 1 : 0;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
  a.ckpt = ckpt; a.buffer = static_cast<float*>(buffer); a.fill = fill; a.out = out;
  a.err = device_error_word();
  if (!a.err) return GDN_ERR_CUDA;
  return launch_status(launch_replay_decode(a, static_cast<cudaStream_t>(stream)));
}

int gdn_replay_state(const gdn_dims* d, int L, const float* ckpt, const void* buffer, const int* fill,
                     float* h_out, void* stream) {
  int st = check_dims(d, false);
  if (st != GDN_OK) return st;
  if (L < 1 || L > GDN_REPLAY_MAX_TOKENS) return GDN_ERR_INVALID_ARG;
  const bool work = (long long)d->B * d->H > 0;
  if (!tensor_ok(ckpt, work) || !tensor_ok(buffer, work) || !gate_ok(fill, work, 4) || !tensor_ok(h_out, work))
    return GDN_ERR_INVALID_ARG;
  if (!work) return GDN_OK;
  ReplayStateArgs a{};
  a.B = d->B; a.H = d->H; a.DK = d->Dk; a.DV = d->Dv; a.L = L;
  a.ckpt = ckpt; a.buffer = static_cast<const float*>(buffer); a.fill = fill; a.h_out = h_out;
  a.err = device_error_word();
  if (!a.err) return GDN_ERR_CUDA;
  return launch_status(launch_replay_state(a, static_cast<cudaStream_t>(stream)));
}

int gdn_selftest_wait_timeout(unsigned max_tries, unsigned long long* cycles, void* stream) {
  if (max_tries == 0 || max_tries > (1u << 16)) return GDN_ERR_INVALID_ARG;
  if (!optional_ok(cycles)) return GDN_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return GDN_ERR_CUDA;
  wait_timeout_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(err, max_tries, cycles);
  return launch_status(cudaGetLastError());
}

int gdn_check_device_error(void) {
  unsigned* p = device_error_word();
  if (!p) return GDN_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return GDN_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_ERR_INTERNAL;
  }
  return GDN_OK;
}

const char* gdn_status_string(int s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument (NULL or misaligned pointer, bad size or flag)";
    case GDN_ERR_UNSUPPORTED: return "unsupported configuration (Dk, Dv in {64, 128}; dtype bf16 or fp32)";
    case GDN_ERR_SHAPE: return "T must be a multiple of 64 on the chunked path";
    case GDN_ERR_CUDA: return "CUDA launch or runtime error";
    case GDN_ERR_INTERNAL: return "a kernel reported an error (a bounded wait timed out, or a replay fill count out of range)";
    case GDN_ERR_SCRATCH_LIMIT: return "problem needs more residual scratch than the static GDN_NOALLOC_SCRATCH_BYTES array";
    default: return "unknown status";
  }
}

int gdn_version(void) { return 100; }

int gdn_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  g_prof_on = on != 0;
  g_prof_used = 0;
  g_prof_failed = false;
  return GDN_OK;
}

int gdn_profile_read(double* ms, int* launches, int n) {
  if (!ms || !launches || n < 0) return GDN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  for (int i = 0; i < n; ++i) {
    ms[i] = 0.0;
    launches[i] = 0;
  }
  if (g_prof_failed) return GDN_ERR_CUDA;
  for (size_t i = 0; i < g_prof_used; ++i) {
    if (cudaEventSynchronize(g_prof[i].b) != cudaSuccess) return GDN_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, g_prof[i].a, g_prof[i].b) != cudaSuccess) return GDN_ERR_CUDA;
    const int id = g_prof[i].id;
    if (id < n) {
      ms[id] += t;
      launches[id] += 1;
    }
  }
  g_prof_used = 0;
  return GDN_OK;
}

const char* gdn_kernel_name(int id) { return (id >= 0 && id < K_COUNT) ? kKernelNames[id] : ""; }

}  // extern "C"
