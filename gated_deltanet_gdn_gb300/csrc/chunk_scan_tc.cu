// State scans on the 5th-generation tensor cores (tcgen05) for bf16 operands with
// Dk = Dv = 128: the forward recurrence over chunks and its reverse for the gradients.
//
// One CTA per (batch, head). The fp32 state lives in tensor memory in transposed form,
// S^T [Dv][Dk]: TMEM lane v holds value column v. Per chunk (C = 64 tokens):
//   forward   U^T  = U'^T + S^T (-W)^T                    (M = Dv, N = C,  K = C, Dk)
//             S^T <- S^T diag(gam) + U^T K-tilde           (M = Dv, N = Dk, K = C)
//   reverse   dU^T = dO^T (scale Aqk) + dS^T K-tilde^T     (M = Dv, N = C,  K = C, Dk)
//             dS^T <- dS^T diag(gam) + dO^T (scale Q-hat) + dU^T (-W)  (N = Dk, K = C)
// which are the transposes of U = U' - W S, S1 = diag(gam) S + K-tilde^T U and of
// dU = scale Aqk^T dO + K-tilde dS, dS0 = diag(gam) dS + scale Q-hat^T dO - W^T dU
// (the chunked WY form of the token recurrence; see chunk_fwd.cu and chunk_bwd.cu).
//
// Forward warp roles (576 threads): warps 0-15 move the state between TMEM and shared
// memory, four per TMEM lane quarter (thread (w, l) owns lane 32 (w % 4) + l and a quarter
// of the columns); warp 16 is the producer that streams each chunk's records into a ring
// of stages (cp.async.bulk) as soon as the tensor cores release a stage; warp 17
// publishes progress to the output CTAs beside the scan. Thread 0 issues every
// tcgen05.mma (bf16 x bf16 -> fp32 in TMEM) on 128-byte swizzled tiles: the records
// exactly as the preparation kernel stored them (K-major or MN-major operands, no
// transposition) and the bf16 copies of S^T / U^T the compute warps write from TMEM
// (double-buffered), which bulk copies also store as the chunk-start state and U records
// the later kernels read. The compute warps add U' to the forward's U^T. The reverse scan
// is the role rscan_role of chunk_scan_tc.cuh (eight compute warps, a producer warp),
// run here by a kernel of its own. Every wait is bounded and sets the device error word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "chunk_out.cuh"
#include "chunk_scan_tc.cuh"
#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

// the forward: 16 compute warps (four per TMEM lane quarter, each on a quarter of the
// state's columns), the producer warp and the publisher warp
constexpr int FWD_COMPUTE = 512;
constexpr int FWD_PRODUCER = FWD_COMPUTE / 32, FWD_PUBLISHER = FWD_PRODUCER + 1;
constexpr int FWD_THREADS = FWD_COMPUTE + 64;

__device__ __forceinline__ void fwd_sync() { asm volatile("bar.sync 1, 512;\n" ::: "memory"); }
__device__ __forceinline__ void out_sync() { asm volatile("bar.sync 2, 256;\n" ::: "memory"); }

// ------------------------------------------------------------------ forward
struct TcFwdLayout {
  static constexpr int W = 0;                    // -W      [C][Dk]  (K-major B of U^T)
  static constexpr int KT = W + C * TD * 2;      // K-tilde [C][Dk]  (MN-major B of S^T)
  static constexpr int UP = KT + C * TD * 2;     // U'^T    [Dv][C]  (added by the threads)
  static constexpr int GAM = UP + C * TD * 2;    // gam     [Dk] fp32
  static constexpr int STAGE = a1k(GAM + TD * 4);
  static constexpr int STAGES = 2;
  static constexpr int SA = STAGES * STAGE;        // S^T bf16 [Dv][Dk], two buffers
  static constexpr int UA = SA + 2 * TD * TD * 2;  // U^T bf16 [Dv][C], two buffers
  static constexpr int BAR = UA + 2 * TD * C * 2;  // full[STAGES], empty[STAGES], u, s, drain
  static constexpr int TSLOT = BAR + 8 * (2 * STAGES + 3);
  static constexpr int BYTES = TSLOT + 16;  // TMEM address, then the publication counter
  static constexpr uint32_t TX = (uint32_t)(3 * C * TD * 2 + TD * 4);
};

// with_out: the grid is cooperative and CTAs B*H.. are output CTAs. Each takes chunk-heads
// (n, bh) in chunk-major order; its warp 8 waits until the scan CTA of bh has published
// that its records of chunk n are stored (a.res.progress[bh] > n) and bulk-loads that
// chunk's four records into one of two stages, while warps 0-7 form the outputs of the
// chunk in the other (out_compute_store). The scan CTAs publish after the bulk copies of a
// chunk's state and U records have completed. Output CTAs only wait on scan CTAs, never
// the other way round.
__global__ void __launch_bounds__(FWD_THREADS, 1) chunk_scan_fwd_tc_kernel(ChunkFwdArgs a, int with_out) {
  pdl_wait();  // no early trigger: one wave for the whole scan, successors must not park beside it
  typedef TcFwdLayout L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int N = a.T / C;
  const int BH = a.B * a.H;
  if (bh >= BH) {  // ---- output CTA: warp 8 loads, warps 0-7 compute (two stages)
    typedef OutLayout<bf16, TD, TD> OL;
    constexpr int OSTAGE = a1k(OL::BYTES);
    uint64_t* ofull = reinterpret_cast<uint64_t*>(sm + 2 * OSTAGE);
    uint64_t* oempty = ofull + 2;
    const int units = N * BH, ncons = (int)gridDim.x - BH;
    const int first = bh - BH;
    const int count = first < units ? (units - first + ncons - 1) / ncons : 0;
    if (tid == 0) {
      for (int s2 = 0; s2 < 2; ++s2) {
        mbar_init(&ofull[s2], 1);
        mbar_init(&oempty[s2], 1);
      }
      fence_mbar_init();
    }
    __syncthreads();
    if (warp >= OUT_THREADS / 32 && warp != FWD_PRODUCER) return;  // warps 0-7 compute, one loads
    if (warp == FWD_PRODUCER) {
      if (lane == 0) {
        for (int k = 0; k < count; ++k) {
          const int u = first + k * ncons, n = u / BH, ob = u % BH, s2 = k & 1;
          if (k >= 2) mbar_wait(&oempty[s2], (uint32_t)((k - 2) >> 1) & 1u, a.err);
          wait_counter(a.res.progress + (size_t)ob * PROGRESS_STRIDE, (unsigned)(n + 1), a.err);
          fence_proxy_async_global();
          const size_t ch = (size_t)ob * N + n;
          uint8_t* st = sm + s2 * OSTAGE;
          mbar_arrive_expect_tx(&ofull[s2], (uint32_t)(2 * C * TD * 2 + C * C * 2 + TD * TD * 2));
          bulk_g2s(st + OL::QH, static_cast<const bf16*>(a.res.qh) + ch * (C * TD), C * TD * 2, &ofull[s2]);
          bulk_g2s(st + OL::AQ, static_cast<const bf16*>(a.res.aqk) + ch * (C * C), C * C * 2, &ofull[s2]);
          bulk_g2s(st + OL::S0, static_cast<const bf16*>(a.res.state) + ch * (TD * TD), TD * TD * 2, &ofull[s2]);
          bulk_g2s(st + OL::U, static_cast<const bf16*>(a.res.u) + ch * (C * TD), C * TD * 2, &ofull[s2]);
        }
        drain_ring(ofull, 2, count);
      }
      return;
    }
    for (int k = 0; k < count; ++k) {
      const int u = first + k * ncons, n = u / BH, ob = u % BH, s2 = k & 1;
      mbar_wait(&ofull[s2], (uint32_t)(k >> 1) & 1u, a.err);
      out_compute_store<bf16, TD, TD>(a, n, ob, sm + s2 * OSTAGE, tid, [] { out_sync(); });
      if (tid == 0) mbar_arrive(&oempty[s2]);
    }
    return;
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* empty = full + L::STAGES;
  uint64_t* bar_u = empty + L::STAGES;
  uint64_t* bar_s = bar_u + 1;
  uint64_t* bar_d = bar_s + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::TSLOT);
  bf16* const sa_buf = reinterpret_cast<bf16*>(sm + L::SA);
  bf16* const ua_buf = reinterpret_cast<bf16*>(sm + L::UA);

  if (tid == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(bar_u, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_d, 1);
    fence_mbar_init();
    *reinterpret_cast<unsigned*>(sm + L::TSLOT + 8) = 0u;  // chunks published
  }
  if (warp == 0) {
    tmem_alloc(tslot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;

  unsigned* pub_s = reinterpret_cast<unsigned*>(sm + L::TSLOT + 8);
  if (warp == FWD_PUBLISHER) {  // ---- publisher (output CTAs beside the scan)
    // Thread 0 sets pub_s to the number of chunks whose state and U records are stored
    // (after their bulk copies completed); this thread forwards the latest value to the
    // output CTAs with a GPU-scope release, which so stays off the chunk chain.
    if (lane == 0 && with_out) {
      unsigned last = 0;
      for (uint32_t i = 0; last < (unsigned)N && i < WAIT_MAX_TRIES; ++i) {
        const unsigned v = ld_acquire_cta(pub_s);
        if (v > last) {
          st_release_gpu(a.res.progress + (size_t)bh * PROGRESS_STRIDE, v);
          last = v;
        } else {
          // after a time-out anywhere the scan's waits give up early; so does this one
          if (i >= WAIT_BAIL_TRIES && (i & 255u) == 0 &&
              (*reinterpret_cast<volatile unsigned*>(a.err) & ERR_WAIT_TIMEOUT))
            break;
          __nanosleep(256);
        }
      }
      if (last < (unsigned)N) atomicOr(a.err, ERR_WAIT_TIMEOUT);
    }
    return;
  }
  if (warp == FWD_PRODUCER) {  // ---- producer
    if (lane == 0) {
      for (int n = 0; n < N; ++n) {
        const int s = n % L::STAGES, k = n / L::STAGES;
        if (k > 0) mbar_wait(&empty[s], (uint32_t)(k - 1) & 1u, a.err);
        uint8_t* st = sm + s * L::STAGE;
        const size_t ch = (size_t)bh * N + n;
        mbar_arrive_expect_tx(&full[s], L::TX);
        bulk_g2s(st + L::W, static_cast<const bf16*>(a.res.wneg) + ch * (C * TD), C * TD * 2, &full[s]);
        bulk_g2s(st + L::KT, static_cast<const bf16*>(a.res.kt) + ch * (C * TD), C * TD * 2, &full[s]);
        bulk_g2s(st + L::UP, static_cast<const bf16*>(a.res.up) + ch * (C * TD), C * TD * 2, &full[s]);
        bulk_g2s(st + L::GAM, a.res.gam + ch * TD, TD * 4, &full[s]);
      }
      drain_ring(full, L::STAGES, N);
    }
    return;
  }

  // ---- compute warps
  // thread: TMEM lane row (value column), state columns 32 qtr .. + 31, U^T tokens 16 qtr ..
  const int row = 32 * (warp & 3) + lane, qtr = warp >> 2;
  const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's lane quarter
  const size_t sb = (size_t)bh * TD * TD;
  {
    float x[32];
    for (int i = 0; i < 32; ++i) x[i] = a.h0 ? a.h0[sb + (size_t)(32 * qtr + i) * TD + row] : 0.f;
    tmem_st32(tl + 32 * qtr, x);
    tmem_wait_st();
  }
  constexpr uint32_t id_1 = umma_idesc_bf16(128, C, false, false);  // S^T (-W)^T
  constexpr uint32_t id_2 = umma_idesc_bf16(128, TD, false, true);  // U^T K-tilde
  bf16* state_rec = static_cast<bf16*>(a.res.state);
  bf16* u_rec = static_cast<bf16*>(a.res.u);
  uint32_t ph_u = 0, ph_s = 0;
#pragma unroll 1
  for (int n = 0; n < N; ++n) {
    const int s = n % L::STAGES;
    uint8_t* st = sm + s * L::STAGE;
    const size_t ch = (size_t)bh * N + n;
    Tile<bf16, TD, TD> Sa{sa_buf + (n & 1) * (TD * TD)};
    Tile<bf16, TD, C> Ua{ua_buf + (n & 1) * (TD * C)};
    if (n > 0) {  // the previous chunk's S^T update is done
      mbar_wait(bar_s, ph_s, a.err);
      ph_s ^= 1u;
      tc_fence_after();
    }
    mbar_wait(&full[s], (uint32_t)(n / L::STAGES) & 1u, a.err);
    // S^T -> bf16 operand (the chunk-start state record)
    float xs[32];
    tmem_ld32(tl + 32 * qtr, xs);
    store_row32(Sa, row, 32 * qtr, xs);
    fence_proxy_async();
    tc_fence_before();
    fwd_sync();
    if (tid == 0) {
      tc_fence_after();
      bulk_s2g(state_rec + ch * (TD * TD), Sa.p, TD * TD * 2);
      bulk_commit();
      const uint64_t dW = desc_k(st + L::W), dSa = desc_k(Sa.p);
#pragma unroll
      for (int ks = 0; ks < TD / 16; ++ks)
        umma_bf16(tm + 128, kstep_k(dSa, ks, PANEL_D), kstep_k(dW, ks, PANEL_C), id_1, ks > 0);
      umma_commit_to(bar_u);
      if (with_out && n > 0) {  // every bulk group but this chunk's state: chunks < n stored
        bulk_wait1();
        fence_proxy_async_global();
        st_release_cta(pub_s, (unsigned)n);
      }
    }
    // S^T <- S^T diag(gam) while the tensor cores form U^T (the S^T update comes after
    // the next barrier)
    {
      const float* gam = reinterpret_cast<const float*>(st + L::GAM) + 32 * qtr;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 g4 = *reinterpret_cast<const float4*>(gam + i);
        xs[i] *= g4.x;
        xs[i + 1] *= g4.y;
        xs[i + 2] *= g4.z;
        xs[i + 3] *= g4.w;
      }
      tmem_st32(tl + 32 * qtr, xs);
      tmem_wait_st();
    }
    mbar_wait(bar_u, ph_u, a.err);
    ph_u ^= 1u;
    tc_fence_after();
    {  // U^T row = U'^T row + (S^T (-W)^T) row -> bf16 operand (the U record)
      uint32_t r16[16];
      tmem_ld16_nowait(tl + 128 + 16 * qtr, r16);
      tmem_wait_ld();
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(r16[i]);
      const bf16* up = reinterpret_cast<const bf16*>(st + L::UP);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 u = *reinterpret_cast<const uint4*>(up + Sw<bf16, TD, C>::off(row, 16 * qtr + 8 * q));
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h2[e]);
          x[8 * q + 2 * e] += f.x;
          x[8 * q + 2 * e + 1] += f.y;
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint4 u;
        u.x = pack_bf16(x[8 * q + 0], x[8 * q + 1]);
        u.y = pack_bf16(x[8 * q + 2], x[8 * q + 3]);
        u.z = pack_bf16(x[8 * q + 4], x[8 * q + 5]);
        u.w = pack_bf16(x[8 * q + 6], x[8 * q + 7]);
        *reinterpret_cast<uint4*>(Ua.ptr(row, 16 * qtr + 8 * q)) = u;
      }
    }
    fence_proxy_async();
    tc_fence_before();
    // the record stores of the previous chunk have read the buffers the next chunk writes
    if (tid == 0) bulk_wait_read1();
    fwd_sync();
    if (tid == 0) {
      tc_fence_after();
      bulk_s2g(u_rec + ch * (C * TD), Ua.p, C * TD * 2);
      bulk_commit();
      const uint64_t dKt = desc_mn(st + L::KT, PANEL_C), dUa = desc_k(Ua.p);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) umma_bf16(tm, kstep_k(dUa, ks, PANEL_D), kstep_mn(dKt, ks), id_2, 1u);
      umma_commit_to(&empty[s]);
      umma_commit_to(bar_s);
    }
  }
  if (N > 0) {
    mbar_wait(bar_s, ph_s, a.err);
    tc_fence_after();
  }
  if (a.h_final) {
    float x[32];
    tmem_ld32(tl + 32 * qtr, x);
#pragma unroll
    for (int i = 0; i < 32; ++i) a.h_final[sb + (size_t)(32 * qtr + i) * TD + row] = x[i];
  }
  if (tid == 0) {  // record stores and every issued MMA complete before TMEM is freed
    bulk_wait0();
    if (with_out) {
      fence_proxy_async_global();
      st_release_cta(pub_s, (unsigned)N);
    }
    drain_mma(bar_d);
  }
  tc_fence_before();
  fwd_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, TMEM_COLS);
}

// ------------------------------------------------------------------ reverse
// One CTA per (batch, head): the reverse scan alone (rscan_role, chunk_scan_tc.cuh), used
// when the fused backward launch of chunk_bwd_tc.cu does not apply.
__global__ void __launch_bounds__(TC_THREADS, 1)
    chunk_scan_bwd_tc_kernel(ChunkBwdArgs a, const __grid_constant__ CUtensorMap dout_map) {
  pdl_wait();  // no early trigger: one wave for the whole scan, successors must not park beside it
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int warp = threadIdx.x >> 5;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + TcBwdLayout::TSLOT);
  if (threadIdx.x == 0) rscan_init(sm);
  if (warp == 0) {
    tmem_alloc(tslot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  rscan_role(a, &dout_map, sm, tm, blockIdx.x, nullptr);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
}

}  // namespace

void* tensor_map_encode_fn() {
  static void* fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = p;
  });
  return fn;
}

bool scan_tc_applies(int bf16_operands, int DK, int DV) { return bf16_operands && DK == TD && DV == TD; }

cudaError_t launch_scan_fwd_tc(const ChunkFwdArgs& a, cudaStream_t s, bool* outputs_done) {
  *outputs_done = false;
  constexpr int OB = 2 * a1k(OutLayout<bf16, TD, TD>::BYTES) + 4 * 8;  // two output stages + barriers
  const int bytes = (TcFwdLayout::BYTES > OB ? TcFwdLayout::BYTES : OB) + 1024;
  cudaError_t e = cudaFuncSetAttribute(chunk_scan_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0, coop = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) return e;
  const int BH = a.B * a.H;
  // outputs beside the scan when SMs are left over: one cooperative grid of one CTA per SM
  // (the kernel's shared memory admits one), so every output CTA's wait has its scan CTA
  // resident
  bool with_out = a.res.progress && coop && BH < nsm && a.T / C > 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(with_out ? nsm : BH);
  cfg.blockDim = dim3(FWD_THREADS);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = with_out ? 2 : 1;
  prof_mark(K_SCAN_FWD_TC, s, true);
  e = cudaLaunchKernelEx(&cfg, chunk_scan_fwd_tc_kernel, a, (int)with_out);
  if (e == cudaErrorCooperativeLaunchTooLarge && with_out) {
    // the context cannot keep a CTA on every SM at once (an SM-limited partition): the
    // scan alone, and the outputs by their own kernel after it
    (void)cudaGetLastError();
    with_out = false;
    cfg.gridDim = dim3(BH);
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, chunk_scan_fwd_tc_kernel, a, 0);
  }
  prof_mark(K_SCAN_FWD_TC, s, false);
  if (e == cudaSuccess) *outputs_done = with_out;
  return e;
}

cudaError_t launch_scan_bwd_tc(const ChunkBwdArgs& a, cudaStream_t s) {
  // dO [B*T][H][Dv] bf16 as a 3-D tensor (Dv innermost); box 64 columns x 1 head x 64
  // tokens, 128-byte swizzled like the shared-memory tiles
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap map{};  // with no chunks (T = 0) nothing is loaded: dh0 = dh_final
  const cuuint64_t dims[3] = {(cuuint64_t)TD, (cuuint64_t)a.H, (cuuint64_t)a.B * a.T};
  const cuuint64_t strides[2] = {(cuuint64_t)TD * 2, (cuuint64_t)a.H * TD * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (a.T / C > 0 &&
      encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.dout), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int bytes = TcBwdLayout::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(chunk_scan_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  prof_mark(K_SCAN_BWD_TC, s, true);
  e = launch_pdl(chunk_scan_bwd_tc_kernel, dim3(a.B * a.H), dim3(TC_THREADS), bytes, s, a, map);
  prof_mark(K_SCAN_BWD_TC, s, false);
  return e;
}

}  // namespace gdn
