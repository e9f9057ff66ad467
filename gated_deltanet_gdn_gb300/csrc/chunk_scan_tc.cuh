// The pieces of the tensor-core state scans (bf16 operands, Dk = Dv = 128) that more than
// one launch uses: shared-memory and TMEM helpers, and the reverse scan as the work of
// one CTA (rscan_role). chunk_scan_tc.cu runs that role in a kernel of its own; the
// fused backward launch of chunk_bwd_tc.cu runs it in the CTAs of its first B*H blocks
// while the other CTAs form the chunk gradients of the chunks it has finished.
//
// Reverse scan per chunk, in reverse order (the transposes of dU = scale Aqk^T dO + K-tilde dS
// and dS0 = diag(gam) dS + scale Q-hat^T dO - W^T dU of the chunked WY form):
//   dU^T = dO^T (scale Aqk) + dS^T K-tilde^T                 (M = Dv, N = C,  K = C, Dk)
//   dS^T <- dS^T diag(gam) + dO^T (scale Q-hat) + dU^T (-W)  (M = Dv, N = Dk, K = C)
// with dS^T resident in TMEM (lane = value column), its bf16 copy and the dU^T copy
// written to shared memory as MMA operands and stored as the dS and dU records.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int TD = 128;                 // Dk = Dv
constexpr int COMPUTE_THREADS = 256;    // warps 0-7
constexpr int TC_THREADS = COMPUTE_THREADS + 32;  // + the producer warp
constexpr int RS_PRODUCER = COMPUTE_THREADS / 32;  // reverse scan: warp 8 streams the records
constexpr int RS_PUBLISHER = RS_PRODUCER + 1;      // and warp 9 (fused launch) publishes progress
constexpr uint32_t TMEM_COLS = 256;     // S^T or dS^T: columns 0..127; U^T or dU^T: 128..191
constexpr int PANEL_C = C * 128;        // bytes of one 64-column panel of a [C][*] bf16 tile
constexpr int PANEL_D = TD * 128;       // bytes of one 64-column panel of a [Dv][*] bf16 tile

__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Row `row` of a bf16 tile with 128-byte panels, 32 consecutive columns from c0 (a
// multiple of 32): four 16-byte stores.
template <int ROWS, int COLS>
__device__ __forceinline__ void store_row32(Tile<bf16, ROWS, COLS> t, int row, int c0, const float* x) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16(x[8 * q + 0], x[8 * q + 1]);
    u.y = pack_bf16(x[8 * q + 2], x[8 * q + 3]);
    u.z = pack_bf16(x[8 * q + 4], x[8 * q + 5]);
    u.w = pack_bf16(x[8 * q + 6], x[8 * q + 7]);
    *reinterpret_cast<uint4*>(t.ptr(row, c0 + 8 * q)) = u;
  }
}

// Two 32-column TMEM loads of this thread's lane, one completion wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,"
      "%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// S^T row slice (64 fp32 columns of this thread's lane from `col`): load it from TMEM
// into x and write its bf16 copy into the operand tile.
__device__ __forceinline__ void state_copy_out(uint32_t taddr, Tile<bf16, TD, TD> Sa, int row, int col, float* x) {
  tmem_ld64(taddr, x);
  store_row32(Sa, row, col, x);
  store_row32(Sa, row, col + 32, x + 32);
}
// Put the slice back into TMEM scaled column-wise by gam (the decay of the state).
__device__ __forceinline__ void state_scale_back(uint32_t taddr, int col, const float* gam, float* x) {
#pragma unroll
  for (int i = 0; i < 64; i += 4) {
    const float4 g = *reinterpret_cast<const float4*>(gam + col + i);
    x[i] *= g.x;
    x[i + 1] *= g.y;
    x[i + 2] *= g.z;
    x[i + 3] *= g.w;
  }
  float lo[32], hi[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    lo[i] = x[i];
    hi[i] = x[32 + i];
  }
  tmem_st32(taddr, lo);
  tmem_st32(taddr + 32, hi);
  tmem_wait_st();
}

// Descriptor helpers. A 128-byte swizzled descriptor's start address field holds
// address / 16 in 14 bits, so moving inside a tile is an add to the low word.
__device__ __forceinline__ uint64_t desc_k(const void* base) { return umma_desc_sw128(smem_u32(base), 16, 1024); }
__device__ __forceinline__ uint64_t desc_mn(const void* base, int panel) {
  return umma_desc_sw128(smem_u32(base), (uint32_t)panel, 1024);
}
// K step ks of a K-major operand whose 64-column panels are `panel` bytes apart
__device__ __forceinline__ uint64_t kstep_k(uint64_t d, int ks, int panel) {
  return d + (uint64_t)(((ks >> 2) * panel + (ks & 3) * 32) >> 4);
}
// K step ks (16 rows of 128 bytes) of an MN-major operand
__device__ __forceinline__ uint64_t kstep_mn(uint64_t d, int ks) { return d + (uint64_t)((ks * 2048) >> 4); }

__device__ __forceinline__ void umma_commit_to(uint64_t* bar) { umma_commit(bar); }

// Every MMA this thread issued has completed (one commit on a barrier used only here).
__device__ __forceinline__ void drain_mma(uint64_t* bar) {
  umma_commit(bar);
  mbar_drain(bar, 0u);
}

// ------------------------------------------------------------------ reverse
struct TcBwdLayout {
  static constexpr int W = 0;                    // -W          [C][Dk] (MN-major B of dS^T)
  static constexpr int QH = W + C * TD * 2;      // scale Q-hat [C][Dk] (MN-major B of dS^T)
  static constexpr int KT = QH + C * TD * 2;     // K-tilde     [C][Dk] (K-major B of dU^T)
  static constexpr int DO = KT + C * TD * 2;     // dO          [C][Dv] (MN-major A)
  static constexpr int AQK = DO + C * TD * 2;    // scale Aqk   [C][C]  (MN-major B of dU^T)
  static constexpr int STAGE = AQK + C * C * 2;
  static constexpr int STAGES = 2;
  static constexpr int GAM = STAGES * STAGE;     // gam [STAGES][Dk] fp32
  static constexpr int SA = a1k(GAM + STAGES * TD * 4);  // dS^T bf16 [Dv][Dk], two buffers
  static constexpr int UA = SA + 2 * TD * TD * 2;  // dU^T bf16 [Dv][C]
  static constexpr int BAR = UA + TD * C * 2;      // full[STAGES], empty[STAGES], u, s, drain
  static constexpr int NBAR = 2 * STAGES + 3;
  static constexpr int TSLOT = BAR + 8 * NBAR;     // TMEM address (standalone kernel)
  static constexpr int PUB = TSLOT + 8;            // chunks whose records are stored
  static constexpr int BYTES = TSLOT + 16;
  static constexpr uint32_t TX = (uint32_t)(4 * C * TD * 2 + C * C * 2 + TD * 4);
};

// Thread 0, before the CTA synchronises and runs rscan_role.
__device__ __forceinline__ void rscan_init(uint8_t* sm) {
  typedef TcBwdLayout L;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  for (int i = 0; i < L::NBAR; ++i) mbar_init(&bars[i], 1);
  *reinterpret_cast<unsigned*>(sm + L::PUB) = 0u;
  fence_mbar_init();
}
// Thread 0, after every thread has returned from rscan_role, before the shared memory
// is used for anything else.
__device__ __forceinline__ void rscan_inval(uint8_t* sm) {
  typedef TcBwdLayout L;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  for (int i = 0; i < L::NBAR; ++i) mbar_inval(&bars[i]);
}

// The reverse scan of (batch, head) bh. Warps 0-7 move dS^T and dU^T between TMEM and
// shared memory (thread (w, l): TMEM lane 32 (w % 4) + l, column half w / 4) and thread 0
// issues every MMA and record store; warp 8 streams each chunk's records into a ring of
// two stages (cp.async.bulk, and a TMA tensor load for dO) as soon as the tensor cores
// release a stage. With progress not NULL, warp 9 forwards the number of chunks whose dS
// and dU records are stored (thread 0 counts them once their bulk stores have completed)
// to progress[bh * PROGRESS_STRIDE] with a GPU-scope release, off the chunk chain. Other
// warps return at once. The caller has run rscan_init, allocated TMEM_COLS or more
// columns at tm and synchronised the CTA; when thread 0 returns, every load, MMA and
// record store of the role has completed. Every wait is bounded.
__device__ __forceinline__ void rscan_role(const ChunkBwdArgs& a, const CUtensorMap* dout_map, uint8_t* sm,
                                           uint32_t tm, int bh, unsigned* progress) {
  typedef TcBwdLayout L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = bh / a.H, h = bh % a.H;
  const int N = a.T / C;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* empty = full + L::STAGES;
  uint64_t* bar_u = empty + L::STAGES;
  uint64_t* bar_s = bar_u + 1;
  uint64_t* bar_d = bar_s + 1;
  unsigned* pub_s = reinterpret_cast<unsigned*>(sm + L::PUB);
  bf16* const sa_buf = reinterpret_cast<bf16*>(sm + L::SA);
  Tile<bf16, TD, C> Ua{reinterpret_cast<bf16*>(sm + L::UA)};
  float* const gams = reinterpret_cast<float*>(sm + L::GAM);

  if (warp == RS_PUBLISHER) {
    if (lane == 0 && progress) {
      unsigned last = 0;
      for (uint32_t i = 0; last < (unsigned)N && i < WAIT_MAX_TRIES; ++i) {
        const unsigned v = ld_acquire_cta(pub_s);
        if (v > last) {
          st_release_gpu(progress + (size_t)bh * PROGRESS_STRIDE, v);
          last = v;
        } else {
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
  if (warp > RS_PUBLISHER) return;
  if (warp == RS_PRODUCER) {  // ---- producer: chunks in reverse order
    if (lane == 0) {
      for (int it = 0; it < N; ++it) {
        const int n = N - 1 - it, s = it % L::STAGES, k = it / L::STAGES;
        if (k > 0) mbar_wait(&empty[s], (uint32_t)(k - 1) & 1u, a.err);
        uint8_t* st = sm + s * L::STAGE;
        const size_t ch = (size_t)bh * N + n;
        mbar_arrive_expect_tx(&full[s], L::TX);
        bulk_g2s(st + L::W, static_cast<const bf16*>(a.res.wneg) + ch * (C * TD), C * TD * 2, &full[s]);
        bulk_g2s(st + L::QH, static_cast<const bf16*>(a.res.qh) + ch * (C * TD), C * TD * 2, &full[s]);
        bulk_g2s(st + L::KT, static_cast<const bf16*>(a.res.kt) + ch * (C * TD), C * TD * 2, &full[s]);
        bulk_g2s(st + L::AQK, static_cast<const bf16*>(a.res.aqk) + ch * (C * C), C * C * 2, &full[s]);
        bulk_g2s(gams + s * TD, a.res.gam + ch * TD, TD * 4, &full[s]);
        const int tok = b * a.T + n * C;
        tma_load_3d(st + L::DO, dout_map, 0, h, tok, &full[s]);
        tma_load_3d(st + L::DO + PANEL_C, dout_map, 64, h, tok, &full[s]);
      }
      drain_ring(full, L::STAGES, N);
    }
    return;
  }
  // ---- compute warps
  const int row = 32 * (warp & 3) + lane, half = warp >> 2;
  const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);
  const size_t sb = (size_t)bh * TD * TD;
  {
    float lo[32], hi[32];
    for (int i = 0; i < 32; ++i) {
      lo[i] = a.dh_final ? a.dh_final[sb + (size_t)(64 * half + i) * TD + row] : 0.f;
      hi[i] = a.dh_final ? a.dh_final[sb + (size_t)(64 * half + 32 + i) * TD + row] : 0.f;
    }
    tmem_st32(tl + 64 * half, lo);
    tmem_st32(tl + 64 * half + 32, hi);
    tmem_wait_st();
  }
  constexpr uint32_t id_a = umma_idesc_bf16(128, C, true, true);    // dO^T Aqk
  constexpr uint32_t id_b = umma_idesc_bf16(128, C, false, false);  // dS^T K-tilde^T
  constexpr uint32_t id_c = umma_idesc_bf16(128, TD, true, true);   // dO^T Q-hat
  constexpr uint32_t id_d = umma_idesc_bf16(128, TD, false, true);  // dU^T (-W)
  bf16* dstate_rec = static_cast<bf16*>(a.ws.dstate);
  bf16* du_rec = static_cast<bf16*>(a.ws.du);
  uint32_t ph_u = 0, ph_s = 0;
#pragma unroll 1
  for (int it = 0; it < N; ++it) {
    const int n = N - 1 - it, s = it % L::STAGES;
    uint8_t* st = sm + s * L::STAGE;
    const size_t ch = (size_t)bh * N + n;
    Tile<bf16, TD, TD> Sa{sa_buf + (it & 1) * (TD * TD)};
    if (it > 0) {
      mbar_wait(bar_s, ph_s, a.err);
      ph_s ^= 1u;
      tc_fence_after();
    }
    mbar_wait(&full[s], (uint32_t)(it / L::STAGES) & 1u, a.err);
    // dS^T -> bf16 operand (the record of the gradient leaving chunk n)
    float xs[64];
    state_copy_out(tl + 64 * half, Sa, row, 64 * half, xs);
    fence_proxy_async();
    tc_fence_before();
    if (tid == 0) bulk_wait_read0();  // the previous dU record store has read Ua
    compute_sync();
    if (tid == 0) {
      tc_fence_after();
      bulk_s2g(dstate_rec + ch * (TD * TD), Sa.p, TD * TD * 2);
      bulk_commit();
      const uint64_t dSa = desc_k(Sa.p);
      const uint64_t dDo = desc_mn(st + L::DO, PANEL_C), dAq = desc_mn(st + L::AQK, PANEL_C);
      const uint64_t dKt = desc_k(st + L::KT);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) umma_bf16(tm + 128, kstep_mn(dDo, ks), kstep_mn(dAq, ks), id_a, ks > 0);
#pragma unroll
      for (int ks = 0; ks < TD / 16; ++ks)
        umma_bf16(tm + 128, kstep_k(dSa, ks, PANEL_D), kstep_k(dKt, ks, PANEL_C), id_b, 1u);
      umma_commit_to(bar_u);
      // every bulk group but this chunk's dS: steps < it stored. Published after each of
      // the first chunks (the gradient CTAs start on them), then after every second one:
      // each publication holds thread 0 on the chain until the copies complete, and the
      // gradient CTAs stay well behind the scan after the start (measured 3 us faster
      // than publishing every chunk at B8 T4096 H6; every fourth: no gain)
      if (progress && it > 0 && (it < 4 || (it & 1) == 0)) {
        bulk_wait1();
        fence_proxy_async_global();
        st_release_cta(pub_s, (unsigned)it);
      }
    }
    // dS^T <- dS^T diag(gam) while the tensor cores form dU^T; every product into dS^T
    // comes after the next barrier
    state_scale_back(tl + 64 * half, 64 * half, gams + s * TD, xs);
    mbar_wait(bar_u, ph_u, a.err);
    ph_u ^= 1u;
    tc_fence_after();
    {  // dU^T row -> bf16 operand (the dU record)
      float x[32];
      tmem_ld32(tl + 128 + 32 * half, x);
      store_row32(Ua, row, 32 * half, x);
    }
    fence_proxy_async();
    tc_fence_before();
    // the dS record store of the previous chunk has read the buffer the next one writes
    if (tid == 0) bulk_wait_read1();
    compute_sync();
    if (tid == 0) {
      tc_fence_after();
      bulk_s2g(du_rec + ch * (C * TD), Ua.p, C * TD * 2);
      bulk_commit();
      const uint64_t dW = desc_mn(st + L::W, PANEL_C), dUa = desc_k(Ua.p);
      const uint64_t dDo = desc_mn(st + L::DO, PANEL_C), dQh = desc_mn(st + L::QH, PANEL_C);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) umma_bf16(tm, kstep_mn(dDo, ks), kstep_mn(dQh, ks), id_c, 1u);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) umma_bf16(tm, kstep_k(dUa, ks, PANEL_D), kstep_mn(dW, ks), id_d, 1u);
      umma_commit_to(&empty[s]);
      umma_commit_to(bar_s);
    }
  }
  if (N > 0) {
    mbar_wait(bar_s, ph_s, a.err);
    tc_fence_after();
  }
  if (a.dh0) {
    float x[64];
    tmem_ld64(tl + 64 * half, x);
#pragma unroll
    for (int i = 0; i < 64; ++i) a.dh0[sb + (size_t)(64 * half + i) * TD + row] = x[i];
  }
  if (tid == 0) {  // record stores and every issued MMA complete before TMEM is reused
    bulk_wait0();
    if (progress) {
      fence_proxy_async_global();
      st_release_cta(pub_s, (unsigned)N);
    }
    drain_mma(bar_d);
  }
}

}  // namespace
}  // namespace gdn
