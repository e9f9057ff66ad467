// Chunk-parallel gradients of the chunked backward on the 5th-generation tensor cores,
// one fused kernel per 64-token chunk and head (bf16 operands, Dk = Dv = 128).
//
// It replaces the chain state products -> score gradients -> channel-group sums of the
// CUDA-core path (chunk_bwd.cu, chunk_grads.cu) for this shape: everything a chunk needs
// after the reverse scan is computed in one CTA, so nothing but the gradients leaves it.
// Inputs per chunk: the forward's records T, U^T and the chunk-start state S0^T, the
// reverse scan's dU^T and dS1^T, dout (3-D TMA tensor load), and q, k, v, g, beta.
// The products (chunked WY backward, header of chunk_bwd.cu), each one tcgen05.mma
// sequence with M = 128 and fp32 accumulation in tensor memory:
//   P1  Y^T  = dU^T T                                   lanes v, columns t
//   P2  D2   = [dO ; Y] U^T         (two 64-token operands stacked to M = 128)
//              rows 0..63: dO U^T -> dAqk = scale (..) masked j <= t
//              rows 64..127: Y U^T -> dAkk = -(..) masked j < t
//   P3  D3   = S0 [dO ; Y]^T        lanes c: columns t -> dQ-hat / scale, 64 + t -> -dBk
//   P4  D4   = dS1 U^T              lanes c: dK-tilde
//   P5  D5   = Ye^T [dAqk ; dAkk]^T lanes c: the x-side score gradients of both families
//   P6  D6   = [Xq ; Xk]^T [dAqk ; dAkk]  lanes c: the y-side score gradients, summed
// with the boundary-split row scaling of the marin.community note "factoring GDN-2 decay
// on TPU" (section Approach): Ye = k exp(G_b - G), Xq = q exp(G - G_b),
// Xk = beta k exp(G - G_b) about the last token b of the first 32-token block. The
// epilogue then runs one thread per key channel and 16 tokens: dq, dk, the
// per-channel decay gradient, its reverse cumulative sum inside the chunk (the last row
// also collects the K-tilde column sums and dgam * gam, dgam = rowsum(dS1 * S0)), and
// dbeta, whose sums over channels and value columns are done in the CTA in fixed order.
// A block whose decay spread would push the row factors out of range (or every block,
// with GDN_FLAG_PAIRWISE_WITHIN_BLOCK) has its in-block score gradients summed pairwise on
// CUDA cores instead, as the note's kernel does for every in-block pair; one decay per
// head (g [B,T,H]) uses the mask form: the C x C factor exp(G_t - G_j) <= 1 is applied to
// dAqk and dAkk, and the operands are q, beta k and k themselves.
//
// Roles (512 threads, one CTA per SM, persistent over chunk-heads): all sixteen warps run
// the epilogues, four per TMEM lane quarter, each on a quarter of the chunk's tokens (16).
// Thread 0 issues P2, thread 32 P3 and the group B loads, thread 64 P4 and P5, thread 96
// P1 and P6, thread 128 the group A loads and thread 160 the q/k/g loads: a tcgen05.mma
// or bulk-copy issue stalls its thread, so the issue work is spread over six warps (the
// loads of the first chunk are issued by thread 0 at the start). Each load
// is issued as soon as the buffer it fills is released (T and dU^T once P1 has read them,
// q and k once P5 and P6 have, the rest once P2-P4 and the gamma-gradient sums have), so
// the next chunk's loads overlap this chunk's later phases. Every wait is bounded.
//
// Two launch shapes. With fewer (batch, head) pairs than SMs, one cooperative grid of one
// CTA per SM runs the reverse scan as well: CTAs 0 .. B*H-1 first run rscan_role
// (chunk_scan_tc.cuh) for their (batch, head), publishing as they go how many chunks'
// dU and dS records are stored, then join the others, which take chunk-heads from a queue
// in the order the scan finishes them and wait (bounded) on those counters before loading
// a chunk's records. Otherwise the reverse scan is a launch of its own before this one,
// and the CTAs stride over the chunk-heads.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "chunk_scan_tc.cuh"
#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int BD = 128;                 // Dk = Dv
constexpr int BT_THREADS = 512;          // 16 warps
constexpr int NTG = 4;                   // token groups (warps per TMEM lane quarter)
constexpr int TPT = C / NTG;             // tokens per thread in the epilogues
constexpr int EB = 4;                    // tokens per batch of the final epilogue
constexpr uint32_t BT_TMEM_COLS = 512;
// TMEM columns
constexpr int TC_D3 = 0, TC_D4 = 128, TC_D5 = 192, TC_D6 = 320, TC_P1 = 384, TC_P2 = 448;
// After E2 has read D2, its columns hold the chunk's q and k (packed bf16 pairs, lanes =
// key channels, columns = tokens) for the final epilogue, until the next chunk's P2.
constexpr int TC_QK = TC_P2;

struct BtLayout {
  // group A: what P1 reads
  static constexpr int TM = 0;                 // T      [C][C]
  static constexpr int DUT = TM + C * C * 2;   // dU^T   [Dv][C]
  static constexpr int VT = DUT + BD * C * 2;  // v      [C][Dv] (3-D TMA tensor load)
  // group B (and the Y rows of DY, written by the epilogue)
  static constexpr int DY = VT + C * BD * 2;   // [dO ; Y] [2C][Dv]
  static constexpr int UT = DY + 2 * C * BD * 2;   // U^T  [Dv][C]
  static constexpr int S0T = UT + BD * C * 2;      // S0^T [Dv][Dk]
  static constexpr int DS1T = S0T + BD * BD * 2;   // dS1^T [Dv][Dk]
  // operands built per chunk
  static constexpr int X = DS1T + BD * BD * 2;     // [Xq | Xk]^T [Dk][2C] (q ; k land here first)
  static constexpr int YE = X + 2 * C * BD * 2;    // Ye^T [Dk][C] (per-channel g lands here first)
  static constexpr int DP = YE + C * BD * 2;       // [dAqk ; dAkk] [2C][C]
  // small arrays (fp32)
  static constexpr int BETA = DP + 2 * C * C * 2;  // [C]
  static constexpr int GSC = BETA + C * 4;         // [C] scalar-decay G per token
  static constexpr int DIAG = GSC + C * 4;         // [C] diagonal of dAqk
  static constexpr int DBV = DIAG + C * 4;         // [4][C] dbeta_v partials per lane quarter
  static constexpr int DBP = DBV + 4 * C * 4;      // [4][C] score dbeta partials
  static constexpr int DGP = DBP + 4 * C * 4;      // [4][C] scalar dg partials
  static constexpr int GX = DGP + 4 * C * 4;       // [NTG][Dk] token-group totals of g
  static constexpr int COLP = GX + NTG * BD * 4;   // [NTG][Dk] K-tilde column partials
  static constexpr int DGAM = COLP + NTG * BD * 4; // [Dk] dgam (room for [NTG][Dk])
  static constexpr int CTOT = GX;                  // [NTG][Dk] token-group totals of dG (final
                                                   // epilogue only; GX is read before it)
  static constexpr int FLAGS = DGAM + NTG * BD * 4;  // int [4]: unsafe1, unsafe2
  static constexpr int BAR = FLAGS + 16;           // 8 mbarriers
  static constexpr int UNITS = BAR + 8 * 8;        // int [4]: claimed units (fused launch)
  static constexpr int TSLOT = UNITS + 16;         // TMEM address (both roles)
  static constexpr int BYTES = TSLOT + 16;
  static constexpr uint32_t TXA = (uint32_t)(C * C * 2 + BD * C * 2 + C * BD * 2);
  static constexpr uint32_t TXB = (uint32_t)(C * BD * 2 + BD * C * 2 + 2 * BD * BD * 2);
  static constexpr uint32_t TXQ = (uint32_t)(2 * C * BD * 2);  // q, k into X
  static constexpr uint32_t TXG = (uint32_t)(C * BD * 2);      // per-channel g into YE
};
static_assert(BtLayout::BYTES + 1024 <= 227 * 1024, "shared memory of one CTA");
static_assert(TcBwdLayout::BYTES <= BtLayout::TSLOT, "the reverse scan role leaves the TMEM address alone");

// The fused launch: CTAs 0 .. nscan - 1 first run the reverse scan of (batch, head)
// blockIdx.x (rscan_role) and publish its progress; every CTA then claims chunk-heads from
// the queue in the order the scan finishes them (all heads' last chunk first) and waits,
// before it loads a chunk's dU and dS records, until that chunk's head has published them.
// queue NULL: no scan, a static stride over the chunk-heads.
struct BwdSync {
  unsigned* progress;  // [B*H][PROGRESS_STRIDE]: chunks the reverse scan has finished
  unsigned* queue;     // the next unit to claim
  int nscan;
};
static_assert(BtLayout::CTOT + NTG * BD * 4 <= BtLayout::COLP, "the dG totals fit in the G totals' place");

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 512;\n" ::: "memory"); }

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
// Input element through the read-only path: the compiler may move these loads ahead of
// the kernel's stores, so each loop below issues its loads as one batch.
__device__ __forceinline__ float ldg_bf16(const bf16* p) {
  return __bfloat162float(__ushort_as_bfloat16(__ldg(reinterpret_cast<const unsigned short*>(p))));
}
__device__ __forceinline__ uint32_t pack2_bf16(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack8_bf16(const float* x) {
  return make_uint4(pack2_bf16(x[0], x[1]), pack2_bf16(x[2], x[3]), pack2_bf16(x[4], x[5]), pack2_bf16(x[6], x[7]));
}

// Sums over the 32 lanes of a warp of TPT = 16 values per lane at once (recursive
// halving: at each step a lane keeps half of its values and adds its partner's copy of
// them, 8 + 4 + 2 + 1 shuffles, then one more for the last pair). On return lane l holds
// the warp total of value (l >> 1) & 15 (lanes 2i and 2i + 1 both hold value i).
__device__ __forceinline__ float warp_sum16(float (&x)[16], int lane) {
#pragma unroll
  for (int h = 8; h >= 1; h >>= 1) {
    const bool up = (lane & (2 * h)) != 0;  // this lane keeps the upper half of its values
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? x[i] : x[i + h];
      const float keep = up ? x[i + h] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * h);
    }
  }
  return x[0] + __shfl_xor_sync(0xffffffffu, x[0], 1);
}

// Sums over the 32 lanes of a warp of 8 values per lane (recursive halving, 4 + 2 + 1
// shuffles, then two more). On return lane l holds the warp total of value (l >> 2) & 7.
__device__ __forceinline__ float warp_sum8(float (&x)[8], int lane) {
#pragma unroll
  for (int h = 4; h >= 1; h >>= 1) {
    const bool up = (lane & (4 * h)) != 0;  // this lane keeps the upper half of its values
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? x[i] : x[i + h];
      const float keep = up ? x[i + h] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4 * h);
    }
  }
  float r = x[0] + __shfl_xor_sync(0xffffffffu, x[0], 2);
  return r + __shfl_xor_sync(0xffffffffu, r, 1);
}

// In-block score gradients summed pairwise (blocks whose row factors would leave the fp32
// range, or every block with GDN_FLAG_PAIRWISE_WITHIN_BLOCK): for token t of block
// [bs, bs + BLK) and channel c, with E(a, b) = exp(G_ac - G_bc),
//   dxa += sum_{j=bs..t} dAqk[t][j] k_jc E(t, j),   dxb += sum_{j=bs..t} dAkk[t][j] k_jc E(t, j)
//   dy  += sum_{s=t..bs+BLK-1} (dAqk[s][t] q_sc + dAkk[s][t] beta_s k_sc) E(s, t)
// Gf: fp32 G of the chunk [C][Dk + 4] in shared memory; q, k rows of the chunk in global
// memory (row stride rs elements).
// Returns (dxa, dxb, dy) to add.
__device__ __noinline__ float3 pairwise_terms(const bf16* dpt, const float* Gf, const bf16* qg, const bf16* kg,
                                              size_t rs, const float* beta_s, int t, int c, int bs) {
  constexpr int LD = BD + 4;
  typedef Sw<bf16, 2 * C, C> DPL;
  const float Gt = Gf[t * LD + c];
  float sa = 0.f, sb = 0.f, sy = 0.f;
  for (int j = bs; j <= t; ++j) {
    const float e = __expf(Gt - Gf[j * LD + c]);
    const float kj = __bfloat162float(kg[(size_t)j * rs + c]);
    sa = fmaf(__bfloat162float(dpt[DPL::off(t, j)]) * kj, e, sa);
    sb = fmaf(__bfloat162float(dpt[DPL::off(C + t, j)]) * kj, e, sb);
  }
  for (int s = t; s < bs + BLK; ++s) {
    const float e = __expf(Gf[s * LD + c] - Gt);
    const float qs = __bfloat162float(qg[(size_t)s * rs + c]);
    const float ks = __bfloat162float(kg[(size_t)s * rs + c]);
    const float v = __bfloat162float(dpt[DPL::off(s, t)]) * qs +
                    __bfloat162float(dpt[DPL::off(C + s, t)]) * beta_s[s] * ks;
    sy = fmaf(v, e, sy);
  }
  return make_float3(sa, sb, sy);
}

template <bool PC>
__global__ void __launch_bounds__(BT_THREADS, 1)
    chunk_bwd_tc_kernel(ChunkBwdArgs a, const __grid_constant__ CUtensorMap dout_map,
                        const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap q_map,
                        const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap g_map,
                        BwdSync sync) {
  pdl_wait();
  pdl_trigger();
  typedef BtLayout L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = a.B * a.H, N = a.T / C, units = N * BH;
  const bool fused = sync.queue != nullptr;
  // static stride: this CTA's units; fused: claimed one ahead into units_s[m % 4]
  const int nunits = fused ? 0 : (units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  int* units_s = reinterpret_cast<int*>(sm + L::UNITS);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::TSLOT);
  const bool scan_cta = (int)blockIdx.x < sync.nscan;
  if (scan_cta && tid == 0) rscan_init(sm);
  if (warp == 0) {
    tmem_alloc(tslot, BT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  if (scan_cta) {  // the reverse scan first; then this CTA joins the gradient work
    rscan_role(a, &dout_map, sm, tm, blockIdx.x, sync.progress);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) rscan_inval(sm);
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* fullA = bars + 0;
  uint64_t* fullB = bars + 1;
  uint64_t* bP1 = bars + 2;
  uint64_t* bP2 = bars + 3;
  uint64_t* bP34 = bars + 4;
  uint64_t* bP56 = bars + 5;
  uint64_t* bDrain = bars + 6;
  uint64_t* fullQ = bars + 7;
  float* beta_s = reinterpret_cast<float*>(sm + L::BETA);
  float* gsc = reinterpret_cast<float*>(sm + L::GSC);
  float* diag_s = reinterpret_cast<float*>(sm + L::DIAG);
  float* dbv_s = reinterpret_cast<float*>(sm + L::DBV);
  float* dbp_s = reinterpret_cast<float*>(sm + L::DBP);
  float* dgp_s = reinterpret_cast<float*>(sm + L::DGP);
  float* gx_s = reinterpret_cast<float*>(sm + L::GX);
  float* colp_s = reinterpret_cast<float*>(sm + L::COLP);
  float* dgam_s = reinterpret_cast<float*>(sm + L::DGAM);
  float* ctot_s = reinterpret_cast<float*>(sm + L::CTOT);
  int* flags_s = reinterpret_cast<int*>(sm + L::FLAGS);

  if (tid == 0) {
    mbar_init(fullA, 1);
    mbar_init(fullB, 1);
    mbar_init(bP1, 1);
    mbar_init(bP2, 1);
    mbar_init(bP34, 2);  // P3 (thread 32) and P4 (thread 64)
    mbar_init(bP56, 2);  // P5 (thread 64) and P6 (thread 96)
    mbar_init(bDrain, 4);  // every issuing thread: 0, 32, 64, 96
    mbar_init(fullQ, 1);
    if (fused) units_s[0] = (int)atomicAdd(sync.queue, 1u);
    fence_mbar_init();
  }
  __syncthreads();

  // the m-th unit of this CTA: static, head-major; fused, in the order the reverse scan
  // finishes chunks (unit index = (N - 1 - n) * B*H + bh)
  auto valid = [&](int m) { return fused ? units_s[m & 3] < units : m < nunits; };
  auto unit_of = [&](int m, int& n, int& bh) {
    if (fused) {
      const int u = units_s[m & 3], it = u / BH;
      bh = u - it * BH;
      n = N - 1 - it;
    } else {
      const int u = (int)blockIdx.x + m * (int)gridDim.x;
      bh = u / N;
      n = u % N;
    }
  };
  // fused: the reverse scan has stored chunk n's dU and dS records. Group A's loader
  // acquires the head's counter; group B's loads of the same chunk are issued later by
  // another thread, after CTA barriers that follow that acquire, so they need only the
  // proxy fence (a GPU-scope acquire costs about 700 cycles of the issuing warp)
  auto wait_scan = [&](int n, int bh, bool acquire) {
    if (fused) {
      if (acquire) wait_counter(sync.progress + (size_t)bh * PROGRESS_STRIDE, (unsigned)(N - n), a.err);
      fence_proxy_async_global();
    }
  };

  // loads, issued by thread 0: group A (T, dU^T, v) and group B (dO, U^T, S0^T, dS1^T)
  auto load_a = [&](int m) {
    int n, bh;
    unit_of(m, n, bh);
    wait_scan(n, bh, true);
    const size_t ch = (size_t)bh * N + n;
    mbar_arrive_expect_tx(fullA, L::TXA);
    bulk_g2s(sm + L::TM, static_cast<const bf16*>(a.res.tmat) + ch * (C * C), C * C * 2, fullA);
    bulk_g2s(sm + L::DUT, static_cast<const bf16*>(a.ws.du) + ch * (C * BD), BD * C * 2, fullA);
    const int b = bh / a.H, h = bh % a.H, tok = b * a.T + n * C;
    tma_load_3d(sm + L::VT, &v_map, 0, h, tok, fullA);                // v, columns 0-63
    tma_load_3d(sm + L::VT + C * 128, &v_map, 64, h, tok, fullA);     // columns 64-127
  };
  auto load_b = [&](int m) {  // after load_a(m): by the same thread, or past CTA barriers
    int n, bh;
    unit_of(m, n, bh);
    wait_scan(n, bh, false);
    const size_t ch = (size_t)bh * N + n;
    mbar_arrive_expect_tx(fullB, L::TXB);
    const int b = bh / a.H, h = bh % a.H, tok = b * a.T + n * C;
    tma_load_3d(sm + L::DY, &dout_map, 0, h, tok, fullB);                 // dO, columns 0-63
    tma_load_3d(sm + L::DY + 2 * C * 128, &dout_map, 64, h, tok, fullB);  // columns 64-127
    bulk_g2s(sm + L::UT, static_cast<const bf16*>(a.res.u) + ch * (C * BD), BD * C * 2, fullB);
    bulk_g2s(sm + L::S0T, static_cast<const bf16*>(a.res.state) + ch * (BD * BD), BD * BD * 2, fullB);
    bulk_g2s(sm + L::DS1T, static_cast<const bf16*>(a.ws.dstate) + ch * (BD * BD), BD * BD * 2, fullB);
  };
  // group Q: q and k into the rows of X (the operand build rewrites them in place) and
  // per-channel g (row-major) into YE, once P5 and P6 of the previous chunk have read them
  auto load_q = [&](int m) {
    int n, bh;
    unit_of(m, n, bh);
    mbar_arrive_expect_tx(fullQ, L::TXQ + (PC ? L::TXG : 0u));
    const int b = bh / a.H, h = bh % a.H, tok = b * a.T + n * C;
    tma_load_3d(sm + L::X, &q_map, 0, h, tok, fullQ);                           // q, columns 0-63
    tma_load_3d(sm + L::X + 2 * C * 128, &q_map, 64, h, tok, fullQ);            // columns 64-127
    tma_load_3d(sm + L::X + C * 128, &k_map, 0, h, tok, fullQ);                 // k, rows C..
    tma_load_3d(sm + L::X + 2 * C * 128 + C * 128, &k_map, 64, h, tok, fullQ);
    if (PC) tma_load_3d(sm + L::YE, &g_map, 0, h, tok, fullQ);
  };
  if (tid == 0 && valid(0)) {
    load_a(0);
    load_b(0);
    load_q(0);
  }

  // ---- all 16 warps. Lane quarter qw = warp % 4 (TMEM lanes 32 qw .. + 31, a value
  // column, a token row of D2 or a key channel), token group tg = warp / 4 (tokens or
  // columns TPT tg .. + TPT - 1).
  const int qw = warp & 3, tg = warp >> 2;
  const int rowl = 32 * qw + lane;
  const uint32_t tl = tm + ((uint32_t)(32 * qw) << 16);
  const int t_beg = TPT * tg;  // this thread's first token
  const int blk = t_beg / BLK; // its 32-token block
  const bool force = (a.flags & FLAG_PAIRWISE) != 0;
  const bool mask_form = !PC && !force;
  const bf16* qg = static_cast<const bf16*>(a.q);
  const bf16* kg = static_cast<const bf16*>(a.k);
  const bf16* gg = static_cast<const bf16*>(a.g);
  const bf16* bg = static_cast<const bf16*>(a.beta);
  const size_t rs = (size_t)a.H;  // token stride in rows
  Tile<bf16, 2 * C, BD> DYt{reinterpret_cast<bf16*>(sm + L::DY)};
  Tile<bf16, 2 * C, BD> Xt{reinterpret_cast<bf16*>(sm + L::X)};      // q ; k as loaded
  Tile<bf16, BD, 2 * C> XTt{reinterpret_cast<bf16*>(sm + L::X)};     // [Xq | Xk]^T, built in their place
  Tile<bf16, BD, C> YeTt{reinterpret_cast<bf16*>(sm + L::YE)};       // Ye^T
  Tile<bf16, 2 * C, C> DPt{reinterpret_cast<bf16*>(sm + L::DP)};
  const bf16* S0T = reinterpret_cast<const bf16*>(sm + L::S0T);
  const bf16* DS1T = reinterpret_cast<const bf16*>(sm + L::DS1T);

  // instruction descriptors
  constexpr uint32_t id_p1 = umma_idesc_bf16(128, C, false, true);     // dU^T (K-major) x T (MN-major)
  constexpr uint32_t id_p2 = umma_idesc_bf16(128, C, false, true);     // DY (K-major) x U^T (MN-major)
  constexpr uint32_t id_p3 = umma_idesc_bf16(128, 2 * C, true, false); // S0 (MN-major) x DY^T (K-major)
  constexpr uint32_t id_p4 = umma_idesc_bf16(128, C, true, true);      // dS1 (MN-major) x U^T (MN-major)
  constexpr uint32_t id_p5 = umma_idesc_bf16(128, 2 * C, false, false); // Ye^T (K-major) x DP^T (K-major)
  constexpr uint32_t id_p6 = umma_idesc_bf16(128, C, false, true);      // X^T (K-major) x DP (MN-major)

  // per-thread values that live from the operand build to the final epilogue: G of this
  // thread's channel over its TPT tokens, and G at the block boundary and the last token
  float Greg[TPT];
  float Gb = 0.f, GC = 0.f;
  int cur_n = 0, cur_bh = 0;  // the chunk whose final epilogue is pending
  int nproc = 0;  // units this CTA processed
  // thread 0, fused: units are claimed two steps ahead, so that an atomic's round trip
  // has a whole step to return before its value is needed (a step-ahead claim held
  // thread 0 about 450 cycles per step). pend0: the unit of step m + 1, stored into
  // units_s during step m; pend1: the unit of step m + 2, claimed at the top of step m.
  unsigned pend0 = 0, pend1 = 0;
  if (fused && tid == 0) pend0 = units_s[0] < units ? atomicAdd(sync.queue, 1u) : (unsigned)units;

#pragma unroll 1
  for (int m = 0;; ++m) {
    const bool cur = valid(m);
    const uint32_t par = (uint32_t)m & 1u;
    int n = 0, bh = 0;
    if (cur) unit_of(m, n, bh);
    if (fused && cur && tid == 0) pend1 = pend0 < (unsigned)units ? atomicAdd(sync.queue, 1u) : (unsigned)units;
    bool q_early = true;  // this chunk's group Q loads were issued at the start of (b)
    // this chunk's beta, read while the previous chunk's final epilogue runs
    float beta_pre = 0.f;
    if (cur && tid < C) {
      const size_t r = ((size_t)(bh / a.H) * a.T + (size_t)n * C + tid) * a.H + (bh % a.H);
      beta_pre = ldg_bf16(bg + r);
    }
    // (a) P1 of this chunk: Y^T = dU^T T
    if (cur && tid == 96) {
      mbar_wait(fullA, par, a.err);
      tc_fence_after();
      const uint64_t dA = desc_kmajor(sm + L::DUT), dB = desc_mnmajor(sm + L::TM, C * 128);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        umma_bf16(tm + TC_P1, kstep_kmajor(dA, ks, BD * 128), kstep_mnmajor(dB, ks), id_p1, ks > 0);
      umma_commit(bP1);
    }
    // (b) the previous chunk's final epilogue, while P1 and this chunk's loads run.
    // Thread: key channel c = rowl, tokens t_beg .. + TPT - 1.
    if (m > 0) {
      const int b0 = cur_bh / a.H, h0 = cur_bh % a.H;
      const size_t row0 = ((size_t)b0 * a.T + (size_t)cur_n * C) * a.H + h0;
      const uint32_t pp = (uint32_t)(m - 1) & 1u;
      mbar_wait(bP34, pp, a.err);
      mbar_wait(bP56, pp, a.err);
      tc_fence_after();
      const int c = rowl;
      const int bs = BLK * blk;
      const bool unsafe1 = flags_s[0] != 0, unsafe2 = flags_s[1] != 0;
      const bool fast = !mask_form && !(unsafe1 || unsafe2);
      q_early = mask_form || fast;  // X is not borrowed for G below
      if (tid == 160 && cur && q_early) load_q(m);
      const bool blk1 = blk == 0;
      const bool pw_rows = !mask_form && !fast && (blk1 ? unsafe1 : unsafe2);
      const bool skip_x = pw_rows && blk1, skip_y = pw_rows && !blk1;
      float* Gf = reinterpret_cast<float*>(sm + L::X);  // fp32 G [C][Dk + 4] (pairwise only)
      if (!mask_form && !fast) {
        // the operands X / Ye are no longer read (P5, P6 completed): G of the chunk goes there
#pragma unroll
        for (int i = 0; i < TPT; ++i) Gf[(t_beg + i) * (BD + 4) + c] = Greg[i];
        epi_sync();
      }
      const float eGb = fast ? __expf(Gb) : 0.f, eCb = fast ? __expf(GC - Gb) : 0.f;
      float dGr[TPT], pdb[TPT];
      float colp = 0.f;
#pragma unroll
      for (int i0 = 0; i0 < TPT; i0 += EB) {
        const int t0 = t_beg + i0;
        uint32_t r3a[EB], r3b[EB], r4[EB], r5a[EB], r5b[EB], r6[EB], rqk[EB];
        tmem_ld4_nowait(tl + TC_QK + t0, rqk);
        tmem_ld4_nowait(tl + TC_D3 + t0, r3a);
        tmem_ld4_nowait(tl + TC_D3 + C + t0, r3b);
        tmem_ld4_nowait(tl + TC_D4 + t0, r4);
        tmem_ld4_nowait(tl + TC_D5 + t0, r5a);
        tmem_ld4_nowait(tl + TC_D5 + C + t0, r5b);
        tmem_ld4_nowait(tl + TC_D6 + t0, r6);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < EB; ++i) {
          const int t = t0 + i;
          const size_t gi = (row0 + (size_t)t * rs) * BD + c;
          const __nv_bfloat162 qk2 = *reinterpret_cast<const __nv_bfloat162*>(&rqk[i]);
          const float qf = __low2float(qk2), kf = __high2float(qk2);
          const float G = Greg[i0 + i];
          const float br = beta_s[t], dgd = diag_s[t];
          const float dqh = a.scale * u2f(r3a[i]), dbk = -u2f(r3b[i]), dkt = u2f(r4[i]);
          float e1 = 1.f, e2 = 1.f, gm, kd;
          if (mask_form) {
            gm = __expf(G);
            kd = __expf(GC - G);
          } else {
            e1 = __expf(G - Gb);
            e2 = __expf(Gb - G);
            gm = fast ? eGb * e1 : __expf(G);
            kd = fast ? eCb * e2 : __expf(GC - G);
          }
          float dxa = skip_x ? 0.f : u2f(r5a[i]) * e1;
          float dxb = skip_x ? 0.f : u2f(r5b[i]) * e1;
          float dy = skip_y ? 0.f : u2f(r6[i]) * e2;
          if (pw_rows) {
            const float3 pw = pairwise_terms(reinterpret_cast<const bf16*>(sm + L::DP), Gf, qg + row0 * BD,
                                             kg + row0 * BD, rs * BD, beta_s, t, c, bs);
            dxa += pw.x;
            dxb += pw.y;
            dy += pw.z;
          }
          const float khat = gm * kf, ktil = kd * kf, dkh = br * dbk;
          const float oq = dqh * gm + dxa + dgd * kf;
          const float ok = br * dxb + dy + dgd * qf + dkh * gm + dkt * kd;
          dGr[i0 + i] = kf * (br * dxb - dy) + qf * (dxa + dqh * gm) + dkh * khat - dkt * ktil;
          colp = fmaf(dkt, ktil, colp);
          static_cast<bf16*>(a.dq)[gi] = __float2bfloat16_rn(oq);
          static_cast<bf16*>(a.dk)[gi] = __float2bfloat16_rn(ok);
          pdb[i0 + i] = kf * dxb + dbk * khat;
        }
      }
      {
        const float sdb = warp_sum16(pdb, lane);
        if ((lane & 1) == 0) dbp_s[qw * C + t_beg + (lane >> 1)] = sdb;
      }
      // reverse cumulative sum of dG per channel inside the chunk: this group's tokens
      // first, then the later groups' totals; the last row also gets the K-tilde column
      // sums and dgam * gam
      float tot = 0.f;
#pragma unroll
      for (int i = TPT - 1; i >= 0; --i) {
        tot += dGr[i];
        dGr[i] = tot;
      }
      colp_s[tg * BD + c] = colp;
      ctot_s[tg * BD + c] = tot;
      tc_fence_before();  // the TMEM reads of this chunk are done before the next products
      epi_sync();
      {
        float suffix = ((colp_s[c] + colp_s[BD + c]) + (colp_s[2 * BD + c] + colp_s[3 * BD + c])) +
                       dgam_s[c] * __expf(GC);
        for (int g2 = NTG - 1; g2 > tg; --g2) suffix += ctot_s[g2 * BD + c];
#pragma unroll
        for (int i = 0; i < TPT; ++i) dGr[i] += suffix;
      }
      if (PC) {
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
          const size_t gi = (row0 + (size_t)(t_beg + i) * rs) * BD + c;
          static_cast<bf16*>(a.dg)[gi] = __float2bfloat16_rn(dGr[i]);
        }
      } else {
        const float sg = warp_sum16(dGr, lane);  // (dGr is not needed afterwards)
        if ((lane & 1) == 0) dgp_s[qw * C + t_beg + (lane >> 1)] = sg;
      }
      epi_sync();
      if (tid < C) {  // per token: fixed-order sums over the four lane quarters
        const int t = tid;
        const size_t r = row0 + (size_t)t * rs;
        const float db = ((dbv_s[t] + dbv_s[C + t]) + (dbv_s[2 * C + t] + dbv_s[3 * C + t])) +
                         ((dbp_s[t] + dbp_s[C + t]) + (dbp_s[2 * C + t] + dbp_s[3 * C + t]));
        static_cast<bf16*>(a.dbeta)[r] = __float2bfloat16_rn(db);
        if (!PC)
          static_cast<bf16*>(a.dg)[r] = __float2bfloat16_rn((dgp_s[t] + dgp_s[C + t]) +
                                                            (dgp_s[2 * C + t] + dgp_s[3 * C + t]));
      }
    }
    if (!cur) {
      nproc = m;
      break;
    }
    if (!q_early) {  // G of the previous chunk has left X (read by the pairwise sums)
      fence_proxy_async();
      epi_sync();
      if (tid == 160) load_q(m);
    }
    const int b = bh / a.H, h = bh % a.H;
    const size_t row0 = ((size_t)b * a.T + (size_t)n * C) * a.H + h;
    cur_n = n;
    cur_bh = bh;
    if (tid < C) beta_s[tid] = beta_pre;
    epi_sync();
    // (c) E1: dv = beta Y, dbeta_v = rowsum(Y * V), Y into the lower half of DY.
    // Thread: value column v = rowl, tokens t_beg .. + TPT - 1.
    {
      const int v = rowl;
      Tile<bf16, C, BD> Vt{reinterpret_cast<bf16*>(sm + L::VT)};
      mbar_wait(bP1, par, a.err);  // P1 was issued after group A (v included) had landed
      tc_fence_after();
      uint32_t y[TPT];
      tmem_ld16_nowait(tl + TC_P1 + t_beg, y);
      tmem_wait_ld();
      float pv[TPT];
#pragma unroll
      for (int i = 0; i < TPT; ++i) {
        const int t = t_beg + i;
        const size_t gi = (row0 + (size_t)t * rs) * BD + v;
        const float yf = u2f(y[i]);
        static_cast<bf16*>(a.dv)[gi] = __float2bfloat16_rn(beta_s[t] * yf);
        pv[i] = yf * __bfloat162float(Vt.at(t, v));
        DYt.at(C + t, v) = __float2bfloat16_rn(yf);
      }
      const float p = warp_sum16(pv, lane);
      if ((lane & 1) == 0) dbv_s[qw * C + t_beg + (lane >> 1)] = p;
    }
    if (fused && tid == 0) {  // before the barrier that precedes the first load of step m + 1
      units_s[(m + 1) & 3] = (int)pend0;
      pend0 = pend1;
    }
    fence_proxy_async();  // the Y rows are read by the tensor cores
    tc_fence_before();
    epi_sync();
    // (d) P2, P3, P4; P1 has read T and dU^T: the next chunk's group A loads
    if (tid == 128 && valid(m + 1)) load_a(m + 1);
    if (tid == 0) {
      mbar_wait(fullB, par, a.err);
      tc_fence_after();
      {  // P2: D2 = DY U^T (M = 2C tokens, N = C, K = Dv)
        const uint64_t dA = desc_kmajor(sm + L::DY), dB = desc_mnmajor(sm + L::UT, BD * 128);
#pragma unroll
        for (int ks = 0; ks < BD / 16; ++ks)
          umma_bf16(tm + TC_P2, kstep_kmajor(dA, ks, 2 * C * 128), kstep_mnmajor(dB, ks), id_p2, ks > 0);
        umma_commit(bP2);
      }
    } else if (tid == 32) {  // P3 and P4 from two more warps: each issue stall is per thread
      mbar_wait(fullB, par, a.err);
      tc_fence_after();
      {  // P3: D3 = S0 DY^T (M = Dk, N = 2C, K = Dv)
        const uint64_t dA = desc_mnmajor(sm + L::S0T, BD * 128), dB = desc_kmajor(sm + L::DY);
#pragma unroll
        for (int ks = 0; ks < BD / 16; ++ks)
          umma_bf16(tm + TC_D3, kstep_mnmajor(dA, ks), kstep_kmajor(dB, ks, 2 * C * 128), id_p3, ks > 0);
      }
      umma_commit(bP34);
    } else if (tid == 64) {
      mbar_wait(fullB, par, a.err);
      tc_fence_after();
      {  // P4: D4 = dS1 U^T (M = Dk, N = C, K = Dv)
        const uint64_t dA = desc_mnmajor(sm + L::DS1T, BD * 128), dB = desc_mnmajor(sm + L::UT, BD * 128);
#pragma unroll
        for (int ks = 0; ks < BD / 16; ++ks)
          umma_bf16(tm + TC_D4, kstep_mnmajor(dA, ks), kstep_mnmajor(dB, ks), id_p4, ks > 0);
      }
      umma_commit(bP34);
    }
    // (e) dgam partials, G, the score operands. Thread: channel c = rowl, tokens
    // t_beg .. + TPT - 1 (value rows 2 TPT tg .. for dgam).
    const int c = rowl;
    const bf16* graw = reinterpret_cast<const bf16*>(sm + L::YE);  // per-channel g [C][Dk]
    float gl[TPT];
    if (!PC) {
#pragma unroll
      for (int i = 0; i < TPT; ++i) gl[i] = ldg_bf16(gg + row0 + (size_t)(t_beg + i) * rs);
    }
    mbar_wait(fullQ, par, a.err);
    float qb[TPT], kb[TPT];  // the build's q and k (X is rewritten in place below)
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      qb[i] = __bfloat162float(Xt.at(t_beg + i, c));
      kb[i] = __bfloat162float(Xt.at(C + t_beg + i, c));
      if (PC) gl[i] = __bfloat162float(graw[(t_beg + i) * BD + c]);
    }
    {  // this group's part of the inclusive cumulative log-decay of channel c
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < TPT; ++i) {
        s += gl[i];
        Greg[i] = s;
      }
      gx_s[tg * BD + c] = s;
    }
    mbar_wait(fullB, par, a.err);
    {  // dgam_c = sum_v dS1[c][v] S0[c][v]: warp w takes channels 8 w .. + 7 (one 16-byte
       // piece of a row of S0^T and dS1^T), lane l rows l + 32 i; then a warp sum
      typedef Sw<bf16, BD, BD> SL;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < BD / 32; ++i) {
        const int off = SL::off(lane + 32 * i, 8 * warp);
        const uint4 s4 = *reinterpret_cast<const uint4*>(S0T + off);
        const uint4 d4 = *reinterpret_cast<const uint4*>(DS1T + off);
        const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w}, dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 sf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sw[e]));
          const float2 df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[e]));
          acc[2 * e] = fmaf(df.x, sf.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(df.y, sf.y, acc[2 * e + 1]);
        }
      }
      const float tot = warp_sum8(acc, lane);
      if ((lane & 3) == 0) dgam_s[8 * warp + (lane >> 2)] = tot;
    }
    if (tid == 0) {
      flags_s[0] = 0;
      flags_s[1] = 0;
    }
    epi_sync();
    {  // the earlier groups' totals, added left to right (G_b after group 1, G_C after 3)
      float p = 0.f, pre = 0.f;
#pragma unroll
      for (int g2 = 0; g2 < NTG; ++g2) {
        if (g2 == tg) pre = p;
        p += gx_s[g2 * BD + c];
        if (g2 == 1) Gb = p;
      }
      GC = p;
#pragma unroll
      for (int i = 0; i < TPT; ++i) Greg[i] += pre;
    }
    if (!PC && c == 0) {
#pragma unroll
      for (int i = 0; i < TPT; ++i) gsc[t_beg + i] = Greg[i];
    }
    // block spreads: exp(G - G_b) of the first block's rows and exp(G_b - G) of the
    // second's must stay in range
    if (PC) {
      if (tg == 0 && !(Greg[0] - Gb <= SAFE_SPREAD)) flags_s[0] = 1;
      if (tg == NTG - 1 && !(Gb - Greg[TPT - 1] <= SAFE_SPREAD)) flags_s[1] = 1;
    }
    if (force && tid == 0) {
      flags_s[0] = 1;
      flags_s[1] = 1;
    }
    epi_sync();
    // E2: the score-gradient tile [dAqk ; dAkk] from D2. Thread: row t' = rowl, columns
    // t_beg .. + TPT - 1.
    mbar_wait(bP2, par, a.err);
    tc_fence_after();
    {
      uint32_t d[TPT];
      tmem_ld16_nowait(tl + TC_P2 + t_beg, d);
      tmem_wait_ld();
      const int tp = rowl, t = tp & (C - 1);
      const bool akk = tp >= C;
      const float Gt = mask_form ? gsc[t] : 0.f;
      float o[TPT];
#pragma unroll
      for (int jj = 0; jj < TPT; ++jj) {
        const int j = t_beg + jj;
        float x;
        if (!akk) {
          x = j <= t ? a.scale * u2f(d[jj]) : 0.f;
          if (j == t) {
            diag_s[t] = x;  // the diagonal only feeds dq and dk directly
            x = 0.f;
          }
        } else {
          x = j < t ? -u2f(d[jj]) : 0.f;
        }
        if (mask_form && j < t) x *= __expf(Gt - gsc[j]);
        o[jj] = x;
      }
#pragma unroll
      for (int q2 = 0; q2 < TPT / 8; ++q2) {
        uint4 u;
        u.x = pack2_bf16(o[8 * q2 + 0], o[8 * q2 + 1]);
        u.y = pack2_bf16(o[8 * q2 + 2], o[8 * q2 + 3]);
        u.z = pack2_bf16(o[8 * q2 + 4], o[8 * q2 + 5]);
        u.w = pack2_bf16(o[8 * q2 + 6], o[8 * q2 + 7]);
        *reinterpret_cast<uint4*>(DPt.ptr(tp, t_beg + 8 * q2)) = u;
      }
    }
    tc_fence_before();  // D2 has been read: its columns take the q, k stash below
    epi_sync();
    {
      const bool unsafe1 = flags_s[0] != 0, unsafe2 = flags_s[1] != 0;
      const bool dead_x = !mask_form && blk == 0 && unsafe1;
      const bool dead_y = !mask_form && blk == 1 && unsafe2;
      // row c of X^T and Ye^T: this thread's tokens in 16-byte pieces of eight
#pragma unroll
      for (int h8 = 0; h8 < TPT / 8; ++h8) {
        float xq[8], xk[8], ye[8];
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          const int i = 8 * h8 + ii, t = t_beg + i;
          const float d = Greg[i] - Gb;
          const float e1 = mask_form ? 1.f : dead_x ? 0.f : __expf(d);
          const float e2 = mask_form ? 1.f : dead_y ? 0.f : __expf(-d);
          xq[ii] = qb[i] * e1;
          xk[ii] = beta_s[t] * kb[i] * e1;
          ye[ii] = kb[i] * e2;
        }
        *reinterpret_cast<uint4*>(XTt.ptr(c, t_beg + 8 * h8)) = pack8_bf16(xq);
        *reinterpret_cast<uint4*>(XTt.ptr(c, C + t_beg + 8 * h8)) = pack8_bf16(xk);
        *reinterpret_cast<uint4*>(YeTt.ptr(c, t_beg + 8 * h8)) = pack8_bf16(ye);
      }
      uint32_t qk[TPT];  // q and k of this channel and token group for the final epilogue
#pragma unroll
      for (int i = 0; i < TPT; ++i) qk[i] = pack2_bf16(qb[i], kb[i]);
      tmem_st16(tl + TC_QK + t_beg, qk);
      tmem_wait_st();
    }
    fence_proxy_async();  // X, Ye and the score-gradient tile are read by the tensor cores
    tc_fence_before();
    epi_sync();
    if (tid == 32 && valid(m + 1)) {
      // P2-P4 and the gamma-gradient sums have read dO, U^T, S0^T and dS1^T: the next
      // chunk's group B loads (the Y rows of DY are written after this chunk's final
      // epilogue, which waits for P3)
      mbar_wait(bP34, par, a.err);
      load_b(m + 1);
    }
    if (tid == 64) {
      tc_fence_after();
      {  // P5: D5 = Ye^T DP^T (M = Dk, N = 2C, K = C)
        const uint64_t dA = desc_kmajor(sm + L::YE), dB = desc_kmajor(sm + L::DP);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks)
          umma_bf16(tm + TC_D5, kstep_kmajor(dA, ks, BD * 128), kstep_kmajor(dB, ks, 2 * C * 128), id_p5, ks > 0);
      }
      umma_commit(bP56);
    } else if (tid == 96) {
      tc_fence_after();
      {  // P6: D6 = X^T DP (M = Dk, N = C, K = 2C)
        const uint64_t dA = desc_kmajor(sm + L::X), dB = desc_mnmajor(sm + L::DP, 2 * C * 128);
#pragma unroll
        for (int ks = 0; ks < 2 * C / 16; ++ks)
          umma_bf16(tm + TC_D6, kstep_kmajor(dA, ks, BD * 128), kstep_mnmajor(dB, ks), id_p6, ks > 0);
      }
      umma_commit(bP56);
    }
  }
  // every MMA and load this CTA issued has completed before TMEM is freed and the CTA
  // retires (in normal operation all were waited for; after a failed wait maybe not)
  if (tid == 0) {
    if (nproc > 0) {
      const uint32_t lp = (uint32_t)(nproc - 1) & 1u;
      mbar_drain(fullA, lp);
      mbar_drain(fullB, lp);
      mbar_drain(fullQ, lp);
    }
  }
  if (tid == 0 || tid == 32 || tid == 64 || tid == 96) {  // each issuing thread's products
    umma_commit(bDrain);
    mbar_drain(bDrain, 0u);
  }
  tc_fence_before();
  epi_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, BT_TMEM_COLS);
}

// Zeroes the fused launch's counters. Launched without programmatic serialisation, so it
// starts after every earlier kernel of the stream has finished with them (a previous
// backward call on the same workspace included); it lets the fused launch be scheduled at
// once, whose griddepcontrol.wait then waits for the zeros. A kernel rather than a memset:
// a memset may queue on a copy engine behind the caller's host copies.
__global__ void chunk_bwd_sync_zero_kernel(unsigned* p, int n) {
  pdl_trigger();
  for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0u;
}

}  // namespace

bool bwd_tc_applies(int DK, int DV) { return DK == BD && DV == BD; }

cudaError_t launch_chunk_bwd_tc(const ChunkBwdArgs& a, cudaStream_t s, bool grads_only) {
  if (a.T / C == 0) return grads_only ? cudaSuccess : launch_scan_bwd_tc(a, s);  // dh0 = dh_final only
  if ((long long)a.B * a.T > 0x7fffffffLL) return cudaErrorInvalidValue;  // TMA token coordinate
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[3] = {(cuuint64_t)BD, (cuuint64_t)a.H, (cuuint64_t)a.B * a.T};
  const cuuint64_t strides[2] = {(cuuint64_t)BD * 2, (cuuint64_t)a.H * BD * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint32_t gbox[3] = {BD, 1, (cuuint32_t)C};  // per-channel g: whole rows, row-major
  // dout, v, q, k [B*T][H][128] (same geometry), g [B*T][H][Dk] when per channel
  CUtensorMap vmap, qmap, kmap, gmap;
  auto enc = [&](CUtensorMap* m, const void* p, const cuuint32_t* bx, CUtensorMapSwizzle sw) {
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p), dims, strides, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  if (!enc(&map, a.dout, box, CU_TENSOR_MAP_SWIZZLE_128B) || !enc(&vmap, a.v, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !enc(&qmap, a.q, box, CU_TENSOR_MAP_SWIZZLE_128B) || !enc(&kmap, a.k, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (a.per_channel) {
    if (!enc(&gmap, a.g, gbox, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
  } else {
    gmap = qmap;  // not read: one decay per token arrives by plain loads
  }
  const int bytes = BtLayout::BYTES + 1024;
  auto kern = a.per_channel ? chunk_bwd_tc_kernel<true> : chunk_bwd_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0, coop = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) return e;
  const int BH = a.B * a.H, units = (a.T / C) * BH;
  // Fewer (batch, head) pairs than SMs: one cooperative grid of one CTA per SM (the shared
  // memory admits one), so every wait of a gradient CTA has the scan CTA it waits for
  // resident. The counters start from zero on every call (chunk_bwd_sync_zero_kernel).
  const bool fused = coop && BH < nsm && units > 0 && a.ws.sync && a.ws.sync_bytes > 0;
  auto two_launches = [&]() {  // the reverse scan, then the gradients over a static stride
    cudaError_t e2;
    if (!grads_only && (e2 = launch_scan_bwd_tc(a, s)) != cudaSuccess) return e2;
    const int grid = units < nsm ? units : nsm;
    if (grid == 0) return cudaSuccess;
    prof_mark(K_BWD_TC, s, true);
    e2 = launch_pdl(kern, dim3(grid), dim3(BT_THREADS), bytes, s, a, map, vmap, qmap, kmap, gmap,
                    BwdSync{nullptr, nullptr, 0});
    prof_mark(K_BWD_TC, s, false);
    return e2;
  };
  if (!fused || grads_only) return two_launches();
  prof_mark(K_BWD_SYNC, s, true);
  chunk_bwd_sync_zero_kernel<<<1, 256, 0, s>>>(a.ws.sync, (int)(a.ws.sync_bytes / 4));
  prof_mark(K_BWD_SYNC, s, false);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  BwdSync sync{a.ws.sync, a.ws.sync + (size_t)BH * PROGRESS_STRIDE, BH};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsm);
  cfg.blockDim = dim3(BT_THREADS);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  prof_mark(K_BWD_TC, s, true);
  e = cudaLaunchKernelEx(&cfg, kern, a, map, vmap, qmap, kmap, gmap, sync);
  prof_mark(K_BWD_TC, s, false);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    // the context cannot keep a CTA on every SM at once (an SM-limited partition)
    (void)cudaGetLastError();
    return two_launches();
  }
  return e;
}

}  // namespace gdn
