// Device helpers shared by the gated delta rule kernels (sm_103a).
//
//  * element types: the "operand type" T of a kernel is __nv_bfloat16 (bf16 inputs,
//    fp32 state / accumulation) or float (fp32 everything; tensor-core products use
//    a three-term TF32 split so that they keep ~fp32 accuracy);
//  * swizzled shared-memory tiles whose byte layout equals what a TMA copy with the
//    matching swizzle mode writes, so a tile can be filled by a bulk copy of an image
//    written in the same layout;
//  * warp-level tensor-core products (mma.sync m16n8k16 bf16, m16n8k8 tf32x3) on
//    those tiles, with either operand read as stored or transposed;
//  * bulk async copies (cp.async.bulk) completing on an mbarrier, with bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

typedef __nv_bfloat16 bf16;

// ------------------------------------------------------------------ conversions
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <class T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Compile-time flag for generic lambdas that are specialised on a condition.
template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

// q/k L2 normalisation: the guard added to the sum of squares.
constexpr float QK_NORM_EPS = 1e-6f;

// V consecutive elements (V = 2 or 4) as floats with one vector load; p aligned to V
// elements.
template <int V>
__device__ __forceinline__ void load_vec(const float* p, float (&x)[V]) {
  static_assert(V == 2 || V == 4, "two or four elements");
  if constexpr (V == 4) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
  } else {
    const float2 u = *reinterpret_cast<const float2*>(p);
    x[0] = u.x; x[1] = u.y;
  }
}
template <int V>
__device__ __forceinline__ void load_vec(const bf16* p, float (&x)[V]) {
  static_assert(V == 2 || V == 4, "two or four elements");
  if constexpr (V == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    x[0] = a.x; x[1] = a.y;
  }
}

// Inverse L2 norm 1 / sqrt(sum_c x_c^2 + QK_NORM_EPS) of a row x[0 .. N-1] (N = 64 or
// 128), read by one full warp: lane l takes the N/32 consecutive elements from
// l N/32 and sums their squares in ascending order with fmaf, then the lanes are
// added by a butterfly (xor 16, 8, 4, 2, 1). Every kernel that normalises q or k uses
// this one definition, so they agree bitwise.
template <int N, class T>
__device__ __forceinline__ float warp_row_inv_norm(const T* x, int lane) {
  constexpr int V = N / 32;
  float v[V];
  load_vec<V>(x + V * lane, v);
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < V; ++j) s = fmaf(v[j], v[j], s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return rsqrtf(s + QK_NORM_EPS);
}

// ------------------------------------------------------------------ swizzled tiles
// A ROWS x COLS tile of T stored as column panels of 128 bytes (fewer when a row is
// shorter). Inside a panel, row r occupies PANB bytes and the 16-byte chunk index is
// XORed with (r / rows-per-128B) like the TMA SWIZZLE_{128,64,32}B modes. Eight
// consecutive rows at the same logical 16-byte chunk land in eight different bank
// groups, so ldmatrix reads are conflict free. Tiles must start 1024-byte aligned.
template <class T, int ROWS, int COLS>
struct Sw {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int ROWB = COLS * ES;
  static constexpr int PANB = ROWB >= 128 ? 128 : ROWB;
  static constexpr int PW = PANB / ES;  // panel width in elements
  static constexpr int ELEMS = ROWS * COLS;
  static constexpr int BYTES = ELEMS * ES;
  static_assert(PANB == 128 || PANB == 64 || PANB == 32, "tile row must be 32, 64 or >=128 bytes");
  static_assert(COLS % PW == 0, "whole panels only");
  __device__ __host__ static __forceinline__ int off(int r, int c) {
    const int panel = c / PW;
    int a = r * PANB + (c % PW) * ES;  // byte offset inside the panel
    if (PANB == 128) a ^= ((a >> 7) & 7) << 4;
    else if (PANB == 64) a ^= ((a >> 7) & 3) << 4;
    else a ^= ((a >> 7) & 1) << 4;
    return panel * (ROWS * PW) + a / ES;
  }
};

template <class T, int ROWS, int COLS>
struct Tile {
  T* p;
  typedef Sw<T, ROWS, COLS> L;
  __device__ __forceinline__ T& at(int r, int c) const { return p[L::off(r, c)]; }
  __device__ __forceinline__ T* ptr(int r, int c) const { return p + L::off(r, c); }
};

// A ROWS x COLS tile stored as COLS / TW consecutive ROWS x TW swizzled sub-tiles (the
// value-column slices the state scan works on).
template <class T, int ROWS, int COLS, int TW>
struct TTile {
  T* p;
  typedef Sw<T, ROWS, TW> L;
  __device__ __forceinline__ static int off(int r, int c) { return (c / TW) * (ROWS * TW) + L::off(r, c % TW); }
  __device__ __forceinline__ T& at(int r, int c) const { return p[off(r, c)]; }
  __device__ __forceinline__ T* ptr(int r, int c) const { return p + off(r, c); }
};

// Plain row-major fp32 matrix in shared memory (elementwise work, no MMA reads).
template <int ROWS, int COLS, int PAD = 0>
struct FTile {
  float* p;
  static constexpr int LD = COLS + PAD;
  static constexpr int BYTES = ROWS * LD * 4;
  __device__ __forceinline__ float& at(int r, int c) const { return p[r * LD + c]; }
};

// ------------------------------------------------------------------ ldmatrix / mma
__device__ __forceinline__ void ldsm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma_tf32(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
// x = hi + lo with hi, lo representable in tf32 (three-term split products keep
// about 21 significant bits)
__device__ __forceinline__ void tf32_split(float x, uint32_t& hi, uint32_t& lo) {
  hi = tf32_rna(x);
  lo = tf32_rna(x - __uint_as_float(hi));
}

// ------------------------------------------------------------------ operand views
// An A operand (M x K) or B operand (K x N) read from a tile either as stored
// (A: tile rows = m; B: tile rows = n, "col" operand) or transposed
// (A: tile rows = k; B: tile rows = k). r0/c0 shift the window inside the tile.
template <class TileT, bool TRANS>
struct AView {
  TileT t;
  int r0, c0;
};
template <class TileT, bool KROWS>
struct BView {
  TileT t;
  int r0, c0;
};
template <bool TRANS, class TileT>
__device__ __forceinline__ AView<TileT, TRANS> aview(TileT t, int r0 = 0, int c0 = 0) {
  return AView<TileT, TRANS>{t, r0, c0};
}
// KROWS = true: B[k][n] = tile(k, n); false: B[k][n] = tile(n, k)
template <bool KROWS, class TileT>
__device__ __forceinline__ BView<TileT, KROWS> bview(TileT t, int r0 = 0, int c0 = 0) {
  return BView<TileT, KROWS>{t, r0, c0};
}

// bf16 fragments ------------------------------------------------------------
template <class TileT>
__device__ __forceinline__ void load_a(uint32_t* a, const AView<TileT, false>& v, int m0, int k0, int lane) {
  ldsm_x4(a, v.t.ptr(v.r0 + m0 + (lane & 15), v.c0 + k0 + (lane >> 4) * 8));
}
template <class TileT>
__device__ __forceinline__ void load_a(uint32_t* a, const AView<TileT, true>& v, int m0, int k0, int lane) {
  ldsm_x4_t(a, v.t.ptr(v.r0 + k0 + (lane & 7) + (lane >> 4) * 8, v.c0 + m0 + ((lane >> 3) & 1) * 8));
}
// two n8 tiles (n0, n0 + 8): b[0..1] first, b[2..3] second
template <class TileT>
__device__ __forceinline__ void load_b2(uint32_t* b, const BView<TileT, false>& v, int n0, int k0, int lane) {
  ldsm_x4(b, v.t.ptr(v.r0 + n0 + (lane & 7) + (lane >> 4) * 8, v.c0 + k0 + ((lane >> 3) & 1) * 8));
}
template <class TileT>
__device__ __forceinline__ void load_b2(uint32_t* b, const BView<TileT, true>& v, int n0, int k0, int lane) {
  ldsm_x4_t(b, v.t.ptr(v.r0 + k0 + (lane & 7) + ((lane >> 3) & 1) * 8, v.c0 + n0 + (lane >> 4) * 8));
}
template <class TileT>
__device__ __forceinline__ void load_b1(uint32_t* b, const BView<TileT, false>& v, int n0, int k0, int lane) {
  ldsm_x2(b, v.t.ptr(v.r0 + n0 + (lane & 7), v.c0 + k0 + ((lane >> 3) & 1) * 8));
}
template <class TileT>
__device__ __forceinline__ void load_b1(uint32_t* b, const BView<TileT, true>& v, int n0, int k0, int lane) {
  ldsm_x2_t(b, v.t.ptr(v.r0 + k0 + (lane & 7) + ((lane >> 3) & 1) * 8, v.c0 + n0));
}

// fp32 (tf32x3) fragments ---------------------------------------------------
template <class TileT>
__device__ __forceinline__ float a_elem(const AView<TileT, false>& v, int m, int k) { return v.t.at(v.r0 + m, v.c0 + k); }
template <class TileT>
__device__ __forceinline__ float a_elem(const AView<TileT, true>& v, int m, int k) { return v.t.at(v.r0 + k, v.c0 + m); }
template <class TileT>
__device__ __forceinline__ float b_elem(const BView<TileT, false>& v, int k, int n) { return v.t.at(v.r0 + n, v.c0 + k); }
template <class TileT>
__device__ __forceinline__ float b_elem(const BView<TileT, true>& v, int k, int n) { return v.t.at(v.r0 + k, v.c0 + n); }

// ------------------------------------------------------------------ warp GEMM
// acc[mt][nt][0..3] += A[m0 + 16 mt .., k] * B[k, n0 + 8 nt ..] for k in [k_begin, k_end).
// Accumulator layout is the mma C fragment: element (row g or g + 8, col 2t or 2t + 1)
// with g = lane / 4, t = lane % 4. NT must be even for bf16 (pairs of n-tiles per ldmatrix).
template <int MT, int NT, class AV, class BV>
__device__ __forceinline__ void warp_gemm_bf16(float (&acc)[MT][NT][4], const AV& A, const BV& B,
                                               int m0, int n0, int k_begin, int k_end, int lane) {
  for (int k0 = k_begin; k0 < k_end; k0 += 16) {
    uint32_t a[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) load_a(a[mt], A, m0 + 16 * mt, k0, lane);
#pragma unroll
    for (int nt = 0; nt + 1 < NT; nt += 2) {
      uint32_t b[4];
      load_b2(b, B, n0 + 8 * nt, k0, lane);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mma_bf16(acc[mt][nt], a[mt], b);
        mma_bf16(acc[mt][nt + 1], a[mt], b + 2);
      }
    }
    if (NT & 1) {
      uint32_t b[2];
      load_b1(b, B, n0 + 8 * (NT - 1), k0, lane);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) mma_bf16(acc[mt][NT - 1], a[mt], b);
    }
  }
}

template <int MT, int NT, class AV, class BV>
__device__ __forceinline__ void warp_gemm_tf32x3(float (&acc)[MT][NT][4], const AV& A, const BV& B,
                                                 int m0, int n0, int k_begin, int k_end, int lane) {
  const int g = lane >> 2, t = lane & 3;
  for (int k0 = k_begin; k0 < k_end; k0 += 8) {
    uint32_t ah[MT][4], al[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int m = m0 + 16 * mt;
      tf32_split(a_elem(A, m + g, k0 + t), ah[mt][0], al[mt][0]);
      tf32_split(a_elem(A, m + g + 8, k0 + t), ah[mt][1], al[mt][1]);
      tf32_split(a_elem(A, m + g, k0 + t + 4), ah[mt][2], al[mt][2]);
      tf32_split(a_elem(A, m + g + 8, k0 + t + 4), ah[mt][3], al[mt][3]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = n0 + 8 * nt;
      uint32_t bh[2], bl[2];
      tf32_split(b_elem(B, k0 + t, n + g), bh[0], bl[0]);
      tf32_split(b_elem(B, k0 + t + 4, n + g), bh[1], bl[1]);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mma_tf32(acc[mt][nt], al[mt], bh);
        mma_tf32(acc[mt][nt], ah[mt], bl);
        mma_tf32(acc[mt][nt], ah[mt], bh);
      }
    }
  }
}

// Same products with the k range fixed at compile time: the loop unrolls, so the
// fragment loads of step k + 1 overlap the MMAs of step k.
template <int MT, int NT, int K0, int K1, class AV, class BV>
__device__ __forceinline__ void warp_gemm_bf16_k(float (&acc)[MT][NT][4], const AV& A, const BV& B, int m0,
                                                 int n0, int lane) {
#pragma unroll
  for (int k0 = K0; k0 < K1; k0 += 16) {
    uint32_t a[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) load_a(a[mt], A, m0 + 16 * mt, k0, lane);
#pragma unroll
    for (int nt = 0; nt + 1 < NT; nt += 2) {
      uint32_t b[4];
      load_b2(b, B, n0 + 8 * nt, k0, lane);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mma_bf16(acc[mt][nt], a[mt], b);
        mma_bf16(acc[mt][nt + 1], a[mt], b + 2);
      }
    }
    if (NT & 1) {
      uint32_t b[2];
      load_b1(b, B, n0 + 8 * (NT - 1), k0, lane);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) mma_bf16(acc[mt][NT - 1], a[mt], b);
    }
  }
}

template <class T> struct Gemm;
template <> struct Gemm<bf16> {
  static constexpr int KSTEP = 16;
  template <int MT, int NT, class AV, class BV>
  __device__ static __forceinline__ void run(float (&acc)[MT][NT][4], const AV& A, const BV& B, int m0,
                                             int n0, int kb, int ke, int lane) {
    warp_gemm_bf16<MT, NT>(acc, A, B, m0, n0, kb, ke, lane);
  }
  template <int MT, int NT, int K0, int K1, class AV, class BV>
  __device__ static __forceinline__ void runk(float (&acc)[MT][NT][4], const AV& A, const BV& B, int m0,
                                              int n0, int lane) {
    warp_gemm_bf16_k<MT, NT, K0, K1>(acc, A, B, m0, n0, lane);
  }
};
template <> struct Gemm<float> {
  static constexpr int KSTEP = 8;
  template <int MT, int NT, class AV, class BV>
  __device__ static __forceinline__ void run(float (&acc)[MT][NT][4], const AV& A, const BV& B, int m0,
                                             int n0, int kb, int ke, int lane) {
    warp_gemm_tf32x3<MT, NT>(acc, A, B, m0, n0, kb, ke, lane);
  }
  template <int MT, int NT, int K0, int K1, class AV, class BV>
  __device__ static __forceinline__ void runk(float (&acc)[MT][NT][4], const AV& A, const BV& B, int m0,
                                              int n0, int lane) {
    warp_gemm_tf32x3<MT, NT>(acc, A, B, m0, n0, K0, K1, lane);
  }
};

template <int MT, int NT>
__device__ __forceinline__ void zero(float (&acc)[MT][NT][4]) {
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
}

// Row / column of accumulator element e (0..3) of an m16n8 fragment.
__device__ __forceinline__ int frag_row(int lane, int e) { return (lane >> 2) + ((e >> 1) << 3); }
__device__ __forceinline__ int frag_col(int lane, int e) { return ((lane & 3) << 1) + (e & 1); }

// ------------------------------------------------------------------ bulk copies
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
// Ends an mbarrier's life: required before its shared memory is used for anything else.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// shared -> global bulk copy, completion tracked with bulk groups
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
// One box of a 3-D tiled tensor map (a CUtensorMap in kernel parameter space) at
// coordinates (c0, c1, c2) into shared memory, completing on an mbarrier
__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// all but the most recently committed bulk group have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;\n" ::: "memory");
}

// Copies rows row0 .. row0 + rows - 1 of a swizzled ROWS x COLS record tile held in
// shared memory as its own rows x COLS tile (row0 a multiple of 8, so the swizzle
// phase of every row is the same in both) to the record in global memory: one bulk
// copy per column panel. Issued by one thread.
template <class T, int ROWS, int COLS>
__device__ __forceinline__ void store_row_block(T* rec, const T* tile, int row0, int rows) {
  constexpr int PW = Sw<T, ROWS, COLS>::PW;
  for (int p = 0; p < COLS / PW; ++p)
    bulk_s2g(rec + (size_t)p * ROWS * PW + (size_t)row0 * PW, tile + (size_t)p * rows * PW,
             (uint32_t)(rows * PW * sizeof(T)));
}

__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Error word bits written by a kernel that gave up on a wait.
enum : unsigned { ERR_WAIT_TIMEOUT = 1u };

// Bounded wait on an mbarrier phase. Each try_wait already suspends for a
// hardware-defined time; 1 << 22 tries is far longer than any copy here needs.
// On time-out the error word gets ERR_WAIT_TIMEOUT and false is returned.
//
// After a time-out no result of the call is valid, and the barriers of the CTA that
// gave up no longer follow their phases, so every later wait there would also run its
// full count. Hence a wait that has already tried WAIT_BAIL_TRIES times gives up at
// once when the error word holds ERR_WAIT_TIMEOUT (set by any CTA of any kernel, until
// the host reads and clears it). Waits of normal operation end within microseconds, far
// below that count, so they never look at the word. Kernels do not leave their loops
// when a wait fails: every thread still reaches every named barrier and the loop runs
// to its end without waiting, and before a CTA frees its tensor memory or exits it
// drains what it issued (mbar_drain below).
constexpr uint32_t WAIT_MAX_TRIES = 1u << 22;
constexpr uint32_t WAIT_BAIL_TRIES = 1u << 12;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  for (uint32_t i = 0; i < WAIT_MAX_TRIES; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i >= WAIT_BAIL_TRIES && (i & 255u) == 0 && err &&
        (*reinterpret_cast<volatile unsigned*>(err) & ERR_WAIT_TIMEOUT))
      return false;
  }
  if (err) atomicOr(err, ERR_WAIT_TIMEOUT);
  return false;
}

// Counters between CTAs of one grid (the forward scan and the output CTAs beside it):
// release store / acquire load at GPU scope, and the fence that orders the bulk copies'
// global writes (async proxy) before the release.
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta(unsigned* p, unsigned v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;\n" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_cta(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}
// all but the most recently committed bulk group have completed (writes included)
__device__ __forceinline__ void bulk_wait1() { asm volatile("cp.async.bulk.wait_group 1;\n" ::: "memory"); }

// Bounded wait, by one thread, until *p >= target (a counter another CTA of the same
// cooperative grid raises with st_release_gpu): same limits and early give-up on the
// error word as mbar_wait, with a short sleep between polls.
__device__ __forceinline__ bool wait_counter(const unsigned* p, unsigned target, unsigned* err,
                                             uint32_t max_tries = WAIT_MAX_TRIES) {
  for (uint32_t i = 0; i < max_tries; ++i) {
    if (ld_acquire_gpu(p) >= target) return true;
    if (i >= WAIT_BAIL_TRIES && (i & 255u) == 0 && err &&
        (*reinterpret_cast<volatile unsigned*>(err) & ERR_WAIT_TIMEOUT))
      return false;
    __nanosleep(512);
  }
  if (err) atomicOr(err, ERR_WAIT_TIMEOUT);
  return false;
}

// Bounded wait used only to drain: the completion of copies or tensor-core operations
// this CTA issued itself, before it frees tensor memory or retires. It does not give up
// early on the error word (operations already issued complete on their own) and
// reports nothing; in normal operation the phase has completed long before.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 20); ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Producer exit: the last (up to `stages`) of the `count` loads issued on a ring of
// single-arrival barriers (load i on barrier i % stages, phase i / stages) have landed.
// In normal operation the consumers waited for them long ago; after a failed wait they
// may not have, and a CTA must not retire with copies into its shared memory in flight.
__device__ __forceinline__ void drain_ring(uint64_t* bars, int stages, int count) {
  for (int i = count > stages ? count - stages : 0; i < count; ++i)
    mbar_drain(&bars[i % stages], (uint32_t)(i / stages) & 1u);
}

// 16-byte vector copy helpers
__device__ __forceinline__ void copy16(void* dst, const void* src) {
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
}
// Two consecutive elements (4 bytes of bf16, 8 bytes of fp32) as floats.
__device__ __forceinline__ float2 ld2(const bf16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
// Four consecutive elements (8 bytes of bf16, 16 bytes of fp32) as floats.
__device__ __forceinline__ void ld4(float (&x)[4], const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  x[0] = __low2float(a); x[1] = __high2float(a); x[2] = __low2float(b); x[3] = __high2float(b);
}
// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) at p into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void ld4(float (&x)[4], const float* p) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
}
__device__ __forceinline__ void st4(bf16* p, const float (&x)[4]) {
  uint2 u;
  *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(x[0], x[1]);
  *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(x[2], x[3]);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void st4(float* p, const float (&x)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}

// ------------------------------------------------------------------ programmatic dependent launch
// The chunk kernels are launched with programmatic stream serialisation: a kernel's grid
// may be scheduled while the previous kernel in the stream is still finishing. Every such
// kernel calls pdl_wait() before it touches global memory (it returns once the previous
// grid has completed and its writes are visible). Kernels of many waves also call
// pdl_trigger() at the start, so the next kernel is scheduled while their last wave runs;
// the single-wave state scans do not, or the next kernel's CTAs would occupy the SMs the
// scans leave free for the whole scan. Both are no-ops for a grid launched without the
// attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ------------------------------------------------------------------ misc helpers
__host__ __device__ constexpr int a1k(int x) { return (x + 1023) / 1024 * 1024; }
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
// Ampere-style 16-byte asynchronous copies (used where the destination is swizzled per 16 bytes)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int NPEND>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(NPEND) : "memory");
}
__device__ __forceinline__ void store2(bf16* p, float x, float y) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x, y);
}
__device__ __forceinline__ void store2(float* p, float x, float y) {
  *reinterpret_cast<float2*>(p) = make_float2(x, y);
}

}  // namespace gdn
