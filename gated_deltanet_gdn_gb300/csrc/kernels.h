// Internal launch interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

constexpr int C = 64;       // chunk length (tokens)
constexpr int BLK = 32;     // block length inside a chunk
constexpr int C2 = 128;     // chunk length with FLAG_CHUNK128: two 64-token blocks
constexpr int NT = 32;      // value columns per warp column group of the mma.sync scans
constexpr int NTS = 64;     // value columns per state-scan CTA (two record slices)
constexpr float SAFE_SPREAD = 80.f;  // max decay spread (nats) for row-scaled in-block scores
constexpr int FLAG_PAIRWISE = 1;     // dims.flags bit: in-block scores always pairwise
constexpr int FLAG_CHUNK128 = 4;     // dims.flags bit: the forward works on 128-token chunks
// the forward scan's chunk counters, one per (batch, head), each on its own 128-byte line
// (counter bh at progress[bh * PROGRESS_STRIDE])
constexpr int PROGRESS_STRIDE = 32;

// Per (batch, head) and chunk, the forward writes these records. Byte sizes of one record
// for operand element size es; every record starts 1024-byte aligned inside its region.
// Each record is a swizzled tile (Sw in common.cuh): Aqk, T [C][C]; -W, Q-hat, K-tilde
// [C][Dk]; U', the chunk-start state and U transposed: U'^T [Dv][C],
// S^T [Dv][Dk] and U^T [Dv][C]. The backward's dS and dU records are likewise
// dS^T [Dv][Dk] and dU^T [Dv][C].
struct ResidualLayout {
  // region base offsets in bytes from the residual pointer (qn, kn, qinv, kinv: only with
  // the q/k L2 normalisation, the normalised rows and their inverse norms; progress: one
  // counter per (batch, head) through which the tensor-core forward scan tells the output
  // CTAs beside it how many chunks' records are stored)
  size_t aqk, tmat, wneg, up, qh, kt, gam, state, u, progress, qn, kn, qinv, kinv, total;
  // bytes of one chunk-head record
  size_t aqk_b, tmat_b, w_b, up_b, qh_b, kt_b, gam_b, state_b, u_b;
  // with 128-token chunks: the 128-token records (merged from the 64-token blocks' aqk,
  // wneg, up, qh, kt and gam above; state and u of the 128-token chunks), same forms with
  // C2 in place of C; the 64-token state and u records are then written by the backward
  size_t aqk2, wneg2, up2, qh2, kt2, gam2, state2, u2;
};

struct BwdWorkspaceLayout {
  // sync (bf16 with Dk = Dv = 128 only): the fused backward launch's counters, sync_bytes
  // bytes, zeroed before each launch: one per (batch, head) on its own 128-byte line (chunks
  // the reverse scan has finished), then the work queue's next unit on a line of its own
  size_t du, dstate, sync, dqh, dbk, dkt, daqk, dakk, dgam, dbv, dbpart, dgpart, total;
  size_t du_b, dstate_b, sync_bytes, dqh_b, dbk_b, dkt_b, daqk_b, dakk_b, dgam_b, dbv_b, dbpart_b, dgpart_b;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline ResidualLayout residual_layout(int B, int T, int H, int DK, int DV, int es, bool qk_norm = false,
                                      bool chunk128 = false) {
  ResidualLayout L{};
  const size_t n = (size_t)B * H * (T / C);
  L.aqk_b = (size_t)C * C * es;
  L.tmat_b = (size_t)C * C * es;
  L.w_b = (size_t)C * DK * es;
  L.up_b = (size_t)C * DV * es;
  L.qh_b = (size_t)C * DK * es;
  L.kt_b = (size_t)C * DK * es;
  L.gam_b = (size_t)DK * 4;
  L.state_b = (size_t)DK * DV * es;
  L.u_b = (size_t)C * DV * es;
  size_t off = 0;
  auto put = [&](size_t& field, size_t rec) {
    field = off;
    off = align_up(off + rec * n, 1024);
  };
  put(L.aqk, L.aqk_b);
  put(L.tmat, L.tmat_b);  // written by the preparation; read by the backward only
  put(L.wneg, L.w_b);
  put(L.up, L.up_b);
  put(L.qh, L.qh_b);
  put(L.kt, L.kt_b);
  put(L.gam, L.gam_b);
  put(L.state, L.state_b);  // with 128-token chunks: formed by the backward, per 64-token block
  put(L.u, L.u_b);
  if (chunk128) {
    const size_t n2 = n / 2;
    auto put2 = [&](size_t& field, size_t rec) {
      field = off;
      off = align_up(off + rec * n2, 1024);
    };
    put2(L.aqk2, (size_t)C2 * C2 * es);
    put2(L.wneg2, (size_t)C2 * DK * es);
    put2(L.up2, (size_t)C2 * DV * es);
    put2(L.qh2, (size_t)C2 * DK * es);
    put2(L.kt2, (size_t)C2 * DK * es);
    put2(L.gam2, (size_t)DK * 4);
    put2(L.state2, L.state_b);
    put2(L.u2, (size_t)C2 * DV * es);
  }
  L.progress = off;
  off = align_up(off + (size_t)B * H * PROGRESS_STRIDE * 4, 1024);
  if (qk_norm) {
    const size_t rows = (size_t)B * T * H;
    L.qn = off;
    off = align_up(off + (size_t)DK * es * rows, 1024);
    L.kn = off;
    off = align_up(off + (size_t)DK * es * rows, 1024);
    L.qinv = off;
    off = align_up(off + rows * 4, 1024);
    L.kinv = off;
    off = align_up(off + rows * 4, 1024);
  }
  L.total = off;
  return L;
}

inline BwdWorkspaceLayout bwd_workspace_layout(int B, int T, int H, int DK, int DV, int es) {
  BwdWorkspaceLayout L{};
  const size_t n = (size_t)B * H * (T / C);
  L.du_b = (size_t)C * DV * es;
  L.dstate_b = (size_t)DK * DV * es;
  L.dqh_b = (size_t)C * DK * es;
  L.dbk_b = (size_t)C * DK * es;
  L.dkt_b = (size_t)C * DK * es;
  L.daqk_b = (size_t)C * C * es;
  L.dakk_b = (size_t)C * C * es;
  L.dgam_b = (size_t)DK * 4;
  L.dbv_b = (size_t)C * 4;
  L.dbpart_b = (size_t)2 * C * 4;
  L.dgpart_b = (size_t)2 * C * 4;
  size_t off = 0;
  auto put = [&](size_t& field, size_t rec) {
    field = off;
    off = align_up(off + rec * n, 1024);
  };
  put(L.du, L.du_b);
  put(L.dstate, L.dstate_b);
  // bf16 with Dk = Dv = 128 runs the fused chunk-gradient kernel (chunk_bwd_tc.cu), which
  // needs only dU and dS from the reverse scan; the other regions serve the CUDA-core
  // kernels (Dk = 64, or fp32 operands)
  if (es == 2 && DK == 128 && DV == 128) {
    L.sync_bytes = (size_t)B * H * PROGRESS_STRIDE * 4 + 128;
    L.sync = off;
    off = align_up(off + L.sync_bytes, 1024);
    L.total = off;
    return L;
  }
  put(L.dqh, L.dqh_b);
  put(L.dbk, L.dbk_b);
  put(L.dkt, L.dkt_b);
  put(L.daqk, L.daqk_b);
  put(L.dakk, L.dakk_b);
  put(L.dgam, L.dgam_b);
  put(L.dbv, L.dbv_b);
  put(L.dbpart, L.dbpart_b);
  put(L.dgpart, L.dgpart_b);
  L.total = off;
  return L;
}

// Pointers into the residual buffer, resolved on the host.
struct ResidualPtrs {
  void *aqk, *tmat, *wneg, *up, *qh, *kt;
  float* gam;
  void *state, *u;
  unsigned* progress;  // [B*H][PROGRESS_STRIDE]: chunks whose state and U records the forward scan has stored
  void *qn, *kn;  // normalised q, k rows (q/k L2 normalisation only)
  float *qinv, *kinv;
};
// The 128-token chunks' records (FLAG_CHUNK128 only).
struct Residual128Ptrs {
  void *aqk, *wneg, *up, *qh, *kt;
  float* gam;
  void *state, *u;
};
struct BwdWorkspacePtrs {
  void *du, *dstate, *dqh, *dbk, *dkt, *daqk, *dakk;
  float *dgam, *dbv, *dbpart, *dgpart;
  unsigned* sync;     // [B*H][PROGRESS_STRIDE] then the queue line (bf16, Dk = Dv = 128)
  size_t sync_bytes;  // 0 when the layout has no sync region
};

struct ChunkFwdArgs {
  int B, T, H, DK, DV, per_channel, bf16, flags;
  const void *q, *k, *v, *g, *beta;
  const float* h0;
  float scale;
  void* out;
  float* h_final;
  ResidualPtrs res;
  Residual128Ptrs res2;  // FLAG_CHUNK128: the 128-token records
  unsigned* err;
};

struct ChunkBwdArgs {
  int B, T, H, DK, DV, per_channel, bf16, flags;
  const void *q, *k, *v, *g, *beta;
  float scale;
  ResidualPtrs res;
  Residual128Ptrs res2;  // FLAG_CHUNK128: the 128-token records
  const void* dout;
  const float* dh_final;
  void *dq, *dk, *dv, *dg, *dbeta;
  float* dh0;
  BwdWorkspacePtrs ws;
  unsigned* err;
};

struct RecurrentArgs {
  int B, T, H, DK, DV, per_channel, bf16, qk_norm;
  const void *q, *k, *v, *g, *beta;
  const float* h0;
  float scale;
  void* out;
  float* h_final;
  unsigned* err;
};

// Replay decode (replay.cu): checkpoint [B,H,DK,DV] fp32, buffer [B,H,L][2 DK + DV] fp32
// slots (k, cumulative log-decay G, delta d), fill [B,H] slots in use.
constexpr int REPLAY_MAX_TOKENS = 8;
struct ReplayArgs {
  int B, H, DK, DV, L, per_channel, bf16, qk_norm;
  const void *q, *k, *v, *g, *beta;
  float scale;
  float* ckpt;
  float* buffer;
  int* fill;
  void* out;
  unsigned* err;
};
struct ReplayStateArgs {
  int B, H, DK, DV, L;
  const float* ckpt;
  const float* buffer;
  const int* fill;
  float* h_out;
  unsigned* err;
};

// Kernel identifiers for the optional per-launch timing (gdn_profile_* in the C ABI).
enum KernelId {
  K_PREP = 0,      // chunk_prep_kernel
  K_SCAN_FWD = 1,  // chunk_scan_fwd_kernel
  K_SCAN_BWD = 2,  // chunk_scan_bwd_kernel
  K_DSTATE = 3,    // chunk_dstate_kernel
  K_GRADS = 4,     // chunk_grads_kernel
  K_RECURRENT = 5, // recurrent_kernel
  K_FINALIZE = 6,  // chunk_bwd_finalize_kernel
  K_OUT = 7,       // chunk_out_kernel
  K_SCAN_FWD_TC = 8,  // chunk_scan_fwd_tc_kernel
  K_SCAN_BWD_TC = 9,  // chunk_scan_bwd_tc_kernel
  K_DECODE = 10,      // decode_kernel
  K_L2NORM = 11,      // l2norm_rows_kernel
  K_L2NORM_BWD = 12,  // l2norm_bwd_kernel
  K_REPLAY = 13,      // replay_decode_kernel
  K_REPLAY_STATE = 14,  // replay_state_kernel
  K_DQA = 15,           // chunk_dqa_kernel (Dk = 64 path)
  K_BWD_TC = 16,        // chunk_bwd_tc_kernel: every chunk product of the backward, fused, tcgen05
  K_PREP_TC = 17,       // chunk_prep_tc_kernel: the chunk preparation on tcgen05
  K_BWD_SYNC = 18,      // chunk_bwd_sync_zero_kernel: zeroes the fused backward's counters
  K_MERGE = 19,         // chunk_merge128_kernel: two 64-token blocks -> one 128-token chunk
  K_MID = 20,           // chunk_mid128_kernel: the 64-token blocks' dU, dS1, states and U
  K_COUNT = 21
};
// Records a CUDA event on s before (begin = true) or after a launch when timing is on.
void prof_mark(KernelId id, cudaStream_t s, bool begin);

// Each returns a cudaError_t from the launches (cudaSuccess when all were accepted).
cudaError_t launch_chunk_fwd(const ChunkFwdArgs& a, cudaStream_t s);
cudaError_t launch_chunk_bwd(const ChunkBwdArgs& a, cudaStream_t s);
cudaError_t launch_recurrent(const RecurrentArgs& a, cudaStream_t s);
cudaError_t launch_chunk_grads(const ChunkBwdArgs& a, cudaStream_t s);  // part of launch_chunk_bwd
// The tensor-core (tcgen05) state scans, used when scan_tc_applies(bf16, Dk, Dv).
bool scan_tc_applies(int bf16_operands, int DK, int DV);
// outputs_done: the launch also formed every chunk's outputs (output CTAs beside the scan)
cudaError_t launch_scan_fwd_tc(const ChunkFwdArgs& a, cudaStream_t s, bool* outputs_done);
cudaError_t launch_scan_bwd_tc(const ChunkBwdArgs& a, cudaStream_t s);
// The chunk preparation on tcgen05 (chunk_prep_tc.cu), bf16 operands with Dk = Dv = 128.
bool prep_tc_applies(int bf16_operands, int DK, int DV);
cudaError_t launch_chunk_prep_tc(const ChunkFwdArgs& a, cudaStream_t s);
// The merge of each pair of 64-token blocks' records into one 128-token chunk's records
// (chunk_merge.cu), FLAG_CHUNK128 only.
cudaError_t launch_chunk_merge128(const ChunkFwdArgs& a, cudaStream_t s);
// The backward of bf16 with Dk = Dv = 128 on tcgen05 (chunk_bwd_tc.cu): the reverse scan and
// the fused chunk-gradient kernel, as one cooperative launch when the (batch, head) pairs
// leave SMs free (the gradient CTAs take each chunk as soon as the scan has finished it),
// else as two launches; it needs only the du, dstate and sync parts of the workspace.
bool bwd_tc_applies(int DK, int DV);
// grads_only: the chunk gradients alone, over a static stride, from dU and dS1 records that
// are already in the workspace (the backward over 128-token chunks forms them first)
cudaError_t launch_chunk_bwd_tc(const ChunkBwdArgs& a, cudaStream_t s, bool grads_only = false);
// cuTensorMapEncodeTiled through the runtime's driver entry point, resolved once (NULL if
// the driver does not provide it); callers cast it to PFN_cuTensorMapEncodeTiled_v12000.
void* tensor_map_encode_fn();
// The single-token decode kernel (decode.cu), used by launch_recurrent when T == 1.
cudaError_t launch_decode(const RecurrentArgs& a, cudaStream_t s);
// q/k L2 normalisation for the chunked path (l2norm.cu): rows = B * T * H.
cudaError_t launch_l2norm_rows(const void* q, const void* k, void* qn, void* kn, float* qinv, float* kinv,
                               size_t rows, int DK, int bf16, cudaStream_t s);
cudaError_t launch_l2norm_bwd(void* dq, void* dk, const void* qn, const void* kn, const float* qinv,
                              const float* kinv, size_t rows, int DK, int bf16, cudaStream_t s);
// Replay decode (replay.cu): one token per (batch, head) against checkpoint + buffer,
// and the fold of a buffer into a full state.
cudaError_t launch_replay_decode(const ReplayArgs& a, cudaStream_t s);
cudaError_t launch_replay_state(const ReplayStateArgs& a, cudaStream_t s);

}  // namespace gdn
