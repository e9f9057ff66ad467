/*
 * gdn.h - C ABI of the GB300 (sm_103a) gated delta rule library (libgdn.so).
 *
 * The operation. For every batch b and head h the state S (Dk x Dv, fp32, row =
 * key channel) evolves token by token:
 *
 *     S   <- diag(exp(g_t)) S              per-key-channel log-decay g_t <= 0
 *     d    = beta_t (v_t - S^T k_t)         delta, scaled by the write gate
 *     S   <- S + k_t d^T                    rank-one write
 *     o_t  = scale * S^T q_t                read after the write
 *
 * Sources: "gated-deltanet" kernel card (hf kernels hub), section Method (the
 * per-token decay, read, delta, write, read, and the state carried between
 * calls in section Usage); marin.community note "factoring GDN-2 decay on TPU",
 * section Background (one decay rate per key channel; a scalar per head is the
 * special case the kernel card uses); atomic-ops 0.1.0, sections Quick start and
 * API (the (q, k, v, g, scale, h0) -> (out, h_final) training call whose
 * backward reuses forward residuals, seq_len a multiple of the chunk size).
 *
 * Layouts (contiguous, row-major):
 *   q, k              [B, T, H, Dk]
 *   v, out, dout      [B, T, H, Dv]
 *   g                 [B, T, H, Dk] if dims.g_per_channel, else [B, T, H]
 *   beta              [B, T, H]
 *   h0, h_final,
 *   dh_final, dh0     [B, H, Dk, Dv]   always float32
 *   dq, dk, dv, dg,
 *   dbeta             same shapes as q, k, v, g, beta
 * dims.dtype is the element type of q, k, v, g, beta, out, dout and of every
 * gradient: GDN_F32 (float) or GDN_BF16 (bfloat16). The state and every
 * accumulation are float32 in both cases.
 *
 * Ownership and execution. Every tensor pointer is a DEVICE pointer owned by
 * the caller; the library never allocates or frees device memory. Each call
 * only enqueues kernels on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and returns; results are ready when the stream reaches that point.
 * Every kernel of a call runs on `stream` (the library owns no stream, event or
 * lock), so calls keep no state between them and may run concurrently on
 * different streams with disjoint buffers (gdn_chunk_fwd_noalloc excepted: see
 * there). Outputs must not alias inputs, except h_final == h0 in gdn_recurrent
 * (in-place state carry).
 *
 * Errors. Arguments are validated before anything is enqueued; a failed
 * check returns a gdn_status and enqueues nothing:
 *   GDN_ERR_INVALID_ARG  NULL dims or required pointer, negative sizes, a
 *                        pointer not aligned to 16 bytes, scale not finite
 *   GDN_ERR_UNSUPPORTED  Dk or Dv not in {64, 128} (each on its own: Dk != Dv
 *                        is supported everywhere), unknown dtype,
 *                        B * H > 65535
 *   GDN_ERR_SHAPE        chunked calls with T not a multiple of 64 (128 with
 *                        GDN_FLAG_CHUNK128)
 *   GDN_ERR_CUDA         a launch was rejected (cudaGetLastError); faults that
 *                        happen later surface at the caller's next
 *                        synchronisation on the stream
 * Inputs are not clipped: non-finite values propagate like the recurrence
 * itself (the rule diverges when beta |k|^2 > 2).
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,
  GDN_ERR_UNSUPPORTED = 2,
  GDN_ERR_SHAPE = 3,
  GDN_ERR_CUDA = 4,
  GDN_ERR_INTERNAL = 5,
  GDN_ERR_SCRATCH_LIMIT = 6 /* gdn_chunk_fwd_noalloc: problem needs more than
                               GDN_NOALLOC_SCRATCH_BYTES of residual scratch */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* dims.flags bits */
/* Score tiles inside each 32-token block are always computed pairwise on CUDA
 * cores instead of from row-scaled tensor-core products (the library already
 * does so by itself for any block whose decay spread makes the row scaling
 * leave the safe exponent range). Results agree to rounding. */
#define GDN_FLAG_PAIRWISE_WITHIN_BLOCK 1
/* q and k are L2-normalised per (token, head) before the rule sees them, the
 * use_qk_l2norm option of the "gated-deltanet" kernel card (sections Usage and
 * Correctness): x / sqrt(sum_c x_c^2 + 1e-6) (the card states no guard for a
 * zero row; 1e-6 is this library's). Accepted by gdn_chunk_fwd, gdn_chunk_bwd
 * (pass the same flags as to the forward that filled the residuals: dq and dk
 * are then gradients with respect to the raw q and k) and gdn_recurrent. With
 * it the residual buffer also holds the normalised rows, so
 * gdn_chunk_residual_bytes depends on the flag. */
#define GDN_FLAG_QK_L2NORM 2
/* gdn_chunk_fwd works on 128-token chunks, each two 64-token blocks, instead
 * of 64-token chunks: the chunk of KernelConfig's bt = 2 bc (atomic-ops 0.1.0,
 * section API) with the 64-query x 64-key cross-block score tile of the
 * marin.community note "factoring GDN-2 decay on TPU" (section Approach),
 * whose factors are taken about the last token of the first block. T must be a
 * multiple of GDN_CHUNK128 (else GDN_ERR_SHAPE); gdn_chunk_residual_bytes
 * depends on the flag. gdn_chunk_bwd takes it with bf16 operands (pass the
 * flags of the forward that filled the residuals); with fp32 operands it
 * returns GDN_ERR_UNSUPPORTED and gdn_chunk_bwd_workspace_bytes 0 (one stage
 * of fp32 128-token records does not fit the reverse scan's shared memory).
 * gdn_recurrent and the replay calls ignore it. Results agree with the
 * 64-token chunking to rounding. */
#define GDN_FLAG_CHUNK128 4

typedef struct {
  int B, T, H;       /* batch, tokens, heads */
  int Dk, Dv;        /* key and value widths: 64 or 128 each */
  int g_per_channel; /* 1: g is [B,T,H,Dk]; 0: g is [B,T,H] (one decay per head) */
  int dtype;         /* gdn_dtype */
  int flags;         /* GDN_FLAG_* */
} gdn_dims;

/* Chunk size of the chunked path (tokens) and its split into two blocks;
 * GDN_CHUNK128 with GDN_FLAG_CHUNK128. */
#define GDN_CHUNK 64
#define GDN_BLOCK 32
#define GDN_CHUNK128 128

/* Bytes of the residual buffer that gdn_chunk_fwd fills and gdn_chunk_bwd
 * reads: per 64-token chunk and head, the chunk-start state, the chunk's
 * decay-weighted score tile, its WY factors and the per-token deltas. Returns 0
 * for invalid dims. The content is private to the library.
 * Source: atomic-ops 0.1.0, section API (a forward variant that returns its
 * residuals for the backward, gdn2_pallas_forward_with_residuals) and section
 * Features (the backward stages reuse forward residuals instead of recomputing
 * them); the records themselves are this library's. It plays the part of the
 * memory estimate that page's API offers (estimate_memory): the caller sizes
 * and owns the buffer. With GDN_FLAG_CHUNK128 it also holds the 128-token
 * chunks' records (the 64-token blocks' records are formed first, then
 * merged). */
size_t gdn_chunk_residual_bytes(const gdn_dims* dims);

/* Bytes of scratch that gdn_chunk_bwd needs (reverse-scan outputs and the
 * per-chunk state-gradient products). Returns 0 for invalid dims and for
 * GDN_FLAG_CHUNK128 with fp32 operands.
 * Source: atomic-ops 0.1.0, sections Features and Limitations (the backward is
 * a chain of stage kernels whose intermediate results are passed between
 * them, one of them the pairwise-decay score backward); this buffer holds what
 * this library's stages pass. Caller-owned, like the residual buffer. */
size_t gdn_chunk_bwd_workspace_bytes(const gdn_dims* dims);

/* Chunked forward (training / prefill), T a multiple of 64 (of 128 with
 * GDN_FLAG_CHUNK128).
 *   h0        initial state, NULL = zeros
 *   scale     output scale (the Python binding passes Dk^-0.5 by default)
 *   out       [B,T,H,Dv] result
 *   h_final   final state, may be NULL
 *   residuals gdn_chunk_residual_bytes(dims) bytes, REQUIRED (also for
 *             forward-only use: it holds the chunk products between kernels),
 *             256-byte aligned
 * Steps: per-chunk cumulative log-decay, boundary-split decay-factorised
 * scores (marin.community note, section Approach), the WY/UT triangular solve
 * (atomic-ops Features: chunk scores -> WY block solve -> recompute ->
 * inter-chunk scan), then the sequential state scan over chunks.
 * With bf16 operands, Dk = Dv = 128 and fewer (batch, head) pairs than SMs,
 * the scan and the chunk outputs run as one cooperative launch of one CTA per
 * SM (output CTAs beside the scan CTAs, synchronised through counters in the
 * residual buffer); it starts once every CTA can be resident at once. Where the
 * context cannot hold one CTA per SM at once (an SM-limited partition), the scan
 * and the outputs run as two launches instead. With GDN_FLAG_CHUNK128 the
 * 64-token blocks' records are formed as above, a merge kernel combines each
 * pair into the records of one 128-token chunk (the cross-block score tile and
 * the off-diagonal block of the WY inverse, T21 = -T22 A21 T11, as products),
 * and the state scan and the outputs run on the CUDA-core kernels over
 * 128-token chunks: half the sequential steps and half the chunk-start states. */
int gdn_chunk_fwd(const gdn_dims* dims, const void* q, const void* k, const void* v,
                  const void* g, const void* beta, const float* h0, float scale, void* out,
                  float* h_final, void* residuals, void* stream);

/* Chunked backward: the gradients of the training call of atomic-ops 0.1.0
 * (sections Quick start and API: gdn2_forward_trainable(q, k, v, ..., g, scale,
 * h0) -> (out, h_final) is differentiable with respect to its inputs and h0,
 * and section Features: a fused backward that reuses forward residuals). The
 * reverse pass itself is hand-derived from the chunked forward (the pages
 * print no formula for it): a reverse scan of the state gradient over the
 * chunks, then chunk-parallel products and the decay gradients (dg is a
 * reverse cumulative sum inside each chunk).
 * Same inputs as the forward plus the residuals it wrote, dout [B,T,H,Dv] and
 * dh_final (NULL = zeros). Writes dq, dk, dv, dg, dbeta and dh0 (may be NULL).
 * workspace: gdn_chunk_bwd_workspace_bytes(dims) bytes, 256-byte aligned,
 * caller-owned, overwritten. With bf16 operands, Dk = Dv = 128 and fewer
 * (batch, head) pairs than SMs, the reverse scan and the chunk gradients run as
 * one cooperative launch of one CTA per SM, synchronised through counters in
 * the workspace that a one-CTA kernel zeroes before it (two launches where the
 * context cannot hold that grid). dims.dtype is that of the forward call that wrote
 * the residuals (bfloat16 or float32 operands; the state gradient is fp32 in
 * both); errors as listed at the top of this file. With GDN_FLAG_CHUNK128
 * (bf16): the reverse scan runs over the 128-token chunks, a kernel forms the
 * 64-token blocks' dU, dS, chunk-start states and U across each block boundary
 * (one reverse and one forward step of the 64-token recurrence), and the
 * 64-token chunk gradients follow. */
int gdn_chunk_bwd(const gdn_dims* dims, const void* q, const void* k, const void* v,
                  const void* g, const void* beta, const float* h0, float scale,
                  const void* residuals, const void* dout, const float* dh_final, void* dq,
                  void* dk, void* dv, void* dg, void* dbeta, float* dh0, void* workspace,
                  void* stream);

/* Chunked forward that allocates nothing and takes no residual buffer.
 *
 * The paper has no counterpart to this call; it exists for callers that cannot
 * call cudaMalloc: code that runs where device memory is owned by someone else
 * (an inference server or plugin host with a fixed memory pool, an embedded or
 * real-time loop that forbids allocation after start-up, a runtime whose
 * allocator would have to be re-entered from a callback). Inputs and outputs
 * are the caller's, exactly as in gdn_chunk_fwd; only the residual records the
 * forward passes between its kernels live in a static device array compiled
 * into the library, GDN_NOALLOC_SCRATCH_BYTES (32 MiB) on every GPU that loads
 * the library, held until the process exits. That fits up to 254 chunk-heads
 * (B * H * T/64) at Dk = Dv = 128 in bf16 (127 in fp32), e.g. B=1, H=3,
 * T=4096; larger problems return GDN_ERR_SCRATCH_LIMIT, before anything is
 * enqueued, and must use gdn_chunk_fwd.
 *
 * The first call on a device resolves the array's device address there (with
 * that device current) and keeps it for the life of the process; make that
 * first call before any stream capture, and make no call after a
 * cudaDeviceReset (or any other teardown of the device's primary context) in
 * the same process, because the kept address would then be stale. Every
 * call shares the one array: calls whose work overlaps on the GPU (on two
 * streams, or from two threads) race on it and must be serialised by the
 * caller. The array keeps the last call's contents; nothing in it needs to
 * start at zero because each call writes every record (and resets the forward
 * scan's chunk counters) before reading it. No
 * cudaMalloc, cudaFree or allocating library routine is called. The residual
 * records are not available afterwards, so this call cannot feed
 * gdn_chunk_bwd. Arguments and other errors as gdn_chunk_fwd. */
#define GDN_NOALLOC_SCRATCH_BYTES (32u << 20)
int gdn_chunk_fwd_noalloc(const gdn_dims* dims, const void* q, const void* k, const void* v,
                          const void* g, const void* beta, const float* h0, float scale,
                          void* out, float* h_final, void* stream);

/* Token-recurrent prefill / decode ("gated-deltanet" kernel card, sections
 * Usage and Method): the exact recurrence in fp32, token by token, any T >= 0.
 * Each state slice is read once and written once per call, and the per-token
 * arithmetic does not depend on how a sequence is split into calls, so a
 * sequence run in several calls (carrying h_final -> h0) equals one call
 * bitwise. h0 NULL = zeros; h_final may equal h0 (in place). T = 0 copies h0
 * to h_final. */
int gdn_recurrent(const gdn_dims* dims, const void* q, const void* k, const void* v,
                  const void* g, const void* beta, const float* h0, float scale, void* out,
                  float* h_final, void* stream);

/* Replay decode: the state of each (batch, head) held as a checkpoint plus a
 * buffer of its last few tokens, after the ReplaySSM summary on the ai4snews
 * "Gated DeltaNet" topic page (item "SSM decoding stops writing state every
 * step"): each step reads the checkpoint, computes the token's output directly
 * from it and the buffered tokens, and appends the token to the buffer; the
 * checkpoint is written only when a step finds the buffer full (it is folded in
 * first). A decode step therefore reads the state but rarely writes it, where
 * gdn_recurrent reads and writes it every step. Outputs equal the recurrence to
 * rounding (not bitwise: the sums run in another order).
 *
 *   L       buffer length in tokens, 1 .. GDN_REPLAY_MAX_TOKENS, fixed for the
 *           life of a buffer
 *   ckpt    [B,H,Dk,Dv] float32 checkpoint, read and (on a fold) written in
 *           place. Start a sequence with ckpt = its state (zeros, or h_final of
 *           a prefill) and fill = 0.
 *   buffer  gdn_replay_buffer_bytes(dims, L) bytes, 16-byte aligned: per (b, h)
 *           L slots of (k, cumulative log-decay since the checkpoint, delta), fp32;
 *           private layout, no initialisation needed
 *   fill    [B,H] int32, slots in use; advanced by each step (to 1 after a
 *           fold). Rolling back the last r <= fill tokens of a sequence (a
 *           rejected speculative draft) is lowering its fill by r before the
 *           next call. A count outside [0, L] sets bit 2 (value 2) of the device
 *           error word and is clamped.
 * gdn_replay_decode processes one token per (b, h): dims.T must be 1, inputs
 * and out as gdn_recurrent with T = 1; dims.flags may hold
 * GDN_FLAG_QK_L2NORM. gdn_replay_state writes the full state the buffer stands
 * for, h_out = fold(ckpt, the fill slots) [B,H,Dk,Dv] (dims.T is ignored); it
 * does not change ckpt, buffer or fill. h_out may be ckpt itself, in which case
 * the caller sets fill to 0 afterwards. Errors as gdn_recurrent, plus
 * GDN_ERR_SHAPE for dims.T != 1 in gdn_replay_decode and GDN_ERR_INVALID_ARG
 * for L out of range. Returns 0 bytes for invalid dims or L. */
#define GDN_REPLAY_MAX_TOKENS 8
size_t gdn_replay_buffer_bytes(const gdn_dims* dims, int L);
int gdn_replay_decode(const gdn_dims* dims, int L, const void* q, const void* k, const void* v,
                      const void* g, const void* beta, float scale, float* ckpt, void* buffer,
                      int* fill, void* out, void* stream);
int gdn_replay_state(const gdn_dims* dims, int L, const float* ckpt, const void* buffer,
                     const int* fill, float* h_out, void* stream);

/* Self-test of the failure path: launches a one-thread kernel that first waits,
 * with the library's cross-CTA counter wait (the one the forward's output CTAs use
 * on the scan), for a counter nothing raises, and gives up after max_tries polls
 * (1 .. 65536), setting bit 1 of the device error word. It then waits on an
 * mbarrier nothing arrives on and gives up after max_tries tries, like every wait
 * in the library's kernels, runs four more of the kernels' own bounded waits on
 * the same barrier (each must give up after 4096 tries or a little more, because
 * the error word is set: after one time-out the library's later waits end early
 * instead of running their full count), and returns; the context stays usable.
 * The next gdn_check_device_error returns GDN_ERR_INTERNAL. cycles: NULL, or a
 * 16-byte aligned device buffer of three unsigned 64-bit words that receives the
 * clock cycles of the first mbarrier wait, of the four later waits together and
 * of the counter wait. Not part of the method: it lets a caller or a test see
 * the error path work without a GPU fault. */
int gdn_selftest_wait_timeout(unsigned max_tries, unsigned long long* cycles, void* stream);

/* Reads and clears the library's device error word on the current device
 * (bits, OR-ed: 1 = a kernel gave up waiting for one of its own asynchronous
 * copies; 2 = a replay fill count was outside [0, L]).
 * Synchronises the device. Returns GDN_OK when the word was zero,
 * GDN_ERR_INTERNAL when it was not, GDN_ERR_CUDA if the read failed. */
int gdn_check_device_error(void);

/* Static description of a status code (never NULL). */
const char* gdn_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int gdn_version(void);

/* Optional per-launch timing, off by default. While enabled, every kernel the
 * library launches is bracketed by two CUDA events recorded on the launch
 * stream (one host thread, one device at a time). gdn_profile_enable(1)
 * starts a fresh record, gdn_profile_enable(0) stops recording.
 * gdn_profile_read(ms, launches, n) waits for the recorded events, writes for
 * each kernel id < n the summed milliseconds and the launch count, clears the
 * record and returns GDN_OK (GDN_ERR_CUDA if an event failed). Kernel ids:
 * 0 chunk preparation, 1 forward state scan, 2 reverse state scan, 3 state
 * products, 4 chunk gradients, 5 recurrent, 6 backward finalisation,
 * 7 chunk outputs, 8 forward state scan on tcgen05 tensor cores, 9 reverse
 * state scan on tcgen05 tensor cores (8 and 9 replace 1 and 2 for bf16
 * operands with Dk = Dv = 128), 10 single-token decode (replaces 5 when T = 1),
 * 11 q/k L2 normalisation, 12 its reverse (GDN_FLAG_QK_L2NORM only),
 * 13 replay decode, 14 replay state fold, 15 the backward's products that need
 * no reverse-scan result (Dk = 64 or fp32 operands), 16 the fused chunk
 * gradients on tcgen05 tensor cores (replaces 3, 4, 6 and 15 for bf16 operands
 * with Dk = Dv = 128; when B * H is below the SM count the same launch also runs
 * the reverse scan, which then replaces 9 too), 17 chunk preparation on tcgen05
 * tensor cores (replaces 0 for bf16 operands with Dk = Dv = 128), 18 the zeroing
 * of that single backward launch's counters; gdn_kernel_name(id) names them
 * ("" for an unknown id). Not part of the paper's method: instrumentation. */
int gdn_profile_enable(int on);
int gdn_profile_read(double* ms, int* launches, int n);
const char* gdn_kernel_name(int id);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
