/*
 * kda.h -- C ABI of libkda.so: the chunkwise-parallel forward of Kimi Delta
 * Attention (KDA) on one GB300 (sm_103a).
 *
 * The operation.  For every (sequence n, head h), with a state S of dk x dv
 * (row i = key channel, column j = value channel):
 *
 *   a_t = max(-softplus(g_logit_t), -5)                (per key channel)
 *   S_t = (I - beta_t k_t k_t^T) Diag(exp(a_t)) S_{t-1} + beta_t k_t v_t^T
 *   o_t = S_t^T (scale * q_t)
 *
 *  - gated delta rule with a diagonal, per-channel decay, computable in a
 *    chunk-parallel form; decay logits through a negative softplus:
 *    Kimi K3 walkthrough (Towards AI, M. Zhao), section "Kimi Delta
 *    Attention (KDA)";
 *  - floor of -5 on the per-step log-decay (at least ~0.67% kept), which
 *    holds a 16-token tile's cumulative log-decay in [-80, 0] so that every
 *    intra-chunk tile, diagonal ones included, is one dense BF16 product:
 *    Kimi K3 architecture (orkas.ai), section "A lower bound that erased a
 *    GPU code path";
 *  - fixed-size recurrent state that does not grow with the sequence:
 *    same page, section "Sequence"; the state as checkpoint/hand-over
 *    quantity: section "The cost is paid in the serving stack".
 * beta is the already-squashed write strength (e.g. a sigmoid output).
 * scale multiplies q (1.0 = none).
 *
 * Layouts (row-major, contiguous, no padding):
 *   q, k, g_logit    [B, T, H, dk]      v, out    [B, T, H, dv]
 *   beta             [B, T, H]
 *   init_state, final_state   [N, H, dk, dv] fp32 (N = B when dense)
 * Packed variable-length batches: cu_seqlens (int32, DEVICE memory, N + 1
 * entries, cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] = T); the
 * tensors are then [1, T, H, .] and the B argument carries N.  Chunks and
 * 16-token tiles restart at every sequence start.
 *
 * Ownership: the caller owns every buffer; the library keeps no pointer
 * after a call returns.  Device pointers must come from the current device.
 * init_state may equal final_state (in-place resume); out must not alias
 * any input.  Either state pointer may be NULL (zero initial state / final
 * state not wanted).
 *
 * Asynchrony: the device entry points enqueue work on `stream` and return;
 * outputs are valid once the stream has reached that point.  Problems the
 * host can see (NULL required pointers, sizes, alignment) return an error
 * before anything is enqueued and nothing is written.  Problems only the
 * device can see (malformed cu_seqlens, a wait that timed out) are written
 * to `dev_status` (kda_chunk_fwd_ex) as a kda_status value; the affected
 * outputs are then unspecified, and no access ever leaves the buffers the
 * arguments describe.
 *
 * Alignment: q, k, v, g_logit, out 16-byte aligned; beta 2-byte (bf16) or
 * 4-byte (fp32); states 16-byte aligned.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* kda_stream_t;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,  /* NULL required pointer, non-positive size, out aliasing */
  KDA_ERR_UNSUPPORTED = 2,  /* dk / dv / chunk / dtype combination not built */
  KDA_ERR_MISALIGNED = 3,   /* a pointer breaks the alignment rule above */
  KDA_ERR_BAD_SEQLENS = 4,  /* cu_seqlens not 0 .. T non-decreasing (device-detected) */
  KDA_ERR_TIMEOUT = 5,      /* a bounded on-chip wait gave up (device-detected) */
  KDA_ERR_CUDA = 6,         /* a CUDA runtime call failed */
  KDA_ERR_WORKSPACE = 7,    /* workspace given but below the path's minimum (see kda_chunk_fwd_ex) */
  KDA_ERR_BOUNDS = 8        /* a device-side bounds check failed (KDA_DEBUG builds only) */
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

/* Implementation choice for kda_chunk_fwd_ex (the result is the same
 * function of the inputs up to rounding). */
typedef enum {
  KDA_ALGO_AUTO = 0,  /* tensor-core path where built (the two-kernel form at
                       * dk = dv = 128), else CUDA-core */
  KDA_ALGO_SIMT = 1,  /* fp32 CUDA-core chunked path (16-token chunks) */
  KDA_ALGO_TC = 2,    /* tcgen05/TMEM/TMA fused path (bf16, dk = dv = 128) */
  KDA_ALGO_SPLIT = 3  /* tensor-core path in two kernels (bf16, dk = dv = 128): every
                       * chunk's state-independent part at once, then the serial
                       * state pass; needs a workspace */
} kda_algo;

/* Human-readable name of a status code (static storage). */
const char* kda_status_string(kda_status s);

/*
 * kda_chunk_fwd -- forward for BF16 inputs (values stored as bf16 bit
 * patterns, uint16_t), fp32 states, bf16 output rounded to nearest even.
 * dk, dv in {16, 32, 64, 128}; B, H >= 1; T >= 0.  Device pointers.
 */
kda_status kda_chunk_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const uint16_t* g_logit, const uint16_t* beta,
                         const float* init_state, uint16_t* out, float* final_state,
                         int B, int T, int H, int dk, int dv, const int32_t* cu_seqlens,
                         kda_stream_t stream);

/* Same, fp32 inputs and output (CUDA-core path, fp32 arithmetic). */
kda_status kda_chunk_fwd_f32(const float* q, const float* k, const float* v,
                             const float* g_logit, const float* beta,
                             const float* init_state, float* out, float* final_state,
                             int B, int T, int H, int dk, int dv, const int32_t* cu_seqlens,
                             kda_stream_t stream);

/*
 * kda_chunk_fwd_ex -- the general entry point.
 *   dtype       KDA_BF16 or KDA_F32 (q, k, v, g_logit, beta, out).
 *   chunk_size  0 (implementation's choice), 16 or 64; no effect on the
 *               result beyond rounding.  16 selects the CUDA-core path.
 *   scale       multiplies q.
 *   algo        kda_algo.
 *   workspace   device scratch of at least kda_workspace_bytes() bytes, or
 *               NULL: the library then takes it from the stream-ordered
 *               allocator (cudaMallocAsync / cudaFreeAsync on `stream`).
 *               256-byte aligned.  The two-kernel path (KDA_ALGO_SPLIT)
 *               also accepts less for a dense batch, down to one chunk
 *               record per (sequence, head) plus the carried state
 *               (N * H * (66048 + 65536) bytes, rounded up to 256): it then
 *               runs the sequence in more, shorter slices; below that
 *               KDA_ERR_WORKSPACE.  A packed batch runs in slices of
 *               chunk columns the same way: at least one column's records
 *               (H * 66048 bytes) after the carried state, the chunk
 *               offsets, the sequence order and the chunk table
 *               (kda_workspace_bytes asks for every column's records,
 *               ceil(T / 64) + N columns at most, while they fit in
 *               32 GiB).
 *               For a dense batch of few long sequences (6 N H state
 *               CTAs at most one per SM, 384 chunks or more per sequence)
 *               kda_workspace_bytes asks for the records of every chunk
 *               (N * H * ceil(T / 64) * 66048 bytes, at most 32 GiB) plus
 *               three [N][G][H][dk][dv] fp32 state buffers, and the call
 *               cuts each sequence into G segments run side by side
 *               (segment summaries, their composition into entry states,
 *               then the reruns); a smaller workspace runs the plain
 *               sliced form.
 *   dev_status  NULL or one device int32; set to KDA_OK at the start of the
 *               work and to a device-detected error if one occurs.
 */
kda_status kda_chunk_fwd_ex(const void* q, const void* k, const void* v, const void* g_logit,
                            const void* beta, const float* init_state, void* out,
                            float* final_state, int B, int T, int H, int dk, int dv,
                            const int32_t* cu_seqlens, kda_dtype dtype, int chunk_size,
                            float scale, int algo, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, kda_stream_t stream);

/*
 * kda_chunk_fwd_ckpt -- kda_chunk_fwd_ex (automatic path, default chunk)
 * that also writes state checkpoints: after every `every` tokens of each
 * sequence (every: a multiple of 64), the state S at that point goes to
 * checkpoints[n][h][c][dk][dv] (fp32, device, 16-byte aligned), c = 0 ..
 * max_per_seq-1 counting boundaries from the sequence start; boundaries
 * beyond max_per_seq are not written, nor are slots of a sequence that
 * ends before them.  The state at a checkpoint is what a later call would
 * take as init_state to resume there: the recurrent half of the prefix
 * cache, checkpointed on a sparse subset of hash boundaries (Kimi K3
 * architecture, orkas.ai, "The cost is paid in the serving stack").
 */
kda_status kda_chunk_fwd_ckpt(const void* q, const void* k, const void* v, const void* g_logit,
                              const void* beta, const float* init_state, void* out,
                              float* final_state, int B, int T, int H, int dk, int dv,
                              const int32_t* cu_seqlens, kda_dtype dtype, float scale,
                              float* checkpoints, int every, int max_per_seq,
                              int32_t* dev_status, kda_stream_t stream);

/*
 * kda_decode -- the recurrent form for a few tokens per sequence (a decode
 * step, or the speculative-decoding rebuild that replays accepted tokens'
 * cached projected inputs from a saved state): the same operation as
 * kda_chunk_fwd_ex with init_state == final_state == `state`, computed
 * token by token with the state slice held on chip, for short T.
 * Dense layouts [N, T, H, .]; `state` [N, H, dk, dv] fp32, read and
 * updated in place.  dtype KDA_BF16 or KDA_F32; dk, dv in {16, 32, 64, 128}.
 */
kda_status kda_decode(const void* q, const void* k, const void* v, const void* g_logit,
                      const void* beta, float* state, void* out, int N, int T, int H, int dk,
                      int dv, kda_dtype dtype, float scale, kda_stream_t stream);

/*
 * kda_chunk_fwd_seg -- kda_chunk_fwd (bf16, dense, dk = dv = 128) with
 * every sequence cut into `nseg` segments of ceil(T / nseg) tokens rounded
 * up to a multiple of 64 that run in parallel: each segment's state update
 * is affine in its entry state (S_out = P S_in + S0, P its cumulative
 * transition, S0 its final state from a zero start); the segments'
 * (P, S0) are computed in parallel, a short scan resolves every entry
 * state, and the segments then run again from those states writing the
 * output (Kimi K3 architecture, orkas.ai, "The cost is paid in the serving
 * stack": a cumulative transition and a zero-start state per segment, then
 * a prefix scan).  Useful when B * H is small against the SM count.
 * workspace: device scratch of kda_seg_workspace_bytes(B, H, nseg, dk, dv)
 * bytes (256-byte aligned), or NULL to take it from the stream-ordered
 * allocator.  nseg = 1 is the plain forward.  (kda_chunk_fwd_ex's
 * automatic path cuts such batches into segments on the two-kernel path;
 * see its workspace note.)
 */
kda_status kda_chunk_fwd_seg(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             const uint16_t* g_logit, const uint16_t* beta,
                             const float* init_state, uint16_t* out, float* final_state, int B,
                             int T, int H, int dk, int dv, float scale, int nseg,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             kda_stream_t stream);

/*
 * kda_chunk_fwd_seg_static -- kda_chunk_fwd_seg (nseg >= 2) that allocates
 * nothing: for callers that may not allocate device memory at all, such as
 * a serving engine that has reserved every byte of HBM for its own pools,
 * or a host framework that neither hands out a workspace nor allows one to
 * be allocated.  (This entry point has no counterpart on the pages; it is a
 * deployment convenience.)  The segment scratch lives in a fixed 16 MiB
 * array compiled into the library, held by every GPU that loads it until
 * the process exits; batches needing more (B * H * nseg > 85 at dk = dv =
 * 128) are refused with KDA_ERR_WORKSPACE before anything is queued.  The
 * caller still provides inputs and outputs.  The first call on a device
 * looks up the array's device address (a runtime query, no allocation);
 * make that first call before any stream capture.  The address is kept for
 * the life of the process, so do not use this entry point on a device after
 * cudaDeviceReset() there (the array then lives at a new address).  The
 * argument rules are those of kda_chunk_fwd_seg.  All calls share the one
 * array and nothing in it needs to start at zero (every value read was
 * written earlier in the same call), so calls that overlap on the GPU race:
 * issue them on one stream, or otherwise one at a time.
 */
kda_status kda_chunk_fwd_seg_static(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    const uint16_t* g_logit, const uint16_t* beta,
                                    const float* init_state, uint16_t* out, float* final_state,
                                    int B, int T, int H, int dk, int dv, float scale, int nseg,
                                    int32_t* dev_status, kda_stream_t stream);

/*
 * Context parallelism: the token axis of a batch split across devices
 * (Kimi K3 architecture, orkas.ai, "The cost is paid in the serving stack";
 * Towards AI walkthrough, "Infrastructure co-design": each device's span is
 * summarised by a cumulative transition and a zero-initialised state, which
 * compose; a prefix scan over one fixed-size all-gather gives each device
 * its entry state).
 *
 * kda_segment_summary -- the summary of the span [0, T) of every sequence of
 * a dense bf16 batch (dk = dv = 128; layouts as kda_chunk_fwd): running the
 * span from a state S_in gives S_out = P S_in + S0.  `summary` (device, fp32,
 * 16-byte aligned, kda_summary_floats(B, H, dk, dv) floats, not overlapping
 * the inputs) receives P [B][H][dk][dk] followed by S0 [B][H][dk][dv].  T = 0
 * gives P = I, S0 = 0.  Asynchronous on `stream`; dev_status as in
 * kda_chunk_fwd_ex.
 */
kda_status kda_segment_summary(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const uint16_t* g_logit, const uint16_t* beta, float* summary,
                               int B, int T, int H, int dk, int dv, int32_t* dev_status,
                               kda_stream_t stream);

/* Floats of one summary: N * H * (dk * dk + dk * dv). */
size_t kda_summary_floats(int N, int H, int dk, int dv);

/*
 * kda_state_compose -- the state after m consecutive spans, from their
 * summaries in order: S = P_{m-1}( ... (P_0 S_init + S0_0) ... ) + S0_{m-1}.
 * `summaries` (device, fp32) holds the m summaries back to back, each laid
 * out as kda_segment_summary writes it; init_state [N][H][dk][dv] or NULL
 * (zero); state_out [N][H][dk][dv] (may equal init_state).  m = 0 copies the
 * initial state.  dk = dv = 128; fp32 arithmetic.  Asynchronous on `stream`.
 */
kda_status kda_state_compose(const float* summaries, int m, const float* init_state,
                             float* state_out, int N, int H, int dk, int dv,
                             kda_stream_t stream);

/* Scratch bytes of kda_chunk_fwd_seg (0 when nseg < 2). */
size_t kda_seg_workspace_bytes(int B, int H, int nseg, int dk, int dv);

/* Device scratch bytes kda_chunk_fwd_ex needs for these sizes (0 = none).
 * N = number of sequences (B, or the cu_seqlens count when packed). */
size_t kda_workspace_bytes(int N, int T, int H, int dk, int dv, int dtype, int chunk_size,
                           int algo, int packed);

/*
 * kda_chunk_fwd_host -- end-to-end call on HOST buffers (pinned memory
 * recommended): copies the inputs (and cu_seqlens) to the device, runs the
 * forward, copies out and final_state back and synchronises `stream`
 * before returning.  Same layouts and rules as kda_chunk_fwd_ex; every
 * pointer here is a host pointer.  dev_buffer: device memory of at least
 * kda_host_staging_bytes() bytes, or NULL (then taken from and returned to
 * the stream-ordered allocator).  The device status is read back and
 * returned as the call's result.  On the two-kernel path (bf16, dk = dv =
 * 128, two or more chunks, or for a packed batch two or more columns of
 * the bound ceil(T / 64) + B) the call runs in up to eight pieces of whole
 * chunks -- chunks [c0, c1) of every sequence of a dense batch, or chunk
 * columns [g0, g1) of a packed one (a contiguous range of token rows):
 * while piece i runs on `stream`, the inputs of piece i + 1 are copied in
 * and the output of piece i - 1 copied out on streams of the call's own,
 * so the copies overlap the kernels; the result is bit-identical to
 * kda_chunk_fwd_ex on device copies of the same inputs.  cu_seqlens is a
 * host array here; it is checked before any copy.
 */
kda_status kda_chunk_fwd_host(const void* q, const void* k, const void* v, const void* g_logit,
                              const void* beta, const float* init_state, void* out,
                              float* final_state, int B, int T, int H, int dk, int dv,
                              const int32_t* cu_seqlens, kda_dtype dtype, float scale,
                              void* dev_buffer, size_t dev_buffer_bytes, kda_stream_t stream);

/* Device bytes kda_chunk_fwd_host stages through for these sizes: inputs,
 * outputs, states and the automatic path's workspace (on the two-kernel
 * path, the chunk records of one piece). */
size_t kda_host_staging_bytes(int B, int T, int H, int dk, int dv, int dtype, int has_init,
                              int has_final, int packed);

/*
 * Test hooks (not part of the hot path): the intra-chunk steps of the
 * tensor-core path for one (sequence n, head h), every chunk, written to
 * fp32 device buffers laid out [n_chunks, 64, .]:
 *   gam  [., 64, dk]  cumulative decay factor e^{G} from the chunk start
 *   aqk  [., 64, 64]  A_qk incl. diagonal (upper part zero)
 *   akk  [., 64, 64]  beta-weighted A_kk, strictly lower
 *   tinv [., 64, 64]  (I + A_kk)^{-1}
 *   w    [., 64, dk], u [., 64, dv]
 * Inputs as kda_chunk_fwd (bf16, dense or packed).  Any output may be NULL.
 */
kda_status kda_debug_intra(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const uint16_t* g_logit, const uint16_t* beta, int B, int T, int H,
                           int dk, int dv, const int32_t* cu_seqlens, int n, int h,
                           float* gam, float* aqk, float* akk, float* tinv, float* w,
                           float* u, kda_stream_t stream);

/*
 * Test hook: one tcgen05 tile product D = A * B^T (bf16 in, fp32 out) with
 * the operand layouts the tensor-core path uses, to check descriptors and
 * lane placement.  A [M][K], B [N][K] row-major bf16 device buffers; D
 * [128][N] fp32 receives all 128 accumulator lanes (lanes an M = 64 tile
 * does not write hold a NaN marker).  M in {64, 128}; N in 16..256 and K in
 * 16..128, multiples of 16.  a_mode: 0 shared K-major, 1 shared MN-major,
 * 2 tensor memory (M = 128 only); b_mode: 0 K-major, 1 MN-major, 2 MN-major
 * with the 128-byte swizzle (N = 64: one swizzle atom wide); pack:
 * order of the 8x16-byte core matrices (0: along K first, 1: along M/N
 * first).  One CTA; asynchronous on `stream`.
 */
kda_status kda_debug_umma(const uint16_t* A, const uint16_t* B, float* D, int M, int N, int K,
                          int a_mode, int b_mode, int pack, int32_t* dev_status,
                          kda_stream_t stream);

/*
 * Profiling hook (not part of the hot path): one of the two kernels of the
 * KDA_ALGO_SPLIT path over a dense bf16 batch (dk = dv = 128), so that each
 * can be timed on its own.  stage 1: the intra-chunk kernel, writes every
 * chunk's record into `workspace`; stage 2: the state kernel, reads them,
 * writes out and final_state.  The workspace must hold the whole sequence
 * in one slice (kda_workspace_bytes(..., KDA_ALGO_SPLIT, 0) does), else
 * KDA_ERR_WORKSPACE.  Stage 2 is meaningful only after stage 1 on the same
 * inputs and workspace.  Asynchronous on `stream`.
 */
kda_status kda_split_stage(int stage, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const uint16_t* g_logit, const uint16_t* beta,
                           const float* init_state, uint16_t* out, float* final_state, int B,
                           int T, int H, float scale, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, kda_stream_t stream);

/*
 * Test hook for the bounded waits of the two-kernel path: after
 * kda_debug_stall_test(flags), calls on that path make their first wait in
 * the intra-chunk kernel (flags bit 0) and / or in the state kernel (bit 1)
 * wait, with a 1 ms limit, on a barrier that nothing ever completes.  The
 * wait gives up, the kernel records KDA_ERR_TIMEOUT in dev_status, waits
 * (bounded) for the copies it has in flight, frees its tensor memory and
 * returns; the outputs of such a call are unspecified.  flags = 0 restores
 * normal calls.  Process-wide; not thread-safe against concurrent calls.
 * Returns KDA_ERR_INVALID_ARG for flags outside 0..3.  No counterpart on
 * the pages: it exists to test the library's own failure path.
 */
kda_status kda_debug_stall_test(int flags);

/*
 * Test hook for the segmented two-kernel form (see kda_chunk_fwd_ex's
 * workspace): segments > 0 makes dense batches on that path use that many
 * segments per sequence wherever each segment still holds a chunk (three
 * at least; kda_workspace_bytes follows), segments < 0 turns the form off,
 * 0 restores the automatic choice.  Process-wide; not thread-safe against
 * concurrent calls.  Always KDA_OK.
 */
kda_status kda_debug_split_segments(int segments);

/* Segments per sequence that kda_chunk_fwd_ex on the two-kernel path
 * (dense bf16 batch, dk = dv = 128, on the current device) cuts each
 * sequence into with a workspace of workspace_bytes: 1 for the plain form.
 * Host-only; a query for schedulers and benchmarks. */
int kda_split_segment_count(int N, int T, int H, size_t workspace_bytes);

/*
 * Debug builds (compiled with -DKDA_DEBUG; kda_build_info() says so): the
 * two-kernel path checks, on the device, every chunk record index against
 * the records the workspace holds and every token row against the input,
 * before it touches global memory; a failed check records KDA_ERR_BOUNDS in
 * dev_status, skips the access and ends the kernel as a timeout does.  This
 * hook makes the next calls' kernels believe the workspace holds only
 * `items` chunk records (0 = the real count), so that the checks can be
 * seen to fire while every access stays inside the real buffer.  No effect
 * in normal builds.  Process-wide; not thread-safe against concurrent calls.
 */
kda_status kda_debug_record_capacity(int64_t items);

/* The path family kda_chunk_fwd_ex would take for these arguments:
 * KDA_ALGO_SIMT, KDA_ALGO_TC (AUTO on the tensor cores: fused, segmented or
 * two-kernel form by the sizes) or KDA_ALGO_SPLIT when asked for; -1 if the
 * combination is unsupported. */
int kda_resolve_algo(int dtype, int dk, int dv, int chunk_size, int algo);

/* The path kda_chunk_fwd_ex takes for these sizes (N sequences, T tokens per
 * row, or in total when packed): KDA_ALGO_SIMT, KDA_ALGO_TC (fused kernel)
 * or KDA_ALGO_SPLIT; -1 if the call would be refused. */
int kda_resolve_path(int N, int T, int H, int dk, int dv, int dtype, int chunk_size, int algo,
                     int packed);

/* Library build identification (static string). */
const char* kda_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
