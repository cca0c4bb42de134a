/*
 * kvgqa.h -- C ABI of the GB300 (sm_103a) cached GQA + RoPE decode/prefill path.
 *
 * One shared library, libkvgqa.so, exports the operations of the
 * positions-aware active-batch decode step over a shared slot KV cache and of
 * its dense case, the equal-length prefill into empty cache rows
 * (microLLM-rocm ARCHITECTURE.md, section "Tensor ownership boundary"):
 *
 *   rope_kv_store_out_            decode-only RoPE of Q/K at each row's own
 *                                 position + K/V store into that row's cell
 *   cached_gqa_attention_out_     GQA attention of each query over its row's
 *                                 cached prefix (split-K + combine)
 *   prefill_gqa_cached_rows_out_  A prompts of T tokens: RoPE, store into the
 *                                 target empty rows, causal GQA attention
 *   prefill_varlen_gqa_cached_rows_out_  prompts of different lengths at their
 *                                 own offsets (chunked prefill), same steps
 *
 * Boundary conventions (same page, sections "Tensor ownership boundary" and
 * "Stable integration boundary"):
 *  - Every tensor crosses as a non-owning descriptor: pointer, accessible
 *    bytes, shape, element strides, dtype and device.  The library never
 *    allocates, frees or keeps a pointer after a call returns.
 *  - Outputs, workspace, device and stream are explicit arguments; ownership
 *    is never inferred from a pointer.
 *  - Unsupported layouts are rejected with a status code, never copied into a
 *    supported one behind the caller's back.
 *  - Every check the host can make (dtype, rank, shape, contiguity, alignment,
 *    device, aliasing, workspace size, scalar ranges) is made before any work
 *    is queued, and failure returns a status with a message from
 *    kvgqa_last_error(); nothing is launched then.
 *  - Values that live only on the device (positions, cache rows) are checked
 *    by the kernels: a row whose metadata is out of range is skipped (nothing
 *    of it is read or written) and a flag is set in the workspace status block,
 *    which kvgqa_read_status() returns on request.  The default path never
 *    synchronises the stream.
 *  - A call that queues work only launches kernels on the given stream (some
 *    with programmatic dependent launch): it can be captured into a CUDA
 *    graph on a non-default stream and replayed, the replay using the
 *    pointers and sizes of the captured call.  The no-allocation entry point
 *    looks up its static array's address at its first call on a device, which
 *    should therefore precede any capture.
 *
 * Data types: Q, K, V, the caches and the outputs are BF16, or all IEEE
 * binary16 (FP16 cached rows; one storage type per call, taken from its first
 * 16-bit tensor, every other 16-bit operand must match or the call returns
 * KVGQA_EDTYPE); "bf16" below stands for that storage type.  Results are
 * rounded once, to nearest even, in it.  Positions and cache rows are int32;
 * softmax and accumulation run in FP32.
 *
 * Layouts (row-major, contiguous, element strides):
 *   decode  q, q_out, out   [A, H_q, D]          k, v  [A, H_kv, D]
 *   prefill q, out          [A, T, H_q, D]       k, v  [A, T, H_kv, D]   (BTHD)
 *   caches  k_cache, v_cache [S, H_kv, max_seq, D]   (one layer; S cache slots)
 *   positions, cache_rows   [A] int32
 * with G = H_q / H_kv query heads per KV head, query head h reading KV head
 * floor(h / G), and D in {64, 128}.
 *
 * Thread safety: calls are reentrant; kvgqa_last_error() is per host thread.
 */
#ifndef KVGQA_H_
#define KVGQA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVGQA_ABI_VERSION 1
#define KVGQA_MAX_DIMS 6

/* Element types of a descriptor. */
typedef enum kvgqa_dtype {
  KVGQA_BF16 = 1,
  KVGQA_I32 = 2,
  KVGQA_F32 = 3,
  KVGQA_U8 = 4,
  KVGQA_F16 = 5    /* IEEE binary16 */
} kvgqa_dtype;

/* Non-owning tensor descriptor.  `data` is a device pointer on `device` (it may
 * be NULL only when the tensor has no elements); `bytes` is how many bytes are
 * accessible from `data` on (the view must lie inside them); `strides` are in
 * elements.  The caller keeps the memory alive until the queued work is done. */
typedef struct kvgqa_tensor {
  void* data;
  int64_t bytes;
  int32_t ndim;
  int32_t dtype;   /* kvgqa_dtype */
  int32_t device;  /* CUDA device ordinal */
  int32_t reserved;
  int64_t shape[KVGQA_MAX_DIMS];
  int64_t strides[KVGQA_MAX_DIMS];
} kvgqa_tensor;

/* Return codes.  Anything but KVGQA_OK means nothing was queued. */
typedef enum kvgqa_status {
  KVGQA_OK = 0,
  KVGQA_EINVAL = 1,      /* bad rank/shape/size/scalar, null descriptor */
  KVGQA_EDTYPE = 2,      /* wrong element type */
  KVGQA_ELAYOUT = 3,     /* non-contiguous strides or misaligned pointer */
  KVGQA_EDEVICE = 4,     /* tensor not on the current device, or not device memory */
  KVGQA_EALIAS = 5,      /* a written tensor overlaps another operand */
  KVGQA_EWORKSPACE = 6,  /* workspace too small or misaligned */
  KVGQA_ECUDA = 7,       /* a CUDA runtime call failed (message has the CUDA error) */
  KVGQA_EUNSUPPORTED = 8, /* a legal shape this build has no kernel for (e.g. D = 96) */
  KVGQA_EFULL = 9         /* slot table: no free cache row */
} kvgqa_status;

/* Bits of the device status word (first 4 bytes of every workspace). */
#define KVGQA_FLAG_POSITION_RANGE 0x1 /* some positions[a] outside [0, max_seq) */
#define KVGQA_FLAG_ROW_RANGE 0x2      /* some cache_rows[a] outside [0, S) */
#define KVGQA_FLAG_TIMEOUT 0x4        /* a bounded in-kernel wait expired; that work was dropped */

/* Every workspace starts with a 256-byte status block; its first int32 is the
 * status word.  Kernels only OR bits into it.  It must be zero before first use
 * (a zero-filled workspace is ready); kvgqa_read_status() clears it. */
#define KVGQA_STATUS_BYTES 256

/* Version of this interface (the descriptor layout, the entry points and
 * their arguments); a caller built against another version should not call
 * in.  Never fails. */
int kvgqa_abi_version(void);

/* Message of the last failing call on this host thread ("" if none). */
const char* kvgqa_last_error(void);

/* Workspace of rope_kv_store_out_: just the status block. */
kvgqa_status rope_kv_store_workspace_size(size_t* bytes);

/*
 * rope_kv_store_out_ -- decode RoPE + K/V store for A active tokens.
 *
 * For every active token a with position p = positions[a] and row
 * r = cache_rows[a]:
 *   q_out[a, h, :]            = RoPE(q[a, h, :], p)    for h < H_q
 *   k_cache[r, g, p, :]       = RoPE(k[a, g, :], p)    for g < H_kv
 *   v_cache[r, g, p, :]       = v[a, g, :]             (bytes copied unchanged)
 * and no other byte of the caches is written, so inactive rows and every other
 * position stay as they were.  RoPE is split-half: pair i = (x[i], x[i+D/2])
 * turns by angle p * theta^(-2i/D) (ARCHITECTURE.md, "Attention layout
 * boundary": even D, nonnegative position, positive base).
 *
 *   q [A,H_q,D] bf16, k/v [A,H_kv,D] bf16, positions/cache_rows [A] int32  (read)
 *   theta  RoPE base, finite and > 0, with every theta^(-2i/D) finite (else
 *          KVGQA_EINVAL; the same holds for every entry point taking theta)
 *   q_out [A,H_q,D] bf16  (written)
 *   k_cache, v_cache [S,H_kv,max_seq,D] bf16  (one cell per token written)
 *   workspace  >= rope_kv_store_workspace_size() bytes, 256-byte aligned
 *   stream  cudaStream_t (NULL = legacy default stream)
 * Preconditions the host cannot see: cache_rows distinct within the call
 * (duplicates race); 0 <= positions[a] < max_seq and 0 <= cache_rows[a] < S, or
 * the token is skipped and the status word flagged.  A = 0 is a no-op.
 */
kvgqa_status rope_kv_store_out_(const kvgqa_tensor* q, const kvgqa_tensor* k,
                                const kvgqa_tensor* v, const kvgqa_tensor* positions,
                                const kvgqa_tensor* cache_rows, double theta,
                                const kvgqa_tensor* q_out, const kvgqa_tensor* k_cache,
                                const kvgqa_tensor* v_cache, const kvgqa_tensor* workspace,
                                void* stream);

/* Workspace of cached_gqa_attention_out_ for these sizes on `device`: the
 * status block, one int32 counter per (row, KV head) and the FP32 split-K
 * partials (it depends on the device's SM count, not on max_seq or the
 * positions).  The counters must be zero before the first call (a zero-filled
 * workspace is ready); every call that completes leaves them at zero.  A call
 * that gave up on a bounded wait (KVGQA_FLAG_TIMEOUT) may leave some short of
 * their count: kvgqa_read_status() then zero-fills the workspace, which makes
 * it ready again. */
kvgqa_status cached_gqa_attention_workspace_size(int64_t A, int64_t H_q, int64_t H_kv,
                                                 int64_t D, int32_t device, size_t* bytes);

/*
 * cached_gqa_attention_out_ -- cached GQA attention of the decode step.
 *
 * For every active token a and query head h, with p = positions[a],
 * r = cache_rows[a], g = floor(h / G):
 *   out[a,h,:] = sum_{j=0..p} softmax_j( scale * q_rot[a,h,:] . k_cache[r,g,j,:] )
 *                * v_cache[r,g,j,:]
 * i.e. the token attends to its row's prefix including its own position (the
 * cell rope_kv_store_out_ just wrote).  Scores, softmax and the weighted sum
 * are FP32; out is rounded to BF16 once.  Nothing past position p of a row is
 * read.  The work is split over the whole GPU by key ranges; the CTA that
 * finishes a split row last merges its partial results (one launch).
 *
 *   q_rot [A,H_q,D] bf16, k_cache/v_cache [S,H_kv,max_seq,D] bf16,
 *   positions/cache_rows [A] int32  (read)
 *   scale  finite (1/sqrt(D) is the usual choice)
 *   out [A,H_q,D] bf16 (written; rows with invalid metadata are left unwritten)
 *   workspace  >= cached_gqa_attention_workspace_size(...) bytes, 256-byte aligned
 * Limits: D in {64,128}; G = H_q / H_kv <= 16;
 * A <= 1024; A * H_kv * max_seq < 2^31.  A = 0 is a no-op.
 */
kvgqa_status cached_gqa_attention_out_(const kvgqa_tensor* q_rot, const kvgqa_tensor* k_cache,
                                       const kvgqa_tensor* v_cache,
                                       const kvgqa_tensor* positions,
                                       const kvgqa_tensor* cache_rows, float scale,
                                       const kvgqa_tensor* out, const kvgqa_tensor* workspace,
                                       void* stream);

/* Workspace of decode_step_out_ and decode_step_single_launch_out_: that of
 * cached_gqa_attention_out_ (status block, counters, partials), then room for
 * the rotated queries (A*H_q*D bf16, 256-byte aligned). */
kvgqa_status decode_step_workspace_size(int64_t A, int64_t H_q, int64_t H_kv, int64_t D,
                                        int32_t device, size_t* bytes);

/*
 * decode_step_out_ -- the whole decode step of one layer: rope_kv_store_out_
 * followed by cached_gqa_attention_out_, in one call.
 *
 * microLLM-rocm ARCHITECTURE.md, section "Tensor ownership boundary":
 * positions and cache rows parameterise decode-only RoPE, the K/V store and
 * cached attention.  For every active token a (p = positions[a],
 * r = cache_rows[a]): the rotated k[a] and the raw v[a] are stored into
 * k_cache/v_cache[r,:,p,:] exactly as rope_kv_store_out_ stores them, and
 * out[a] is the attention of the rotated q[a] over keys 0..p of row r, as
 * cached_gqa_attention_out_ computes it (the rotated queries are rounded to
 * BF16 first, as there).  The results are bit-identical to the two calls.
 * It is faster than them: knowing that the kernel before its attention is its
 * own store kernel (which writes only the rotated queries, into the
 * workspace, and the new cells), the attention streams every cache tile that
 * holds no new cell while the store still runs.
 *
 *   q [A,H_q,D], k/v [A,H_kv,D] bf16, positions/cache_rows [A] int32  (read)
 *   theta > 0 and finite, scale finite
 *   k_cache/v_cache [S,H_kv,max_seq,D] bf16 (read; the cells (r,:,p,:) written)
 *   out [A,H_q,D] bf16 (written; rows with invalid metadata are left
 *     unwritten, their cells untouched, and a status bit is set)
 *   workspace  >= decode_step_workspace_size(...) bytes, 256-byte aligned,
 *     counters zero before the first call (left zero by every call that
 *     completes; after KVGQA_FLAG_TIMEOUT, kvgqa_read_status() re-zeroes)
 * Limits as cached_gqa_attention_out_.  cache_rows must be distinct.  A = 0
 * is a no-op.  There is no q_out: callers that need the rotated queries use
 * the two-call path.
 */
kvgqa_status decode_step_out_(const kvgqa_tensor* q, const kvgqa_tensor* k, const kvgqa_tensor* v,
                              const kvgqa_tensor* positions, const kvgqa_tensor* cache_rows,
                              double theta, float scale, const kvgqa_tensor* k_cache,
                              const kvgqa_tensor* v_cache, const kvgqa_tensor* out,
                              const kvgqa_tensor* workspace, void* stream);

/*
 * decode_step_single_launch_out_ -- decode_step_out_ in one kernel launch:
 * the attention kernel rotates each segment's queries in shared memory and
 * stores the new cells itself (the rotated queries never leave the chip).
 * Same arguments, workspace and results (bit-identical); measured slower
 * than decode_step_out_ on GB300, kept for launch-bound callers.
 */
kvgqa_status decode_step_single_launch_out_(const kvgqa_tensor* q, const kvgqa_tensor* k,
                                            const kvgqa_tensor* v, const kvgqa_tensor* positions,
                                            const kvgqa_tensor* cache_rows, double theta, float scale,
                                            const kvgqa_tensor* k_cache, const kvgqa_tensor* v_cache,
                                            const kvgqa_tensor* out, const kvgqa_tensor* workspace,
                                            void* stream);

/*
 * cached_gqa_attention_static_scratch_out_ -- the same attention as
 * cached_gqa_attention_out_, for callers that cannot allocate device memory.
 *
 * The pages describe no such operation; it exists for callers that have no
 * way to obtain a workspace: code that runs where cudaMalloc is unavailable or
 * forbidden (inside an allocator hook, under an external memory budget that
 * owns every byte, or a host runtime that only ever hands out its inputs and
 * outputs).  Instead of a workspace, the split-K partials go to a scratch array
 * that the library itself holds in device memory: a file-scope static device
 * array of 4 MiB (KVGQA_STATIC_SCRATCH_BYTES), present on every GPU that loads
 * the library until the process exits.  Nothing is allocated by this call: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * The first call on a device looks up the device address of that array (once
 * per device, with that device current); make that first call before any
 * stream capture.  Sizes whose partials do not fit the array are rejected
 * with KVGQA_EUNSUPPORTED.  Every call shares the one array: before its kernel
 * each call clears the array's status word and per-row counters with
 * cudaMemsetAsync on `stream` (which allocates nothing), so no call depends on
 * what an earlier one left, not even one that gave up on a bounded wait; the
 * kernel then overwrites the partials before reading them.  Calls whose work
 * overlaps on the GPU (different streams, or different host threads) race on
 * the array.  Device-side range checks still skip rows with invalid positions
 * or cache rows, but this variant has no status word for the caller to read.
 */
#define KVGQA_STATIC_SCRATCH_BYTES (4u << 20)
kvgqa_status cached_gqa_attention_static_scratch_out_(const kvgqa_tensor* q_rot,
                                                      const kvgqa_tensor* k_cache,
                                                      const kvgqa_tensor* v_cache,
                                                      const kvgqa_tensor* positions,
                                                      const kvgqa_tensor* cache_rows, float scale,
                                                      const kvgqa_tensor* out, void* stream);

/* Workspace of prefill_gqa_cached_rows_out_ and prefill_varlen_gqa_cached_rows_out_:
 * the status block, the rotated queries (A*T*H_q*D 16-bit values, rounded up
 * to 256 bytes) and, used by the varlen call, an order of its work items (one
 * int32 per 128-query tile of each prompt). */
kvgqa_status prefill_gqa_cached_rows_workspace_size(int64_t A, int64_t T, int64_t H_q,
                                                    int64_t H_kv, int64_t D, size_t* bytes);

/*
 * prefill_gqa_cached_rows_out_ -- equal-length prefill into empty rows.
 *
 * A prompts of T tokens each, at positions 0..T-1 (the target rows are empty;
 * ARCHITECTURE.md, "Tensor ownership boundary": equal-length pending prompts run
 * as one batch and each prefix lands in its target empty shared-cache row).
 * With r = cache_rows[a]:
 *   k_cache[r, g, t, :] = RoPE(k[a, t, g, :], t),  v_cache[r, g, t, :] = v[a, t, g, :]
 *   for t < T; nothing else in the caches is written;
 *   out[a, t, h, :] = causal GQA attention of RoPE(q[a,t,h,:], t) over cached
 *   positions 0..t of row r, KV head floor(h/G), scores scaled by `scale`.
 * The prompts are written straight into their rows (no temporary cache).
 *
 *   q [A,T,H_q,D], k/v [A,T,H_kv,D] bf16 (BTHD), cache_rows [A] int32 (read)
 *   theta > 0, scale finite
 *   k_cache/v_cache [S,H_kv,max_seq,D] bf16 with T <= max_seq (rows r written)
 *   out [A,T,H_q,D] bf16 (written)
 *   workspace >= prefill_gqa_cached_rows_workspace_size(...) bytes, 256-byte aligned
 * Precondition: cache_rows distinct.  A = 0 or T = 0 is a no-op.
 */
kvgqa_status prefill_gqa_cached_rows_out_(const kvgqa_tensor* q, const kvgqa_tensor* k,
                                          const kvgqa_tensor* v, const kvgqa_tensor* cache_rows,
                                          double theta, float scale, const kvgqa_tensor* k_cache,
                                          const kvgqa_tensor* v_cache, const kvgqa_tensor* out,
                                          const kvgqa_tensor* workspace, void* stream);

/*
 * prefill_varlen_gqa_cached_rows_out_ -- prompts of different lengths, each
 * at its own position offset, into rows that may already hold a prefix
 * (chunked prefill).
 *
 * ARCHITECTURE.md, "Tensor ownership boundary", keeps prompts of different
 * lengths in separate equal-length groups; this call runs them in one launch.
 * Its RoPE takes a nonnegative position offset per prompt ("Attention layout
 * boundary").  Prompt a holds len = lengths[a] tokens, padded to T in q/k/v,
 * at positions off = offsets[a] .. off+len-1 of row r = cache_rows[a]:
 *   k_cache[r, g, off+t, :] = RoPE(k[a, t, g, :], off+t),
 *   v_cache[r, g, off+t, :] = v[a, t, g, :]            for t < len;
 *   out[a, t, h, :] = GQA attention of RoPE(q[a,t,h,:], off+t) over cached
 *   positions 0..off+t of row r (the prefix the row held, then the prompt's
 *   own keys up to t), KV head floor(h/G), scores scaled by `scale`.
 * Rows t >= len of out are not written.  offsets = 0, lengths = T is
 * prefill_gqa_cached_rows_out_; len = 1 is one decode token at position off;
 * prefilling a prompt in consecutive chunks equals prefilling it at once.
 *
 *   q [A,T,H_q,D], k/v [A,T,H_kv,D] bf16 (BTHD, T = the longest prompt or more)
 *   offsets, lengths, cache_rows [A] int32 (read)
 *   theta > 0, scale finite
 *   k_cache/v_cache [S,H_kv,max_seq,D] bf16 with T <= max_seq (rows r written)
 *   out [A,T,H_q,D] bf16 (rows t < lengths[a] written)
 *   workspace >= prefill_gqa_cached_rows_workspace_size(...) bytes, 256-byte aligned
 * Device-side checks: a prompt with len outside [0, T], off < 0 or
 * off + len > max_seq sets KVGQA_FLAG_POSITION_RANGE, one whose row is outside
 * [0, S) sets KVGQA_FLAG_ROW_RANGE; neither is read or written.  len = 0 is a
 * no-op for that prompt.
 * Preconditions: cache_rows distinct; positions 0..off-1 of each row hold the
 * prefix the prompt continues.  Cells past off+len are never read.
 */
kvgqa_status prefill_varlen_gqa_cached_rows_out_(const kvgqa_tensor* q, const kvgqa_tensor* k,
                                                 const kvgqa_tensor* v, const kvgqa_tensor* offsets,
                                                 const kvgqa_tensor* lengths, const kvgqa_tensor* cache_rows,
                                                 double theta, float scale, const kvgqa_tensor* k_cache,
                                                 const kvgqa_tensor* v_cache, const kvgqa_tensor* out,
                                                 const kvgqa_tensor* workspace, void* stream);

/*
 * Slot table and step metadata (host side, no kernels).
 *
 * microLLM-rocm ARCHITECTURE.md, section "Tensor ownership boundary": a
 * continuous-batch scheduler owns the request-to-row map of the shared slot
 * cache; it admits only at step boundaries, resets a row when its request
 * ends (length, stop or cancel) and reuses the lowest free slot; CPU-origin
 * token/position/row metadata of a step travel in one [3,A] host-to-device
 * copy, split on the device into zero-copy views.
 *
 * kvgqa_slots_create    a table of num_slots rows of max_seq positions.
 * kvgqa_slots_admit     lowest free row for `request`, whose row will hold
 *                       prompt_len tokens (the prefill writes them); an
 *                       admitted request keeps its row.  KVGQA_EFULL when no
 *                       row is free.
 * kvgqa_slots_release   free the request's row (reason 0 stop, 1 length,
 *                       2 cancel); KVGQA_EINVAL for an unknown request.
 * kvgqa_slots_step      one decode step for n admitted requests in the
 *                       caller's order: writes token i, its position (the
 *                       row's length) and its row into meta[0][i], meta[1][i],
 *                       meta[2][i] of a host int32 [3][capacity] array, then
 *                       advances every length; a row that becomes full is
 *                       released (reason length) and flagged in finished[i]
 *                       (may be NULL).  Unknown, repeated or full requests
 *                       fail with KVGQA_EINVAL and change nothing.
 * kvgqa_slots_query     rows in use, free rows, and releases per reason.
 * kvgqa_metadata_upload one cudaMemcpyAsync of the whole host [3][capacity]
 *                       int32 array (pinned memory for an asynchronous copy)
 *                       into a device int32 tensor [3, capacity]; rows 1 and
 *                       2 of that tensor, cut to the step's A entries, are the
 *                       positions and cache_rows of the decode calls.
 * The table is not thread-safe; one scheduler thread owns it.
 */
typedef struct kvgqa_slots kvgqa_slots;
kvgqa_status kvgqa_slots_create(int32_t num_slots, int32_t max_seq, kvgqa_slots** out);
kvgqa_status kvgqa_slots_destroy(kvgqa_slots* slots);
kvgqa_status kvgqa_slots_admit(kvgqa_slots* slots, int64_t request, int32_t prompt_len, int32_t* row);
kvgqa_status kvgqa_slots_release(kvgqa_slots* slots, int64_t request, int32_t reason);
kvgqa_status kvgqa_slots_step(kvgqa_slots* slots, const int64_t* requests, const int32_t* tokens, int32_t n,
                              int32_t* meta, int32_t capacity, uint8_t* finished);
kvgqa_status kvgqa_slots_query(const kvgqa_slots* slots, int32_t* active, int32_t* free_rows,
                               int64_t released[3]);
kvgqa_status kvgqa_metadata_upload(const int32_t* host_meta, int32_t capacity, const kvgqa_tensor* device_meta,
                                   void* stream);

/* Opt-in: synchronise `stream`, return the status word of `workspace` in
 * *flags (KVGQA_FLAG_* bits; 0 = every device-side check passed) and clear it.
 * When KVGQA_FLAG_TIMEOUT is among them, the whole workspace is zero-filled
 * (a call that gave up on a wait may have left split-K counters short of
 * their count), so it is ready for any call again.  This is the only call
 * that waits for the device. */
kvgqa_status kvgqa_read_status(const kvgqa_tensor* workspace, void* stream, int32_t* flags);

/* Diagnostic: check on the device that the library's waits end.  Launches on
 * `stream` one CTA that holds tensor memory and waits, with the bounded wait
 * every kernel here uses, on an mbarrier nothing ever arrives on.  After the
 * bound (2 s) the wait gives up and sets KVGQA_FLAG_TIMEOUT in the status word
 * of `workspace`; the CTA frees its tensor memory and returns, and the
 * context stays usable (the same path a kernel takes when a copy or MMA it
 * waits for never completes).  No counterpart in the pages: a test hook.
 *   workspace  >= 256 bytes, 256-byte aligned, device memory (status word set)
 * Read the result with kvgqa_read_status(). */
kvgqa_status kvgqa_check_bounded_wait(const kvgqa_tensor* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVGQA_H_ */
