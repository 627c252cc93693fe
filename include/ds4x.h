/*
 * ds4x.h — C ABI of libds4x.so, the GB300 (sm_103a) implementation of the
 * DeepSeek V4 Flash sparse-attention "lightning indexer" hot path:
 *
 *     score  ->  top-k (k_top = 512)  ->  sparse multi-query attention
 *
 * Sources for what the path computes:
 *   [K]  "How I made DeepSeek 12x faster on a Mac Studio", section "1: the kernels":
 *        the lightning indexer scores compressed KV and keeps the top 512 rows per
 *        token (PRs #830/#831 = the scorer, #832 = the streaming top-k whose output
 *        is byte-identical to a full sort).
 *   [S]  "How I turned one oversized DeepSeek optimization into three merged oMLX
 *        PRs", section "The three changes that merged", item 3 (PR #2563): when every
 *        pooled row fits inside index_topk, scoring and top-k are skipped and the
 *        sequential indices are emitted.
 *   [A]  same page, item 1 (PR #2559): attention over pooled compressed rows chosen
 *        by an index list.
 *   The pages never print the indexer formula; this library's definition is
 *        score[t,s] = sum_h w[t,h] * ReLU( q[t,h,:] . k[s,:] )
 *   with row s visible to a token at position p iff (s+1)*ratio <= p+1, top-k ties
 *   broken toward the lower row index, indices emitted in ascending row order, and
 *   the attention  out[t,h,:] = sum_j softmax_j(scale * q_attn[t,h,:].kv[idx_j,:]) kv[idx_j,:]
 *   (kv is both key and value; softmax in fp32).
 *
 * Conventions shared by every entry point
 *   - Every tensor argument is a DEVICE pointer to a dense row-major array owned by the
 *     caller; the library allocates nothing and keeps no state between calls.
 *     Pointers must be 16-byte aligned.
 *   - fp16 / bf16 tensors are passed as raw 16-bit storage (const void*).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Every call is asynchronous on that stream; calls on different streams that
 *     write disjoint outputs may run concurrently.
 *   - Arguments are validated on the host before anything is launched. On a
 *     validation error nothing is launched and no output is touched.
 *   - Return value: DS4X_OK, or a negative ds4x_status (see ds4x_status_string).
 *     DS4X_ERR_CUDA is returned when a launch fails (the CUDA error is left for the
 *     caller to inspect with cudaGetLastError / cudaPeekAtLastError).
 *   - There is no CPU fallback: unsupported shapes return DS4X_ERR_UNSUPPORTED.
 *
 * Visibility:  n_vis(p) = min(S, floor((p+1)/ratio)) rows are visible to a token at
 *              position p (positions are int32; a negative position sees no row).
 */
#ifndef DS4X_H
#define DS4X_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { DS4X_F16 = 0, DS4X_BF16 = 1 } ds4x_dtype;

typedef enum {
  DS4X_OK = 0,
  DS4X_ERR_INVALID = -1,     /* null/misaligned pointer, negative size, bad ld, ...  */
  DS4X_ERR_UNSUPPORTED = -2, /* a shape this library has no kernel for               */
  DS4X_ERR_CUDA = -3,        /* a kernel launch or device query failed              */
  DS4X_ERR_WORKSPACE = -4,   /* workspace_bytes smaller than the *_workspace_bytes() */
  DS4X_ERR_TIMEOUT = -5      /* a bounded device-side wait gave up                  */
} ds4x_status;

/* Shapes the kernels accept (anything else -> DS4X_ERR_UNSUPPORTED):
 *   indexer heads H in {16, 32, 64, 128}, indexer dim D in {64, 128}
 *   attention heads Hq = 64, attention dim Dkv = 512
 *   1 <= k_top <= DS4X_MAX_KTOP                                                  */
#define DS4X_MAX_KTOP 1024
/*   0 <= window <= DS4X_MAX_WINDOW for the local-plus-pooled entries                 */
#define DS4X_MAX_WINDOW 1024

/* ---------------------------------------------------------------------------
 * ds4x_indexer_score — the lightning-indexer scorer ([K] #830/#831).
 *
 *   scores[t*ld_scores + s] = sum_h w[t,h] * max(0, sum_d q[t,h,d]*k[s,d])  if s < n_vis(positions[t])
 *                           = -INFINITY                                      if n_vis <= s < S
 *   columns S..ld_scores-1 are not written.
 *
 *   q          [T, H, D] fp16          w  [T, H] fp16        k [S, D] fp16
 *   positions  [T] int32                scores [T, ld_scores] fp32, ld_scores >= S
 *   ratio >= 1.  The head products are accumulated in fp32 on the tensor cores and the
 *   head sum in fp32; the full T x H x S product tensor never reaches memory.
 *   T == 0 or S == 0 is a no-op.
 * ------------------------------------------------------------------------- */
int ds4x_indexer_score(const void* q, const void* w, const void* k, const int32_t* positions,
                       int32_t T, int32_t H, int32_t D, int32_t S, int32_t ratio,
                       float* scores, int64_t ld_scores, void* stream);

/* ---------------------------------------------------------------------------
 * ds4x_topk — per-token exact top-k_top of the visible scores ([K] #832, [S] #2563).
 *
 *   For token t with n = n_vis(positions[t]):
 *     n <= k_top : indices[t,:] = 0, 1, ..., n-1, then -1 padding (scores are not read)
 *     n >  k_top : the k_top rows s < n with the largest scores[t*ld+s], ties broken by
 *                  the lower row index, emitted in ascending row order.
 *   counts[t] = min(n, k_top) when counts != NULL.
 *
 *   scores [T, ld_scores] fp32 (only s < n_vis is read)   indices [T, k_top] int32
 *   counts [T] int32 or NULL
 *   workspace: device scratch of at least ds4x_topk_workspace_bytes(T, S, k_top) bytes
 *   (may be NULL when that is 0).  Undefined for NaN scores.
 * ------------------------------------------------------------------------- */
int ds4x_topk(const float* scores, int64_t ld_scores, const int32_t* positions,
              int32_t T, int32_t S, int32_t ratio, int32_t k_top,
              int32_t* indices, int32_t* counts,
              void* workspace, size_t workspace_bytes, void* stream);

size_t ds4x_topk_workspace_bytes(int32_t T, int32_t S, int32_t k_top);

/* ---------------------------------------------------------------------------
 * ds4x_topk_static_scratch — ds4x_topk for callers that cannot allocate device memory.
 * No counterpart on the pages: a convenience of this library.
 *
 *   Same arguments and results as ds4x_topk, minus the workspace.  Meant for callers that must
 *   not allocate device memory at call time (a serving process that gave all of HBM to its KV
 *   cache at start-up, a plugin running under a host framework that owns the allocator) and so
 *   cannot hand over a workspace.  The candidate lists of the split mode (one long row spread
 *   over many CTAs) live instead in a fixed array of DS4X_TOPK_STATIC_SCRATCH_BYTES compiled
 *   into the library; every GPU that loads the library holds that array until the process exits.
 *   - Calls needing more than that (ds4x_topk_workspace_bytes(T, S, k_top) > the maximum) return
 *     DS4X_ERR_WORKSPACE and launch nothing.  The split mode is used only while T is below the
 *     GPU's SM count and rows are longer than 8192, so the need is 0 for T >= SM count: e.g. at
 *     262144-row rows, T = 1..35 fits, T = 36..(SM count - 1) is refused and larger T runs one CTA
 *     per token without any scratch.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 *     that device current); make that first call before any stream capture.
 *   - Allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *   - All calls on a device share the one array: calls that overlap on the GPU (different streams,
 *     no ordering between them) race on it and must not be issued.  Sequential calls are fine; a
 *     call never reads what an earlier call left in the array.
 * ------------------------------------------------------------------------- */
#define DS4X_TOPK_STATIC_SCRATCH_BYTES (4u << 20)
int ds4x_topk_static_scratch(const float* scores, int64_t ld_scores, const int32_t* positions,
                             int32_t T, int32_t S, int32_t ratio, int32_t k_top,
                             int32_t* indices, int32_t* counts, void* stream);

/* ---------------------------------------------------------------------------
 * ds4x_sparse_attn — multi-query attention over the selected compressed rows ([A]).
 *
 *   For token t, head h, over the valid entries j of indices[t, 0..k_top-1]
 *   (valid = 0 <= idx < S; -1 padding and out-of-range entries are skipped):
 *     l_j          = scale * sum_d q_attn[t,h,d] * kv[idx_j, d]
 *     out[t,h,:]   = sum_j exp(l_j - m) kv[idx_j,:] / sum_j exp(l_j - m),   m = max_j l_j
 *     lse[t,h]     = m + log(sum_j exp(l_j - m))
 *   A token with no valid entry gets out = 0 and lse = -INFINITY.
 *
 *   q_attn [T, Hq, Dkv] and kv [S, Dkv] and out [T, Hq, Dkv] all of `dtype`
 *   indices [T, k_top] int32      lse [T, Hq] fp32 or NULL
 *   Softmax statistics in fp32; the probabilities enter the second product in `dtype`;
 *   out is rounded to `dtype` with round-to-nearest-even.
 * ------------------------------------------------------------------------- */
int ds4x_sparse_attn(const void* q_attn, const void* kv, ds4x_dtype dtype,
                     const int32_t* indices, int32_t T, int32_t Hq, int32_t Dkv,
                     int32_t S, int32_t k_top, float scale,
                     void* out, float* lse, void* stream);

/* ---------------------------------------------------------------------------
 * ds4x_index_and_attend — the whole path for one chunk of query tokens:
 *   score (only for tokens with n_vis > k_top: the [S] shortcut) -> top-k -> attention.
 *   Equal to ds4x_indexer_score + ds4x_topk + ds4x_sparse_attn with the same arguments;
 *   the scores live only in `workspace` (at least ds4x_workspace_bytes(T, S, k_top)).
 *   q, w, k fp16 as in ds4x_indexer_score; q_attn, kv, out of kv_dtype.
 *   When the tokens fill less than half of the GPU's SMs (2T <= SM count, e.g. decode), the
 *   attention of each token is split over several CTAs by chunks of its selected rows and the
 *   parts are merged by their softmax statistics.  Each part is normalized by its own row sum
 *   and stored in kv_dtype (a convex combination of kv rows: inside the dtype's range), so out
 *   and lse then differ from the unsplit result by fp32 rounding order and that one rounding of
 *   the parts.  The workspace holds
 *   [scores T x S fp32 | top-k scratch | split-attention scratch] (256-byte aligned parts).
 * ------------------------------------------------------------------------- */
int ds4x_index_and_attend(const void* q, const void* w, const void* k, const int32_t* positions,
                          const void* q_attn, const void* kv, ds4x_dtype kv_dtype,
                          int32_t T, int32_t H, int32_t D, int32_t S, int32_t ratio,
                          int32_t k_top, int32_t Hq, int32_t Dkv, float scale,
                          int32_t* indices, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, void* stream);

size_t ds4x_workspace_bytes(int32_t T, int32_t S, int32_t k_top);

/* ---------------------------------------------------------------------------
 * ds4x_index_and_attend_host — ds4x_index_and_attend on HOST buffers: the inputs are copied
 *   to the device, the path runs, the outputs are copied back, and the copies overlap the
 *   work.  The tokens are cut into about n_chunks sub-chunks (0: the library chooses, about 512
 *   tokens each; from four on, a quarter-size first and last sub-chunk are added, since the first
 *   copy in and the last copy out overlap nothing); the sub-chunks' q and q_attn are copied in on an internal stream, computed on
 *   `stream` and their indices and out copied back on a second internal stream, rotating over
 *   three device staging slots, so that both copy directions and the kernels run at once.  The
 *   shared rows k and kv and every token's w and position are copied once, first; every
 *   token's lse is copied back once, last.  Results are those of ds4x_index_and_attend on each
 *   sub-chunk (the same per token).
 *
 *   q, w, positions, q_attn, k, kv: host memory, layouts as in ds4x_index_and_attend.
 *   indices, out, lse (lse may be NULL): host memory, written by the call.
 *   Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to
 *   run asynchronously and overlap; pageable memory gives the same results, serialised.
 *   device_buffer: device memory the call owns for its duration, 16-byte aligned, at least
 *   ds4x_index_and_attend_host_bytes(...) bytes (staging for k, kv, every token's w, position
 *   and lse, three sub-chunks of q, q_attn, indices and out, and the fused workspace).
 *   Ordering: the copies start after all work enqueued on `stream` before the call; on return
 *   everything is enqueued and `stream` waits for the last copy out, so a synchronisation of
 *   `stream` (or any work enqueued on it later) sees the outputs in host memory.  The host
 *   buffers and device_buffer must stay allocated and untouched until then (the copies run after
 *   the call returns).
 *   Errors: as ds4x_index_and_attend; DS4X_ERR_WORKSPACE when device_bytes is too small,
 *   DS4X_ERR_INVALID for NULL or misaligned pointers or n_chunks < 0.
 * ------------------------------------------------------------------------- */
int ds4x_index_and_attend_host(const void* q, const void* w, const void* k, const int32_t* positions,
                               const void* q_attn, const void* kv, ds4x_dtype kv_dtype,
                               int32_t T, int32_t H, int32_t D, int32_t S, int32_t ratio,
                               int32_t k_top, int32_t Hq, int32_t Dkv, float scale,
                               int32_t* indices, void* out, float* lse, int32_t n_chunks,
                               void* device_buffer, size_t device_bytes, void* stream);

size_t ds4x_index_and_attend_host_bytes(int32_t T, int32_t H, int32_t D, int32_t S, int32_t k_top,
                                        int32_t Hq, int32_t Dkv, int32_t n_chunks);

/* ---------------------------------------------------------------------------
 * Local-plus-pooled attention ([A]: ratio-128 compressed attention draws on local and pooled
 * key/value state, and the native kernel takes both in one pass; the ds4.c overview keeps the
 * live raw sliding-window KV rows as state of their own).  The pages give no window size and no
 * joining rule; this library's definition:
 *
 *   the rows of token t (position p = positions[t]) are its valid selected pooled rows
 *   kv[indices[t, j]] (as in ds4x_sparse_attn) followed by the raw window rows kv_local[r] for
 *   every position a = local_pos0 + r with  max(0, p - window + 1) <= a <= p  and  0 <= r < L;
 *   out and lse are the softmax attention of ds4x_sparse_attn over all of these rows at once
 *   (same query, same scale, nothing de-duplicated).
 *
 *   kv_local [L, Dkv] of the kv dtype: raw rows of consecutive positions starting at
 *   local_pos0 >= 0.  For a prefill chunk at positions pos0..pos0+T-1 it holds positions
 *   pos0-window+1 (or 0) .. pos0+T-1: the previous window-1 raw rows and the chunk's own.
 *   Window positions outside the buffer are not attended.  window = 0 or L = 0 gives exactly
 *   the pooled-only result (kv_local may then be NULL).  0 <= window <= DS4X_MAX_WINDOW.
 *   The window rows are extra 64-row chunks of the same kernel, after the pooled ones.
 * ------------------------------------------------------------------------- */

/* Attention alone over the two row sources; arguments otherwise as ds4x_sparse_attn, plus
 * positions [T] int32 (device). */
int ds4x_local_pooled_attn(const void* q_attn, const void* kv, const void* kv_local, ds4x_dtype dtype,
                           const int32_t* indices, const int32_t* positions, int32_t T, int32_t Hq,
                           int32_t Dkv, int32_t S, int32_t k_top, int32_t local_pos0, int32_t L,
                           int32_t window, float scale, void* out, float* lse, void* stream);

/* The whole path with the window: ds4x_index_and_attend's indices, then ds4x_local_pooled_attn.
 * workspace: at least ds4x_workspace_bytes_local(T, S, k_top, window) bytes (the split mode of
 * small T divides the pooled and the window chunks alike); may be NULL when that is 0. */
int ds4x_index_and_attend_local(const void* q, const void* w, const void* k, const int32_t* positions,
                                const void* q_attn, const void* kv, const void* kv_local,
                                ds4x_dtype kv_dtype, int32_t T, int32_t H, int32_t D, int32_t S,
                                int32_t ratio, int32_t k_top, int32_t Hq, int32_t Dkv,
                                int32_t local_pos0, int32_t L, int32_t window, float scale,
                                int32_t* indices, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream);

size_t ds4x_workspace_bytes_local(int32_t T, int32_t S, int32_t k_top, int32_t window);

/* ds4x_index_and_attend_host with the window: kv_local is HOST memory too, copied once with k
 * and kv; device_buffer of at least ds4x_index_and_attend_local_host_bytes(...) bytes. */
int ds4x_index_and_attend_local_host(const void* q, const void* w, const void* k,
                                     const int32_t* positions, const void* q_attn, const void* kv,
                                     const void* kv_local, ds4x_dtype kv_dtype, int32_t T, int32_t H,
                                     int32_t D, int32_t S, int32_t ratio, int32_t k_top, int32_t Hq,
                                     int32_t Dkv, int32_t local_pos0, int32_t L, int32_t window,
                                     float scale, int32_t* indices, void* out, float* lse,
                                     int32_t n_chunks, void* device_buffer, size_t device_bytes,
                                     void* stream);

size_t ds4x_index_and_attend_local_host_bytes(int32_t T, int32_t H, int32_t D, int32_t S,
                                              int32_t k_top, int32_t Hq, int32_t Dkv, int32_t L,
                                              int32_t window, int32_t n_chunks);

/* ---------------------------------------------------------------------------
 * ds4x_compress — the compressor: one pooled row per `ratio` positions, with the partial block
 * carried from call to call as the "frontier" ([S] item 3: the skip path still advances the
 * indexer compressor and its cache; the ds4.c overview keeps "compressor frontier" tensors with
 * the compressed rows).  The pages give no formula; this library's definition:
 *
 *   the sequence is the n_frontier held-over positions (frontier_x, frontier_g) followed by the
 *   T new positions (x, g); block j = sequence positions j*ratio .. j*ratio + ratio - 1, and
 *     rows[j, d] = sum_i a_i x_i[d],   a_i = exp(z_i) / sum_i' exp(z_i'),   z_i = g_i[d] + bias[i, d]
 *   (i = position inside the block; softmax in fp32, rows rounded to `dtype`, equal gates give the
 *   mean).  The (n_frontier + T) % ratio positions after the last full block are copied to
 *   frontier_x_out / frontier_g_out: the next call's frontier.
 *
 *   x, g [T, D] and frontier_x, frontier_g [n_frontier, D] of `dtype` (raw rows and gate logits,
 *   the outputs of the compressor's projections); bias [ratio, D] fp32 (learned per-position
 *   weights); rows [(n_frontier + T) / ratio, D] of `dtype` (e.g. the next rows of k or kv);
 *   frontier_*_out [(n_frontier + T) % ratio, D].  D % 8 == 0, 1 <= ratio <= DS4X_MAX_RATIO,
 *   0 <= n_frontier < ratio.  The outputs must not overlap the inputs (keep two frontier buffers
 *   and swap them between calls).  One launch; HBM-bound (every input byte read once).
 * ------------------------------------------------------------------------- */
#define DS4X_MAX_RATIO 65536
int ds4x_compress(const void* x, const void* g, const float* bias, ds4x_dtype dtype, int32_t T,
                  int32_t D, int32_t ratio, const void* frontier_x, const void* frontier_g,
                  int32_t n_frontier, void* rows, void* frontier_x_out, void* frontier_g_out,
                  void* stream);

/* ---------------------------------------------------------------------------
 * ds4x_decode — the decode loop: n_steps query tokens at consecutive positions
 * pos0, pos0+1, ..., one fused step (ds4x_index_and_attend with T = 1) each, with the
 * compressed rows appended as the positions complete them ([K]: decode at long context;
 * [S]: one pooled row per `ratio` positions).
 *
 *   Before step i (position p = pos0 + i) the loop appends, while S < floor((p+1)/ratio),
 *   the next unused staged rows k_new[a], kv_new[a] (a = 0, 1, ...) at row S of k and kv
 *   and increments S (stopping when the n_new staged rows or the capacity run out; the step
 *   then sees min(S, floor((p+1)/ratio)) rows).  The step writes
 *     positions[i] = p, indices[i, :], out[i, :, :], lse[i, :]  (lse may be NULL)
 *   exactly as ds4x_index_and_attend would for that one token with the current S.
 *
 *   q [n_steps, H, D] fp16, w [n_steps, H] fp16, q_attn [n_steps, Hq, Dkv] kv_dtype
 *   k [capacity, D] fp16 and kv [capacity, Dkv] kv_dtype: rows 0..S0-1 valid on entry,
 *     rows S0.. are overwritten by the appends (read and written by the call)
 *   k_new [n_new, D], kv_new [n_new, Dkv]: staged rows in append order (NULL when n_new = 0)
 *   positions [n_steps] int32 (written), indices [n_steps, k_top] int32, out like q_attn
 *   workspace: at least ds4x_decode_workspace_bytes(capacity, k_top) bytes
 *   S_final (host pointer, may be NULL): receives S after the last step.
 *   Requires pos0 >= 0, H % 8 == 0 and k_top % 4 == 0 (per-step rows stay 16-byte aligned).
 *   The loop runs on the host and only issues kernel launches on `stream` (no synchronization,
 *   no allocation), so a call may be captured into a CUDA graph after a first call on the device.
 * ------------------------------------------------------------------------- */
int ds4x_decode(const void* q, const void* w, const void* q_attn, void* k, void* kv, ds4x_dtype kv_dtype,
                int32_t capacity, int32_t S0, const void* k_new, const void* kv_new, int32_t n_new,
                int32_t pos0, int32_t n_steps, int32_t H, int32_t D, int32_t ratio, int32_t k_top,
                int32_t Hq, int32_t Dkv, float scale, int32_t* positions, int32_t* indices, void* out,
                float* lse, void* workspace, size_t workspace_bytes, int32_t* S_final, void* stream);
size_t ds4x_decode_workspace_bytes(int32_t capacity, int32_t k_top);

/* ---------------------------------------------------------------------------
 * ds4x_decode_local — ds4x_decode with local-plus-pooled attention: each step also attends to the
 * raw rows of its last `window` positions (see ds4x_local_pooled_attn), the decode form of [A]'s
 * local-plus-pooled kernel.
 *
 *   kv_raw [raw_capacity, Dkv] of kv_dtype: row a holds the raw row of position a; rows below
 *   pos0 (the window's history) are the caller's, rows pos0 .. pos0 + n_steps - 1 are written
 *   by the call from kv_raw_new [n_steps, Dkv] (step i's own raw row) before the first step.
 *   raw_capacity >= pos0 + n_steps.  Step i (position p) attends to its selected pooled rows and
 *   to kv_raw rows max(0, p - window + 1) .. p in one softmax; window = 0 is ds4x_decode.
 *   workspace: at least ds4x_decode_local_workspace_bytes(capacity, k_top, window) bytes.
 *   Everything else as ds4x_decode.
 * ------------------------------------------------------------------------- */
int ds4x_decode_local(const void* q, const void* w, const void* q_attn, void* k, void* kv,
                      ds4x_dtype kv_dtype, int32_t capacity, int32_t S0, const void* k_new,
                      const void* kv_new, int32_t n_new, int32_t pos0, int32_t n_steps, int32_t H,
                      int32_t D, int32_t ratio, int32_t k_top, int32_t Hq, int32_t Dkv, float scale,
                      void* kv_raw, int32_t raw_capacity, const void* kv_raw_new, int32_t window,
                      int32_t* positions, int32_t* indices, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, int32_t* S_final, void* stream);
size_t ds4x_decode_local_workspace_bytes(int32_t capacity, int32_t k_top, int32_t window);

/* Human-readable name of a ds4x_status value (static storage, never NULL). */
const char* ds4x_status_string(int status);

/* Number of kernel launches issued by the most recent successful call on this host
 * thread (for launch accounting in benchmarks). */
int ds4x_last_launch_count(void);

/* ---------------------------------------------------------------------------
 * Device status.  Every wait inside the kernels is bounded (about one second); a wait that
 * gives up records DS4X_ERR_TIMEOUT in a status word of the current device and the kernel
 * returns without finishing its work.  ds4x_device_status synchronizes `stream`, returns
 * DS4X_OK or DS4X_ERR_TIMEOUT, and clears the word when `clear` != 0.
 * ------------------------------------------------------------------------- */
int ds4x_device_status(void* stream, int clear);

/* Diagnostic of the timeout path: launches one kernel whose single waiting thread waits on
 * a barrier that nothing completes, giving up after `timeout_ns` nanoseconds; the status
 * word then reads DS4X_ERR_TIMEOUT.  No fault, no hang.  timeout_ns in [1000, 2e9]. */
int ds4x_selftest_bounded_wait(int64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DS4X_H */
