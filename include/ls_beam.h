/*
 * ls_beam — hierarchical ("coarse-select, then fine-rank") beam-search step and
 * beam-cache refresh for NVIDIA GB300 (sm_103a).
 *
 * Method: LightSeq inference article (31duo.com, itemid-283120), section on the
 * hierarchical rewrite of decoding.  Per beam, a first traversal of the logits
 * computes log_sum_exp and an "R-top-k" threshold (split the logits into groups,
 * take each group's max, the k-th largest of those maxima never exceeds the true
 * k-th largest logit).  A second traversal keeps the logits at or above R-top-k,
 * rescores them as beam_score + logit - log_sum_exp and queues them on the device;
 * one sort of that short queue per batch yields the exact top-k (token, parent
 * beam, score) of every sequence.  The article then refreshes the cache by parent
 * beam (its latency breakdown figure puts that at 10% / 6% of inference).
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers unless the argument says "host".
 *    The caller owns every buffer; the library allocates nothing.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Calls are stream-ordered and return once the work is enqueued; nothing here
 *    synchronises except ls_read_status / ls_read_row_stats.
 *  - Argument errors are found on the host before anything is enqueued and return
 *    LS_ERR_INVALID_ARG.  A failed CUDA launch returns LS_ERR_CUDA.  Conditions the
 *    GPU detects (a bounded wait that ran out, an out-of-range parent index) set a
 *    status word in the workspace, read with ls_read_status.
 *  - Buffer extents cannot be checked through this interface: each array must hold
 *    at least the elements its comment states.
 */
#ifndef LS_BEAM_H
#define LS_BEAM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LS_API __attribute__((visibility("default")))
#else
#define LS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LS_OK = 0,
  LS_ERR_INVALID_ARG = 1, /* bad argument, found on the host; nothing enqueued */
  LS_ERR_UNSUPPORTED = 2, /* valid request outside what the library supports */
  LS_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  LS_ERR_TIMEOUT = 4,     /* a bounded device wait ran out (reported by ls_read_status) */
  LS_ERR_INTERNAL = 5     /* device-detected inconsistency, e.g. a parent index out of range */
} ls_status;

typedef enum { LS_DTYPE_F32 = 0, LS_DTYPE_F16 = 1, LS_DTYPE_BF16 = 2 } ls_dtype;

/* Largest beam width supported. */
#define LS_MAX_K 64

/*
 * Bytes of device workspace ls_beam_step needs for (batch, k, vocab).  Host-only,
 * needs no GPU.  Returns 0 for arguments ls_beam_step would reject.
 * Follows the article's memory-reuse rule (every dynamic shape gets a static
 * maximum and buffers are allocated once, at start-up): allocate the workspace once
 * for the largest shape served and reuse it for every step of that or a smaller shape.
 */
LS_API size_t ls_beam_step_workspace_size(int batch, int k, int vocab);

/*
 * Zero-fill a workspace (enqueued on `stream`).  Required once before the first
 * ls_beam_step on it, and again after any call reported a device error.
 * workspace: device, workspace_bytes long.
 */
LS_API ls_status ls_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * One beam-search step (article: hierarchical decoding — first traversal, second
 * traversal into the candidate queue, then one sort of the queue per batch).
 *
 *  logits      [batch, k, vocab] row-major, logit_dtype (f32, f16 or bf16), device.
 *              Any address aligned to the element size; 16-byte alignment is fastest.
 *  bias        [vocab] f32 or NULL; added to every beam's logits before anything else.
 *  beam_scores [batch, k] f32 accumulated log-probabilities of the live beams.
 *  finished    [batch, k] uint8 0/1 or NULL (= none finished).  A finished beam
 *              contributes exactly one candidate, (eos_id, its beam score unchanged),
 *              and its logits are not read.
 *  eos_id      in [0, vocab).
 *  k           beam width, 1 <= k <= LS_MAX_K, k <= vocab; k * vocab < 2^31.
 *  out_token, out_parent  [batch, k] int32: token id in [0, vocab) and parent beam in [0, k).
 *  out_score   [batch, k] f32: beam_score[parent] + x - lse[parent], x = logit + bias.
 *  out_finished [batch, k] uint8 or NULL: finished[parent] || token == eos_id.
 *  Per batch the k outputs are the exact top-k of all k*vocab (beam, token) pairs,
 *  sorted by descending score; equal scores are ordered by parent beam, then by the
 *  larger logit, then by the smaller token id.  A beam whose scores are all -inf
 *  (beam score -inf, or every logit -inf) offers tokens 0, 1, ... with score -inf.
 *  NaN or +inf inputs are not supported (no fault; the result is unspecified).
 *  workspace   device buffer of at least ls_beam_step_workspace_size(batch, k, vocab)
 *              bytes, zero-filled once by ls_workspace_init.  Calls that share a
 *              workspace must be ordered (same stream, or synchronised).
 *  batch == 0 is a no-op.
 */
LS_API ls_status ls_beam_step(const void* logits, ls_dtype logit_dtype, const float* bias,
                       const float* beam_scores, const uint8_t* finished, int batch, int k,
                       int vocab, int eos_id, int32_t* out_token, int32_t* out_parent,
                       float* out_score, uint8_t* out_finished, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * The beam step fused into the output projection that produces its logits (the step
 * before the article's first traversal, which reads the [batch, k, vocab] logits the
 * projection wrote).  logits = hidden . weight^T are accumulated on the tensor cores a
 * tile at a time and never stored: each tile's epilogue runs the first traversal on it
 * (per beam and chunk of 256 to 1024 tokens the max, the sum of exp and the group
 * maxima, and the candidates at or above the chunk's R-top-k bound), then the fine rank of
 * ls_beam_step runs on those candidates.
 *
 *  hidden      [batch, k, dim] row-major, dtype, device, 16-byte aligned: each beam's last
 *              decoder state.
 *  weight      [vocab, dim] row-major, dtype, device, 16-byte aligned: the projection,
 *              one row per token (x[v] = hidden . weight[v] + bias[v]).
 *  dtype       LS_DTYPE_F16 or LS_DTYPE_BF16, both operands.  The products are exact and
 *              are summed in f32 on the tensor cores in an unspecified order, so a logit
 *              differs from the exact dot product by a few f32 roundings of partial sums of
 *              at most sum_d |hidden[d] * weight[v, d]|.
 *  dim         hidden size: a multiple of 8, at least 8.
 *  k           1 <= k <= 32 (k up to LS_MAX_K returns LS_ERR_UNSUPPORTED).
 *  All other arguments, the results (outputs, order, ties, finished beams, -inf) and the
 *  workspace (ls_beam_step_workspace_size(batch, k, vocab) bytes, shared with ls_beam_step)
 *  are those of ls_beam_step with x = logit + bias.  The rows of finished beams are
 *  multiplied but not used.  Argument errors return LS_ERR_INVALID_ARG with nothing
 *  enqueued; a device wait that runs out is reported by ls_read_status.
 */
LS_API ls_status ls_logits_beam_step(const void* hidden, const void* weight, ls_dtype dtype, int dim,
                                     const float* bias, const float* beam_scores,
                                     const uint8_t* finished, int batch, int k, int vocab, int eos_id,
                                     int32_t* out_token, int32_t* out_parent, float* out_score,
                                     uint8_t* out_finished, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * Beam-cache refresh by parent beam (article: "update the cache" after selection):
 *   dst[l, b*k+j, h, p, :] = src[l, b*k + parent[b*k+j], h, p, :]   for p < len.
 * Layout [layers, batch*k, heads, max_len, head_dim], element size from dtype
 * (the copy is bitwise).  Positions p >= len of dst are not written.
 * src and dst must not overlap (ping-pong buffers).  parent [batch, k] int32 in [0, k);
 * an out-of-range parent leaves that row of dst unwritten and, when `workspace` is
 * not NULL, sets LS_ERR_INTERNAL in its status word.  workspace: NULL or a workspace
 * initialised by ls_workspace_init (only its status word is used).
 * len == 0 or an empty shape is a no-op.
 */
LS_API ls_status ls_cache_reorder(const void* src, void* dst, ls_dtype dtype, const int32_t* parent,
                           int layers, int batch, int k, int heads, int max_len, int len,
                           int head_dim, void* workspace, void* stream);

/*
 * Beam-cache refresh in place, copy on change (article: "update the cache" after the
 * selection): for every row j whose parent is not j itself,
 *   cache[l, b*k+j, h, p, :] = (state before the call) cache[l, b*k + parent[b*k+j], h, p, :]
 * for p < len; rows with parent[b*k+j] == j and positions p >= len are not touched.  The
 * result on [0, len) equals ls_cache_reorder from a copy of the cache.
 *
 * cache [layers, batch*k, heads, max_len, head_dim] of dtype, device; parent [batch, k]
 * int32 in [0, k), device; k <= LS_MAX_K.  An out-of-range parent leaves that row as it is
 * and, when `workspace` is not NULL, sets LS_ERR_INTERNAL in its status word.  workspace:
 * NULL or a workspace initialised by ls_workspace_init.  Of it the call uses the status word
 * and, for the bulk-copy kernel, a work counter in bytes 64-71 from which its CTAs take their
 * items; each launch leaves the counter at zero, so calls that share a workspace must be
 * ordered (one stream, or events).  Without a workspace each CTA takes a fixed share of the
 * items.  len == 0 or an empty shape is a no-op.  Nothing is allocated.
 */
LS_API ls_status ls_cache_refresh_inplace(void* cache, ls_dtype dtype, const int32_t* parent, int layers,
                                          int batch, int k, int heads, int max_len, int len, int head_dim,
                                          void* workspace, void* stream);

/*
 * One beam-search step followed by the in-place cache refresh by its parents (article:
 * hierarchical decoding, then "update the cache"): the result equals ls_beam_step and then
 * ls_cache_refresh_inplace(cache, ..., out_parent, ...) on the same stream.  The arguments
 * are those of the two calls; out_parent is required.
 *
 * By default the two run as two launches.  With LS_BEAM_DEBUG=steprefresh, where the step
 * of each batch runs in one CTA (k <= 8 and batch large enough to fill the GPU), that CTA
 * refreshes its own batch's rows as soon as it has ranked them, so the refresh of early
 * batches overlaps the step of the others.  On c5 that form measured slower (7.49 against
 * 6.83 ms per 64-step search: the per-batch refresh inherits the step's two batches per
 * SM, while the standalone refresh spreads over every SM).  A bounded wait of that refresh
 * that runs out sets LS_ERR_TIMEOUT in the workspace's status word (read with
 * ls_read_status).  The cache must not overlap any other argument.  Nothing is allocated.
 */
LS_API ls_status ls_beam_step_refresh_inplace(const void* logits, ls_dtype logit_dtype, const float* bias,
                                              const float* beam_scores, const uint8_t* finished, int batch, int k,
                                              int vocab, int eos_id, int32_t* out_token, int32_t* out_parent,
                                              float* out_score, uint8_t* out_finished, void* cache,
                                              ls_dtype cache_dtype, int layers, int heads, int max_len, int len,
                                              int head_dim, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Workspace bytes for ls_sample on `rows` rows of `vocab` logits keeping top_k candidates
 * (0 for unsupported shapes: top_k outside [1, LS_MAX_K] or above vocab).
 */
LS_API size_t ls_sample_workspace_size(int rows, int top_k, int vocab);

/*
 * Sampling decoding (article: decoding by sampling, next to beam search): one token per
 * sequence from the top_k candidates of its logits, optionally cut to the top-p prefix,
 * drawn by inverse CDF at the caller's uniform.  The first traversal is the beam step's:
 * log_sum_exp and the R-top-k bound in one pass over the logits, then only the logits at
 * or above the bound are ranked.
 *
 *  logits      [rows, vocab] row-major, logit_dtype, device; bias [vocab] f32 or NULL,
 *              added first (x = logit + bias).
 *  u           [rows] f32 uniforms in [0, 1), device (the random numbers are the caller's).
 *  top_k       1..LS_MAX_K, <= vocab: the top_k tokens by x (ties: smaller token id first)
 *              with probabilities proportional to exp(x), renormalised over them.
 *  top_p       in (0, 1]: below 1, only the shortest prefix of those (best first) whose
 *              cumulative probability reaches top_p is kept and renormalised.
 *  out_token   [rows] int32: the first kept candidate whose cumulative probability
 *              exceeds u.
 *  out_logprob [rows] f32 or NULL: x(token) - log sum_v exp(x_v) over the whole row.
 *  workspace   device, >= ls_sample_workspace_size(rows, top_k, vocab) bytes, zero-filled
 *              once by ls_workspace_init; calls sharing it must be ordered.
 *  rows == 0 is a no-op.  NaN or +inf logits are not supported.
 */
LS_API ls_status ls_sample(const void* logits, ls_dtype logit_dtype, const float* bias, const float* u,
                           int rows, int vocab, int top_k, float top_p, int32_t* out_token,
                           float* out_logprob, void* workspace, size_t workspace_bytes, void* stream);

/*
 * End of a search: the token sequence of every final beam, read back through the
 * per-step parent pointers (article: decoding keeps, for every new beam, the beam it
 * continued — the same parent index the cache refresh follows).
 *
 *  token_hist, parent_hist  [steps, batch, k] int32, device: the out_token / out_parent of
 *              decode steps 1..steps (step t's beam j appended token_hist[t, b, j] to beam
 *              parent_hist[t, b, j] of step t-1).
 *  out_seq     [batch, k, steps] int32, device: out_seq[b, j, t] = the token final beam j
 *              of batch b took at step t (final beams in the order of the last step, i.e.
 *              best first).
 *  out_len     [batch, k] int32, device: 1 + the first t whose token is eos_id, or steps.
 *  workspace   NULL, or a workspace initialised by ls_workspace_init: a parent outside
 *              [0, k) on a walked path then sets LS_ERR_INTERNAL in its status word (the
 *              walk stays in bounds; that beam's output is unspecified).
 *  steps == 0 or batch == 0 is a no-op.  Buffers are caller-owned; nothing is allocated.
 */
LS_API ls_status ls_backtrack(const int32_t* token_hist, const int32_t* parent_hist, int steps, int batch,
                              int k, int eos_id, int32_t* out_seq, int32_t* out_len, void* workspace,
                              void* stream);

/*
 * Synchronise `stream`, return the status the device recorded in `workspace` since
 * the last read, and clear it.  LS_OK when nothing was recorded.
 */
LS_API ls_status ls_read_status(void* workspace, void* stream);

/* Static description of a status code. */
LS_API const char* ls_status_string(ls_status status);

/*
 * Diagnostic readback of the last ls_beam_step on `workspace` (synchronises `stream`).
 * All outputs are HOST arrays, each may be NULL:
 *   lse      [batch*k] f32 log_sum_exp of each live beam (NaN for finished beams)
 *   rtopk    [batch*k] f32 the beam's R-top-k threshold (the k-th largest of its
 *            group maxima; -inf when fewer than k groups hold a value)
 *   ncand    [batch*k] int32 candidates of that beam that entered the final sort
 *            (-1 when the batch took the exact fallback)
 *   path     [batch]   int32 0 = candidate queue, 1 = exact fallback (queue overflow),
 *            2 = exact fallback (forced for testing), 3 = exact fallback (large queue)
 */
LS_API ls_status ls_read_row_stats(const void* workspace, int batch, int k, int vocab, float* lse,
                            float* rtopk, int32_t* ncand, int32_t* path, void* stream);

/*
 * The beam step for callers that cannot allocate device memory (no counterpart in the
 * article; it exists for callers such as plugins of a host framework that owns all
 * device memory, or serving loops with a fixed memory budget, where cudaMalloc is not
 * available at request time).  Same arguments and results as ls_beam_step, without the
 * workspace: the scratch lives in a fixed 64 MiB array in this library's device memory,
 * held by every GPU that loads the library until the process exits.  The library
 * allocates nothing here either.
 *  - Shapes whose ls_beam_step_workspace_size exceeds 64 MiB return LS_ERR_UNSUPPORTED.
 *  - The first call on a device looks up that device's address of the array (the
 *    device must be current); make that first call before any stream capture.
 *  - All calls share the one array, which keeps the last call's contents; its status
 *    word is cleared at the start of each call, and ls_beam_step_noalloc_status reads it
 *    for the call before.  Calls whose work overlaps on the GPU (different streams, or
 *    threads without ordering) race on it.
 *  - Argument errors return LS_ERR_INVALID_ARG before anything is enqueued, as for
 *    ls_beam_step.  After cudaDeviceReset the library is not used on that device again
 *    (its device code, the array included, went with the context).
 */
LS_API ls_status ls_beam_step_noalloc(const void* logits, ls_dtype logit_dtype, const float* bias,
                                      const float* beam_scores, const uint8_t* finished, int batch,
                                      int k, int vocab, int eos_id, int32_t* out_token,
                                      int32_t* out_parent, float* out_score, uint8_t* out_finished,
                                      void* stream);

/*
 * Device-detected status of the last ls_beam_step_noalloc on the current device (no
 * counterpart in the article): synchronises `stream`, returns what the device recorded in
 * the fixed array's status word since that call began (LS_OK, or e.g. LS_ERR_TIMEOUT when a
 * bounded device wait ran out) and clears it.  Read it after the call and before the next
 * one, which clears the word again.  LS_ERR_CUDA if the array cannot be reached.
 */
LS_API ls_status ls_beam_step_noalloc_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LS_BEAM_H */
