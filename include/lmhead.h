/*
 * lmhead.h -- C ABI of the GB300 (sm_103a) fused LM-head scoring library.
 *
 * What it computes, for hidden states h[N,H] and an LM-head weight W[V,H]
 * (bf16, row-major), targets y[N] and a keep mask keep[N]:
 *
 *   for every kept row i (keep[i] != 0), with z = h[i] W^T (never stored):
 *     lse[i]      = log sum_v exp(z_v)
 *     logprob[i]  = z_{y[i]} - lse[i]
 *     entropy[i]  = -sum_v p_v log p_v,       p = softmax(z)
 *   and for a gradient g_lp[i] on logprob and g_ent[i] on entropy:
 *     dz_v        = g_lp (1[v = y] - p_v) - g_ent p_v (log p_v + entropy)
 *     dhidden[i]  = dz W            dW += dz^T h[i]
 *   skipped rows get logprob = entropy = lse = 0, dhidden = 0, and add
 *   nothing to dW.
 *
 * Sources (cited by page title and section):
 *   [P1] prime-rl pull request #3326, "Don't compute the logprobs and their
 *        gradients for tokens no loss component reads": maintainer comment
 *        (the FLOPs are in the [N,H] x [H,V] vocab matmul) and "Overview"
 *        (keep mask = union of RL loss mask, CE weights and ref-KL weights
 *        after the next-token shift; compact -> chunked logprob/entropy ->
 *        expand with zeros; token chunk 8192).
 *   [P2] SkyRL pull request #2374, "feat(megatron): fuse LM-head entropy for
 *        RL": "How it works" (one projection gives log-prob and entropy;
 *        metric-only entropy adds no gradient work; entropy-loss mode keeps
 *        the entropy derivative) and the gemini-code-assist review (entropy
 *        = -(p log p) over the vocabulary; the backward reuses the forward
 *        entropy instead of recomputing it).
 *   [P3] twinkle pull request #283, "Fix three memory defects in the Megatron
 *        path", section 1 "selective_log_softmax pins one full-vocab copy per
 *        row": float32 results for bf16 input; chunked work; softmax
 *        recomputed in backward rather than saved.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers on the current CUDA device,
 *     allocated and owned by the caller.  The library never allocates device
 *     memory (the caller passes a workspace) and keeps no per-call state,
 *     except the library-wide scratch array of lmhead_compact_noalloc
 *     (described there).
 *     A pointer that is neither device memory of the current device nor
 *     managed memory (a host pointer, another GPU's memory) is refused with
 *     LMHEAD_EINVAL before anything is launched.
 *   - Matrices are row-major and contiguous.  hidden, weight (and dhidden)
 *     must be 16-byte aligned; H must be a multiple of 8.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  A host-detectable error is returned at once
 *     and nothing is launched.  Errors found on the device (a target out of
 *     range on a kept row, a pipeline wait that ran out) are recorded in a
 *     status word inside the workspace; lmhead_get_status() reads it.
 *   - No C++ exception crosses this boundary and the library never exits the
 *     process.
 *   - Outputs are float32 (logprob, entropy, lse, dW) and bf16 (dhidden).
 *     Results are deterministic: each output element is written once per
 *     launch, and dW's accumulation over chunks adds each element once per
 *     chunk (a TMA reduce-add at L2), chunk after chunk in a fixed order.
 *   - Environment, read on every call: LMHEAD_GEMM = "single", "pair" or
 *     "wide" runs all four contractions on the one-CTA (128 x 256 tiles),
 *     CTA-pair (256 x 256 tiles, two accumulators) or wide CTA-pair (256 x
 *     512 tiles, one accumulator) tcgen05 kernel; unset, dHidden and dW run on
 *     wide tiles when H spans an even number of 256-column tiles, and
 *     everything else on 256 x 256 tiles, unless LMHEAD_WIDE names
 *     the contractions on wide tiles ("fwd,dz,dh,dw" or a subset, "none").
 *     LMHEAD_DH_SPLIT = 1 .. 4 caps the K parts of the dHidden tiles of a
 *     partly filled last wave (default 4; 1 never splits K).  The variants
 *     accumulate in the same order and differ at most by which dHidden tiles
 *     are split (the tile count differs by variant).  LMHEAD_FAULT =
 *     "tensor_map", "launch" or "stall" makes the next calls fail on purpose
 *     for tests: a tensor-map encode or a launch reports LMHEAD_ECUDA, or the
 *     GEMM producers issue no loads so that the bounded pipeline waits run
 *     out (LMHEAD_ETIMEOUT).
 */
#ifndef LMHEAD_H
#define LMHEAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LMHEAD_OK = 0,
  LMHEAD_EINVAL = 1,       /* bad argument: NULL / non-device pointer, size,
                              alignment                                       */
  LMHEAD_EWORKSPACE = 2,   /* workspace smaller than lmhead_workspace_size()   */
  LMHEAD_ETARGET = 3,      /* (device) a kept row's target is outside [0, V)   */
  LMHEAD_ECUDA = 4,        /* a CUDA runtime call failed                       */
  LMHEAD_ETIMEOUT = 5,     /* (device) a pipeline wait gave up; results invalid*/
  LMHEAD_EUNSUPPORTED = 6, /* the current device is not an sm_103 GPU          */
  LMHEAD_EBOUNDS = 7       /* (device) an index outside its array was skipped:
                              a caller's index (lmhead_expand), or in the
                              LMHEAD_DEBUG build any checked internal index  */
} lmhead_status;

/* Opaque cudaStream_t. */
typedef void* lmhead_stream_t;

/* Default rows per chunk of kept tokens ([P1] Overview: token chunk 8192). */
#define LMHEAD_DEFAULT_CHUNK_ROWS 8192

/*
 * Bytes of device workspace that lmhead_fwd / lmhead_bwd / lmhead_compact
 * need for these sizes (the same figure serves all three).  chunk_rows <= 0
 * selects LMHEAD_DEFAULT_CHUNK_ROWS.  The figure grows as
 * O(N + C*(H + V)) with C = chunk_rows: it never holds [N, V] logits
 * ([P3] section 1: memory scales with chunks, not with rows).
 * Returns 0 for invalid sizes (N < 0, H or V < 1).
 * The figure never decreases with N, so a workspace sized for N_max serves
 * every call with N <= N_max (same H, V, chunk_rows): each call lays the
 * workspace out from its own N.  Calls that share a workspace must not
 * overlap on the GPU (order them on one stream): it holds their intermediate
 * buffers and their status word.
 */
size_t lmhead_workspace_size(int64_t N, int H, int V, int want_entropy, int chunk_rows);

/*
 * Keep mask after the next-token shift ([P1] Overview).
 *   loss_mask, ce_weight, kl_weight : float32 [N] token-aligned loss
 *       components, each nullable (NULL = reads no token).  Any non-zero
 *       value counts as "read".
 *   seq_offsets : int32 [n_seq + 1], ascending, seq_offsets[0] = 0 and
 *       seq_offsets[n_seq] = N: the packed sequences.
 *   keep (out)  : uint8 [N]; keep[i] = 1 iff row i+1 is in the same sequence
 *       as row i and some component is non-zero at token i+1.
 */
lmhead_status lmhead_build_keep_mask(const float* loss_mask, const float* ce_weight,
                                     const float* kl_weight, const int32_t* seq_offsets,
                                     int32_t n_seq, int64_t N, uint8_t* keep,
                                     lmhead_stream_t stream);

/*
 * Stable stream compaction of the kept rows ([P1] Overview: "compact").
 *   keep      : uint8 [N], nullable (NULL = every row kept).
 *   targets   : int64 [N]; only kept rows are read and must lie in [0, V)
 *               (else the device status becomes LMHEAD_ETARGET and the
 *               compacted target is stored as 0).
 *   idx (out)       : int32 [N]; idx[0..Nk) = kept rows in ascending order.
 *   targets_c (out) : int32 [N]; targets_c[k] = targets[idx[k]].
 *   d_nk (out)      : int32 [1] on the device: Nk.
 *   workspace       : >= lmhead_workspace_size(N, 1, 1, 0, 0) bytes.
 */
lmhead_status lmhead_compact(const uint8_t* keep, const int64_t* targets, int64_t N, int V,
                             int32_t* idx, int32_t* targets_c, int32_t* d_nk,
                             void* workspace, size_t ws_bytes, lmhead_stream_t stream);

/*
 * Forward: logprob, entropy and lse of every row ([P2] How it works, [P3]
 * section 1).  Only the kept rows are projected; the vocab matmul runs on the
 * tensor cores in bf16 with float32 accumulation and an online-softmax
 * epilogue, chunk_rows kept rows at a time; no [N, V] buffer exists.
 *   hidden  : bf16 [N, H]     weight : bf16 [V, H]     targets : int64 [N]
 *   keep    : uint8 [N], nullable (NULL = all rows kept)
 *   logprob, lse (out) : float32 [N]
 *   entropy (out)      : float32 [N]; may be NULL iff want_entropy == 0
 *                        (then it is not computed).
 *   Skipped rows get +0.0 in every output.
 */
lmhead_status lmhead_fwd(const void* hidden, const void* weight, const int64_t* targets,
                         const uint8_t* keep, int64_t N, int H, int V, int want_entropy,
                         float* logprob, float* entropy, float* lse, int chunk_rows,
                         void* workspace, size_t ws_bytes, lmhead_stream_t stream);

/*
 * Backward of L = sum_i grad_logprob[i] logprob[i] + grad_entropy[i] entropy[i]
 * ([P2] How it works and gemini-code-assist review; [P3] section 1).  The
 * logits are recomputed tile by tile from hidden and weight; lse and entropy
 * are the forward's outputs (not recomputed).
 *   hidden, weight, targets, keep, N, H, V : as passed to lmhead_fwd.
 *   lse     : float32 [N] from lmhead_fwd.
 *   entropy : float32 [N] from lmhead_fwd; read only when grad_entropy is
 *             given (may be NULL otherwise).
 *   grad_logprob : float32 [N].
 *   grad_entropy : float32 [N], nullable: NULL = metric-only entropy, no
 *             entropy term in the gradient.
 *   dhidden (out): bf16 [N, H]; rows of skipped tokens are written as 0.
 *   dweight (out): float32 [V, H]; overwritten when dw_accumulate == 0,
 *             added to when dw_accumulate != 0 (gradient accumulation).
 */
lmhead_status lmhead_bwd(const void* hidden, const void* weight, const int64_t* targets,
                         const uint8_t* keep, int64_t N, int H, int V, const float* lse,
                         const float* entropy, const float* grad_logprob,
                         const float* grad_entropy, void* dhidden, float* dweight,
                         int dw_accumulate, int chunk_rows, void* workspace, size_t ws_bytes,
                         lmhead_stream_t stream);

/*
 * Largest N accepted by lmhead_compact_noalloc (4096 scan blocks of 4096 rows).
 */
#define LMHEAD_NOALLOC_MAX_ROWS 16777216

/*
 * lmhead_compact_noalloc -- the same stable compaction as lmhead_compact, for
 * callers that cannot allocate device memory.  (The pages have no counterpart
 * of this entry point; it exists for such callers only.)
 *
 * Who needs it: code that has no device allocator of its own -- a plugin or
 * hook running inside a framework whose caching allocator owns the GPU's
 * memory, or a service that reserves all its memory at start-up and must not
 * call cudaMalloc later (cudaMalloc can synchronise the device and can fail
 * with out-of-memory mid-run).  Instead of a caller workspace, its scratch
 * (the per-block kept-row counts, 16 KiB) is a fixed array inside the library
 * that every GPU loading the library holds until the process exits.  The call
 * performs no cudaMalloc/cudaFree and calls no allocating library routine.
 *
 *   keep, targets, N, V, idx, targets_c, d_nk : as for lmhead_compact.
 *   d_status (out) : int32 [1] on the device; set to 0 by the call, then to
 *                    LMHEAD_ETARGET if a kept row's target is outside [0, V).
 *   Returns LMHEAD_EINVAL for N > LMHEAD_NOALLOC_MAX_ROWS (and for the
 *   argument errors of lmhead_compact), LMHEAD_EUNSUPPORTED off sm_103.
 *
 * The first call on a device looks up the array's device address (a one-time
 * set-up per device and CUDA context, done with that device current; a new
 * context on the device, e.g. after cudaDeviceReset, gets a fresh look-up);
 * make that first call before any stream capture.  Every call on a device
 * shares the one array and it keeps the last call's contents: calls whose
 * work overlaps on the GPU (e.g. on two streams at once) race and must be
 * ordered by the caller.
 */
lmhead_status lmhead_compact_noalloc(const uint8_t* keep, const int64_t* targets, int64_t N,
                                     int V, int32_t* idx, int32_t* targets_c, int32_t* d_nk,
                                     int32_t* d_status, lmhead_stream_t stream);

/*
 * Block-sparse form (tile skipping in place; [P2] "How it works": block-sparse
 * forward and backward skip inactive tiles instead of compacting).  Same
 * arguments, results and workspace as lmhead_fwd / lmhead_bwd; instead of
 * compacting kept rows, the 256-row tiles of the batch that hold at least one
 * kept row are scored where they lie (hidden is read in place, no gather or
 * scatter); rows of those tiles that are not kept get the same zeros and add
 * nothing to dW.  It does the work of every row of an active tile, so it pays
 * off only when kept rows come in tile-aligned spans.
 */
lmhead_status lmhead_fwd_blocksparse(const void* hidden, const void* weight,
                                     const int64_t* targets, const uint8_t* keep, int64_t N,
                                     int H, int V, int want_entropy, float* logprob,
                                     float* entropy, float* lse, int chunk_rows, void* workspace,
                                     size_t ws_bytes, lmhead_stream_t stream);
lmhead_status lmhead_bwd_blocksparse(const void* hidden, const void* weight,
                                     const int64_t* targets, const uint8_t* keep, int64_t N,
                                     int H, int V, const float* lse, const float* entropy,
                                     const float* grad_logprob, const float* grad_entropy,
                                     void* dhidden, float* dweight, int dw_accumulate,
                                     int chunk_rows, void* workspace, size_t ws_bytes,
                                     lmhead_stream_t stream);

/*
 * Vocabulary-parallel form ([P2] gemini-code-assist review: with the LM head
 * split over the vocabulary, each rank reduces its own logits and one
 * exchange after the loop completes the log-softmax and the entropy; greptile
 * / cursor reviews: the fused op returns the rank-local dZ W hidden gradient
 * and the caller reduces it).  A rank holds W[v_begin : v_begin + V_shard].
 *
 * lmhead_fwd_shard: per kept row, the shard's partial reduction
 *     partials[i] = (m, s, u, t) with m = max_v z_v, s = sum exp(z_v - m),
 *     u = sum exp(z_v - m)(z_v - m), t = z_y if y is in the shard else -inf;
 *     float32 [N, 4], 16-byte aligned; skipped rows get (-inf, 0, 0, -inf).
 *   targets are global vocabulary ids, checked against [0, V_total).
 *   Other arguments as for lmhead_fwd (V = V_shard).
 * lmhead_merge_shards: partials of all shards, float32 [num_shards, N, 4]
 *   (e.g. gathered across ranks by the caller), -> logprob, entropy, lse
 *   [N] (skipped rows +0.0).
 * lmhead_bwd_shard: as lmhead_bwd for the shard, with the merged (whole
 *   vocabulary) lse and entropy; dhidden_partial (bf16 [N, H]) receives this
 *   shard's dZ W_shard, to be summed over shards by the caller; dweight_shard
 *   is float32 [V_shard, H].
 */
lmhead_status lmhead_fwd_shard(const void* hidden, const void* weight_shard,
                               const int64_t* targets, const uint8_t* keep, int64_t N, int H,
                               int V_shard, int64_t v_begin, int64_t V_total, int want_entropy,
                               float* partials, int chunk_rows, void* workspace,
                               size_t ws_bytes, lmhead_stream_t stream);
lmhead_status lmhead_merge_shards(const float* partials, int num_shards, const uint8_t* keep,
                                  int64_t N, int want_entropy, float* logprob, float* entropy,
                                  float* lse, lmhead_stream_t stream);
lmhead_status lmhead_bwd_shard(const void* hidden, const void* weight_shard,
                               const int64_t* targets, const uint8_t* keep, int64_t N, int H,
                               int V_shard, int64_t v_begin, int64_t V_total, const float* lse,
                               const float* entropy, const float* grad_logprob,
                               const float* grad_entropy, void* dhidden_partial,
                               float* dweight_shard, int dw_accumulate, int chunk_rows,
                               void* workspace, size_t ws_bytes, lmhead_stream_t stream);

/*
 * Expand compacted per-row values back to all rows ([P1] Overview: expand
 * back, skipped positions get zeros).
 *   src  : float32 [Nk]   idx : int32 [Nk] (from lmhead_compact)
 *   d_nk : int32 [1] on the device (from lmhead_compact)
 *   dst (out) : float32 [N]; dst[idx[k]] = src[k], +0.0 elsewhere.
 *   d_status (out, nullable) : int32 [1] on the device.  idx and d_nk come
 *            from the caller: an entry of idx outside [0, N), or Nk > N, is
 *            skipped (nothing is written for it) and sets *d_status to
 *            LMHEAD_EBOUNDS (the caller clears it).
 */
lmhead_status lmhead_expand(const float* src, const int32_t* idx, const int32_t* d_nk,
                            int64_t N, float* dst, int32_t* d_status, lmhead_stream_t stream);

/* Element types of a logit matrix. */
#define LMHEAD_DTYPE_BF16 0
#define LMHEAD_DTYPE_F32 1

/*
 * Scoring of logits that already exist ([P3] section 1, the chunked float32
 * `selective_log_softmax`): for every kept row i of a logit matrix z[N, V],
 *   lse[i] = log sum_v exp(z_iv), logprob[i] = z_{i,y_i} - lse[i],
 *   entropy[i] = -sum_v p_iv log p_iv, computed and returned in float32 (no
 *   bf16 quantisation of the log-prob).  Bound by HBM bandwidth (one read of
 *   the logits).
 *   logits : [N, V] row-major with row stride ld elements (ld >= V), element
 *            type logits_dtype (LMHEAD_DTYPE_BF16 or LMHEAD_DTYPE_F32).  16-byte
 *            aligned rows take the vectorised path; others are still correct.
 *   targets, keep : as for lmhead_fwd (keep nullable = all rows kept).
 *   logprob, lse (out) : float32 [N]; entropy (out) float32 [N], may be NULL
 *            iff want_entropy == 0.  Skipped rows get +0.0.
 *   d_status (out, nullable) : int32 [1] on the device, set to LMHEAD_ETARGET
 *            if a kept row's target is outside [0, V) (the caller clears it);
 *            such a row is scored against target 0.
 */
lmhead_status lmhead_selective_log_softmax_fwd(const void* logits, int logits_dtype, int64_t ld,
                                               const int64_t* targets, const uint8_t* keep,
                                               int64_t N, int V, int want_entropy,
                                               float* logprob, float* entropy, float* lse,
                                               int32_t* d_status, lmhead_stream_t stream);

/*
 * Backward of the above: dlogits[i, v] = g_lp (1[v = y] - p) - g_ent p (log p + H)
 * with p recomputed from the logits and the forward's lse and entropy
 * ([P3] section 1: the softmax is recomputed, not saved).
 *   lse, entropy : float32 [N] from the forward (entropy read only when
 *            grad_entropy is given).
 *   grad_logprob : float32 [N]; grad_entropy : float32 [N], nullable.
 *   dlogits (out) : [N, V] of the logits' element type, row stride ld_out;
 *            rows of skipped tokens are written as 0.  May not alias logits.
 */
lmhead_status lmhead_selective_log_softmax_bwd(const void* logits, int logits_dtype, int64_t ld,
                                               const int64_t* targets, const uint8_t* keep,
                                               int64_t N, int V, const float* lse,
                                               const float* entropy, const float* grad_logprob,
                                               const float* grad_entropy, void* dlogits,
                                               int64_t ld_out, int32_t* d_status,
                                               lmhead_stream_t stream);

/*
 * Device-side status of the last lmhead_* call that used this workspace:
 * synchronises `stream`, then returns LMHEAD_OK, LMHEAD_ETARGET or
 * LMHEAD_ETIMEOUT (or LMHEAD_ECUDA if the stream reports an error).
 */
lmhead_status lmhead_get_status(const void* workspace, lmhead_stream_t stream);

/*
 * Where the last call on this workspace ran out of time, if it did (the
 * LMHEAD_ETIMEOUT of lmhead_get_status): synchronises `stream` and returns
 * 0 if no pipeline wait gave up, else (site << 24) | cta with cta the index
 * of the first CTA whose wait gave up and site the wait --
 *   1 a TMA producer waiting for a free shared-memory stage,
 *   2 the MMA issuer waiting for the epilogue to release an accumulator,
 *   3 the MMA issuer waiting for a filled stage,
 *   4 an epilogue warp waiting for a finished accumulator,
 *   5 a producer letting its last loads land before the CTA exits,
 *   6 the MMA issuer letting its last MMAs finish before the CTA exits.
 * Returns -1 for a NULL workspace or a failed CUDA call.  A diagnostic: it
 * names the wait that gave up when a run reports LMHEAD_ETIMEOUT.
 */
int32_t lmhead_get_timeout_record(const void* workspace, lmhead_stream_t stream);

/*
 * Device address (int32, 1 element) where lmhead_fwd / lmhead_bwd /
 * lmhead_compact leave Nk, the number of kept rows of their last call on this
 * workspace -- for logging the kept-token fraction Nk/N ([P1] Overview:
 * perf/lm_head_token_fraction) without synchronising the host.  NULL for a
 * NULL workspace.  The value is valid once that call has completed on its
 * stream.
 */
const int32_t* lmhead_workspace_kept_rows(const void* workspace);

/* Human-readable name of a status code (static string). */
const char* lmhead_strerror(lmhead_status status);

/*
 * Diagnostics (no effect on results).
 *   lmhead_profile_enable(1) makes later calls record a CUDA event pair around
 *   every kernel launch; lmhead_profile_read() synchronises on those events
 *   and reports, per kernel kind k (0 <= k < lmhead_profile_kinds()), the
 *   launches and their summed device milliseconds since the last read, then
 *   clears them.  lmhead_profile_kind_name(k) names kind k.
 *   lmhead_launch_count() is the number of kernels this library has launched
 *   in the process so far.
 */
void lmhead_profile_enable(int on);
int lmhead_profile_kinds(void);
const char* lmhead_profile_kind_name(int kind);
lmhead_status lmhead_profile_read(int64_t* launches, double* total_ms);
int64_t lmhead_launch_count(void);

/* Library version string. */
const char* lmhead_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LMHEAD_H */
