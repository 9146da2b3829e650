/*
 * tri.h -- C ABI of the GB300 KV-cache compression library (libtri.so).
 *
 * The library scores every cached key of every KV head with the TriAttention
 * trigonometric series, keeps a per-head budget of keys under a protected
 * prompt prefix and recent window, compacts K/V in place, and offers the
 * Random Attention variant that keeps a uniform random subset instead of
 * scoring. Every call is asynchronous on the caller's CUDA stream.
 *
 * Sources, cited by page title and section / equation:
 *   [TA] "TriAttention: Efficient Long Reasoning with Trigonometric KV
 *        Compression" (paper summary page), section 3.4.
 *   [TB] the TriAttention blog page (same title), "TriAttention Scoring",
 *        code-level implementation and S_norm paragraphs, "actual flow".
 *   [RA] "Random Attention: Rethinking KV Cache Eviction for Efficient
 *        Reasoning", section 2 (Eq. 2), section 3 (Eq. 3, Algorithm 1),
 *        Appendix F (engine details).
 *
 * Conventions for every entry point
 *   - A "slice" is one (sequence, layer, KV head) row block of the cache;
 *     slice s = (seq * n_layers + layer) * n_kv_heads + head.
 *   - Pointers documented as "device" must be device (or managed) memory
 *     owned by the caller; the library never allocates, frees or retains
 *     caller memory and keeps no per-call state (calls are thread-safe).
 *   - Scratch memory, where an entry point needs it, is passed in by the
 *     caller with its size from the matching *_workspace_bytes() query.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and return TRI_ERR_INVALID_ARG / TRI_ERR_UNSUPPORTED; nothing is
 *     launched in that case. TRI_ERR_CUDA means a launch failed (the CUDA
 *     error is left for the caller's cudaGetLastError()).
 *   - Input faults only visible on the device (n_valid > n_cap, a NaN score,
 *     a malformed keep list) are reported through the caller's optional
 *     device word *dev_status (first error wins, TRI_DEV_* codes); kernels
 *     never trap. A slice with a fault is skipped by the kernel that found
 *     it.
 */
#ifndef TRI_H_
#define TRI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA stream handle, the same type as cudaStream_t (NULL = the legacy
 * default stream). */
typedef struct CUstream_st* tri_stream_t;

typedef enum {
  TRI_OK = 0,
  TRI_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size or budget    */
  TRI_ERR_UNSUPPORTED = 2, /* head_dim, dtype or device not supported          */
  TRI_ERR_CUDA = 3,        /* a kernel launch failed                           */
  TRI_ERR_TIMEOUT = 4      /* reserved: no entry point waits on anything today */
} tri_status;

/* Device status word values (written with atomicCAS from 0, first error wins). */
#define TRI_DEV_OK 0
#define TRI_DEV_NVALID_OVER_CAP 1 /* n_valid[s] > n_cap: slice skipped            */
#define TRI_DEV_NAN_SCORE 2       /* a candidate score was NaN (ranked lowest)    */
#define TRI_DEV_BAD_KEEP 3        /* keep list not ascending / out of range       */
#define TRI_DEV_TIMEOUT 4         /* a bounded in-kernel wait gave up (~2 s)      */
#define TRI_DEV_GROUP_NVALID 5    /* slices sharing a keep list differ in n_valid */
#define TRI_DEV_BAD_BLOCK 6       /* a block table entry is outside [0, num_blocks) */

typedef enum { TRI_F32 = 0, TRI_BF16 = 1 } tri_dtype;

/* How band f pairs two coordinates of a head vector into one complex number:
 * interleaved (x[2f], x[2f+1]) as [TA] "RoPE in complex form" writes it, or
 * half-split (x[f], x[f+d/2]) -- the other rotation style [TB]'s invert_rope
 * call accepts. Both the query statistics and the keys use the same style. */
typedef enum { TRI_ROPE_INTERLEAVED = 0, TRI_ROPE_HALF = 1 } tri_rope_style;

/* Norm term: weighted S_norm = sum_f (1 - R_f) E|q_f| |k_f| ([TA] "Adaptive
 * Weighting via Q/K Concentration"), or the unweighted ablation
 * S_norm^(0) = sum_f E|q_f| |k_f| ([TA] "The Norm-Based Term"). */
typedef enum { TRI_NORM_WEIGHTED = 0, TRI_NORM_UNWEIGHTED = 1 } tri_norm_mode;

/* What the cached K rows hold. Pre-RoPE keys k_i (the form [TA] scores) with
 * their positions in `pos`; or post-RoPE keys k~_i = RoPE(k_i, p_i), band f
 * multiplied by e^{i w_f p_i} in the same pairing style -- what engines store
 * ([TB] "scoring": vLLM keeps post-RoPE K and inverts RoPE before scoring;
 * [RA] Appendix F). For post-RoPE keys the score needs no positions: with
 * k_f = e^{-i w_f p_i} k~_f it is Re sum_f c_f G_f e^{i w_f p_cur} conj(k~_f)
 * + sum_f wgt_f E|q_f| |k~_f|, the same value. */
typedef enum { TRI_KEYS_PRE_ROPE = 0, TRI_KEYS_POST_ROPE = 1 } tri_key_layout;

/* The cache. K and V rows are head_dim elements, contiguous; slice s starts
 * at element s * slice_stride of k (and of v); row i of the slice at element
 * s * slice_stride + i * head_dim. k and v: device, 16-byte aligned,
 * slice_stride * element size a multiple of 16 bytes. */
typedef struct {
  void* k;               /* [n_slices][n_cap][head_dim] keys (see key_layout)    */
  void* v;               /* [n_slices][n_cap][head_dim] values                   */
  int32_t* pos;          /* device [n_slices][n_cap] token positions, or NULL:
                            NULL means position = slot index (a fresh cache)    */
  int32_t* pos_out;      /* device [n_slices][n_cap]: where compaction writes the
                            survivors' positions; may equal pos                 */
  int32_t* n_valid;      /* device [n_slices]: cached rows per slice; compaction
                            sets it to the number kept                          */
  int64_t slice_stride;  /* elements between slices, >= n_cap * head_dim        */
  int32_t n_seq, n_layers, n_kv_heads;
  int32_t n_cap;         /* row capacity of a slice                              */
  int32_t head_dim;      /* 64 or 128                                            */
  tri_dtype dtype;       /* element type of k and v                              */
  int32_t* dev_status;   /* device int32 status word (TRI_DEV_*), or NULL        */
  tri_key_layout key_layout; /* pre- or post-RoPE keys (0 = pre-RoPE)            */
  /* Paged caches (block_table != NULL; [RA] section 6: scoring walks the
   * engine's block tables, and eviction moves the survivors to the front of
   * the request's blocks and returns the unused tail). k and v are then block pools, and
   * logical row r of slice (seq, layer, head) is at element
   *   block_table[seq][r / block_size] * block_stride + layer * layer_stride
   *   + head * head_stride + (r % block_size) * head_dim
   * of k (and of v): every (block, layer, head) holds block_size contiguous
   * rows. One table per sequence, shared by its layers and heads; n_cap =
   * (table entries per sequence) * block_size; slice_stride is ignored. All
   * fields below are ignored when block_table is NULL. */
  const int32_t* block_table; /* device [n_seq][n_cap / block_size], or NULL    */
  int32_t block_size;         /* rows per block: a power of two, at least 16      */
  int32_t num_blocks;         /* blocks per pool; every used entry must be below  */
  int64_t block_stride, layer_stride, head_stride; /* elements; x elem size % 16 == 0 */
} tri_kv;

/* Per-(layer, KV head) query statistics, [TA] "Offline Calibration
 * Procedure"; index lh = layer * n_kv_heads + head, F = head_dim / 2. */
typedef struct {
  float* center;    /* device [n_layers * n_kv_heads][F][2]: E[q_f] (re, im)       */
  float* mean_norm; /* device [n_layers * n_kv_heads][F]:    E|q_f|                */
  float* mrl;       /* device [n_layers * n_kv_heads][F]:    R_f = |E q_f| / E|q_f|*/
} tri_centers;

/* ------------------------------------------------------------------------ */
const char* tri_status_string(tri_status s); /* static text, never NULL */
int32_t tri_abi_version(void);               /* 3 */
/* Kernels this library has launched in this process (all devices, all
 * threads); used to count launches inside a timed region. */
uint64_t tri_launch_count(void);

/* ------------------------------------------------------------------------
 * tri_calibrate_centers -- offline per-head query statistics.
 * [TA] "Offline Calibration Procedure" and "Measurement via Mean Resultant
 * Length": for each layer, KV head h and band f, pooling the `group` query
 * heads h*group .. h*group+group-1 that share KV head h (the reading chosen
 * for GQA: one centre per KV head, as [TB] shapes the norm coefficient
 * [num_kv_heads, freq_count]):
 *   center = mean of q_f (complex), mean_norm = mean of |q_f|,
 *   mrl = |center| / mean_norm (0 when mean_norm is 0).
 * q: device [n_layers][n_q_heads][n_tok][head_dim] pre-RoPE queries of type
 * dtype, 16-byte aligned. n_q_heads must be a multiple of group. Sums are in
 * fp32 with a fixed-order two-level reduction (deterministic).
 * ws: device scratch of at least tri_calibrate_workspace_bytes(...) bytes,
 * 16-byte aligned (may be NULL when that size is 0).
 * ------------------------------------------------------------------------ */
size_t tri_calibrate_workspace_bytes(int32_t n_layers, int32_t n_q_heads, int32_t group,
                                     int32_t head_dim, int64_t n_tok);
tri_status tri_calibrate_centers(const void* q, tri_dtype dtype, int32_t n_layers,
                                 int32_t n_q_heads, int32_t group, int32_t head_dim,
                                 int64_t n_tok, tri_rope_style style, tri_centers out,
                                 void* ws, size_t ws_bytes, tri_stream_t stream);

/* ------------------------------------------------------------------------
 * tri_calibrate_centers_noalloc -- tri_calibrate_centers without scratch.
 * (The pages have no counterpart: this is a convenience of this library.)
 * For callers that cannot allocate device memory: a plugin inside an engine
 * that owns all device memory through its own pool and forbids direct driver
 * allocations, or latency-critical code that must not call cudaMalloc /
 * cudaFree because those can synchronise the device and stall other streams.
 * Same arguments, result and arithmetic as tri_calibrate_centers, minus the
 * scratch: the partial sums go to a fixed array of
 * TRI_CALIBRATE_NOALLOC_MAX_SCRATCH_BYTES bytes inside the library, which
 * every GPU that loads the library holds until the process exits. This call
 * allocates nothing.
 *   - Shapes whose scratch (tri_calibrate_workspace_bytes) exceeds the array
 *     return TRI_ERR_INVALID_ARG before anything is enqueued.
 *   - Every call looks up the array's address in the current device's
 *     context (a host-side query; it stays right after cudaDeviceReset and
 *     under another context). The first call on a device may load the
 *     library's device code there: make that first call before any stream
 *     capture begins.
 *   - All calls share the one array, and each call fully rewrites the part it
 *     reads, so nothing carries over between calls; but calls whose kernels
 *     overlap on the GPU (e.g. on two streams without ordering) race on it.
 * ------------------------------------------------------------------------ */
#define TRI_CALIBRATE_NOALLOC_MAX_SCRATCH_BYTES (4u * 1024u * 1024u)
tri_status tri_calibrate_centers_noalloc(const void* q, tri_dtype dtype, int32_t n_layers,
                                         int32_t n_q_heads, int32_t group, int32_t head_dim,
                                         int64_t n_tok, tri_rope_style style, tri_centers out,
                                         tri_stream_t stream);

/* ------------------------------------------------------------------------
 * tri_score -- offset-averaged TriAttention score of cached keys.
 * For every row i of slice s with n_prompt <= i < n_valid[s] - n_recent
 * (protected rows are not scored and their score entries are left as they
 * were), with p_i its position, age = p_cur[seq] - p_i, and the statistics of
 * the slice's (layer, KV head):
 *   S~(i) = (1/|D|) sum_{delta in D} sum_f |c_f||k_f| cos(w_f (age+delta) + arg c_f - arg k_f)
 *         + sum_f wgt_f E|q_f| |k_f|
 * [TA] "The Trigonometric Series Term" (S_trig), "Adaptive Weighting via Q/K
 * Concentration" (S_norm, wgt_f = 1 - R_f; wgt_f = 1 under
 * TRI_NORM_UNWEIGHTED), "The combined score", "Handling Multiple Future
 * Positions" (average over the future offsets D); w_f = rope_theta^(-2f/d).
 * Computed as the per-band complex multiply-accumulate
 *   Re sum_f (c_f G_f e^{i w_f age}) conj(k_f) + norm term,
 *   G_f = (1/|D|) sum_delta e^{i w_f delta},
 * which is the same quantity ([TB] "implementation in code": the query-side
 * phase carries the distance).
 * offsets: HOST array of n_offsets (1..64) token offsets (D).
 * p_cur: device [n_seq] int64, position of the newest cached token of each
 * sequence (the current query position). With a position array (kv->pos),
 * every valid row's age p_cur - pos[i] must lie in [0, 2^32). scores: device [n_slices][n_cap]
 * fp32. Arithmetic: fp32 FMA; phases in 64-bit fixed-point turns.
 * ------------------------------------------------------------------------ */
tri_status tri_score(const tri_kv* kv, const tri_centers* c, double rope_theta,
                     tri_rope_style style, tri_norm_mode norm_mode, const int32_t* offsets,
                     int32_t n_offsets, const int64_t* p_cur, int32_t n_prompt,
                     int32_t n_recent, float* scores, tri_stream_t stream);

/* ------------------------------------------------------------------------
 * tri_select_topk -- per-slice budgeted selection.
 * If n_valid[s] <= budget nothing is evicted: keep = 0 .. n_valid-1, then -1.
 * Otherwise keep = [0, n_prompt) U top-(budget - n_prompt - n_recent) of the
 * candidates [n_prompt, n_valid - n_recent) by score U [n_valid - n_recent,
 * n_valid), in ascending slot order ([TA] "Retention and eviction"; [RA]
 * Eq. 2 and section 2's never-scored recent buffer; [TB] "actual flow": the
 * prompt is protected; [RA] Appendix F: keep-sets sorted chronologically).
 * Equal scores keep the lower slot; -0 equals +0; NaN ranks lowest and sets
 * TRI_DEV_NAN_SCORE. budget counts every survivor, protected rows included;
 * requires budget >= n_prompt + n_recent.
 * scores: device [n_slices][n_cap]; keep_idx: device [n_slices][budget].
 * ------------------------------------------------------------------------ */
tri_status tri_select_topk(const float* scores, const tri_kv* kv, int32_t n_prompt,
                           int32_t n_recent, int32_t budget, int32_t* keep_idx,
                           tri_stream_t stream);

/* ------------------------------------------------------------------------
 * tri_compact_kv -- in-place, order-preserving compaction.
 * For each slice, with n_keep = the number of leading non-negative entries of
 * keep_idx[s] (ascending, keep_idx[s][j] >= j, < n_cap): for j < n_keep, row
 * j of K and V <- row keep_idx[s][j] (as if done for j ascending, one row at
 * a time); pos_out[s][j] <- pos[s][keep[j]] (or keep[j] when pos is NULL);
 * n_valid[s] <- n_keep. [RA] Appendix F: KV tensors compacted with a gather.
 * Rows >= n_keep keep their old bytes. A malformed keep list sets
 * TRI_DEV_BAD_KEEP and leaves that slice untouched. kv->pos_out required.
 * ------------------------------------------------------------------------ */
tri_status tri_compact_kv(const tri_kv* kv, const int32_t* keep_idx, int32_t budget,
                          tri_stream_t stream);

/* ------------------------------------------------------------------------
 * rand_evict -- Random Attention keep lists (no score is computed).
 * [RA] section 3, Eq. 3 and Algorithm 1: prompt rows score +inf (kept), every
 * other candidate draws an i.i.d. uniform u_i, independently per KV head and
 * per eviction; keep the top (budget - n_prompt - n_recent) by (u desc, slot
 * asc); the recent buffer is kept unscored ([RA] section 2). u_i is word
 * (i mod 4) of Philox-4x32-10 (Salmon et al., SC'11) with
 *   counter = (i / 4, head + 65536 * layer, seq, round),
 *   key     = (low 32 bits of seed, high 32 bits of seed).
 * Output layout and the n_valid <= budget case as tri_select_topk.
 * n_layers must be <= 65535 and n_kv_heads <= 65536.
 * ------------------------------------------------------------------------ */
tri_status rand_evict(const tri_kv* kv, uint64_t seed, uint32_t round, int32_t n_prompt,
                      int32_t n_recent, int32_t budget, int32_t* keep_idx,
                      tri_stream_t stream);

/* ------------------------------------------------------------------------
 * rand_evict_scoped -- rand_evict with the draw shared across heads: [RA]
 * Appendix D's shared-draw control keeps the prompt and uses ONE random
 * keep-set for every head (no cross-head diversity). Scope PER_HEAD is
 * rand_evict; PER_LAYER gives every KV head of a (seq, layer) the draw of
 * head 0 (counter word 1 = 65536 * layer); PER_SEQUENCE gives every head of
 * every layer the draw of (layer 0, head 0) (counter word 1 = 0). Slices that
 * share a draw and have the same n_valid get identical keep lists.
 * ------------------------------------------------------------------------ */
typedef enum { TRI_DRAW_PER_HEAD = 0, TRI_DRAW_PER_LAYER = 1, TRI_DRAW_PER_SEQUENCE = 2 } tri_draw_scope;
tri_status rand_evict_scoped(const tri_kv* kv, uint64_t seed, uint32_t round, tri_draw_scope scope,
                             int32_t n_prompt, int32_t n_recent, int32_t budget, int32_t* keep_idx,
                             tri_stream_t stream);

/* ------------------------------------------------------------------------
 * tri_select_compact -- exactly tri_select_topk then tri_compact_kv with the
 * same arguments, each slice selected and compacted by one CTA in a single
 * launch (one slice's selection overlaps other slices' row traffic; this
 * pays when selecting is cheap next to the rows moved, as for the Random
 * Attention draws).
 * rand_evict_compact -- likewise rand_evict_scoped then tri_compact_kv.
 * keep_idx is written as by the selection; kv->pos_out required.
 * ------------------------------------------------------------------------ */
tri_status tri_select_compact(const float* scores, const tri_kv* kv, int32_t n_prompt, int32_t n_recent,
                              int32_t budget, int32_t* keep_idx, tri_stream_t stream);
tri_status rand_evict_compact(const tri_kv* kv, uint64_t seed, uint32_t round, tri_draw_scope scope,
                              int32_t n_prompt, int32_t n_recent, int32_t budget, int32_t* keep_idx,
                              tri_stream_t stream);

/* ------------------------------------------------------------------------
 * tri_compress -- one compression event: score + select + compact.
 * Exactly tri_score (rows [n_prompt, n_valid - n_recent)), tri_select_topk
 * and tri_compact_kv called in sequence with the same arguments, with the
 * scores kept in caller scratch. When a slice fits one CTA of the score
 * kernel (n_cap at most 4096 rows of 256 B, 8192 of 128 B, ...: 32 tiles of
 * 32 KB) one CTA scores, selects and compacts each slice in a single launch;
 * otherwise the three kernels run in turn.
 * keep_idx: device [n_slices][budget], written as by tri_select_topk.
 * ws: device scratch of at least tri_compress_workspace_bytes(kv) bytes,
 * 16-byte aligned (the scores [n_slices][n_cap]; nothing in it needs to be
 * initialised; the candidates' scores are left there). kv->pos_out required.
 * ------------------------------------------------------------------------ */
size_t tri_compress_workspace_bytes(const tri_kv* kv);
tri_status tri_compress(const tri_kv* kv, const tri_centers* c, double rope_theta,
                        tri_rope_style style, tri_norm_mode norm_mode, const int32_t* offsets,
                        int32_t n_offsets, const int64_t* p_cur, int32_t n_prompt,
                        int32_t n_recent, int32_t budget, int32_t* keep_idx, void* ws,
                        size_t ws_bytes, tri_stream_t stream);

/* ------------------------------------------------------------------------
 * GQA: one score per query head, z-score + max.
 * [TA] "Handling Grouped-Query Attention (GQA)": the G query heads that share
 * a KV head each score every cached key with their own statistics; per head
 * the scores are z-normalised with their mean and standard deviation over all
 * cached keys, and the final score of a key is the maximum over the G heads.
 *
 * tri_score_heads -- for every row 0 <= i < n_valid[s] of every slice and
 * every query head g < group: scores_g[s][g][i] = S~(g)(i), the tri_score
 * formula with the statistics of query head (layer, h * group + g), i.e. row
 * (layer * n_kv_heads + h) * group + g of `centers` (as tri_calibrate_centers
 * writes them with group = 1); and stats[s][g] = (mean, std) of those scores
 * over the n_valid rows (population std: divided by n_valid; 0 and 0 for an
 * empty slice). group: 1..8. scores_g: device [n_slices][group][n_cap] fp32
 * (rows >= n_valid untouched); stats: device [n_slices][group][2] fp32.
 * ws: device scratch of tri_score_heads_workspace_bytes(kv, group) bytes,
 * 16-byte aligned (fp64 per-CTA partial sums; no initial contents needed).
 * bf16 keys: one pass over K for the whole group, the contraction over the
 * heads on the tensor cores with fp16 features (Re z_f, -Im z_f, |k_f|) and
 * each head's coefficients as an fp16 pair (hi + lo): the score's error is
 * at most ~2^-11 * sqrt(2) * sum_f E|q(g)_f| |k_f| plus fp32 rounding. A key
 * band with |k_f| >= 65520 does not fit fp16: its scores come out non-finite
 * and tri_select_topk_zmax reports TRI_DEV_NAN_SCORE. fp32 keys: fp32
 * arithmetic on the CUDA cores, up to four heads per pass over K (ceil(G/4)
 * passes). The statistics are summed in a fixed order (deterministic).
 *
 * tri_select_topk_zmax -- tri_select_topk with the score of candidate i
 * replaced by S_final(i) = max_g (scores_g[s][g][i] - mean_g) / std_g (a head
 * with std 0 contributes 0), computed in fp32 as (x - mean) * (1 / std).
 * final_scores: optional device [n_slices][n_cap]; when not NULL, S_final of
 * every valid row is written there (the values the selection ranked).
 * ------------------------------------------------------------------------ */
size_t tri_score_heads_workspace_bytes(const tri_kv* kv, int32_t group);
tri_status tri_score_heads(const tri_kv* kv, const tri_centers* centers, int32_t group,
                           double rope_theta, tri_rope_style style, tri_norm_mode norm_mode,
                           const int32_t* offsets, int32_t n_offsets, const int64_t* p_cur,
                           float* scores_g, float* stats, void* ws, size_t ws_bytes,
                           tri_stream_t stream);
tri_status tri_select_topk_zmax(const float* scores_g, const float* stats, int32_t group,
                                const tri_kv* kv, int32_t n_prompt, int32_t n_recent,
                                int32_t budget, int32_t* keep_idx, float* final_scores,
                                tri_stream_t stream);

/* ------------------------------------------------------------------------
 * tri_select_union -- one keep list for the n_kv_heads KV heads of each
 * (seq, layer): union-based selection ([TB] "eviction (union-based
 * selection)"):
 *   1. every head h picks its own top k_head candidates by its own score
 *      (as tri_select_topk with budget n_prompt + n_recent + k_head);
 *   2. U = the union of those picks;
 *   3. the B - n_prompt - n_recent kept candidates are U's best by the
 *      combined score, or all of U and the best of the rest when U is smaller;
 *   4. plus [0, n_prompt) and [n - n_recent, n); ascending.
 * Combined score (a reading; the page leaves it open): [TA]'s normalise-then-
 * max, c(i) = max_h (s_h(i) - mean_h) / std_h with mean and population std of
 * each head's scores over all n valid rows (a head with std 0 gives 0),
 * computed in fp32 as (x - mean) * (1 / std); order (in U first, c desc,
 * slot asc). scores: [n_slices][n_cap], EVERY valid row scored (tri_score
 * with n_prompt = n_recent = 0). All heads of a (seq, layer) must hold the
 * same n_valid (else TRI_DEV_GROUP_NVALID). n_kv_heads: 1..8; n_cap <=
 * 524288. keep_idx: [n_slices][budget], identical rows within a group.
 * final_scores: optional [n_seq * n_layers][n_cap], c(i) of every valid row.
 * ws: tri_select_union_workspace_bytes(kv, n_prompt, n_recent, k_head) bytes,
 * 16-byte aligned.
 * ------------------------------------------------------------------------ */
size_t tri_select_union_workspace_bytes(const tri_kv* kv, int32_t n_prompt, int32_t n_recent, int32_t k_head);
tri_status tri_select_union(const float* scores, const tri_kv* kv, int32_t n_prompt, int32_t n_recent,
                            int32_t budget, int32_t k_head, int32_t* keep_idx, float* final_scores, void* ws,
                            size_t ws_bytes, tri_stream_t stream);

/* ------------------------------------------------------------------------
 * tri_paged_blocks_used -- after a compaction of a paged cache: the blocks
 * each sequence still uses, ceil(max over its slices of n_valid / block_size);
 * table entries from there on hold no live row and can go back to the
 * caller's allocator ([RA] section 6: unused tail blocks go back). blocks_used: device
 * [n_seq] int32. Requires a paged cache (block_table != NULL).
 * ------------------------------------------------------------------------ */
tri_status tri_paged_blocks_used(const tri_kv* kv, int32_t* blocks_used, tri_stream_t stream);

/* ------------------------------------------------------------------------
 * tri_selftest_wait_timeout -- a check of the failure path every kernel
 * shares: one thread waits on an mbarrier that nothing arrives on for
 * limit_ns nanoseconds of the GPU's global timer (1000 <= limit_ns <=
 * 1000000000), then sets *dev_status to TRI_DEV_TIMEOUT (first error wins)
 * and returns -- what each bounded in-kernel wait does after about 2 s.
 * The context stays usable. dev_status: device int32, required, 4-byte
 * aligned. Stream-ordered; TRI_ERR_INVALID_ARG for a null status word or a
 * limit out of range (nothing is launched then).
 * ------------------------------------------------------------------------ */
tri_status tri_selftest_wait_timeout(int32_t* dev_status, uint64_t limit_ns, tri_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TRI_H_ */
