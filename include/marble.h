/*
 * marble.h -- C ABI of a single-GPU (GB300, sm_103a) library for exact, mask-aware
 * blockwise attention over packed multimodal sequences, carrying the online-softmax
 * state (O, m, l) in fp32 across a sequence of key/value shards ("ring steps" run
 * back to back on one GPU).
 *
 * Sources for the operations (cited by page title and section):
 *   [MARBLE]  "MARBLE: exact sequence parallelism for packed multimodal masks"
 *             (Luma AI): s01 "Packed multimodal masks" (four per-token tracks and the
 *             mask_mod predicate), s03 "Block classification", "PTRR: balancing ring
 *             attention steps", "Exact ring attention accumulation", s04 "Sparse
 *             all-to-all and strategy selection", "Layout transforms", "Planning cost".
 *   [RING]    "RingAttention and Context Parallelism: Mathematical Foundations ..."
 *             (llms.blog): "The Online Softmax Formulation", "Execution Algorithm".
 *   [LIBRA]   "Libra: Taming Attention Workload Skew ..." (arXiv 2607.23250):
 *             s2.2 Eq. 1 (CoreAttn = softmax(QK^T/sqrt(d_h) + M) V).
 *
 * Conventions for every call
 *   - Pointers named "device" must be CUDA device pointers (or managed memory) on the
 *     device that was current when the plan was created; "host" pointers are ordinary
 *     host memory.  Export/copy calls accept either (the copy direction is inferred).
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream) unless
 *     stated otherwise.  Arguments are validated before anything is launched; an invalid
 *     argument returns MARBLE_ERR_INVALID_ARG and launches nothing.
 *   - The caller owns every tensor it passes.  A plan owns only its own device
 *     workspace: allocated by marble_plan, grown by the backward calls for their scratch
 *     of bf16 dS tiles, and freed by marble_plan_destroy (which keeps up to two dS
 *     scratch buffers per device for later plans).  This memory comes from a
 *     stream-ordered pool the library keeps per device.  The calls that read sizes or
 *     status back to the host (marble_plan, marble_plan_stats, marble_check) do so through
 *     a small pinned host buffer the library keeps per calling thread.  No call allocates
 *     memory that the caller sees.
 *   - No C++ exception crosses this boundary.  marble_last_error() returns a
 *     thread-local, human-readable message for the last failing call on this thread.
 *   - The step-list and fused calls spread launches over up to four side streams of the
 *     library, and plans are freed on a library stream.  With CUDA's default of 8 hardware
 *     work queues (CUDA_DEVICE_MAX_CONNECTIONS) these share queues with the caller's
 *     streams, so that a caller's copy can wait behind unrelated attention kernels; set
 *     CUDA_DEVICE_MAX_CONNECTIONS=32 before the process creates its CUDA context (the
 *     Python binding does so at import unless the variable is set).
 *   - Every wait inside a kernel is bounded in time; a wait that runs out sets an error
 *     word owned by the plan and the kernel returns.  marble_check() reports it as
 *     MARBLE_ERR_TIMEOUT.  Asynchronous CUDA faults surface as MARBLE_ERR_CUDA.
 *
 * Token order and layouts
 *   - The plan's tracks are given in ORIGINAL order; the original position of a token
 *     is its index (pos = index).  marble_plan computes a token permutation (`perm`,
 *     new index -> original index).  All attention tensors below are in the plan's NEW
 *     order: the caller gathers Q/K/V (and dO) with marble_permute first and scatters
 *     results back with marble_permute(..., inverse = 1).
 *   - Virtual shard r holds new tokens [r*N/P, (r+1)*N/P), i.e. new blocks
 *     [r*nb/P, (r+1)*nb/P) with nb = N/128.
 *   - Q, O, dO: bf16 [N, Hq, d]; K, V: bf16 [N, Hkv, d]; token-major, contiguous.
 *     O_acc, dQ_acc: fp32 [N, Hq, d]; dK_acc, dV_acc: fp32 [N, Hkv, d].
 *     m, l, LSE, delta: fp32 [Hq, N].
 *     All base pointers must be 16-byte aligned.
 *   - Grouped-query attention: q head h reads kv head h / (Hq / Hkv).
 *   - Supported head dims: d = 64 and d = 128.  Hq must be a multiple of Hkv.
 */
#ifndef MARBLE_H_
#define MARBLE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *marble_stream_t;

typedef enum {
  MARBLE_OK = 0,
  MARBLE_ERR_INVALID_ARG = 1, /* bad pointer, size, layout or metadata */
  MARBLE_ERR_UNSUPPORTED = 2, /* valid request outside what this build implements */
  MARBLE_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a kernel failed */
  MARBLE_ERR_OOM = 4,         /* plan workspace allocation failed */
  MARBLE_ERR_TIMEOUT = 5      /* a bounded in-kernel wait ran out (see marble_check) */
} marble_status_t;

#define MARBLE_BLOCK 128               /* tokens per block (MARBLE s03) */
#define MARBLE_WINDOW_INF 2147483647   /* W for globally causal layers */
#define MARBLE_TILE_FULL 1             /* every pair provably legal: no mask evaluated */
#define MARBLE_TILE_PARTIAL 2          /* mixed: the mask predicate runs per pair */
#define MARBLE_KV_NEEDED (-1)          /* kv_shard value: every needed KV block at once */
#define MARBLE_STEP_FIRST 1u           /* flags bit: this is the first step of the rows */
#define MARBLE_STEP_BF16_MERGE 2u      /* flags bit: standard ring merge in bf16 (baseline) */
#define MARBLE_STEP_FP32_MERGE 4u      /* flags bit: merge of fp32 partials by their LSE */

typedef enum {
  MARBLE_ORDER_CONTIGUOUS = 0, /* identity order: shard r = contiguous token range */
  MARBLE_ORDER_PTRR_BLOCK = 1, /* PTRR over 128-token blocks (MARBLE s03 "PTRR") */
  MARBLE_ORDER_PTRR_CHUNK = 2, /* PTRR over contiguous chunks of chunk_tokens tokens
                                  (MARBLE s03 "Chunked ring attention") */
  MARBLE_ORDER_CHUNK_SEARCH = 3 /* contiguous chunks, layout searched for the lowest
                                   layout cost C (MARBLE s03 "Chunked ring attention") */
} marble_order_t;

/*
 * Plan descriptor.  MARBLE s01: four integers per token encode the packed mask -- a
 * sample id, a segment id shared by the tokens of one bidirectional span (or of all
 * spans of one image group), a noise-group id for generated spans, and the original
 * position (here: the index).  The predicate is
 *   allowed(q, k) = (0 <= pos[q]-pos[k] < W  or  seg[q] == seg[k] >= 0)
 *                   and (noise[k] < 0 or noise[q] == noise[k]) and sample[q] == sample[k].
 * Requirements (checked; MARBLE_ERR_INVALID_ARG otherwise):
 *   n_tokens > 0, a multiple of 128, < 2^31;
 *   sample_id non-decreasing along the pack and >= 0 (each sample one contiguous run);
 *   seg_id >= -1, noise_id >= -1 (-1 = none);
 *   window >= 0 (MARBLE_WINDOW_INF for global layers);
 *   1 <= num_shards <= 256 and nb % num_shards == 0;
 *   PTRR_CHUNK: chunk_tokens a positive multiple of 128 dividing n_tokens, and the
 *   number of chunks divisible by num_shards.
 *   CHUNK_SEARCH: range_cost >= 0, and n_tokens / 128 divisible by num_shards (one chunk
 *   per rank is always a candidate).  The search (MARBLE s03 "Chunked ring attention"):
 *   W[r, j] = legal (q, k) pairs between rank r's queries and rank j's keys; a layout of k
 *   contiguous chunks per rank costs C = sum_s max_r W[r, (r - s) mod P] + range_cost * P * k.
 *   For k = 1, 2, 4, ..., 64 (equal chunks of whole blocks, at most 1024 chunks in all):
 *   deal the chunks with PTRR's rule once in the order of their work and once in sequence
 *   order, keep the start with the lower first term (the work order on a tie), then swap
 *   chunks between ranks while that strictly lowers it: passes over chunk pairs (a, b),
 *   a < b ascending, first improvement taken, until a pass makes no swap (64 passes at
 *   most).  The lowest C wins, the fewer chunks on a tie; each rank keeps its chunks in
 *   sequence order.  The search runs on the host over pair counts summed on the device.
 * The three track arrays are device int32[n_tokens]; they are read during marble_plan
 * only (the plan keeps its own permuted copy).
 */
typedef struct {
  int64_t n_tokens;
  const int32_t *sample_id;
  const int32_t *seg_id;
  const int32_t *noise_id;
  int32_t window;
  int32_t num_shards;
  int32_t order;        /* marble_order_t */
  int32_t chunk_tokens; /* PTRR_CHUNK only */
  int64_t range_cost;   /* CHUNK_SEARCH only: tau, the fixed cost of one contiguous range in
                           one ring step, in legal pairs */
  int32_t no_key_intervals; /* 1: partial tiles always evaluate the four-track predicate;
                               0 (default): key-interval test where it is exact.  The test is
                               lo_k <= i_q < hi_k with i_q the query's index in the order the
                               tracks are given in (MARBLE s03 "Block classification") */
  const int32_t *pos_id;    /* NULL: a token's position is its index.  Otherwise device
                               int32[n_tokens] >= 0, the original position of every token of
                               a permuted pack (MARBLE s04 "Layout transforms": tokens carry
                               their position), read during marble_plan only.  On globally
                               causal layers (window MARBLE_WINDOW_INF) the key intervals are
                               then computed from the positions: exact for a key when the
                               queries of its sample at a position >= its own form one range
                               of indices (the vision-group layout gives this), when the
                               positions are a permutation of [0, n_tokens) and each sample
                               holds one range of them.  With a window and a position track
                               the interval test is off. */
} marble_plan_desc_t;

typedef struct marble_plan marble_plan_t; /* opaque; immutable after creation */

/*
 * Build a plan on the current device (MARBLE s03 "Block classification", "PTRR";
 * s04 "Sparse all-to-all", "Layout transforms"; s04 "Planning cost": a plan depends only
 * on the metadata and is reused by every layer, forward and backward).
 * Steps, all in CUDA kernels: validate the tracks; per-block summaries (min/max of each
 * track plus a 64-bit segment bitmap); classify every block pair of the candidate band
 * as full / partial / empty from the summaries alone; per-row cost = non-empty tiles;
 * token order (contiguous or PTRR); permuted tracks; per (q block, kv shard) tile lists
 * for the forward and dQ, per (kv block, q shard) lists for dK/dV, and the needed-KV
 * block index of every q shard.
 * Synchronises `stream` a few times (to size its arrays), the last time after its last
 * kernel: the tracks are read only during the call, and their buffers may be reused as soon
 * as it returns.  On success *out owns device memory until marble_plan_destroy.  Errors: INVALID_ARG (descriptor or metadata),
 * UNSUPPORTED, OOM, CUDA.
 */
marble_status_t marble_plan(const marble_plan_desc_t *desc, marble_stream_t stream,
                            marble_plan_t **out);

/* Frees the plan without synchronising: the workspace returns to the library's memory
 * pool in stream order, once the work of every earlier call that used the plan has
 * completed, on whatever streams those calls ran; the plan handle is invalid as soon as
 * the call returns.  The backward's dS^T scratch is kept instead for the backward calls of
 * later plans on the device (at most two such buffers; the stream of the call that takes
 * one waits for the last use by its previous plan), so that a training loop with one plan
 * per batch does not have the pool map a new scratch for every batch.  NULL is accepted.
 * Errors: CUDA (the plan is freed on the host all the same). */
marble_status_t marble_plan_destroy(marble_plan_t *plan);

typedef struct {
  int64_t n_tokens, n_blocks, num_shards;
  int64_t nnz;          /* non-empty tiles */
  int64_t n_full, n_partial;
  int64_t legal_pairs;  /* legal (q, k) pairs of the mask, per head */
  int64_t shard_cost_max, shard_cost_sum; /* non-empty tiles per q shard: max, sum */
  int64_t step_cost;    /* sum_s max_r W[r, (r-s) mod P], W in tiles (MARBLE s03,
                           chunk-layout cost C without the per-range term) */
  int64_t needed_total; /* sum over q shards of needed kv blocks */
  int64_t needed_remote;/* ... of which lie outside the q shard's own kv shard */
  int64_t chunks_per_rank; /* CHUNK_SEARCH: k of the chosen layout (0 for other orders) */
  int64_t layout_cost;  /* CHUNK_SEARCH: its C in legal pairs, range term included */
  int64_t layout_step_cost; /* CHUNK_SEARCH: its sum_s max_r W[r, (r-s) mod P], in pairs */
  int64_t step_cost_pairs;  /* any order: sum_s max_r W[r, (r-s) mod P], W in legal pairs */
} marble_plan_stats_t;

/*
 * The chunk-layout search of MARBLE_ORDER_CHUNK_SEARCH on caller-supplied work, on the
 * host (no device involved): block_pairs is a host int64 [n_blocks][n_blocks] matrix of
 * legal pairs (or any non-negative work) between q block a and kv block b, n_blocks a
 * multiple of num_shards and at most 65536.  Writes out[0] = k (chunks per rank), out[1] =
 * the layout cost C and out[2] = its step cost sum_s max_r W[r, (r-s) mod P], and the rank
 * of every chunk (k * num_shards entries, chunk c = blocks [c, c + 1) * n_blocks / (k *
 * num_shards)) to the host array chunk_rank, which must hold min(n_blocks, 1024) entries.
 * Errors: INVALID_ARG.
 */
marble_status_t marble_chunk_layout_search(const int64_t *block_pairs, int64_t n_blocks,
                                           int32_t num_shards, int64_t range_cost,
                                           int32_t *chunk_rank, int64_t *out);

/*
 * The vision-group layout (MARBLE s04 "Layout transforms"), on the host: for host int32
 * arrays sample[n] and seg[n] of a pack (same rules as marble_plan_desc_t), writes perm[n],
 * new index -> index in the given order.  In every sample the tokens outside image groups
 * come first, in order, then the group spans, the last span first; an image group is a
 * segment id with more than one run of consecutive tokens in the sample, a span one such
 * run.  Apply perm to every per-token array (activations and the three tracks) and pass the
 * tokens' original positions (perm itself, for a pack in position order) as pos_id: the
 * mask is unchanged, and each key's visible queries form one range in the new order.
 * Errors: INVALID_ARG.
 */
marble_status_t marble_layout_vision_groups(const int32_t *sample, const int32_t *seg, int64_t n,
                                            int32_t *perm);

/* Plan statistics; counts legal pairs with a kernel over the partial tiles (full tiles
 * contribute 128*128 each).  Synchronises `stream`. */
marble_status_t marble_plan_stats(const marble_plan_t *plan, marble_stream_t stream,
                                  marble_plan_stats_t *out);

typedef enum {
  MARBLE_FIELD_PERM = 0,         /* int32[N]   new token -> original token */
  MARBLE_FIELD_BLOCK_PERM = 1,   /* int32[nb]  new block -> original block */
  MARBLE_FIELD_TRACKS_PERM = 2,  /* int32[4][N] sample, seg, noise, pos in new order */
  MARBLE_FIELD_TILE_ROWPTR = 3,  /* int64[nb+1] tile map CSR, ORIGINAL block coords */
  MARBLE_FIELD_TILE_COL = 4,     /* int32[nnz]  original kv block, ascending per row */
  MARBLE_FIELD_TILE_TAG = 5,     /* uint8[nnz]  MARBLE_TILE_FULL / MARBLE_TILE_PARTIAL */
  MARBLE_FIELD_STEP_PTR = 6,     /* int64[nb*P+1] list of (new q block i, kv shard j)
                                    at [ptr[i*P+j], ptr[i*P+j+1]) */
  MARBLE_FIELD_STEP_COL = 7,     /* int32[nnz] new kv block, ascending per list */
  MARBLE_FIELD_STEP_TAG = 8,     /* uint8[nnz] */
  MARBLE_FIELD_COLT_PTR = 9,     /* int64[nb*P+1] list of (new kv block k, q shard r)
                                    at [ptr[k*P+r], ptr[k*P+r+1]) */
  MARBLE_FIELD_COLT_ROW = 10,    /* int32[nnz] new q block, ascending per list */
  MARBLE_FIELD_COLT_TAG = 11,    /* uint8[nnz] */
  MARBLE_FIELD_NEEDED_PTR = 12,  /* int64[P+1] */
  MARBLE_FIELD_NEEDED = 13,      /* int32[needed_total] sorted unique new kv blocks that
                                    q shard r's rows need (local blocks included) */
  MARBLE_FIELD_KEY_INTERVALS = 14, /* int32[2][N] new order: lo, hi of every key's
                                      visible-query interval (indices in the order the
                                      tracks were given in) */
  MARBLE_FIELD_INTERVAL_BLOCKS = 15 /* uint8[nb] new order: 1 if every key of the block
                                       has an exact interval */
} marble_field_t;

/* Size in bytes of an exported field (host call, no synchronisation). */
marble_status_t marble_plan_field_bytes(const marble_plan_t *plan, int32_t field,
                                        size_t *bytes);

/* Copy a plan field to `dst` (host or device), asynchronously on `stream`.  `bytes`
 * must equal marble_plan_field_bytes(). */
marble_status_t marble_plan_export(const marble_plan_t *plan, int32_t field, void *dst,
                                   size_t bytes, marble_stream_t stream);

/*
 * Gather (inverse = 0: dst[i] = src[perm[i]]) or scatter (inverse = 1:
 * dst[perm[i]] = src[i]) rows of `row_bytes` bytes per token between original and plan
 * order (MARBLE s04 "Layout transforms").  src and dst are device pointers of
 * N * row_bytes bytes that must not overlap; row_bytes must be a positive multiple of 4
 * and both pointers 16-byte aligned.
 */
marble_status_t marble_permute(const marble_plan_t *plan, const void *src, void *dst,
                               int64_t row_bytes, int32_t inverse, marble_stream_t stream);

/*
 * marble_permute fused with the fp32 -> bf16 cast of marble_cast_bf16, for fp32 results
 * that leave plan order as bf16 (the gradient accumulators): inverse = 1 writes
 * dst[perm[i]] = bf16(src[i]), inverse = 0 writes dst[i] = bf16(src[perm[i]]), rows of
 * `row_elems` elements, each rounded to nearest even (MARBLE s04 "Layout transforms").
 * src: device fp32 [N, row_elems]; dst: device bf16 [N, row_elems]; the two must not
 * overlap.  row_elems must be a positive multiple of 4 and both pointers 16-byte aligned.
 * Errors: INVALID_ARG for a null plan, a bad row_elems, a pointer that is not device
 * memory or not aligned, or overlapping buffers; CUDA if the launch fails.
 */
marble_status_t marble_permute_cast_bf16(const marble_plan_t *plan, const float *src,
                                         void *dst, int64_t row_elems, int32_t inverse,
                                         marble_stream_t stream);

/* Queries, keys and values in plan order (layouts above). scale <= 0 selects 1/sqrt(d)
 * (LIBRA Eq. 1). */
typedef struct {
  const void *q; /* device bf16 [N, hq, d] */
  const void *k; /* device bf16 [N, hkv, d] */
  const void *v; /* device bf16 [N, hkv, d] */
  int32_t hq, hkv, d;
  float scale;
} marble_qkv_t;

/* Online-softmax state of every (token, q head), caller-owned, plan order.
 * o_acc: unnormalised fp32 accumulator [N, hq, d]; m: running row maximum of the
 * scaled scores, kept in base-2 units (score * scale * log2(e)); l: running row sum of
 * exp2(score*scale*log2(e) - m).  (O_acc, m, l) always satisfy O_acc = sum_k 2^(s_k - m) v_k
 * and l = sum_k 2^(s_k - m) over the keys seen so far. */
typedef struct {
  float *o_acc; /* device fp32 [N, hq, d] */
  float *m;     /* device fp32 [hq, N] */
  float *l;     /* device fp32 [hq, N] */
} marble_state_t;

/*
 * One ring step of the forward (MARBLE s03 "Exact ring attention accumulation";
 * RING "The Online Softmax Formulation"): for every row of q shard `q_shard` and every
 * q head, process the tiles the plan lists between the row's block and kv shard
 * `kv_shard` (or, with kv_shard == MARBLE_KV_NEEDED, every tile of the row: one pass
 * over the local and needed remote blocks, MARBLE s04) and update (O_acc, m, l) in
 * fp32.  Full tiles skip the mask; partial tiles evaluate the predicate per pair; empty
 * tiles are never loaded.
 * flags & MARBLE_STEP_FIRST: the state of this shard's rows is uninitialised; every row
 * of the shard starts from (O = 0, m = -inf, l = 0), including rows with no tile in this
 * step (which are written as such).  Otherwise the stored state is resumed.
 * The ring pairing of MARBLE s03 is kv_shard = (q_shard - s) mod P at step s; any order
 * of the P kv shards gives the same result up to fp32 rounding.
 * flags & MARBLE_STEP_BF16_MERGE: instead of carrying the fp32 state, run the standard
 * ring-attention merge that MARBLE s03 compares against: the step's output is normalised
 * and rounded to bf16, then merged with the stored output by log-sum-exp weights and
 * rounded to bf16 again.  O_acc then holds bf16-representable values, m the running
 * log-sum-exp in base 2 (ln -> log2) and l = 1 (0 while a row has seen no legal key), so
 * that marble_attn_finalize gives O and LSE unchanged.
 * flags & MARBLE_STEP_FP32_MERGE: the same merge with no rounding: each step's output is an
 * fp32 partial with its LSE and the partials are merged in fp32 (MARBLE s03 and s06: the
 * route to exactness through fp32 split-KV partials).  O_acc holds the normalised fp32
 * output, m and l as above.
 * At most one of the two merge bits may be set, and every step of a pass over the same rows
 * must carry the same merge bits.
 * Errors: INVALID_ARG (shard out of range, null/misaligned pointer, d not 64/128,
 * hq % hkv != 0), CUDA.
 */
marble_status_t marble_attn_step(const marble_plan_t *plan, const marble_qkv_t *qkv,
                                 int32_t q_shard, int32_t kv_shard,
                                 const marble_state_t *state, uint32_t flags,
                                 marble_stream_t stream);

/*
 * A list of forward ring steps in one call: step i is exactly
 * marble_attn_step(plan, qkv, q_shards[i], kv_shards[i], state, flags[i], stream), launched
 * in list order on `stream` (each step is still its own kernel launch and the state passes
 * through HBM between steps).  The host arrays q_shards, kv_shards, flags hold n_steps
 * entries and are read before the call returns.  Saves per-call validation and tensor-map
 * set-up when a whole ring schedule is issued at once.
 */
marble_status_t marble_attn_steps(const marble_plan_t *plan, const marble_qkv_t *qkv,
                                  int32_t n_steps, const int32_t *q_shards,
                                  const int32_t *kv_shards, const uint32_t *flags,
                                  const marble_state_t *state, marble_stream_t stream);

/*
 * Normalise once at the end (MARBLE s03: "only the last call normalizes the output,
 * writes the LSE and casts to bf16"):  O = O_acc / l as bf16 [N, hq, d] and
 * LSE = ln(sum_k exp(s_k)) = (m + log2 l) * ln 2 as fp32 [hq, N].  A row with l = 0 (no
 * legal key) gives O = 0 and LSE = -inf.  Covers all N tokens.
 */
marble_status_t marble_attn_finalize(const marble_plan_t *plan, const marble_state_t *state,
                                     int32_t hq, int32_t d, void *o_bf16, float *lse,
                                     marble_stream_t stream);

/* Backward preprocessing: delta = rowsum(dO * O) as fp32 [hq, N] from bf16 O and dO
 * (the O emitted by marble_attn_finalize). */
marble_status_t marble_attn_bwd_prep(const marble_plan_t *plan, const void *o,
                                     const void *d_o, int32_t hq, int32_t d, float *delta,
                                     marble_stream_t stream);

/*
 * One ring step of the backward (MARBLE s03: each step runs the attention backward
 * against the FINAL LSE; the fp32 dQ accumulator is carried across steps and each kv
 * shard's fp32 dK/dV accumulators travel with the shard; s03 closing rule: gradients
 * summed across calls are summed in fp32).  For the tiles between q shard `q_shard` and
 * kv shard `kv_shard` (or every tile of the q shard's rows with MARBLE_KV_NEEDED):
 *   P = exp(S*scale - LSE), dV += P^T dO, dP = dO V^T, dS = P * (dP - delta),
 *   dK += scale * dS^T Q, dQ += scale * dS K,
 * accumulated in place into dq_acc [N, hq, d], dk_acc / dv_acc [N, hkv, d] (fp32).
 * The accumulators must be zeroed by the caller before the first step.
 * flags: reserved, pass 0.
 */
marble_status_t marble_attn_bwd(const marble_plan_t *plan, const marble_qkv_t *qkv,
                                const void *d_o, const float *lse, const float *delta,
                                int32_t q_shard, int32_t kv_shard, float *dq_acc,
                                float *dk_acc, float *dv_acc, uint32_t flags,
                                marble_stream_t stream);

/* A list of backward ring steps in one call: step i is marble_attn_bwd(..., q_shards[i],
 * kv_shards[i], ..., flags = 0), with the same result as issuing them in list order on
 * `stream`; host arrays of n_steps entries.  Each step runs a dK/dV kernel, which also
 * writes the step's bf16 dS tiles to a scratch array the plan owns, and a dQ GEMM reads them:
 *   - a list that holds every (q shard, kv shard) pair of the ring exactly once, when the dS
 *     tiles of the whole pack fit the 32 GB scratch cap (nnz tiles x hq x 32 KB): every
 *     step's dK/dV kernel, then ONE dQ GEMM over every q block's whole row, so each dQ row
 *     block is accumulated on chip over all its steps and added to dq_acc once (a q shard's
 *     dQ is local to it on a real ring, so its GEMM may wait for the ring's end);
 *   - such a list in q-shard runs (r-major), when the tiles of two q shards fit the cap: the
 *     same whole-row GEMM per q shard after its last step, a few q shards' tiles held at once;
 *   - otherwise a dQ GEMM after each step, the scratch holding the tiles of up to four steps
 *     (two when four would exceed the cap).
 *   Whole rows are used only while no q block's row is longer than half an SM's share of the
 *   GEMM's tiles (one such unit would set the launch's length).
 * Two environment variables, read on every call, reach the other paths on small packs (tests):
 * MARBLE_DS_SCRATCH_CAP_MB lowers the 32 GB cap; MARBLE_WHOLE_ROWS=always skips the row test.
 * Results differ between the paths only in fp32 summation order.
 * The scratch grows on demand; backward calls on one plan must therefore be ordered with
 * respect to each other.  The launches spread over side streams of the device, forked from
 * `stream` at the start and joined back into it at the end; launches that add into the same
 * dK/dV rows (one kv shard) stay on one stream, so results do not depend on timing. */
marble_status_t marble_attn_bwd_steps(const marble_plan_t *plan, const marble_qkv_t *qkv,
                                      const void *d_o, const float *lse, const float *delta,
                                      int32_t n_steps, const int32_t *q_shards,
                                      const int32_t *kv_shards, float *dq_acc, float *dk_acc,
                                      float *dv_acc, marble_stream_t stream);

/*
 * The whole forward ring in one launch (MARBLE s03 "Exact ring attention accumulation" and
 * "PTRR"; RING "Execution Algorithm"): the same result as marble_attn_steps over every
 * (q_shard r, kv_shard (r - s) mod P, FIRST at s = 0) for s = 0 .. P-1, up to fp32 rounding.
 * Every (q block, q head) of every shard visits its tiles in that ring order, step after
 * step, with its fp32 (O_acc, m, l) held on chip from its first step to its last; the state
 * is written to `state` once, in the form marble_attn_step leaves it (so marble_attn_finalize
 * follows as usual), rows with no tile included.  The state never passes through HBM between
 * steps, and the pass is one persistent launch instead of P^2.  Only the carried fp32 state
 * (no merge flags).  Errors: as marble_attn_steps.
 */
marble_status_t marble_attn_fwd_fused(const marble_plan_t *plan, const marble_qkv_t *qkv,
                                      const marble_state_t *state, marble_stream_t stream);

/*
 * The whole backward ring (MARBLE s03: each kv shard's fp32 dK/dV accumulator travels with
 * the shard around the ring while dQ is carried per q shard): the same result as
 * marble_attn_bwd_steps over every (r, (r - s) mod P), up to fp32 rounding.  For every kv
 * shard j, one dK/dV launch visits the q shards in ring order (j, j + 1, ..., j - 1) and keeps
 * the dK/dV of each of its kv blocks in TMEM across all of them, adding it to dk_acc / dv_acc
 * once.  When the dS tiles of the whole pack fit the 32 GB scratch cap (and the rows balance,
 * as in marble_attn_bwd_steps), one dQ GEMM over every q block's whole row follows all of
 * them.  Otherwise
 * the dQ GEMM of each step (q shard, j) follows its kv shard's launch, and when the dS tiles
 * of a kv shard's whole ring would exceed half of the cap, its ring is split into consecutive
 * ranges of steps, each added once.  Accumulators must be zeroed by the caller; scratch and
 * ordering as marble_attn_bwd_steps.  Errors: as marble_attn_bwd_steps.
 */
marble_status_t marble_attn_bwd_fused(const marble_plan_t *plan, const marble_qkv_t *qkv,
                                      const void *d_o, const float *lse, const float *delta,
                                      float *dq_acc, float *dk_acc, float *dv_acc,
                                      marble_stream_t stream);

/* Cast fp32 -> bf16 (round to nearest even) for n elements, e.g. gradient accumulators;
 * n must be a multiple of 4 and both pointers 16-byte aligned. */
marble_status_t marble_cast_bf16(const float *src, void *dst, int64_t n,
                                 marble_stream_t stream);

/*
 * Synchronise `stream` and report the plan's device error word: MARBLE_ERR_TIMEOUT if a
 * bounded in-kernel wait ran out since the last check (the word is then cleared),
 * MARBLE_ERR_CUDA on an asynchronous CUDA error, MARBLE_OK otherwise.
 */
marble_status_t marble_check(const marble_plan_t *plan, marble_stream_t stream);

/* Upper bound, in nanoseconds, on every in-kernel wait of later launches in this
 * process (default 2e9 ns; also read once from env MARBLE_WAIT_LIMIT_MS). */
marble_status_t marble_set_wait_limit_ns(uint64_t ns);

/*
 * Process-wide cap on the side streams that marble_attn_steps and marble_attn_bwd_steps
 * spread their launches over (default 4, the most they use; 0 runs every launch in list
 * order on the caller's stream).  Results do not depend on it.  Errors: INVALID_ARG if n is
 * outside [0, 4].
 */
marble_status_t marble_set_side_streams(int32_t n);

/*
 * Give back to the device the memory the library keeps for reuse on the current device:
 * the dS^T scratch buffers that destroyed plans left for later plans, and the unused part
 * of the library's memory pool (which otherwise keeps freed blocks for later allocations).
 * Memory of plans that are still alive is not touched.  Waits for the library's teardown
 * stream, so that every free queued by marble_plan_destroy has happened; queues no work on
 * any other stream.  Errors: CUDA.
 */
marble_status_t marble_release_memory(void);

/*
 * Per-kernel device timing, a measurement hook (off by default).  While it is on, every
 * marble_attn_step(s) / marble_attn_bwd(_steps) call records CUDA events, on the stream each
 * kernel runs on, before its first and after its last launch of that kernel, and counts the
 * launches.  marble_timing_read synchronises on those events, adds up their spans since the
 * previous read and writes out[0..5] = forward ms, forward launches, dQ-kernel ms, dQ-kernel
 * launches, dK/dV-kernel ms, dK/dV-kernel launches.  Launches on different streams overlap
 * in time (see marble_set_side_streams), and a launch that waits for SMs held by another
 * stream's launch has that wait in its span; with the side streams capped at 0 every launch
 * runs alone and a span is its duration.  Returns MARBLE_ERR_INVALID_ARG if `out` is null.
 */
marble_status_t marble_timing_enable(int on);
marble_status_t marble_timing_read(double *out);

/* Test hook: launch one CTA that waits, with the normal bounded wait, on a barrier that
 * nothing completes; it gives up after `limit_ns` and sets the plan's error word, so a
 * following marble_check returns MARBLE_ERR_TIMEOUT.  Nothing faults or hangs. */
marble_status_t marble_debug_wait_timeout(const marble_plan_t *plan, uint64_t limit_ns,
                                          marble_stream_t stream);

/*
 * Tile map without allocation.  The paper has no counterpart for this call: it is a
 * library convenience for callers that cannot call cudaMalloc.  Typical cases:
 *   - a planner that runs for every packed batch on a side stream while the previous
 *     training step still runs, and cannot afford the device-wide synchronisation that
 *     cudaMalloc may imply;
 *   - a process whose device memory is owned by another allocator (a framework caching
 *     allocator that has reserved the pool) or is capped by a fixed budget.
 * It computes the same global tile map as marble_plan (MARBLE_FIELD_TILE_ROWPTR / _COL /
 * _TAG: per-row CSR in original block coordinates, kv blocks ascending, tags FULL /
 * PARTIAL) into caller buffers, and allocates nothing.  Its intermediate scratch
 * (per-block summaries, candidate bands, per-row counts, a validation word; about 64 bytes
 * per 128-token block) lives in a fixed array inside the library, sized for at most
 * MARBLE_TILE_MAP_STATIC_MAX_TOKENS tokens; every GPU that loads the library holds that
 * array (about 1 MiB) until the process exits.
 *   n_tokens  multiple of 128, at most MARBLE_TILE_MAP_STATIC_MAX_TOKENS (larger packs are
 *             rejected with MARBLE_ERR_INVALID_ARG: use marble_plan);
 *   sample_id, seg_id, noise_id, window: as in marble_plan_desc_t (device int32[n_tokens]);
 *   row_ptr   device int64[n_tokens/128 + 1], written completely; row_ptr[nb] = number of
 *             non-empty tiles.  If the metadata fails validation, row_ptr[0] is set to -1;
 *   col, tag  device int32[capacity], uint8[capacity]; entries at CSR index >= capacity are
 *             not written (compare row_ptr[nb] with capacity to detect a short buffer).
 * Every pointer must be device (or managed) memory of the current device; others are
 * rejected with MARBLE_ERR_INVALID_ARG.
 * Asynchronous on `stream`; host-side argument errors return before any launch.  The first
 * call on a device looks up the device address of the scratch array on that device (a
 * host-side step, done once per device, with that device current); make that first call
 * before any stream capture.  The address belongs to the device's context: do not call this
 * again after cudaDeviceReset in the same process.  All calls on a device share the one scratch array, so calls
 * whose executions overlap on the GPU (different streams, or several host threads) race;
 * serialise them, e.g. on one stream.
 */
#define MARBLE_TILE_MAP_STATIC_MAX_TOKENS 2097152
marble_status_t marble_tile_map_static(int64_t n_tokens, const int32_t *sample_id,
                                       const int32_t *seg_id, const int32_t *noise_id,
                                       int32_t window, int64_t *row_ptr, int32_t *col,
                                       uint8_t *tag, int64_t capacity, marble_stream_t stream);

/* Thread-local message describing the last error on this thread ("" if none). */
const char *marble_last_error(void);

/* Library version string. */
const char *marble_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MARBLE_H_ */
