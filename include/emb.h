/*
 * emb.h -- C ABI of the GB300 sparse-embedding library (libemb.so).
 *
 * The library implements the sparse embedding layer of a DLRM-style recommender on one
 * GPU: IDs are mapped to table rows (directly, or through an open-addressing hash table
 * that inserts unseen keys), rows are gathered and pooled per (sample, feature), the
 * pooled vectors and the dense vector go through the pairwise dot interaction, and the
 * backward pass dedups the batch's rows, reduces their gradients and applies sparse
 * Adagrad to the touched rows only.  Around that path: Adagrad Decay, feature admission
 * and eviction for the hashed table, tiered storage for static tables (host tier plus an
 * HBM row cache), a cross interaction layer and an int8 row codec.
 *
 * Sources (web pages, by title and section):
 *  - HugeCTR interview (zhidx), section 2: embeddings map categorical IDs to vectors that
 *    sit before the feature interaction; IDs of unknown range go through a hash table.
 *    Section 3 (1): GPU hash table and a memory-saving sparse optimiser; (5) pooling fused
 *    with its neighbour kernel; (6) CUDA Graph over the many kernels of a step.
 *  - Merlin Distributed Embeddings article, "Background": lookup is memory-bandwidth bound;
 *    the wrapper takes a list of tables (input_dim, output_dim); "synthetic model
 *    benchmark": global batch 65536 with the Adagrad optimiser.
 *  - DeepRec announcement, "EmbeddingVariable": dynamic vocabulary in a lock-free hash
 *    table touched once per forward and once per backward; new features start from the
 *    initializer value, generally 0.
 *  - OneEmbedding article, "operator optimisation": FusedDotFeatureInteraction and
 *    FusedCrossFeatureInteraction; "usability": interaction(dense_fields, embedding).
 *  - DeepRec announcement, "Adagrad Decay Optimizer": period-based accumulator discount.
 *
 * Conventions (every entry point):
 *  - Pointers named d_* are device pointers owned by the caller; h_* are host pointers
 *    owned by the caller.  The context owns the tables, accumulators, hash arrays and all
 *    workspace; it allocates them in emb_create and frees them in emb_destroy.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Calls
 *    that take a stream only enqueue work on it and return without waiting.
 *  - Argument errors are returned at once (EMB_EINVAL, EMB_ESTATE) and enqueue nothing.
 *    Data errors found on the device (an ID out of range, a negative hashed key, a full
 *    hash table, malformed offsets) set bits of a device flag word read by emb_get_status;
 *    the offending lookup contributes zero and takes no update.
 *  - Layouts: bag index = b*T + t (sample-major); ids are table-local row numbers (static
 *    tables) or raw keys in [0, 2^63) (hashed table, shared by all T features).
 *    offsets: int32 [B*T+1] with offsets[0] = 0 (multi-hot) or NULL (one ID per bag).
 *    pooled / d_pooled: fp32 [B][T][D].  dense / d_dense: fp32 [B][D].
 *    interaction out / dout: fp32 [B][D + P], P = F(F-1)/2, F = T+1; out = [dense ||
 *    x_i . x_j for i = 1..F-1, j = 0..i-1], x_0 = dense, x_t+1 = pooled[t].
 *  - One context serves one stream at a time; calls on one context must be ordered.
 */
#ifndef EMB_H_
#define EMB_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum emb_status {
  EMB_OK = 0,
  EMB_EINVAL = 1, /* bad argument or configuration; nothing enqueued */
  EMB_ENOMEM = 2, /* device allocation failed in emb_create; nothing left allocated */
  EMB_ESTATE = 3, /* call out of order, e.g. a backward with no forward before it */
  EMB_ECUDA = 4   /* a CUDA runtime call or a kernel launch failed */
} emb_status;

/* device flag bits (emb_get_status) */
#define EMB_FLAG_ID_RANGE 0x1u    /* static ID outside [0, rows[t]) */
#define EMB_FLAG_BAD_KEY 0x2u     /* hashed key negative (outside [0, 2^63)) */
#define EMB_FLAG_TABLE_FULL 0x4u  /* no free hash slot within the probe limit (tiered
                                     tables: no free cache slot) */
#define EMB_FLAG_BAD_OFFSETS 0x8u /* offsets decreasing, negative or beyond nnz */
#define EMB_FLAG_WAIT_LIMIT 0x10u /* a bounded in-kernel wait on an asynchronous copy gave up;
                                     the results of that call are not valid */

enum { EMB_F32 = 0, EMB_BF16 = 1 };
enum { EMB_POOL_SUM = 0, EMB_POOL_MEAN = 1 };
enum { EMB_ADAGRAD = 0, EMB_ADAGRAD_ROWWISE = 1 };

typedef struct emb_config {
  int32_t num_tables;  /* T >= 1: features (fields) per sample */
  int32_t dim;         /* D: row width; D*sizeof(elem) a multiple of 16 bytes, D <= 512 */
  const int64_t* rows; /* host [T]: rows of each static table; NULL when hashed */
  int32_t hashed;      /* 1: one open-addressing table keyed by int64, shared by all T */
  int64_t capacity;    /* hashed: slots, a power of two <= 2^31 */
  int32_t dtype;       /* EMB_F32 or EMB_BF16 parameter storage */
  int32_t pooling;     /* EMB_POOL_SUM or EMB_POOL_MEAN */
  int32_t optimizer;   /* EMB_ADAGRAD (fp32 accumulator per element) or
                          EMB_ADAGRAD_ROWWISE (one fp32 accumulator per row) */
  float lr, eps;       /* acc += g^2; w -= lr * g / (sqrt(acc) + eps) */
  float init_acc;      /* initial accumulator value */
  float init_lo, init_hi; /* static rows start at U(init_lo, init_hi) (counter-based spec) */
  float hash_init;     /* value of every element of a newly inserted hashed row */
  uint64_t seed;       /* seed of the counter-based row initialiser */
  int64_t max_batch;   /* largest B any call will pass */
  int64_t max_lookups; /* largest nnz (IDs per batch) any call will pass */
} emb_config;

typedef struct emb_ctx emb_ctx;

/* Text of a status code.  Never NULL. */
const char* emb_status_str(emb_status s);

/* Validate `cfg`, allocate and initialise every table, accumulator and workspace on the
 * current device, and return a context in *out.  Static rows take the counter-based
 * initial values (SplitMix64 stream of `seed`, element (t, id, col) = output number
 * ((t<<40)+id)*512+col+1, u = (z>>40)/2^24, v = lo + (hi-lo)*u in float); accumulators
 * take init_acc; hashed slots start empty with w = hash_init, acc = init_acc.
 * Synchronous.  EMB_EINVAL for a bad config (checked before any CUDA call), EMB_ENOMEM
 * when an allocation fails (everything already allocated is freed).
 * Four environment variables, read here, tune the context without changing results beyond
 * floating-point summation order: EMB_FUSED_FWD = "simt" runs the fused interaction forward
 * on the FMA pipes instead of the tensor cores, and EMB_FUSED_BWD = "simt" the fused
 * interaction backward (the tensor-core kernels serve fp32 one-hot tables with D = 128 and
 * T+1 <= 32; "tc" or unset selects them); EMB_HOST_CHUNKS = 1..8 sets how many sample
 * chunks emb_train_step_host pipelines for those shapes (default 2); EMB_ONCE_DIRECT = "1"
 * makes every interaction step on the tensor-core backward (per-element Adagrad) update the
 * rows looked up once in its batch inside the backward, "0" never (all rows go through the
 * gradient buffer and the update kernel), unset: when the previous batch had at least one
 * unique row per ten lookups (see emb_step_tracks_once).  A fifth exists for tests of the
 * failure path only: EMB_WAIT_POLLS = n caps the first bounded in-kernel wait of the
 * tensor-core backward (its wait for the tensor core) at n polls, 0 meaning it gives up at
 * once; the kernel then raises EMB_FLAG_WAIT_LIMIT, waits at the full limit for the work
 * it has in flight, and leaves, so the results of that step are not valid. */
emb_status emb_create(const emb_config* cfg, emb_ctx** out);

/* Tiered storage for static tables (HugeCTR interview and Merlin article: embedding tables
 * outgrow device memory; the design here is this library's own).  As emb_create for static
 * tables (cfg->hashed must be 0), but every row and accumulator lives in host-mapped pinned
 * memory (the host tier, written with the initial values by the device) and HBM holds a
 * cache of `cache_rows` rows (a power of two, 2 .. 2^31) indexed by global row.  A lookup
 * whose row is not cached claims a cache slot; right after deduplication the row is copied
 * in from the host tier, so every kernel of the step works on HBM.  emb_evict writes the
 * rows it removes back to the host tier (same policy: idle steps or low count; the per-key
 * counts are kept from the start), and emb_read_rows reads a row from the cache or, if not
 * cached, from the host tier.  Results equal those of the static table.  A batch must find
 * room for its rows: once the cache is full a new row is rejected like a full hashed table
 * (EMB_FLAG_TABLE_FULL) and adds zero, so callers evict between steps (emb_evict, or the
 * watermark check of emb_set_tier_watermark after every step). */
emb_status emb_create_tiered(const emb_config* cfg, int64_t cache_rows, emb_ctx** out);

/* Tiered contexts: bring a later batch's rows into the cache ahead of its step (DeepRec
 * announcement, "Embedding multi-level hybrid storage": features move between storage
 * levels asynchronously).  d_ids / d_offsets / nnz / batch as emb_forward, device
 * buffers whose contents must be ready in the order of `stream` (a copy made on another
 * stream must be waited for on `stream` first) and stay valid until the work on `stream`
 * has run.  Enqueued on `stream` (meant to be a second stream, so that the copy from the
 * host tier runs while the current step computes); it starts after the latest change of
 * the cache (a forward's dedup and fill, an eviction), and the next forward, eviction or
 * watermark check waits for it, so a step never sees a row half copied.  Every valid lookup's row that is not
 * cached claims a slot and is copied in; a full cache is not flagged here (the batch's own
 * forward retries those rows and flags them).  Every row of the batch, brought in or
 * found cached, counts as last used at the number of the step in flight (the pending
 * step while a forward awaits its backward, else the last completed one), so neither the
 * watermark check nor an idle-time eviction takes it out before its step; rows brought in
 * start with a lookup count of zero (an emb_evict with a count minimum does remove them).
 * Results of every step equal those without the prefetch.  EMB_EINVAL for a non-tiered
 * context or malformed arguments (ids out of range are skipped, as the forward flags
 * them). */
emb_status emb_prefetch(emb_ctx* ctx, const int64_t* d_ids, const int32_t* d_offsets,
                        int64_t nnz, int64_t batch, void* stream);

/* Tiered contexts: the cache's watermarks (DeepRec announcement, "Embedding multi-level
 * hybrid storage": heat statistics keep hot features on the fast level and offload rare
 * ones).  With high > 0, at the end of every backward step, on its stream, when more than
 * `high` cache rows are in use the rows idle longest are written back to the host tier
 * until at most `low` remain: the device counts the cached rows by idle steps (current
 * step - last step looked up, 0 .. 62 and 63 for 63 or more) and evicts every row idle for
 * more than the smallest threshold t that reaches `low` (t = 0 evicts all rows the current
 * step did not look up, the most it can free; the step's own rows always stay).  The
 * decision is taken on the device, so no step waits for the host.  high = 0 switches it
 * off (the default).  0 <= low < high <= cache_rows; between steps only (EMB_ESTATE after
 * a forward without its backward); EMB_EINVAL for a non-tiered context. */
emb_status emb_set_tier_watermark(emb_ctx* ctx, int64_t high, int64_t low);

/* Tiered contexts: the number of cache rows in use (synchronous: waits for the device). */
emb_status emb_tier_occupancy(emb_ctx* ctx, int64_t* h_rows);

/* Free everything the context owns (waits for the device first).  NULL is a no-op. */
void emb_destroy(emb_ctx* ctx);

/* Forward lookup + pooling (HugeCTR interview sec. 2; Merlin article "Background").
 * d_ids: [nnz]; d_offsets: [B*T+1] or NULL (then nnz must equal B*T);
 * d_pooled: [B][T][D] fp32 output (sum, or mean over the bag length L; L = 0 gives 0).
 * Hashed: unseen keys are inserted (DeepRec "EmbeddingVariable").  Records the
 * row of every lookup and the batch's unique rows for the next backward call. */
emb_status emb_forward(emb_ctx* ctx, const int64_t* d_ids, const int32_t* d_offsets,
                       int64_t nnz, int64_t batch, float* d_pooled, void* stream);

/* Dot interaction (OneEmbedding "operator optimisation"): d_out[B][D+P] from d_dense
 * [B][D] and d_pooled [B][T][D].  Needs T+1 <= 32, D <= 512. */
emb_status emb_interact(emb_ctx* ctx, const float* d_dense, const float* d_pooled,
                        int64_t batch, float* d_out, void* stream);

/* Backward of emb_interact.  The pages give no formula: this is the chain rule of the dot
 * interaction of the OneEmbedding article, "operator optimisation" (pair order as in
 * emb_interact): G[i][j] = G[j][i] = dout[D + pair(i,j)], dX = G X,
 * d_dense = dX_0 + dout[0:D], d_pooled[t] = dX_{t+1}.  d_dout [B][D+P], d_dense and
 * d_pooled as for emb_interact; d_ddense [B][D] and d_dpooled [B][T][D] are overwritten.
 * Same argument checks as emb_interact. */
emb_status emb_interact_backward(emb_ctx* ctx, const float* d_dout, const float* d_dense,
                                 const float* d_pooled, int64_t batch, float* d_ddense,
                                 float* d_dpooled, void* stream);

/* Backward of the last emb_forward + sparse Adagrad (Merlin article "synthetic model
 * benchmark"; HugeCTR interview sec. 3 (1)).  d_dpooled: [B][T][D] gradient of the
 * pooled output.  The gradients of all lookups of one row are summed (scaled by 1/L
 * under mean pooling), then each touched row takes one Adagrad step; untouched rows are
 * not written.  EMB_ESTATE unless the previous call on ctx was a forward. */
emb_status emb_backward_adagrad(emb_ctx* ctx, const float* d_dpooled, void* stream);

/* Fused forward: lookup + pooling + dot interaction in one pass over the rows; the pooled
 * vectors are never written to memory (HugeCTR interview sec. 3 (5), pooling fused with
 * its neighbour).  Same inputs as emb_forward plus d_dense [B][D]; d_out [B][D+P]. */
emb_status emb_forward_interact(emb_ctx* ctx, const int64_t* d_ids, const int32_t* d_offsets,
                                int64_t nnz, int64_t batch, const float* d_dense,
                                float* d_out, void* stream);

/* Fused backward of emb_forward_interact: recomputes each sample's pooled vectors from the
 * (not yet updated) rows, applies the interaction backward, sums the row gradients per
 * unique row and applies Adagrad.  d_dout [B][D+P], d_dense [B][D] (the same dense input
 * as the forward), d_ddense [B][D] output.  EMB_ESTATE unless the previous call on ctx
 * was emb_forward_interact. */
emb_status emb_backward_interact_adagrad(emb_ctx* ctx, const float* d_dout,
                                         const float* d_dense, float* d_ddense, void* stream);

/* One training step from host buffers: copies ids, offsets, dense and dout to the device,
 * runs emb_forward_interact + emb_backward_interact_adagrad, and copies out [B][D+P] and
 * d_dense [B][D] back.  Host buffers should be page-locked for asynchronous copies.  The
 * copies overlap the kernels on two internal streams (dout is uploaded during the forward,
 * out downloaded during the backward); all of the step's work is ordered after the work
 * already enqueued on `stream`, and `stream` is ordered after all of it.  The device staging
 * buffers and the internal streams are created on the first call on a context.  Returns
 * once the work is enqueued; synchronise `stream` before reading h_out / h_ddense. */
emb_status emb_train_step_host(emb_ctx* ctx, const int64_t* h_ids, const int32_t* h_offsets,
                               int64_t nnz, int64_t batch, const float* h_dense,
                               const float* h_dout, float* h_out, float* h_ddense,
                               void* stream);

/* No passage (status reporting of this library): wait for `stream`, then return the device
 * flag word (EMB_FLAG_*) in *flags and clear it.  EMB_EINVAL for a NULL context or flags. */
emb_status emb_get_status(emb_ctx* ctx, void* stream, uint32_t* flags);

/* No passage (read-back for checks and checkpoints; the DeepRec announcement's incremental
 * model export is the nearest the pages come).
 * Read rows (synchronous; waits for the device).  Static: h_ids are table-local rows of
 * `table`.  Hashed: h_ids are keys (table ignored); h_found[i] = 0 for an absent key.
 * h_w: [n][D] fp32 (bf16 widened exactly); h_acc: [n][D] (per element) or [n] (row-wise).
 * Any of h_w, h_acc, h_found may be NULL.  EMB_EINVAL for a static id out of range. */
emb_status emb_read_rows(emb_ctx* ctx, int32_t table, const int64_t* h_ids, int64_t n,
                         float* h_w, float* h_acc, int8_t* h_found);

/* Cross interaction: one layer of a deep & cross network over each sample's feature
 * vector.  OneFlow OneEmbedding article, "operator optimisation": FusedCrossFeatureInteraction,
 * with the cross layer of "Deep & Cross Network for Ad Click Predictions" (figure cited
 * there): out = x0 * (xl . w) + b + xl per sample.  Backward by the chain rule, with
 * s = xl . w and t = x0 . dout per sample: dxl = dout + w t, dx0 = dout s,
 * dw = sum over samples of xl t, db = sum of dout (dw, db overwritten; fp32 outputs, sums
 * over samples accumulated in double per CTA).  x0, xl, out, dout, dx0, dxl: fp32 [B][K]
 * (K = F * D for the concatenated dense and pooled vectors); w, b, dw, db: fp32 [K]; device
 * buffers owned by the caller; enqueued on `stream`, no context needed.  EMB_EINVAL for
 * B < 0, K outside [1, EMB_CROSS_MAX_K] or a NULL buffer. */
#define EMB_CROSS_MAX_K 9216
emb_status emb_cross_forward(const float* d_x0, const float* d_xl, const float* d_w,
                             const float* d_b, int64_t B, int32_t K, float* d_out, void* stream);
emb_status emb_cross_backward(const float* d_x0, const float* d_xl, const float* d_w,
                              const float* d_dout, int64_t B, int32_t K, float* d_dx0,
                              float* d_dxl, float* d_dw, float* d_db, void* stream);

/* int8 row codec for the rows the layer exchanges (pooled rows, their gradients).  Merlin
 * Distributed Embeddings article, opening section: rows are exchanged between GPUs in
 * reduced precision; the format is not given.  Reading taken: per row of d floats,
 * scale = max|x| / 127 and code = x / scale rounded to nearest, ties to even, clamped to
 * [-127, 127] (a zero row: scale 0, codes 0); decoding gives code * scale.  Every step is one
 * IEEE fp32 operation, so results are fixed bit for bit.  Inputs must be finite.
 * d_x: fp32 [n][d]; d_q: int8 [n][d]; d_scale: fp32 [n]; device buffers owned by the caller.
 * Enqueued on `stream`; no context needed.  EMB_EINVAL for n < 0, d < 1 or a NULL buffer. */
emb_status emb_quantize_rows(const float* d_x, int64_t n, int32_t d, int8_t* d_q,
                             float* d_scale, void* stream);
emb_status emb_dequantize_rows(const int8_t* d_q, const float* d_scale, int64_t n, int32_t d,
                               float* d_x, void* stream);

/* Adagrad Decay.  DeepRec announcement, "Adagrad Decay Optimizer": the accumulator is
 * discounted by period, with one discount for every sample of a period; the rule is not
 * given.  Reading taken: backward steps after this call are grouped into periods of
 * period_steps steps (the first period is 0); when a row is updated, its accumulator is first
 * multiplied by rate^(periods since the period of its previous update, or since period 0),
 * then the step adds g^2 (per element) or mean g^2 (row-wise).  rate in (0, 1];
 * period_steps 0 turns the decay off.  Between steps only (EMB_ESTATE otherwise);
 * allocates one uint32 per table row on first use (EMB_ENOMEM).  While it is on, rows looked
 * up once are not updated inside the interaction backward (see EMB_ONCE_DIRECT). */
emb_status emb_set_adagrad_decay(emb_ctx* ctx, float rate, uint32_t period_steps);

/* Feature admission and eviction for the hashed table.  DeepRec announcement,
 * "EmbeddingVariable": admission methods and eviction strategies are named, not defined;
 * the reading taken here:
 *  - every backward step is numbered (1, 2, ...); it adds each key's lookups in its batch to
 *    the key's count and stamps the key with the step number;
 *  - admission: a key's row takes the Adagrad update of a step only once its count, this
 *    step's lookups included, has reached min_count; until then the row keeps its initial
 *    value (its lookups read w = hash_init).  min_count 0 or 1: every key at once.  The
 *    first call also starts the per-key counts and last steps that admission and eviction
 *    read (a hashed context keeps none before it, so steps before the call are not
 *    counted).  Hashed contexts only (EMB_EINVAL otherwise); between steps only (EMB_ESTATE
 *    after a forward without its backward).  While a minimum above 1 is set, rows looked up
 *    once are not updated inside the interaction backward (see EMB_ONCE_DIRECT). */
emb_status emb_set_admission(emb_ctx* ctx, uint32_t min_count);

/*  - eviction: remove every key whose idle time (current step - its last step) exceeds
 *    max_idle_steps (when max_idle_steps > 0) or whose count is below min_count.  Its slot
 *    becomes reusable, its row and accumulator return to their initial values and its
 *    count to zero, so a key looked up again later starts afresh.  Enqueued on `stream`;
 *    when h_evicted is not NULL the call waits and stores the number of keys removed.
 *    Hashed contexts only; between steps only, after emb_set_admission (EMB_ESTATE
 *    otherwise). */
emb_status emb_evict(emb_ctx* ctx, uint32_t max_idle_steps, uint32_t min_count, void* stream,
                     int64_t* h_evicted);

/*  - the count and last step of n hashed keys (synchronous; 0 and 0 for an absent key).
 *    h_count / h_last_step: [n] host buffers, either may be NULL. */
emb_status emb_read_key_stats(emb_ctx* ctx, const int64_t* h_keys, int64_t n, uint32_t* h_count,
                              uint32_t* h_last_step);
/*    (Tiered tables: emb_evict and emb_read_key_stats take global rows as keys, i.e. the sum
 *    of the rows of the tables before t plus the table-local id.) */

/* No passage (read-back of the dedup step, for checks): unique rows of the last forward
 * (synchronous): *h_num_unique = U; the first min(U, cap)
 * entries of h_keys get the global row (sum of rows of the tables before t, plus id) or
 * the hashed key, and h_counts their occurrence counts, in no particular order. */
emb_status emb_read_unique(emb_ctx* ctx, int64_t* h_keys, int32_t* h_counts, int64_t cap,
                           int64_t* h_num_unique);

/* No passage (read-back for checks and checkpoints; cf. the DeepRec announcement's
 * incremental model export): every occupied slot of the hashed table (synchronous):
 * *h_count = number of keys; the
 * first min(count, cap) keys with their rows (h_w [cap][D]) and accumulators go to the
 * host buffers, in slot order.  EMB_EINVAL for a static-table context. */
emb_status emb_export_hash(emb_ctx* ctx, int64_t* h_keys, float* h_w, float* h_acc,
                           int64_t cap, int64_t* h_count);

/* Kernel timing: with enable = 1 every kernel launch is bracketed by CUDA events on its
 * stream; emb_profile_read waits for them and returns, for kernel number idx, its name,
 * the summed device time in milliseconds and its launch count since the last reset
 * (EMB_EINVAL past the last kernel).  emb_profile_reset clears the sums. */
emb_status emb_profile(emb_ctx* ctx, int32_t enable);
emb_status emb_profile_read(emb_ctx* ctx, int32_t idx, const char** name, double* total_ms,
                            int64_t* launches);
emb_status emb_profile_reset(emb_ctx* ctx);

/* Number of kernels this context has launched since it was created. */
int64_t emb_launch_count(const emb_ctx* ctx);

/* 1 when the step of the last forward tracks the rows looked up once in its batch (the
 * interaction backward then applies their Adagrad update itself, and the update after it
 * only the other rows'), else 0; -1 for a NULL context.  Either way every row gets the same
 * update; only the kernel that applies it differs. */
int32_t emb_step_tracks_once(const emb_ctx* ctx);

/* Largest n accepted by emb_unique_keys_noalloc. */
#define EMB_NOALLOC_MAX_KEYS 524288

/* Unique keys of a batch, for callers that cannot allocate device memory.  The source pages
 * have no counterpart of this call: it is the dedup step of the backward (unique rows of a
 * batch and each lookup's unique index) offered on its own to callers that may not call
 * cudaMalloc -- serving processes that fix their device memory budget at start-up, or
 * plug-ins and callbacks that are handed only their input and output buffers.
 * It needs no context and allocates nothing: its scratch (a hash set of 2^20 slots, 12 MiB)
 * is a fixed array in the library's device image, held by every GPU that loads the library
 * until the process exits.
 *   d_keys     [n] int64 keys; a negative key is skipped (inverse -1)
 *   d_unique   [n] output: the distinct non-negative keys in slots 0..U-1, in no fixed order
 *   d_inverse  [n] output: index into d_unique of each key, or -1
 *   d_num_unique  [1] int32 output: U
 * Stream-ordered and asynchronous.  n above EMB_NOALLOC_MAX_KEYS, a negative n, or a NULL
 * buffer returns EMB_EINVAL before anything is enqueued.  Every call resets and reuses the
 * same scratch, so calls that may overlap on the GPU (different streams or host threads)
 * race and must be serialised by the caller.  The first call on each device looks up the
 * scratch's device address (cudaGetSymbolAddress, with that device current); make that
 * first call before any stream capture. */
emb_status emb_unique_keys_noalloc(const int64_t* d_keys, int64_t n, int64_t* d_unique,
                                   int32_t* d_inverse, int32_t* d_num_unique, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EMB_H_ */
