/*
 * emb.h -- C ABI of the GB300 sparse embedding training step.
 *
 * One training step of a multi-table, multi-hot embedding layer on one GPU:
 *   emb_forward          lookup + pooling + concatenation, one fused kernel
 *   emb_backward_update  dedup of the touched rows, per-row gradient reduction
 *                        and the SGD / Adagrad update, in place
 *   emb_unique           the stand-alone dedup primitive
 *
 * The operations are the ones the GTC 2022 "Merlin HugeCTR" slides name
 * (slides "COMMON EMBEDDING PRIMITIVES" and "HUGECTR EMBEDDING LAYER": table
 * lookup, pooling/reduction, concatenation, fused into one kernel; slide
 * "WEIGHT CONVERSION FOR MIXED PRECISION TRAINING": FP32 optimizer math, FP16
 * tables), with the reduction-based (RB) and unique-based (UB) backward
 * flavours named in "NVIDIA EMBark revoluciona la formacion en sistemas de
 * recomendacion a escala", section "Integracion del cluster".
 *
 * Conventions shared by every call
 *  - Pointers are DEVICE pointers unless their name ends in _host.  Device
 *    arrays must be aligned to their element size (int64: 8 bytes, int32 and
 *    fp32: 4, fp16/bf16: 2); the pooled output and grad_out to 16 bytes (the
 *    kernels move 4 columns at a time).  A misaligned pointer returns
 *    EMB_ERR_INVALID_ARG with nothing enqueued.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call that takes a stream only enqueues work on it and
 *    returns without waiting, except the *_host copies and emb_sync_status.
 *  - Return value: EMB_OK or a negative emb_status.  Problems the host can see
 *    (null pointers, sizes beyond the limits given at creation, bad enums)
 *    return at once with nothing enqueued.  Problems only the GPU can see (a
 *    key outside [0, rows), a bag whose table id is not j / batch, a full hash
 *    table, a bounded wait that ran out) never trap: the offending lookup or
 *    row is skipped and a sticky error word in the layer records it, returned
 *    and cleared by emb_sync_status.
 *  - Thread safety: a layer may be used from one host thread at a time; calls
 *    on one layer must be issued on one stream (or be ordered by the caller).
 */
#ifndef EMB_H
#define EMB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EMB_OK = 0,
    EMB_ERR_INVALID_ARG = -1,   /* bad argument, detected on the host (or a bad table id on the GPU) */
    EMB_ERR_OOM = -2,           /* device allocation failed */
    EMB_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed */
    EMB_ERR_KEY_RANGE = -4,     /* GPU saw a key outside [0, rows) */
    EMB_ERR_CAPACITY = -5,      /* GPU hash table full */
    EMB_ERR_TIMEOUT = -6,       /* a bounded GPU wait gave up (reserved: no current kernel waits) */
    EMB_ERR_STATE = -7          /* call out of order (e.g. backward before any forward) */
} emb_status;

typedef enum { EMB_F32 = 0, EMB_F16 = 1, EMB_BF16 = 2 } emb_dtype;
typedef enum { EMB_POOL_SUM = 0, EMB_POOL_MEAN = 1 } emb_pooling;
typedef enum {
    EMB_OPT_SGD = 0,
    EMB_OPT_ADAGRAD = 1,            /* one fp32 accumulator per element */
    EMB_OPT_ROWWISE_ADAGRAD = 2     /* one fp32 accumulator per row */
} emb_opt;
typedef enum {
    EMB_BWD_REDUCTION = 0,      /* RB: sort (row id, bag) pairs, reduce each run of equal ids */
    EMB_BWD_UNIQUE_SORT = 1,    /* UB: sort-based dedup to unique/inverse/counts first, then reduce */
    EMB_BWD_UNIQUE_HASH = 2     /* UB: hash-based dedup first, then reduce by inverse index */
} emb_bwd_variant;

/* One embedding table.  dim must be a multiple of 4 in [4, 128]; rows >= 1.
 * lr / eps / init_acc: SGD uses lr; both Adagrads use all three (init_acc is
 * the initial accumulator value).  The layer stores weights in `dtype` and the
 * accumulators in fp32 (rows*dim of them for Adagrad, rows for row-wise
 * Adagrad); all arithmetic is fp32.
 * master_fp32 (fp16/bf16 tables only; EMB_ERR_INVALID_ARG for fp32): GTC 2022
 * HugeCTR slides, "WEIGHT CONVERSION FOR MIXED PRECISION TRAINING" -- the
 * optimizer keeps FP32 weights and the FP16 copy the forward reads is
 * converted from them.  The layer then holds rows*dim fp32 master values;
 * every update steps the master in fp32 and stores the 16-bit weight as the
 * new master rounded to nearest-even, so steps smaller than half a 16-bit
 * ulp accumulate instead of being rounded away.
 * dynamic (GTC 2022 HugeCTR slides, "HUGECTR EMBEDDING LAYER": embeddings
 * behind a GPU hash table): the table's keys are arbitrary int64 ids, not row
 * indices, and `rows` is the capacity.  emb_forward finds each key's row in an
 * open-addressing map over the rows (linear probing from a hash of table and
 * key) and, for a key it has not seen, takes a free row and gives it initial
 * values: the counter-based values of emb_init_uniform with splitmix64
 * output number (key << 8) ^ (t << 57) ^ c, the table's init_acc and, with
 * master_fp32, the fp32 value as master.  Nothing is evicted: a lookup that
 * finds the table full is skipped and reported as EMB_ERR_CAPACITY.  The key
 * -2^63 is reserved and reported like an out-of-range key.  Everything after
 * the lookup (dedup ids, row I/O) uses the row, which emb_find_keys gives. */
typedef struct {
    int64_t rows;
    int32_t dim;
    int32_t dtype;     /* emb_dtype */
    int32_t pooling;   /* emb_pooling */
    int32_t opt;       /* emb_opt */
    float lr;
    float eps;
    float init_acc;
    int32_t master_fp32; /* 1: keep an fp32 master copy of a 16-bit table (see below); 0: none */
    int32_t dynamic;     /* 1: keys are arbitrary int64 ids mapped to rows by a hash map (see below) */
} emb_table_spec;

typedef struct emb_layer emb_layer;   /* opaque; owns tables, optimizer state and workspace */

/* Create a layer of `num_tables` tables (1..4096).  GTC 2022 HugeCTR slides,
 * "CHALLENGES OF EMBEDDING LAYER": the tables' memory demand is the first
 * challenge the slide names (there answered by spreading tables over GPUs),
 * and lower precision such as FP16 the common answer; here every table (fp32,
 * fp16 or bf16), its optimizer state and the step's workspace are held in this
 * one GPU's memory.  The sum of all rows must be
 * below 2^32 - 1.  `max_batch` (>= 1) and `max_nnz` (>= 0, < 2^31) bound every
 * later forward: the workspace for that many bags and lookups is allocated
 * here, once, so the step itself allocates nothing.  Weights are NOT
 * initialised (call emb_init_uniform or emb_set_rows).  On success *out owns
 * the device memory until emb_destroy.  Allocation failure: EMB_ERR_OOM with
 * nothing leaked and *out untouched.
 * Test hooks, read here from the environment (unset in normal use):
 * EMB_TEST_ALLOC_LIMIT_BYTES caps what this call may allocate (to reach the
 * EMB_ERR_OOM path); EMB_TEST_REDUCE_CHUNK (a power of two in [32, 256])
 * raises the layer's reduction chunk length, so small inputs run the kernels
 * large multi-hot inputs get.  Neither changes any result. */
int emb_create(const emb_table_spec* specs, int32_t num_tables, int32_t max_batch,
               int64_t max_nnz, emb_layer** out);

/* Free everything the layer owns.  Synchronises the device first.  NULL is a
 * no-op.  No passage: library convenience. */
int emb_destroy(emb_layer* layer);

/* Fill every table with the counter-based uniform values
 *   w(t, r, c) = lo + (hi - lo) * ((h >> 40) * 2^-24),  h = splitmix64 output
 *   number n = t*2^44 + r*2^12 + c of the stream started from state `seed`,
 * evaluated in fp32 with one rounding per operation and then rounded to
 * nearest-even into the table dtype; set every Adagrad accumulator to its
 * table's init_acc and every fp32 master to the fp32 value.  A dynamic table
 * is emptied instead (all keys forgotten); its rows get the same kind of
 * values, from this seed/lo/hi, when keys take them.  Asynchronous on
 * `stream`.  No passage: library convenience (the pages give no
 * initialisation; this counter-based one lets tests regenerate any row). */
int emb_init_uniform(emb_layer* layer, uint64_t seed, float lo, float hi, void* stream);

/* Forward: lookup + pooling + concatenation (GTC 2022 HugeCTR slides, "COMMON
 * EMBEDDING PRIMITIVES"; Merlin overview article, section "HugeCTR").
 *   keys       int64[nnz]            local row ids, bags back to back
 *   offsets    int64[T*batch + 1]    CSR boundaries, bag j = t*batch + b
 *                                    (table-major); offsets[0] = 0,
 *                                    non-decreasing, offsets[T*batch] = nnz
 *   table_ids  int32[T*batch]        table of bag j; must equal j / batch
 *   out        fp32[batch, sum(dim)] out[b, doff_t + c] = s_j * sum over the
 *                                    bag of W_t[key][c]; s_j = 1 (sum) or
 *                                    1/L_j (mean); an empty bag gives 0;
 *                                    doff_t = dim_0 + ... + dim_(t-1)
 * All of keys/offsets/table_ids/out are caller-owned; none is kept after the
 * call.  The lookup's global row ids and bag ids are kept in the layer's
 * workspace for the next emb_backward_update.  A key outside [0, rows_t) or a
 * wrong table id is skipped (contributes 0, gets no gradient) and flagged
 * (EMB_ERR_KEY_RANGE / EMB_ERR_INVALID_ARG at emb_sync_status).  Offsets
 * that leave [0, nnz] or decrease are clamped on the GPU (into [0, nnz],
 * then to the bag start) before any key is read, and flagged as
 * EMB_ERR_INVALID_ARG at emb_sync_status; the pooled output and a following
 * backward are then meaningless but every access stays inside the caller's
 * arrays and the layer's workspace. */
int emb_forward(emb_layer* layer, const int64_t* keys, const int64_t* offsets,
                const int32_t* table_ids, int64_t nnz, int32_t batch, float* out,
                void* stream);

/* Backward + update for the most recent emb_forward on this layer: the
 * reduction-based (RB) or unique-based (UB) backward of "NVIDIA EMBark
 * revoluciona la formacion en sistemas de recomendacion a escala", section
 * "Integracion del cluster" (RB reduces the gradients of equal keys; UB
 * dedups the keys first), with the FP32 optimizer of the GTC 2022 HugeCTR
 * slides, "WEIGHT CONVERSION FOR MIXED PRECISION TRAINING":
 *   G_u[c] = sum over lookups i of row u of s_bag(i) * grad_out[b(i), doff_t + c]
 * then one optimizer step per touched row u (untouched rows are not read):
 *   SGD:     W <- W - lr*G
 *   Adagrad: A <- A + G*G ; W <- W - lr*G/(sqrt(A)+eps)     (per element)
 *   row-wise Adagrad: a <- a + (1/dim) * sum_c G[c]^2 (one accumulator a per
 *            row) ; W <- W - lr*G/(sqrt(a)+eps).  The pages name only the
 *            fp32 optimizer; this is the row-wise form of the open DLRM
 *            embedding libraries, which moves 4 bytes of state per row
 *            instead of 4*dim.
 * fp32 math, W stored back rounded to nearest-even into its dtype.
 * grad_out: fp32[batch, sum(dim)], caller-owned, same layout as `out`.
 * variant: emb_bwd_variant.  All variants give the same indices and the same
 * update up to fp32 rounding order; each variant is deterministic.
 * EMB_ERR_STATE if no forward preceded it. */
int emb_backward_update(emb_layer* layer, const float* grad_out, int32_t variant, void* stream);

/* Early dedup.  With variant >= 0 (an emb_bwd_variant), every later
 * emb_forward also enqueues the dedup of that backward variant on an
 * internal stream of the layer: the global ids and bags are extracted and
 * sorted (or hashed) while the pooling kernel runs on the caller's stream --
 * the dedup needs only the batch's keys, not the pooled output.  A following
 * emb_backward_update on the caller's stream waits for it and, if called with
 * the same variant, goes straight to the segmented reduction (with another
 * variant it redoes the dedup).  Results are identical to the default mode.
 * variant = -1 (default) turns it off.  The caller's input buffers must stay
 * valid until that backward is enqueued; no extra memory is used.  Passage:
 * "NVIDIA EMBark ...", section "Integracion del cluster" (the UB dedup needs
 * only the keys), and the fused embedding kernels of the GTC 2022 HugeCTR
 * slides, "HUGECTR EMBEDDING LAYER". */
int emb_set_early_dedup(emb_layer* layer, int32_t variant);

/* Keep (1) or drop (0, default) the dedup by-products of later backwards so
 * emb_dedup_result can return them.  EMB_BWD_REDUCTION then also writes the
 * sorted unique ids, counts and segment offsets it otherwise never forms.
 * No passage: library convenience (tests and callers that want the dedup). */
int emb_set_keep_dedup(emb_layer* layer, int32_t keep);

/* Copy the dedup result of the last emb_backward_update (with keep_dedup on)
 * into caller device buffers, each sized for the forward's nnz (NULL = skip):
 *   unique       int64[U]    global row ids row_base[t] + key, ascending
 *   inverse      int32[nnz]  unique[inverse[i]] = global id of lookup i;
 *                            skipped lookups get U.  Not formed by
 *                            EMB_BWD_REDUCTION (EMB_ERR_STATE if requested)
 *   counts       int32[U]    lookups per unique row
 *   seg_offsets  int32[U+1]  exclusive prefix sum of counts
 *   sorted_bags  int32[nnz]  bag id of each lookup, grouped by unique row,
 *                            ascending lookup order inside a group
 *   num_unique_host          U (the call synchronises `stream` for it)
 * EMB_ERR_STATE if there is no such result.  Passage: "NVIDIA EMBark ...",
 * section "Integracion del cluster" (the unique keys, inverse index and
 * counts of the UB dedup). */
int emb_dedup_result(emb_layer* layer, int64_t* unique, int32_t* inverse, int32_t* counts,
                     int32_t* seg_offsets, int32_t* sorted_bags, int64_t* num_unique_host,
                     void* stream);

/* Stand-alone dedup of arbitrary int64 keys: the dedup step that the
 * unique-based (UB) backward of "NVIDIA EMBark revoluciona la formacion en
 * sistemas de recomendacion a escala", section "Integracion del cluster",
 * runs before reducing gradients:
 *   unique       int64[n]    distinct keys, ascending, in unique[0..U)
 *   inverse      int32[n]    unique[inverse[i]] == keys[i]
 *   counts       int32[n]    counts[k] = #{i : keys[i] == unique[k]}, k < U
 *   seg_offsets  int32[n+1]  nullable; exclusive prefix sum of counts, [0..U]
 *   num_unique   int64[1]    U, written on the device
 * n in [0, 2^31).  `workspace` is caller-owned device memory of at least
 * emb_unique_workspace(n) bytes, 256-byte aligned; the call keeps no pointer
 * after it returns.  Sort-based (own LSD radix sort over the key range), so
 * the result is deterministic. */
int emb_unique_workspace(int64_t n, size_t* bytes);
int emb_unique(const int64_t* keys, int64_t n, int64_t* unique, int32_t* inverse,
               int32_t* counts, int32_t* seg_offsets, int64_t* num_unique,
               void* workspace, size_t workspace_bytes, void* stream);

/* emb_unique without any allocation, for callers that cannot allocate device
 * memory at call time: for instance a plugin whose enqueue path runs inside a
 * host framework that forbids cudaMalloc there (it may synchronise the device,
 * and fails outright under a fixed memory budget), or a serving thread that
 * must not touch the allocator while requests are in flight.  There is no
 * counterpart on the pages: this is a library convenience, not part of the
 * embedding method.
 *
 * Arguments and results are exactly those of emb_unique, minus the workspace:
 * the scratch is one array compiled into the library (12 MB of device
 * memory, held on every GPU that loads the library until the process exits).
 * n must be at most EMB_UNIQUE_NOALLOC_MAX_KEYS; larger n returns
 * EMB_ERR_INVALID_ARG and enqueues nothing.  The first call on a device looks
 * up the array's address on that device (the device current at the call), so
 * make that first call before any stream capture.  All calls share the one
 * array: calls whose GPU work overlaps -- on different streams or from
 * different threads without ordering -- race on it and give wrong results; the
 * contents left by the previous call are never relied on.  The address looked
 * up on a device stays in use for the life of the process: after
 * cudaDeviceReset on that device the function must not be called again. */
#define EMB_UNIQUE_NOALLOC_MAX_KEYS 262144
int emb_unique_noalloc(const int64_t* keys, int64_t n, int64_t* unique, int32_t* inverse,
                       int32_t* counts, int32_t* seg_offsets, int64_t* num_unique, void* stream);

/* Copy rows [row0, row0+n) of table t between the layer and host memory.
 * weights_host holds n*dim values of the table dtype (fp32, or the raw 16-bit
 * patterns of fp16/bf16); state_host (nullable; Adagrad tables only) n*dim
 * fp32, or n fp32 for row-wise Adagrad.  Synchronous: the call waits for
 * `stream`.  No passage: library convenience (checkpoint and resume, tests). */
int emb_get_rows(emb_layer* layer, int32_t t, int64_t row0, int64_t n, void* weights_host,
                 float* state_host, void* stream);
int emb_set_rows(emb_layer* layer, int32_t t, int64_t row0, int64_t n,
                 const void* weights_host, const float* state_host, void* stream);

/* Inference cache of table t (GTC 2022 HugeCTR slides, slide "HUGECTR:
 * SCALABLE, ACCELERATED RECSYS TRAINING": inference served through an
 * embedding cache on the GPU in front of the hierarchical parameter server,
 * HPS): fp16 copies of n chosen
 * rows (device int64 row ids; a dynamic table's rows from emb_find_keys),
 * looked up through a hash map from row to cache slot.  Replaces any earlier
 * cache of the table; n = 0 removes it.  The copies are a snapshot of the
 * rows at this call (16-bit tables are converted from their stored values
 * to fp16): training steps do not refresh them.  Tables of 2^31 rows or more
 * take no cache (EMB_ERR_INVALID_ARG).  Allocates device memory for the cache
 * and synchronises `stream`; EMB_ERR_OOM when it cannot allocate.
 * An id outside [0, rows) is skipped and flagged like a bad key. */
int emb_cache_build(emb_layer* layer, int32_t t, const int64_t* rows, int64_t n, void* stream);

/* Inference-only forward: the pooled, concatenated output of emb_forward
 * (same arguments, layout and error reporting), reading every row held in
 * its table's cache from the fp16 cache and every other row from the table.
 * Dynamic tables look keys up without inserting; an id the table does not
 * hold contributes nothing and is not an error.  Nothing is kept for a
 * backward: a following emb_backward_update still refers to the last
 * emb_forward.  Allocates nothing.  Passage: as for emb_cache_build. */
int emb_forward_infer(emb_layer* layer, const int64_t* keys, const int64_t* offsets,
                      const int32_t* table_ids, int64_t nnz, int32_t batch, float* out,
                      void* stream);

/* Rows of n keys (device int64) of dynamic table t, into rows_out (device
 * int64; -1 for a key the table does not hold).  Inserts nothing.
 * Asynchronous; EMB_ERR_INVALID_ARG for a table that is not dynamic.
 * Passage: GTC 2022 HugeCTR slides, "HUGECTR EMBEDDING LAYER" (the GPU hash
 * table from keys to embedding rows). */
int emb_find_keys(emb_layer* layer, int32_t t, const int64_t* keys, int64_t n, int64_t* rows_out,
                  void* stream);

/* The fp32 master copy of rows [row0, row0+n) of table t (a table created
 * with master_fp32 = 1; EMB_ERR_INVALID_ARG otherwise), n*dim fp32 in host
 * memory, for checkpoints and tests.  Synchronous: the call waits for
 * `stream`.  Setting the master does not touch the 16-bit weights: set both
 * (emb_set_rows) to restore a checkpoint.  Passage: GTC 2022 HugeCTR slides,
 * "WEIGHT CONVERSION FOR MIXED PRECISION TRAINING" (the FP32 weights behind
 * FP16 tables). */
int emb_get_master_rows(emb_layer* layer, int32_t t, int64_t row0, int64_t n, float* master_host,
                        void* stream);
int emb_set_master_rows(emb_layer* layer, int32_t t, int64_t row0, int64_t n,
                        const float* master_host, void* stream);
/* Gather n arbitrary rows' master values (device int64 ids) into a device
 * buffer of n*dim fp32.  Asynchronous; out-of-range ids are skipped and
 * flagged like bad keys.  Passage: as for emb_get_master_rows. */
int emb_gather_master_rows(emb_layer* layer, int32_t t, const int64_t* rows, int64_t n, float* master_out,
                           void* stream);

/* Gather n arbitrary rows (device int64 ids, each in [0, rows_t)) of table t
 * into device buffers: weights_out n*dim of the table dtype, state_out
 * (nullable) n*dim fp32 (row-wise Adagrad: n fp32).  Asynchronous.
 * Out-of-range ids are skipped and flagged like bad keys.  No passage:
 * library convenience (tests and checkpoints). */
int emb_gather_rows(emb_layer* layer, int32_t t, const int64_t* rows, int64_t n,
                    void* weights_out, float* state_out, void* stream);

/* Wait for `stream`, then return and clear the sticky device error word
 * (EMB_OK if the GPU saw nothing wrong).  No passage: library convenience. */
int emb_sync_status(emb_layer* layer, void* stream);

/* Number of kernels the library launched on behalf of this layer since the
 * last reset (reset = 1 clears it after reading).  No passage: library
 * convenience (measurement). */
int emb_launch_count(emb_layer* layer, int64_t* count_host, int32_t reset);

/* Phase timing.  With enable = 1 the layer records CUDA events on the call's
 * stream around each phase of every later step -- EMB_PHASE_FORWARD (the
 * fused lookup/pooling kernel), EMB_PHASE_DEDUP (global-id sort or hash
 * dedup, from the start of emb_backward_update up to the reduction) and
 * EMB_PHASE_REDUCE_UPDATE (segmented reduction + optimizer kernels) -- and
 * adds their elapsed times.  With early dedup the dedup phase runs on the
 * layer's internal stream, overlapping the forward.  A step's events are
 * read back only when a ring of 64 steps comes round to its slot again, so
 * timing adds no host wait to a step.  emb_phase_times waits for the last
 * recorded events, writes the accumulated milliseconds of the n (<= 3)
 * phases and the number of steps they cover, and, with reset = 1, clears
 * them.  No passage: library convenience (measurement). */
enum { EMB_PHASE_FORWARD = 0, EMB_PHASE_DEDUP = 1, EMB_PHASE_REDUCE_UPDATE = 2, EMB_NUM_PHASES = 3 };
int emb_set_timing(emb_layer* layer, int32_t enable);
int emb_phase_times(emb_layer* layer, float* ms_host, int32_t n, int64_t* steps_host, int32_t reset);

/* Static description of an emb_status value.  No passage: library convenience. */
const char* emb_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* EMB_H */
