/* mt.h -- C ABI of the merged dynamic embedding table (GB300, sm_103a).
 *
 * The hot path of a dynamic hash embedding table as described in "MTGenRec:
 * An Efficient Distributed Training System for Generative Recommendation
 * Models in Meituan" (TL;DR and abstract: dynamic hash tables replacing
 * static ones so keys can be inserted and deleted while training runs, feature
 * tables merged into one, ID deduplication in two stages) and in "MTGR: Industrial-Scale Generative
 * Recommendation Framework in Meituan" (section 5, Embedding Management: keys
 * lead to embeddings plus bookkeeping data; Embedding Lookup: no duplicate IDs
 * on either side of an exchange).
 *
 * Conventions that hold for every call:
 *  - Plain C types only.  `mt_stream` is a cudaStream_t passed as void*
 *    (NULL = the legacy default stream).
 *  - The library never allocates device memory.  The caller provides the
 *    table arena, every workspace and every output, as device pointers,
 *    unless a parameter says "host".  Device buffers passed here must be
 *    16-byte aligned; arenas and workspaces 256-byte aligned.
 *  - Calls are asynchronous and stream-ordered on `stream`, except
 *    mt_stats, mt_export, mt_get_error, mt_get_adam_state,
 *    mt_set_adam_state, mt_table_grow, mt_compact and mt_shard_lookup, which
 *    synchronise it (they read or publish host-side values).  One table must
 *    be used from one stream at a time.
 *  - A negative return value is an error detected on the host; nothing has
 *    been enqueued.  Errors found on the device (an ID out of range, the
 *    probe limit or the row pool exhausted) latch the first code into a
 *    device error word that mt_stats / mt_get_error report; the affected
 *    positions get row -1 and zero output, and the call otherwise completes.
 *  - No kernel of this library waits on another block or another launch:
 *    every probe loop is bounded by the table's probe limit, and where the
 *    last block of a launch finishes a scan it only reads what the earlier
 *    blocks published before they counted themselves done.
 */
#ifndef MT_H
#define MT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MT_ABI_VERSION 2

/* Status codes. */
enum {
  MT_OK = 0,
  MT_EINVAL = -1,   /* bad argument (even probe step, bad dim, bad offsets, ...) */
  MT_ENOSPACE = -2, /* arena or workspace too small or misaligned */
  MT_EFULL = -3,    /* device: probe limit reached or row pool exhausted */
  MT_EKEY = -4,     /* device: an ID outside [0, 2^56) */
  MT_ECUDA = -5,    /* a CUDA runtime call failed */
  MT_ETOOBIG = -6   /* batch larger than a fixed-size entry point allows (mt_lookup_static) */
};

/* Element types of rows and gradients. */
enum { MT_F32 = 0, MT_BF16 = 1 };

/* Merged key = (table_id << 56) | id with table_id in [0, 254] and id in
 * [0, 2^56) (feature tables merged into one table, MTGenRec TL;DR).  Table id 255 is
 * reserved for the two slot sentinels. */
#define MT_KEY_EMPTY 0xFFFFFFFFFFFFFFFFull
#define MT_KEY_TOMBSTONE 0xFFFFFFFFFFFFFFFEull
#define MT_MAX_FEATURES 256

#define MT_MAX_DIM 1024
#define MT_HIST_BINS 64

typedef struct mt_table mt_table; /* opaque host handle, owned by the library */
typedef void* mt_stream;

/* Table configuration.
 *  log2_slots  n: the key store has M = 2^n slots, 1 <= n <= 31.
 *  dim         d: embedding width; a multiple of 4 (fp32 rows) or 8 (bf16
 *              rows), 4 <= d <= MT_MAX_DIM.
 *  row_dtype   MT_F32 or MT_BF16 storage of the embedding; the Adam moments
 *              m and v are always fp32.
 *  max_probes  probe limit per key; 0 means M.
 *  probe_step  S of the probe sequence h_t = (h0 + t*S) mod M (MTGenRec,
 *              Theorem 1).  Used mod M; it must be odd, which makes the
 *              sequence visit every slot.  An even S is MT_EINVAL.
 *  hash_seed   h0 = top n bits of splitmix64-finaliser(key ^ hash_seed).
 *  init_seed   fresh rows: column j = scale * (2q - 2^24) / 2^24 with q
 *              24 bits of word (j/2)%4 of Philox4x64-10(counter (j/8,0,0,0),
 *              key (merged key, init_seed)): bits 63..40 for an even j, bits
 *              39..16 for an odd j; m = v = 0.
 *  init_scale  0 means fp32(1/sqrt(d)).
 *  num_rows    R, rows in the row pool; 0 means M.  1 <= R <= M. */
typedef struct {
  uint32_t log2_slots;
  uint32_t dim;
  uint32_t row_dtype;
  uint32_t max_probes;
  uint64_t probe_step;
  uint64_t hash_seed;
  uint64_t init_seed;
  float init_scale;
  uint32_t flags; /* must be 0 (reserved) */
  int64_t num_rows;
} mt_config;

/* Per-batch result of mt_lookup; all pointers are device buffers of
 * capacity n (the batch size) owned by the caller.  It stays valid for
 * mt_backward_adam until the next mt_lookup or mt_erase on the table. */
typedef struct {
  uint64_t* unique_keys; /* [n]: first U entries: the distinct merged keys in first-occurrence order */
  int32_t* inverse;      /* [n]: unique_keys[inverse[i]] is the key of position i; -1 for an invalid ID */
  int32_t* counts;       /* [n]: first U entries: number of positions holding each unique key */
  int32_t* unique_rows;  /* [n]: first U entries: row of each unique key, -1 when it has none */
  int64_t* num_unique;   /* [1]: U */
  int32_t* ranks;        /* [n] or NULL: rank of position i among the counts[inverse[i]] positions of its
                            key, in an unspecified order (-1 for an invalid ID).  With ranks the backward
                            groups positions by key without hashing them again. */
} mt_lookup_result;

/* Adam hyper-parameters (Meituan TensorFlow article, section 3.2 names Adam;
 * the update is Kingma & Ba's with bias correction, see mt_backward_adam). */
typedef struct {
  float lr, beta1, beta2, eps;
} mt_adam;

/* Occupancy of the key store (MTGenRec, Theorem 1 probe sequence). */
typedef struct {
  int64_t live;               /* slots holding a key */
  int64_t tombstones;         /* slots holding MT_KEY_TOMBSTONE */
  int64_t capacity;           /* M */
  int64_t num_rows;           /* R */
  int64_t rows_free;          /* rows on the free list */
  int64_t step;               /* Adam steps taken (mt_backward_adam calls) */
  int64_t total_displacement; /* sum over live keys of their probe index t */
  double load_factor;         /* live / M */
  int64_t probe_hist[MT_HIST_BINS]; /* live keys by probe index t; the last bin holds t >= 63 */
  int32_t device_error;       /* first latched device error code, 0 if none */
  int32_t reserved;
} mt_stats_out;

/* ---- table ------------------------------------------------------------- */

/* A table lives in caller-owned device memory in two kinds of parts: one key
 * store (a header, M 16-byte slots {key, row, insert step} and the row free
 * list, R int32) and up to MT_MAX_ROW_SEGMENTS row segments holding the row
 * records [emb d x row dtype | m d x fp32 | v d x fp32], each part padded to
 * 16 bytes.  Keys lead to rows through the key store only (MTGR section 5,
 * Embedding Management), so growing the table or compacting its key store
 * rebuilds the key store and never moves a row. */
#define MT_MAX_ROW_SEGMENTS 8

/* Bytes of a single arena holding the key store followed by all R rows (the
 * layout mt_table_create uses).  Returns 0 for an invalid configuration. */
size_t mt_table_bytes(const mt_config* cfg);

/* Bytes of the key store alone for `cfg` (header, M slots, free list of
 * cfg->num_rows entries).  Returns 0 for an invalid configuration. */
size_t mt_keystore_bytes(const mt_config* cfg);

/* Bytes of a row segment of `rows` records for `cfg`'s dim and row dtype. */
size_t mt_rows_bytes(const mt_config* cfg, int64_t rows);

/* Build a table in caller-owned device memory `dev_mem` (>= mt_table_bytes
 * bytes, 256-byte aligned; owned by the caller and used by the table until
 * it is destroyed): the key store first, then one row segment of all R rows.
 * Marks every slot EMPTY and every row free, enqueued on `stream`.  *out
 * receives a host handle. */
int mt_table_create(const mt_config* cfg, void* dev_mem, size_t bytes, mt_stream stream, mt_table** out);

/* The same with the key store and the rows in separate caller-owned buffers:
 * `keystore` (>= mt_keystore_bytes) and `rows` (>= mt_rows_bytes(cfg, R)),
 * both 256-byte aligned and not overlapping. */
int mt_table_create_split(const mt_config* cfg, void* keystore, size_t keystore_bytes, void* rows,
                          size_t rows_bytes, mt_stream stream, mt_table** out);

/* Free the host handle (not the arena). */
int mt_table_destroy(mt_table* t);

/* The configuration with defaults filled in (S reduced mod M, max_probes,
 * init_scale, num_rows). */
int mt_table_config(const mt_table* t, mt_config* out);

/* ---- forward: encode, two-stage dedup, find/insert, gather -------------- */

/* Workspace bytes mt_lookup needs for a batch of n IDs. */
size_t mt_lookup_workspace_bytes(const mt_table* t, int64_t n);

/* Lookup of one batch of n IDs (MTGenRec TL;DR: merged tables and two-stage
 * ID deduplication; MTGR section 5, Embedding Lookup).
 *  ids           device int64 [n]: raw feature IDs.
 *  feat_offsets  host int64 [F+1]: positions [feat_offsets[f], feat_offsets[f+1])
 *                belong to feature table f; 0 = off[0] <= ... <= off[F] = n.
 *                NULL means F = 1 covering all n.
 *  table_ids     host uint8 [F]: the table id of each feature, < 255.  NULL
 *                means table id 0 for every feature.
 *  insert_missing  1: absent keys are inserted with a fresh row ("real-time
 *                insertions", MTGenRec abstract); 0: they get row -1.
 *  out_rows      device [n, d] of the row dtype, or NULL to skip the gather:
 *                out_rows[i] = embedding of key i (zeros for an invalid ID or
 *                an absent key).
 *  res           caller-owned result buffers (see mt_lookup_result).
 *  ws, ws_bytes  device workspace of mt_lookup_workspace_bytes(t, n) bytes;
 *                its contents are scratch and need no initialisation.
 * Device errors: an ID outside [0, 2^56) latches MT_EKEY (inverse -1); a full
 * chain or an empty row pool latches MT_EFULL (row -1). */
int mt_lookup(mt_table* t, const int64_t* ids, int64_t n, const int64_t* feat_offsets, const uint8_t* table_ids,
              int F, int insert_missing, void* out_rows, const mt_lookup_result* res, void* ws, size_t ws_bytes,
              mt_stream stream);

/* The same lookup for callers that cannot allocate device memory when they
 * call it (an operator or plugin interface that only passes its inputs and
 * outputs, or a serving process whose memory budget is fixed at start-up):
 * the workspace comes from a static device array inside the library instead
 * of `ws`, so at most MT_LOOKUP_STATIC_MAX_IDS IDs per call; larger n returns
 * MT_ETOOBIG with nothing enqueued.  The pages have no counterpart; this is
 * an interface convenience, not part of the method.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every GPU that loads the library holds the array (6 MiB) until exit.
 *  - All calls share the array: calls whose work overlaps on the GPU (other
 *    streams or host threads) race on it.  The array keeps the last call's
 *    contents; each call clears what it needs cleared.
 *  - Otherwise identical to mt_lookup: same arguments, results and errors. */
#define MT_LOOKUP_STATIC_MAX_IDS 65536
int mt_lookup_static(mt_table* t, const int64_t* ids, int64_t n, const int64_t* feat_offsets, const uint8_t* table_ids,
                     int F, int insert_missing, void* out_rows, const mt_lookup_result* res, mt_stream stream);

/* ---- backward: per-unique gradient sum + sparse row-wise Adam ------------ */

/* Workspace bytes mt_backward_adam needs for a batch of n IDs. */
size_t mt_backward_workspace_bytes(const mt_table* t, int64_t n);

/* Backward of the lookup `res` (same n): g_u = sum of grads[i] over positions
 * i with inverse[i] = u, accumulated in at least fp32 pair precision and
 * rounded once to fp32; then, for every unique key with a row, one Adam step
 * in fp32 with the table's step counter t (advanced once per call):
 *   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*g*g;
 *   w = w - step_size * (m / (sqrt(v) * inv_sqrt_bc2 + eps))
 * with step_size = lr / (1-b1^t) and inv_sqrt_bc2 = 1 / sqrt(1-b2^t), i.e.
 * Kingma & Ba's m_hat / (sqrt(v_hat) + eps) with the bias corrections folded
 * into per-step scalars (1-b1, 1-b2 and both scalars evaluated in double,
 * then rounded to fp32; every per-element operation rounds once).  b1^t and
 * b2^t are the table's beta-power accumulators (Meituan TensorFlow article,
 * section 3.2): starting from 1, each call multiplies them (in double) by
 * that call's b1 and b2.
 * Rows absent from the batch are not touched.
 *  grads      device [n, d] of grad_dtype (MT_F32 or MT_BF16).
 *  gsum_out   device fp32 [n, d] or NULL: the first U rows receive g_u.
 *  ws         device workspace of mt_backward_workspace_bytes(t, n) bytes. */
int mt_backward_adam(mt_table* t, const mt_lookup_result* res, int64_t n, const void* grads, int grad_dtype,
                     const mt_adam* hp, float* gsum_out, void* ws, size_t ws_bytes, mt_stream stream);

/* ---- pooled bags of a jagged batch ------------------------------------------ */

/* A bag is a run of consecutive positions [bag_offsets[b], bag_offsets[b+1])
 * of a lookup batch; in a jagged sequence batch one bag holds one user's
 * tokens of one feature (MTGR section 5, Load Balance: user sequences of very
 * different lengths).  Pooling replaces the bag's rows by their sum or mean. */
#define MT_POOL_SUM 0
#define MT_POOL_MEAN 1

/* Workspace bytes mt_pool_forward needs for num_bags bags (an fp64 [num_bags, d] accumulator). */
size_t mt_pool_workspace_bytes(const mt_table* t, int64_t num_bags);

/* Pooled embeddings of the lookup `res` (same n, as the table holds the rows
 * now): out[b] = sum of the rows of the keys at the bag's positions (zero
 * rows for invalid IDs and absent keys), divided by the bag's length for
 * MT_POOL_MEAN; accumulated as exact fp32 pairs and fp64, rounded once to
 * fp32.  Empty bags give zeros.
 *  bag_offsets  device int64 [num_bags + 1], non-decreasing within [0, n];
 *               positions outside [bag_offsets[0], bag_offsets[num_bags])
 *               are in no bag.  Offsets that break this latch MT_EINVAL on
 *               the device (those bags read as zeros; every access stays in
 *               bounds).
 *  out          device fp32 [num_bags, d].
 *  ws           device workspace of mt_pool_workspace_bytes(t, num_bags) bytes. */
int mt_pool_forward(mt_table* t, const mt_lookup_result* res, int64_t n, const int64_t* bag_offsets,
                    int64_t num_bags, int mode, float* out, void* ws, size_t ws_bytes, mt_stream stream);

/* Workspace bytes mt_backward_adam_pooled needs. */
size_t mt_backward_pooled_workspace_bytes(const mt_table* t, int64_t n, int64_t num_bags);

/* Backward of mt_pool_forward followed by mt_backward_adam, with no
 * per-position gradient rows: every position of bag b takes the gradient
 * dpooled[b] (MT_POOL_SUM) or dpooled[b] * s_b rounded once to fp32 with
 * s_b = fp32(1 / len_b) (MT_POOL_MEAN); positions in no bag take zero.  Then
 * exactly the per-unique sum and Adam step of mt_backward_adam (the table's
 * step counter advances once).
 *  dpooled   device fp32 [num_bags, d].
 *  ws        device workspace of mt_backward_pooled_workspace_bytes bytes. */
int mt_backward_adam_pooled(mt_table* t, const mt_lookup_result* res, int64_t n, const int64_t* bag_offsets,
                            int64_t num_bags, int mode, const float* dpooled, const mt_adam* hp, float* gsum_out,
                            void* ws, size_t ws_bytes, mt_stream stream);

/* ---- automatic table merging ------------------------------------------------ */

/* Feature tables merged into shared tables (MTGenRec TL;DR and abstract:
 * automatic table merging, so a batch needs fewer lookups).  The pages give
 * no grouping rule; this one is used: features whose tables have the same
 * row shape (dim and row dtype) share a merged table, in order of first
 * appearance, each feature keeping its own key space through its table id
 * (0, 1, 2, ... in feature order; a merged table holds at most 255 features,
 * more open another one of the same shape). */
typedef struct {
  uint32_t dim;       /* the feature table's embedding width */
  uint32_t row_dtype; /* MT_F32 or MT_BF16 */
  int64_t capacity;   /* keys the feature's table is expected to hold (>= 0) */
} mt_feature_spec;

typedef struct {
  int32_t group;    /* the merged table the feature goes to */
  uint8_t table_id; /* its table id there */
  uint8_t pad[3];
} mt_feature_placement;

typedef struct {
  uint32_t dim, row_dtype;
  uint32_t log2_slots; /* the smallest n >= 1 with capacity <= max_load * 2^n */
  int32_t num_features;
  int64_t capacity;    /* the sum of its features' capacities */
} mt_merge_group;

/* Plan the merged tables of F features (1 <= F <= MT_MAX_FEATURES) with
 * 0 < max_load <= 1: placement [F] and groups [F] (host) receive the plan,
 * *num_groups the number of merged tables.  MT_EINVAL for a bad row shape, a
 * negative capacity, or a group that would need more than 2^31 slots. */
int mt_plan_merge(const mt_feature_spec* features, int F, double max_load, mt_feature_placement* placement,
                  mt_merge_group* groups, int* num_groups);

/* Workspace bytes mt_lookup_grouped needs for a batch of n IDs in F feature
 * segments, however the features split it among the groups. */
size_t mt_lookup_grouped_workspace_bytes(int64_t n, int F);

/* Lookup of one batch of F feature segments over the merged tables of a plan:
 * the segments of the features placed in group g are routed, in feature
 * order, into one batch for tables[g] (its feature offsets and table ids from
 * the plan), and looked up there as mt_lookup does.
 *  tables       host array [G] of distinct merged tables (rows of group g's shape).
 *  ids          device int64 [n]; feat_offsets host int64 [F + 1] (0 .. n).
 *  out_rows     host array [G] of device pointers [group_n[g], d_g] (entries
 *               or the array may be NULL).
 *  results      host array [G], each of capacity >= the group's IDs.
 *  group_n      host int64 [G]: receives each group's number of IDs.
 * When more than one group receives IDs, the groups run side by side on the
 * library's own side streams of the current device: up to four per host
 * thread, so that calls from different threads (or one thread's stream
 * capture) never share one; a thread's streams are created on its first such
 * call, go back to a pool when it exits and are kept until the process exits.
 * They wait for the work enqueued on `stream` before the call, and work
 * enqueued on `stream` after the call waits for all of them, also when the
 * call returns an error.  Under stream capture this records parallel branches
 * of the graph.
 * The backward of group g is mt_backward_adam(tables[g], &results[g],
 * group_n[g], ...) with that group's gradient rows, or all groups at once with
 * mt_backward_adam_grouped. */
int mt_lookup_grouped(mt_table* const* tables, int G, const mt_feature_placement* placement, const int64_t* ids,
                      int64_t n, const int64_t* feat_offsets, int F, int insert_missing, void* const* out_rows,
                      const mt_lookup_result* results, int64_t* group_n, void* ws, size_t ws_bytes,
                      mt_stream stream);

/* Workspace bytes mt_backward_adam_grouped needs: the groups' backward
 * workspaces (mt_backward_workspace_bytes(tables[g], group_n[g])) side by side. */
size_t mt_backward_grouped_workspace_bytes(mt_table* const* tables, int G, const int64_t* group_n);

/* mt_backward_adam of every group of a grouped lookup: group g's call gets
 * tables[g], &results[g], group_n[g], grads[g] (device [group_n[g], d_g] of
 * grad_dtype) and gsum_out[g] (gsum_out may be NULL; so may its entries), and
 * the groups run side by side as in mt_lookup_grouped.  The tables must be
 * distinct (each call advances its table's step counter).  Every group's
 * arguments are checked before anything is enqueued. */
int mt_backward_adam_grouped(mt_table* const* tables, int G, const mt_lookup_result* results, const int64_t* group_n,
                             const void* const* grads, int grad_dtype, const mt_adam* hp, float* const* gsum_out,
                             void* ws, size_t ws_bytes, mt_stream stream);

/* ---- sharded two-stage deduplication (G logical shards on one GPU) ------- */

/* The distributed form of the lookup (MTGR section 5, Embedding Lookup:
 * deduplicated IDs on both sides of the cross-device all-to-all; MTGenRec
 * TL;DR: two-stage ID deduplication), with G logical ranks on one GPU.  Each
 * rank r owns the keys whose owner(key) (a second hash of the key mapped to
 * [0, G)) is r and keeps them in its shard table; each rank has its own
 * batch.  Forward: stage-1 unique per rank; the (rank, owner) counts are read
 * on the host (the sizes of a variable all-to-all); every rank writes its
 * unique keys into the owners' receive buffers (the exchange, a device-local
 * copy here); stage-2 unique, find/insert and gather at each owner; rows back
 * to the ranks, and each rank expands them through its inverse.  Backward:
 * per-rank sums per unique key, sums to the owners, per-key sums over the
 * ranks and one Adam step on every shard.  The shards must share dim, row
 * dtype, init seed and init scale (a key's row does not depend on its owner).
 * These calls synchronise the stream (the exchange sizes are read on the
 * host), so they cannot be captured in a CUDA graph. */
#define MT_MAX_SHARDS 16
typedef struct mt_shard_group mt_shard_group; /* opaque host handle */

/* Group G distinct tables (1 <= G <= MT_MAX_SHARDS) as the shards of one logical table. */
int mt_shard_group_create(mt_table* const* shards, int G, mt_shard_group** out);
int mt_shard_group_destroy(mt_shard_group* g);

/* Workspace bytes for batches of n[r] IDs (host int64 [G]); the lookup and its
 * backward take the same workspace, which keeps the exchange layout between them. */
size_t mt_shard_workspace_bytes(const mt_shard_group* g, const int64_t* n);

/* Forward of one step of all G ranks.
 *  ids          host array of G device pointers: rank r's IDs, int64 [n[r]].
 *  n            host int64 [G].
 *  feat_offsets host int64 [G * (F + 1)]: rank r's feature offsets (as in
 *               mt_lookup); NULL means F = 1 for every rank.
 *  table_ids    host uint8 [F] (< 255), shared by the ranks; NULL means 0.
 *  out_rows     host array of G device pointers [n[r], d] (entries or the
 *               array may be NULL: no rows for that rank).
 *  results      host array of G mt_lookup_result: rank r's unique keys in
 *               first-occurrence order of its own batch, inverse, counts,
 *               ranks (nullable) and num_unique; unique_rows are set to -1
 *               (the rows live in the owners' shards).
 * The rows a rank receives equal what one table holding every key would give.
 * The ranks' stage-1 lookups, and then the owners' stage-2 lookups, run side by
 * side on the library's side streams (as in mt_lookup_grouped), joined back
 * into `stream`; the host reads of the exchange sizes synchronise it. */
int mt_shard_lookup(mt_shard_group* g, const int64_t* const* ids, const int64_t* n, const int64_t* feat_offsets,
                    const uint8_t* table_ids, int F, int insert_missing, void* const* out_rows,
                    const mt_lookup_result* results, void* ws, size_t ws_bytes, mt_stream stream);

/* Backward of the last mt_shard_lookup (same results and workspace): grads is a
 * host array of G device pointers [n[r], d] of grad_dtype.  Every key's
 * gradient is summed over all positions of all ranks (rank sums rounded to
 * fp32, then summed exactly at the owner and rounded once), then one Adam step
 * is applied by its owner; every shard's step counter advances once.  The
 * ranks' sums, and then the owners' Adam steps, run side by side on the side
 * streams, joined back into `stream`.
 *  gsum_out  NULL, or a host array of G device pointers fp32 [U_r, d] (entries
 *            may be NULL): rank r's unique keys' sums over all ranks. */
int mt_shard_backward_adam(mt_shard_group* g, const mt_lookup_result* results, const void* const* grads,
                           int grad_dtype, const mt_adam* hp, float* const* gsum_out, void* ws, size_t ws_bytes,
                           mt_stream stream);

/* ---- deletion ------------------------------------------------------------ */

/* Workspace bytes mt_erase needs for n keys. */
size_t mt_erase_workspace_bytes(int64_t n);

/* Delete n merged keys (keys deleted while training runs, MTGenRec abstract): a live
 * key's slot becomes MT_KEY_TOMBSTONE, which later probes pass over and
 * later inserts may reuse, and its row returns to the free list.  A key
 * inserted again later starts from its initial row with m = v = 0.
 *  keys   device uint64 [n] merged keys (duplicates allowed).
 *  found  device uint8 [n] or NULL: 1 when the key was live before the call
 *         (every duplicate of a live key reports 1). */
int mt_erase(mt_table* t, const uint64_t* keys, int64_t n, uint8_t* found, void* ws, size_t ws_bytes,
             mt_stream stream);

/* ---- inspection ------------------------------------------------------------ */

/* Capacity expansion (MTGR section 5, Embedding Management: the key store is
 * replicated, the embeddings are not).  new_cfg may have more slots
 * (log2_slots) and more rows (num_rows) but must otherwise equal the table's
 * configuration (dim, row dtype, probe step, seeds, init scale, flags;
 * max_probes 0 means the new M).  A new key store is built in `keystore`
 * (>= mt_keystore_bytes(new_cfg), 256-byte aligned, overlapping none of the
 * table's memory): the header and the Adam state are copied, the free list
 * is copied and extended by the new rows, and every live key is inserted
 * again along its probe sequence in the larger slot array.  The new rows
 * (new_cfg->num_rows - R of them) form a new row segment in `rows`
 * (>= mt_rows_bytes(new_cfg, new R - R) bytes; NULL when no rows are added);
 * existing rows stay where they are, with the same row indices.  At most
 * MT_MAX_ROW_SEGMENTS segments (else MT_EINVAL).  Synchronises `stream`.  On
 * success the table uses the new key store, and the old one (which the caller
 * may free, unless it shares an allocation with rows) is no longer read.  If
 * a key does not fit within the new max_probes, MT_EFULL is returned and the
 * table keeps its old key store, unchanged.  CUDA graphs captured before the
 * call must be captured again. */
int mt_table_grow(mt_table* t, const mt_config* new_cfg, void* keystore, size_t keystore_bytes, void* rows,
                  size_t rows_bytes, mt_stream stream);

/* Bytes of the slot array mt_compact needs: M x 16. */
size_t mt_compact_workspace_bytes(const mt_table* t);

/* Tombstone compaction of the key store.  Every live key is inserted again,
 * with its row and insertion step, along its probe sequence
 * h_t = (h0 + t*S) mod M into the fresh slot array `ws` (>=
 * mt_compact_workspace_bytes, 256-byte aligned, not the table's slots),
 * which then becomes the table's slot array: no slots are copied back.
 * Tombstones disappear and chains shorten; rows, the free list, the step
 * counter and every key's row stay as they were.  On success *released
 * receives the slot array the table used before: that memory belongs to the
 * caller again (it lies in the caller's key store, or in an earlier `ws`)
 * and may serve as the next call's `ws`; `ws` must stay allocated while the
 * table uses it.  If a key would need more than max_probes probes in the new
 * order (possible only with a small max_probes), MT_EFULL is returned and the
 * table is unchanged (*released = NULL).  Synchronises `stream`.  CUDA graphs
 * captured before the call must be captured again. */
int mt_compact(mt_table* t, void* ws, size_t ws_bytes, void** released, mt_stream stream);

/* Scan the key store: live keys, tombstones, and each live key's probe index
 * t = (slot - h0) * S^-1 mod M (S is odd, so S^-1 mod 2^n exists; MTGenRec
 * Theorem 1).  Synchronises `stream`. */
int mt_stats(mt_table* t, mt_stats_out* out, mt_stream stream);

/* Copy up to `capacity` live (key, row) pairs into device buffers keys/rows
 * (in no particular order) and the number of live keys into *count (host).
 * Synchronises `stream`.  (export by a scan of the key store, MTGR section 5.) */
int mt_export(mt_table* t, uint64_t* keys, int32_t* rows, int64_t capacity, int64_t* count, mt_stream stream);

/* Read n rows (device int32 row indices; -1 gives zeros) as fp32 into device
 * buffers emb, m, v ([n, d] each; any may be NULL). */
int mt_read_rows(const mt_table* t, const int32_t* rows, int64_t n, float* emb, float* m, float* v,
                 mt_stream stream);

/* Workspace bytes mt_import needs for n keys. */
size_t mt_import_workspace_bytes(int64_t n);

/* Checkpoint restore (with mt_export, mt_read_rows and the Adam state
 * below): for each of n merged keys, find the key or insert it as a lookup
 * would (first tombstone-or-EMPTY slot of its chain, a row from the free
 * list), then write its row: embedding emb[i] (fp32; stored with
 * round-to-nearest-even when the rows are bf16), moments m[i] and v[i].
 *  keys        device uint64 [n] merged keys; they must be distinct (with
 *              duplicates the table's contents are unspecified, but every
 *              access stays in bounds).  A sentinel key latches MT_EKEY.
 *  emb, m, v   device fp32 [n, d].
 *  ws          device, >= mt_import_workspace_bytes(n), 256-byte aligned.
 * A full chain or an empty row pool latches MT_EFULL for that key. */
int mt_import(mt_table* t, const uint64_t* keys, int64_t n, const float* emb, const float* m, const float* v,
              void* ws, size_t ws_bytes, mt_stream stream);

/* The table's Adam state: steps taken and the beta-power accumulators
 * b1^t and b2^t (see mt_backward_adam).  Both synchronise `stream`. */
int mt_get_adam_state(mt_table* t, int64_t* step, double* b1pow, double* b2pow, mt_stream stream);
int mt_set_adam_state(mt_table* t, int64_t step, double b1pow, double b2pow, mt_stream stream);

/* The first latched device error (0 if none) into *device_error (host);
 * clears it when `clear` is non-zero.  Synchronises `stream`. */
int mt_get_error(mt_table* t, int32_t* device_error, int clear, mt_stream stream);

/* Adam steps taken so far (host-side count of mt_backward_adam calls). */
int64_t mt_step(const mt_table* t);

/* ---- tracing ------------------------------------------------------------- */

/* Per-kernel device time, measured with CUDA events recorded on the
 * launching stream around each kernel while profiling is on. */
typedef struct {
  char name[40];
  int64_t launches;
  double total_ms;
} mt_kernel_time;

/* Turn per-kernel event timing on or off for every table of the process
 * (off by default; when on, each launch adds two event records). */
int mt_profile_enable(int on);

/* Synchronise the recorded events and return accumulated per-kernel totals
 * (up to `capacity` entries; *count receives how many kernels have totals);
 * clears the totals when `reset` is non-zero. */
int mt_profile_report(mt_kernel_time* out, int capacity, int* count, int reset);

/* Number of kernels this library has launched in the process. */
int64_t mt_kernel_launches(void);

const char* mt_strerror(int code);
int mt_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MT_H */
