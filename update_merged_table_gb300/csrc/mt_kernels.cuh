// Kernel parameter blocks and host-side launchers shared by the kernel files
// and the C ABI (mt_api.cu).
#pragma once

#include "mt_internal.cuh"

namespace mt {

// ---- forward ----------------------------------------------------------------

constexpr int kTile = 2048;              // positions per lookup tile (one CTA)
constexpr int kThreads = 256;            // threads per lookup CTA (number, expand)
constexpr int kPPT = kTile / kThreads;   // positions per thread
constexpr int kThreadsA = 512;           // threads per stage-1 CTA (k_local)
constexpr int kPPTA = kTile / kThreadsA; // positions per stage-1 thread
constexpr int kHS = 2 * kTile;           // shared-memory hash slots (backward fill)
constexpr int kHSA = 3 * kTile / 2;      // shared-memory hash slots of stage 1 (load <= 2/3)
constexpr int kThreadsR = 256;           // threads per resolve CTA (k_resolve)
constexpr int kThreadsC = 256;           // threads per global-claim CTA (k_claim)
constexpr uint16_t kNoIdx = 0xFFFF;

// One slot of the stage-2 scratch hash.  The lookup clears the slots to all
// ones, so a fresh slot holds key EMPTY, first = "none" and cnt = 2^32 - 1,
// i.e. cnt stores (positions - 1): an atomicAdd of c returns (positions
// added before) - 1.  After numbering, `first` holds the key's unique index
// and `cnt` its table row.
struct __align__(16) ScSlot {
  unsigned long long key;
  uint32_t first;  // smallest position holding the key (atomicMin), then its unique index
  uint32_t cnt;    // positions holding the key, minus one; then its table row
};
static_assert(sizeof(ScSlot) == 16, "scratch slot is 16 bytes");

struct LookupParams {
  TableDev T;
  const long long* ids;
  long long n;
  int F;
  int insert_missing;
  int keys_in;            // 1: ids[] already hold merged keys (no encoding; sentinels are invalid)
  int no_table;           // 1: deduplicate only; the table is not read (unique rows -1)
  long long feat_off[MT_MAX_FEATURES + 1];
  unsigned char table_ids[MT_MAX_FEATURES];
  void* out_rows;
  unsigned long long* unique_keys;
  int32_t* inverse;
  int32_t* counts;
  int32_t* unique_rows;
  long long* num_unique;
  int32_t* ranks;         // nullable
  // workspace (the scratch slots and the distinct-key counter are cleared to all ones per call)
  ScSlot* sc;             // [ss] stage-2 scratch hash
  unsigned long long ss;  // scratch slots (>= n + 1; not a power of two)
  uint32_t* ulist_n;      // distinct keys listed so far, minus one
  uint32_t* fresh_n;      // fresh rows listed so far, minus one (the word after ulist_n)
  uint32_t* rec_n;        // tile-local uniques listed so far, minus one (the word after fresh_n)
  ulonglong2* rec;        // [n] records {key, first position | count << 32}, each tile's together
  int2* rec_sr;           // [n] {scratch slot of the record's key, rank base (positions of the key in records
                          // claimed before)}
  int32_t* tile_rec;      // [ntiles] where each tile's records start
  int32_t* fresh_row;     // [n] rows inserted by this lookup
  unsigned long long* fresh_key;  // [n] their keys
  int32_t* ulist;         // [n] scratch slot of each distinct key, in claim order
  int32_t* urow;          // [n] table row of each distinct key (-1: none), beside ulist
  int32_t* tile_L;        // [ntiles] tile-local uniques per tile
  unsigned long long* owner_nb;  // [ntiles * kTile / 64] bit i clear: position i is its key's first (cleared
                                 // to all ones)
  uint16_t* wpre;         // [ntiles * kTile / 64] first positions in the tile before each 64-position word
  int32_t* prow;          // [ntiles * kTile] table row of each position (-1: none), for the gather
  int32_t* tile_pre;      // [ntiles + 1] first positions before each tile (its count, then the exclusive prefix)
  uint32_t* done;         // k_prefix blocks finished (zeroed by k_local)
  uint32_t* llr;          // [ntiles * kTile] per position: tile-local unique (low half, 0xFFFF: invalid ID) |
                          // rank among its key's positions in the tile (high half)
  int ntiles;
  int resolve_grid;
  size_t clear_bytes;     // bytes from sc on cleared to all ones per call (slots, counters, first-position bits)
};

struct LookupWsLayout {
  size_t sc, ulist_n, ulist, rec, rec_sr, fresh_row, fresh_key, urow, tile_L, owner_nb, tile_pre, done,
      wpre, prow, tile_rec, llr, total;
  size_t clear_bytes;  // bytes from the start of the workspace cleared to all ones per call
  unsigned long long ss;
  int ntiles;
};
LookupWsLayout lookup_ws_layout(long long n);
// Points the workspace fields of p into w laid out as L (n > 0).
void bind_lookup_ws(LookupParams& p, char* w, const LookupWsLayout& L);
cudaError_t launch_lookup(const LookupParams& p, cudaStream_t s);

// ---- backward ---------------------------------------------------------------

constexpr int kChunk = 32;          // most positions a light unique has (one team-chunk)
constexpr int kTeamShare = 64;      // positions per team in a heavy unique's warp-chunk
constexpr int kScanTile = 2048;     // uniques per scan block
constexpr int kScanThreads = 256;

struct BackwardParams {
  TableDev T;
  long long n;
  const int32_t* pos_map;  // nullable: gradient row of each position (-1: none); NULL means row = position
  long long grad_rows;     // rows of `grads` (n, or the number of bags)
  const int32_t* inverse;
  const int32_t* ranks;  // nullable: rank of each position among its unique's positions
  const int32_t* counts;
  const int32_t* unique_rows;
  const long long* num_unique;
  const void* grads;
  int grad_dtype;
  float lr, beta1, beta2, eps;
  float one_minus_b1, one_minus_b2;
  float* gsum_out;
  int reduce_only;      // 1: gradient sums only; no Adam step and no step counter change
  // workspace
  int32_t* ctr;         // [3] positions, heavy warp-chunks and heavy uniques placed so far (zeroed per call;
                        //     their totals once k_bw_plan is done)
  int2* seg;            // [n] {segment start, count} of each unique; the fill advances the start to the end
  int4* chunks;         // [light0 + n] descriptors {start, end, row, u or -(heavy index + 1)}: the warp-chunks of
                        //     heavy uniques (more than kChunk positions) from 0; unique u's team-chunk at
                        //     light0 + u (empty, {0, 0, -1, -1}, for a heavy unique)
  int4* heavy_info;     // [heavy_cap] {u, warp-chunks, segment start, first chunk} of each heavy unique
  int32_t* pos_sorted;  // [n] positions grouped by unique
  double* acc64;        // [heavy_cap * d] cross-chunk sums of heavy uniques
  int32_t* arrive;      // [heavy_cap] chunks finished per heavy unique
  int32_t* work;        // [4] heavy warp-chunks handed out (zeroed per call), -, step_size and inv_sqrt_bc2 (fp32 bits)
  int nblk;
  int light0;           // where the light uniques' team-chunks start in chunks (bounds the heavy warp-chunks)
  int ntiles;
  int team_shift;       // log2 lanes per team (one team covers VEC columns per lane)
  int warp_chunk;       // positions per heavy warp-chunk: kTeamShare x teams per warp
};

struct BackwardWsLayout {
  size_t ctr, seg, chunks, heavy_info, pos_sorted, acc64, arrive, work, total;
  long long heavy_cap;
  int nblk, ntiles, light0;
};
BackwardWsLayout backward_ws_layout(long long n, uint32_t dim);
// Points the workspace fields of p into w laid out as L.
void bind_backward_ws(BackwardParams& p, char* w, const BackwardWsLayout& L);
int backward_team_shift(uint32_t dim, int row_dtype);
cudaError_t launch_backward(const BackwardParams& p, cudaStream_t s);

// ---- pooled bags ---------------------------------------------------------------

struct PoolParams {
  TableDev T;
  long long n;
  const int32_t* inverse;
  const int32_t* unique_rows;
  const long long* num_unique;
  const long long* bag_offsets;  // [num_bags + 1] device
  long long num_bags;
  int mode;                      // MT_POOL_SUM or MT_POOL_MEAN
  int team_shift;                // log2 lanes per team (VEC columns per lane)
  float* out;                    // [num_bags, d]
  double* acc;                   // [num_bags, d] workspace: sums of bags split over chunks
};
cudaError_t launch_pool(const PoolParams& p, cudaStream_t s);
cudaError_t launch_pos_bag(const long long* bo, long long B, long long n, int32_t* pos_bag, Header* hdr,
                           cudaStream_t s);
cudaError_t launch_pool_scale(const long long* bo, long long B, int d, const float* dpooled, float* dscaled,
                              cudaStream_t s);

// ---- table maintenance --------------------------------------------------------

cudaError_t launch_table_init(const TableDev& T, cudaStream_t s);
cudaError_t launch_erase(const TableDev& T, const unsigned long long* keys, long long n, unsigned char* found,
                         int32_t* ws_slot, cudaStream_t s);
cudaError_t launch_compact(const TableDev& T, Slot* fresh, cudaStream_t s);
cudaError_t launch_import(const TableDev& T, const unsigned long long* keys, long long n, const float* emb,
                          const float* m, const float* v, int32_t* ws_rows, cudaStream_t s);
cudaError_t launch_grow(const TableDev& T, const TableDev& T2, cudaStream_t s);
cudaError_t launch_stats(const TableDev& T, cudaStream_t s);
cudaError_t launch_export(const TableDev& T, unsigned long long* keys, int32_t* rows, long long capacity,
                          cudaStream_t s);
cudaError_t launch_read_rows(const TableDev& T, const int32_t* rows, long long n, float* emb, float* m, float* v,
                             cudaStream_t s);

// Counts every kernel launch of the library and, while profiling is on,
// brackets it with CUDA events on its stream (mt_profile.cu).
class LaunchScope {
 public:
  LaunchScope(const char* name, cudaStream_t s);
  ~LaunchScope();
  LaunchScope(const LaunchScope&) = delete;
  LaunchScope& operator=(const LaunchScope&) = delete;

 private:
  const char* name_;
  cudaStream_t stream_;
  cudaEvent_t start_;
};

#define MT_CAT2(a, b) a##b
#define MT_CAT(a, b) MT_CAT2(a, b)
// Put at the start of a block that launches exactly one kernel.
#define MT_LAUNCH(name, stream) ::mt::LaunchScope MT_CAT(mt_launch_scope_, __LINE__)(name, stream)

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch settings (grid sizes, shared-memory attributes) are cached per
// device: a process may drive tables on several GPUs.  Entries are written
// with idempotent values, so concurrent first calls only repeat the work.
constexpr int kMaxDevices = 64;
inline int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

// ---- side streams ---------------------------------------------------------------

// Independent tables (merged groups, logical ranks) each run a chain of small
// latency-bound launches: they run side by side on the library's side streams
// of the current device and host thread (created on first use, pooled when the
// thread exits, never destroyed), forked from the caller's stream by an event
// and joined back into it before the call returns (under stream capture:
// parallel branches of the graph).
constexpr int kSideStreams = 4;
cudaError_t side_streams(cudaStream_t* out);
// Work enqueued on side[0 .. k) from now on waits for everything enqueued on s so far.
cudaError_t fork_streams(cudaStream_t s, const cudaStream_t* side, int k);
// Work enqueued on s from now on waits for everything enqueued on side[0 .. k) so far.
cudaError_t join_streams(cudaStream_t s, const cudaStream_t* side, int k);

// Where the work of the i-th table with work goes: a side stream when several
// tables have work, else the caller's stream.
struct GroupStreams {
  cudaStream_t caller = nullptr;
  cudaStream_t side[kSideStreams] = {};
  int used = 0;  // side streams forked
  cudaError_t begin(cudaStream_t s, int active) {
    caller = s;
    used = 0;
    if (active < 2) return cudaSuccess;
    const cudaError_t e = side_streams(side);
    if (e != cudaSuccess) return e;
    used = active < kSideStreams ? active : kSideStreams;
    return fork_streams(s, side, used);
  }
  cudaStream_t stream(int slot) const { return used ? side[slot % used] : caller; }
  cudaError_t end() {
    const cudaError_t e = used ? join_streams(caller, side, used) : cudaSuccess;
    used = 0;
    return e;
  }
};

// Streaming multiprocessors of the current device (queried once per device).
int sm_count();

// Blocks of `threads` for `work` items, capped at `per_sm` blocks per SM
// (grid-stride kernels loop over the rest).
inline int grid_for(long long work, int threads, int per_sm) {
  long long g = (work + threads - 1) / threads;
  const long long cap = (long long)sm_count() * per_sm;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

}  // namespace mt
