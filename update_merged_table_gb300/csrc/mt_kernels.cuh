// Kernel parameter blocks and host-side launchers shared by the kernel files
// and the C ABI (mt_api.cu).
#pragma once

#include "mt_internal.cuh"

namespace mt {

// ---- forward ----------------------------------------------------------------

constexpr int kTile = 2048;              // positions per lookup tile (one CTA)
constexpr int kThreads = 256;            // threads per lookup CTA
constexpr int kPPT = kTile / kThreads;   // positions per thread
constexpr int kThreadsA = 512;           // threads per dedup CTA (k_dedup_claim)
constexpr int kPPTA = kTile / kThreadsA; // positions per dedup thread
constexpr int kHS = 2 * kTile;           // shared-memory hash slots (backward fill)
constexpr int kHSA = 3 * kTile / 2;      // shared-memory hash slots of stage 1 (load <= 2/3)
constexpr uint16_t kNoIdx = 0xFFFF;

struct LookupParams {
  TableDev T;
  const long long* ids;
  long long n;
  int F;
  int insert_missing;
  long long feat_off[MT_MAX_FEATURES + 1];
  unsigned char table_ids[MT_MAX_FEATURES];
  void* out_rows;
  unsigned long long* unique_keys;
  int32_t* inverse;
  int32_t* counts;
  int32_t* unique_rows;
  long long* num_unique;
  int32_t* ranks;         // nullable
  // workspace
  // stage-2 global scratch hash, one array per field (keys and first
  // positions start all-ones; unique indices are written before they are read)
  unsigned long long* sc_key;
  uint32_t* sc_minpos;
  int32_t* sc_uidx;
  int32_t* sc_row;        // table row of the key, written by its claimer (-1: absent)
  unsigned long long scratch_mask;
  int32_t* tile_L;        // [ntiles] local uniques per tile
  unsigned long long* tile_status;  // [ntiles] owner-count scan: flag << 32 | count (cleared by k_dedup_claim)
  int32_t* ticket;        // tiles handed to k_assign_resolve blocks in start order
  uint32_t* lfirst;       // [ntiles * kTile] first global position of local unique l
  uint32_t* lsslot;       // [ntiles * kTile] its scratch slot
  uint16_t* lidx;         // [ntiles * kTile] local unique index of each position
  int ntiles;
};

struct LookupWsLayout {
  size_t sc_key, sc_minpos, sc_uidx, sc_row, tile_L, tile_status, ticket, lfirst, lsslot, lidx, total;
  unsigned long long scratch_slots;
  int ntiles;
};
LookupWsLayout lookup_ws_layout(long long n);
cudaError_t launch_lookup(const LookupParams& p, cudaStream_t s);

// ---- backward ---------------------------------------------------------------

constexpr int kChunk = 32;          // most positions a light unique has (one team-chunk)
constexpr int kTeamShare = 64;      // positions per team in a heavy unique's warp-chunk
constexpr int kScanTile = 2048;     // uniques per scan block
constexpr int kScanThreads = 256;

struct BackwardParams {
  TableDev T;
  long long n;
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
  // workspace
  int32_t* bsum;        // [nblk * 3] per scan block: sums of counts, heavy chunks, heavy uniques
  int32_t* boff;        // [(nblk + 1) * 3] exclusive offsets (+ totals)
  int2* seg;            // [n] {segment start, count} of each unique; the fill advances the start to the end
  int4* chunks;         // [n] descriptors {start, end, row, u or -(heavy index + 1)}: the warp-chunks of
                        //     heavy uniques (more than kChunk positions) first, then one team-chunk per light unique
  int4* heavy_info;     // [heavy_cap] {u, warp-chunks, segment start, first chunk} of each heavy unique
  int32_t* pos_sorted;  // [n] positions grouped by unique
  double* acc64;        // [heavy_cap * d] cross-chunk sums of heavy uniques
  int32_t* arrive;      // [heavy_cap] chunks finished per heavy unique
  int32_t* work;        // [4] heavy warp-chunks handed out (zeroed per call), -, step_size and inv_sqrt_bc2 (fp32 bits)
  int nblk;
  int ntiles;
  int team_shift;       // log2 lanes per team (one team covers VEC columns per lane)
  int warp_chunk;       // positions per heavy warp-chunk: kTeamShare x teams per warp
};

struct BackwardWsLayout {
  size_t bsum, boff, seg, chunks, heavy_info, pos_sorted, acc64, arrive, work, total;
  long long heavy_cap;
  int nblk, ntiles;
};
BackwardWsLayout backward_ws_layout(long long n, uint32_t dim);
int backward_team_shift(uint32_t dim, int row_dtype);
cudaError_t launch_backward(const BackwardParams& p, cudaStream_t s);

// ---- table maintenance --------------------------------------------------------

cudaError_t launch_table_init(const TableDev& T, cudaStream_t s);
cudaError_t launch_erase(const TableDev& T, const unsigned long long* keys, long long n, unsigned char* found,
                         int32_t* ws_slot, cudaStream_t s);
cudaError_t launch_compact(const TableDev& T, void* ws, cudaStream_t s);
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

}  // namespace mt
