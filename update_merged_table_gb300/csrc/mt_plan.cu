// Automatic table merging: a plan that puts feature tables into merged
// tables, and the lookup that routes a batch's feature segments to them.
//
// Pages: "MTGenRec" TL;DR and abstract (feature tables merged into one
// automatically, so a batch needs fewer lookups).  The pages give no
// grouping rule; the plainest one the rest supports is used: features whose
// tables have the same row shape (dim and row dtype) can share one table, and
// inside it each keeps its own key space through its table id (the merged key
// (table_id << 56) | id).
#include <cstring>
#include <mutex>
#include <vector>

#include "mt_kernels.cuh"

namespace mt {
int lookup_group_status(const mt_lookup_result* res, const void* out_rows);
int backward_group_status(const mt_table* t, const mt_lookup_result* res, int64_t n, const void* grads,
                          int grad_dtype, const mt_adam* hp, const float* gsum_out);

namespace {

constexpr int kRouteSegs = 64;  // segments per routing launch (kernel parameter space)

struct RouteSegs {
  long long src[kRouteSegs];  // first position of the segment in the batch
  long long dst[kRouteSegs];  // first position in the group's batch
  long long len[kRouteSegs];
  int count;
};

// The group's batch: each of its feature segments copied from the batch.
__global__ void __launch_bounds__(256) k_route(const long long* ids, long long* out, const RouteSegs segs) {
  for (int s = blockIdx.y; s < segs.count; s += gridDim.y) {
    const long long len = segs.len[s];
    const long long* src = ids + segs.src[s];
    long long* dst = out + segs.dst[s];
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < len; i += (long long)gridDim.x * blockDim.x)
      dst[i] = __ldg(&src[i]);
  }
}

}  // namespace

// The library's side streams: one set of kSideStreams per device and host
// thread, so that a call on one thread (or a stream capture it is making)
// never enqueues onto a stream that another thread's call is using.  When a
// thread exits, its sets go back to a pool that later threads draw from;
// streams are never destroyed.  The pool and its lock are never freed, so a
// thread may exit at any point of the process's shutdown.
namespace {
struct SideSet {
  cudaStream_t s[kSideStreams];
};
std::mutex& side_pool_mu() {
  static std::mutex* m = new std::mutex;
  return *m;
}
std::vector<SideSet>* side_pool() {  // [kMaxDevices]
  static std::vector<SideSet>* v = new std::vector<SideSet>[kMaxDevices];
  return v;
}
struct ThreadSides {
  SideSet set[kMaxDevices] = {};
  bool have[kMaxDevices] = {};
  ~ThreadSides() {
    std::lock_guard<std::mutex> lk(side_pool_mu());
    for (int d = 0; d < kMaxDevices; ++d)
      if (have[d]) side_pool()[d].push_back(set[d]);
  }
};
thread_local ThreadSides t_sides;
}  // namespace

cudaError_t side_streams(cudaStream_t* out) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  ThreadSides& ts = t_sides;
  if (!ts.have[dev]) {
    SideSet x{};
    bool pooled = false;
    {
      std::lock_guard<std::mutex> lk(side_pool_mu());
      std::vector<SideSet>& v = side_pool()[dev];
      if (!v.empty()) {
        x = v.back();
        v.pop_back();
        pooled = true;
      }
    }
    for (int k = 0; k < kSideStreams && !pooled; ++k) {
      const cudaError_t e = cudaStreamCreateWithFlags(&x.s[k], cudaStreamNonBlocking);
      if (e != cudaSuccess) {
        for (int q = 0; q < k; ++q) cudaStreamDestroy(x.s[q]);
        return e;
      }
    }
    ts.set[dev] = x;
    ts.have[dev] = true;
  }
  for (int k = 0; k < kSideStreams; ++k) out[k] = ts.set[dev].s[k];
  return cudaSuccess;
}

cudaError_t fork_streams(cudaStream_t s, const cudaStream_t* side, int k) {
  cudaEvent_t ev;
  cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(ev, s);
  for (int i = 0; i < k && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(side[i], ev, 0);
  cudaEventDestroy(ev);  // released once the waits are resolved
  return e;
}

cudaError_t join_streams(cudaStream_t s, const cudaStream_t* side, int k) {
  cudaError_t first = cudaSuccess;
  for (int i = 0; i < k; ++i) {
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) {
      e = cudaEventRecord(ev, side[i]);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev, 0);
      cudaEventDestroy(ev);
    }
    if (first == cudaSuccess) first = e;
  }
  return first;
}

}  // namespace mt

extern "C" {

int mt_plan_merge(const mt_feature_spec* features, int F, double max_load, mt_feature_placement* placement,
                  mt_merge_group* groups, int* num_groups) {
  if (num_groups == nullptr) return MT_EINVAL;
  *num_groups = 0;
  if (features == nullptr || placement == nullptr || groups == nullptr || F < 1 || F > MT_MAX_FEATURES)
    return MT_EINVAL;
  if (!(max_load > 0.0 && max_load <= 1.0)) return MT_EINVAL;
  int G = 0;
  for (int f = 0; f < F; ++f) {
    const mt_feature_spec& x = features[f];
    const uint32_t vec = x.row_dtype == MT_F32 ? 4 : 8;
    if ((x.row_dtype != MT_F32 && x.row_dtype != MT_BF16) || x.dim < 4 || x.dim > MT_MAX_DIM || x.dim % vec != 0 ||
        x.capacity < 0)
      return MT_EINVAL;
    int g = -1;
    for (int q = 0; q < G; ++q)  // the first open group of the same row shape
      if (groups[q].dim == x.dim && groups[q].row_dtype == x.row_dtype && groups[q].num_features < 255) {
        g = q;
        break;
      }
    if (g < 0) {
      g = G++;
      std::memset(&groups[g], 0, sizeof(groups[g]));
      groups[g].dim = x.dim;
      groups[g].row_dtype = x.row_dtype;
    }
    placement[f].group = g;
    placement[f].table_id = (uint8_t)groups[g].num_features;
    groups[g].num_features += 1;
    groups[g].capacity += x.capacity;
  }
  for (int g = 0; g < G; ++g) {  // the smallest M = 2^n (n >= 1) with capacity <= max_load * M
    uint32_t n = 1;
    while (n <= 31 && (double)groups[g].capacity > max_load * (double)(1ull << n)) ++n;
    if (n > 31) return MT_EINVAL;
    groups[g].log2_slots = n;
  }
  *num_groups = G;
  return MT_OK;
}

size_t mt_lookup_grouped_workspace_bytes(int64_t n, int F) {
  if (n < 0 || n > 0x7FFFFFFF || F < 1 || F > MT_MAX_FEATURES) return 0;
  // the routed IDs, then one lookup workspace per group with IDs (at most min(F, n) of them).  Split into
  // groups, a batch needs at most one more tile, one more scratch-hash rounding and one more set of array
  // alignments per group: the workspace of a one-ID lookup.
  const long long groups = n < F ? n : F;
  return mt::align_up((size_t)(n > 0 ? n : 1) * 8, 256) + mt::align_up(mt::lookup_ws_layout(n).total, 256) +
         (size_t)groups * mt::align_up(mt::lookup_ws_layout(1).total, 256);
}

int mt_lookup_grouped(mt_table* const* tables, int G, const mt_feature_placement* placement, const int64_t* ids,
                      int64_t n, const int64_t* feat_offsets, int F, int insert_missing, void* const* out_rows,
                      const mt_lookup_result* results, int64_t* group_n, void* ws, size_t ws_bytes,
                      mt_stream stream) {
  if (tables == nullptr || placement == nullptr || results == nullptr || group_n == nullptr || G < 1) return MT_EINVAL;
  if (n < 0 || n > 0x7FFFFFFF || feat_offsets == nullptr || F < 1 || F > MT_MAX_FEATURES) return MT_EINVAL;
  if (n > 0 && (ids == nullptr || ((uintptr_t)ids % 8) != 0)) return MT_EINVAL;
  if (feat_offsets[0] != 0 || feat_offsets[F] != n) return MT_EINVAL;
  for (int f = 0; f < F; ++f) {
    if (feat_offsets[f + 1] < feat_offsets[f]) return MT_EINVAL;
    if (placement[f].group < 0 || placement[f].group >= G || placement[f].table_id == 0xFF) return MT_EINVAL;
  }
  for (int g = 0; g < G; ++g) {
    if (tables[g] == nullptr) return MT_EINVAL;
    for (int q = 0; q < g; ++q)  // distinct tables: the groups' lookups run side by side
      if (tables[q] == tables[g]) return MT_EINVAL;
  }
  if (ws == nullptr || ((uintptr_t)ws % 256) != 0) return MT_ENOSPACE;
  // each group's IDs, its slice of the routed IDs and its own lookup workspace (the groups run side by side)
  std::vector<long long> ng(G, 0), rbase(G, 0);
  std::vector<size_t> wso(G, 0), wsz(G, 0);
  for (int f = 0; f < F; ++f) ng[placement[f].group] += feat_offsets[f + 1] - feat_offsets[f];
  size_t off = mt::align_up((size_t)(n > 0 ? n : 1) * 8, 256);
  long long rb = 0;
  int active = 0;
  for (int g = 0; g < G; ++g) {
    rbase[g] = rb;
    rb += ng[g];
    if (ng[g] > 0) {
      wsz[g] = mt::lookup_ws_layout(ng[g]).total;
      wso[g] = off;
      off = mt::align_up(off + wsz[g], 256);
      ++active;
    }
  }
  if (ws_bytes < off) return MT_ENOSPACE;
  for (int g = 0; g < G; ++g) {
    const int st = mt::lookup_group_status(&results[g], out_rows ? out_rows[g] : nullptr);
    if (st != MT_OK) return st;
  }
  long long* routed = static_cast<long long*>(ws);
  mt::GroupStreams gs;
  if (gs.begin(reinterpret_cast<cudaStream_t>(stream), active) != cudaSuccess) return MT_ECUDA;
  int rc = MT_OK, slot = 0;
  for (int g = 0; g < G && rc == MT_OK; ++g) {
    const cudaStream_t s = ng[g] > 0 ? gs.stream(slot++) : gs.caller;
    // the group's features in batch order, their segments routed into its slice of the routed IDs
    std::vector<int64_t> offs(1, 0);
    std::vector<uint8_t> tids;
    mt::RouteSegs segs;
    std::memset(&segs, 0, sizeof(segs));
    long long* dst = routed + rbase[g];
    for (int f = 0; f < F; ++f) {
      if (placement[f].group != g) continue;
      const long long len = feat_offsets[f + 1] - feat_offsets[f];
      if (len > 0) {
        segs.src[segs.count] = feat_offsets[f];
        segs.dst[segs.count] = offs.back();
        segs.len[segs.count] = len;
        if (++segs.count == mt::kRouteSegs) {
          MT_LAUNCH("k_route", s);
          mt::k_route<<<dim3(64, mt::kRouteSegs), 256, 0, s>>>(reinterpret_cast<const long long*>(ids), dst, segs);
          segs.count = 0;
        }
      }
      offs.push_back(offs.back() + len);
      tids.push_back(placement[f].table_id);
    }
    if (segs.count > 0) {
      MT_LAUNCH("k_route", s);
      mt::k_route<<<dim3(64, segs.count), 256, 0, s>>>(reinterpret_cast<const long long*>(ids), dst, segs);
    }
    if (cudaGetLastError() != cudaSuccess) {
      rc = MT_ECUDA;
      break;
    }
    group_n[g] = ng[g];
    if (tids.empty()) {  // no feature of this batch goes to the group: an empty lookup
      offs.push_back(0);
      tids.push_back(0);
    }
    rc = mt_lookup(tables[g], reinterpret_cast<const int64_t*>(dst), ng[g], offs.data(), tids.data(),
                   (int)tids.size(), insert_missing, out_rows ? out_rows[g] : nullptr, &results[g],
                   ng[g] > 0 ? static_cast<char*>(ws) + wso[g] : nullptr, wsz[g], reinterpret_cast<mt_stream>(s));
  }
  // every group's work is ordered before the caller's later work, also after an error
  if (gs.end() != cudaSuccess && rc == MT_OK) rc = MT_ECUDA;
  return rc;
}

size_t mt_backward_grouped_workspace_bytes(mt_table* const* tables, int G, const int64_t* group_n) {
  if (tables == nullptr || group_n == nullptr || G < 1) return 0;
  size_t off = 0;
  for (int g = 0; g < G; ++g) {
    if (tables[g] == nullptr || group_n[g] < 0) return 0;
    off = mt::align_up(off + mt_backward_workspace_bytes(tables[g], group_n[g]), 256);
  }
  return off > 0 ? off : 256;
}

int mt_backward_adam_grouped(mt_table* const* tables, int G, const mt_lookup_result* results, const int64_t* group_n,
                             const void* const* grads, int grad_dtype, const mt_adam* hp, float* const* gsum_out,
                             void* ws, size_t ws_bytes, mt_stream stream) {
  if (tables == nullptr || results == nullptr || group_n == nullptr || grads == nullptr || G < 1) return MT_EINVAL;
  for (int g = 0; g < G; ++g)
    if (tables[g] == nullptr || group_n[g] < 0) return MT_EINVAL;
  if (ws == nullptr || ((uintptr_t)ws % 256) != 0 || ws_bytes < mt_backward_grouped_workspace_bytes(tables, G, group_n))
    return MT_ENOSPACE;
  for (int g = 0; g < G; ++g) {
    for (int q = 0; q < g; ++q)  // the tables must be distinct: each call advances its table's step
      if (tables[q] == tables[g]) return MT_EINVAL;
    const int st = mt::backward_group_status(tables[g], &results[g], group_n[g], grads[g], grad_dtype, hp,
                                             gsum_out ? gsum_out[g] : nullptr);
    if (st != MT_OK) return st;
  }
  int active = 0;
  for (int g = 0; g < G; ++g) active += group_n[g] > 0;
  mt::GroupStreams gs;
  if (gs.begin(reinterpret_cast<cudaStream_t>(stream), active) != cudaSuccess) return MT_ECUDA;
  int rc = MT_OK, slot = 0;
  size_t off = 0;
  for (int g = 0; g < G && rc == MT_OK; ++g) {
    const size_t need = mt_backward_workspace_bytes(tables[g], group_n[g]);
    const cudaStream_t s = group_n[g] > 0 ? gs.stream(slot++) : gs.caller;
    rc = mt_backward_adam(tables[g], &results[g], group_n[g], grads[g], grad_dtype, hp,
                          gsum_out ? gsum_out[g] : nullptr, static_cast<char*>(ws) + off, need,
                          reinterpret_cast<mt_stream>(s));
    off = mt::align_up(off + need, 256);
  }
  if (gs.end() != cudaSuccess && rc == MT_OK) rc = MT_ECUDA;
  return rc;
}

}  // extern "C"
