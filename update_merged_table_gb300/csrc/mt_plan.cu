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
#include <vector>

#include "mt_kernels.cuh"

namespace mt {
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

size_t mt_lookup_grouped_workspace_bytes(int64_t n) {
  if (n < 0 || n > 0x7FFFFFFF) return 0;
  return mt::align_up((size_t)(n > 0 ? n : 1) * 8, 256) + mt::lookup_ws_layout(n).total;
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
  for (int g = 0; g < G; ++g)
    if (tables[g] == nullptr) return MT_EINVAL;
  if (ws == nullptr || ws_bytes < mt_lookup_grouped_workspace_bytes(n) || ((uintptr_t)ws % 256) != 0)
    return MT_ENOSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  long long* routed = static_cast<long long*>(ws);
  void* lws = static_cast<char*>(ws) + mt::align_up((size_t)(n > 0 ? n : 1) * 8, 256);
  const size_t lws_bytes = ws_bytes - mt::align_up((size_t)(n > 0 ? n : 1) * 8, 256);
  for (int g = 0; g < G; ++g) {
    // the group's features in batch order, their segments routed into one contiguous batch
    std::vector<int64_t> offs(1, 0);
    std::vector<uint8_t> tids;
    mt::RouteSegs segs;
    std::memset(&segs, 0, sizeof(segs));
    for (int f = 0; f < F; ++f) {
      if (placement[f].group != g) continue;
      const long long len = feat_offsets[f + 1] - feat_offsets[f];
      if (len > 0) {
        segs.src[segs.count] = feat_offsets[f];
        segs.dst[segs.count] = offs.back();
        segs.len[segs.count] = len;
        if (++segs.count == mt::kRouteSegs) {
          MT_LAUNCH("k_route", s);
          mt::k_route<<<dim3(64, mt::kRouteSegs), 256, 0, s>>>(reinterpret_cast<const long long*>(ids), routed, segs);
          segs.count = 0;
        }
      }
      offs.push_back(offs.back() + len);
      tids.push_back(placement[f].table_id);
    }
    if (segs.count > 0) {
      MT_LAUNCH("k_route", s);
      mt::k_route<<<dim3(64, segs.count), 256, 0, s>>>(reinterpret_cast<const long long*>(ids), routed, segs);
    }
    if (cudaGetLastError() != cudaSuccess) return MT_ECUDA;
    const int64_t ng = offs.back();
    group_n[g] = ng;
    if (tids.empty()) {  // no feature of this batch goes to the group: an empty lookup
      offs.push_back(0);
      tids.push_back(0);
    }
    const int rc = mt_lookup(tables[g], reinterpret_cast<const int64_t*>(routed), ng, offs.data(), tids.data(),
                             (int)tids.size(), insert_missing, out_rows ? out_rows[g] : nullptr, &results[g], lws,
                             lws_bytes, stream);
    if (rc != MT_OK) return rc;
  }
  return MT_OK;
}

}  // extern "C"
