// mt_lookup_static: the lookup for callers that cannot allocate device
// memory when they call it.
//
// Some callers have no way to hand us a workspace: a plugin or operator
// interface that passes only input and output buffers, or a serving process
// that fixed its memory budget at start-up and may not call cudaMalloc (or a
// caching allocator) afterwards.  For them this entry point takes its scratch
// from a file-scope device array, sized for batches of up to
// MT_LOOKUP_STATIC_MAX_IDS IDs.  Every GPU that loads the library holds the
// array until the process exits.
//
// In host code the array's name is only a host-side stand-in, not a device
// address, so its device address is looked up with cudaGetSymbolAddress once
// per device (on the first call made with that device current) and cached.
// That first call should therefore come before any stream capture.
//
// All calls share the one array and it keeps the previous call's contents;
// the lookup clears what must start empty (its scratch hash) itself.  Calls
// whose work overlaps on the GPU (other streams, other host threads) race on
// the array and must not be issued.
#include <mutex>

#include "mt_kernels.cuh"

namespace {

constexpr size_t kStaticScratchBytes = 6u << 20;  // 6 MiB: the lookup workspace for MT_LOOKUP_STATIC_MAX_IDS IDs

__device__ __align__(256) unsigned char g_lookup_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[mt::kMaxDevices] = {};

// Device address of the scratch array on the current device, or nullptr.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= mt::kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_lookup_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int mt_lookup_static(mt_table* t, const int64_t* ids, int64_t n, const int64_t* feat_offsets,
                                const uint8_t* table_ids, int F, int insert_missing, void* out_rows,
                                const mt_lookup_result* res, mt_stream stream) {
  if (n < 0) return MT_EINVAL;
  if (n > MT_LOOKUP_STATIC_MAX_IDS) return MT_ETOOBIG;
  const size_t need = mt::lookup_ws_layout(n).total;
  if (need > kStaticScratchBytes) return MT_ETOOBIG;
  void* ws = scratch_on_current_device();
  if (ws == nullptr) return MT_ECUDA;
  return mt_lookup(t, ids, n, feat_offsets, table_ids, F, insert_missing, out_rows, res, ws, kStaticScratchBytes,
                   stream);
}
