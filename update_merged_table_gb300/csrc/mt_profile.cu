// Per-kernel timing with CUDA events and a process-wide launch counter.
//
// Every kernel launch of the library is wrapped in a LaunchScope.  The scope
// always counts the launch; when profiling is on it also records a CUDA
// event before and after the kernel on the launching stream.  The report
// synchronises those events and accumulates the elapsed time per kernel name.
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "mt_kernels.cuh"

namespace mt {

namespace {

struct Pending {
  const char* name;
  cudaEvent_t start, stop;
};

struct Totals {
  const char* name;
  long long launches;
  double ms;
};

std::mutex g_mu;
bool g_enabled = false;
long long g_launches = 0;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free_events;
std::vector<Totals> g_totals;

cudaEvent_t take_event() {
  if (!g_free_events.empty()) {
    cudaEvent_t e = g_free_events.back();
    g_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

Totals& totals_for(const char* name) {
  for (auto& t : g_totals)
    if (std::strcmp(t.name, name) == 0) return t;
  g_totals.push_back(Totals{name, 0, 0.0});
  return g_totals.back();
}

}  // namespace

LaunchScope::LaunchScope(const char* name, cudaStream_t s) : name_(name), stream_(s), start_(nullptr) {
  std::lock_guard<std::mutex> lk(g_mu);
  ++g_launches;
  if (!g_enabled) return;
  start_ = take_event();
  if (start_ != nullptr) cudaEventRecord(start_, s);
}

LaunchScope::~LaunchScope() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (start_ == nullptr) return;
  cudaEvent_t stop = take_event();
  if (stop == nullptr) {
    g_free_events.push_back(start_);
    return;
  }
  cudaEventRecord(stop, stream_);
  g_pending.push_back(Pending{name_, start_, stop});
}

}  // namespace mt

extern "C" {

int mt_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(mt::g_mu);
  mt::g_enabled = on != 0;
  return MT_OK;
}

int mt_profile_report(mt_kernel_time* out, int capacity, int* count, int reset) {
  if (count == nullptr || capacity < 0 || (capacity > 0 && out == nullptr)) return MT_EINVAL;
  std::lock_guard<std::mutex> lk(mt::g_mu);
  int rc = MT_OK;
  for (auto& p : mt::g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.stop) != cudaSuccess || cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess)
      rc = MT_ECUDA;
    mt::Totals& t = mt::totals_for(p.name);
    t.launches += 1;
    t.ms += ms;
    mt::g_free_events.push_back(p.start);
    mt::g_free_events.push_back(p.stop);
  }
  mt::g_pending.clear();
  const int n = (int)mt::g_totals.size();
  *count = n;
  for (int i = 0; i < n && i < capacity; ++i) {
    std::memset(&out[i], 0, sizeof(out[i]));
    std::strncpy(out[i].name, mt::g_totals[i].name, sizeof(out[i].name) - 1);
    out[i].launches = mt::g_totals[i].launches;
    out[i].total_ms = mt::g_totals[i].ms;
  }
  if (reset) mt::g_totals.clear();
  return rc;
}

int64_t mt_kernel_launches(void) {
  std::lock_guard<std::mutex> lk(mt::g_mu);
  return mt::g_launches;
}

}  // extern "C"
