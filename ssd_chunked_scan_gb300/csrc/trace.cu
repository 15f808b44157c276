// Launch accounting and optional per-kernel timing of libssd.
//
// Every kernel launch made by the library goes through a LaunchTrace scope.
// The scope always bumps a process-wide launch counter; when tracing is
// enabled (ssd_trace_enable) it also brackets the launch with two CUDA events
// on the launching stream, so per-kernel device time can be read back with
// ssd_trace_get after the work has finished.
#include <mutex>
#include <string>
#include <vector>
#include <atomic>

#include "../../include/ssd.h"
#include "common.cuh"

namespace ssd {
namespace {

struct Rec {
  const char *name;
  cudaEvent_t a, b;
};

std::atomic<long long> g_launches{0};
std::atomic<int> g_enabled{0};
thread_local bool t_quiet = false;
std::mutex g_mu;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_free;

cudaEvent_t get_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

struct Agg {
  std::string name;
  long long launches = 0;
  double ms = 0.0;
};
std::vector<Agg> g_agg;

}  // namespace

LaunchTrace::Quiet::Quiet() : prev_(t_quiet) { t_quiet = true; }
LaunchTrace::Quiet::~Quiet() { t_quiet = prev_; }

LaunchTrace::LaunchTrace(const char *name, cudaStream_t s) : name_(name), s_(s), a_(nullptr) {
  if (!t_quiet && g_enabled.load(std::memory_order_relaxed)) {
    std::lock_guard<std::mutex> lk(g_mu);
    a_ = get_event();
    if (a_) cudaEventRecord(static_cast<cudaEvent_t>(a_), s_);
  }
}

LaunchTrace::~LaunchTrace() {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (a_) {
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t b = get_event();
    if (b) {
      cudaEventRecord(b, s_);
      g_recs.push_back(Rec{name_, static_cast<cudaEvent_t>(a_), b});
    } else {
      g_free.push_back(static_cast<cudaEvent_t>(a_));
    }
  }
}

}  // namespace ssd

extern "C" {

SSD_API long long ssd_launch_count(void) { return ssd::g_launches.load(); }

SSD_API int ssd_trace_enable(int on) {
  ssd::g_enabled.store(on ? 1 : 0);
  return SSD_OK;
}

// Waits for every traced launch, folds them into per-kernel totals and
// returns the number of distinct kernel names recorded since the last reset.
SSD_API int ssd_trace_collect(void) {
  std::lock_guard<std::mutex> lk(ssd::g_mu);
  for (auto &r : ssd::g_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess) return -SSD_ERR_CUDA;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -SSD_ERR_CUDA;
    bool found = false;
    for (auto &a : ssd::g_agg)
      if (a.name == r.name) { a.launches++; a.ms += ms; found = true; break; }
    if (!found) ssd::g_agg.push_back(ssd::Agg{r.name, 1, ms});
    ssd::g_free.push_back(r.a);
    ssd::g_free.push_back(r.b);
  }
  ssd::g_recs.clear();
  return (int)ssd::g_agg.size();
}

SSD_API int ssd_trace_get(int i, char *name, int name_len, long long *launches, double *total_ms) {
  std::lock_guard<std::mutex> lk(ssd::g_mu);
  if (i < 0 || i >= (int)ssd::g_agg.size() || !name || name_len < 1) return SSD_ERR_ARG;
  const auto &a = ssd::g_agg[i];
  int n = 0;
  for (; n + 1 < name_len && n < (int)a.name.size(); ++n) name[n] = a.name[n];
  name[n] = 0;
  if (launches) *launches = a.launches;
  if (total_ms) *total_ms = a.ms;
  return SSD_OK;
}

SSD_API int ssd_trace_reset(void) {
  std::lock_guard<std::mutex> lk(ssd::g_mu);
  for (auto &r : ssd::g_recs) {
    ssd::g_free.push_back(r.a);
    ssd::g_free.push_back(r.b);
  }
  ssd::g_recs.clear();
  ssd::g_agg.clear();
  return SSD_OK;
}

}  // extern "C"
