// Launch instrumentation: a launch counter and optional CUDA-event brackets around the launches
// of one kernel class (used by the benchmark to time its dominant kernel on the launching stream,
// including inside captured CUDA graphs, where each record becomes an external event node).
#include <atomic>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "lora_kernels.h"

namespace lora {

namespace {
std::atomic<unsigned long long> g_launches{0};
std::mutex g_mu;
int g_kind = 0;
std::vector<cudaEvent_t> g_starts, g_stops;
size_t g_used = 0;

// Under stream capture a plain record only orders streams inside the capture; the external flag
// makes it an event-record node that fires (and timestamps) on every replay.
void record(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
  else
    cudaEventRecord(e, st);
}
}  // namespace

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("LORA_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

void prof_begin(int kind, cudaStream_t st) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (kind == 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_kind == kind && g_used < g_starts.size()) record(g_starts[g_used], st);
}

void prof_end(int kind, cudaStream_t st) {
  if (kind == 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_kind == kind && g_used < g_stops.size()) {
    record(g_stops[g_used], st);
    ++g_used;
  }
}

}  // namespace lora

extern "C" {

int lora_profile_arm(int32_t kernel_class, void* const* start_events, void* const* stop_events,
                     int32_t n) {
  if (kernel_class < 0 || n < 0 || (n > 0 && (!start_events || !stop_events)))
    return LORA_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (!start_events[i] || !stop_events[i]) return LORA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(lora::g_mu);
  lora::g_kind = kernel_class;
  lora::g_starts.assign(n, nullptr);
  lora::g_stops.assign(n, nullptr);
  for (int i = 0; i < n; ++i) {
    lora::g_starts[i] = (cudaEvent_t)start_events[i];
    lora::g_stops[i] = (cudaEvent_t)stop_events[i];
  }
  lora::g_used = 0;
  return LORA_OK;
}

int32_t lora_profile_used(void) {
  std::lock_guard<std::mutex> lk(lora::g_mu);
  return (int32_t)lora::g_used;
}

uint64_t lora_launch_counter(void) { return lora::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
