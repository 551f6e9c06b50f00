// lizard_trace.cu -- optional per-kernel device timing with CUDA events.
//
// When tracing is enabled on a host thread, every kernel this library enqueues from
// that thread is bracketed by two events recorded on the launch stream.  Reading the
// log synchronises on the events and returns (name, milliseconds) pairs.  Events are
// pooled and reused; nothing is recorded while tracing is off.
#include <string.h>

#include <vector>

#include "lizard_internal.h"

namespace lz {
namespace {

struct Rec {
  const char* name;
  cudaEvent_t start, stop;
};

struct TraceState {
  bool on = false;
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  int open = -1;  // index of the record awaiting its stop event
};

thread_local TraceState g_trace;

cudaEvent_t take_event() {
  if (!g_trace.pool.empty()) {
    cudaEvent_t e = g_trace.pool.back();
    g_trace.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

void trace_begin(const char* name, cudaStream_t s) {
  if (!g_trace.on) return;
  Rec r{name, take_event(), take_event()};
  if (!r.start || !r.stop) return;
  cudaEventRecord(r.start, s);
  g_trace.recs.push_back(r);
  g_trace.open = (int)g_trace.recs.size() - 1;
}

void trace_end(cudaStream_t s) {
  if (!g_trace.on || g_trace.open < 0) return;
  cudaEventRecord(g_trace.recs[g_trace.open].stop, s);
  g_trace.open = -1;
}

}  // namespace lz

extern "C" {

lizard_status lizard_trace_enable(int32_t enable) {
  lz::g_trace.on = enable != 0;
  return LIZARD_OK;
}

int32_t lizard_trace_read(char* names, int32_t name_len, float* ms, int32_t max_records) {
  auto& t = lz::g_trace;
  int32_t n = 0;
  for (auto& r : t.recs) {
    if (n < max_records && names && ms && name_len > 0) {
      float v = -1.f;
      if (cudaEventSynchronize(r.stop) == cudaSuccess) cudaEventElapsedTime(&v, r.start, r.stop);
      strncpy(names + (size_t)n * name_len, r.name, (size_t)name_len - 1);
      names[(size_t)n * name_len + name_len - 1] = '\0';
      ms[n] = v;
      ++n;
    }
    t.pool.push_back(r.start);
    t.pool.push_back(r.stop);
  }
  t.recs.clear();
  t.open = -1;
  return n;
}

}  // extern "C"
