// Kernel tracing for rpa_forward (rpa_trace_begin / rpa_trace_end): CUDA
// events recorded around each launch on the caller's stream, or event-record
// nodes when the stream is being captured into a CUDA graph.
#include <cuda_runtime.h>

#include <vector>

#include "rpa.h"
#include "rpa_internal.h"

namespace rpa {
namespace {

struct Mark {
  int kernel;        // -1: start of an rpa_forward call on `stream`
  cudaEvent_t event;
  void* stream;
};

bool g_on = false;
int g_capacity = 0;
int g_launches = 0;
std::vector<Mark> g_marks;
std::vector<cudaEvent_t> g_pool;  // events reused across trace sessions

cudaEvent_t take_event() {
  size_t used = g_marks.size();
  if (used < g_pool.size()) return g_pool[used];
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  g_pool.push_back(e);
  return e;
}

void record(int kernel, void* stream) {
  cudaEvent_t e = take_event();
  if (e == nullptr) return;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Under stream capture the mark becomes an event-record node of the graph
  // (recorded on every replay); otherwise a plain record.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return;
  const unsigned flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u;
  if (cudaEventRecordWithFlags(e, s, flags) != cudaSuccess) return;
  g_marks.push_back({kernel, e, stream});
}

}  // namespace

void trace_start(void* stream) {
  if (!g_on || g_launches >= g_capacity) return;
  record(-1, stream);
}

void trace_mark(int kernel, void* stream) {
  if (!g_on || g_launches >= g_capacity) return;
  ++g_launches;
  record(kernel, stream);
}

}  // namespace rpa

extern "C" {

rpa_status_t rpa_trace_begin(int32_t capacity) {
  if (capacity < 1 || capacity > 65536) return RPA_ERR_INVALID_ARG;
  rpa::g_on = true;
  rpa::g_capacity = capacity;
  rpa::g_launches = 0;
  rpa::g_marks.clear();
  return RPA_OK;
}

rpa_status_t rpa_trace_end(rpa_trace_record* records, int32_t* count) {
  if (count == nullptr || (records == nullptr && *count > 0)) return RPA_ERR_INVALID_ARG;
  rpa::g_on = false;
  int32_t n = 0;
  rpa_status_t st = RPA_OK;
  for (size_t i = 1; i < rpa::g_marks.size(); ++i) {
    const rpa::Mark& m = rpa::g_marks[i];
    if (m.kernel < 0) continue;
    if (n >= *count) break;
    // The previous mark on the same stream: a mixed batch's prefill runs on
    // a second stream beside the decode.
    size_t j = i - 1;
    while (j > 0 && rpa::g_marks[j].stream != m.stream) --j;
    if (rpa::g_marks[j].stream != m.stream) continue;
    float ms = 0.f;
    if (cudaEventSynchronize(m.event) != cudaSuccess ||
        cudaEventElapsedTime(&ms, rpa::g_marks[j].event, m.event) != cudaSuccess) {
      st = RPA_ERR_CUDA;
      break;
    }
    records[n].kernel = m.kernel;
    records[n].ms = ms;
    ++n;
  }
  rpa::g_marks.clear();
  *count = n;
  return st;
}

}  // extern "C"
