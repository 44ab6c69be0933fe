// Opt-in kernel timing for benchmarks.  While enabled on a host thread, the
// launchers record a pair of CUDA events on the caller's stream around their
// main kernel; kv_int4_timing_collect() waits for the recorded pairs and sums
// their durations.  Event objects are created on first use and reused; no
// device memory is allocated.

#include <cuda_runtime.h>

#include "../../include/kvint4.h"
#include "internal.h"

namespace kvint4 {

namespace {
constexpr int kMaxPairs = 4096;

struct Pair {
  cudaEvent_t a = nullptr, b = nullptr;
};

struct ThreadTiming {
  bool enabled = false;
  Pair pairs[kTimedKinds][kMaxPairs];
  int used[kTimedKinds] = {};
  int dropped[kTimedKinds] = {};
  int open[kTimedKinds] = {};  // 1 while a begin has no matching end
};

thread_local ThreadTiming tt;

bool ensure(Pair& p) {
  if (!p.a && cudaEventCreate(&p.a) != cudaSuccess) return false;
  if (!p.b && cudaEventCreate(&p.b) != cudaSuccess) return false;
  return true;
}
}  // namespace

void timing_begin(TimedKind kind, cudaStream_t stream) {
  if (!tt.enabled) return;
  const int k = (int)kind;
  if (tt.used[k] >= kMaxPairs || !ensure(tt.pairs[k][tt.used[k]])) {
    tt.dropped[k]++;
    return;
  }
  if (cudaEventRecord(tt.pairs[k][tt.used[k]].a, stream) != cudaSuccess) {
    tt.dropped[k]++;
    return;
  }
  tt.open[k] = 1;
}

void timing_end(TimedKind kind, cudaStream_t stream) {
  const int k = (int)kind;
  if (!tt.enabled || !tt.open[k]) return;
  tt.open[k] = 0;
  if (cudaEventRecord(tt.pairs[k][tt.used[k]].b, stream) != cudaSuccess) {
    tt.dropped[k]++;
    return;
  }
  tt.used[k]++;
}

}  // namespace kvint4

using namespace kvint4;

extern "C" {

int kv_int4_timing_enable(int enable) {
  tt.enabled = enable != 0;
  return KV_INT4_OK;
}

int kv_int4_timing_collect(double* ms_out, int* launches_out, int* dropped_out) {
  int rc = KV_INT4_OK;
  for (int k = 0; k < kTimedKinds; k++) {
    double total = 0.0;
    for (int i = 0; i < tt.used[k]; i++) {
      float ms = 0.f;
      if (cudaEventSynchronize(tt.pairs[k][i].b) != cudaSuccess ||
          cudaEventElapsedTime(&ms, tt.pairs[k][i].a, tt.pairs[k][i].b) != cudaSuccess) {
        rc = KV_INT4_ERR_CUDA;
        continue;
      }
      total += ms;
    }
    if (ms_out) ms_out[k] = total;
    if (launches_out) launches_out[k] = tt.used[k];
    if (dropped_out) dropped_out[k] = tt.dropped[k];
    tt.used[k] = 0;
    tt.dropped[k] = 0;
    tt.open[k] = 0;
  }
  return rc;
}

}  // extern "C"
