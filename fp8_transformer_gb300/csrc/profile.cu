// Optional per-launch timing of the library's kernels with CUDA events on the launching
// stream (te_profile_begin / te_profile_end).  Off unless a caller turns it on.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "kernels.h"
#include "te_gb300.h"

namespace te {
namespace {

struct Record {
  int kind;
  cudaEvent_t start, stop;
};

struct Profiler {
  std::mutex mu;
  bool on = false;
  int max_records = 0;
  std::vector<Record> records;
  int launches[TE_KERNEL_KINDS] = {};
};

Profiler& prof() {
  static Profiler p;
  return p;
}

}  // namespace

ProfileScope::ProfileScope(int kind, cudaStream_t stream) : kind_(kind), stream_(stream) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  if (!p.on) return;
  p.launches[kind]++;
  if (int(p.records.size()) >= p.max_records) return;
  Record r{kind, nullptr, nullptr};
  if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.stop) != cudaSuccess) return;
  cudaEventRecord(r.start, stream);
  p.records.push_back(r);
  slot_ = int(p.records.size()) - 1;
}

ProfileScope::~ProfileScope() {
  if (slot_ < 0) return;
  Profiler& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  if (slot_ < int(p.records.size())) cudaEventRecord(p.records[slot_].stop, stream_);
}

}  // namespace te

using namespace te;

extern "C" {

te_status te_profile_begin(int32_t max_records) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  for (Record& r : p.records) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  p.records.clear();
  for (int& l : p.launches) l = 0;
  p.max_records = max_records > 0 ? max_records : 0;
  p.records.reserve(size_t(p.max_records));
  p.on = true;
  return TE_OK;
}

te_status te_profile_end(float* total_ms, int32_t* launches) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  p.on = false;
  te_status st = TE_OK;
  float sum[TE_KERNEL_KINDS] = {};
  for (Record& r : p.records) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      st = TE_ERR_CUDA;
    sum[r.kind] += ms;
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  p.records.clear();
  for (int k = 0; k < TE_KERNEL_KINDS; ++k) {
    if (total_ms) total_ms[k] = sum[k];
    if (launches) launches[k] = p.launches[k];
  }
  return st;
}

}  // extern "C"
