// Kernel timing trace: a pair of CUDA events around every kernel launch of
// the library while a trace is open.  Host-side state only.
#include <mutex>
#include <vector>

#include "trace.h"

namespace fusekv {

namespace {

struct Record {
  const char* name;
  cudaEvent_t start;
  cudaEvent_t stop;
};

std::mutex g_mu;
bool g_on = false;
std::vector<cudaEvent_t> g_pool;   // 2 * capacity events
std::vector<Record> g_records;
size_t g_capacity = 0;

}  // namespace

int trace_open(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_records.size() >= g_capacity) return -1;
  const size_t i = g_records.size();
  Record r{nullptr, g_pool[2 * i], g_pool[2 * i + 1]};
  if (cudaEventRecord(r.start, s) != cudaSuccess) return -1;
  g_records.push_back(r);
  return (int)i;
}

void trace_close(int slot, const char* name, cudaStream_t s) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (slot >= (int)g_records.size()) return;
  g_records[slot].name = name;
  cudaEventRecord(g_records[slot].stop, s);
}

}  // namespace fusekv

using namespace fusekv;

extern "C" {

fuse_status_t fuse_trace_begin(int32_t max_records) {
  if (max_records <= 0) return FUSE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  for (cudaEvent_t e : g_pool) cudaEventDestroy(e);
  g_pool.clear();
  g_records.clear();
  g_pool.resize(2 * (size_t)max_records);
  for (auto& e : g_pool) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      g_pool.clear();
      g_on = false;
      return FUSE_ERR_CUDA;
    }
  }
  g_capacity = (size_t)max_records;
  g_on = true;
  return FUSE_OK;
}

fuse_status_t fuse_trace_end(fuse_trace_entry_t* out, int32_t max_out, int32_t* n_out) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = false;
  fuse_status_t st = FUSE_OK;
  int32_t n = 0;
  for (const Record& r : g_records) {
    if (cudaEventSynchronize(r.stop) != cudaSuccess) {
      st = FUSE_ERR_CUDA;
      break;
    }
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
      st = FUSE_ERR_CUDA;
      break;
    }
    if (out && n < max_out) {
      out[n].kernel = r.name ? r.name : "?";
      out[n].ms = ms;
    }
    ++n;
  }
  if (n_out) *n_out = out ? (n < max_out ? n : max_out) : n;
  for (cudaEvent_t e : g_pool) cudaEventDestroy(e);
  g_pool.clear();
  g_records.clear();
  g_capacity = 0;
  return st;
}

}  // extern "C"
