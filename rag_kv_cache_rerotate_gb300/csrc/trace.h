// Kernel timing trace hooks used around every kernel launch of the library.
#pragma once

#include <cuda_runtime.h>

#include "fusekv.h"

namespace fusekv {

// Records the start event of one launch on stream s; -1 when no trace is open.
int trace_open(cudaStream_t s);
// Records the stop event of the launch opened as `slot` and names it.
void trace_close(int slot, const char* name, cudaStream_t s);

// Runs one launcher between a trace_open / trace_close pair.
template <typename F>
cudaError_t traced(const char* name, cudaStream_t s, F&& launch) {
  const int slot = trace_open(s);
  const cudaError_t e = launch();
  trace_close(slot, name, s);
  return e;
}

}  // namespace fusekv
