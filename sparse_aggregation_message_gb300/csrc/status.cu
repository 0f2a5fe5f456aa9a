// Error reporting shared by every entry point.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include <atomic>

#include "internal.h"

namespace gnn {

static thread_local char g_last_error[512] = "";

gnn_status fail(gnn_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

static std::atomic<unsigned long long> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Bit 0: a kernel found bad data; bit 1: a bounded wait gave up.
__device__ unsigned g_device_flags = 0;

unsigned* device_flags() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_flags) != cudaSuccess) return nullptr;
  return static_cast<unsigned*>(p);
}

}  // namespace gnn

extern "C" const char* gnn_last_error(void) { return gnn::g_last_error; }

extern "C" int gnn_version(void) { return 1 * 10000 + 0 * 100 + 0; }

extern "C" unsigned long long gnn_kernel_launches(void) {
  return gnn::g_launches.load(std::memory_order_relaxed);
}

extern "C" gnn_status gnn_sync_check(gnn_stream_t stream) {
  // every stream: a flag may come from a kernel on a second stream (the
  // asynchronous layers' aux stream)
  GNN_CUDA(cudaStreamSynchronize(gnn::as_stream(stream)));
  GNN_CUDA(cudaDeviceSynchronize());
  unsigned flags = 0;
  GNN_CUDA(cudaMemcpyFromSymbol(&flags, gnn::g_device_flags, sizeof(flags)));
  if (flags) {
    const unsigned zero = 0;
    GNN_CUDA(cudaMemcpyToSymbol(gnn::g_device_flags, &zero, sizeof(zero)));
    if (flags & 2u) return gnn::fail(GNN_ERR_TIMEOUT, "a bounded device wait gave up");
    return gnn::fail(GNN_ERR_DEVICE_CHECK, "a kernel flagged invalid data (flags=0x%x)", flags);
  }
  return GNN_OK;
}
