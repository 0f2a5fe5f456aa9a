// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gnnagg.h"

namespace gnn {

// Records a message for gnn_last_error() and returns `code`.
gnn_status fail(gnn_status code, const char* fmt, ...);

// Device-side flag word raised by kernels (bit 0: bad data, bit 1: timeout).
unsigned* device_flags();

inline cudaStream_t as_stream(gnn_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

#define GNN_CUDA(expr)                                                              \
  do {                                                                              \
    cudaError_t e_ = (expr);                                                        \
    if (e_ != cudaSuccess)                                                          \
      return ::gnn::fail(GNN_ERR_CUDA, "%s failed: %s (%s:%d)", #expr,              \
                         cudaGetErrorString(e_), __FILE__, __LINE__);               \
  } while (0)

// Counts library kernel launches (reported by gnn_kernel_launches).
void count_launch();

#define GNN_CHECK_LAUNCH()        \
  do {                            \
    ::gnn::count_launch();        \
    GNN_CUDA(cudaGetLastError()); \
  } while (0)

#define GNN_REQUIRE(cond, ...)                                                      \
  do {                                                                              \
    if (!(cond)) return ::gnn::fail(GNN_ERR_INVALID_ARG, __VA_ARGS__);              \
  } while (0)

// Carves 256-byte aligned pieces out of a caller workspace.  With base NULL
// it only measures.
struct Arena {
  char* base;
  size_t cap;
  size_t used = 0;
  Arena(void* b, size_t c) : base(static_cast<char*>(b)), cap(c) {}
  template <class T>
  T* take(size_t count) {
    size_t bytes = (count * sizeof(T) + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += bytes;
    return p;
  }
  void* take_bytes(size_t bytes) { return take<char>(bytes); }
  bool ok() const { return base == nullptr || used <= cap; }
};

inline bool is_valid_bits(int b) { return b == 1 || b == 2 || b == 4 || b == 8 || b == 32; }

constexpr int kMaxF = 1024;

}  // namespace gnn
