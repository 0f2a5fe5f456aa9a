// Setup calls (not on the per-layer hot path): CSR construction with GCN
// normalisation (SYLVIE guide, section 2) and the boundary index with per-node
// widths (sections 3, 7 and 9).  Sorting, deduplication and scans use CUB's
// device primitives; everything else is plain kernels.  Results are canonical
// (sorted), so they do not depend on the order atomics hand out positions.
#include <cub/cub.cuh>
#include <cuda_runtime.h>
#include <math.h>

#include "device.cuh"
#include "internal.h"

namespace gnn {

static int bits_for(uint64_t x) {  // bits needed to hold values < x (>= 1)
  int b = 1;
  while (b < 63 && (uint64_t(1) << b) < x) ++b;
  return b;
}

__device__ __forceinline__ int64_t part_of(int64_t x, int64_t n, int P) {
  return ((x + 1) * (int64_t)P - 1) / n;
}

template <class T>
__device__ __forceinline__ int64_t lower_bound_dev(const T* a, int64_t len, T key) {
  int64_t lo = 0, hi = len;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

template <class T>
__device__ __forceinline__ int64_t upper_bound_dev(const T* a, int64_t len, T key) {
  int64_t lo = 0, hi = len;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (a[mid] <= key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ int64_t row_of(const int64_t* rowptr, int n, int64_t e) {
  return upper_bound_dev(rowptr, (int64_t)n + 1, e) - 1;
}

#define GRID1(count) (unsigned)(((count) + 255) / 256), 256

// ------------------------------------------------------------------ CSR build
__global__ void emit_edge_keys(int64_t m, const int32_t* __restrict__ src,
                               const int32_t* __restrict__ dst, int n, int shift, bool sym,
                               bool drop_loops, uint64_t* __restrict__ keys,
                               unsigned long long* __restrict__ count, unsigned* flags) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= m) return;
  const int32_t u = src[i], v = dst[i];
  if (u < 0 || u >= n || v < 0 || v >= n) {
    atomicOr(flags, 1u);
    return;
  }
  if (drop_loops && u == v) return;
  const unsigned long long at = atomicAdd(count, sym ? 2ull : 1ull);
  keys[at] = ((uint64_t)v << shift) | (uint64_t)u;
  if (sym) keys[at + 1] = ((uint64_t)u << shift) | (uint64_t)v;
}

__global__ void emit_loop_keys(int n, int shift, uint64_t* __restrict__ keys,
                               const unsigned long long* __restrict__ count) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  keys[*count + i] = ((uint64_t)i << shift) | (uint64_t)i;
}

__global__ void csr_rowptr_kernel(int n, const uint64_t* __restrict__ keys, int64_t nnz,
                                  int shift, int64_t* __restrict__ rowptr) {
  const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v > n) return;
  rowptr[v] = lower_bound_dev(keys, nnz, (uint64_t)v << shift);
}

// GCN weight 1/sqrt(d_v d_u) or mean weight 1/d_v, in fp64 rounded to fp32;
// val_t (optional) receives the weight of the transposed entry (u, v).
__global__ void csr_fill_kernel(const uint64_t* __restrict__ keys, int64_t nnz, int shift,
                                const int64_t* __restrict__ rowptr, int mean,
                                int32_t* __restrict__ col, float* __restrict__ val,
                                float* __restrict__ val_t) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= nnz) return;
  const uint64_t k = keys[e];
  const int64_t v = (int64_t)(k >> shift);
  const int64_t u = (int64_t)(k & ((uint64_t(1) << shift) - 1));
  col[e] = (int32_t)u;
  const double dv = (double)(rowptr[v + 1] - rowptr[v]);
  const double du = (double)(rowptr[u + 1] - rowptr[u]);
  if (mean) {
    val[e] = (float)(1.0 / dv);
    if (val_t) val_t[e] = (float)(1.0 / du);
  } else {
    val[e] = (float)(1.0 / sqrt(dv * du));
    if (val_t) val_t[e] = val[e];
  }
}

struct CsrWs {
  uint64_t* a;
  uint64_t* b;
  unsigned long long* count;
  void* temp;
  size_t temp_bytes;
};

static gnn_status csr_ws_layout(int32_t n, int64_t m, uint32_t flags, void* base, size_t cap,
                                CsrWs* out, size_t* total) {
  const bool sym = flags & GNN_CSR_SYMMETRIZE;
  const bool loops = flags & GNN_CSR_SELF_LOOPS;
  const int64_t cap_keys = (sym ? 2 * m : m) + (loops ? n : 0);
  size_t t1 = 0, t2 = 0;
  GNN_CUDA(cub::DeviceRadixSort::SortKeys(nullptr, t1, (uint64_t*)nullptr, (uint64_t*)nullptr,
                                          cap_keys > 0 ? cap_keys : 1, 0, 64));
  GNN_CUDA(cub::DeviceSelect::Unique(nullptr, t2, (uint64_t*)nullptr, (uint64_t*)nullptr,
                                     (unsigned long long*)nullptr, cap_keys > 0 ? cap_keys : 1));
  Arena ar(base, cap);
  out->a = ar.take<uint64_t>(cap_keys + 1);
  out->b = ar.take<uint64_t>(cap_keys + 1);
  out->count = ar.take<unsigned long long>(4);
  out->temp_bytes = t1 > t2 ? t1 : t2;
  out->temp = ar.take_bytes(out->temp_bytes);
  *total = ar.used;
  if (!ar.ok()) return fail(GNN_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", cap, ar.used);
  return GNN_OK;
}

// ------------------------------------------------------------------ boundary
__global__ void cut_keys_kernel(int n, const int64_t* __restrict__ rowptr,
                                const int32_t* __restrict__ col, int64_t nnz, int P, int shift,
                                uint64_t* __restrict__ keys, int64_t* __restrict__ eidx,
                                unsigned long long* __restrict__ count) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= nnz) return;
  const int64_t v = row_of(rowptr, n, e);
  const int64_t u = col[e];
  const int64_t pv = part_of(v, n, P), pu = part_of(u, n, P);
  if (pv == pu) return;
  const unsigned long long at = atomicAdd(count, 1ull);
  keys[at] = ((uint64_t)pv << shift) | (uint64_t)u;
  eidx[at] = e;
}

__global__ void part_start_kernel(int n, int P, int64_t* __restrict__ ps) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p <= P) ps[p] = ((int64_t)p * n) / P;
}

__global__ void slots_decode_kernel(const uint64_t* __restrict__ sk, int64_t S, int shift,
                                    int32_t* __restrict__ slot_node) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s < S) slot_node[s] = (int32_t)(sk[s] & ((uint64_t(1) << shift) - 1));
}

__global__ void send_start_kernel(const uint64_t* __restrict__ sk, int64_t S, int shift, int P,
                                  int64_t* __restrict__ send_start) {
  const int q = blockIdx.x * blockDim.x + threadIdx.x;
  if (q <= P) send_start[q] = lower_bound_dev(sk, S, (uint64_t)q << shift);
}

__global__ void copy_col_kernel(const int32_t* __restrict__ col, int64_t nnz,
                                int32_t* __restrict__ col_remap) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e < nnz) col_remap[e] = col[e];
}

// For every cut entry: its slot, the remapped column, and the backward key.
__global__ void cut_remap_kernel(int n, const int64_t* __restrict__ rowptr,
                                 const float* __restrict__ val, const uint64_t* __restrict__ keys,
                                 const int64_t* __restrict__ eidx, int64_t nc,
                                 const uint64_t* __restrict__ sk, int64_t S, int shift,
                                 int32_t* __restrict__ col_remap, uint64_t* __restrict__ key2,
                                 float* __restrict__ v2) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nc) return;
  const int64_t s = lower_bound_dev(sk, S, keys[i]);
  const int64_t e = eidx[i];
  col_remap[e] = ~(int32_t)s;
  const int64_t v = row_of(rowptr, n, e);
  key2[i] = ((uint64_t)s << shift) | (uint64_t)v;
  v2[i] = val[e];
}

// Row v's entries reordered: local sources first, then remote slots, each
// group keeping CSR order; weights follow their entries.
__global__ void reorder_rows_kernel(int n, const int64_t* __restrict__ rowptr,
                                    const int32_t* __restrict__ remap_csr,
                                    const float* __restrict__ val, const float* __restrict__ val_t,
                                    int32_t* __restrict__ col_remap, float* __restrict__ val_remap,
                                    float* __restrict__ val_remap_t, int32_t* __restrict__ local_cnt) {
  const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= n) return;
  const int64_t beg = rowptr[v], end = rowptr[v + 1];
  int64_t cnt = 0;
  for (int64_t e = beg; e < end; ++e) cnt += remap_csr[e] >= 0;
  local_cnt[v] = (int32_t)cnt;
  int64_t li = beg, ri = beg + cnt;
  for (int64_t e = beg; e < end; ++e) {
    const int32_t c = remap_csr[e];
    const float w = val[e];
    const int64_t at = c >= 0 ? li++ : ri++;
    col_remap[at] = c;
    val_remap[at] = w;
    if (val_remap_t) val_remap_t[at] = val_t[e];
  }
}

__global__ void slot_csr_kernel(const uint64_t* __restrict__ key2, int64_t nc, int shift,
                                int32_t* __restrict__ slot_col) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < nc) slot_col[i] = (int32_t)(key2[i] & ((uint64_t(1) << shift) - 1));
}

__global__ void bound_ptr_kernel(const uint64_t* __restrict__ keys, int64_t len, int shift,
                                 int64_t count, int64_t* __restrict__ ptr) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i <= count) ptr[i] = lower_bound_dev(keys, len, (uint64_t)i << shift);
}

__global__ void own_keys_kernel(const int32_t* __restrict__ slot_node, int64_t S, int shiftS,
                                uint64_t* __restrict__ k3) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s < S) k3[s] = ((uint64_t)slot_node[s] << shiftS) | (uint64_t)s;
}

__global__ void own_slot_kernel(const uint64_t* __restrict__ k3, int64_t S, int shiftS,
                                int32_t* __restrict__ own_slot) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s < S) own_slot[s] = (int32_t)(k3[s] & ((uint64_t(1) << shiftS) - 1));
}

__global__ void pool_degrees_kernel(int n, const int64_t* __restrict__ rowptr,
                                    const int64_t* __restrict__ own_ptr,
                                    uint32_t* __restrict__ deg, unsigned long long* count) {
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= n) return;
  if (own_ptr[u + 1] > own_ptr[u]) {
    const unsigned long long at = atomicAdd(count, 1ull);
    deg[at] = (uint32_t)(rowptr[u + 1] - rowptr[u]);
  }
}

__global__ void node_bits_kernel(int n, const int64_t* __restrict__ rowptr,
                                 const int64_t* __restrict__ own_ptr,
                                 const uint32_t* __restrict__ sorted_deg,
                                 const unsigned long long* __restrict__ pool_count,
                                 gnn_bit_rule rule, int base, uint8_t* __restrict__ node_bits) {
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= n) return;
  if (own_ptr[u + 1] == own_ptr[u]) {
    node_bits[u] = 0;
    return;
  }
  const int64_t np = (int64_t)*pool_count;
  const uint32_t d = (uint32_t)(rowptr[u + 1] - rowptr[u]);
  const int64_t c = upper_bound_dev(sorted_deg, np, d);
  int level = 0;
  for (int i = 0; i + 1 < rule.n_levels; ++i) level += (100 * c > (int64_t)rule.pct[i] * np) ? 1 : 0;
  const int mask = rule.bits[level];
  const int w = mask == 32 ? 32 : (mask * base > 8 ? 8 : mask * base);
  node_bits[u] = (uint8_t)w;
}

__global__ void slot_bits_kernel(const int32_t* __restrict__ slot_node, int64_t S,
                                 const uint8_t* __restrict__ node_bits, int F,
                                 uint8_t* __restrict__ slot_bits, int64_t* __restrict__ rb) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s > S) return;
  if (s == S) {
    rb[s] = 0;
    return;
  }
  const int b = node_bits[slot_node[s]];
  slot_bits[s] = (uint8_t)b;
  rb[s] = rowbytes_dev(b, F);
}

__global__ void rowbytes_kernel(const uint8_t* __restrict__ slot_bits, int64_t S, int F,
                                int64_t* __restrict__ rb) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s < S) rb[s] = rowbytes_dev(slot_bits[s], F);
  else if (s == S) rb[s] = 0;
}

// ------------------------------------------------------------------ row split
__global__ void split_flag_kernel(int n, const int64_t* __restrict__ rowptr, int T,
                                  int32_t* __restrict__ flag, int64_t* __restrict__ pc) {
  const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v > n) return;
  if (v == n) {
    flag[v] = 0;
    pc[v] = 0;
    return;
  }
  const int64_t d = rowptr[v + 1] - rowptr[v];
  const bool f = d > T;
  flag[v] = f ? 1 : 0;
  pc[v] = f ? (d + T - 1) / T : 0;
}

__global__ void split_fill_kernel(int n, const int64_t* __restrict__ rowptr, int T,
                                  const int32_t* __restrict__ flag, const int32_t* __restrict__ pos,
                                  const int64_t* __restrict__ pp, int32_t* __restrict__ long_rows,
                                  int64_t* __restrict__ piece_ptr, int32_t* __restrict__ piece_row,
                                  int64_t* __restrict__ piece_beg) {
  const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v > n) return;
  if (v == n) {
    piece_ptr[pos[n]] = pp[n];
    return;
  }
  if (!flag[v]) return;
  const int32_t i = pos[v];
  long_rows[i] = (int32_t)v;
  piece_ptr[i] = pp[v];
  const int64_t beg = rowptr[v], end = rowptr[v + 1];
  int64_t p = pp[v];
  for (int64_t e = beg; e < end; e += T, ++p) {
    piece_row[p] = (int32_t)v;
    piece_beg[p] = e;
  }
}

struct SplitWs {
  int32_t* flag;
  int32_t* pos;
  int64_t* pc;
  int64_t* pp;
  void* temp;
  size_t temp_bytes;
};

static gnn_status split_ws_layout(int n, void* base, size_t cap, SplitWs* w, size_t* total) {
  size_t t1 = 0, t2 = 0;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, t1, (int32_t*)nullptr, (int32_t*)nullptr, (int64_t)n + 1));
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, t2, (int64_t*)nullptr, (int64_t*)nullptr, (int64_t)n + 1));
  Arena ar(base, cap);
  w->flag = ar.take<int32_t>((size_t)n + 1);
  w->pos = ar.take<int32_t>((size_t)n + 1);
  w->pc = ar.take<int64_t>((size_t)n + 1);
  w->pp = ar.take<int64_t>((size_t)n + 1);
  w->temp_bytes = t1 > t2 ? t1 : t2;
  w->temp = ar.take_bytes(w->temp_bytes);
  *total = ar.used;
  if (!ar.ok()) return fail(GNN_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", cap, ar.used);
  return GNN_OK;
}

static gnn_status split_scan(const gnn_csr& csr, int T, SplitWs& w, int32_t* n_long,
                             int64_t* n_pieces, cudaStream_t st) {
  split_flag_kernel<<<GRID1((int64_t)csr.n + 1), 0, st>>>(csr.n, csr.rowptr, T, w.flag, w.pc);
  GNN_CHECK_LAUNCH();
  size_t tb = w.temp_bytes;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(w.temp, tb, w.flag, w.pos, (int64_t)csr.n + 1, st));
  tb = w.temp_bytes;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(w.temp, tb, w.pc, w.pp, (int64_t)csr.n + 1, st));
  GNN_CUDA(cudaMemcpyAsync(n_long, w.pos + csr.n, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaMemcpyAsync(n_pieces, w.pp + csr.n, sizeof(int64_t), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaStreamSynchronize(st));
  return GNN_OK;
}

struct BndWs {
  uint64_t* k0;  // cut keys (unsorted, paired with eidx)
  uint64_t* k1;  // sorted cut keys / backward keys
  uint64_t* k2;  // slot keys / sorted backward keys
  uint64_t* k3;  // owner keys (sorted in place via k1)
  int64_t* eidx;
  float* v1;
  float* v2;
  uint32_t* d1;
  uint32_t* d2;
  int64_t* rb;
  unsigned long long* count;  // [0] cut entries, [1] slots, [2] pool size
  void* temp;
  size_t temp_bytes;
};

static gnn_status bnd_ws_layout(int64_t nnz, int32_t n, void* base, size_t cap, BndWs* w,
                                size_t* total) {
  const int64_t E = nnz > 0 ? nnz : 1;
  const int64_t N = n > 0 ? n : 1;
  size_t t = 0, x = 0;
  GNN_CUDA(cub::DeviceRadixSort::SortKeys(nullptr, x, (uint64_t*)nullptr, (uint64_t*)nullptr, E, 0, 64));
  t = x > t ? x : t;
  GNN_CUDA(cub::DeviceSelect::Unique(nullptr, x, (uint64_t*)nullptr, (uint64_t*)nullptr,
                                     (unsigned long long*)nullptr, E));
  t = x > t ? x : t;
  GNN_CUDA(cub::DeviceRadixSort::SortPairs(nullptr, x, (uint64_t*)nullptr, (uint64_t*)nullptr,
                                           (float*)nullptr, (float*)nullptr, E, 0, 64));
  t = x > t ? x : t;
  GNN_CUDA(cub::DeviceRadixSort::SortKeys(nullptr, x, (uint32_t*)nullptr, (uint32_t*)nullptr, N, 0, 32));
  t = x > t ? x : t;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, x, (int64_t*)nullptr, (int64_t*)nullptr, E + 1));
  t = x > t ? x : t;
  Arena ar(base, cap);
  w->k0 = ar.take<uint64_t>(E);
  w->k1 = ar.take<uint64_t>(E);
  w->k2 = ar.take<uint64_t>(E);
  w->k3 = ar.take<uint64_t>(E);
  w->eidx = ar.take<int64_t>(E);
  w->v1 = ar.take<float>(E);
  w->v2 = ar.take<float>(E);
  w->d1 = ar.take<uint32_t>(N);
  w->d2 = ar.take<uint32_t>(N);
  w->rb = ar.take<int64_t>(E + 1);
  w->count = ar.take<unsigned long long>(4);
  w->temp_bytes = t;
  w->temp = ar.take_bytes(t);
  *total = ar.used;
  if (!ar.ok()) return fail(GNN_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", cap, ar.used);
  return GNN_OK;
}

// Cut entries -> sorted unique slot keys in w.k2; returns counts on the host.
static gnn_status cut_and_slots(const gnn_csr& csr, int P, int shift, BndWs& w, int64_t* nc,
                                int64_t* S, cudaStream_t st) {
  GNN_CUDA(cudaMemsetAsync(w.count, 0, 4 * sizeof(unsigned long long), st));
  if (csr.nnz > 0)
    cut_keys_kernel<<<GRID1(csr.nnz), 0, st>>>(csr.n, csr.rowptr, csr.col, csr.nnz, P, shift,
                                               w.k0, w.eidx, w.count);
  GNN_CHECK_LAUNCH();
  unsigned long long h = 0;
  GNN_CUDA(cudaMemcpyAsync(&h, w.count, sizeof(h), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaStreamSynchronize(st));
  *nc = (int64_t)h;
  if (*nc == 0) {
    *S = 0;
    return GNN_OK;
  }
  const int end_bit = bits_for((uint64_t)P) + shift;
  size_t tb = w.temp_bytes;
  GNN_CUDA(cub::DeviceRadixSort::SortKeys(w.temp, tb, w.k0, w.k1, *nc, 0, end_bit, st));
  tb = w.temp_bytes;
  GNN_CUDA(cub::DeviceSelect::Unique(w.temp, tb, w.k1, w.k2, w.count + 1, *nc, st));
  GNN_CUDA(cudaMemcpyAsync(&h, w.count + 1, sizeof(h), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaStreamSynchronize(st));
  *S = (int64_t)h;
  return GNN_OK;
}

static gnn_status compute_bits(const gnn_csr& csr, const gnn_bit_rule& rule, int base, int F,
                               gnn_boundary& b, BndWs& w, cudaStream_t st) {
  const int n = csr.n;
  GNN_CUDA(cudaMemsetAsync(w.count + 2, 0, sizeof(unsigned long long), st));
  pool_degrees_kernel<<<GRID1(n), 0, st>>>(n, csr.rowptr, b.own_ptr, w.d1, w.count + 2);
  GNN_CHECK_LAUNCH();
  unsigned long long np = 0;
  GNN_CUDA(cudaMemcpyAsync(&np, w.count + 2, sizeof(np), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaStreamSynchronize(st));
  if (np > 0) {
    size_t tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceRadixSort::SortKeys(w.temp, tb, w.d1, w.d2, (int64_t)np, 0, 32, st));
  }
  node_bits_kernel<<<GRID1(n), 0, st>>>(n, csr.rowptr, b.own_ptr, w.d2, w.count + 2, rule, base,
                                        b.node_bits);
  GNN_CHECK_LAUNCH();
  const int64_t S = b.n_slots;
  slot_bits_kernel<<<GRID1(S + 1), 0, st>>>(b.slot_node, S, b.node_bits, F, b.slot_bits, w.rb);
  GNN_CHECK_LAUNCH();
  size_t tb = w.temp_bytes;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(w.temp, tb, w.rb, b.slot_off, S + 1, st));
  b.F = F;
  return GNN_OK;
}

static gnn_status check_rule(const gnn_bit_rule* rule, int base) {
  if (!rule) return fail(GNN_ERR_INVALID_ARG, "bit rule is NULL");
  if (rule->n_levels < 1 || rule->n_levels > 4)
    return fail(GNN_ERR_INVALID_ARG, "bit rule: n_levels must be 1..4");
  for (int i = 0; i < rule->n_levels; ++i)
    if (!is_valid_bits(rule->bits[i]))
      return fail(GNN_ERR_INVALID_ARG, "bit rule: bits must be 1, 2, 4, 8 or 32");
  for (int i = 0; i + 1 < rule->n_levels; ++i) {
    if (rule->pct[i] < 0 || rule->pct[i] > 100)
      return fail(GNN_ERR_INVALID_ARG, "bit rule: pct must be 0..100");
    if (i > 0 && rule->pct[i] < rule->pct[i - 1])
      return fail(GNN_ERR_INVALID_ARG, "bit rule: pct must ascend");
  }
  if (!(base == 1 || base == 2 || base == 4 || base == 8))
    return fail(GNN_ERR_INVALID_ARG, "base_bits must be 1, 2, 4 or 8");
  return GNN_OK;
}

}  // namespace gnn

using namespace gnn;

extern "C" gnn_status gnn_csr_build_workspace(int32_t n, int64_t n_edges, uint32_t flags,
                                              size_t* ws_bytes) {
  GNN_REQUIRE(n >= 0 && n_edges >= 0 && ws_bytes, "gnn_csr_build_workspace: bad arguments");
  CsrWs w;
  return csr_ws_layout(n, n_edges, flags, nullptr, 0, &w, ws_bytes);
}

extern "C" gnn_status gnn_csr_build(int32_t n, int64_t n_edges, const int32_t* src,
                                    const int32_t* dst, uint32_t flags, int64_t capacity,
                                    gnn_csr* out, void* ws, size_t ws_bytes,
                                    gnn_stream_t stream) {
  GNN_REQUIRE(out, "gnn_csr_build: out is NULL");
  GNN_REQUIRE(n >= 0 && n_edges >= 0 && capacity >= 0, "gnn_csr_build: negative size");
  GNN_REQUIRE(n_edges == 0 || (src && dst), "gnn_csr_build: NULL edge list");
  GNN_REQUIRE(out->rowptr && (capacity == 0 || (out->col && out->val)),
              "gnn_csr_build: NULL output arrays");
  GNN_REQUIRE((flags & ~15u) == 0, "gnn_csr_build: unknown flag bits");
  cudaStream_t st = as_stream(stream);
  CsrWs w;
  size_t need = 0;
  gnn_status s = csr_ws_layout(n, n_edges, flags, ws, ws_bytes, &w, &need);
  if (s != GNN_OK) return s;
  GNN_REQUIRE(ws, "gnn_csr_build: NULL workspace");
  const bool sym = flags & GNN_CSR_SYMMETRIZE, loops = flags & GNN_CSR_SELF_LOOPS;
  const int shift = bits_for((uint64_t)(n > 0 ? n : 1));
  // the build's own bad-endpoint flag lives in its workspace (count[3]), so
  // a flag another kernel raised in the library-wide word is left for
  // gnn_sync_check to report
  unsigned* dflags = reinterpret_cast<unsigned*>(w.count + 3);
  GNN_CUDA(cudaMemsetAsync(w.count, 0, 4 * sizeof(unsigned long long), st));
  if (n_edges > 0)
    emit_edge_keys<<<GRID1(n_edges), 0, st>>>(n_edges, src, dst, n, shift, sym, loops, w.a,
                                              w.count, dflags);
  GNN_CHECK_LAUNCH();
  if (loops && n > 0) {
    emit_loop_keys<<<GRID1(n), 0, st>>>(n, shift, w.a, w.count);
    GNN_CHECK_LAUNCH();
  }
  unsigned long long cnt = 0;
  unsigned bad = 0;
  GNN_CUDA(cudaMemcpyAsync(&cnt, w.count, sizeof(cnt), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaMemcpyAsync(&bad, dflags, sizeof(bad), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaStreamSynchronize(st));
  if (bad) return fail(GNN_ERR_INVALID_ARG, "gnn_csr_build: an edge endpoint is outside [0, n)");
  const int64_t total = (int64_t)cnt + (loops ? n : 0);
  const int end_bit = 2 * shift;
  uint64_t* sorted = w.a;
  int64_t nnz = total;
  if (total > 0) {
    size_t tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceRadixSort::SortKeys(w.temp, tb, w.a, w.b, total, 0, end_bit, st));
    sorted = w.b;
    if (flags & GNN_CSR_DEDUP) {
      tb = w.temp_bytes;
      GNN_CUDA(cub::DeviceSelect::Unique(w.temp, tb, w.b, w.a, w.count + 1, total, st));
      GNN_CUDA(cudaMemcpyAsync(&cnt, w.count + 1, sizeof(cnt), cudaMemcpyDeviceToHost, st));
      GNN_CUDA(cudaStreamSynchronize(st));
      nnz = (int64_t)cnt;
      sorted = w.a;
    }
  }
  out->n = n;
  out->nnz = nnz;
  const bool mean = flags & GNN_CSR_MEAN;
  out->symmetric = sym && !mean ? 1 : 0;
  // A^T weights exist on the pattern only when it is symmetric
  float* val_t = sym && mean ? out->val_t : nullptr;
  if (!(sym && mean)) out->val_t = nullptr;
  if (nnz > capacity)
    return fail(GNN_ERR_CAPACITY, "gnn_csr_build: %lld entries exceed capacity %lld",
                (long long)nnz, (long long)capacity);
  csr_rowptr_kernel<<<GRID1((int64_t)n + 1), 0, st>>>(n, sorted, nnz, shift, out->rowptr);
  GNN_CHECK_LAUNCH();
  if (nnz > 0) {
    csr_fill_kernel<<<GRID1(nnz), 0, st>>>(sorted, nnz, shift, out->rowptr, mean ? 1 : 0,
                                           out->col, out->val, val_t);
    GNN_CHECK_LAUNCH();
  }
  GNN_CUDA(cudaStreamSynchronize(st));
  return GNN_OK;
}

static gnn_status check_csr_setup(const gnn_csr* csr, const char* who) {
  if (!csr || csr->n < 1 || csr->nnz < 0 || !csr->rowptr || (csr->nnz > 0 && (!csr->col || !csr->val)))
    return fail(GNN_ERR_INVALID_ARG, "%s: invalid csr", who);
  return GNN_OK;
}

extern "C" gnn_status gnn_boundary_workspace(const gnn_csr* csr, int32_t P, size_t* ws_bytes) {
  gnn_status s = check_csr_setup(csr, "gnn_boundary_workspace");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(P >= 1 && ws_bytes, "gnn_boundary_workspace: bad arguments");
  BndWs w;
  return bnd_ws_layout(csr->nnz, csr->n, nullptr, 0, &w, ws_bytes);
}

extern "C" gnn_status gnn_boundary_count(const gnn_csr* csr, int32_t P, int64_t* n_slots,
                                         int64_t* nnz_cut, void* ws, size_t ws_bytes,
                                         gnn_stream_t stream) {
  gnn_status s = check_csr_setup(csr, "gnn_boundary_count");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(P >= 1 && n_slots && nnz_cut && ws, "gnn_boundary_count: bad arguments");
  BndWs w;
  size_t need = 0;
  if ((s = bnd_ws_layout(csr->nnz, csr->n, ws, ws_bytes, &w, &need)) != GNN_OK) return s;
  const int shift = bits_for((uint64_t)csr->n);
  return cut_and_slots(*csr, P, shift, w, nnz_cut, n_slots, as_stream(stream));
}

extern "C" gnn_status gnn_boundary_index(const gnn_csr* csr, const gnn_bit_rule* rule,
                                         uint8_t base_bits, int32_t F, gnn_boundary* out,
                                         void* ws, size_t ws_bytes, gnn_stream_t stream) {
  gnn_status s = check_csr_setup(csr, "gnn_boundary_index");
  if (s != GNN_OK) return s;
  if ((s = check_rule(rule, base_bits)) != GNN_OK) return s;
  GNN_REQUIRE(out && ws && F >= 1, "gnn_boundary_index: bad arguments");
  GNN_REQUIRE(out->P >= 1, "gnn_boundary_index: out->P must be set");
  GNN_REQUIRE(out->part_start && out->send_start && out->col_remap && out->val_remap &&
                  out->local_cnt && out->own_ptr && out->node_bits && out->slot_off &&
                  out->slot_rowptr,
              "gnn_boundary_index: NULL output array");
  GNN_REQUIRE(out->n_slots == 0 || (out->slot_node && out->own_slot && out->slot_bits),
              "gnn_boundary_index: NULL slot array");
  GNN_REQUIRE(out->nnz_cut == 0 || (out->slot_col && out->slot_val),
              "gnn_boundary_index: NULL backward array");
  cudaStream_t st = as_stream(stream);
  BndWs w;
  size_t need = 0;
  if ((s = bnd_ws_layout(csr->nnz, csr->n, ws, ws_bytes, &w, &need)) != GNN_OK) return s;
  const int n = csr->n, P = out->P;
  const int shift = bits_for((uint64_t)n);
  int64_t nc = 0, S = 0;
  if ((s = cut_and_slots(*csr, P, shift, w, &nc, &S, st)) != GNN_OK) return s;
  if (S != out->n_slots || nc != out->nnz_cut)
    return fail(GNN_ERR_INVALID_ARG, "gnn_boundary_index: out sizes (%lld slots, %lld cut) do not "
                "match the graph (%lld, %lld)", (long long)out->n_slots, (long long)out->nnz_cut,
                (long long)S, (long long)nc);
  out->n = n;
  part_start_kernel<<<GRID1(P + 1), 0, st>>>(n, P, out->part_start);
  send_start_kernel<<<GRID1(P + 1), 0, st>>>(w.k2, S, shift, P, out->send_start);
  if (S > 0) slots_decode_kernel<<<GRID1(S), 0, st>>>(w.k2, S, shift, out->slot_node);
  // col_remap in CSR order goes to a temporary first (w.v2 is free here)
  int32_t* remap_csr = reinterpret_cast<int32_t*>(w.v2);
  if (csr->nnz > 0) copy_col_kernel<<<GRID1(csr->nnz), 0, st>>>(csr->col, csr->nnz, remap_csr);
  GNN_CHECK_LAUNCH();
  const int shiftS = bits_for((uint64_t)(S > 0 ? S : 1));
  if (nc > 0) {
    // backward entries keyed (s, v): slot s's rows v in ascending order
    cut_remap_kernel<<<GRID1(nc), 0, st>>>(n, csr->rowptr, csr->val, w.k0, w.eidx, nc, w.k2, S,
                                          shift, remap_csr, w.k1, w.v1);
    GNN_CHECK_LAUNCH();
    size_t tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceRadixSort::SortPairs(w.temp, tb, w.k1, w.k3, w.v1, out->slot_val, nc, 0,
                                             shiftS + shift, st));
    slot_csr_kernel<<<GRID1(nc), 0, st>>>(w.k3, nc, shift, out->slot_col);
    GNN_CHECK_LAUNCH();
  }
  bound_ptr_kernel<<<GRID1(S + 1), 0, st>>>(w.k3, nc, shift, S, out->slot_rowptr);
  GNN_CHECK_LAUNCH();
  float* vrt = csr->val_t ? out->val_remap_t : nullptr;
  if (!csr->val_t) out->val_remap_t = nullptr;
  reorder_rows_kernel<<<GRID1(n), 0, st>>>(n, csr->rowptr, remap_csr, csr->val, csr->val_t,
                                           out->col_remap, out->val_remap, vrt, out->local_cnt);
  GNN_CHECK_LAUNCH();
  // owner lists keyed (u, s)
  if (S > 0) {
    own_keys_kernel<<<GRID1(S), 0, st>>>(out->slot_node, S, shiftS, w.k0);
    GNN_CHECK_LAUNCH();
    size_t tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceRadixSort::SortKeys(w.temp, tb, w.k0, w.k1, S, 0, shiftS + shift, st));
    own_slot_kernel<<<GRID1(S), 0, st>>>(w.k1, S, shiftS, out->own_slot);
    GNN_CHECK_LAUNCH();
  }
  bound_ptr_kernel<<<GRID1((int64_t)n + 1), 0, st>>>(w.k1, S, shiftS, n, out->own_ptr);
  GNN_CHECK_LAUNCH();
  if ((s = compute_bits(*csr, *rule, base_bits, F, *out, w, st)) != GNN_OK) return s;
  GNN_CUDA(cudaStreamSynchronize(st));
  return GNN_OK;
}

extern "C" gnn_status gnn_boundary_set_bits(const gnn_csr* csr, const gnn_bit_rule* rule,
                                            uint8_t base_bits, int32_t F, gnn_boundary* bnd,
                                            void* ws, size_t ws_bytes, gnn_stream_t stream) {
  gnn_status s = check_csr_setup(csr, "gnn_boundary_set_bits");
  if (s != GNN_OK) return s;
  if ((s = check_rule(rule, base_bits)) != GNN_OK) return s;
  GNN_REQUIRE(bnd && ws && F >= 1 && bnd->own_ptr && bnd->node_bits && bnd->slot_off &&
                  (bnd->n_slots == 0 || (bnd->slot_node && bnd->slot_bits)),
              "gnn_boundary_set_bits: bad arguments");
  BndWs w;
  size_t need = 0;
  if ((s = bnd_ws_layout(csr->nnz, csr->n, ws, ws_bytes, &w, &need)) != GNN_OK) return s;
  cudaStream_t st = as_stream(stream);
  if ((s = compute_bits(*csr, *rule, base_bits, F, *bnd, w, st)) != GNN_OK) return s;
  GNN_CUDA(cudaStreamSynchronize(st));
  return GNN_OK;
}

extern "C" gnn_status gnn_slot_offsets_workspace(int64_t n_slots, size_t* ws_bytes) {
  GNN_REQUIRE(n_slots >= 0 && ws_bytes, "gnn_slot_offsets_workspace: bad arguments");
  size_t t = 0;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, t, (int64_t*)nullptr, (int64_t*)nullptr, n_slots + 1));
  Arena ar(nullptr, 0);
  ar.take<int64_t>(n_slots + 1);
  ar.take_bytes(t);
  *ws_bytes = ar.used;
  return GNN_OK;
}

extern "C" gnn_status gnn_slot_offsets(const uint8_t* slot_bits, int64_t n_slots, int32_t F,
                                       int64_t* slot_off, void* ws, size_t ws_bytes,
                                       gnn_stream_t stream) {
  GNN_REQUIRE(n_slots >= 0 && F >= 1 && slot_off && ws && (n_slots == 0 || slot_bits),
              "gnn_slot_offsets: bad arguments");
  size_t t = 0;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, t, (int64_t*)nullptr, (int64_t*)nullptr, n_slots + 1));
  Arena ar(ws, ws_bytes);
  int64_t* rb = ar.take<int64_t>(n_slots + 1);
  void* temp = ar.take_bytes(t);
  if (!ar.ok()) return fail(GNN_ERR_INVALID_ARG, "gnn_slot_offsets: workspace too small");
  cudaStream_t st = as_stream(stream);
  rowbytes_kernel<<<GRID1(n_slots + 1), 0, st>>>(slot_bits, n_slots, F, rb);
  GNN_CHECK_LAUNCH();
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(temp, t, rb, slot_off, n_slots + 1, st));
  return GNN_OK;
}

extern "C" gnn_status gnn_csr_split_workspace(const gnn_csr* csr, size_t* ws_bytes) {
  gnn_status s = check_csr_setup(csr, "gnn_csr_split_workspace");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(ws_bytes, "gnn_csr_split_workspace: NULL ws_bytes");
  SplitWs w;
  return split_ws_layout(csr->n, nullptr, 0, &w, ws_bytes);
}

extern "C" gnn_status gnn_csr_split_count(const gnn_csr* csr, int32_t split_len, int32_t* n_long,
                                          int64_t* n_pieces, void* ws, size_t ws_bytes,
                                          gnn_stream_t stream) {
  gnn_status s = check_csr_setup(csr, "gnn_csr_split_count");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(split_len >= 32 && n_long && n_pieces && ws, "gnn_csr_split_count: bad arguments");
  SplitWs w;
  size_t need = 0;
  if ((s = split_ws_layout(csr->n, ws, ws_bytes, &w, &need)) != GNN_OK) return s;
  return split_scan(*csr, split_len, w, n_long, n_pieces, as_stream(stream));
}

extern "C" gnn_status gnn_csr_split(gnn_csr* csr, void* ws, size_t ws_bytes, gnn_stream_t stream) {
  gnn_status s = check_csr_setup(csr, "gnn_csr_split");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(csr->split_len >= 32 && ws, "gnn_csr_split: split_len must be >= 32");
  GNN_REQUIRE(csr->piece_ptr && (csr->n_long == 0 || csr->long_rows) &&
                  (csr->n_pieces == 0 || (csr->piece_row && csr->piece_beg)),
              "gnn_csr_split: NULL plan array");
  SplitWs w;
  size_t need = 0;
  if ((s = split_ws_layout(csr->n, ws, ws_bytes, &w, &need)) != GNN_OK) return s;
  cudaStream_t st = as_stream(stream);
  int32_t nl = 0;
  int64_t np = 0;
  if ((s = split_scan(*csr, csr->split_len, w, &nl, &np, st)) != GNN_OK) return s;
  if (nl != csr->n_long || np != csr->n_pieces)
    return fail(GNN_ERR_INVALID_ARG, "gnn_csr_split: n_long/n_pieces (%d, %lld) do not match the "
                "graph (%d, %lld)", csr->n_long, (long long)csr->n_pieces, nl, (long long)np);
  split_fill_kernel<<<GRID1((int64_t)csr->n + 1), 0, st>>>(csr->n, csr->rowptr, csr->split_len,
                                                         w.flag, w.pos, w.pp, csr->long_rows,
                                                         csr->piece_ptr, csr->piece_row,
                                                         csr->piece_beg);
  GNN_CHECK_LAUNCH();
  GNN_CUDA(cudaStreamSynchronize(st));
  return GNN_OK;
}

// ------------------------------------------------------------------ long slots
__global__ void long_flag_kernel(int64_t S, const int64_t* __restrict__ srp, int T,
                                 int32_t* __restrict__ flag) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s > S) return;
  flag[s] = (s < S && srp[s + 1] - srp[s] > T) ? 1 : 0;
}

__global__ void long_fill_kernel(int64_t S, const int32_t* __restrict__ flag,
                                 const int32_t* __restrict__ pos, int32_t* __restrict__ out) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s < S && flag[s]) out[pos[s]] = (int32_t)s;
}

static gnn_status long_slots_scan(const gnn_boundary& b, int T, void* ws, size_t ws_bytes,
                                  int32_t** flag, int32_t** pos, int32_t* count, cudaStream_t st) {
  const int64_t S = b.n_slots;
  size_t t = 0;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, t, (int32_t*)nullptr, (int32_t*)nullptr, S + 1));
  Arena ar(ws, ws_bytes);
  *flag = ar.take<int32_t>((size_t)S + 1);
  *pos = ar.take<int32_t>((size_t)S + 1);
  void* temp = ar.take_bytes(t);
  if (!ar.ok()) return fail(GNN_ERR_INVALID_ARG, "long slots: workspace too small");
  long_flag_kernel<<<GRID1(S + 1), 0, st>>>(S, b.slot_rowptr, T, *flag);
  GNN_CHECK_LAUNCH();
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(temp, t, *flag, *pos, S + 1, st));
  GNN_CUDA(cudaMemcpyAsync(count, *pos + S, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaStreamSynchronize(st));
  return GNN_OK;
}

extern "C" gnn_status gnn_boundary_long_slots_count(const gnn_boundary* bnd, int32_t long_slot_len,
                                                    int32_t* n_long_slots, void* ws,
                                                    size_t ws_bytes, gnn_stream_t stream) {
  GNN_REQUIRE(bnd && n_long_slots && ws && long_slot_len >= 32 && bnd->slot_rowptr,
              "gnn_boundary_long_slots_count: bad arguments");
  int32_t *flag, *pos;
  return long_slots_scan(*bnd, long_slot_len, ws, ws_bytes, &flag, &pos, n_long_slots,
                         as_stream(stream));
}

// Halo visiting order: key (first backward entry v) << 32 | s, sorted.
__global__ void halo_key_kernel(int64_t S, const int64_t* __restrict__ srp,
                                const int32_t* __restrict__ scol, uint64_t* __restrict__ key) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= S) return;
  const int64_t b = srp[s];
  const uint32_t v = b < srp[s + 1] ? (uint32_t)scol[b] : 0xffffffffu;
  key[s] = ((uint64_t)v << 32) | (uint64_t)s;
}

__global__ void halo_order_kernel(int64_t S, const uint64_t* __restrict__ key,
                                  int32_t* __restrict__ order) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < S) order[i] = (int32_t)(key[i] & 0xffffffffu);
}

static gnn_status halo_order_fill(const gnn_boundary& b, void* ws, size_t ws_bytes,
                                  cudaStream_t st) {
  const int64_t S = b.n_slots;
  if (S == 0) return GNN_OK;
  size_t t = 0;
  GNN_CUDA(cub::DeviceRadixSort::SortKeys(nullptr, t, (uint64_t*)nullptr, (uint64_t*)nullptr, S, 0, 64));
  Arena ar(ws, ws_bytes);
  uint64_t* k0 = ar.take<uint64_t>((size_t)S);
  uint64_t* k1 = ar.take<uint64_t>((size_t)S);
  void* temp = ar.take_bytes(t);
  if (!ar.ok()) return fail(GNN_ERR_INVALID_ARG, "halo order: workspace too small");
  halo_key_kernel<<<GRID1(S), 0, st>>>(S, b.slot_rowptr, b.slot_col, k0);
  GNN_CHECK_LAUNCH();
  GNN_CUDA(cub::DeviceRadixSort::SortKeys(temp, t, k0, k1, S, 0, 64, st));
  halo_order_kernel<<<GRID1(S), 0, st>>>(S, k1, b.halo_order);
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

extern "C" gnn_status gnn_boundary_long_slots(gnn_boundary* bnd, void* ws, size_t ws_bytes,
                                              gnn_stream_t stream) {
  GNN_REQUIRE(bnd && ws && bnd->long_slot_len >= 32 && bnd->slot_rowptr &&
                  (bnd->n_long_slots == 0 || bnd->long_slots),
              "gnn_boundary_long_slots: bad arguments");
  cudaStream_t st = as_stream(stream);
  int32_t *flag, *pos, count = 0;
  gnn_status s = long_slots_scan(*bnd, bnd->long_slot_len, ws, ws_bytes, &flag, &pos, &count, st);
  if (s != GNN_OK) return s;
  if (count != bnd->n_long_slots)
    return fail(GNN_ERR_INVALID_ARG, "gnn_boundary_long_slots: n_long_slots %d does not match %d",
                bnd->n_long_slots, count);
  if (bnd->n_slots > 0) {
    long_fill_kernel<<<GRID1(bnd->n_slots), 0, st>>>(bnd->n_slots, flag, pos, bnd->long_slots);
    GNN_CHECK_LAUNCH();
  }
  GNN_CUDA(cudaStreamSynchronize(st));
  if (bnd->halo_order && bnd->n_slots > 0) {
    if (bnd->nnz_cut > 0 && !bnd->slot_col)
      return fail(GNN_ERR_INVALID_ARG, "gnn_boundary_long_slots: slot_col is NULL");
    if ((s = halo_order_fill(*bnd, ws, ws_bytes, st)) != GNN_OK) return s;
    GNN_CUDA(cudaStreamSynchronize(st));
  }
  return GNN_OK;
}
