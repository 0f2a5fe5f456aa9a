// Stochastic integer quantisation + packing of message rows, and the
// standalone receive-side unpacking (SYLVIE guide, section 6).
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"
#include "kernels.h"

namespace gnn {

// Rows per group: a group walks QK consecutive rows and loads the next row
// (and its width and offset) before it quantises the current one, so the
// row's HBM latency overlaps the quantiser's arithmetic.
#ifndef GNN_QUANT_ROWS
#define GNN_QUANT_ROWS 1
#endif

template <int G, int CPL>
__device__ __forceinline__ void load_row(const float* __restrict__ X, int64_t ldx,
                                         const int32_t* __restrict__ row_idx, int64_t r, int nch,
                                         int gl, float4 (&v)[CPL]) {
  const int64_t src = row_idx ? (int64_t)__ldg(row_idx + r) : r;
  const float4* x = reinterpret_cast<const float4*>(X + src * ldx);
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = gl + i * G;
    v[i] = c < nch ? __ldg(x + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int G, int CPL, int QK = GNN_QUANT_ROWS>
__global__ void __launch_bounds__(256) quant_pack_kernel(
    const float* __restrict__ X, int64_t ldx, int F, const int32_t* __restrict__ row_idx,
    int64_t n_rows, const uint8_t* __restrict__ row_bits, const int64_t* __restrict__ row_off,
    uint32_t seed, uint8_t* __restrict__ packed, float2* __restrict__ meta, int64_t r0) {
  const int lane = threadIdx.x & 31;
  const int gl = lane & (G - 1);
  const int64_t i0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / G) * QK;
  if (i0 >= n_rows) return;  // uniform across the group
  const uint32_t gmask = group_mask(G, lane);
  const int nch = (F + 3) >> 2;
  float4 v[CPL];
  load_row<G, CPL>(X, ldx, row_idx, r0 + i0, nch, gl, v);
  int b = __ldg(row_bits + r0 + i0);
  int64_t off = __ldg(row_off + r0 + i0);
#pragma unroll 1
  for (int j = 0; j < QK; ++j) {
    const int64_t idx = i0 + j;
    if (idx >= n_rows) break;  // uniform
    const int64_t r = r0 + idx;  // row (and row key) of this step
    float4 nv[CPL];
    int nb = 0;
    int64_t noff = 0;
    if (QK > 1 && j + 1 < QK && idx + 1 < n_rows) {
      load_row<G, CPL>(X, ldx, row_idx, r + 1, nch, gl, nv);
      nb = __ldg(row_bits + r + 1);
      noff = __ldg(row_off + r + 1);
    }
    quantize_pack_row<G, CPL>(v, F, b, row_key(seed, (uint32_t)r), packed + off, meta + r, gl,
                              gmask);
    if (QK > 1) {
#pragma unroll
      for (int i = 0; i < CPL; ++i) v[i] = nv[i];
      b = nb;
      off = noff;
    }
  }
}

// Forward messages grouped by their node: a group walks K consecutive
// entries of the owner lists (own_slot: the slots of node 0, then node 1,
// ...), so consecutive slots mostly share a node.  When the node changes the
// group loads the node's row and prepares it (min, max, scale and every
// element's quotient, quant_prepare) -- once for all the slots that send it
// -- and each slot then only draws its codes with its own row key (the slot
// index) and writes its packed row and meta.  The bytes are those of the
// per-slot quantiser: the quotients do not depend on the slot.
template <int G, int CPL, int K>
__global__ void __launch_bounds__(256, 4) quant_pack_owned_kernel(
    const float* __restrict__ X, int64_t ldx, int F, int64_t S,
    const int32_t* __restrict__ own_slot, const int32_t* __restrict__ slot_node,
    const uint8_t* __restrict__ slot_bits, const int64_t* __restrict__ slot_off, uint32_t seed,
    uint8_t* __restrict__ packed, float2* __restrict__ meta) {
  const int lane = threadIdx.x & 31;
  const int gl = lane & (G - 1);
  const int64_t k0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / G) * K;
  if (k0 >= S) return;  // uniform across the group
  const uint32_t gmask = group_mask(G, lane);
  const int nch = (F + 3) >> 2;
  const int kn = (int)min((int64_t)K, S - k0);
  // lane j of the group holds entry k0 + (a multiple of G) + j: its slot,
  // node, width and offset
  int my_s = 0, my_u = -1, my_b = 0;
  int64_t my_off = 0;
  float4 t[CPL];
  float mn = 0.f, scale = 0.f;
  bool flat = true;
  int cur_u = -1, cur_b = 0;
#pragma unroll 1
  for (int j = 0; j < kn; ++j) {
    const int jj = j % G;
    if (jj == 0) {  // the next G entries' slots, nodes, widths and offsets
      my_s = 0;
      my_u = -1;
      my_b = 0;
      my_off = 0;
      if (j + gl < kn) {
        my_s = __ldg(own_slot + k0 + j + gl);
        my_u = __ldg(slot_node + my_s);
        my_b = __ldg(slot_bits + my_s);
        my_off = __ldg(slot_off + my_s);
      }
    }
    const int s = __shfl_sync(gmask, my_s, jj, G);
    const int u = __shfl_sync(gmask, my_u, jj, G);
    const int b = __shfl_sync(gmask, my_b, jj, G);
    const int64_t off = __shfl_sync(gmask, my_off, jj, G);
    const float4* x = reinterpret_cast<const float4*>(X + (int64_t)u * ldx);
    if (b == 32) {  // fp32 pass-through (testing): the row as it is
      float4 v[CPL];
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = gl + i * G;
        v[i] = c < nch ? __ldg(x + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      store_raw_row<G, CPL>(v, F, packed + off, gl);
      if (gl == 0) meta[s] = make_float2(0.f, 0.f);
      continue;
    }
    if (u != cur_u || b != cur_b) {  // a new row: load and prepare it
      float4 v[CPL];
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = gl + i * G;
        v[i] = c < nch ? __ldg(x + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      quant_prepare<G, CPL>(v, F, b, gl, gmask, t, mn, scale, flat);
      cur_u = u;
      cur_b = b;
    }
    pack_codes_b<G, CPL>(t, F, b, flat, row_key(seed, (uint32_t)s),
                         reinterpret_cast<uint32_t*>(packed + off), gl, gmask);
    if (gl == 0) meta[s] = make_float2(mn, scale);
  }
}

template <int G>
__global__ void __launch_bounds__(256) dequant_unpack_kernel(
    const uint8_t* __restrict__ packed, const float2* __restrict__ meta,
    const int64_t* __restrict__ row_off, const uint8_t* __restrict__ row_bits, int64_t n_rows,
    int F, float* __restrict__ out, int64_t ldo) {
  const int lane = threadIdx.x & 31;
  const int gl = lane & (G - 1);
  const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / G;
  if (r >= n_rows) return;
  const int b = __ldg(row_bits + r);
  const float2 m = __ldg(meta + r);
  const uint8_t* row = packed + __ldg(row_off + r);
  float* o = out + r * ldo;
  const int nch = (F + 3) >> 2;
  for (int c = gl; c < nch; c += G) store_chunk_f32(o, c, F, dequant_chunk(row, b, m.x, m.y, c));
}

__global__ void __launch_bounds__(256) quant_divide_kernel(const float* __restrict__ a,
                                                          const float* __restrict__ b,
                                                          float* __restrict__ q, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
  {
    const Divisor d = make_divisor(__ldg(b + i));
    q[i] = d.fast ? div_rn<true>(__ldg(a + i), d) : div_rn<false>(__ldg(a + i), d);
  }
}

// Chunk slots a packed row of width 1 (the widest padding) spans.
static int quant_chunk_slots(int F) { return 32 * ((F + 127) / 128) > (F + 3) / 4 ? 32 * ((F + 127) / 128) : (F + 3) / 4; }

template <int G, int CPL>
static void launch_qp(const float* X, int64_t ldx, int F, const int32_t* row_idx, int64_t n_rows,
                      const uint8_t* bits, const int64_t* off, uint32_t seed, uint8_t* packed,
                      float2* meta, cudaStream_t st, int64_t r0) {
  const int64_t threads = ((n_rows + GNN_QUANT_ROWS - 1) / GNN_QUANT_ROWS) * G;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  quant_pack_kernel<G, CPL><<<(unsigned)grid, block, 0, st>>>(X, ldx, F, row_idx, n_rows, bits,
                                                               off, seed, packed, meta, r0);
}

gnn_status launch_quant_pack(const float* X, int64_t ldx, int F, const int32_t* row_idx,
                             int64_t n_rows, const uint8_t* bits, const int64_t* off,
                             uint32_t seed, uint8_t* packed, float2* meta, cudaStream_t st) {
  return launch_quant_pack_range(X, ldx, F, row_idx, 0, n_rows, bits, off, seed, packed, meta, st);
}

gnn_status launch_quant_pack_range(const float* X, int64_t ldx, int F, const int32_t* row_idx,
                                   int64_t r0, int64_t n_rows, const uint8_t* bits,
                                   const int64_t* off, uint32_t seed, uint8_t* packed,
                                   float2* meta, cudaStream_t st) {
  if (n_rows == 0) return GNN_OK;
  const int slots = quant_chunk_slots(F);
  if (slots <= 32) {
    launch_qp<8, 4>(X, ldx, F, row_idx, n_rows, bits, off, seed, packed, meta, st, r0);
  } else {
    switch ((slots + 31) / 32) {
      case 1: launch_qp<32, 1>(X, ldx, F, row_idx, n_rows, bits, off, seed, packed, meta, st, r0); break;
      case 2: launch_qp<32, 2>(X, ldx, F, row_idx, n_rows, bits, off, seed, packed, meta, st, r0); break;
      case 3: launch_qp<32, 3>(X, ldx, F, row_idx, n_rows, bits, off, seed, packed, meta, st, r0); break;
      case 4: launch_qp<32, 4>(X, ldx, F, row_idx, n_rows, bits, off, seed, packed, meta, st, r0); break;
      case 5: launch_qp<32, 5>(X, ldx, F, row_idx, n_rows, bits, off, seed, packed, meta, st, r0); break;
      case 6: launch_qp<32, 6>(X, ldx, F, row_idx, n_rows, bits, off, seed, packed, meta, st, r0); break;
      case 7: launch_qp<32, 7>(X, ldx, F, row_idx, n_rows, bits, off, seed, packed, meta, st, r0); break;
      case 8: launch_qp<32, 8>(X, ldx, F, row_idx, n_rows, bits, off, seed, packed, meta, st, r0); break;
      default: return fail(GNN_ERR_UNSUPPORTED, "quant_pack: F=%d exceeds %d", F, kMaxF);
    }
  }
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

// Owner-list entries per group of the node-grouped kernel, and the slot
// count from which it serves gnn_quant_pack_owned.  Measured on the R-MAT
// scale graph (37.9M slots of 7.2M nodes, 5.2 per node) at F = 256: K = 4,
// 8, 16 took 15.2, 12.7, 11.2 ms against 14.2 ms for the per-slot kernel;
// one group per node took 22.9 ms (most nodes send nothing and hubs run
// long).  On the DC-SBM graphs' 0.8M-3.4M slots the per-slot kernel is
// faster (Yelp-shaped 0.41 against 0.71 ms), so it serves them.
#ifndef GNN_OWNED_K
#define GNN_OWNED_K 16
#endif
#ifndef GNN_OWNED_MIN_SLOTS
#define GNN_OWNED_MIN_SLOTS (int64_t(1) << 24)
#endif
template <int G, int CPL>
static void launch_qpo(const gnn_boundary& b, const float* X, int64_t ldx, int F, uint32_t seed,
                       uint8_t* packed, float2* meta, cudaStream_t st) {
  constexpr int K = GNN_OWNED_K;
  const int64_t S = b.n_slots;
  const int64_t threads = ((S + K - 1) / K) * G;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  quant_pack_owned_kernel<G, CPL, K><<<(unsigned)grid, block, 0, st>>>(
      X, ldx, F, S, b.own_slot, b.slot_node, b.slot_bits, b.slot_off, seed, packed, meta);
}

gnn_status launch_quant_pack_owned(const gnn_boundary& b, const float* X, int64_t ldx, int F,
                                   uint32_t seed, uint8_t* packed, float2* meta, cudaStream_t st) {
  if (b.n_slots == 0) return GNN_OK;
  if (b.n_slots < GNN_OWNED_MIN_SLOTS || !b.own_slot)  // the per-slot kernel: the same bytes
    return launch_quant_pack(X, ldx, F, b.slot_node, b.n_slots, b.slot_bits, b.slot_off, seed,
                             packed, meta, st);
  const int slots = quant_chunk_slots(F);
  if (slots <= 32) {
    launch_qpo<8, 4>(b, X, ldx, F, seed, packed, meta, st);
  } else {
    switch ((slots + 31) / 32) {
      case 1: launch_qpo<32, 1>(b, X, ldx, F, seed, packed, meta, st); break;
      case 2: launch_qpo<32, 2>(b, X, ldx, F, seed, packed, meta, st); break;
      case 3: launch_qpo<32, 3>(b, X, ldx, F, seed, packed, meta, st); break;
      case 4: launch_qpo<32, 4>(b, X, ldx, F, seed, packed, meta, st); break;
      case 5: launch_qpo<32, 5>(b, X, ldx, F, seed, packed, meta, st); break;
      case 6: launch_qpo<32, 6>(b, X, ldx, F, seed, packed, meta, st); break;
      case 7: launch_qpo<32, 7>(b, X, ldx, F, seed, packed, meta, st); break;
      case 8: launch_qpo<32, 8>(b, X, ldx, F, seed, packed, meta, st); break;
      default: return fail(GNN_ERR_UNSUPPORTED, "quant_pack_owned: F=%d exceeds %d", F, kMaxF);
    }
  }
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

gnn_status launch_dequant_unpack(const uint8_t* packed, const float2* meta, const int64_t* off,
                                 const uint8_t* bits, int64_t n_rows, int F, float* out,
                                 int64_t ldo, cudaStream_t st) {
  if (n_rows == 0) return GNN_OK;
  const int nch = (F + 3) / 4;
  const int block = 256;
  if (nch <= 8) {
    const int64_t grid = (n_rows * 8 + block - 1) / block;
    dequant_unpack_kernel<8><<<(unsigned)grid, block, 0, st>>>(packed, meta, off, bits, n_rows, F,
                                                               out, ldo);
  } else {
    const int64_t grid = (n_rows * 32 + block - 1) / block;
    dequant_unpack_kernel<32><<<(unsigned)grid, block, 0, st>>>(packed, meta, off, bits, n_rows,
                                                                F, out, ldo);
  }
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

}  // namespace gnn

using namespace gnn;

extern "C" gnn_status gnn_quant_pack(const float* X, int64_t ldx, int32_t F, const int32_t* row_idx,
                                     int64_t n_rows, const uint8_t* row_bits,
                                     const int64_t* row_off, uint32_t seed, uint8_t* packed,
                                     float* meta, gnn_stream_t stream) {
  GNN_REQUIRE(n_rows >= 0, "gnn_quant_pack: n_rows < 0");
  GNN_REQUIRE(F >= 1, "gnn_quant_pack: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_quant_pack: F=%d > %d", F, kMaxF);
  if (n_rows == 0) return GNN_OK;
  GNN_REQUIRE(X && row_bits && row_off && packed && meta, "gnn_quant_pack: NULL pointer");
  GNN_REQUIRE(ldx >= F && ldx % 4 == 0, "gnn_quant_pack: ldx must be >= F and a multiple of 4");
  GNN_REQUIRE(((uintptr_t)X & 15) == 0 && ((uintptr_t)packed & 15) == 0 && ((uintptr_t)meta & 7) == 0,
              "gnn_quant_pack: X and packed must be 16-byte aligned, meta 8-byte aligned");
  return launch_quant_pack(X, ldx, F, row_idx, n_rows, row_bits, row_off, seed, packed,
                           reinterpret_cast<float2*>(meta), as_stream(stream));
}

extern "C" gnn_status gnn_quant_pack_slots(const float* X, int64_t ldx, int32_t F,
                                           const int32_t* slot_node, int64_t s0, int64_t s1,
                                           const uint8_t* slot_bits, const int64_t* slot_off,
                                           uint32_t seed, uint8_t* packed, float* meta,
                                           gnn_stream_t stream) {
  GNN_REQUIRE(s0 >= 0 && s1 >= s0, "gnn_quant_pack_slots: need 0 <= s0 <= s1");
  GNN_REQUIRE(F >= 1, "gnn_quant_pack_slots: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_quant_pack_slots: F=%d > %d", F, kMaxF);
  if (s1 == s0) return GNN_OK;
  GNN_REQUIRE(X && slot_node && slot_bits && slot_off && packed && meta,
              "gnn_quant_pack_slots: NULL pointer");
  GNN_REQUIRE(ldx >= F && ldx % 4 == 0, "gnn_quant_pack_slots: ldx must be >= F and a multiple of 4");
  GNN_REQUIRE(((uintptr_t)X & 15) == 0 && ((uintptr_t)packed & 15) == 0 && ((uintptr_t)meta & 7) == 0,
              "gnn_quant_pack_slots: X and packed must be 16-byte aligned, meta 8-byte aligned");
  return launch_quant_pack_range(X, ldx, F, slot_node, s0, s1 - s0, slot_bits, slot_off, seed,
                                 packed, reinterpret_cast<float2*>(meta), as_stream(stream));
}

extern "C" gnn_status gnn_quant_pack_owned(const gnn_boundary* bnd, const float* X, int64_t ldx,
                                           int32_t F, uint32_t seed, uint8_t* packed, float* meta,
                                           gnn_stream_t stream) {
  GNN_REQUIRE(bnd, "gnn_quant_pack_owned: bnd is NULL");
  GNN_REQUIRE(F >= 1, "gnn_quant_pack_owned: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_quant_pack_owned: F=%d > %d", F, kMaxF);
  if (bnd->n_slots == 0) return GNN_OK;
  GNN_REQUIRE(bnd->n_slots > 0 && bnd->n_slots < (int64_t(1) << 31),
              "gnn_quant_pack_owned: n_slots out of range");
  GNN_REQUIRE(X && bnd->own_slot && bnd->slot_node && bnd->slot_bits && bnd->slot_off && packed &&
                  meta,
              "gnn_quant_pack_owned: NULL pointer");
  GNN_REQUIRE(ldx >= F && ldx % 4 == 0, "gnn_quant_pack_owned: ldx must be >= F and a multiple of 4");
  GNN_REQUIRE(((uintptr_t)X & 15) == 0 && ((uintptr_t)packed & 15) == 0 && ((uintptr_t)meta & 7) == 0,
              "gnn_quant_pack_owned: X and packed must be 16-byte aligned, meta 8-byte aligned");
  return launch_quant_pack_owned(*bnd, X, ldx, F, seed, packed, reinterpret_cast<float2*>(meta),
                                 as_stream(stream));
}

extern "C" gnn_status gnn_quant_divide(const float* a, const float* b, float* q, int64_t n,
                                       gnn_stream_t stream) {
  GNN_REQUIRE(n >= 0, "gnn_quant_divide: n < 0");
  if (n == 0) return GNN_OK;
  GNN_REQUIRE(a && b && q, "gnn_quant_divide: NULL pointer");
  int64_t grid = (n + 255) / 256;
  if (grid > 152 * 32) grid = 152 * 32;
  quant_divide_kernel<<<(unsigned)grid, 256, 0, as_stream(stream)>>>(a, b, q, n);
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

extern "C" gnn_status gnn_dequant_unpack(const uint8_t* packed, const float* meta,
                                         const int64_t* row_off, const uint8_t* row_bits,
                                         int64_t n_rows, int32_t F, float* out, int64_t ldo,
                                         gnn_stream_t stream) {
  GNN_REQUIRE(n_rows >= 0, "gnn_dequant_unpack: n_rows < 0");
  GNN_REQUIRE(F >= 1, "gnn_dequant_unpack: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_dequant_unpack: F=%d > %d", F, kMaxF);
  if (n_rows == 0) return GNN_OK;
  GNN_REQUIRE(packed && meta && row_off && row_bits && out, "gnn_dequant_unpack: NULL pointer");
  GNN_REQUIRE(ldo >= F && ldo % 4 == 0, "gnn_dequant_unpack: ldo must be >= F and a multiple of 4");
  GNN_REQUIRE(((uintptr_t)out & 15) == 0 && ((uintptr_t)packed & 15) == 0 && ((uintptr_t)meta & 7) == 0,
              "gnn_dequant_unpack: out and packed must be 16-byte aligned, meta 8-byte aligned");
  return launch_dequant_unpack(packed, reinterpret_cast<const float2*>(meta), row_off, row_bits,
                               n_rows, F, out, ldo, as_stream(stream));
}
