// Attention aggregator on the boundary-quantised path (SYLVIE guide, section
// 2: GAT weights the neighbour aggregation by attention coefficients; section
// 12: one head).  Single-head graph attention on the transformed rows:
//   Y = bf16(H) W,  s_l = Y a_l,  s_r = Y a_r,
//   e_vu = LeakyReLU(s_l[v] + s_r[u]) (slope 0.2), alpha_v. = softmax(e_v.),
//   H' = act(sum_u alpha_vu Y_u).
// A remote source is known to the receiving partition only by its dequantised
// message Y~_u, so its score is a_r . Y~_u.  The backward message of a boundary
// copy is its gradient: the fixed-order halo partial sum_v alpha_vu dZ_v plus
// the score term a_r * sum_v g_vu (g the gradient at the pre-activation score),
// quantised like the forward messages; the owner adds it to dY_u.
//
// The aggregations run through the row kernels of spmm.cu with the attention
// as entry weights; this file holds the scores, the edge softmax, the SDDMM of
// the backward and the small reductions around them.
#include <cuda_runtime.h>
#include <math.h>

#include "device.cuh"
#include "gemm.h"
#include "internal.h"
#include "kernels.h"

namespace gnn {
namespace {

constexpr float kSlope = 0.2f;
constexpr int kBlock = 256;

// SDDMM launch shape: threads per block, resident blocks asked of the
// register allocator, and entries gathered per round by 2-chunk lanes.
#ifndef GNN_GAT_SD_BLOCK
#define GNN_GAT_SD_BLOCK 64
#endif
#ifndef GNN_GAT_SD_MINB
#define GNN_GAT_SD_MINB 16
#endif
#ifndef GNN_GAT_SD_U2
#define GNN_GAT_SD_U2 4
#endif

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ int64_t warp_id() {
  return ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
}

// Element j of a packed message row (width b, meta (mn, scale)), as the
// receiver dequantises it.
__device__ __forceinline__ float dequant_elem(const uint8_t* __restrict__ row, int b, float mn,
                                              float scale, int j) {
  if (b == 32) return __ldg(reinterpret_cast<const float*>(row) + j);
  const uint32_t bitpos = (uint32_t)(j * b);
  const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(row) + (bitpos >> 5));
  const uint32_t code = (w >> (bitpos & 31u)) & ((1u << b) - 1u);
  return __fadd_rn(__fmul_rn(scale, (float)code), mn);
}

// ---------------------------------------------------------------- index maps
// tpos[k] for a local entry k of row u reading v: the position of row v's
// local entry reading u (local entries keep ascending ids); -1 for remote.
__global__ void gat_tpos_kernel(int n, const int64_t* __restrict__ rowptr,
                                const int32_t* __restrict__ cr, const int32_t* __restrict__ lc,
                                int64_t* __restrict__ tpos) {
  const int64_t u = warp_id();
  if (u >= n) return;
  const int lane = threadIdx.x & 31;
  const int64_t beg = rowptr[u], end = rowptr[u + 1];
  for (int64_t k = beg + lane; k < end; k += 32) {
    const int32_t v = cr[k];
    int64_t at = -1;
    if (v >= 0) {
      const int64_t end_v = rowptr[v] + (lc ? lc[v] : rowptr[v + 1] - rowptr[v]);
      int64_t lo = rowptr[v], hi = end_v;
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (cr[mid] < (int32_t)u) lo = mid + 1;
        else hi = mid;
      }
      if (lo < end_v && cr[lo] == (int32_t)u) at = lo;  // else the pattern is not symmetric
    }
    tpos[k] = at;
  }
}

// spos[j] for slot-CSR entry j (slot s, row v): the position of row v's remote
// entry reading slot s (a row's remote entries hold ascending slots).
__global__ void gat_spos_kernel(int64_t S, const int64_t* __restrict__ rowptr,
                                const int32_t* __restrict__ cr, const int32_t* __restrict__ lc,
                                const int64_t* __restrict__ srp, const int32_t* __restrict__ scol,
                                int64_t* __restrict__ spos) {
  const int64_t s = warp_id();
  if (s >= S) return;
  const int lane = threadIdx.x & 31;
  for (int64_t j = srp[s] + lane; j < srp[s + 1]; j += 32) {
    const int v = scol[j];
    const int64_t end_v = rowptr[v + 1];
    int64_t lo = rowptr[v] + lc[v], hi = end_v;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if ((int64_t)~cr[mid] < s) lo = mid + 1;
      else hi = mid;
    }
    spos[j] = (lo < end_v && (int64_t)~cr[lo] == s) ? lo : -1;
  }
}

// ---------------------------------------------------------------- forward
__global__ void gat_node_scores_kernel(int n, const float* __restrict__ Y, int64_t ldy, int F,
                                       const float* __restrict__ a_l, const float* __restrict__ a_r,
                                       float* __restrict__ s_l, float* __restrict__ s_r) {
  const int64_t v = warp_id();
  if (v >= n) return;
  const int lane = threadIdx.x & 31;
  float pl = 0.f, pr = 0.f;
  for (int j = lane; j < F; j += 32) {
    const float y = __ldg(Y + v * ldy + j);
    pl = fmaf(y, __ldg(a_l + j), pl);
    pr = fmaf(y, __ldg(a_r + j), pr);
  }
  pl = warp_sum(pl);
  pr = warp_sum(pr);
  if (lane == 0) {
    s_l[v] = pl;
    s_r[v] = pr;
  }
}

__global__ void gat_slot_scores_kernel(int64_t S, const uint8_t* __restrict__ packed,
                                       const float2* __restrict__ meta,
                                       const int64_t* __restrict__ off,
                                       const uint8_t* __restrict__ bits, int F,
                                       const float* __restrict__ a_r, float* __restrict__ s_slot) {
  const int64_t s = warp_id();
  if (s >= S) return;
  const int lane = threadIdx.x & 31;
  const int b = __ldg(bits + s);
  const float2 m = __ldg(meta + s);
  const uint8_t* row = packed + __ldg(off + s);
  float pr = 0.f;
  for (int j = lane; j < F; j += 32) pr = fmaf(dequant_elem(row, b, m.x, m.y, j), __ldg(a_r + j), pr);
  pr = warp_sum(pr);
  if (lane == 0) s_slot[s] = pr;
}

__device__ __forceinline__ float pre_score(float sl, int32_t c, const float* __restrict__ s_r,
                                           const float* __restrict__ s_slot) {
  return sl + (c >= 0 ? __ldg(s_r + c) : __ldg(s_slot + ~c));
}

__device__ __forceinline__ float lrelu(float x) { return x > 0.f ? x : kSlope * x; }

// alpha[k] = exp(e_k - max) / sum over the row, a group of G lanes per row:
// e is formed once (kept in alpha), then exponentiated and summed, then
// divided.  Each lane touches only its own entries.  Rows longer than
// long_len are left to gat_softmax_long_kernel.
template <int G>
__global__ void gat_softmax_kernel(int n, const int64_t* __restrict__ rowptr,
                                   const int32_t* __restrict__ cr, const float* __restrict__ s_l,
                                   const float* __restrict__ s_r, const float* __restrict__ s_slot,
                                   float* __restrict__ alpha, int64_t long_len) {
  const int64_t v = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / G;
  if (v >= n) return;  // uniform across the group
  const int gl = threadIdx.x & (G - 1);
  const uint32_t gmask = group_mask(G, threadIdx.x & 31);
  const int64_t beg = rowptr[v], end = rowptr[v + 1];
  if (long_len > 0 && end - beg > long_len) return;
  const float sl = s_l[v];
  float m = -INFINITY;
  for (int64_t k = beg + gl; k < end; k += G) {
    const float e = lrelu(pre_score(sl, cr[k], s_r, s_slot));
    alpha[k] = e;
    m = fmaxf(m, e);
  }
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(gmask, m, o));
  float sum = 0.f;
  for (int64_t k = beg + gl; k < end; k += G) {
    const float w = expf(alpha[k] - m);
    alpha[k] = w;
    sum += w;
  }
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(gmask, sum, o);
  for (int64_t k = beg + gl; k < end; k += G) alpha[k] = alpha[k] / sum;
}

// The same for the long rows (the split plan's list), one block per row.
__global__ void __launch_bounds__(kBlock) gat_softmax_long_kernel(
    int n_long, const int32_t* __restrict__ long_rows, const int64_t* __restrict__ rowptr,
    const int32_t* __restrict__ cr, const float* __restrict__ s_l, const float* __restrict__ s_r,
    const float* __restrict__ s_slot, float* __restrict__ alpha) {
  __shared__ float red[kBlock / 32];
  __shared__ float bcast;
  if ((int)blockIdx.x >= n_long) return;
  const int v = long_rows[blockIdx.x];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t beg = rowptr[v], end = rowptr[v + 1];
  const float sl = s_l[v];
  float m = -INFINITY;
  for (int64_t k = beg + threadIdx.x; k < end; k += blockDim.x) {
    const float e = lrelu(pre_score(sl, cr[k], s_r, s_slot));
    alpha[k] = e;
    m = fmaxf(m, e);
  }
  m = warp_max(m);
  if (lane == 0) red[wid] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = red[0];
    for (int q = 1; q < kBlock / 32; ++q) t = fmaxf(t, red[q]);
    bcast = t;
  }
  __syncthreads();
  m = bcast;
  float sum = 0.f;
  for (int64_t k = beg + threadIdx.x; k < end; k += blockDim.x) {
    const float w = expf(alpha[k] - m);
    alpha[k] = w;
    sum += w;
  }
  sum = warp_sum(sum);
  __syncthreads();
  if (lane == 0) red[wid] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int q = 0; q < kBlock / 32; ++q) t += red[q];
    bcast = t;
  }
  __syncthreads();
  sum = bcast;
  for (int64_t k = beg + threadIdx.x; k < end; k += blockDim.x) alpha[k] = alpha[k] / sum;
}

// ---------------------------------------------------------------- backward
// Sums of U values across the warp, one per group of 32/U lanes: d[i] of all
// lanes is reduced, and lane L returns the sum for i = (L >> (5 - log2 U)) &
// (U - 1).  A reduce-scatter: each halving step keeps half of the values and
// adds the partner's other half (U - 1 shuffles in all), then the remaining
// lanes of a group add up (5 - log2 U shuffles).
template <int U>
__device__ __forceinline__ float reduce_scatter(float (&d)[U], int lane) {
  constexpr int P = U == 1 ? 0 : U == 2 ? 1 : U == 4 ? 2 : U == 8 ? 3 : U == 16 ? 4 : 5;
  static_assert((1 << P) == U, "U must be a power of two up to 32");
#pragma unroll
  for (int st = 0; st < P; ++st) {
    const int o = 16 >> st;
    const int h = U >> (st + 1);
    const bool hi = (lane >> (4 - st)) & 1;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float keep = hi ? d[i + h] : d[i];
      const float send = hi ? d[i] : d[i + h];
      d[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float v = d[0];
#pragma unroll
  for (int o = 16 >> P; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct Units {  // rows, or pieces of the split plan first
  int n;
  int64_t n_pieces;
  int T;
  const int32_t* piece_row;
  const int64_t* piece_beg;
};

// dalpha_k = dZ_v . x_k for the entries of one unit (a row, or a piece of a
// long row), written to g[k]; cpart[unit] = sum_k alpha_k dalpha_k.  A whole
// row then finishes in place: g_k = alpha_k (dalpha_k - c_v) LeakyReLU'(pre_k)
// and ds_l[v] = sum_k g_k.  Each group of 32 lanes holds dZ_v in registers and
// gathers U entries' rows at a time.
template <int CPL, int U>
__global__ void __launch_bounds__(GNN_GAT_SD_BLOCK, GNN_GAT_SD_MINB) gat_sddmm_kernel(
    Units un, const int64_t* __restrict__ rowptr, const int32_t* __restrict__ cr,
    const float* __restrict__ alpha, const float* __restrict__ Y, int64_t ldy, int F,
    const float* __restrict__ dZ, int64_t ldz, const uint8_t* __restrict__ packed,
    const float2* __restrict__ meta, const int64_t* __restrict__ off,
    const uint8_t* __restrict__ bits, const float* __restrict__ s_l,
    const float* __restrict__ s_r, const float* __restrict__ s_slot, float* __restrict__ g,
    float* __restrict__ cpart, float* __restrict__ ds_l) {
  const int64_t unit = warp_id();
  const int lane = threadIdx.x & 31;
  if (unit >= un.n_pieces + un.n) return;
  const bool piece = unit < un.n_pieces;
  int64_t row, beg, end;
  if (piece) {
    row = un.piece_row[unit];
    beg = un.piece_beg[unit];
    end = min(beg + (int64_t)un.T, rowptr[row + 1]);
  } else {
    row = unit - un.n_pieces;
    beg = rowptr[row];
    end = rowptr[row + 1];
    if (un.T > 0 && end - beg > un.T) return;  // its pieces cover it
  }
  const int nch = (F + 3) >> 2;
  const float4* Y4 = reinterpret_cast<const float4*>(Y);
  const int64_t ldy4 = ldy >> 2;
  float4 z[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = lane + 32 * i;
    z[i] = c < nch ? __ldg(reinterpret_cast<const float4*>(dZ + row * ldz) + c)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float c_acc = 0.f;
  for (int64_t base = beg; base < end; base += 32) {
    const int64_t e = base + lane;
    int32_t cc = 0;
    float a = 0.f;
    int sb = 0;
    uint32_t so16 = 0;
    float2 sm = make_float2(0.f, 0.f);
    if (e < end) {
      cc = cr[e];
      a = alpha[e];
      if (cc < 0) {
        const int s = ~cc;
        sb = __ldg(bits + s);
        so16 = (uint32_t)(__ldg(off + s) >> 4);
        sm = __ldg(meta + s);
      }
    }
    const int cnt = (int)min((int64_t)32, end - base);
    constexpr int GP = 32 / U;  // lanes that end up holding one entry's sum
    const uint32_t rmask = __ballot_sync(0xffffffffu, e < end && cc < 0);  // remote entries
    const uint32_t raw = __ballot_sync(0xffffffffu, e < end && cc < 0 && sb == 32);
    for (int k = 0; k < cnt; k += U) {
      float d[U];
      const int lim = cnt - k;
      const uint32_t vmask = lim >= U ? (1u << U) - 1u : (1u << lim) - 1u;  // the round's entries
      if (((rmask >> k) & vmask) == vmask && ((raw >> k) & vmask) == 0u) {
        // all entries remote and packed: each chunk's 32-bit word for every
        // entry is loaded before any is decoded
        uint32_t wd[U][CPL];
        float mnk[U], sck[U];
        int bk[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int src = k + u < cnt ? k + u : k;
          bk[u] = __shfl_sync(0xffffffffu, sb, src);
          const uint32_t ok = __shfl_sync(0xffffffffu, so16, src);
          mnk[u] = __shfl_sync(0xffffffffu, sm.x, src);
          sck[u] = __shfl_sync(0xffffffffu, sm.y, src);
          const uint32_t* row = reinterpret_cast<const uint32_t*>(packed + ((size_t)ok << 4));
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            wd[u][i] = c < nch ? __ldg(row + (((uint32_t)c * (uint32_t)bk[u]) >> 3)) : 0u;
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int b = bk[u];
          const uint32_t m = (1u << b) - 1u;
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            if (c < nch) {
              const uint32_t bits4 = wd[u][i] >> (((uint32_t)c * (uint32_t)b * 4u) & 31u);
              acc = fmaf(z[i].x, __fadd_rn(__fmul_rn(sck[u], (float)(bits4 & m)), mnk[u]), acc);
              acc = fmaf(z[i].y, __fadd_rn(__fmul_rn(sck[u], (float)((bits4 >> b) & m)), mnk[u]), acc);
              acc = fmaf(z[i].z, __fadd_rn(__fmul_rn(sck[u], (float)((bits4 >> (2 * b)) & m)), mnk[u]), acc);
              acc = fmaf(z[i].w, __fadd_rn(__fmul_rn(sck[u], (float)((bits4 >> (3 * b)) & m)), mnk[u]), acc);
            }
          }
          d[u] = acc;
        }
      } else if (((rmask >> k) & ((1u << U) - 1u)) == 0u) {
        // all U entries local: their rows' loads go out together
        float4 x[U][CPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int ck = __shfl_sync(0xffffffffu, cc, k + u < cnt ? k + u : k);
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            x[u][i] = c < nch ? __ldg(Y4 + (int64_t)ck * ldy4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            acc = fmaf(z[i].x, x[u][i].x, acc);
            acc = fmaf(z[i].y, x[u][i].y, acc);
            acc = fmaf(z[i].z, x[u][i].z, acc);
            acc = fmaf(z[i].w, x[u][i].w, acc);
          }
          d[u] = acc;
        }
      } else {  // local and remote entries mixed: one entry at a time
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int src = k + u < cnt ? k + u : k;
          const int32_t ck = __shfl_sync(0xffffffffu, cc, src);
          int bk = 0;
          uint32_t ok = 0;
          float mnk = 0.f, sck = 0.f;
          if (ck < 0) {  // uniform across the warp
            bk = __shfl_sync(0xffffffffu, sb, src);
            ok = __shfl_sync(0xffffffffu, so16, src);
            mnk = __shfl_sync(0xffffffffu, sm.x, src);
            sck = __shfl_sync(0xffffffffu, sm.y, src);
          }
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            if (c < nch) {
              const float4 x = ck >= 0 ? __ldg(Y4 + (int64_t)ck * ldy4 + c)
                                       : dequant_chunk(packed + ((size_t)ok << 4), bk, mnk, sck, c);
              acc = fmaf(z[i].x, x.x, acc);
              acc = fmaf(z[i].y, x.y, acc);
              acc = fmaf(z[i].z, x.z, acc);
              acc = fmaf(z[i].w, x.w, acc);
            }
          }
          d[u] = acc;
        }
      }
      const float t = reduce_scatter<U>(d, lane);
      const int idx = lane / GP;
      const float ae = __shfl_sync(0xffffffffu, a, k + idx);
      if (lane % GP == 0 && k + idx < cnt) {
        g[base + k + idx] = t;
        c_acc = fmaf(ae, t, c_acc);
      }
    }
  }
  c_acc = warp_sum(c_acc);
  if (piece) {
    if (lane == 0) cpart[unit] = c_acc;
    return;
  }
  __syncwarp();
  const float sl = s_l[row];
  float dsl = 0.f;
  for (int64_t k = beg + lane; k < end; k += 32) {
    const float pre = pre_score(sl, cr[k], s_r, s_slot);
    const float gk = alpha[k] * (g[k] - c_acc) * (pre > 0.f ? 1.f : kSlope);
    g[k] = gk;
    dsl += gk;
  }
  dsl = warp_sum(dsl);
  if (lane == 0) ds_l[row] = dsl;
}

// Long rows: c_v from their pieces (piece order), then g and ds_l as above;
// one block per row.
__global__ void __launch_bounds__(kBlock) gat_long_rows_kernel(int n_long, const int32_t* __restrict__ long_rows,
                                     const int64_t* __restrict__ piece_ptr,
                                     const float* __restrict__ cpart,
                                     const int64_t* __restrict__ rowptr,
                                     const int32_t* __restrict__ cr,
                                     const float* __restrict__ alpha,
                                     const float* __restrict__ s_l, const float* __restrict__ s_r,
                                     const float* __restrict__ s_slot, float* __restrict__ g,
                                     float* __restrict__ ds_l) {
  __shared__ float red[kBlock / 32];
  const int64_t i = blockIdx.x;
  if (i >= n_long) return;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int row = long_rows[i];
  float c = 0.f;
  for (int64_t p = piece_ptr[i]; p < piece_ptr[i + 1]; ++p) c += cpart[p];
  const float sl = s_l[row];
  float dsl = 0.f;
  for (int64_t k = rowptr[row] + threadIdx.x; k < rowptr[row + 1]; k += blockDim.x) {
    const float pre = pre_score(sl, cr[k], s_r, s_slot);
    const float gk = alpha[k] * (g[k] - c) * (pre > 0.f ? 1.f : kSlope);
    g[k] = gk;
    dsl += gk;
  }
  dsl = warp_sum(dsl);
  if (lane == 0) red[wid] = dsl;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int q = 0; q < kBlock / 32; ++q) t += red[q];
    ds_l[row] = t;
  }
}

// Attention and score gradients at the transposed positions: alpha_t / g_t
// (col_remap order, local entries; 0 for remote ones) and slot_alpha / slot_g
// (slot-CSR order).
__global__ void gat_gather_kernel(int64_t nnz, const int64_t* __restrict__ tpos, int64_t nc,
                                  const int64_t* __restrict__ spos,
                                  const float* __restrict__ alpha, const float* __restrict__ g,
                                  float* __restrict__ alpha_t, float* __restrict__ g_t,
                                  float* __restrict__ slot_alpha, float* __restrict__ slot_g) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < nnz) {
    const int64_t p = tpos[i];
    alpha_t[i] = p >= 0 ? alpha[p] : 0.f;
    g_t[i] = p >= 0 ? g[p] : 0.f;
  } else if (i - nnz < nc) {
    const int64_t p = spos[i - nnz];
    slot_alpha[i - nnz] = p >= 0 ? alpha[p] : 0.f;
    slot_g[i - nnz] = p >= 0 ? g[p] : 0.f;
  }
}

// ds_r[u] = sum of g over u's local transposed entries (one warp per row).
__global__ void gat_row_sum_kernel(int n, const int64_t* __restrict__ rowptr,
                                   const int32_t* __restrict__ lc, const float* __restrict__ g_t,
                                   float* __restrict__ ds_r) {
  const int64_t u = warp_id();
  if (u >= n) return;
  const int lane = threadIdx.x & 31;
  const int64_t beg = rowptr[u], end = lc ? beg + lc[u] : rowptr[u + 1];
  float s = 0.f;
  for (int64_t k = beg + lane; k < end; k += 32) s += g_t[k];
  s = warp_sum(s);
  if (lane == 0) ds_r[u] = s;
}

// r[s] = sum of g over slot s's entries, in entry order (fp32, from +0): the
// score term of the backward message.
__global__ void gat_slot_sum_kernel(int64_t S, const int64_t* __restrict__ srp,
                                    const float* __restrict__ slot_g, float* __restrict__ r) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= S) return;
  float acc = 0.f;
  for (int64_t j = srp[s]; j < srp[s + 1]; ++j) acc = __fadd_rn(acc, slot_g[j]);
  r[s] = acc;
}

// dY[u] += ds_r[u] a_r + ds_l[u] a_l: a block of (F/4) x rows threads, one
// float4 of a row each.
__global__ void gat_score_terms_kernel(int64_t n, int F, const float* __restrict__ ds_r,
                                       const float* __restrict__ ds_l,
                                       const float* __restrict__ a_r,
                                       const float* __restrict__ a_l, float* __restrict__ dY,
                                       int64_t ldy) {
  const int c = threadIdx.x;  // chunk; F is a multiple of 16
  const int64_t u = (int64_t)blockIdx.x * blockDim.y + threadIdx.y;
  if (u >= n || 4 * c >= F) return;
  const float r = ds_r[u], l = ds_l[u];
  const float4 ar = __ldg(reinterpret_cast<const float4*>(a_r) + c);
  const float4 al = __ldg(reinterpret_cast<const float4*>(a_l) + c);
  float4* p = reinterpret_cast<float4*>(dY + u * ldy) + c;
  float4 v = *p;
  v.x += fmaf(r, ar.x, l * al.x);
  v.y += fmaf(r, ar.y, l * al.y);
  v.z += fmaf(r, ar.z, l * al.z);
  v.w += fmaf(r, ar.w, l * al.w);
  *p = v;
}

// part_l[b] / part_r[b] = the column sums of rows [b*rpb, (b+1)*rpb) of X
// weighted by w_l and by w_r, in one pass over X.  Thread t covers chunk
// t % nch of the rows t / nch + k*rp (rp = 256 / nch row phases), four rows
// in flight; the row phases are then added in order through shared memory.
__global__ void __launch_bounds__(256) gat_colsum2_kernel(int64_t rows, int64_t rpb, int F,
                                                          const float* __restrict__ w_l,
                                                          const float* __restrict__ w_r,
                                                          const float* __restrict__ X, int64_t ldx,
                                                          float* __restrict__ part_l,
                                                          float* __restrict__ part_r) {
  __shared__ float4 sl[256], sr[256];
  const int nch = (F + 3) >> 2;
  const int rp = 256 / nch;  // F <= 1024: at least one row phase
  const int t = threadIdx.x;
  const int c = t % nch, ph = t / nch;
  const int64_t r0 = (int64_t)blockIdx.x * rpb;
  const int64_t r1 = min(rows, r0 + rpb);
  float4 al = make_float4(0.f, 0.f, 0.f, 0.f), ar = al;
  if (ph < rp) {
    int64_t r = r0 + ph;
    for (; r + 3 * rp < r1; r += 4 * rp) {
      float4 x[4];
      float a[4], b[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t rr = r + q * rp;
        x[q] = __ldg(reinterpret_cast<const float4*>(X + rr * ldx) + c);
        a[q] = __ldg(w_l + rr);
        b[q] = __ldg(w_r + rr);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        fma4(al, a[q], x[q]);
        fma4(ar, b[q], x[q]);
      }
    }
    for (; r < r1; r += rp) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(X + r * ldx) + c);
      fma4(al, __ldg(w_l + r), x);
      fma4(ar, __ldg(w_r + r), x);
    }
  }
  sl[t] = al;
  sr[t] = ar;
  __syncthreads();
  if (t < nch) {
    float4 sa = sl[t], sb = sr[t];
    for (int q = 1; q < rp; ++q) {
      add4(sa, sl[q * nch + t]);
      add4(sb, sr[q * nch + t]);
    }
    float* pl = part_l + (int64_t)blockIdx.x * F + 4 * t;
    float* pr = part_r + (int64_t)blockIdx.x * F + 4 * t;
    const float va[4] = {sa.x, sa.y, sa.z, sa.w}, vb[4] = {sb.x, sb.y, sb.z, sb.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (4 * t + e < F) {
        pl[e] = va[e];
        pr[e] = vb[e];
      }
  }
}

// part[b] = sum over slots [b*rpb, (b+1)*rpb) of w[s] times slot s's
// dequantised message (the receiver's values).  Thread t covers chunk
// t % nch (four elements from one 32-bit word) of the slots t / nch + k*rp,
// four slots in flight; row phases are added in order through shared memory.
__global__ void __launch_bounds__(256) gat_colsum_slots_kernel(int64_t S, int64_t rpb, int F,
                                                               const float* __restrict__ w,
                                                               const uint8_t* __restrict__ packed,
                                                               const float2* __restrict__ meta,
                                                               const int64_t* __restrict__ off,
                                                               const uint8_t* __restrict__ bits,
                                                               float* __restrict__ part) {
  __shared__ float4 sh[256];
  const int nch = (F + 3) >> 2;
  const int rp = 256 / nch;
  const int t = threadIdx.x;
  const int c = t % nch, ph = t / nch;
  const int64_t r0 = (int64_t)blockIdx.x * rpb;
  const int64_t r1 = min(S, r0 + rpb);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (ph < rp) {
    int64_t s = r0 + ph;
    for (; s + 3 * rp < r1; s += 4 * rp) {
      float4 x[4];
      float a[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t ss = s + q * rp;
        const float2 m = __ldg(meta + ss);
        x[q] = dequant_chunk(packed + __ldg(off + ss), __ldg(bits + ss), m.x, m.y, c);
        a[q] = __ldg(w + ss);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) fma4(acc, a[q], x[q]);
    }
    for (; s < r1; s += rp) {
      const float2 m = __ldg(meta + s);
      fma4(acc, __ldg(w + s), dequant_chunk(packed + __ldg(off + s), __ldg(bits + s), m.x, m.y, c));
    }
  }
  sh[t] = acc;
  __syncthreads();
  if (t < nch) {
    float4 sa = sh[t];
    for (int q = 1; q < rp; ++q) add4(sa, sh[q * nch + t]);
    float* pp = part + (int64_t)blockIdx.x * F + 4 * t;
    const float va[4] = {sa.x, sa.y, sa.z, sa.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (4 * t + e < F) pp[e] = va[e];
  }
}

__global__ void gat_colsum_reduce_kernel(int nparts, int F, const float* __restrict__ part,
                                         float* __restrict__ out) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= F) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int b = 0;
  for (; b + 8 <= nparts; b += 8) {
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] += part[(int64_t)(b + q) * F + j];
  }
  for (int q = 0; b < nparts; ++b, ++q) acc[q] += part[(int64_t)b * F + j];
  float sum = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) sum += acc[q];
  out[j] = sum;
}

unsigned warps_grid(int64_t warps) { return (unsigned)((warps * 32 + kBlock - 1) / kBlock); }
unsigned threads_grid(int64_t t) { return (unsigned)((t + kBlock - 1) / kBlock); }

constexpr int kColsumBlocks = 608;  // 4 per SM

int64_t colsum_rows_per_block(int64_t rows) {
  return rows > 0 ? (rows + kColsumBlocks - 1) / kColsumBlocks : 1;
}
int colsum_blocks(int64_t rows) {
  return rows > 0 ? (int)((rows + colsum_rows_per_block(rows) - 1) / colsum_rows_per_block(rows)) : 0;
}

int64_t round_up64(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct GatWs {
  float *s_l, *s_r, *s_slot, *g, *cpart, *alpha_t, *g_t, *slot_alpha, *slot_g, *ds_l, *ds_r, *r;
  float *dz, *dy, *part_l, *part_r, *spmm;
  void* dense;
  size_t dense_bytes;
  size_t bytes;
};

GatWs gat_ws_layout(void* base, size_t cap, const gnn_csr& csr, const gnn_boundary* bnd, int F_in,
                    int F_out, bool* ok) {
  Arena ar(base, cap);
  GatWs w{};
  const size_t n = (size_t)csr.n, nnz = (size_t)csr.nnz;
  const size_t S = bnd ? (size_t)bnd->n_slots : 0, nc = bnd ? (size_t)bnd->nnz_cut : 0;
  const size_t ldy = (size_t)round_up64(F_out, 4);
  w.s_l = ar.take<float>(n);
  w.s_r = ar.take<float>(n);
  w.s_slot = ar.take<float>(S > 0 ? S : 1);
  w.g = ar.take<float>(nnz > 0 ? nnz : 1);
  w.cpart = ar.take<float>(csr.n_pieces > 0 ? (size_t)csr.n_pieces : 1);
  w.alpha_t = ar.take<float>(nnz > 0 ? nnz : 1);
  w.g_t = ar.take<float>(nnz > 0 ? nnz : 1);
  w.slot_alpha = ar.take<float>(nc > 0 ? nc : 1);
  w.slot_g = ar.take<float>(nc > 0 ? nc : 1);
  w.ds_l = ar.take<float>(n);
  w.ds_r = ar.take<float>(n);
  w.r = ar.take<float>(S > 0 ? S : 1);
  w.dz = ar.take<float>(n * ldy);
  w.dy = ar.take<float>(n * ldy);
  w.part_l = ar.take<float>((size_t)kColsumBlocks * F_out);
  w.part_r = ar.take<float>((size_t)2 * kColsumBlocks * F_out);
  const size_t sp = spmm_workspace_bytes(csr, F_out);
  w.spmm = sp ? reinterpret_cast<float*>(ar.take_bytes(sp)) : nullptr;
  size_t db = 0;
  gnn_dense_workspace(csr.n, F_in, F_out, &db);
  w.dense_bytes = db;
  w.dense = ar.take_bytes(db);
  w.bytes = ar.used;
  *ok = ar.ok();
  return w;
}

gnn_status check_gat(const gnn_csr* csr, const gnn_boundary* bnd, int F_in, int F_out,
                     const char* who, bool offsets = true) {
  if (!csr || csr->n < 1 || !csr->rowptr || (csr->nnz > 0 && !csr->col))
    return fail(GNN_ERR_INVALID_ARG, "%s: invalid csr", who);
  if (F_in < 1 || F_in > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "%s: F_in=%d", who, F_in);
  if (F_out < 16 || F_out % 16 || F_out > 256)
    return fail(GNN_ERR_UNSUPPORTED, "%s: F_out must be a multiple of 16 in [16, 256]", who);
  if (bnd && (bnd->n != csr->n || (offsets && bnd->F != F_out) || !bnd->col_remap || !bnd->local_cnt))
    return fail(GNN_ERR_INVALID_ARG, "%s: boundary must match csr with offsets for F_out", who);
  return GNN_OK;
}

}  // namespace
}  // namespace gnn

using namespace gnn;

extern "C" gnn_status gnn_gat_index(const gnn_csr* csr, const gnn_boundary* bnd, int64_t* tpos,
                                    int64_t* spos, gnn_stream_t stream) {
  GNN_REQUIRE(csr && csr->n >= 1 && csr->rowptr && tpos, "gnn_gat_index: bad arguments");
  GNN_REQUIRE(csr->symmetric || csr->val_t, "gnn_gat_index: needs a symmetrised pattern");
  GNN_REQUIRE(!bnd || ((bnd->nnz_cut == 0 || spos) && bnd->col_remap && bnd->local_cnt &&
                       bnd->slot_rowptr && (bnd->nnz_cut == 0 || bnd->slot_col)),
              "gnn_gat_index: boundary arrays or spos missing");
  cudaStream_t st = as_stream(stream);
  const int32_t* cr = bnd ? bnd->col_remap : csr->col;
  const int32_t* lc = bnd ? bnd->local_cnt : nullptr;
  gat_tpos_kernel<<<warps_grid(csr->n), kBlock, 0, st>>>(csr->n, csr->rowptr, cr, lc, tpos);
  GNN_CHECK_LAUNCH();
  if (bnd && bnd->n_slots > 0) {
    gat_spos_kernel<<<warps_grid(bnd->n_slots), kBlock, 0, st>>>(
        bnd->n_slots, csr->rowptr, cr, lc, bnd->slot_rowptr, bnd->slot_col, spos);
    GNN_CHECK_LAUNCH();
  }
  return GNN_OK;
}

extern "C" gnn_status gnn_gat_workspace(const gnn_csr* csr, const gnn_boundary* bnd, int32_t F_in,
                                        int32_t F_out, size_t* ws_bytes) {
  gnn_status s = check_gat(csr, bnd, F_in, F_out, "gnn_gat_workspace", false);
  if (s != GNN_OK) return s;
  GNN_REQUIRE(ws_bytes, "gnn_gat_workspace: NULL ws_bytes");
  bool ok;
  *ws_bytes = gat_ws_layout(nullptr, 0, *csr, bnd, F_in, F_out, &ok).bytes;
  return GNN_OK;
}

extern "C" gnn_status gnn_gat_layer_fwd(const gnn_csr* csr, const gnn_boundary* bnd,
                                        const float* H_in, int64_t ldh, int32_t F_in,
                                        const uint16_t* W, int32_t F_out, const float* a_l,
                                        const float* a_r, int32_t relu, uint32_t seed,
                                        uint8_t* packed, float* meta, uint16_t* Hb, int64_t ldhb,
                                        float* Y, int64_t ldy, float* alpha, float* H_out,
                                        int64_t ldo, void* ws, size_t ws_bytes,
                                        gnn_stream_t stream) {
  gnn_status s = check_gat(csr, bnd, F_in, F_out, "gnn_gat_layer_fwd");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(H_in && W && a_l && a_r && Hb && Y && alpha && H_out, "gnn_gat_layer_fwd: NULL pointer");
  GNN_REQUIRE(((uintptr_t)a_l & 15) == 0 && ((uintptr_t)a_r & 15) == 0,
              "gnn_gat_layer_fwd: a_l and a_r must be 16-byte aligned");
  GNN_REQUIRE(ldh >= F_in && ldh % 4 == 0 && ((uintptr_t)H_in & 15) == 0, "gnn_gat_layer_fwd: bad H_in");
  GNN_REQUIRE(ldhb >= round_up64(F_in, 16) && ldhb % 8 == 0 && ((uintptr_t)Hb & 15) == 0,
              "gnn_gat_layer_fwd: bad Hb");
  GNN_REQUIRE(ldy >= round_up64(F_out, 4) && ldy % 4 == 0 && ((uintptr_t)Y & 15) == 0,
              "gnn_gat_layer_fwd: bad Y");
  GNN_REQUIRE(ldo >= F_out && ldo % 4 == 0 && ((uintptr_t)H_out & 15) == 0, "gnn_gat_layer_fwd: bad H_out");
  const bool slots = bnd && bnd->n_slots > 0;
  GNN_REQUIRE(!slots || (packed && meta && ((uintptr_t)packed & 15) == 0 && ((uintptr_t)meta & 7) == 0 &&
                         bnd->slot_node && bnd->slot_bits && bnd->slot_off),
              "gnn_gat_layer_fwd: message buffers required with a boundary");
  bool ok;
  GatWs w = gat_ws_layout(ws, ws_bytes, *csr, bnd, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_gat_layer_fwd: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  cudaStream_t st = as_stream(stream);
  const int n = csr->n;
  // Y = bf16(H) W
  if ((s = launch_cast_bf16(n, F_in, H_in, ldh, Hb, ldhb, st)) != GNN_OK) return s;
  s = gnn_dense_fwd(Hb, ldhb, n, F_in, W, F_out, 0, Y, ldy, w.dense, w.dense_bytes, stream);
  if (s != GNN_OK) return s;
  gat_node_scores_kernel<<<warps_grid(n), kBlock, 0, st>>>(n, Y, ldy, F_out, a_l, a_r, w.s_l, w.s_r);
  GNN_CHECK_LAUNCH();
  if (slots) {
    s = launch_quant_pack_owned(*bnd, Y, ldy, F_out, seed, packed, reinterpret_cast<float2*>(meta),
                                st);
    if (s != GNN_OK) return s;
    gat_slot_scores_kernel<<<warps_grid(bnd->n_slots), kBlock, 0, st>>>(
        bnd->n_slots, packed, reinterpret_cast<const float2*>(meta), bnd->slot_off, bnd->slot_bits,
        F_out, a_r, w.s_slot);
    GNN_CHECK_LAUNCH();
  }
  const int32_t* cr = bnd ? bnd->col_remap : csr->col;
  // ordinary rows a warp each; the split plan's long rows a block each
  const bool plan = csr->split_len > 0 && csr->n_long > 0;
  gat_softmax_kernel<32><<<warps_grid(n), kBlock, 0, st>>>(n, csr->rowptr, cr, w.s_l, w.s_r,
                                                           w.s_slot, alpha, plan ? csr->split_len : 0);
  GNN_CHECK_LAUNCH();
  if (plan) {
    gat_softmax_long_kernel<<<(unsigned)csr->n_long, kBlock, 0, st>>>(
        csr->n_long, csr->long_rows, csr->rowptr, cr, w.s_l, w.s_r, w.s_slot, alpha);
  }
  GNN_CHECK_LAUNCH();
  return launch_spmm_fwd_w(*csr, bnd, alpha, Y, ldy, F_out, packed,
                           reinterpret_cast<const float2*>(meta), H_out, ldo, w.spmm, relu, st);
}

extern "C" gnn_status gnn_gat_layer_bwd(
    const gnn_csr* csr, const gnn_boundary* bnd, const int64_t* tpos, const int64_t* spos,
    const float* dH_out, int64_t ldg, const float* H_out, int64_t ldo, int32_t relu,
    const uint16_t* Hb, int64_t ldhb, const float* Y, int64_t ldy, const float* alpha,
    const uint8_t* packed_fwd, const float* meta_fwd, const uint16_t* W, const float* a_l,
    const float* a_r, int32_t F_in, int32_t F_out, uint32_t seed, uint8_t* packed_ws,
    float* meta_ws, float* dW, float* da_l, float* da_r, float* dH_in, int64_t ldh, float* g_out,
    void* ws, size_t ws_bytes, gnn_stream_t stream) {
  gnn_status s = check_gat(csr, bnd, F_in, F_out, "gnn_gat_layer_bwd");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(tpos && dH_out && Hb && Y && alpha && W && a_l && a_r && dW && da_l && da_r,
              "gnn_gat_layer_bwd: NULL pointer");
  GNN_REQUIRE(ldg >= F_out && ldg % 4 == 0 && ((uintptr_t)dH_out & 15) == 0, "gnn_gat_layer_bwd: bad dH_out");
  GNN_REQUIRE(((uintptr_t)a_l & 15) == 0 && ((uintptr_t)a_r & 15) == 0,
              "gnn_gat_layer_bwd: a_l and a_r must be 16-byte aligned");
  GNN_REQUIRE(!relu || (H_out && ldo >= F_out && ldo % 4 == 0 && ((uintptr_t)H_out & 15) == 0),
              "gnn_gat_layer_bwd: relu needs H_out");
  GNN_REQUIRE(ldy >= round_up64(F_out, 4) && ldy % 4 == 0 && ((uintptr_t)Y & 15) == 0,
              "gnn_gat_layer_bwd: bad Y");
  GNN_REQUIRE(!dH_in || (ldh >= round_up64(F_in, 4) && ldh % 4 == 0 && ((uintptr_t)dH_in & 15) == 0),
              "gnn_gat_layer_bwd: bad dH_in");
  const bool slots = bnd && bnd->n_slots > 0;
  GNN_REQUIRE(!slots || (spos && packed_fwd && meta_fwd && packed_ws && meta_ws &&
                         ((uintptr_t)packed_ws & 15) == 0 && ((uintptr_t)meta_ws & 7) == 0 &&
                         bnd->slot_rowptr && bnd->slot_col && bnd->own_ptr && bnd->own_slot),
              "gnn_gat_layer_bwd: message buffers, spos and slot arrays required with a boundary");
  bool ok;
  GatWs w = gat_ws_layout(ws, ws_bytes, *csr, bnd, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_gat_layer_bwd: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  cudaStream_t st = as_stream(stream);
  const int n = csr->n;
  const int64_t ldy4 = round_up64(F_out, 4);
  const int32_t* cr = bnd ? bnd->col_remap : csr->col;
  const float2* mf = reinterpret_cast<const float2*>(meta_fwd);
  const int64_t S = slots ? bnd->n_slots : 0;
  float* g = g_out ? g_out : w.g;
  // dZ
  const float* dz = dH_out;
  int64_t ldz = ldg;
  if (relu) {
    if ((s = launch_relu_mask_f32(n, F_out, dH_out, ldg, H_out, ldo, w.dz, ldy4, st)) != GNN_OK) return s;
    dz = w.dz;
    ldz = ldy4;
  }
  // scores again (from Y and the forward messages)
  gat_node_scores_kernel<<<warps_grid(n), kBlock, 0, st>>>(n, Y, ldy, F_out, a_l, a_r, w.s_l, w.s_r);
  GNN_CHECK_LAUNCH();
  if (slots) {
    gat_slot_scores_kernel<<<warps_grid(S), kBlock, 0, st>>>(S, packed_fwd, mf, bnd->slot_off,
                                                            bnd->slot_bits, F_out, a_r, w.s_slot);
    GNN_CHECK_LAUNCH();
  }
  // SDDMM and the softmax backward
  Units un{n, 0, 0, nullptr, nullptr};
  if (csr->split_len > 0 && csr->n_pieces > 0) {
    un.n_pieces = csr->n_pieces;
    un.T = csr->split_len;
    un.piece_row = csr->piece_row;
    un.piece_beg = csr->piece_beg;
  }
  const int nch = (F_out + 3) / 4;
  const unsigned gs =
      (unsigned)(((un.n_pieces + n) * 32 + GNN_GAT_SD_BLOCK - 1) / GNN_GAT_SD_BLOCK);
  const uint8_t* pk = slots ? packed_fwd : nullptr;
  const int64_t* so = slots ? bnd->slot_off : nullptr;
  const uint8_t* sbits = slots ? bnd->slot_bits : nullptr;
  if (nch <= 32)
    gat_sddmm_kernel<1, 8><<<gs, GNN_GAT_SD_BLOCK, 0, st>>>(un, csr->rowptr, cr, alpha, Y, ldy, F_out, dz, ldz, pk,
                                                  mf, so, sbits, w.s_l, w.s_r, w.s_slot, g, w.cpart,
                                                  w.ds_l);
  else
    gat_sddmm_kernel<2, GNN_GAT_SD_U2><<<gs, GNN_GAT_SD_BLOCK, 0, st>>>(un, csr->rowptr, cr, alpha, Y, ldy, F_out, dz, ldz, pk,
                                                  mf, so, sbits, w.s_l, w.s_r, w.s_slot, g, w.cpart,
                                                  w.ds_l);
  GNN_CHECK_LAUNCH();
  if (un.n_pieces > 0) {
    gat_long_rows_kernel<<<(unsigned)csr->n_long, kBlock, 0, st>>>(
        csr->n_long, csr->long_rows, csr->piece_ptr, w.cpart, csr->rowptr, cr, alpha, w.s_l, w.s_r,
        w.s_slot, g, w.ds_l);
    GNN_CHECK_LAUNCH();
  }
  // transposed attention and score gradients; ds_r and the slots' score sums
  const int64_t nc = slots ? bnd->nnz_cut : 0;
  gat_gather_kernel<<<threads_grid(csr->nnz + nc), kBlock, 0, st>>>(
      csr->nnz, tpos, nc, spos, alpha, g, w.alpha_t, w.g_t, w.slot_alpha, w.slot_g);
  GNN_CHECK_LAUNCH();
  gat_row_sum_kernel<<<warps_grid(n), kBlock, 0, st>>>(n, csr->rowptr, bnd ? bnd->local_cnt : nullptr,
                                                       w.g_t, w.ds_r);
  GNN_CHECK_LAUNCH();
  if (slots) {
    gat_slot_sum_kernel<<<threads_grid(S), kBlock, 0, st>>>(S, bnd->slot_rowptr, w.slot_g, w.r);
    GNN_CHECK_LAUNCH();
    // backward messages: fixed-order halo partial of dZ with the attention,
    // plus the score term, quantised and packed
    s = launch_halo_quant_pack_ex(*bnd, dz, ldz, F_out, seed, packed_ws,
                                  reinterpret_cast<float2*>(meta_ws), w.slot_alpha, w.r, a_r, st);
    if (s != GNN_OK) return s;
  }
  // dY = local transposed aggregation + owned messages, then the score terms
  s = launch_spmm_bwd_local_w(*csr, bnd, w.alpha_t, dz, ldz, F_out, packed_ws,
                              reinterpret_cast<const float2*>(meta_ws), w.dy, ldy4, w.spmm, st);
  if (s != GNN_OK) return s;
  {
    const dim3 blk(F_out / 4, kBlock / (F_out / 4));
    gat_score_terms_kernel<<<(unsigned)((n + blk.y - 1) / blk.y), blk, 0, st>>>(
        n, F_out, w.ds_r, w.ds_l, a_r, a_l, w.dy, ldy4);
  }
  GNN_CHECK_LAUNCH();
  // da_l = sum_v ds_l[v] Y_v;  da_r = sum_u ds_r[u] Y_u + sum_s r[s] Y~_s
  const int bn = colsum_blocks(n), bs = colsum_blocks(S);
  if (bn > 0) {
    gat_colsum2_kernel<<<bn, 256, 0, st>>>(n, colsum_rows_per_block(n), F_out, w.ds_l, w.ds_r, Y, ldy,
                                           w.part_l, w.part_r);
    GNN_CHECK_LAUNCH();
  }
  gat_colsum_reduce_kernel<<<1, 256, 0, st>>>(bn, F_out, w.part_l, da_l);
  GNN_CHECK_LAUNCH();
  if (bs > 0) {
    gat_colsum_slots_kernel<<<bs, 256, 0, st>>>(S, colsum_rows_per_block(S), F_out, w.r, packed_fwd, mf,
                                                bnd->slot_off, bnd->slot_bits,
                                                w.part_r + (int64_t)bn * F_out);
    GNN_CHECK_LAUNCH();
  }
  gat_colsum_reduce_kernel<<<1, 256, 0, st>>>(bn + bs, F_out, w.part_r, da_r);
  GNN_CHECK_LAUNCH();
  // dW = Hb^T bf16(dY), dH_in = bf16(dY) W^T
  return gnn_dense_bwd(Hb, ldhb, n, F_in, W, F_out, w.dy, ldy4, nullptr, 0, 0, dH_in,
                       dH_in ? ldh : 0, dW, w.dense, w.dense_bytes, stream);
}
