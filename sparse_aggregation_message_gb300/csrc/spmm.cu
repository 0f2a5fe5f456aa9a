// GCN aggregation kernels (SYLVIE guide sections 2, 3 and 11):
//   forward  M = A H, remote sources replaced by their dequantised messages;
//   backward halo partials of every slot (fixed fp32 order) fused with their
//            quantisation and packing, then dH = local A^T G + owned messages.
//
// One group of G lanes owns one output row (or one piece of a long row); lane
// g holds the float4 chunks c = g + i*G (i < CPL) of the row in registers, so
// every gathered source row is read with coalesced 16-byte loads.  A group
// walks its entries G at a time: the G lanes load G (col, val) pairs -- and,
// for remote entries, the slot's width, offset and meta -- in one coalesced
// step, then broadcast them with shuffles while all lanes gather U entries at
// a time (U loads in flight per lane and chunk).
//
// Load balance on power-law graphs: rows longer than the CSR's split_len are
// cut into pieces of split_len entries.  Pieces run as their own groups at
// the front of the grid and leave fp32 partial rows in the workspace; a fixup
// kernel adds a row's pieces in piece order (deterministic) and writes it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "device.cuh"
#include "internal.h"
#include "kernels.h"

namespace gnn {

enum SpmmMode { kPlain = 0, kFwdRemote = 1, kBwdOwned = 2 };

struct SlotMsgs {
  const uint8_t* packed;
  const float2* meta;
  const int64_t* off;
  const uint8_t* bits;
};

struct RowSplit {
  int T;  // split_len; 0 = no plan
  int n_long;
  int64_t n_pieces;
  const int32_t* long_rows;
  const int64_t* piece_ptr;
  const int32_t* piece_row;
  const int64_t* piece_beg;
};

// Prefetch hints for the rows a batch will gather: each lane asks L2 for the
// 128-byte lines of its own entry's byte range [lo, hi) as soon as the
// batch's entry data arrive, so the later rounds of the batch (which load
// only a few entries at a time) find their rows in L2 instead of waiting on
// HBM one round after another.  0: off; 1: L2; 2: L1.
#ifndef GNN_PF_REMOTE
#define GNN_PF_REMOTE 0
#endif
#ifndef GNN_PF_LOCAL
#define GNN_PF_LOCAL 0
#endif
#ifndef GNN_PF_HALO
#define GNN_PF_HALO 0
#endif

template <int LEVEL>
__device__ __forceinline__ void prefetch_lines(const void* base, uint32_t lo, uint32_t hi) {
  if (LEVEL == 0 || hi <= lo) return;
  const uintptr_t a0 = (reinterpret_cast<uintptr_t>(base) + lo) & ~uintptr_t(127);
  const uintptr_t a1 = reinterpret_cast<uintptr_t>(base) + hi;
  for (uintptr_t a = a0; a < a1; a += 128) {
    if (LEVEL == 1)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    else
      asm volatile("prefetch.global.L1 [%0];" ::"l"(a));
  }
}

// acc += sum over local entries [beg, end) of val * H[col].  The group covers
// chunks c0 + gl + i*G (i < CPL) below c_end.  One accumulator per chunk; U
// entries are gathered before they are added, so U*CPL 16-byte loads per lane
// are in flight.
template <int G, int CPL, int U>
__device__ __forceinline__ void gather_local(int64_t beg, int64_t end, const int32_t* __restrict__ col,
                                             const float* __restrict__ val,
                                             const float4* __restrict__ H4, int64_t ldh4, int c0,
                                             int c_end, int gl, uint32_t gmask, float4 (&acc)[CPL]) {
  for (int64_t base = beg; base < end; base += G) {
    const int64_t e = base + gl;
    int cc = 0;
    float w = 0.f;
    if (e < end) {
      cc = __ldg(col + e);
      w = __ldg(val + e);
      prefetch_lines<GNN_PF_LOCAL>(H4 + (int64_t)cc * ldh4, 16u * c0, 16u * c_end);
    }
    const int cnt = (int)min((int64_t)G, end - base);
    for (int k = 0; k < cnt; k += U) {
      float4 x[U][CPL];
      float wk[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool valid = k + u < cnt;
        const int src = valid ? k + u : k;
        wk[u] = valid ? __shfl_sync(gmask, w, src, G) : 0.f;
        const int ck = __shfl_sync(gmask, cc, src, G);
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = c0 + gl + i * G;
          x[u][i] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (valid && c < c_end) x[u][i] = __ldg(H4 + (int64_t)ck * ldh4 + c);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) fma4(acc[i], wk[u], x[u][i]);
      }
    }
  }
}

// acc += sum over remote entries [beg, end) (slot ~col) of val * the slot's
// dequantised message.  The G lanes load G entries' (val, slot width, offset,
// meta) in one coalesced step and broadcast them with shuffles; a round then
// loads, for UR entries, the one 32-bit word that holds each chunk's four
// codes (widths 1, 2, 4, 8 never straddle a word) before it dequantises and
// adds them in entry order -- one register per chunk in flight instead of
// four.  A round that meets a raw fp32 slot (width 32) reads float4 chunks.
// OWNED: entries [beg, end) of own_slot (slot ids, weight 1) instead: the
// messages a row owns, added in list order (w = 1 makes each fused
// multiply-add an exact add).
template <int G, int CPL, int UR, bool OWNED = false>
__device__ __forceinline__ void gather_remote(int64_t beg, int64_t end,
                                                    const int32_t* __restrict__ col,
                                                    const float* __restrict__ val, int c0,
                                                    int c_end, const SlotMsgs& msg, int gl,
                                                    uint32_t gmask, float4 (&acc)[CPL]) {
  for (int64_t base = beg; base < end; base += G) {
    const int64_t e = base + gl;
    float w = 0.f;
    int sb = 0;
    uint32_t so16 = 0;
    float2 sm = make_float2(0.f, 0.f);
    if (e < end) {
      const int s = OWNED ? __ldg(col + e) : ~__ldg(col + e);
      w = OWNED ? 1.f : __ldg(val + e);
      sb = __ldg(msg.bits + s);
      so16 = (uint32_t)(__ldg(msg.off + s) >> 4);
      sm = __ldg(msg.meta + s);
      // bytes of the row the group's chunks [c0, c_end) read
      const uint32_t lo = sb == 32 ? 16u * c0 : ((uint32_t)(4 * c0 * sb) >> 5) << 2;
      const uint32_t hi = sb == 32 ? 16u * c_end : (((uint32_t)(4 * c_end * sb) + 31u) >> 5) << 2;
      prefetch_lines<GNN_PF_REMOTE>(msg.packed + ((size_t)so16 << 4), lo, hi);
    }
    const int cnt = (int)min((int64_t)G, end - base);
    for (int k = 0; k < cnt; k += UR) {
      float wk[UR], mnk[UR], sck[UR];
      int bk[UR];
      uint32_t ok[UR];
      bool raw = false;
#pragma unroll
      for (int u = 0; u < UR; ++u) {
        const bool valid = k + u < cnt;
        const int src = valid ? k + u : k;
        wk[u] = valid ? __shfl_sync(gmask, w, src, G) : 0.f;
        bk[u] = __shfl_sync(gmask, sb, src, G);
        ok[u] = __shfl_sync(gmask, so16, src, G);
        mnk[u] = __shfl_sync(gmask, sm.x, src, G);
        sck[u] = __shfl_sync(gmask, sm.y, src, G);
        raw |= valid && bk[u] == 32;
      }
      if (raw) {
#pragma unroll
        for (int u = 0; u < UR; ++u) {
          if (k + u >= cnt) continue;
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = c0 + gl + i * G;
            if (c < c_end)
              fma4(acc[i], wk[u], dequant_chunk(msg.packed + ((size_t)ok[u] << 4), bk[u], mnk[u], sck[u], c));
          }
        }
        continue;
      }
      uint32_t wd[UR][CPL];
#pragma unroll
      for (int u = 0; u < UR; ++u) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = c0 + gl + i * G;
          wd[u][i] = 0u;
          if (k + u < cnt && c < c_end) {
            const uint32_t bitpos = (uint32_t)(4 * c * bk[u]);
            wd[u][i] = __ldg(reinterpret_cast<const uint32_t*>(msg.packed + ((size_t)ok[u] << 4)) +
                             (bitpos >> 5));
          }
        }
      }
#pragma unroll
      for (int u = 0; u < UR; ++u) {
        const int b = bk[u];
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = c0 + gl + i * G;
          const uint32_t bits4 = wd[u][i] >> ((uint32_t)(4 * c * b) & 31u);
          fma4(acc[i], wk[u], dequant4(bits4, b, mnk[u], sck[u]));
        }
      }
    }
  }
}

// The same sum with the round split in two phases: first the packed words of
// UR entries are requested (each entry's width and offset taken from its
// lane by shuffle), then each entry's weight, width and meta are taken again
// and its words decoded.  Only the words are held across the phase, so far
// more entries are in flight per lane than when every entry's five values
// are kept (latency of the random message reads is what bounds this loop
// when most sources are remote).
template <int G, int CPL, int UR, bool OWNED = false>
__device__ __forceinline__ void gather_remote_split(int64_t beg, int64_t end,
                                                    const int32_t* __restrict__ col,
                                                    const float* __restrict__ val, int c0,
                                                    int c_end, const SlotMsgs& msg, int gl,
                                                    uint32_t gmask, float4 (&acc)[CPL]) {
  for (int64_t base = beg; base < end; base += G) {
    const int64_t e = base + gl;
    float w = 0.f;
    int sb = 0;
    uint32_t so16 = 0;
    float2 sm = make_float2(0.f, 0.f);
    if (e < end) {
      const int s = OWNED ? __ldg(col + e) : ~__ldg(col + e);
      w = OWNED ? 1.f : __ldg(val + e);
      sb = __ldg(msg.bits + s);
      so16 = (uint32_t)(__ldg(msg.off + s) >> 4);
      sm = __ldg(msg.meta + s);
      const uint32_t lo = sb == 32 ? 16u * c0 : ((uint32_t)(4 * c0 * sb) >> 5) << 2;
      const uint32_t hi = sb == 32 ? 16u * c_end : (((uint32_t)(4 * c_end * sb) + 31u) >> 5) << 2;
      prefetch_lines<GNN_PF_REMOTE>(msg.packed + ((size_t)so16 << 4), lo, hi);
    }
    const int cnt = (int)min((int64_t)G, end - base);
    for (int k = 0; k < cnt; k += UR) {
      uint32_t wd[UR][CPL];
      bool raw = false;
#pragma unroll
      for (int u = 0; u < UR; ++u) {
        const bool valid = k + u < cnt;
        const int src = valid ? k + u : k;
        const int b = __shfl_sync(gmask, sb, src, G);
        const uint32_t o16 = __shfl_sync(gmask, so16, src, G);
        raw |= valid && b == 32;
        const uint32_t* rowp = reinterpret_cast<const uint32_t*>(msg.packed + ((size_t)o16 << 4));
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = c0 + gl + i * G;
          wd[u][i] = 0u;
          if (valid && c < c_end && b != 32) wd[u][i] = __ldg(rowp + ((uint32_t)(4 * c * b) >> 5));
        }
      }
#pragma unroll
      for (int u = 0; u < UR; ++u) {
        const bool valid = k + u < cnt;
        const int src = valid ? k + u : k;
        const float wk = valid ? __shfl_sync(gmask, w, src, G) : 0.f;
        const int b = __shfl_sync(gmask, sb, src, G);
        const float mn = __shfl_sync(gmask, sm.x, src, G);
        const float sc = __shfl_sync(gmask, sm.y, src, G);
        if (b == 32) continue;  // raw rows: below
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = c0 + gl + i * G;
          const uint32_t bits4 = wd[u][i] >> ((uint32_t)(4 * c * b) & 31u);
          fma4(acc[i], wk, dequant4(bits4, b, mn, sc));
        }
      }
      if (raw) {  // fp32 pass-through rows (width 32), read as float4 chunks
#pragma unroll
        for (int u = 0; u < UR; ++u) {
          const bool valid = k + u < cnt;
          const int src = valid ? k + u : k;
          const float wk = __shfl_sync(gmask, w, src, G);
          const int b = __shfl_sync(gmask, sb, src, G);
          const uint32_t o16 = __shfl_sync(gmask, so16, src, G);
          if (!valid || b != 32) continue;
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = c0 + gl + i * G;
            if (c < c_end) fma4(acc[i], wk, dequant_chunk(msg.packed + ((size_t)o16 << 4), 32, 0.f, 0.f, c));
          }
        }
      }
    }
  }
}

// The same sum with each batch's per-entry values -- (slot offset, weight,
// min, scale) and the width -- staged in shared memory instead of held in
// registers and broadcast by shuffles: a round then requests the packed words
// of UR entries (reading each entry's offset and width back with broadcast
// shared loads), and decodes them after all UR requests are in flight.  Only
// the words stay in registers across the round, so UR can be large.
// rec/recb: this warp's 32 records (index = lane).
template <int G, int CPL, int UR, bool OWNED = false>
__device__ __forceinline__ void gather_remote_smem(int64_t beg, int64_t end,
                                                   const int32_t* __restrict__ col,
                                                   const float* __restrict__ val, int c0,
                                                   int c_end, const SlotMsgs& msg, int gl,
                                                   uint32_t gmask, float4 (&acc)[CPL],
                                                   uint4* rec, int* recb) {
  const int lane = threadIdx.x & 31;
  const int g0 = lane & ~(G - 1);  // the group's first record
  for (int64_t base = beg; base < end; base += G) {
    const int64_t e = base + gl;
    if (e < end) {
      const int s = OWNED ? __ldg(col + e) : ~__ldg(col + e);
      const float w = OWNED ? 1.f : __ldg(val + e);
      const int sb = __ldg(msg.bits + s);
      const uint32_t so16 = (uint32_t)(__ldg(msg.off + s) >> 4);
      const float2 sm = __ldg(msg.meta + s);
      rec[lane] = make_uint4(so16, __float_as_uint(w), __float_as_uint(sm.x), __float_as_uint(sm.y));
      recb[lane] = sb;
    }
    __syncwarp(gmask);
    const int cnt = (int)min((int64_t)G, end - base);
    for (int k = 0; k < cnt; k += UR) {
      uint32_t wd[UR][CPL];
      int bk[UR];
      bool raw = false;
#pragma unroll
      for (int u = 0; u < UR; ++u) {
        const bool valid = k + u < cnt;
        const int idx = g0 + (valid ? k + u : k);
        const int b = recb[idx];
        bk[u] = b;
        raw |= valid && b == 32;
        const uint32_t* rowp =
            reinterpret_cast<const uint32_t*>(msg.packed + ((size_t)rec[idx].x << 4));
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = c0 + gl + i * G;
          wd[u][i] = 0u;
          if (valid && c < c_end && b != 32) wd[u][i] = __ldg(rowp + ((uint32_t)(4 * c * b) >> 5));
        }
      }
#pragma unroll
      for (int u = 0; u < UR; ++u) {
        const bool valid = k + u < cnt;
        const uint4 r = rec[g0 + (valid ? k + u : k)];
        const float wk = valid ? __uint_as_float(r.y) : 0.f;
        const int b = bk[u];
        if (b == 32) continue;  // raw rows: below
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = c0 + gl + i * G;
          const uint32_t bits4 = wd[u][i] >> ((uint32_t)(4 * c * b) & 31u);
          fma4(acc[i], wk, dequant4(bits4, b, __uint_as_float(r.z), __uint_as_float(r.w)));
        }
      }
      if (raw) {  // fp32 pass-through rows (width 32), read as float4 chunks
#pragma unroll
        for (int u = 0; u < UR; ++u) {
          if (k + u >= cnt || bk[u] != 32) continue;
          const uint4 r = rec[g0 + k + u];
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = c0 + gl + i * G;
            if (c < c_end)
              fma4(acc[i], __uint_as_float(r.y),
                   dequant_chunk(msg.packed + ((size_t)r.x << 4), 32, 0.f, 0.f, c));
          }
        }
      }
    }
    __syncwarp(gmask);  // every lane is done with this batch's records
  }
}

#ifndef GNN_REMOTE_SPLIT
#define GNN_REMOTE_SPLIT 0
#endif
#ifndef GNN_REMOTE_SMEM
#define GNN_REMOTE_SMEM 1
#endif
#ifndef GNN_REMOTE_SMEM_UR
#define GNN_REMOTE_SMEM_UR 4
#endif
#ifndef GNN_REMOTE_SPLIT_UR
#define GNN_REMOTE_SPLIT_UR 8
#endif

// acc += dequantised messages of the slots row r owns (backward), in the
// owner list's order; the slots' widths, offsets and meta are loaded for G
// slots at once and their words UR slots at a time.
template <int G, int CPL, int UR>
__device__ __forceinline__ void add_owned(int64_t r, const int64_t* __restrict__ own_ptr,
                                          const int32_t* __restrict__ own_slot,
                                          const SlotMsgs& msg, int c0, int c_end, int gl,
                                          uint32_t gmask, float4 (&acc)[CPL]) {
  gather_remote<G, CPL, UR, true>(__ldg(own_ptr + r), __ldg(own_ptr + r + 1), own_slot, nullptr, c0,
                                  c_end, msg, gl, gmask, acc);
}

// Writes the group's chunks of row r: fp32 chunks below nch, bf16 chunks
// below nch_b (zeros past F), both limited to the group's slice [c0, c1);
// with relu, max(x, 0) of each; with hmask, x where hmask's row is > 0, else 0.
template <int G, int CPL>
__device__ __forceinline__ void store_row(int64_t r, float4 (&acc)[CPL], int F, int nch,
                                          int nch_b, int c0, int c1, int gl,
                                          float* __restrict__ M, int64_t ldm,
                                          __nv_bfloat16* __restrict__ Mb, int64_t ldmb, int relu,
                                          const float* __restrict__ hmask, int64_t ldhm) {
  if (hmask) {  // keep x where the mask row is positive (the next ReLU's gate)
    const float4* mrow = reinterpret_cast<const float4*>(hmask + r * ldhm);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = c0 + gl + i * G;
      if (c < c1 && c < nch) {
        const float4 h = __ldg(mrow + c);
        if (!(h.x > 0.f)) acc[i].x = 0.f;
        if (!(h.y > 0.f)) acc[i].y = 0.f;
        if (!(h.z > 0.f)) acc[i].z = 0.f;
        if (!(h.w > 0.f)) acc[i].w = 0.f;
      }
    }
  }
  if (relu) {
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      acc[i].x = fmaxf(acc[i].x, 0.f);
      acc[i].y = fmaxf(acc[i].y, 0.f);
      acc[i].z = fmaxf(acc[i].z, 0.f);
      acc[i].w = fmaxf(acc[i].w, 0.f);
    }
  }
  if (M) {
    float* mrow = M + r * ldm;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = c0 + gl + i * G;
      if (c < c1 && c < nch) store_chunk_f32(mrow, c, F, acc[i]);
    }
  }
  if (Mb) {
    __nv_bfloat16* brow = Mb + r * ldmb;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = c0 + gl + i * G;
      if (c < c1 && c < nch_b)
        store_chunk_bf16(brow, c, F, c < nch ? acc[i] : make_float4(0.f, 0.f, 0.f, 0.f));
    }
  }
}

// Feature slices: wide rows are cut into ns slices of cs chunks, each owned
// by its own group (the slices re-read the row's (col, val) pairs).
struct Slices {
  int ns;
  int cs;
};

// Threads per block of the rows kernel: one warp with messages (forward
// with remote rows, backward), two without.  Small blocks free their slot as
// soon as their few rows finish, which keeps more warps resident when row
// lengths vary.
template <int MODE>
constexpr int rows_block() {
  return MODE == 0 ? 64 : 32;
}
// Entries gathered per round: local (U, by chunks per lane; the forward with
// remote rows has its own) and remote (UR) entries, each measured best on the
// power-law workloads; the 3-chunk layout gathers 2 local entries.
#ifndef GNN_U1
#define GNN_U1 6
#endif
#ifndef GNN_U2
#define GNN_U2 3
#endif
#ifndef GNN_U1_FWD
#define GNN_U1_FWD 6
#endif
#ifndef GNN_U2_FWD
#define GNN_U2_FWD 4
#endif
#ifndef GNN_UR1
#define GNN_UR1 3
#endif
#ifndef GNN_UR2
#define GNN_UR2 2
#endif
#ifndef GNN_UR3
#define GNN_UR3 2
#endif
// Widest feature slice a group covers (in 16-byte chunks).
#ifndef GNN_SLICE_CHUNKS
#define GNN_SLICE_CHUNKS 96
#endif

// Rows per group for the kernels with messages when a row is one slice: a
// group walks RK consecutive rows, their bounds read at once (lane k: row k),
// so no row waits on its own bounds.
#ifndef GNN_ROWS_MULTI
#define GNN_ROWS_MULTI 8
#endif

template <int G, int CPL, int MODE, int U, int UR, int RK>
__device__ __forceinline__ void rows_group(
    int64_t grp, int n, const int64_t* __restrict__ rowptr, const int32_t* __restrict__ col,
    const float* __restrict__ val, const int32_t* __restrict__ local_cnt,
    const float4* __restrict__ H4, int64_t ldh4, int F, int nch, const SlotMsgs& msg,
    const int64_t* __restrict__ own_ptr, const int32_t* __restrict__ own_slot, const RowSplit& sp,
    int c0, int c1, float* __restrict__ M, int64_t ldm, __nv_bfloat16* __restrict__ Mb,
    int64_t ldmb, int nch_b, int relu, const float* __restrict__ hmask, int64_t ldhm, int gl,
    uint32_t gmask, uint4* rec, int* recb) {
  const int64_t row0 = grp * RK;
  if (row0 >= n) return;  // uniform across the group
  long long my_b = 0, my_e = 0;
  int my_lc = 0;
  auto load_bounds = [&](int64_t first) {
    my_b = my_e = 0;
    my_lc = 0;
    if (first + gl < n && first + gl < row0 + RK) {
      my_b = __ldg(rowptr + first + gl);
      my_e = __ldg(rowptr + first + gl + 1);
      my_lc = __ldg(local_cnt + first + gl);
    }
  };
  load_bounds(row0);
#pragma unroll 1
  for (int j = 0; j < RK; ++j) {
    const int64_t row = row0 + j;
    if (row >= n) break;  // uniform
    const int jj = j % G;
    if (j > 0 && jj == 0) load_bounds(row);
    const int64_t beg = __shfl_sync(gmask, my_b, jj, G), end = __shfl_sync(gmask, my_e, jj, G);
    const int lc = __shfl_sync(gmask, my_lc, jj, G);
    if (sp.T > 0 && end - beg > sp.T) continue;  // a long row: its pieces cover it
    float4 acc[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t mid = beg + lc;
    gather_local<G, CPL, U>(beg, min(end, mid), col, val, H4, ldh4, c0, min(c1, nch), gl, gmask, acc);
    if constexpr (MODE == kFwdRemote) {
      if (GNN_REMOTE_SMEM)
        gather_remote_smem<G, CPL, GNN_REMOTE_SMEM_UR>(max(beg, mid), end, col, val, c0,
                                                       min(c1, nch), msg, gl, gmask, acc, rec, recb);
      else
        gather_remote<G, CPL, UR>(max(beg, mid), end, col, val, c0, min(c1, nch), msg, gl, gmask,
                                  acc);
    }
    if constexpr (MODE == kBwdOwned)
      add_owned<G, CPL, UR>(row, own_ptr, own_slot, msg, c0, min(c1, nch), gl, gmask, acc);
    store_row<G, CPL>(row, acc, F, nch, nch_b, c0, c1, gl, M, ldm, Mb, ldmb, relu, hmask, ldhm);
  }
}

// 1024 resident threads per SM (64 registers each); the 3-chunk forward with
// remote rows needs up to 80 and keeps 768.
template <int G, int CPL, int MODE, int U, int UR>
__global__ void __launch_bounds__(rows_block<MODE>(), ((MODE == 1 && CPL == 3) ? 768 : 1024) / rows_block<MODE>())
    spmm_rows_kernel(
    int n, const int64_t* __restrict__ rowptr, const int32_t* __restrict__ col,
    const float* __restrict__ val, const int32_t* __restrict__ local_cnt,
    const float* __restrict__ H, int64_t ldh, int F,
    SlotMsgs msg, const int64_t* __restrict__ own_ptr, const int32_t* __restrict__ own_slot,
    RowSplit sp, Slices sl, float* __restrict__ partial, float* __restrict__ M, int64_t ldm,
    __nv_bfloat16* __restrict__ Mb, int64_t ldmb, int nch_b, int relu,
    const float* __restrict__ hmask, int64_t ldhm) {
  const int lane = threadIdx.x & 31;
  const int gl = lane & (G - 1);
  const int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / G;
  const uint32_t gmask = group_mask(G, lane);
  const int nch = (F + 3) >> 2;
  const float4* H4 = reinterpret_cast<const float4*>(H);
  const int64_t ldh4 = ldh >> 2;
  const int slice = (int)(g % sl.ns);
  const int64_t unit = g / sl.ns;
  const int c0 = slice * sl.cs, c1 = c0 + sl.cs;
  float4 acc[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);

  __shared__ uint4 srec[(MODE == kFwdRemote && GNN_REMOTE_SMEM) ? rows_block<MODE>() : 1];
  __shared__ int sbits[(MODE == kFwdRemote && GNN_REMOTE_SMEM) ? rows_block<MODE>() : 1];
  uint4* rec = srec + ((MODE == kFwdRemote && GNN_REMOTE_SMEM) ? (threadIdx.x & ~31) : 0);
  int* recb = sbits + ((MODE == kFwdRemote && GNN_REMOTE_SMEM) ? (threadIdx.x & ~31) : 0);
  if constexpr (MODE != kPlain && GNN_ROWS_MULTI > 1) {
    if (sl.ns == 1 && unit >= sp.n_pieces) {
      rows_group<G, CPL, MODE, U, UR, GNN_ROWS_MULTI>(
          unit - sp.n_pieces, n, rowptr, col, val, local_cnt, H4, ldh4, F, nch, msg, own_ptr,
          own_slot, sp, c0, c1, M, ldm, Mb, ldmb, nch_b, relu, hmask, ldhm, gl, gmask, rec, recb);
      return;
    }
  }
  const bool piece = unit < sp.n_pieces;
  int64_t row, beg, end;
  if (piece) {  // a piece of a long row -> partial row `unit`
    row = __ldg(sp.piece_row + unit);
    beg = __ldg(sp.piece_beg + unit);
    end = min(beg + (int64_t)sp.T, __ldg(rowptr + row + 1));
  } else {
    row = unit - sp.n_pieces;
    if (row >= n) return;  // uniform across the group
    beg = __ldg(rowptr + row);
    end = __ldg(rowptr + row + 1);
    if (sp.T > 0 && end - beg > sp.T) return;  // a long row: its pieces cover it
  }
  // local entries lead each row, remote slots follow
  const int64_t mid =
      MODE == kPlain ? end : (piece ? __ldg(rowptr + row) : beg) + __ldg(local_cnt + row);
  gather_local<G, CPL, U>(beg, min(end, mid), col, val, H4, ldh4, c0, min(c1, nch), gl, gmask, acc);
  if constexpr (MODE == kFwdRemote) {
    if (GNN_REMOTE_SMEM) {
      gather_remote_smem<G, CPL, GNN_REMOTE_SMEM_UR>(max(beg, mid), end, col, val, c0,
                                                     min(c1, nch), msg, gl, gmask, acc, rec, recb);
    } else if (GNN_REMOTE_SPLIT)
      gather_remote_split<G, CPL, GNN_REMOTE_SPLIT_UR>(max(beg, mid), end, col, val, c0,
                                                        min(c1, nch), msg, gl, gmask, acc);
    else
      gather_remote<G, CPL, UR>(max(beg, mid), end, col, val, c0, min(c1, nch), msg, gl, gmask, acc);
  }
  if (piece) {
    float4* prow = reinterpret_cast<float4*>(partial) + unit * nch;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = c0 + gl + i * G;
      if (c < c1 && c < nch) prow[c] = acc[i];
    }
    return;
  }
  if (MODE == kBwdOwned)
    add_owned<G, CPL, UR>(row, own_ptr, own_slot, msg, c0, min(c1, nch), gl, gmask, acc);
  store_row<G, CPL>(row, acc, F, nch, nch_b, c0, c1, gl, M, ldm, Mb, ldmb, relu, hmask, ldhm);
}

// Long rows: sum of their pieces' partial rows, 16 pieces at a time and then
// the block sums, always in piece order (deterministic, short fp32 chains).
template <int G, int CPL, int MODE>
__global__ void __launch_bounds__(256) spmm_fixup_kernel(
    RowSplit sp, Slices sl, const float* __restrict__ partial, int F, SlotMsgs msg,
    const int64_t* __restrict__ own_ptr, const int32_t* __restrict__ own_slot,
    float* __restrict__ M, int64_t ldm, __nv_bfloat16* __restrict__ Mb, int64_t ldmb,
    int nch_b, int relu, const float* __restrict__ hmask, int64_t ldhm) {
  const int lane = threadIdx.x & 31;
  const int gl = lane & (G - 1);
  const int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / G;
  const int64_t i = g / sl.ns;
  if (i >= sp.n_long) return;
  const int slice = (int)(g % sl.ns);
  const int c0 = slice * sl.cs, c1 = c0 + sl.cs;
  const int nch = (F + 3) >> 2;
  const int64_t row = __ldg(sp.long_rows + i);
  const int64_t pb = __ldg(sp.piece_ptr + i), pe = __ldg(sp.piece_ptr + i + 1);
  float4 acc[CPL];
#pragma unroll
  for (int k = 0; k < CPL; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* P4 = reinterpret_cast<const float4*>(partial);
  for (int64_t p0 = pb; p0 < pe; p0 += 16) {
    float4 blk[CPL];
#pragma unroll
    for (int k = 0; k < CPL; ++k) blk[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t p1 = min(pe, p0 + 16);
    for (int64_t p = p0; p < p1; ++p) {
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        const int c = c0 + gl + k * G;
        if (c < c1 && c < nch) add4(blk[k], __ldg(P4 + p * nch + c));
      }
    }
#pragma unroll
    for (int k = 0; k < CPL; ++k) add4(acc[k], blk[k]);
  }
  if (MODE == kBwdOwned)
    add_owned<G, CPL, 2>(row, own_ptr, own_slot, msg, c0, min(c1, nch), gl, group_mask(G, lane), acc);
  store_row<G, CPL>(row, acc, F, nch, nch_b, c0, c1, gl, M, ldm, Mb, ldmb, relu, hmask, ldhm);
}

// P = fl(P + fl(r * a_r[j])) for the elements j of chunk c below F (the score
// term of an attention layer's backward message).
__device__ __forceinline__ void add_score_term(float4& p, float r, const float* __restrict__ a_r,
                                               int c, int F) {
  const int j = 4 * c;
  if (j < F) p.x = __fadd_rn(p.x, __fmul_rn(r, __ldg(a_r + j)));
  if (j + 1 < F) p.y = __fadd_rn(p.y, __fmul_rn(r, __ldg(a_r + j + 1)));
  if (j + 2 < F) p.z = __fadd_rn(p.z, __fmul_rn(r, __ldg(a_r + j + 2)));
  if (j + 3 < F) p.w = __fadd_rn(p.w, __fmul_rn(r, __ldg(a_r + j + 3)));
}

// Backward messages: halo partial of slot s over its entries in ascending v,
// every product and sum rounded to fp32 (start +0), then quantised and packed
// in registers with row key s.
//
// Blocks [0, n_long) each take one long slot: the block's threads load E
// entry rows at a time into shared memory (all loads in flight together),
// then thread t adds chunk t of those rows in entry order.  The remaining
// blocks give every ordinary slot a group of G lanes that loads U entries
// ahead of their adds.  Both keep each element's additions in entry order,
// so the result is the same as one sequential loop.  Rows of up to three
// chunks per lane keep 64 registers (four blocks per SM: the loads of a slot
// are few and short, so more slots in flight pay more than deeper unrolling).
// Ordinary slots, HK > 1: each group of G lanes walks HK consecutive slots of
// the visiting order.  The bounds of all HK slots are read at once, and the
// first batch of the next slot's entries is requested before the current
// slot is quantised, so only the row gathers are left on each slot's chain
// of dependent loads.  Every slot's sum keeps its fixed order.
template <int G, int CPL, int U, int HK>
__device__ __forceinline__ void halo_group_slots(
    int64_t block, const int64_t* __restrict__ srp, const int32_t* __restrict__ scol,
    const float* __restrict__ sval, const float4* __restrict__ G4, int64_t ldg4, int F,
    const uint8_t* __restrict__ slot_bits, const int64_t* __restrict__ slot_off, uint32_t seed,
    uint8_t* __restrict__ packed, float2* __restrict__ meta, int long_len,
    const float* __restrict__ score_r, const float* __restrict__ a_r,
    const int32_t* __restrict__ order, int64_t s_lo, int64_t s_hi) {
  const int lane = threadIdx.x & 31;
  const int gl = lane & (G - 1);
  const uint32_t gmask = group_mask(G, lane);
  const int nch = (F + 3) >> 2;
  const int64_t count = s_hi - s_lo;
  // HK consecutive slots of the visiting order: their first entries are
  // neighbouring gradient rows, which the group then re-reads from cache
  const int64_t i0 = ((block * blockDim.x + threadIdx.x) / G) * HK;
  if (i0 >= count) return;  // uniform across the group
  // the slots' ids and bounds, G slots at a time (lane k holds slot k of the chunk)
  long long my_s = 0, my_b = 0, my_e = 0;
  auto load_bounds = [&](int64_t j0) {
    my_s = my_b = my_e = 0;
    const int64_t i = i0 + j0 + gl;
    if (i < count && j0 + gl < HK) {
      my_s = order ? (long long)__ldg(order + i) : (long long)(s_lo + i);
      my_b = __ldg(srp + my_s);
      my_e = __ldg(srp + my_s + 1);
    }
  };
  load_bounds(0);
  // the first entry batch of the group's first slot
  int v_next = 0;
  float w_next = 0.f;
  {
    const int64_t b0 = __shfl_sync(gmask, my_b, 0, G), e0 = __shfl_sync(gmask, my_e, 0, G);
    if (b0 + gl < e0) {
      v_next = __ldg(scol + b0 + gl);
      w_next = __ldg(sval + b0 + gl);
    }
  }
#pragma unroll 1
  for (int j = 0; j < HK; ++j) {
    if (i0 + j >= count) break;  // uniform
    const int jj = j % G;  // the slot's lane in the current chunk
    const int64_t s = __shfl_sync(gmask, my_s, jj, G);
    const int64_t beg = __shfl_sync(gmask, my_b, jj, G), end = __shfl_sync(gmask, my_e, jj, G);
    const bool skip = long_len > 0 && end - beg > long_len;  // summed by a long-slot block
    float4 acc[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!skip) {
      for (int64_t base = beg; base < end; base += G) {
        const int64_t e = base + gl;
        int v = v_next;
        float w = w_next;
        if (base != beg) {
          v = 0;
          w = 0.f;
          if (e < end) {
            v = __ldg(scol + e);
            w = __ldg(sval + e);
          }
        }
        const int cnt = (int)min((int64_t)G, end - base);
        for (int k = 0; k < cnt; k += U) {
          float4 x[U][CPL];
          float wk[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int src = (k + u < cnt) ? k + u : k;
            const int vk = __shfl_sync(gmask, v, src, G);
            wk[u] = __shfl_sync(gmask, w, src, G);
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
              const int c = gl + i * G;
              if (c < nch) x[u][i] = __ldg(G4 + (int64_t)vk * ldg4 + c);
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (k + u < cnt) {
#pragma unroll
              for (int i = 0; i < CPL; ++i) {
                if (gl + i * G < nch) mul_add4(acc[i], wk[u], x[u][i]);
              }
            }
          }
        }
      }
    }
    // the next slot's first entry batch, requested before this slot is quantised
    v_next = 0;
    w_next = 0.f;
    if (j + 1 < HK && i0 + j + 1 < count) {
      if (jj + 1 == G) load_bounds(j + 1);  // the next chunk of G slots
      const int jn = (j + 1) % G;
      const int64_t nb = __shfl_sync(gmask, my_b, jn, G), ne = __shfl_sync(gmask, my_e, jn, G);
      if (nb + gl < ne) {
        v_next = __ldg(scol + nb + gl);
        w_next = __ldg(sval + nb + gl);
      }
    }
    if (skip) continue;
    if (score_r) {
      const float r = __ldg(score_r + s);
#pragma unroll
      for (int i = 0; i < CPL; ++i)
        if (gl + i * G < nch) add_score_term(acc[i], r, a_r, gl + i * G, F);
    }
    quantize_pack_row<G, CPL>(acc, F, __ldg(slot_bits + s), row_key(seed, (uint32_t)s),
                              packed + __ldg(slot_off + s), meta + s, gl, gmask);
  }
}

#ifndef GNN_HALO_MULTI
#define GNN_HALO_MULTI 64
#endif
// Slots per group, measured at F = 256 (two chunks per lane): 64 on the
// R-MAT graph's 37.9M slots (67.4 -> 46.7 ms), 16 on the DC-SBM-shaped
// graphs' 0.8M-3.4M slots (Yelp-shaped 0.71 -> 0.69 ms, products-shaped
// 3.14 -> 2.58 ms; 64 there is slower than one).  The other row layouts
// measured slower with more than one slot per group and keep one.
constexpr int halo_slots_per_group(int G, int CPL, bool many_slots) {
  return (G == 32 && CPL == 2) ? (many_slots ? GNN_HALO_MULTI : 16) : 1;
}
constexpr int64_t kManySlots = int64_t(1) << 24;

#ifndef GNN_RING_SPLIT
#define GNN_RING_SPLIT 1
#endif
template <int G, int CPL>
__device__ __forceinline__ void quantize_pack_row_sel(const float4 (&v)[CPL], int F, int b,
                                                      uint32_t key, uint8_t* __restrict__ out,
                                                      float2* __restrict__ meta, int gl,
                                                      uint32_t gmask) {
  if (GNN_RING_SPLIT)
    quantize_pack_row_split<G, CPL>(v, F, b, key, out, meta, gl, gmask);
  else
    quantize_pack_row<G, CPL>(v, F, b, key, out, meta, gl, gmask);
}

// One long slot summed by a whole block: the block's threads load E entry
// rows at a time into shared memory (all loads in flight together), then
// thread t adds chunk t of those rows in entry order; warp 0 quantises.
template <int CPLQ>
__device__ __forceinline__ void halo_long_block(
    int blk, const int64_t* __restrict__ srp, const int32_t* __restrict__ scol,
    const float* __restrict__ sval, const float4* __restrict__ G4, int64_t ldg4, int F,
    const uint8_t* __restrict__ slot_bits, const int64_t* __restrict__ slot_off, uint32_t seed,
    uint8_t* __restrict__ packed, float2* __restrict__ meta, const int32_t* __restrict__ long_slots,
    int E, const float* __restrict__ score_r, const float* __restrict__ a_r, int64_t s_lo,
    int64_t s_hi, float4* tile) {
  __shared__ int sv[32];
  __shared__ float sw[32];
  const int lane = threadIdx.x & 31;
  const int nch = (F + 3) >> 2;
  const int64_t s = __ldg(long_slots + blk);
  if (s < s_lo || s >= s_hi) return;  // outside the requested slot range (block-uniform)
  const int64_t beg = __ldg(srp + s), end = __ldg(srp + s + 1);
  const int t = threadIdx.x;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t base = beg; base < end; base += E) {
    const int cnt = (int)min((int64_t)E, end - base);
    if (t < cnt) {
      sv[t] = __ldg(scol + base + t);
      sw[t] = __ldg(sval + base + t);
    }
    __syncthreads();
    for (int idx = t; idx < cnt * nch; idx += blockDim.x) {
      const int e = idx / nch, c = idx - e * nch;
      tile[idx] = __ldg(G4 + (int64_t)sv[e] * ldg4 + c);
    }
    __syncthreads();
    if (t < nch) {
      for (int e = 0; e < cnt; ++e) mul_add4(acc, sw[e], tile[e * nch + t]);
    }
    __syncthreads();
  }
  if (t < nch) {
    if (score_r) add_score_term(acc, __ldg(score_r + s), a_r, t, F);
    tile[t] = acc;
  }
  __syncthreads();
  if (t < 32) {
    float4 v[CPLQ];
#pragma unroll
    for (int i = 0; i < CPLQ; ++i) {
      const int c = lane + 32 * i;
      v[i] = c < nch ? tile[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    quantize_pack_row_sel<32, CPLQ>(v, F, __ldg(slot_bits + s), row_key(seed, (uint32_t)s),
                                    packed + __ldg(slot_off + s), meta + s, lane, 0xffffffffu);
  }
}

// Ordinary slots through a per-warp ring of R + 1 gradient rows in shared
// memory.  A warp takes HK (<= 32) consecutive slots of the visiting order
// and walks their entries as one stream of T entries: entry k + R is
// requested (each lane copies its own chunks with 16-byte asynchronous
// copies) as entry k is added, so R rows stay in flight at every step -- also
// while a finished slot is quantised -- and no register holds a row in
// flight.  Each lane reads back only the chunks it copied, so no barrier is
// needed; the row a copy overwrites was added one step earlier.  Lane k holds
// slot k's first entry, length and start in the stream (an exclusive scan of
// the lengths); a batch of 32 stream positions loads its (col, val) pairs in
// one step (each lane finds its position's slot by a binary search over the
// starts), and the consumer finds the next slot with entries from a ballot
// mask, so the per-entry work is two shuffles, the copies, one weight store
// and the adds.  Every slot's sum keeps its fixed order (entries ascending,
// product and sum each rounded).  Measured on the R-MAT graph at F = 256:
// 42.3 ms, against 45.9 ms for a first version that tracked slots and
// entries with 64-bit cursors and loaded (col, val) per slot.
template <int CPL, int R, int HK>
__device__ __forceinline__ void halo_ring_stream(
    int64_t block, const int64_t* __restrict__ srp, const int32_t* __restrict__ scol,
    const float* __restrict__ sval, const float4* __restrict__ G4, int64_t ldg4, int F,
    const uint8_t* __restrict__ slot_bits, const int64_t* __restrict__ slot_off, uint32_t seed,
    uint8_t* __restrict__ packed, float2* __restrict__ meta, int long_len,
    const float* __restrict__ score_r, const float* __restrict__ a_r,
    const int32_t* __restrict__ order, int64_t s_lo, int64_t s_hi, float4* ring, float* wring) {
  constexpr uint32_t FULL = 0xffffffffu;
  constexpr uint32_t RING = R + 1;
  const int lane = threadIdx.x & 31;
  const int nch = (F + 3) >> 2;
  const int64_t count = s_hi - s_lo;
  const int64_t i0 = ((block * blockDim.x + threadIdx.x) >> 5) * HK;
  if (i0 >= count) return;  // uniform across the warp
  const int nslots = (int)min((int64_t)HK, count - i0);
  long long my_s = 0, my_b = 0;
  int my_n = 0;
  if (lane < nslots) {
    my_s = order ? (long long)__ldg(order + i0 + lane) : (long long)(s_lo + i0 + lane);
    my_b = __ldg(srp + my_s);
    my_n = (int)(__ldg(srp + my_s + 1) - my_b);
    if (long_len > 0 && my_n > long_len) my_n = 0;  // summed by a long-slot block
  }
  // exclusive scan of the lengths: my_start; T = total entries of the run
  int incl = my_n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  const int my_start = incl - my_n;
  const int T = __shfl_sync(FULL, incl, 31);
  const uint32_t nonempty = __ballot_sync(FULL, my_n > 0);
  // batch of stream positions [tb, tb + 32): lane l holds (col, val) of tb + l
  int vb = 0;
  float wb = 0.f;
  auto load_batch = [&](int tb) {
    const int p = tb + lane;
    vb = 0;
    wb = 0.f;
    int k = 0;  // the last slot whose start is <= p
#pragma unroll
    for (int step = 16; step > 0; step >>= 1) {
      const int st = __shfl_sync(FULL, my_start, (k + step) & 31);
      if (k + step < nslots && st <= p) k += step;
    }
    const long long b = __shfl_sync(FULL, my_b, k);
    const int st = __shfl_sync(FULL, my_start, k);
    if (p < T) {
      vb = __ldg(scol + b + (p - st));
      wb = __ldg(sval + b + (p - st));
    }
  };
  int tf = 0;  // next stream position to fetch
  auto fetch_one = [&]() {
    if (tf < T) {
      if ((tf & 31) == 0) load_batch(tf);
      const int v = __shfl_sync(FULL, vb, tf & 31);
      const uint32_t r = (uint32_t)tf % RING;
      wring[r * 32 + lane] = __shfl_sync(FULL, wb, tf & 31);
      const float4* src = G4 + (int64_t)v * ldg4;
      float4* dst = ring + r * (32 * CPL);
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < nch) cp_async16(dst + c, src + c);
      }
    }
    cp_async_commit();
    ++tf;
  };
#pragma unroll 1
  for (int k = 0; k < R; ++k) fetch_one();
  float4 acc[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  int kc = nonempty ? __ffs(nonempty) - 1 : 32;
  int end_c = kc < 32 ? __shfl_sync(FULL, incl, kc) : 0;
#pragma unroll 1
  for (int tc = 0; tc < T; ++tc) {
    cp_async_wait<R - 1>();
    const uint32_t r = (uint32_t)tc % RING;
    const float w = wring[r * 32 + lane];
    const float4* src = ring + r * (32 * CPL);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      if (c < nch) mul_add4(acc[i], w, src[c]);
    }
    fetch_one();
    if (tc + 1 == end_c) {  // slot kc complete
      const int64_t s = __shfl_sync(FULL, my_s, kc);
      if (score_r) {
        const float rs = __ldg(score_r + s);
#pragma unroll
        for (int i = 0; i < CPL; ++i)
          if (lane + 32 * i < nch) add_score_term(acc[i], rs, a_r, lane + 32 * i, F);
      }
      quantize_pack_row_sel<32, CPL>(acc, F, __ldg(slot_bits + s), row_key(seed, (uint32_t)s),
                                 packed + __ldg(slot_off + s), meta + s, lane, FULL);
#pragma unroll
      for (int i = 0; i < CPL; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      const uint32_t later = kc < 31 ? nonempty & ~((2u << kc) - 1u) : 0u;
      kc = later ? __ffs(later) - 1 : 32;
      end_c = kc < 32 ? __shfl_sync(FULL, incl, kc) : 0;
    }
  }
  cp_async_wait<0>();
}

// Shared memory of a ring block: per warp (R + 1) rows of 32 * CPL chunks
// and (R + 1) x 32 weights.
constexpr size_t halo_ring_warp_bytes(int CPL, int R) {
  return (size_t)(R + 1) * 32 * CPL * 16 + (size_t)(R + 1) * 32 * 4;
}

template <int CPL, int R, int HK>
__global__ void __launch_bounds__(256) halo_ring_kernel(
    int64_t S, const int64_t* __restrict__ srp, const int32_t* __restrict__ scol,
    const float* __restrict__ sval, const float* __restrict__ Gm, int64_t ldg, int F,
    const uint8_t* __restrict__ slot_bits, const int64_t* __restrict__ slot_off, uint32_t seed,
    uint8_t* __restrict__ packed, float2* __restrict__ meta, int n_long,
    const int32_t* __restrict__ long_slots, int long_len, int E, const float* __restrict__ score_r,
    const float* __restrict__ a_r, const int32_t* __restrict__ order, int64_t s_lo, int64_t s_hi) {
  extern __shared__ float4 tile[];
  const float4* G4 = reinterpret_cast<const float4*>(Gm);
  const int64_t ldg4 = ldg >> 2;
  if ((int)blockIdx.x < n_long) {
    halo_long_block<CPL>(blockIdx.x, srp, scol, sval, G4, ldg4, F, slot_bits, slot_off, seed,
                         packed, meta, long_slots, E, score_r, a_r, s_lo, s_hi, tile);
    return;
  }
  const int warp = threadIdx.x >> 5;
  char* base = reinterpret_cast<char*>(tile) + (size_t)warp * halo_ring_warp_bytes(CPL, R);
  float4* ring = reinterpret_cast<float4*>(base);
  float* wring = reinterpret_cast<float*>(base + (size_t)(R + 1) * 32 * CPL * 16);
  halo_ring_stream<CPL, R, HK>(blockIdx.x - n_long, srp, scol, sval, G4, ldg4, F, slot_bits,
                               slot_off, seed, packed, meta, long_len, score_r, a_r, order, s_lo,
                               s_hi, ring, wring);
}

template <int G, int CPL, int U, int HK>
__global__ void __launch_bounds__(256, (G == 32 && CPL <= 3) ? 4 : 1) halo_quant_pack_kernel(
    int64_t S, const int64_t* __restrict__ srp, const int32_t* __restrict__ scol,
    const float* __restrict__ sval, const float* __restrict__ Gm, int64_t ldg, int F,
    const uint8_t* __restrict__ slot_bits, const int64_t* __restrict__ slot_off, uint32_t seed,
    uint8_t* __restrict__ packed, float2* __restrict__ meta, int n_long,
    const int32_t* __restrict__ long_slots, int long_len, int E, const float* __restrict__ score_r,
    const float* __restrict__ a_r, const int32_t* __restrict__ order, int64_t s_lo, int64_t s_hi) {
  constexpr int CPLQ = (G * CPL + 31) / 32;  // chunks per lane when one warp quantises
  extern __shared__ float4 tile[];
  const int lane = threadIdx.x & 31;
  const int nch = (F + 3) >> 2;
  const float4* G4 = reinterpret_cast<const float4*>(Gm);
  const int64_t ldg4 = ldg >> 2;

  if ((int)blockIdx.x < n_long) {
    halo_long_block<CPLQ>(blockIdx.x, srp, scol, sval, G4, ldg4, F, slot_bits, slot_off, seed,
                          packed, meta, long_slots, E, score_r, a_r, s_lo, s_hi, tile);
    return;
  }

  const int gl = lane & (G - 1);
  if constexpr (HK > 1) {
    halo_group_slots<G, CPL, U, HK>(blockIdx.x - n_long, srp, scol, sval, G4, ldg4, F, slot_bits,
                                    slot_off, seed, packed, meta, long_len, score_r, a_r, order,
                                    s_lo, s_hi);
    return;
  }
  const int64_t i = ((int64_t)(blockIdx.x - n_long) * blockDim.x + threadIdx.x) / G;
  if (i >= s_hi - s_lo) return;
  // visiting order (no effect on results), or the slots of [s_lo, s_hi) in turn
  const int64_t s = order ? (int64_t)__ldg(order + i) : s_lo + i;
  const int64_t beg = __ldg(srp + s), end = __ldg(srp + s + 1);
  if (long_len > 0 && end - beg > long_len) return;  // summed by a long-slot block
  const uint32_t gmask = group_mask(G, lane);
  float4 acc[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t base = beg; base < end; base += G) {
    const int64_t e = base + gl;
    int v = 0;
    float w = 0.f;
    if (e < end) {
      v = __ldg(scol + e);
      w = __ldg(sval + e);
      prefetch_lines<GNN_PF_HALO>(G4 + (int64_t)v * ldg4, 0u, 16u * nch);
    }
    const int cnt = (int)min((int64_t)G, end - base);
    for (int k = 0; k < cnt; k += U) {
      float4 x[U][CPL];
      float wk[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int src = (k + u < cnt) ? k + u : k;
        const int vk = __shfl_sync(gmask, v, src, G);
        wk[u] = __shfl_sync(gmask, w, src, G);
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = gl + i * G;
          if (c < nch) x[u][i] = __ldg(G4 + (int64_t)vk * ldg4 + c);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (k + u < cnt) {
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            if (gl + i * G < nch) mul_add4(acc[i], wk[u], x[u][i]);
          }
        }
      }
    }
  }
  if (score_r) {
    const float r = __ldg(score_r + s);
#pragma unroll
    for (int i = 0; i < CPL; ++i)
      if (gl + i * G < nch) add_score_term(acc[i], r, a_r, gl + i * G, F);
  }
  quantize_pack_row<G, CPL>(acc, F, __ldg(slot_bits + s), row_key(seed, (uint32_t)s),
                            packed + __ldg(slot_off + s), meta + s, gl, gmask);
}

// ---------------------------------------------------------------- dispatch
static RowSplit row_split_of(const gnn_csr& csr) {
  RowSplit sp{};
  if (csr.split_len > 0) {
    sp.T = csr.split_len;
    sp.n_long = csr.n_long;
    sp.n_pieces = csr.n_pieces;
    sp.long_rows = csr.long_rows;
    sp.piece_ptr = csr.piece_ptr;
    sp.piece_row = csr.piece_row;
    sp.piece_beg = csr.piece_beg;
  }
  return sp;
}

template <int MODE>
static gnn_status dispatch_rows(const gnn_csr& csr, const int32_t* colv, const float* valv,
                                const int32_t* local_cnt, const float* H, int64_t ldh, int F,
                                SlotMsgs msg, const int64_t* own_ptr, const int32_t* own_slot,
                                float* partial, float* M, int64_t ldm, __nv_bfloat16* Mb,
                                int64_t ldmb, cudaStream_t st, int relu = 0,
                                const float* hmask = nullptr, int64_t ldhm = 0, int ldb_pad = 0) {
  const int nch = (F + 3) / 4;
  // bf16 columns written (zeros past F): round_up(F, 16), or ldb_pad
  const int nch_b = Mb ? (ldb_pad > 0 ? ldb_pad / 4 : ((F + 15) / 16) * 4) : nch;
  const int need = nch_b > nch ? nch_b : nch;
  const RowSplit sp = row_split_of(csr);
  // feature slices of at most GNN_SLICE_CHUNKS chunks keep every lane's registers low
  Slices sl{1, need};
  if (need > GNN_SLICE_CHUNKS) {
    sl.ns = (need + GNN_SLICE_CHUNKS - 1) / GNN_SLICE_CHUNKS;
    sl.cs = (need + sl.ns - 1) / sl.ns;
  }
  const int cpl = (sl.cs + 31) / 32;
  constexpr int block = rows_block<MODE>();
#define GNN_ROWS(G_, CPL_, U_, UR_)                                                            \
  do {                                                                                         \
    const int64_t row_units = (MODE != kPlain && sl.ns == 1)                                   \
                                  ? ((int64_t)csr.n + GNN_ROWS_MULTI - 1) / GNN_ROWS_MULTI     \
                                  : (int64_t)csr.n;                                            \
    const int64_t groups = (row_units + sp.n_pieces) * sl.ns;                                  \
    const int64_t grid = (groups * G_ + block - 1) / block;                                    \
    spmm_rows_kernel<G_, CPL_, MODE, U_, UR_><<<(unsigned)grid, block, 0, st>>>(               \
        csr.n, csr.rowptr, colv, valv, local_cnt, H, ldh, F, msg, own_ptr, own_slot, sp, sl,   \
        partial, M, ldm, Mb, ldmb, nch_b, relu, hmask, ldhm);                                  \
    GNN_CHECK_LAUNCH();                                                                        \
    if (sp.n_long > 0) {                                                                       \
      const int64_t g2 = ((int64_t)sp.n_long * sl.ns * G_ + 255) / 256;                        \
      spmm_fixup_kernel<G_, CPL_, MODE><<<(unsigned)g2, 256, 0, st>>>(                         \
          sp, sl, partial, F, msg, own_ptr, own_slot, M, ldm, Mb, ldmb, nch_b, relu, hmask,    \
          ldhm);                                                                               \
      GNN_CHECK_LAUNCH();                                                                      \
    }                                                                                          \
  } while (0)
  // entries gathered per round: ~8 float4 loads in flight per lane for local
  // rows; remote rows carry four more values per entry and gather fewer
  constexpr int U1 = MODE == kFwdRemote ? GNN_U1_FWD : GNN_U1;
  constexpr int U2 = MODE == kFwdRemote ? GNN_U2_FWD : GNN_U2;
  if (sl.cs <= 4) GNN_ROWS(4, 1, U1, GNN_UR1);
  else if (sl.cs <= 8) GNN_ROWS(8, 1, U1, GNN_UR1);
  else if (sl.cs <= 16) GNN_ROWS(16, 1, U1, GNN_UR1);
  else if (cpl == 1) GNN_ROWS(32, 1, U1, GNN_UR1);
  else if (cpl == 2) GNN_ROWS(32, 2, U2, GNN_UR2);
  else if (cpl == 3) GNN_ROWS(32, 3, 2, GNN_UR3);
  else return fail(GNN_ERR_UNSUPPORTED, "spmm: F=%d exceeds %d", F, kMaxF);
#undef GNN_ROWS
  return GNN_OK;
}

gnn_status launch_spmm_fwd(const gnn_csr& csr, const gnn_boundary* bnd, const float* H,
                           int64_t ldh, int F, const uint8_t* packed, const float2* meta,
                           float* M, int64_t ldm, uint16_t* Mb, int64_t ldmb, float* partial,
                           cudaStream_t st, int relu) {
  if (csr.n == 0) return GNN_OK;
  auto* mb = reinterpret_cast<__nv_bfloat16*>(Mb);
  if (!bnd)
    return dispatch_rows<kPlain>(csr, csr.col, csr.val, nullptr, H, ldh, F, SlotMsgs{}, nullptr,
                                 nullptr, partial, M, ldm, mb, ldmb, st, relu);
  SlotMsgs msg{packed, meta, bnd->slot_off, bnd->slot_bits};
  return dispatch_rows<kFwdRemote>(csr, bnd->col_remap, bnd->val_remap, bnd->local_cnt, H, ldh, F,
                                   msg, nullptr, nullptr, partial, M, ldm, mb, ldmb, st, relu);
}

gnn_status launch_spmm_bwd_masked(const gnn_csr& csr, const gnn_boundary* bnd, const float* Gm,
                                  int64_t ldg, int F, uint32_t seed, uint8_t* packed_ws,
                                  float2* meta_ws, const float* hmask, int64_t ldhm, uint16_t* dZ,
                                  int64_t ldz, float* partial, cudaStream_t st) {
  if (csr.n == 0) return GNN_OK;
  auto* zb = reinterpret_cast<__nv_bfloat16*>(dZ);
  if (!bnd) {
    const float* wt = csr.val_t ? csr.val_t : csr.val;
    return dispatch_rows<kPlain>(csr, csr.col, wt, nullptr, Gm, ldg, F, SlotMsgs{}, nullptr,
                                 nullptr, partial, nullptr, 0, zb, ldz, st, 0, hmask, ldhm,
                                 (int)ldz);
  }
  gnn_status s = launch_halo_quant_pack(*bnd, Gm, ldg, F, seed, packed_ws, meta_ws, st);
  if (s != GNN_OK) return s;
  return launch_spmm_bwd_local_masked(csr, *bnd, Gm, ldg, F, packed_ws, meta_ws, hmask, ldhm, dZ,
                                      ldz, partial, st);
}

gnn_status launch_spmm_bwd_local_masked(const gnn_csr& csr, const gnn_boundary& bnd,
                                        const float* Gm, int64_t ldg, int F, const uint8_t* packed,
                                        const float2* meta, const float* hmask, int64_t ldhm,
                                        uint16_t* dZ, int64_t ldz, float* partial,
                                        cudaStream_t st) {
  if (csr.n == 0) return GNN_OK;
  auto* zb = reinterpret_cast<__nv_bfloat16*>(dZ);
  SlotMsgs msg{packed, meta, bnd.slot_off, bnd.slot_bits};
  const float* wt = bnd.val_remap_t ? bnd.val_remap_t : bnd.val_remap;
  return dispatch_rows<kBwdOwned>(csr, bnd.col_remap, wt, bnd.local_cnt, Gm, ldg, F, msg,
                                  bnd.own_ptr, bnd.own_slot, partial, nullptr, 0, zb, ldz, st, 0,
                                  hmask, ldhm, (int)ldz);
}

gnn_status launch_spmm_fwd_w(const gnn_csr& csr, const gnn_boundary* bnd, const float* weights,
                             const float* H, int64_t ldh, int F, const uint8_t* packed,
                             const float2* meta, float* M, int64_t ldm, float* partial, int relu,
                             cudaStream_t st) {
  if (csr.n == 0) return GNN_OK;
  if (!bnd)
    return dispatch_rows<kPlain>(csr, csr.col, weights, nullptr, H, ldh, F, SlotMsgs{}, nullptr,
                                 nullptr, partial, M, ldm, nullptr, 0, st, relu);
  SlotMsgs msg{packed, meta, bnd->slot_off, bnd->slot_bits};
  return dispatch_rows<kFwdRemote>(csr, bnd->col_remap, weights, bnd->local_cnt, H, ldh, F, msg,
                                   nullptr, nullptr, partial, M, ldm, nullptr, 0, st, relu);
}

gnn_status launch_spmm_bwd_local_w(const gnn_csr& csr, const gnn_boundary* bnd,
                                   const float* weights, const float* Gm, int64_t ldg, int F,
                                   const uint8_t* packed, const float2* meta, float* dH,
                                   int64_t ldh, float* partial, cudaStream_t st) {
  if (csr.n == 0) return GNN_OK;
  if (!bnd)
    return dispatch_rows<kPlain>(csr, csr.col, weights, nullptr, Gm, ldg, F, SlotMsgs{}, nullptr,
                                 nullptr, partial, dH, ldh, nullptr, 0, st);
  SlotMsgs msg{packed, meta, bnd->slot_off, bnd->slot_bits};
  return dispatch_rows<kBwdOwned>(csr, bnd->col_remap, weights, bnd->local_cnt, Gm, ldg, F, msg,
                                  bnd->own_ptr, bnd->own_slot, partial, dH, ldh, nullptr, 0, st);
}

static int quant_chunk_slots(int F) {
  const int a = 32 * ((F + 127) / 128), b = (F + 3) / 4;
  return a > b ? a : b;
}

gnn_status launch_halo_quant_pack(const gnn_boundary& b, const float* Gm, int64_t ldg, int F,
                                  uint32_t seed, uint8_t* packed_ws, float2* meta_ws,
                                  cudaStream_t st) {
  return launch_halo_quant_pack_ex(b, Gm, ldg, F, seed, packed_ws, meta_ws, b.slot_val, nullptr,
                                   nullptr, st);
}

// Backward messages of 32-lane row layouts through the ring kernel
// (GNN_HALO_RING 1) or through register gathers (0).
#ifndef GNN_HALO_RING
#define GNN_HALO_RING 1
#endif
#ifndef GNN_RING_R
#define GNN_RING_R 3
#endif
// Rows in flight per warp of the ring kernel, by chunks per lane (shared
// memory per warp: (R + 1) rows of 512 * CPL bytes).  Measured on the R-MAT
// graph at F = 256 (37.9M slots, 256-thread blocks, 64 registers): R = 2, 3,
// 4, 5, 7 took 48.5, 45.9, 49.0, 46.4, 55.7 ms against 50.8 ms for the
// register kernel; deeper rings cost resident warps (shared memory) faster
// than they add rows in flight.
constexpr int halo_ring_depth(int CPL) { return CPL <= 2 ? GNN_RING_R : (CPL <= 4 ? 3 : 2); }
constexpr int kRingSlotsPerWarp = 32;
// Where the ring pays (measured): wide rows (F = 602, 5 chunks per lane:
// 7.9 against 11.5 ms on the Reddit-shaped graph) and the 16.8M-slot R-MAT
// graph at F = 256 (46.2 against 52.8 ms).  On the Yelp-shaped graph's 0.8M
// slots at F = 300 the register kernel is faster (0.85 against 1.00 ms).
#ifndef GNN_RING_MIN_SLOTS
#define GNN_RING_MIN_SLOTS (int64_t(1) << 24)
#endif
static bool halo_use_ring(int G, int CPL, int64_t count) {
  return GNN_HALO_RING && G == 32 && CPL <= 8 && (CPL >= 4 || count >= GNN_RING_MIN_SLOTS);
}

template <int CPL>
static gnn_status launch_halo_ring(const gnn_boundary& b, const float* Gm, int64_t ldg, int F,
                                   uint32_t seed, uint8_t* packed_ws, float2* meta_ws,
                                   const float* sval, const float* score_r, const float* a_r,
                                   cudaStream_t st, int64_t s_lo, int64_t s_hi,
                                   const int32_t* order, int n_long, int long_len, int E,
                                   size_t long_smem) {
  constexpr int R = halo_ring_depth(CPL);
  constexpr int block = 256;
  const size_t ring = (size_t)(block / 32) * halo_ring_warp_bytes(CPL, R);
  const size_t dyn = ring > long_smem ? ring : long_smem;
  static bool attr_set[8] = {};  // per device
  int dev = 0;
  GNN_CUDA(cudaGetDevice(&dev));
  if (dev >= 8 || !attr_set[dev]) {
    // long-slot blocks stage at most 48 KB; the ring needs `ring` bytes
    const int need = (int)(ring > 49152 ? ring : 49152);
    GNN_CUDA(cudaFuncSetAttribute(halo_ring_kernel<CPL, R, kRingSlotsPerWarp>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, need));
    if (dev < 8) attr_set[dev] = true;
  }
  const int64_t count = s_hi - s_lo;
  const int64_t warps = (count + kRingSlotsPerWarp - 1) / kRingSlotsPerWarp;
  const int64_t grid = n_long + (warps + block / 32 - 1) / (block / 32);
  halo_ring_kernel<CPL, R, kRingSlotsPerWarp><<<(unsigned)grid, block, dyn, st>>>(
      b.n_slots, b.slot_rowptr, b.slot_col, sval, Gm, ldg, F, b.slot_bits, b.slot_off, seed,
      packed_ws, meta_ws, n_long, b.long_slots, long_len, E, score_r, a_r, order, s_lo, s_hi);
  return GNN_OK;  // the caller checks and counts the launch
}

gnn_status launch_halo_quant_pack_ex(const gnn_boundary& b, const float* Gm, int64_t ldg, int F,
                                     uint32_t seed, uint8_t* packed_ws, float2* meta_ws,
                                     const float* sval, const float* score_r, const float* a_r,
                                     cudaStream_t st, int64_t s_lo, int64_t s_hi) {
  const int64_t S = b.n_slots;
  if (s_hi < 0) s_hi = S;
  if (S == 0 || s_hi <= s_lo) return GNN_OK;
  // the visiting order covers every slot: a partial range walks its slots in turn
  const int32_t* order = (s_lo == 0 && s_hi == S) ? b.halo_order : nullptr;
  const int64_t count = s_hi - s_lo;
  const int slots = quant_chunk_slots(F);
  const int nch = (F + 3) / 4;
  const int block = 256;
  const bool use_long = b.long_slot_len > 0 && b.n_long_slots > 0 && b.long_slots;
  const int n_long = use_long ? b.n_long_slots : 0;
  const int long_len = use_long ? b.long_slot_len : 0;
  // entries staged per round by a long-slot block: at most 32 and 48 KB
  int E = 3072 / nch;
  if (E > 32) E = 32;
  if (E < 1) E = 1;
  const size_t smem = use_long ? (size_t)E * nch * sizeof(float4) : 0;
  const size_t smem_q = (size_t)nch * sizeof(float4);
  const size_t dyn = smem > smem_q ? smem : (use_long ? smem_q : 0);
#define GNN_HALO_K(G_, CPL_, U_, HK_)                                                            \
  do {                                                                                           \
    const int64_t grid = n_long + (((count + (HK_) - 1) / (HK_)) * G_ + block - 1) / block;      \
    halo_quant_pack_kernel<G_, CPL_, U_, HK_><<<(unsigned)grid, block, dyn, st>>>(               \
        S, b.slot_rowptr, b.slot_col, sval, Gm, ldg, F, b.slot_bits, b.slot_off, seed,           \
        packed_ws, meta_ws, n_long, b.long_slots, long_len, E, score_r, a_r, order, s_lo, s_hi); \
  } while (0)
#define GNN_HALO(G_, CPL_, U_)                                                                   \
  do {                                                                                           \
    if (halo_use_ring(G_, CPL_, count)) {                                                        \
      gnn_status rs = launch_halo_ring<CPL_>(b, Gm, ldg, F, seed, packed_ws, meta_ws, sval,       \
                                             score_r, a_r, st, s_lo, s_hi, order, n_long,         \
                                             long_len, E, smem);                                  \
      if (rs != GNN_OK) return rs;                                                               \
    } else if (count >= kManySlots)                                                              \
      GNN_HALO_K(G_, CPL_, U_, halo_slots_per_group(G_, CPL_, true));                            \
    else                                                                                         \
      GNN_HALO_K(G_, CPL_, U_, halo_slots_per_group(G_, CPL_, false));                           \
  } while (0)
  if (slots <= 32) GNN_HALO(8, 4, 2);
  else {
    switch ((slots + 31) / 32) {
      case 1: GNN_HALO(32, 1, 4); break;
      case 2: GNN_HALO(32, 2, 2); break;
      case 3: GNN_HALO(32, 3, 1); break;
      case 4: GNN_HALO(32, 4, 2); break;
      case 5: GNN_HALO(32, 5, 2); break;
      case 6: GNN_HALO(32, 6, 2); break;
      case 7: GNN_HALO(32, 7, 2); break;
      case 8: GNN_HALO(32, 8, 2); break;
      default: return fail(GNN_ERR_UNSUPPORTED, "spmm_bwd: F=%d exceeds %d", F, kMaxF);
    }
  }
#undef GNN_HALO
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

gnn_status launch_spmm_bwd_local(const gnn_csr& csr, const gnn_boundary& bnd, const float* Gm,
                                 int64_t ldg, int F, const uint8_t* packed, const float2* meta,
                                 float* dH, int64_t ldh, float* partial, cudaStream_t st);

gnn_status launch_spmm_bwd(const gnn_csr& csr, const gnn_boundary* bnd, const float* Gm,
                           int64_t ldg, int F, uint32_t seed, uint8_t* packed_ws,
                           float2* meta_ws, float* dH, int64_t ldh, float* partial,
                           cudaStream_t st) {
  if (csr.n == 0) return GNN_OK;
  if (!bnd)
    return dispatch_rows<kPlain>(csr, csr.col, csr.val_t ? csr.val_t : csr.val, nullptr, Gm, ldg,
                                 F, SlotMsgs{}, nullptr, nullptr, partial, dH, ldh, nullptr, 0, st);
  gnn_status s = launch_halo_quant_pack(*bnd, Gm, ldg, F, seed, packed_ws, meta_ws, st);
  if (s != GNN_OK) return s;
  return launch_spmm_bwd_local(csr, *bnd, Gm, ldg, F, packed_ws, meta_ws, dH, ldh, partial, st);
}

gnn_status launch_spmm_bwd_local(const gnn_csr& csr, const gnn_boundary& bnd, const float* Gm,
                                 int64_t ldg, int F, const uint8_t* packed, const float2* meta,
                                 float* dH, int64_t ldh, float* partial, cudaStream_t st) {
  if (csr.n == 0) return GNN_OK;
  SlotMsgs msg{packed, meta, bnd.slot_off, bnd.slot_bits};
  // row u's local entries weighted by A^T: A[v][u] for each local source v
  const float* wt = bnd.val_remap_t ? bnd.val_remap_t : bnd.val_remap;
  return dispatch_rows<kBwdOwned>(csr, bnd.col_remap, wt, bnd.local_cnt, Gm, ldg, F, msg,
                                  bnd.own_ptr, bnd.own_slot, partial, dH, ldh, nullptr, 0, st);
}

size_t spmm_workspace_bytes(const gnn_csr& csr, int F) {
  if (csr.split_len <= 0) return 0;
  return (size_t)csr.n_pieces * (size_t)((F + 3) / 4) * 16u;
}

}  // namespace gnn

using namespace gnn;

static gnn_status check_csr(const gnn_csr* csr, const char* who) {
  if (!csr) return fail(GNN_ERR_INVALID_ARG, "%s: csr is NULL", who);
  if (csr->n < 0 || csr->nnz < 0) return fail(GNN_ERR_INVALID_ARG, "%s: negative csr size", who);
  if (csr->n > 0 && (!csr->rowptr || (csr->nnz > 0 && (!csr->col || !csr->val))))
    return fail(GNN_ERR_INVALID_ARG, "%s: csr arrays are NULL", who);
  if (csr->split_len < 0 || (csr->split_len > 0 && csr->split_len < 32))
    return fail(GNN_ERR_INVALID_ARG, "%s: split_len must be 0 or >= 32", who);
  if (csr->split_len > 0 &&
      (csr->n_long < 0 || csr->n_pieces < 0 || !csr->piece_ptr ||
       (csr->n_long > 0 && !csr->long_rows) ||
       (csr->n_pieces > 0 && (!csr->piece_row || !csr->piece_beg))))
    return fail(GNN_ERR_INVALID_ARG, "%s: incomplete split plan", who);
  return GNN_OK;
}

static gnn_status check_ws(const gnn_csr* csr, int F, void* ws, size_t ws_bytes, const char* who) {
  const size_t need = spmm_workspace_bytes(*csr, F);
  if (need == 0) return GNN_OK;
  if (!ws || ws_bytes < need || ((uintptr_t)ws & 15) != 0)
    return fail(GNN_ERR_INVALID_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)",
                who, need, ws_bytes);
  return GNN_OK;
}

static gnn_status check_bnd(const gnn_csr* csr, const gnn_boundary* b, int F, bool bwd,
                            const char* who) {
  if (!b) return GNN_OK;
  if (b->n != csr->n || b->P < 1) return fail(GNN_ERR_INVALID_ARG, "%s: boundary does not match csr", who);
  if (b->F != F)
    return fail(GNN_ERR_INVALID_ARG, "%s: boundary offsets are for F=%d, call has F=%d", who, b->F, F);
  if (!b->col_remap || !b->val_remap || !b->local_cnt ||
      (b->n_slots > 0 && (!b->slot_off || !b->slot_bits)))
    return fail(GNN_ERR_INVALID_ARG, "%s: boundary arrays are NULL", who);
  if (bwd && (!b->own_ptr || (b->n_slots > 0 && (!b->slot_rowptr || !b->own_slot)) ||
              (b->nnz_cut > 0 && (!b->slot_col || !b->slot_val))))
    return fail(GNN_ERR_INVALID_ARG, "%s: boundary backward arrays are NULL", who);
  if (bwd && !csr->symmetric && !b->val_remap_t)
    return fail(GNN_ERR_INVALID_ARG, "%s: A is not symmetric and the boundary has no val_remap_t",
                who);
  if (bwd && b->long_slot_len > 0 &&
      (b->long_slot_len < 32 || b->n_long_slots < 0 || (b->n_long_slots > 0 && !b->long_slots)))
    return fail(GNN_ERR_INVALID_ARG, "%s: incomplete long-slot list", who);
  return GNN_OK;
}

extern "C" gnn_status gnn_spmm_workspace(const gnn_csr* csr, int32_t F, size_t* ws_bytes) {
  gnn_status st = check_csr(csr, "gnn_spmm_workspace");
  if (st != GNN_OK) return st;
  GNN_REQUIRE(F >= 1 && ws_bytes, "gnn_spmm_workspace: bad arguments");
  *ws_bytes = spmm_workspace_bytes(*csr, F);
  return GNN_OK;
}

extern "C" gnn_status gnn_spmm_fwd(const gnn_csr* csr, const gnn_boundary* bnd, const float* H,
                                   int64_t ldh, int32_t F, const uint8_t* packed,
                                   const float* meta, float* M, int64_t ldm, uint16_t* Mb,
                                   int64_t ldmb, void* ws, size_t ws_bytes, gnn_stream_t stream) {
  return gnn::spmm_fwd_checked(csr, bnd, H, ldh, F, packed, meta, M, ldm, Mb, ldmb, ws, ws_bytes,
                               stream, 0);
}

gnn_status gnn::spmm_fwd_checked(const gnn_csr* csr, const gnn_boundary* bnd, const float* H,
                                 int64_t ldh, int32_t F, const uint8_t* packed, const float* meta,
                                 float* M, int64_t ldm, uint16_t* Mb, int64_t ldmb, void* ws,
                                 size_t ws_bytes, gnn_stream_t stream, int relu) {
  gnn_status st = check_csr(csr, "gnn_spmm_fwd");
  if (st != GNN_OK) return st;
  GNN_REQUIRE(F >= 1, "gnn_spmm_fwd: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_fwd: F=%d > %d", F, kMaxF);
  if ((st = check_bnd(csr, bnd, F, false, "gnn_spmm_fwd")) != GNN_OK) return st;
  if ((st = check_ws(csr, F, ws, ws_bytes, "gnn_spmm_fwd")) != GNN_OK) return st;
  if (csr->n == 0) return GNN_OK;
  GNN_REQUIRE(H && (M || Mb), "gnn_spmm_fwd: H is NULL or no output given");
  GNN_REQUIRE(ldh >= F && ldh % 4 == 0 && ((uintptr_t)H & 15) == 0,
              "gnn_spmm_fwd: ldh must be >= F, a multiple of 4, H 16-byte aligned");
  GNN_REQUIRE(!M || (ldm >= F && ldm % 4 == 0 && ((uintptr_t)M & 15) == 0),
              "gnn_spmm_fwd: ldm must be >= F, a multiple of 4, M 16-byte aligned");
  GNN_REQUIRE(!Mb || (ldmb >= (F + 15) / 16 * 16 && ldmb % 8 == 0 && ((uintptr_t)Mb & 15) == 0),
              "gnn_spmm_fwd: ldmb must be >= round_up(F,16), a multiple of 8, Mb 16-byte aligned");
  GNN_REQUIRE(!bnd || bnd->n_slots == 0 || (packed && meta),
              "gnn_spmm_fwd: packed/meta required with a boundary");
  return launch_spmm_fwd(*csr, bnd, H, ldh, F, packed, reinterpret_cast<const float2*>(meta), M,
                         ldm, Mb, ldmb, static_cast<float*>(ws), as_stream(stream), relu);
}

extern "C" gnn_status gnn_spmm_bwd(const gnn_csr* csr, const gnn_boundary* bnd, const float* G,
                                   int64_t ldg, int32_t F, uint32_t seed, uint8_t* packed_ws,
                                   float* meta_ws, float* dH, int64_t ldh, void* ws,
                                   size_t ws_bytes, gnn_stream_t stream) {
  gnn_status st = check_csr(csr, "gnn_spmm_bwd");
  if (st != GNN_OK) return st;
  GNN_REQUIRE(F >= 1, "gnn_spmm_bwd: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_bwd: F=%d > %d", F, kMaxF);
  if (!csr->symmetric && !csr->val_t)
    return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_bwd: needs A^T (a symmetric CSR or val_t)");
  if ((st = check_bnd(csr, bnd, F, true, "gnn_spmm_bwd")) != GNN_OK) return st;
  if ((st = check_ws(csr, F, ws, ws_bytes, "gnn_spmm_bwd")) != GNN_OK) return st;
  if (csr->n == 0) return GNN_OK;
  GNN_REQUIRE(G && dH, "gnn_spmm_bwd: NULL G or dH");
  GNN_REQUIRE(ldg >= F && ldg % 4 == 0 && ((uintptr_t)G & 15) == 0,
              "gnn_spmm_bwd: ldg must be >= F, a multiple of 4, G 16-byte aligned");
  GNN_REQUIRE(ldh >= F && ldh % 4 == 0 && ((uintptr_t)dH & 15) == 0,
              "gnn_spmm_bwd: ldh must be >= F, a multiple of 4, dH 16-byte aligned");
  GNN_REQUIRE(!bnd || bnd->n_slots == 0 ||
                  (packed_ws && meta_ws && ((uintptr_t)packed_ws & 15) == 0 && ((uintptr_t)meta_ws & 7) == 0),
              "gnn_spmm_bwd: packed_ws (16-byte aligned) and meta_ws required with a boundary");
  return launch_spmm_bwd(*csr, bnd, G, ldg, F, seed, packed_ws,
                         reinterpret_cast<float2*>(meta_ws), dH, ldh, static_cast<float*>(ws),
                         as_stream(stream));
}

extern "C" gnn_status gnn_spmm_bwd_masked(const gnn_csr* csr, const gnn_boundary* bnd,
                                          const float* G, int64_t ldg, int32_t F, uint32_t seed,
                                          uint8_t* packed_ws, float* meta_ws, const float* H_mask,
                                          int64_t ldhm, uint16_t* dZ, int64_t ldz, void* ws,
                                          size_t ws_bytes, gnn_stream_t stream) {
  gnn_status st = check_csr(csr, "gnn_spmm_bwd_masked");
  if (st != GNN_OK) return st;
  GNN_REQUIRE(F >= 1, "gnn_spmm_bwd_masked: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_bwd_masked: F=%d > %d", F, kMaxF);
  if (!csr->symmetric && !csr->val_t)
    return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_bwd_masked: needs A^T (a symmetric CSR or val_t)");
  if ((st = check_bnd(csr, bnd, F, true, "gnn_spmm_bwd_masked")) != GNN_OK) return st;
  if ((st = check_ws(csr, F, ws, ws_bytes, "gnn_spmm_bwd_masked")) != GNN_OK) return st;
  if (csr->n == 0) return GNN_OK;
  GNN_REQUIRE(G && dZ, "gnn_spmm_bwd_masked: NULL G or dZ");
  GNN_REQUIRE(ldg >= F && ldg % 4 == 0 && ((uintptr_t)G & 15) == 0,
              "gnn_spmm_bwd_masked: ldg must be >= F, a multiple of 4, G 16-byte aligned");
  GNN_REQUIRE(ldz >= (F + 63) / 64 * 64 && ldz % 8 == 0 && ((uintptr_t)dZ & 15) == 0,
              "gnn_spmm_bwd_masked: ldz must be >= round_up(F, 64), a multiple of 8, dZ 16-byte aligned");
  GNN_REQUIRE(!H_mask || (ldhm >= F && ldhm % 4 == 0 && ((uintptr_t)H_mask & 15) == 0),
              "gnn_spmm_bwd_masked: ldhm must be >= F, a multiple of 4, H_mask 16-byte aligned");
  GNN_REQUIRE(!bnd || bnd->n_slots == 0 ||
                  (packed_ws && meta_ws && ((uintptr_t)packed_ws & 15) == 0 && ((uintptr_t)meta_ws & 7) == 0),
              "gnn_spmm_bwd_masked: packed_ws (16-byte aligned) and meta_ws required with a boundary");
  return launch_spmm_bwd_masked(*csr, bnd, G, ldg, F, seed, packed_ws,
                                reinterpret_cast<float2*>(meta_ws), H_mask, ldhm, dZ, ldz,
                                static_cast<float*>(ws), as_stream(stream));
}

extern "C" gnn_status gnn_spmm_bwd_local_masked(const gnn_csr* csr, const gnn_boundary* bnd,
                                                const float* G, int64_t ldg, int32_t F,
                                                const uint8_t* packed, const float* meta,
                                                const float* H_mask, int64_t ldhm, uint16_t* dZ,
                                                int64_t ldz, void* ws, size_t ws_bytes,
                                                gnn_stream_t stream) {
  gnn_status st = check_csr(csr, "gnn_spmm_bwd_local_masked");
  if (st != GNN_OK) return st;
  GNN_REQUIRE(bnd, "gnn_spmm_bwd_local_masked: boundary is NULL (use gnn_spmm_bwd_masked)");
  GNN_REQUIRE(F >= 1, "gnn_spmm_bwd_local_masked: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_bwd_local_masked: F=%d > %d", F, kMaxF);
  if (!csr->symmetric && !csr->val_t)
    return fail(GNN_ERR_UNSUPPORTED,
                "gnn_spmm_bwd_local_masked: needs A^T (a symmetric CSR or val_t)");
  if ((st = check_bnd(csr, bnd, F, true, "gnn_spmm_bwd_local_masked")) != GNN_OK) return st;
  if ((st = check_ws(csr, F, ws, ws_bytes, "gnn_spmm_bwd_local_masked")) != GNN_OK) return st;
  if (csr->n == 0) return GNN_OK;
  GNN_REQUIRE(G && dZ, "gnn_spmm_bwd_local_masked: NULL G or dZ");
  GNN_REQUIRE(ldg >= F && ldg % 4 == 0 && ((uintptr_t)G & 15) == 0,
              "gnn_spmm_bwd_local_masked: ldg must be >= F, a multiple of 4, G 16-byte aligned");
  GNN_REQUIRE(ldz >= (F + 63) / 64 * 64 && ldz % 8 == 0 && ((uintptr_t)dZ & 15) == 0,
              "gnn_spmm_bwd_local_masked: ldz must be >= round_up(F, 64), a multiple of 8, dZ "
              "16-byte aligned");
  GNN_REQUIRE(!H_mask || (ldhm >= F && ldhm % 4 == 0 && ((uintptr_t)H_mask & 15) == 0),
              "gnn_spmm_bwd_local_masked: ldhm must be >= F, a multiple of 4, H_mask 16-byte "
              "aligned");
  GNN_REQUIRE(bnd->n_slots == 0 || (packed && meta && ((uintptr_t)packed & 15) == 0),
              "gnn_spmm_bwd_local_masked: packed (16-byte aligned) and meta required");
  return launch_spmm_bwd_local_masked(*csr, *bnd, G, ldg, F, packed,
                                      reinterpret_cast<const float2*>(meta), H_mask, ldhm, dZ, ldz,
                                      static_cast<float*>(ws), as_stream(stream));
}

// ---------------------------------------------------------------- no-allocation forward
// Some callers cannot call cudaMalloc once they are running: a serving loop
// whose device memory is fully reserved at start-up, or a plugin that a host
// framework hands only input and output pointers while keeping every
// allocation to itself.  gnn_spmm_fwd_noalloc serves them: the partial rows of
// the split plan live in the fixed device array below instead of a caller
// workspace.  Every GPU that loads this library holds the array until the
// process exits.
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kNoAllocMaxDevices = 64;
static __device__ __align__(256) float g_noalloc_partials[kNoAllocScratchBytes / sizeof(float)];
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kNoAllocMaxDevices] = {};
CUcontext g_noalloc_ctx[kNoAllocMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent, fetched once through the runtime (the
// library links no driver library).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuCtxGetCurrent", &p, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}
}  // namespace

// Device address of the array on the current device.  Host code only knows a
// host-side stand-in for the symbol, so the address is looked up with that
// device current and cached together with the context it was found in: a
// new context on the device (after cudaDeviceReset, or once the primary
// context was released and created again) is seen and the address looked up
// afresh, so a stale address from a dead context is never used.
static gnn_status noalloc_scratch(float** out) {
  int dev = 0;
  GNN_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_fwd_noalloc: device %d out of range", dev);
  GNN_CUDA(cudaSetDevice(dev));  // makes the device's primary context current on this thread
  CUcontext ctx = nullptr;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get || get(&ctx) != CUDA_SUCCESS)
    return fail(GNN_ERR_CUDA, "gnn_spmm_fwd_noalloc: cannot read the current context");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx) {
    void* p = nullptr;
    GNN_CUDA(cudaGetSymbolAddress(&p, g_noalloc_partials));
    g_noalloc_ptr[dev] = static_cast<float*>(p);
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_ptr[dev];
  return GNN_OK;
}

extern "C" gnn_status gnn_spmm_fwd_noalloc(const gnn_csr* csr, const gnn_boundary* bnd,
                                           const float* H, int64_t ldh, int32_t F,
                                           const uint8_t* packed, const float* meta, float* M,
                                           int64_t ldm, uint16_t* Mb, int64_t ldmb,
                                           gnn_stream_t stream) {
  gnn_status st = check_csr(csr, "gnn_spmm_fwd_noalloc");
  if (st != GNN_OK) return st;
  GNN_REQUIRE(F >= 1, "gnn_spmm_fwd_noalloc: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_fwd_noalloc: F=%d > %d", F, kMaxF);
  const size_t need = spmm_workspace_bytes(*csr, F);
  if (need > kNoAllocScratchBytes)
    return fail(GNN_ERR_UNSUPPORTED,
                "gnn_spmm_fwd_noalloc: the split plan needs %zu bytes of scratch at F=%d; the "
                "static buffer holds %zu (use gnn_spmm_fwd with a workspace)",
                need, F, kNoAllocScratchBytes);
  if ((st = check_bnd(csr, bnd, F, false, "gnn_spmm_fwd_noalloc")) != GNN_OK) return st;
  if (csr->n == 0) return GNN_OK;
  GNN_REQUIRE(H && (M || Mb), "gnn_spmm_fwd_noalloc: H is NULL or no output given");
  GNN_REQUIRE(ldh >= F && ldh % 4 == 0 && ((uintptr_t)H & 15) == 0,
              "gnn_spmm_fwd_noalloc: ldh must be >= F, a multiple of 4, H 16-byte aligned");
  GNN_REQUIRE(!M || (ldm >= F && ldm % 4 == 0 && ((uintptr_t)M & 15) == 0),
              "gnn_spmm_fwd_noalloc: ldm must be >= F, a multiple of 4, M 16-byte aligned");
  GNN_REQUIRE(!Mb || (ldmb >= (F + 15) / 16 * 16 && ldmb % 8 == 0 && ((uintptr_t)Mb & 15) == 0),
              "gnn_spmm_fwd_noalloc: ldmb must be >= round_up(F,16), a multiple of 8, Mb 16-byte aligned");
  GNN_REQUIRE(!bnd || bnd->n_slots == 0 || (packed && meta),
              "gnn_spmm_fwd_noalloc: packed/meta required with a boundary");
  float* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != GNN_OK) return st;
  return launch_spmm_fwd(*csr, bnd, H, ldh, F, packed, reinterpret_cast<const float2*>(meta), M,
                         ldm, Mb, ldmb, scratch, as_stream(stream));
}

extern "C" gnn_status gnn_halo_quant_pack(const gnn_boundary* bnd, const float* G, int64_t ldg,
                                          int32_t F, uint32_t seed, uint8_t* packed, float* meta,
                                          gnn_stream_t stream) {
  GNN_REQUIRE(bnd, "gnn_halo_quant_pack: boundary is NULL");
  GNN_REQUIRE(F >= 1, "gnn_halo_quant_pack: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_halo_quant_pack: F=%d > %d", F, kMaxF);
  GNN_REQUIRE(bnd->F == F, "gnn_halo_quant_pack: boundary offsets are for F=%d, call has F=%d",
              bnd->F, F);
  if (bnd->n_slots == 0) return GNN_OK;
  GNN_REQUIRE(bnd->slot_rowptr && bnd->slot_bits && bnd->slot_off &&
                  (bnd->nnz_cut == 0 || (bnd->slot_col && bnd->slot_val)),
              "gnn_halo_quant_pack: boundary arrays are NULL");
  GNN_REQUIRE(bnd->long_slot_len == 0 ||
                  (bnd->long_slot_len >= 32 && bnd->n_long_slots >= 0 &&
                   (bnd->n_long_slots == 0 || bnd->long_slots)),
              "gnn_halo_quant_pack: incomplete long-slot list");
  GNN_REQUIRE(G && ldg >= F && ldg % 4 == 0 && ((uintptr_t)G & 15) == 0,
              "gnn_halo_quant_pack: ldg must be >= F, a multiple of 4, G 16-byte aligned");
  GNN_REQUIRE(packed && meta && ((uintptr_t)packed & 15) == 0 && ((uintptr_t)meta & 7) == 0,
              "gnn_halo_quant_pack: packed (16-byte aligned) and meta required");
  return launch_halo_quant_pack(*bnd, G, ldg, F, seed, packed, reinterpret_cast<float2*>(meta),
                                as_stream(stream));
}

extern "C" gnn_status gnn_halo_quant_pack_slots(const gnn_boundary* bnd, const float* G,
                                                int64_t ldg, int32_t F, int64_t s0, int64_t s1,
                                                uint32_t seed, uint8_t* packed, float* meta,
                                                gnn_stream_t stream) {
  GNN_REQUIRE(bnd, "gnn_halo_quant_pack_slots: boundary is NULL");
  GNN_REQUIRE(s0 >= 0 && s0 <= s1 && s1 <= bnd->n_slots,
              "gnn_halo_quant_pack_slots: need 0 <= s0 <= s1 <= n_slots");
  GNN_REQUIRE(F >= 1, "gnn_halo_quant_pack_slots: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_halo_quant_pack_slots: F=%d > %d", F, kMaxF);
  GNN_REQUIRE(bnd->F == F, "gnn_halo_quant_pack_slots: boundary offsets are for F=%d, call has F=%d",
              bnd->F, F);
  if (s1 == s0) return GNN_OK;
  GNN_REQUIRE(bnd->slot_rowptr && bnd->slot_bits && bnd->slot_off &&
                  (bnd->nnz_cut == 0 || (bnd->slot_col && bnd->slot_val)),
              "gnn_halo_quant_pack_slots: boundary arrays are NULL");
  GNN_REQUIRE(bnd->long_slot_len == 0 ||
                  (bnd->long_slot_len >= 32 && bnd->n_long_slots >= 0 &&
                   (bnd->n_long_slots == 0 || bnd->long_slots)),
              "gnn_halo_quant_pack_slots: incomplete long-slot list");
  GNN_REQUIRE(G && ldg >= F && ldg % 4 == 0 && ((uintptr_t)G & 15) == 0,
              "gnn_halo_quant_pack_slots: ldg must be >= F, a multiple of 4, G 16-byte aligned");
  GNN_REQUIRE(packed && meta && ((uintptr_t)packed & 15) == 0 && ((uintptr_t)meta & 7) == 0,
              "gnn_halo_quant_pack_slots: packed (16-byte aligned) and meta required");
  return launch_halo_quant_pack_ex(*bnd, G, ldg, F, seed, packed, reinterpret_cast<float2*>(meta),
                                   bnd->slot_val, nullptr, nullptr, as_stream(stream), s0, s1);
}

extern "C" gnn_status gnn_spmm_bwd_local(const gnn_csr* csr, const gnn_boundary* bnd,
                                         const float* G, int64_t ldg, int32_t F,
                                         const uint8_t* packed, const float* meta, float* dH,
                                         int64_t ldh, void* ws, size_t ws_bytes,
                                         gnn_stream_t stream) {
  gnn_status st = check_csr(csr, "gnn_spmm_bwd_local");
  if (st != GNN_OK) return st;
  GNN_REQUIRE(bnd, "gnn_spmm_bwd_local: boundary is NULL (use gnn_spmm_bwd)");
  GNN_REQUIRE(F >= 1, "gnn_spmm_bwd_local: F must be >= 1");
  if (F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_bwd_local: F=%d > %d", F, kMaxF);
  if (!csr->symmetric && !csr->val_t)
    return fail(GNN_ERR_UNSUPPORTED, "gnn_spmm_bwd_local: needs A^T (a symmetric CSR or val_t)");
  if ((st = check_bnd(csr, bnd, F, true, "gnn_spmm_bwd_local")) != GNN_OK) return st;
  if ((st = check_ws(csr, F, ws, ws_bytes, "gnn_spmm_bwd_local")) != GNN_OK) return st;
  if (csr->n == 0) return GNN_OK;
  GNN_REQUIRE(G && dH, "gnn_spmm_bwd_local: NULL G or dH");
  GNN_REQUIRE(ldg >= F && ldg % 4 == 0 && ((uintptr_t)G & 15) == 0,
              "gnn_spmm_bwd_local: ldg must be >= F, a multiple of 4, G 16-byte aligned");
  GNN_REQUIRE(ldh >= F && ldh % 4 == 0 && ((uintptr_t)dH & 15) == 0,
              "gnn_spmm_bwd_local: ldh must be >= F, a multiple of 4, dH 16-byte aligned");
  GNN_REQUIRE(bnd->n_slots == 0 || (packed && meta && ((uintptr_t)packed & 15) == 0),
              "gnn_spmm_bwd_local: packed (16-byte aligned) and meta required");
  return launch_spmm_bwd_local(*csr, *bnd, G, ldg, F, packed, reinterpret_cast<const float2*>(meta),
                               dH, ldh, static_cast<float*>(ws), as_stream(stream));
}
