// Cluster-blocked aggregation for community-ordered graphs (the layout idea
// of the TorchGT guide, "Cluster-aware Graph Parallelism": put the pairs of
// nodes with high locality next to each other) applied to the aggregation of
// the SYLVIE guide's section 2.
//
// The local entries are cut into T x T tiles (row block x column block).  A
// tile with at least min_entries entries is "dense": a thread block stages
// the tile's T source rows (a 128-column slice of them) in shared memory with
// bulk asynchronous copies, double-buffered on mbarriers, and every entry of
// the tile then reads its source row from shared memory instead of the
// memory system.  All other entries -- sparse tiles and the remote ones --
// form a residual CSR in the usual aggregation order, which the row kernels
// of spmm.cu aggregate first into an fp32 partial; the tile kernel adds the
// tiles to it in tile order and stores the result.
#include <cub/cub.cuh>
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"
#include "kernels.h"
#include "tc.cuh"

namespace gnn {
namespace {

constexpr int kTile = 128;         // T
constexpr int kSlice = 128;        // staged columns per block (floats)
constexpr int kTileThreads = 512;  // 16 warps, 8 rows each
constexpr int kWarps = kTileThreads / 32;
constexpr int kRowsPerWarp = kTile / kWarps;
constexpr size_t kStageBytes = (size_t)kTile * kSlice * sizeof(float);
// Entries of a tile row whose shared-memory rows are read before they are added.
#ifndef GNN_BLK_U
#define GNN_BLK_U 1
#endif
// A tile's metadata (row offsets, columns, weights) staged in shared memory
// one tile ahead; tiles with more entries read it from global memory.
constexpr int kMetaEntries = 4096;
struct MetaStage {
  int32_t trp[kTile + 4];
  float val[kMetaEntries];
  uint8_t col[kMetaEntries + 16];
};
constexpr size_t kSmemBytes = 2 * kStageBytes + 2 * sizeof(MetaStage);

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst)), "l"(src)
               : "memory");
}

#define GRIDB(count) (unsigned)(((count) + 255) / 256), 256

int bits_for(uint64_t x) {
  int b = 0;
  while ((uint64_t(1) << b) < x) ++b;
  return b < 1 ? 1 : b;
}

__device__ __forceinline__ int64_t warp_id() {
  return ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
}

// ---------------------------------------------------------------- plan build
__global__ void bl_local_count_kernel(int n, const int64_t* __restrict__ rowptr,
                                      const int32_t* __restrict__ lc, int64_t* __restrict__ cnt) {
  const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v > n) return;
  cnt[v] = v == n ? 0 : (lc ? (int64_t)lc[v] : rowptr[v + 1] - rowptr[v]);
}

// key = ((row block * nb + column block) << 16) | (row % T) << 8 | (col % T)
__global__ void bl_keys_kernel(int n, const int64_t* __restrict__ rowptr,
                               const int32_t* __restrict__ cr, const int64_t* __restrict__ loff,
                               int64_t nb, uint64_t* __restrict__ keys, int64_t* __restrict__ pay) {
  const int64_t v = warp_id();
  if (v >= n) return;
  const int lane = threadIdx.x & 31;
  const int64_t beg = rowptr[v], cnt = loff[v + 1] - loff[v], o = loff[v];
  const uint64_t rb = (uint64_t)(v / kTile), rin = (uint64_t)(v % kTile);
  for (int64_t j = lane; j < cnt; j += 32) {
    const int64_t k = beg + j;
    const int32_t c = cr[k];
    const uint64_t tile = rb * (uint64_t)nb + (uint64_t)(c / kTile);
    keys[o + j] = (tile << 16) | (rin << 8) | (uint64_t)(c % kTile);
    pay[o + j] = k;
  }
}

__global__ void bl_hi_kernel(int64_t m, const uint64_t* __restrict__ keys, uint64_t* __restrict__ hi) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < m) hi[i] = keys[i] >> 16;
}

__global__ void bl_flag_kernel(int64_t runs, const int64_t* __restrict__ cnt, int64_t min_entries,
                               uint8_t* __restrict__ flag, int64_t* __restrict__ cnt_tail) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < runs) flag[i] = cnt[i] >= min_entries ? 1 : 0;
  if (i == runs) cnt_tail[i] = 0;
}

// One block per dense tile: marks its entries and (with outputs) writes their
// columns, weights and the tile's row offsets.
__global__ void bl_tile_kernel(int64_t nd, const int64_t* __restrict__ doff,
                               const int64_t* __restrict__ dcnt, const uint64_t* __restrict__ keys,
                               const int64_t* __restrict__ pay, const float* __restrict__ val,
                               uint8_t* __restrict__ dense, const int64_t* __restrict__ tile_ptr,
                               uint8_t* __restrict__ ent_col, float* __restrict__ ent_val,
                               int32_t* __restrict__ tile_rowptr) {
  const int64_t t = blockIdx.x;
  if (t >= nd) return;
  const int64_t o = doff[t], c = dcnt[t];
  for (int64_t i = threadIdx.x; i < c; i += blockDim.x) {
    const int64_t k = pay[o + i];
    dense[k] = 1;
    if (ent_col) {
      ent_col[tile_ptr[t] + i] = (uint8_t)(keys[o + i] & 0xFF);
      ent_val[tile_ptr[t] + i] = val[k];
    }
  }
  if (tile_rowptr) {
    for (int r = threadIdx.x; r <= kTile; r += blockDim.x) {
      int64_t lo = 0, hi = c;  // first entry with row >= r
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int)((keys[o + mid] >> 8) & 0xFF) < r) lo = mid + 1;
        else hi = mid;
      }
      tile_rowptr[t * (kTile + 1) + r] = (int32_t)lo;
    }
  }
}

// Residual counts per row (all entries, and the local ones).
__global__ void bl_res_count_kernel(int n, const int64_t* __restrict__ rowptr,
                                    const int32_t* __restrict__ lc,
                                    const uint8_t* __restrict__ dense, int64_t* __restrict__ rcnt,
                                    int32_t* __restrict__ rlc) {
  const int64_t v = warp_id();
  const int lane = threadIdx.x & 31;
  if (v > n) return;
  if (v == n) {
    if (lane == 0) rcnt[n] = 0;
    return;
  }
  const int64_t beg = rowptr[v], end = rowptr[v + 1];
  const int64_t lend = lc ? beg + lc[v] : end;
  int d = 0;
  for (int64_t k = beg + lane; k < lend; k += 32) d += dense[k];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
  if (lane == 0) {
    rcnt[v] = (end - beg) - d;
    if (rlc) rlc[v] = (int32_t)((lend - beg) - d);
  }
}

// The residual entries of each row, in their original order (warp per row,
// ballot compaction).
__global__ void bl_res_fill_kernel(int n, const int64_t* __restrict__ rowptr,
                                   const int32_t* __restrict__ cr, const float* __restrict__ val,
                                   const uint8_t* __restrict__ dense,
                                   const int64_t* __restrict__ rrp, int32_t* __restrict__ rcol,
                                   float* __restrict__ rval) {
  const int64_t v = warp_id();
  if (v >= n) return;
  const int lane = threadIdx.x & 31;
  const int64_t beg = rowptr[v], end = rowptr[v + 1];
  int64_t at = rrp[v];
  for (int64_t base = beg; base < end; base += 32) {
    const int64_t k = base + lane;
    const bool keep = k < end && !dense[k];
    const uint32_t m = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int64_t p = at + __popc(m & ((1u << lane) - 1u));
      rcol[p] = cr[k];
      rval[p] = val[k];
    }
    at += __popc(m);
  }
}

__global__ void bl_rb_kernel(int n_rb, int64_t nd, const uint64_t* __restrict__ dtile, int64_t nb,
                             int64_t* __restrict__ rb_ptr, int32_t* __restrict__ tile_cb) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < nd) tile_cb[i] = (int32_t)(dtile[i] % (uint64_t)nb);
  if (i <= n_rb) {
    int64_t lo = 0, hi = nd;  // first tile of row block i
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if ((int64_t)(dtile[mid] / (uint64_t)nb) < i) lo = mid + 1;
      else hi = mid;
    }
    rb_ptr[i] = lo;
  }
}

struct PlanWs {
  int64_t *loff, *pay0, *pay1, *cnt, *run_off, *dcnt, *doff, *rcnt, *counters;
  uint64_t *keys0, *keys1, *hi, *uniq, *dtile;
  uint8_t *flag, *dense;
  void* temp;
  size_t temp_bytes;
  size_t bytes;
};

PlanWs plan_ws(void* base, size_t cap, int n, int64_t nnz, int64_t nl, bool* ok) {
  Arena ar(base, cap);
  PlanWs w{};
  const size_t m = (size_t)(nl > 0 ? nl : 1);
  w.loff = ar.take<int64_t>((size_t)n + 1);
  w.keys0 = ar.take<uint64_t>(m);
  w.keys1 = ar.take<uint64_t>(m);
  w.pay0 = ar.take<int64_t>(m);
  w.pay1 = ar.take<int64_t>(m);
  w.hi = ar.take<uint64_t>(m);
  w.uniq = ar.take<uint64_t>(m);
  w.cnt = ar.take<int64_t>(m + 1);
  w.run_off = ar.take<int64_t>(m + 1);
  w.flag = ar.take<uint8_t>(m);
  w.dtile = ar.take<uint64_t>(m);
  w.dcnt = ar.take<int64_t>(m + 1);
  w.doff = ar.take<int64_t>(m);
  w.dense = ar.take<uint8_t>((size_t)(nnz > 0 ? nnz : 1));
  w.rcnt = ar.take<int64_t>((size_t)n + 1);
  w.counters = ar.take<int64_t>(4);
  size_t t = 0, x = 0;
  cub::DeviceScan::ExclusiveSum(nullptr, x, (int64_t*)nullptr, (int64_t*)nullptr, (int64_t)n + 1);
  t = x > t ? x : t;
  cub::DeviceRadixSort::SortPairs(nullptr, x, (uint64_t*)nullptr, (uint64_t*)nullptr,
                                  (int64_t*)nullptr, (int64_t*)nullptr, (int64_t)m, 0, 64);
  t = x > t ? x : t;
  cub::DeviceRunLengthEncode::Encode(nullptr, x, (uint64_t*)nullptr, (uint64_t*)nullptr,
                                     (int64_t*)nullptr, (int64_t*)nullptr, (int64_t)m);
  t = x > t ? x : t;
  cub::DeviceScan::ExclusiveSum(nullptr, x, (int64_t*)nullptr, (int64_t*)nullptr, (int64_t)m + 1);
  t = x > t ? x : t;
  cub::DeviceSelect::Flagged(nullptr, x, (uint64_t*)nullptr, (uint8_t*)nullptr, (uint64_t*)nullptr,
                             (int64_t*)nullptr, (int64_t)m);
  t = x > t ? x : t;
  cub::DeviceSelect::Flagged(nullptr, x, (int64_t*)nullptr, (uint8_t*)nullptr, (int64_t*)nullptr,
                             (int64_t*)nullptr, (int64_t)m);
  t = x > t ? x : t;
  w.temp_bytes = t;
  w.temp = ar.take_bytes(t);
  w.bytes = ar.used;
  *ok = ar.ok();
  return w;
}

struct Source {
  const int32_t* cr;
  const float* val;
  const int32_t* lc;
};

Source source_of(const gnn_csr& csr, const gnn_boundary* bnd) {
  if (bnd) return Source{bnd->col_remap, bnd->val_remap, bnd->local_cnt};
  return Source{csr.col, csr.val, nullptr};
}

// Steps shared by counting and building: keys, sort, tiles, dense marks and
// residual counts.  Synchronises (the run and tile counts size the rest).
gnn_status plan_core(const gnn_csr& csr, const gnn_boundary* bnd, int64_t min_entries,
                     const PlanWs& w, int64_t* n_local, int64_t* n_tiles, int64_t* n_entries,
                     int64_t* n_res, int32_t* res_lc, cudaStream_t st) {
  const int n = csr.n;
  const Source src = source_of(csr, bnd);
  const int64_t nb = (n + kTile - 1) / kTile;
  size_t tb;
  bl_local_count_kernel<<<GRIDB((int64_t)n + 1), 0, st>>>(n, csr.rowptr, src.lc, w.cnt);
  GNN_CHECK_LAUNCH();
  tb = w.temp_bytes;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(w.temp, tb, w.cnt, w.loff, (int64_t)n + 1, st));
  int64_t nl = 0;
  GNN_CUDA(cudaMemcpyAsync(&nl, w.loff + n, sizeof(nl), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaStreamSynchronize(st));
  *n_local = nl;
  GNN_CUDA(cudaMemsetAsync(w.dense, 0, (size_t)(csr.nnz > 0 ? csr.nnz : 1), st));
  int64_t nd = 0;
  if (nl > 0) {
    bl_keys_kernel<<<(unsigned)(((int64_t)n * 32 + 255) / 256), 256, 0, st>>>(
        n, csr.rowptr, src.cr, w.loff, nb, w.keys0, w.pay0);
    GNN_CHECK_LAUNCH();
    const int end_bit = 16 + bits_for((uint64_t)nb * (uint64_t)nb);
    tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceRadixSort::SortPairs(w.temp, tb, w.keys0, w.keys1, w.pay0, w.pay1, nl, 0,
                                             end_bit, st));
    bl_hi_kernel<<<GRIDB(nl), 0, st>>>(nl, w.keys1, w.hi);
    GNN_CHECK_LAUNCH();
    tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceRunLengthEncode::Encode(w.temp, tb, w.hi, w.uniq, w.cnt, w.counters, nl, st));
    int64_t runs = 0;
    GNN_CUDA(cudaMemcpyAsync(&runs, w.counters, sizeof(runs), cudaMemcpyDeviceToHost, st));
    GNN_CUDA(cudaStreamSynchronize(st));
    bl_flag_kernel<<<GRIDB(runs + 1), 0, st>>>(runs, w.cnt, min_entries, w.flag, w.cnt);
    GNN_CHECK_LAUNCH();
    tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceScan::ExclusiveSum(w.temp, tb, w.cnt, w.run_off, runs + 1, st));
    tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceSelect::Flagged(w.temp, tb, w.uniq, w.flag, w.dtile, w.counters + 1, runs, st));
    tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceSelect::Flagged(w.temp, tb, w.cnt, w.flag, w.dcnt, w.counters + 1, runs, st));
    tb = w.temp_bytes;
    GNN_CUDA(cub::DeviceSelect::Flagged(w.temp, tb, w.run_off, w.flag, w.doff, w.counters + 1, runs, st));
    GNN_CUDA(cudaMemcpyAsync(&nd, w.counters + 1, sizeof(nd), cudaMemcpyDeviceToHost, st));
    GNN_CUDA(cudaStreamSynchronize(st));
  }
  *n_tiles = nd;
  int64_t ne = 0;
  if (nd > 0) {
    GNN_CUDA(cudaMemsetAsync(w.dcnt + nd, 0, sizeof(int64_t), st));
    tb = w.temp_bytes;
    // tile entry offsets land in w.run_off (its run offsets are no longer needed)
    GNN_CUDA(cub::DeviceScan::ExclusiveSum(w.temp, tb, w.dcnt, w.run_off, nd + 1, st));
    GNN_CUDA(cudaMemcpyAsync(&ne, w.run_off + nd, sizeof(ne), cudaMemcpyDeviceToHost, st));
    bl_tile_kernel<<<(unsigned)nd, 256, 0, st>>>(nd, w.doff, w.dcnt, w.keys1, w.pay1, src.val,
                                                 w.dense, nullptr, nullptr, nullptr, nullptr);
    GNN_CHECK_LAUNCH();
  }
  bl_res_count_kernel<<<(unsigned)((((int64_t)n + 1) * 32 + 255) / 256), 256, 0, st>>>(
      n, csr.rowptr, src.lc, w.dense, w.rcnt, res_lc);
  GNN_CHECK_LAUNCH();
  tb = w.temp_bytes;
  GNN_CUDA(cub::DeviceScan::ExclusiveSum(w.temp, tb, w.rcnt, w.loff, (int64_t)n + 1, st));
  int64_t nr = 0;
  GNN_CUDA(cudaMemcpyAsync(&nr, w.loff + n, sizeof(nr), cudaMemcpyDeviceToHost, st));
  GNN_CUDA(cudaStreamSynchronize(st));
  *n_entries = ne;
  *n_res = nr;
  return GNN_OK;
}

gnn_status check_plan_args(const gnn_csr* csr, const gnn_boundary* bnd, int32_t T,
                           int32_t min_entries, const char* who) {
  if (!csr || csr->n < 1 || !csr->rowptr || (csr->nnz > 0 && (!csr->col || !csr->val)))
    return fail(GNN_ERR_INVALID_ARG, "%s: invalid csr", who);
  if (T != kTile) return fail(GNN_ERR_UNSUPPORTED, "%s: tile edge T must be %d", who, kTile);
  if (min_entries < 1) return fail(GNN_ERR_INVALID_ARG, "%s: min_entries must be >= 1", who);
  if (!csr->symmetric)
    return fail(GNN_ERR_UNSUPPORTED, "%s: needs symmetric weights (A = A^T)", who);
  if (bnd && (bnd->n != csr->n || !bnd->col_remap || !bnd->val_remap || !bnd->local_cnt))
    return fail(GNN_ERR_INVALID_ARG, "%s: boundary does not match csr", who);
  return GNN_OK;
}

// ---------------------------------------------------------------- tile kernel
struct TilesDev {
  int n;
  const int64_t* rb_ptr;
  const int32_t* tile_cb;
  const int64_t* tile_ptr;
  const int32_t* tile_rowptr;
  const uint8_t* ent_col;
  const float* ent_val;
};

// Block (row block rb, column slice s): acc = the row block's dense tiles, in
// order, over columns [128 s, 128 s + 128); out = R + acc (fp32 and/or bf16,
// optional gate by hmask > 0).  Warp w owns rows w + 16 i.  Thread 0 posts
// each tile's byte count on the stage's mbarrier and warp 0 issues one bulk
// copy per source row; the next tile's copies fly while this one is summed.
__global__ void __launch_bounds__(kTileThreads, 1) blocked_tiles_kernel(
    TilesDev tp, const float* __restrict__ X, int64_t ldx, int F, const float* __restrict__ R,
    int64_t ldr, float* __restrict__ M, int64_t ldm, __nv_bfloat16* __restrict__ Mb,
    int64_t ldmb, int nch_b, const float* __restrict__ hmask, int64_t ldhm,
    unsigned* __restrict__ flags) {
  extern __shared__ __align__(128) float4 stage4[];
  __shared__ __align__(8) uint64_t full[2];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rb = blockIdx.x, s = blockIdx.y;
  const int64_t v0 = (int64_t)rb * kTile;
  const int nrows = (int)min((int64_t)kTile, (int64_t)tp.n - v0);
  const int col0 = s * kSlice;                       // first column of the slice
  const int64_t width = min((int64_t)kSlice, ldx - col0);  // staged floats per row
  const int nchunk = width > 0 ? (int)(width >> 2) : 0;
  const int nch = (F + 3) >> 2;
  const int cg = s * (kSlice / 4) + lane;            // this lane's global chunk
  const int64_t t0 = tp.rb_ptr[rb], t1 = tp.rb_ptr[rb + 1];
  if (threadIdx.x == 0) {
    tc::mbar_init(&full[0], 1);
    tc::mbar_init(&full[1], 1);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();

  MetaStage* meta = reinterpret_cast<MetaStage*>(reinterpret_cast<char*>(stage4) + 2 * kStageBytes);
  // all threads: this tile's metadata into meta[ms] (4-byte asynchronous copies)
  auto issue_meta = [&](int64_t t, int ms) {
    const int64_t eb = tp.tile_ptr[t], ne = tp.tile_ptr[t + 1] - eb;
    if (ne <= kMetaEntries) {
      MetaStage& m = meta[ms];
      for (int i = threadIdx.x; i <= kTile; i += kTileThreads)
        cp_async4(&m.trp[i], tp.tile_rowptr + t * (kTile + 1) + i);
      for (int64_t i = threadIdx.x; i < ne; i += kTileThreads) cp_async4(&m.val[i], tp.ent_val + eb + i);
      const int64_t c0 = eb & ~(int64_t)3;
      const int64_t nw = (eb + ne - c0 + 3) >> 2;
      for (int64_t i = threadIdx.x; i < nw; i += kTileThreads)
        cp_async4(&m.col[4 * i], tp.ent_col + c0 + 4 * i);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  auto issue = [&](int64_t t, int st) {  // warp 0
    const int cb = tp.tile_cb[t];
    const int64_t u0 = (int64_t)cb * kTile;
    const int rows = (int)min((int64_t)kTile, (int64_t)tp.n - u0);
    const uint32_t bytes = (uint32_t)(width * 4);
    if (lane == 0) tc::mbar_expect_tx(&full[st], bytes * (uint32_t)rows);
    __syncwarp();
    float4* dst0 = stage4 + (size_t)st * (kStageBytes / 16);
    for (int j = lane; j < rows; j += 32) {
      const float* src = X + (u0 + j) * ldx + col0;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              tc::smem_u32(dst0 + (size_t)j * (kSlice / 4))),
          "l"(src), "r"(bytes), "r"(tc::smem_u32(&full[st]))
          : "memory");
    }
  };

  float4 acc[kRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (warp == 0 && t0 < t1 && nchunk > 0) issue(t0, 0);
  if (t0 < t1 && nchunk > 0) {
    issue_meta(t0, 0);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
  }
  int64_t issued = (t0 < t1 && nchunk > 0) ? t0 + 1 : t0;
  int64_t failed = -1;
  for (int64_t t = t0; t < t1 && nchunk > 0; ++t) {
    const int st = (int)((t - t0) & 1);
    const uint32_t ph = (uint32_t)(((t - t0) >> 1) & 1);
    if (warp == 0 && t + 1 < t1) issue(t + 1, st ^ 1);
    if (t + 1 < t1) {
      issued = t + 2;
      issue_meta(t + 1, st ^ 1);
    }
    // every thread leaves together if any wait gave up (no one left at a barrier)
    const bool got = tc::mbar_wait(&full[st], ph, flags, &abort_flag);
    if (!__syncthreads_and(got)) {
      failed = t;
      break;
    }
    const float4* stg = stage4 + (size_t)st * (kStageBytes / 16);
    const int64_t eb = tp.tile_ptr[t];
    const bool staged = tp.tile_ptr[t + 1] - eb <= kMetaEntries;
    const int32_t* trp = staged ? meta[st].trp : tp.tile_rowptr + t * (kTile + 1);
    const float* ev = staged ? meta[st].val : tp.ent_val + eb;
    const uint8_t* ec = staged ? meta[st].col + (eb & 3) : tp.ent_col + eb;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int r = warp + kWarps * i;
      if (r >= nrows) continue;
      const int b = trp[r], e = trp[r + 1];
      for (int base = b; base < e; base += 32) {
        const int k = base + lane;
        int c = 0;
        float w = 0.f;
        if (k < e) {
          c = ec[k];
          w = ev[k];
        }
        const int cnt = min(32, e - base);
        for (int q = 0; q < cnt; q += GNN_BLK_U) {
          float4 x[GNN_BLK_U];
          float wq[GNN_BLK_U];
#pragma unroll
          for (int u = 0; u < GNN_BLK_U; ++u) {  // the round's shared loads first
            const bool valid = q + u < cnt;
            const int src = valid ? q + u : q;
            const int cq = __shfl_sync(0xffffffffu, c, src);
            wq[u] = valid ? __shfl_sync(0xffffffffu, w, src) : 0.f;
            x[u] = lane < nchunk ? stg[(size_t)cq * (kSlice / 4) + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < GNN_BLK_U; ++u) fma4(acc[i], wq[u], x[u]);
        }
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // the next tile's metadata is in
    __syncthreads();  // and this tile's stages are free for the tile after next
  }
  if (failed >= 0) {
    // wait (bounded) for this block's copies still in flight, then leave
    asm volatile("cp.async.wait_all;" ::: "memory");
    abort_flag = 0;
    __syncthreads();
    for (int64_t t = failed; t < issued; ++t) {
      const int st = (int)((t - t0) & 1);
      const uint32_t ph = (uint32_t)(((t - t0) >> 1) & 1);
      tc::mbar_wait(&full[st], ph, flags, &abort_flag);
    }
    return;
  }
  // out = R + acc
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int r = warp + kWarps * i;
    if (r >= nrows) continue;
    const int64_t v = v0 + r;
    float4 x = acc[i];
    if (cg < nch) {
      add4(x, __ldg(reinterpret_cast<const float4*>(R + v * ldr) + cg));
      if (hmask) {
        const float4 h = __ldg(reinterpret_cast<const float4*>(hmask + v * ldhm) + cg);
        if (!(h.x > 0.f)) x.x = 0.f;
        if (!(h.y > 0.f)) x.y = 0.f;
        if (!(h.z > 0.f)) x.z = 0.f;
        if (!(h.w > 0.f)) x.w = 0.f;
      }
      if (M) store_chunk_f32(M + v * ldm, cg, F, x);
    }
    if (Mb && cg < nch_b) store_chunk_bf16(Mb + v * ldmb, cg, F, cg < nch ? x : make_float4(0.f, 0.f, 0.f, 0.f));
  }
}

struct BlockedRun {
  float* R;
  float* partial;
  size_t bytes;
};

BlockedRun blocked_ws(void* base, size_t cap, const gnn_blocked& bp, int n, int F, bool* ok) {
  Arena ar(base, cap);
  BlockedRun w{};
  w.R = ar.take<float>((size_t)n * (size_t)((F + 3) / 4 * 4));
  const size_t sp = spmm_workspace_bytes(bp.residual, F);
  w.partial = sp ? reinterpret_cast<float*>(ar.take_bytes(sp)) : nullptr;
  w.bytes = ar.used;
  *ok = ar.ok();
  return w;
}

gnn_status launch_tiles(const gnn_blocked& bp, const float* X, int64_t ldx, int F, const float* R,
                        int64_t ldr, float* M, int64_t ldm, uint16_t* Mb, int64_t ldmb, int nch_b,
                        const float* hmask, int64_t ldhm, cudaStream_t st) {
  const int nch = (F + 3) / 4;
  const int need = nch_b > nch ? nch_b : nch;
  const int slices = (need + (kSlice / 4) - 1) / (kSlice / 4);
  const size_t smem = kSmemBytes;
  static bool attr = false;
  if (!attr) {
    GNN_CUDA(cudaFuncSetAttribute(blocked_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem));
    attr = true;
  }
  unsigned* flags = device_flags();
  if (!flags) return fail(GNN_ERR_CUDA, "blocked aggregation: device flag word unavailable");
  TilesDev tp{bp.residual.n, bp.rb_tile_ptr, bp.tile_cb, bp.tile_ptr, bp.tile_rowptr, bp.ent_col,
              bp.ent_val};
  blocked_tiles_kernel<<<dim3((unsigned)bp.n_rb, (unsigned)slices), kTileThreads, smem, st>>>(
      tp, X, ldx, F, R, ldr, M, ldm, reinterpret_cast<__nv_bfloat16*>(Mb), ldmb, nch_b, hmask,
      ldhm, flags);
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

gnn_status check_blocked(const gnn_csr* csr, const gnn_boundary* bnd, const gnn_blocked* bp,
                         int F, const char* who) {
  if (!csr || !bp || bp->T != kTile || bp->residual.n != csr->n ||
      bp->n_rb != (csr->n + kTile - 1) / kTile || !bp->rb_tile_ptr || !bp->residual.rowptr ||
      (bp->n_tiles > 0 && (!bp->tile_cb || !bp->tile_ptr || !bp->tile_rowptr)) ||
      (bp->n_entries > 0 && (!bp->ent_col || !bp->ent_val)) ||
      (bp->residual.nnz > 0 && (!bp->residual.col || !bp->residual.val)) ||
      (bnd && !bp->res_local_cnt))
    return fail(GNN_ERR_INVALID_ARG, "%s: plan does not match the csr/boundary", who);
  if (!csr->symmetric) return fail(GNN_ERR_UNSUPPORTED, "%s: needs symmetric weights", who);
  if (F < 1 || F > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "%s: F=%d", who, F);
  if (bnd && bnd->F != F)
    return fail(GNN_ERR_INVALID_ARG, "%s: boundary offsets are for F=%d, call has F=%d", who, bnd->F, F);
  return GNN_OK;
}

}  // namespace
}  // namespace gnn

using namespace gnn;

extern "C" gnn_status gnn_blocked_workspace(const gnn_csr* csr, const gnn_boundary* bnd,
                                            int32_t T, int32_t min_entries, size_t* ws_bytes) {
  gnn_status s = check_plan_args(csr, bnd, T, min_entries, "gnn_blocked_workspace");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(ws_bytes, "gnn_blocked_workspace: NULL ws_bytes");
  bool ok;
  *ws_bytes = plan_ws(nullptr, 0, csr->n, csr->nnz, csr->nnz, &ok).bytes;
  return GNN_OK;
}

extern "C" gnn_status gnn_blocked_count(const gnn_csr* csr, const gnn_boundary* bnd, int32_t T,
                                        int32_t min_entries, int64_t* n_tiles, int64_t* n_entries,
                                        int64_t* n_residual, void* ws, size_t ws_bytes,
                                        gnn_stream_t stream) {
  gnn_status s = check_plan_args(csr, bnd, T, min_entries, "gnn_blocked_count");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(n_tiles && n_entries && n_residual, "gnn_blocked_count: NULL output");
  bool ok;
  PlanWs w = plan_ws(ws, ws_bytes, csr->n, csr->nnz, csr->nnz, &ok);
  GNN_REQUIRE(ws && ok, "gnn_blocked_count: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  int64_t nl;
  return plan_core(*csr, bnd, min_entries, w, &nl, n_tiles, n_entries, n_residual, nullptr,
                   as_stream(stream));
}

extern "C" gnn_status gnn_blocked_build(const gnn_csr* csr, const gnn_boundary* bnd, int32_t T,
                                        int32_t min_entries, gnn_blocked* out, void* ws,
                                        size_t ws_bytes, gnn_stream_t stream) {
  gnn_status s = check_plan_args(csr, bnd, T, min_entries, "gnn_blocked_build");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(out && out->rb_tile_ptr && out->residual.rowptr && (!bnd || out->res_local_cnt),
              "gnn_blocked_build: output arrays missing");
  bool ok;
  PlanWs w = plan_ws(ws, ws_bytes, csr->n, csr->nnz, csr->nnz, &ok);
  GNN_REQUIRE(ws && ok, "gnn_blocked_build: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  cudaStream_t st = as_stream(stream);
  const int n = csr->n;
  const int64_t nb = (n + kTile - 1) / kTile;
  int64_t nl, nd, ne, nr;
  s = plan_core(*csr, bnd, min_entries, w, &nl, &nd, &ne, &nr, bnd ? out->res_local_cnt : nullptr, st);
  if (s != GNN_OK) return s;
  GNN_REQUIRE(out->n_tiles == nd && out->n_entries == ne && out->residual.nnz == nr,
              "gnn_blocked_build: sizes differ from gnn_blocked_count's");
  GNN_REQUIRE((nd == 0 || (out->tile_cb && out->tile_ptr && out->tile_rowptr)) &&
                  (ne == 0 || (out->ent_col && out->ent_val)) &&
                  (nr == 0 || (out->residual.col && out->residual.val)),
              "gnn_blocked_build: output arrays missing");
  out->T = kTile;
  out->n_rb = (int32_t)nb;
  const Source src = source_of(*csr, bnd);
  if (nd > 0) {
    // tile entry offsets (left in w.run_off by plan_core)
    GNN_CUDA(cudaMemcpyAsync(out->tile_ptr, w.run_off, (size_t)(nd + 1) * sizeof(int64_t),
                             cudaMemcpyDeviceToDevice, st));
    bl_tile_kernel<<<(unsigned)nd, 256, 0, st>>>(nd, w.doff, w.dcnt, w.keys1, w.pay1, src.val,
                                                 w.dense, out->tile_ptr, out->ent_col, out->ent_val,
                                                 out->tile_rowptr);
    GNN_CHECK_LAUNCH();
  }
  bl_rb_kernel<<<GRIDB(nd > nb + 1 ? nd : nb + 1), 0, st>>>((int)nb, nd, w.dtile, nb,
                                                            out->rb_tile_ptr, out->tile_cb);
  GNN_CHECK_LAUNCH();
  // residual CSR: row offsets (in w.loff) and entries in their order
  GNN_CUDA(cudaMemcpyAsync(out->residual.rowptr, w.loff, (size_t)(n + 1) * sizeof(int64_t),
                           cudaMemcpyDeviceToDevice, st));
  if (nr > 0) {
    bl_res_fill_kernel<<<(unsigned)(((int64_t)n * 32 + 255) / 256), 256, 0, st>>>(
        n, csr->rowptr, src.cr, src.val, w.dense, w.loff, out->residual.col, out->residual.val);
    GNN_CHECK_LAUNCH();
  }
  out->residual.n = n;
  out->residual.symmetric = 0;
  out->residual.nnz = nr;
  GNN_CUDA(cudaStreamSynchronize(st));
  return GNN_OK;
}

extern "C" gnn_status gnn_blocked_spmm_workspace(const gnn_blocked* bp, int32_t F,
                                                 size_t* ws_bytes) {
  GNN_REQUIRE(bp && ws_bytes && F >= 1, "gnn_blocked_spmm_workspace: bad arguments");
  bool ok;
  *ws_bytes = blocked_ws(nullptr, 0, *bp, bp->residual.n, F, &ok).bytes;
  return GNN_OK;
}

extern "C" gnn_status gnn_spmm_fwd_blocked(const gnn_csr* csr, const gnn_boundary* bnd,
                                           const gnn_blocked* bp, const float* H, int64_t ldh,
                                           int32_t F, const uint8_t* packed, const float* meta,
                                           float* M, int64_t ldm, uint16_t* Mb, int64_t ldmb,
                                           void* ws, size_t ws_bytes, gnn_stream_t stream) {
  gnn_status s = check_blocked(csr, bnd, bp, F, "gnn_spmm_fwd_blocked");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(H && (M || Mb), "gnn_spmm_fwd_blocked: H is NULL or no output given");
  GNN_REQUIRE(ldh >= F && ldh % 4 == 0 && ((uintptr_t)H & 15) == 0, "gnn_spmm_fwd_blocked: bad H");
  GNN_REQUIRE(!M || (ldm >= F && ldm % 4 == 0 && ((uintptr_t)M & 15) == 0), "gnn_spmm_fwd_blocked: bad M");
  GNN_REQUIRE(!Mb || (ldmb >= (F + 15) / 16 * 16 && ldmb % 8 == 0 && ((uintptr_t)Mb & 15) == 0),
              "gnn_spmm_fwd_blocked: bad Mb");
  GNN_REQUIRE(!bnd || bnd->n_slots == 0 || (packed && meta), "gnn_spmm_fwd_blocked: messages required");
  bool ok;
  BlockedRun w = blocked_ws(ws, ws_bytes, *bp, csr->n, F, &ok);
  GNN_REQUIRE(ws && ok, "gnn_spmm_fwd_blocked: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  cudaStream_t st = as_stream(stream);
  const int64_t ldr = (F + 3) / 4 * 4;
  // residual (sparse tiles and remote entries) into the fp32 partial R
  gnn_boundary rb = bnd ? *bnd : gnn_boundary{};
  if (bnd) {
    rb.col_remap = bp->residual.col;
    rb.val_remap = bp->residual.val;
    rb.local_cnt = bp->res_local_cnt;
  }
  s = launch_spmm_fwd(bp->residual, bnd ? &rb : nullptr, H, ldh, F, packed,
                      reinterpret_cast<const float2*>(meta), w.R, ldr, nullptr, 0, w.partial, st);
  if (s != GNN_OK) return s;
  const int nch_b = Mb ? (F + 15) / 16 * 4 : 0;
  return launch_tiles(*bp, H, ldh, F, w.R, ldr, M, ldm, Mb, ldmb, nch_b, nullptr, 0, st);
}

extern "C" gnn_status gnn_spmm_bwd_blocked(const gnn_csr* csr, const gnn_boundary* bnd,
                                           const gnn_blocked* bp, const float* G, int64_t ldg,
                                           int32_t F, uint32_t seed, uint8_t* packed_ws,
                                           float* meta_ws, const float* H_mask, int64_t ldhm,
                                           float* dH, int64_t ldh, uint16_t* dZ, int64_t ldz,
                                           void* ws, size_t ws_bytes, gnn_stream_t stream) {
  gnn_status s = check_blocked(csr, bnd, bp, F, "gnn_spmm_bwd_blocked");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(G && (dH || dZ), "gnn_spmm_bwd_blocked: G is NULL or no output given");
  GNN_REQUIRE(ldg >= F && ldg % 4 == 0 && ((uintptr_t)G & 15) == 0, "gnn_spmm_bwd_blocked: bad G");
  GNN_REQUIRE(!dH || (ldh >= F && ldh % 4 == 0 && ((uintptr_t)dH & 15) == 0), "gnn_spmm_bwd_blocked: bad dH");
  GNN_REQUIRE(!dZ || (ldz >= (F + 63) / 64 * 64 && ldz % 8 == 0 && ((uintptr_t)dZ & 15) == 0),
              "gnn_spmm_bwd_blocked: dZ needs ldz >= round_up(F, 64)");
  GNN_REQUIRE(!H_mask || (ldhm >= F && ldhm % 4 == 0 && ((uintptr_t)H_mask & 15) == 0),
              "gnn_spmm_bwd_blocked: bad H_mask");
  GNN_REQUIRE(!bnd || bnd->n_slots == 0 ||
                  (packed_ws && meta_ws && ((uintptr_t)packed_ws & 15) == 0 && ((uintptr_t)meta_ws & 7) == 0 &&
                   bnd->own_ptr && bnd->own_slot && bnd->slot_rowptr),
              "gnn_spmm_bwd_blocked: message buffers required with a boundary");
  bool ok;
  BlockedRun w = blocked_ws(ws, ws_bytes, *bp, csr->n, F, &ok);
  GNN_REQUIRE(ws && ok, "gnn_spmm_bwd_blocked: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  cudaStream_t st = as_stream(stream);
  const int64_t ldr = (F + 3) / 4 * 4;
  if (bnd) {
    // backward messages (unchanged), then the residual with the owned adds
    s = launch_halo_quant_pack(*bnd, G, ldg, F, seed, packed_ws, reinterpret_cast<float2*>(meta_ws), st);
    if (s != GNN_OK) return s;
    gnn_boundary rb = *bnd;
    rb.col_remap = bp->residual.col;
    rb.val_remap = bp->residual.val;
    rb.val_remap_t = nullptr;
    rb.local_cnt = bp->res_local_cnt;
    s = launch_spmm_bwd_local(bp->residual, rb, G, ldg, F, packed_ws,
                              reinterpret_cast<const float2*>(meta_ws), w.R, ldr, w.partial, st);
  } else {
    s = launch_spmm_fwd(bp->residual, nullptr, G, ldg, F, nullptr, nullptr, w.R, ldr, nullptr, 0,
                        w.partial, st);
  }
  if (s != GNN_OK) return s;
  if (dH) {
    s = launch_tiles(*bp, G, ldg, F, w.R, ldr, dH, ldh, nullptr, 0, 0, dZ ? nullptr : H_mask,
                     ldhm, st);
    if (s != GNN_OK || !dZ) return s;
  }
  return launch_tiles(*bp, G, ldg, F, w.R, ldr, nullptr, 0, dZ, ldz, (int)(ldz / 4), H_mask, ldhm,
                      st);
}
