// Dense transform of the GCN layer on tcgen05 tensor cores (SYLVIE guide,
// section 2: z = W h after aggregation; section 7: the weight gradient).
//
//   gemm_tn:   C[M x N] = A[M x K] * B[N x K]^T, A and B bf16 with K contiguous
//              ("K-major"), fp32 accumulate in TMEM, fp32 out, optional ReLU.
//              Used for Z = Mb W (B = W^T) and dM = dZ W^T (B = W).
//   gemm_mn:   C[Mi x Nj] = sum_k A[k, i] B[k, j] with A, B bf16 row-major
//              (i, j contiguous: "MN-major"), split over k into fp32 partial
//              tiles that a second kernel adds in fixed order.  Used for
//              dW = Mb^T dZ, the reduction over all nodes.
//
// Both kernels are persistent and warp-specialised (192 threads): warp 0
// issues TMA tile loads into a 4-stage ring of 128-byte-swizzled shared
// memory tiles, warp 1 allocates TMEM and issues tcgen05.mma from one thread,
// warps 2-5 drain the accumulator (TMEM -> registers -> global).  Two TMEM
// accumulators let the drain of one tile overlap the MMAs of the next.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "gemm.h"
#include "tc.cuh"

namespace gnn {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;           // 16 KB
constexpr int B_STAGE = 256 * BK * 2;          // 32 KB (N tile up to 256)
constexpr int OUT_SUB = 32 * 32 * 4;           // one epilogue warp's 32 x 32 fp32 sub-tile
constexpr int OUT_STAGE = 4 * 2 * OUT_SUB;     // 4 warps, double-buffered: 32 KB
constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) + 1024 /*barriers*/ + 1024 /*align*/;
constexpr int SMEM_TN_BYTES = SMEM_BYTES + OUT_STAGE;
constexpr int THREADS = 192;

struct Smem {
  uint8_t* a;
  uint8_t* b;
  uint8_t* out;  // epilogue staging (gemm_tn only), 1024-byte aligned
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint32_t* tmem_base;
  volatile int* abort_flag;
};

__device__ __forceinline__ Smem carve(uint8_t* raw) {
  Smem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.a = base;
  s.b = base + STAGES * A_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.b + STAGES * B_STAGE);
  s.full = bars;
  s.empty = bars + STAGES;
  s.tfull = bars + 2 * STAGES;
  s.tempty = bars + 2 * STAGES + 2;
  s.tmem_base = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_base + 1);
  s.out = s.b + STAGES * B_STAGE + 1024;
  return s;
}

__device__ __forceinline__ uint32_t tmem_cols_for(int BN) {
  uint32_t c = 32;
  while (c < (uint32_t)(2 * BN)) c <<= 1;
  return c;
}

__device__ __forceinline__ void setup_ctas(const Smem& s, int BN) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(&s.full[i], 1);
      tc::mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s.tfull[i], 1);
      tc::mbar_init(&s.tempty[i], 128);
    }
    *s.abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(s.tmem_base, tmem_cols_for(BN));
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

__device__ __forceinline__ void teardown(const Smem& s, int BN, uint32_t tmem) {
  tc::fence_before_sync();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tmem_cols_for(BN));
  }
}

}  // namespace

struct TnArgs {
  int M, N, K, BN;
  int n_store;  // output columns written per row (multiple of 4, <= ldo)
  float* out;
  int64_t ldo;
  int relu;
  unsigned* flags;
};

__global__ void __launch_bounds__(THREADS, 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, TnArgs g) {
  extern __shared__ uint8_t smem_raw[];
  const Smem s = carve(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BN = g.BN;
  setup_ctas(s, BN);
  const uint32_t tmem = *s.tmem_base;
  const int num_m = (g.M + BM - 1) / BM;
  const int num_n = (g.N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int num_kb = (g.K + BK - 1) / BK;

  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
    int st = 0;
    uint32_t ph = 0;
    const uint32_t bytes = A_STAGE + BN * BK * 2;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      const int m0 = (t % num_m) * BM, n0 = (t / num_m) * BN;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!tc::mbar_wait(&s.empty[st], ph ^ 1, g.flags, s.abort_flag)) goto done;
        tc::mbar_expect_tx(&s.full[st], bytes);
        tc::tma_load_2d(s.a + st * A_STAGE, &tmA, &s.full[st], kb * BK, m0);
        tc::tma_load_2d(s.b + st * B_STAGE, &tmB, &s.full[st], kb * BK, n0);
        if (++st == STAGES) { st = 0; ph ^= 1; }
      }
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = tc::idesc_bf16(BM, BN, false, false);
    int st = 0;
    uint32_t ph = 0;
    int it = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!tc::mbar_wait(&s.tempty[acc], aph ^ 1, g.flags, s.abort_flag)) goto done;
      tc::fence_after_sync();
      const uint32_t d = tmem + acc * BN;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!tc::mbar_wait(&s.full[st], ph, g.flags, s.abort_flag)) goto done;
        tc::fence_after_sync();
        const uint32_t a0 = tc::smem_u32(s.a + st * A_STAGE);
        const uint32_t b0 = tc::smem_u32(s.b + st * B_STAGE);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          tc::mma_bf16(d, tc::sw128_desc(a0 + k * 32, 16), tc::sw128_desc(b0 + k * 32, 16), idesc,
                       (kb | k) ? 1u : 0u);
        tc::mma_commit(&s.empty[st]);
        if (++st == STAGES) { st = 0; ph ^= 1; }
      }
      tc::mma_commit(&s.tfull[acc]);
    }
  } else if (warp >= 2) {
    // Each epilogue warp owns 32 accumulator rows (its TMEM lane quarter).
    // Per 32-column chunk: TMEM -> registers (ReLU) -> a 128-byte-swizzled
    // 32 x 32 fp32 sub-tile in shared memory -> one TMA store (rows and
    // columns outside the output are clipped by the tensor map).  Two
    // staging buffers per warp let a store drain while the next fills.
    const int q = warp & 3;
    uint8_t* stage0 = s.out + (warp - 2) * 2 * OUT_SUB;
    int it = 0, nbuf = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
      const int m0 = (t % num_m) * BM, n0 = (t / num_m) * BN;
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!tc::mbar_wait(&s.tfull[acc], aph, g.flags, s.abort_flag)) goto done;
      tc::fence_after_sync();
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + acc * BN + c0, *reinterpret_cast<float(*)[16]>(v));
        if (c0 + 16 < BN)
          tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + acc * BN + c0 + 16,
                        *reinterpret_cast<float(*)[16]>(v + 16));
        else {
#pragma unroll
          for (int j = 16; j < 32; ++j) v[j] = 0.f;
        }
        if (c0 + 32 >= BN) {  // accumulator fully read: hand it back to the MMA warp
          tc::fence_before_sync();
          tc::mbar_arrive(&s.tempty[acc]);
        }
        if (g.relu) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j], 0.f);
        }
        uint8_t* stage = stage0 + nbuf * OUT_SUB;
        if (lane == 0) tc::bulk_wait_read<1>();  // this buffer's previous store has read it
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<float4*>(stage + lane * 128 + ((k ^ (lane & 7)) << 4)) =
              make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        tc::fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::tma_store_2d(&tmC, stage, n0 + c0, m0 + q * 32);
          tc::bulk_commit();
        }
        nbuf ^= 1;
      }
    }
  }
done:
  if (warp >= 2 && lane == 0) tc::bulk_wait_all();  // stores finish before the block exits
  teardown(s, BN, tmem);
}

struct MnArgs {
  int Mi, Nj, K;   // output rows (A columns), output columns (B columns), reduction length
  int BN;          // multiple of 64
  int kb_per_split, splits;
  float* part;     // [splits][num_mt*128][num_nt*BN]
  unsigned* flags;
};

__global__ void __launch_bounds__(THREADS, 1)
    gemm_mn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   MnArgs g) {
  extern __shared__ uint8_t smem_raw[];
  const Smem s = carve(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BN = g.BN;
  setup_ctas(s, BN);
  const uint32_t tmem = *s.tmem_base;
  const int num_mt = (g.Mi + BM - 1) / BM;
  const int num_nt = (g.Nj + BN - 1) / BN;
  const int units = num_mt * num_nt * g.splits;
  const int num_kb = (g.K + BK - 1) / BK;
  const int ldp = num_nt * BN;
  constexpr int BOX = BK * 128;  // one 64-wide MN block of BK rows: 8 KB

  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
    int st = 0;
    uint32_t ph = 0;
    const uint32_t bytes = 2 * BOX + (BN / 64) * BOX;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int mt = u % num_mt, nt = (u / num_mt) % num_nt, ks = u / (num_mt * num_nt);
      const int kb0 = ks * g.kb_per_split;
      const int kb1 = min(num_kb, kb0 + g.kb_per_split);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!tc::mbar_wait(&s.empty[st], ph ^ 1, g.flags, s.abort_flag)) goto done;
        tc::mbar_expect_tx(&s.full[st], bytes);
        for (int j = 0; j < 2; ++j)
          tc::tma_load_2d(s.a + st * A_STAGE + j * BOX, &tmA, &s.full[st], mt * BM + 64 * j, kb * BK);
        for (int j = 0; j < BN / 64; ++j)
          tc::tma_load_2d(s.b + st * B_STAGE + j * BOX, &tmB, &s.full[st], nt * BN + 64 * j, kb * BK);
        if (++st == STAGES) { st = 0; ph ^= 1; }
      }
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = tc::idesc_bf16(BM, BN, true, true);
    int st = 0;
    uint32_t ph = 0;
    int it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
      const int ks = u / (num_mt * num_nt);
      const int kb0 = ks * g.kb_per_split;
      const int kb1 = min(num_kb, kb0 + g.kb_per_split);
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!tc::mbar_wait(&s.tempty[acc], aph ^ 1, g.flags, s.abort_flag)) goto done;
      tc::fence_after_sync();
      const uint32_t d = tmem + acc * BN;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!tc::mbar_wait(&s.full[st], ph, g.flags, s.abort_flag)) goto done;
        tc::fence_after_sync();
        const uint32_t a0 = tc::smem_u32(s.a + st * A_STAGE);
        const uint32_t b0 = tc::smem_u32(s.b + st * B_STAGE);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          tc::mma_bf16(d, tc::sw128_desc(a0 + k * 2048, BOX), tc::sw128_desc(b0 + k * 2048, BOX),
                       idesc, (kb > kb0 || k) ? 1u : 0u);
        tc::mma_commit(&s.empty[st]);
        if (++st == STAGES) { st = 0; ph ^= 1; }
      }
      tc::mma_commit(&s.tfull[acc]);
    }
  } else if (warp >= 2) {
    const int q = warp & 3;
    int it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
      const int mt = u % num_mt, nt = (u / num_mt) % num_nt, ks = u / (num_mt * num_nt);
      const int kb0 = ks * g.kb_per_split;
      const bool empty_range = kb0 >= num_kb;
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!tc::mbar_wait(&s.tfull[acc], aph, g.flags, s.abort_flag)) goto done;
      tc::fence_after_sync();
      const int row = mt * BM + q * 32 + lane;
      float* prow = g.part + ((int64_t)ks * num_mt * BM + row) * ldp + nt * BN;
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + acc * BN + c0, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4*>(prow + c0 + j) =
              empty_range ? make_float4(0.f, 0.f, 0.f, 0.f)
                          : make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&s.tempty[acc]);
    }
  }
done:
  teardown(s, BN, tmem);
}

// out[i][j] = sum_s part[s][i][j] in split order, i < Mi, j < Nj.
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, int64_t split_stride,
                                     int ldp, int Mi, int Nj, float* __restrict__ out, int64_t ldo) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)Mi * Nj) return;
  const int i = (int)(idx / Nj), j = (int)(idx % Nj);
  const float* p = part + (int64_t)i * ldp + j;
  float acc = 0.f;
  for (int s2 = 0; s2 < splits; ++s2) acc += __ldg(p + (int64_t)s2 * split_stride);
  out[(int64_t)i * ldo + j] = acc;
}

// dZ = dH' * 1[H' > 0] (or dH' without ReLU), rounded to bf16, zero-padded
// to ldz columns.
__global__ void relu_mask_bf16_kernel(int64_t n, int F, const float* __restrict__ dH, int64_t ldg,
                                      const float* __restrict__ Hout, int64_t ldh, int relu,
                                      __nv_bfloat16* __restrict__ dZ, int64_t ldz) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_row = (int)(ldz / 4);
  if (idx >= n * per_row) return;
  const int64_t r = idx / per_row;
  const int c = (int)(idx % per_row) * 4;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (c < F) {
    const float4 g4 = *reinterpret_cast<const float4*>(dH + r * ldg + c);
    v[0] = g4.x; v[1] = g4.y; v[2] = g4.z; v[3] = g4.w;
    if (relu) {
      const float4 h4 = *reinterpret_cast<const float4*>(Hout + r * ldh + c);
      if (!(h4.x > 0.f)) v[0] = 0.f;
      if (!(h4.y > 0.f)) v[1] = 0.f;
      if (!(h4.z > 0.f)) v[2] = 0.f;
      if (!(h4.w > 0.f)) v[3] = 0.f;
    }
    for (int k = 0; k < 4; ++k)
      if (c + k >= F) v[k] = 0.f;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
  uint2 p;
  p.x = *reinterpret_cast<uint32_t*>(&lo);
  p.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dZ + r * ldz + c) = p;
}

// Xb = bf16(X) (nearest-even), columns F..ldb-1 zero.
__global__ void cast_bf16_kernel(int64_t n, int F, const float* __restrict__ X, int64_t ldx,
                                 __nv_bfloat16* __restrict__ Xb, int64_t ldb) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_row = (int)(ldb / 4);
  if (idx >= n * per_row) return;
  const int64_t r = idx / per_row;
  const int c = (int)(idx % per_row) * 4;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (c < F) {
    const float4 x4 = *reinterpret_cast<const float4*>(X + r * ldx + c);
    v[0] = x4.x; v[1] = x4.y; v[2] = x4.z; v[3] = x4.w;
    for (int k = 0; k < 4; ++k)
      if (c + k >= F) v[k] = 0.f;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
  uint2 p;
  p.x = *reinterpret_cast<uint32_t*>(&lo);
  p.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(Xb + r * ldb + c) = p;
}

// dZ = dH' * 1[H' > 0] in fp32, columns F..ldz-1 zero.
__global__ void relu_mask_f32_kernel(int64_t n, int F, const float* __restrict__ dH, int64_t ldg,
                                     const float* __restrict__ Hout, int64_t ldh,
                                     float* __restrict__ dZ, int64_t ldz) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_row = (int)(ldz / 4);
  if (idx >= n * per_row) return;
  const int64_t r = idx / per_row;
  const int c = (int)(idx % per_row) * 4;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < F) {
    v = *reinterpret_cast<const float4*>(dH + r * ldg + c);
    const float4 h4 = *reinterpret_cast<const float4*>(Hout + r * ldh + c);
    if (!(h4.x > 0.f) || c >= F) v.x = 0.f;
    if (!(h4.y > 0.f) || c + 1 >= F) v.y = 0.f;
    if (!(h4.z > 0.f) || c + 2 >= F) v.z = 0.f;
    if (!(h4.w > 0.f) || c + 3 >= F) v.w = 0.f;
  }
  *reinterpret_cast<float4*>(dZ + r * ldz + c) = v;
}

// Wt[j][i] = W[i][j] (i < F_in), zero for F_in <= i < K.
__global__ void transpose_w_kernel(const __nv_bfloat16* __restrict__ W, int F_in, int F_out, int K,
                                   __nv_bfloat16* __restrict__ Wt) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)F_out * K) return;
  const int j = (int)(idx / K), i = (int)(idx % K);
  Wt[idx] = i < F_in ? W[(int64_t)i * F_out + j] : __float2bfloat16(0.f);
}

// ---------------------------------------------------------------- host side
// The tensor-map encoder comes from the driver through the runtime, so the
// library itself does not link against libcuda.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

static gnn_status make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  if (((uintptr_t)base & 15) || (row_bytes & 15))
    return fail(GNN_ERR_INVALID_ARG, "dense transform: operands need 16-byte aligned rows");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(GNN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                            const_cast<void*>(base), dims, strides, box, es,
                                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GNN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return GNN_OK;
}

// fp32 output map for the epilogue's TMA stores (128-byte swizzle, 32 x 32 box).
static gnn_status make_tmap_f32(CUtensorMap* map, void* base, uint64_t inner, uint64_t outer,
                                uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  if (((uintptr_t)base & 15) || (row_bytes & 15))
    return fail(GNN_ERR_INVALID_ARG, "dense transform: output needs 16-byte aligned rows");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(GNN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GNN_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", (int)r);
  return GNN_OK;
}

static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

static gnn_status ensure_smem_attr() {
  static bool done = false;
  if (!done) {
    GNN_CUDA(cudaFuncSetAttribute(gemm_tn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TN_BYTES));
    GNN_CUDA(cudaFuncSetAttribute(gemm_mn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    done = true;
  }
  return GNN_OK;
}

gnn_status launch_gemm_tn(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, int M,
                          int N, int K, float* out, int64_t ldo, int n_store, int relu,
                          cudaStream_t st) {
  if (M == 0) return GNN_OK;
  if (N < 1 || K < 1) return fail(GNN_ERR_INVALID_ARG, "dense transform: empty N or K");
  gnn_status s = ensure_smem_attr();
  if (s != GNN_OK) return s;
  // N tile: a multiple of 16 (MMA shape); with several tiles a multiple of 32,
  // so the epilogue's 32-column stores never reach into the next tile
  const int num_n = (N + 255) / 256;
  const int BN = num_n == 1 ? (N + 15) / 16 * 16 : ((N + num_n - 1) / num_n + 31) / 32 * 32;
  CUtensorMap ta, tb, tcm;
  if ((s = make_tmap(&ta, A, (uint64_t)lda, (uint64_t)M, (uint64_t)lda * 2, BK, BM)) != GNN_OK) return s;
  if ((s = make_tmap(&tb, B, (uint64_t)ldb, (uint64_t)N, (uint64_t)ldb * 2, BK, (uint32_t)BN)) != GNN_OK) return s;
  if ((s = make_tmap_f32(&tcm, out, (uint64_t)n_store, (uint64_t)M, (uint64_t)ldo * 4, 32, 32)) != GNN_OK)
    return s;
  unsigned* flags = device_flags();
  if (!flags) return fail(GNN_ERR_CUDA, "device flag word unavailable");
  TnArgs g{M, N, K, BN, n_store, out, ldo, relu, flags};
  const int tiles = ((M + BM - 1) / BM) * num_n;
  const int grid = tiles < sm_count() ? tiles : sm_count();
  gemm_tn_kernel<<<grid, THREADS, SMEM_TN_BYTES, st>>>(ta, tb, tcm, g);
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

size_t gemm_mn_workspace_bytes(int Mi, int Nj, int K) {
  int splits = 0, kbps = 0, BN = 0;
  gemm_mn_plan(Mi, Nj, K, &splits, &kbps, &BN);
  const int num_mt = (Mi + BM - 1) / BM, num_nt = (Nj + BN - 1) / BN;
  return (size_t)splits * num_mt * BM * num_nt * BN * sizeof(float);
}

void gemm_mn_plan(int Mi, int Nj, int K, int* splits, int* kb_per_split, int* BN) {
  const int num_nt = (Nj + 255) / 256;
  *BN = ((Nj + num_nt - 1) / num_nt + 63) / 64 * 64;
  const int num_mt = (Mi + BM - 1) / BM;
  const int num_kb = (K + BK - 1) / BK;
  const int tiles = num_mt * num_nt;
  int want = (2 * sm_count() + tiles - 1) / tiles;  // about two units per SM
  if (want > num_kb) want = num_kb;
  if (want < 1) want = 1;
  *kb_per_split = (num_kb + want - 1) / want;
  *splits = (num_kb + *kb_per_split - 1) / *kb_per_split;
  if (*splits < 1) *splits = 1;
}

gnn_status launch_gemm_mn(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, int Mi,
                          int Nj, int K, float* out, int64_t ldo, float* part, cudaStream_t st) {
  gnn_status s = ensure_smem_attr();
  if (s != GNN_OK) return s;
  int splits, kbps, BN;
  gemm_mn_plan(Mi, Nj, K, &splits, &kbps, &BN);
  const int num_mt = (Mi + BM - 1) / BM, num_nt = (Nj + BN - 1) / BN;
  if (K == 0) {
    GNN_CUDA(cudaMemset2DAsync(out, ldo * sizeof(float), 0, Nj * sizeof(float), Mi, st));
    return GNN_OK;
  }
  CUtensorMap ta, tb;
  if ((s = make_tmap(&ta, A, (uint64_t)lda, (uint64_t)K, (uint64_t)lda * 2, 64, BK)) != GNN_OK) return s;
  if ((s = make_tmap(&tb, B, (uint64_t)ldb, (uint64_t)K, (uint64_t)ldb * 2, 64, BK)) != GNN_OK) return s;
  unsigned* flags = device_flags();
  if (!flags) return fail(GNN_ERR_CUDA, "device flag word unavailable");
  MnArgs g{Mi, Nj, K, BN, kbps, splits, part, flags};
  const int units = num_mt * num_nt * splits;
  const int grid = units < sm_count() ? units : sm_count();
  gemm_mn_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, g);
  GNN_CHECK_LAUNCH();
  const int ldp = num_nt * BN;
  const int64_t split_stride = (int64_t)num_mt * BM * ldp;
  const int64_t total = (int64_t)Mi * Nj;
  splitk_reduce_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(part, splits, split_stride,
                                                                       ldp, Mi, Nj, out, ldo);
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

gnn_status launch_relu_mask_bf16(int64_t n, int F, const float* dH, int64_t ldg, const float* Hout,
                                 int64_t ldh, int relu, uint16_t* dZ, int64_t ldz,
                                 cudaStream_t st) {
  if (n == 0) return GNN_OK;
  const int64_t total = n * (ldz / 4);
  relu_mask_bf16_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
      n, F, dH, ldg, Hout, ldh, relu, reinterpret_cast<__nv_bfloat16*>(dZ), ldz);
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

gnn_status launch_cast_bf16(int64_t n, int F, const float* X, int64_t ldx, uint16_t* Xb,
                            int64_t ldb, cudaStream_t st) {
  if (n == 0) return GNN_OK;
  const int64_t total = n * (ldb / 4);
  cast_bf16_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
      n, F, X, ldx, reinterpret_cast<__nv_bfloat16*>(Xb), ldb);
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

gnn_status launch_relu_mask_f32(int64_t n, int F, const float* dH, int64_t ldg, const float* Hout,
                                int64_t ldh, float* dZ, int64_t ldz, cudaStream_t st) {
  if (n == 0) return GNN_OK;
  const int64_t total = n * (ldz / 4);
  relu_mask_f32_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(n, F, dH, ldg, Hout, ldh,
                                                                        dZ, ldz);
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

gnn_status launch_transpose_w(const uint16_t* W, int F_in, int F_out, int K, uint16_t* Wt,
                              cudaStream_t st) {
  const int64_t total = (int64_t)F_out * K;
  transpose_w_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(W), F_in, F_out, K, reinterpret_cast<__nv_bfloat16*>(Wt));
  GNN_CHECK_LAUNCH();
  return GNN_OK;
}

}  // namespace gnn
