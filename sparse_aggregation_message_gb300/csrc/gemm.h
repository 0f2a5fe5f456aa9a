// Launch wrappers of the tcgen05 dense transform and its elementwise helpers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gnnagg.h"

namespace gnn {

// out[M x n_store] = A[M x K] * B[N x K]^T (bf16, K contiguous, row strides
// lda/ldb elements, multiples of 8), optional ReLU.  Columns N..n_store-1 of
// out come from zero-filled B rows.
gnn_status launch_gemm_tn(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, int M,
                          int N, int K, float* out, int64_t ldo, int n_store, int relu,
                          cudaStream_t st);

// out[Mi x Nj] = sum_{k<K} A[k][i] B[k][j] (bf16 row-major, strides lda/ldb
// multiples of 8), through split-k partial tiles in `part`
// (gemm_mn_workspace_bytes) added in fixed order.
gnn_status launch_gemm_mn(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, int Mi,
                          int Nj, int K, float* out, int64_t ldo, float* part, cudaStream_t st);
size_t gemm_mn_workspace_bytes(int Mi, int Nj, int K);
void gemm_mn_plan(int Mi, int Nj, int K, int* splits, int* kb_per_split, int* BN);

gnn_status launch_relu_mask_bf16(int64_t n, int F, const float* dH, int64_t ldg, const float* Hout,
                                 int64_t ldh, int relu, uint16_t* dZ, int64_t ldz, cudaStream_t st);

// Xb = bf16(X) with row stride ldb (a multiple of 4), columns F.. zero.
gnn_status launch_cast_bf16(int64_t n, int F, const float* X, int64_t ldx, uint16_t* Xb,
                            int64_t ldb, cudaStream_t st);

// dZ = dH' * 1[H' > 0] in fp32 with row stride ldz (a multiple of 4).
gnn_status launch_relu_mask_f32(int64_t n, int F, const float* dH, int64_t ldg, const float* Hout,
                                int64_t ldh, float* dZ, int64_t ldz, cudaStream_t st);

gnn_status launch_transpose_w(const uint16_t* W, int F_in, int F_out, int K, uint16_t* Wt,
                              cudaStream_t st);

}  // namespace gnn
