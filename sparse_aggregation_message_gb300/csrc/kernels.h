// Launch wrappers shared between the library's translation units.  They do
// no argument checking; the extern "C" entry points do that first.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gnnagg.h"

namespace gnn {

gnn_status launch_quant_pack(const float* X, int64_t ldx, int F, const int32_t* row_idx,
                             int64_t n_rows, const uint8_t* bits, const int64_t* off,
                             uint32_t seed, uint8_t* packed, float2* meta, cudaStream_t st);
// Rows [r0, r0 + n_rows) of the row lists (row key = row index).
gnn_status launch_quant_pack_range(const float* X, int64_t ldx, int F, const int32_t* row_idx,
                                   int64_t r0, int64_t n_rows, const uint8_t* bits,
                                   const int64_t* off, uint32_t seed, uint8_t* packed,
                                   float2* meta, cudaStream_t st);

// Every slot's forward message, node by node along the owner lists.
gnn_status launch_quant_pack_owned(const gnn_boundary& b, const float* X, int64_t ldx, int F,
                                   uint32_t seed, uint8_t* packed, float2* meta, cudaStream_t st);

gnn_status launch_dequant_unpack(const uint8_t* packed, const float2* meta, const int64_t* off,
                                 const uint8_t* bits, int64_t n_rows, int F, float* out,
                                 int64_t ldo, cudaStream_t st);

// M = A H (bnd NULL) or the partitioned forward aggregation; fp32 and/or bf16
// outputs (either may be NULL), ReLU'd when relu != 0.
// `partial` holds one fp32 row per piece of csr's split plan (may be NULL
// without a plan).
gnn_status launch_spmm_fwd(const gnn_csr& csr, const gnn_boundary* bnd, const float* H,
                           int64_t ldh, int F, const uint8_t* packed, const float2* meta,
                           float* M, int64_t ldm, uint16_t* Mb, int64_t ldmb, float* partial,
                           cudaStream_t st, int relu = 0);

gnn_status launch_spmm_bwd(const gnn_csr& csr, const gnn_boundary* bnd, const float* G,
                           int64_t ldg, int F, uint32_t seed, uint8_t* packed_ws,
                           float2* meta_ws, float* dH, int64_t ldh, float* partial,
                           cudaStream_t st);

gnn_status launch_spmm_bwd_local(const gnn_csr& csr, const gnn_boundary& bnd, const float* G,
                                 int64_t ldg, int F, const uint8_t* packed, const float2* meta,
                                 float* dH, int64_t ldh, float* partial, cudaStream_t st);

gnn_status launch_halo_quant_pack(const gnn_boundary& b, const float* Gm, int64_t ldg, int F,
                                  uint32_t seed, uint8_t* packed_ws, float2* meta_ws,
                                  cudaStream_t st);

// The halo quant-pack with other entry weights (sval, slot-CSR order) and,
// when score_r is given, the score term fl(P + fl(score_r[s] * a_r[j])) added
// to each slot's partial before it is quantised.
// Slots [s_lo, s_hi) only (s_hi < 0: every slot).
gnn_status launch_halo_quant_pack_ex(const gnn_boundary& b, const float* Gm, int64_t ldg, int F,
                                     uint32_t seed, uint8_t* packed_ws, float2* meta_ws,
                                     const float* sval, const float* score_r, const float* a_r,
                                     cudaStream_t st, int64_t s_lo = 0, int64_t s_hi = -1);

// Aggregations with caller weights in place of the CSR's (CSR order without
// a boundary, col_remap order with one): the forward (fp32 out, optional
// ReLU) and the owner-side backward (local entries plus owned messages).
gnn_status launch_spmm_fwd_w(const gnn_csr& csr, const gnn_boundary* bnd, const float* weights,
                             const float* H, int64_t ldh, int F, const uint8_t* packed,
                             const float2* meta, float* M, int64_t ldm, float* partial, int relu,
                             cudaStream_t st);
gnn_status launch_spmm_bwd_local_w(const gnn_csr& csr, const gnn_boundary* bnd,
                                   const float* weights, const float* Gm, int64_t ldg, int F,
                                   const uint8_t* packed, const float2* meta, float* dH,
                                   int64_t ldh, float* partial, cudaStream_t st);

// The backward aggregation with the next layer's ReLU gate and bf16 rounding
// fused into its store: dZ = bf16((A^T G) * 1[hmask > 0]) (hmask NULL: no
// gate), columns F..ldz-1 zero.
gnn_status launch_spmm_bwd_masked(const gnn_csr& csr, const gnn_boundary* bnd, const float* Gm,
                                  int64_t ldg, int F, uint32_t seed, uint8_t* packed_ws,
                                  float2* meta_ws, const float* hmask, int64_t ldhm, uint16_t* dZ,
                                  int64_t ldz, float* partial, cudaStream_t st);

// The owner-side half of launch_spmm_bwd_masked: local A^T entries plus the
// owned messages in packed/meta, gated and stored as bf16.
gnn_status launch_spmm_bwd_local_masked(const gnn_csr& csr, const gnn_boundary& bnd,
                                        const float* Gm, int64_t ldg, int F, const uint8_t* packed,
                                        const float2* meta, const float* hmask, int64_t ldhm,
                                        uint16_t* dZ, int64_t ldz, float* partial, cudaStream_t st);

size_t spmm_workspace_bytes(const gnn_csr& csr, int F);

// gnn_spmm_fwd with its argument checks, the output ReLU'd when relu != 0.
gnn_status spmm_fwd_checked(const gnn_csr* csr, const gnn_boundary* bnd, const float* H,
                            int64_t ldh, int32_t F, const uint8_t* packed, const float* meta,
                            float* M, int64_t ldm, uint16_t* Mb, int64_t ldmb, void* ws,
                            size_t ws_bytes, gnn_stream_t stream, int relu);

}  // namespace gnn
