// Dense transform and whole-layer entry points: one GCN layer of the SYLVIE
// guide's section 11 data path on one stream -- quantise the boundary rows,
// aggregate with dequantised remote rows, transform with W (tcgen05) and
// activate; the backward mirrors it with the embedding gradients.
#include <cuda_runtime.h>

#include "gemm.h"
#include "internal.h"
#include "kernels.h"

namespace gnn {

static int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct DenseWs {
  uint16_t* wt;    // W^T [F_out x ldb] (forward)
  uint16_t* dz;    // dZ bf16 [n x ldz] (backward)
  float* part;     // split-k partials of dW
  size_t bytes;
};

static DenseWs dense_ws_layout(void* base, size_t cap, int64_t n, int F_in, int F_out,
                               bool* ok) {
  Arena ar(base, cap);
  DenseWs w{};
  const int64_t ldb = round_up(F_in, 16), ldz = round_up(F_out, 64);
  w.wt = ar.take<uint16_t>((size_t)F_out * ldb);
  w.dz = ar.take<uint16_t>((size_t)n * ldz);
  w.part = reinterpret_cast<float*>(ar.take_bytes(gemm_mn_workspace_bytes(F_in, F_out, (int)n)));
  w.bytes = ar.used;
  *ok = ar.ok();
  return w;
}

static gnn_status check_dims(int64_t n, int F_in, int F_out, const char* who) {
  if (n < 0 || n > (int64_t)0x7fffffff) return fail(GNN_ERR_INVALID_ARG, "%s: bad row count", who);
  if (F_in < 1 || F_out < 1) return fail(GNN_ERR_INVALID_ARG, "%s: F_in/F_out must be >= 1", who);
  if (F_in > kMaxF) return fail(GNN_ERR_UNSUPPORTED, "%s: F_in=%d > %d", who, F_in, kMaxF);
  if (F_out % 16 != 0 || F_out > 256)
    return fail(GNN_ERR_UNSUPPORTED, "%s: F_out must be a multiple of 16 and <= 256", who);
  return GNN_OK;
}

static gnn_status dense_fwd_impl(const uint16_t* Mb, int64_t ldmb, int64_t n, int F_in,
                                 const uint16_t* W, int F_out, int relu, float* H_out,
                                 int64_t ldo, const DenseWs& w, cudaStream_t st) {
  const int64_t K = round_up(F_in, 16);
  gnn_status s = launch_transpose_w(W, F_in, F_out, (int)K, w.wt, st);
  if (s != GNN_OK) return s;
  return launch_gemm_tn(Mb, ldmb, w.wt, K, (int)n, F_out, (int)K, H_out, ldo, F_out, relu, st);
}

static gnn_status dense_bwd_impl(const uint16_t* Mb, int64_t ldmb, int64_t n, int F_in,
                                 const uint16_t* W, int F_out, const float* dH_out, int64_t ldg,
                                 const float* H_out, int64_t ldo, int relu, float* dM,
                                 int64_t ldm, float* dW, const DenseWs& w, cudaStream_t st) {
  const int64_t ldz = round_up(F_out, 64);
  gnn_status s = launch_relu_mask_bf16(n, F_out, dH_out, ldg, H_out, ldo, relu, w.dz, ldz, st);
  if (s != GNN_OK) return s;
  if (dM) {
    // dM = dZ W^T: A = dZ [n x F_out], B = W [F_in x F_out], both K-major
    s = launch_gemm_tn(w.dz, ldz, W, F_out, (int)n, F_in, F_out, dM, ldm, (int)round_up(F_in, 4),
                       0, st);
    if (s != GNN_OK) return s;
  }
  if (dW) {
    // dW = Mb^T dZ: reduction over the n rows of both (MN-major operands)
    s = launch_gemm_mn(Mb, ldmb, w.dz, ldz, F_in, F_out, (int)n, dW, F_out, w.part, st);
    if (s != GNN_OK) return s;
  }
  return GNN_OK;
}

}  // namespace gnn

using namespace gnn;

extern "C" gnn_status gnn_dense_workspace(int64_t n, int32_t F_in, int32_t F_out, size_t* ws_bytes) {
  gnn_status s = check_dims(n, F_in, F_out, "gnn_dense_workspace");
  if (s != GNN_OK) return s;
  GNN_REQUIRE(ws_bytes, "gnn_dense_workspace: NULL ws_bytes");
  bool ok;
  *ws_bytes = dense_ws_layout(nullptr, 0, n, F_in, F_out, &ok).bytes;
  return GNN_OK;
}

static gnn_status check_mb(const uint16_t* Mb, int64_t ldmb, int F_in, const char* who) {
  if (!Mb || ldmb < (F_in + 15) / 16 * 16 || ldmb % 8 || ((uintptr_t)Mb & 15))
    return fail(GNN_ERR_INVALID_ARG, "%s: Mb needs ldmb >= round_up(F_in,16), a multiple of 8, "
                "16-byte alignment", who);
  return GNN_OK;
}

extern "C" gnn_status gnn_dense_fwd(const uint16_t* Mb, int64_t ldmb, int64_t n, int32_t F_in,
                                    const uint16_t* W, int32_t F_out, int32_t relu, float* H_out,
                                    int64_t ldo, void* ws, size_t ws_bytes, gnn_stream_t stream) {
  gnn_status s = check_dims(n, F_in, F_out, "gnn_dense_fwd");
  if (s != GNN_OK) return s;
  if (n == 0) return GNN_OK;
  if ((s = check_mb(Mb, ldmb, F_in, "gnn_dense_fwd")) != GNN_OK) return s;
  GNN_REQUIRE(W && H_out && ldo >= F_out && ldo % 4 == 0 && ((uintptr_t)H_out & 15) == 0,
              "gnn_dense_fwd: bad W or H_out");
  bool ok;
  DenseWs w = dense_ws_layout(ws, ws_bytes, n, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_dense_fwd: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  return dense_fwd_impl(Mb, ldmb, n, F_in, W, F_out, relu, H_out, ldo, w, as_stream(stream));
}

extern "C" gnn_status gnn_dense_bwd(const uint16_t* Mb, int64_t ldmb, int64_t n, int32_t F_in,
                                    const uint16_t* W, int32_t F_out, const float* dH_out,
                                    int64_t ldg, const float* H_out, int64_t ldo, int32_t relu,
                                    float* dM, int64_t ldm, float* dW, void* ws, size_t ws_bytes,
                                    gnn_stream_t stream) {
  gnn_status s = check_dims(n, F_in, F_out, "gnn_dense_bwd");
  if (s != GNN_OK) return s;
  if ((s = check_mb(Mb, ldmb, F_in, "gnn_dense_bwd")) != GNN_OK) return s;
  GNN_REQUIRE(W && dH_out && ldg >= F_out && ldg % 4 == 0 && ((uintptr_t)dH_out & 15) == 0,
              "gnn_dense_bwd: bad W or dH_out");
  GNN_REQUIRE(!relu || (H_out && ldo >= F_out && ldo % 4 == 0 && ((uintptr_t)H_out & 15) == 0),
              "gnn_dense_bwd: relu needs H_out");
  GNN_REQUIRE(!dM || (ldm >= (F_in + 3) / 4 * 4 && ldm % 4 == 0 && ((uintptr_t)dM & 15) == 0),
              "gnn_dense_bwd: dM needs ldm >= round_up(F_in,4), a multiple of 4");
  bool ok;
  DenseWs w = dense_ws_layout(ws, ws_bytes, n, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_dense_bwd: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  return dense_bwd_impl(Mb, ldmb, n, F_in, W, F_out, dH_out, ldg, H_out, ldo, relu, dM, ldm, dW,
                        w, as_stream(stream));
}

extern "C" gnn_status gnn_dense_bwd_z(const uint16_t* Mb, int64_t ldmb, int64_t n, int32_t F_in,
                                      const uint16_t* W, int32_t F_out, const uint16_t* dZ,
                                      int64_t ldz, float* dM, int64_t ldm, float* dW, void* ws,
                                      size_t ws_bytes, gnn_stream_t stream) {
  gnn_status s = check_dims(n, F_in, F_out, "gnn_dense_bwd_z");
  if (s != GNN_OK) return s;
  if ((s = check_mb(Mb, ldmb, F_in, "gnn_dense_bwd_z")) != GNN_OK) return s;
  GNN_REQUIRE(W && dZ && ldz >= round_up(F_out, 64) && ldz % 8 == 0 && ((uintptr_t)dZ & 15) == 0,
              "gnn_dense_bwd_z: dZ needs ldz >= round_up(F_out, 64), a multiple of 8");
  GNN_REQUIRE(!dM || (ldm >= (F_in + 3) / 4 * 4 && ldm % 4 == 0 && ((uintptr_t)dM & 15) == 0),
              "gnn_dense_bwd_z: dM needs ldm >= round_up(F_in,4), a multiple of 4");
  bool ok;
  DenseWs w = dense_ws_layout(ws, ws_bytes, n, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_dense_bwd_z: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  if (n == 0) return GNN_OK;
  cudaStream_t st = as_stream(stream);
  if (dM) {
    s = launch_gemm_tn(dZ, ldz, W, F_out, (int)n, F_in, F_out, dM, ldm, (int)round_up(F_in, 4), 0,
                       st);
    if (s != GNN_OK) return s;
  }
  if (dW) return launch_gemm_mn(Mb, ldmb, dZ, ldz, F_in, F_out, (int)n, dW, F_out, w.part, st);
  return GNN_OK;
}

// ------------------------------------------------------------------ layers// ------------------------------------------------------------------ layers
struct LayerWs {
  DenseWs dense;
  float* dM;
  float* spmm;
  size_t bytes;
};

static LayerWs layer_ws_layout(void* base, size_t cap, const gnn_csr& csr, int F_in, int F_out,
                               bool* ok) {
  LayerWs w{};
  bool ok1;
  DenseWs probe = dense_ws_layout(nullptr, 0, csr.n, F_in, F_out, &ok1);
  Arena ar(base, cap);
  void* dbase = ar.take_bytes(probe.bytes);
  w.dense = dense_ws_layout(dbase, probe.bytes, csr.n, F_in, F_out, &ok1);
  w.dM = ar.take<float>((size_t)csr.n * (size_t)round_up(F_in, 4));
  const size_t sp = spmm_workspace_bytes(csr, F_in);
  w.spmm = sp ? reinterpret_cast<float*>(ar.take_bytes(sp)) : nullptr;
  w.bytes = ar.used;
  *ok = ar.ok();
  return w;
}

extern "C" gnn_status gnn_layer_workspace(const gnn_csr* csr, int32_t F_in, int32_t F_out,
                                          size_t* ws_bytes) {
  GNN_REQUIRE(csr && ws_bytes, "gnn_layer_workspace: NULL argument");
  gnn_status s = check_dims(csr->n, F_in, F_out, "gnn_layer_workspace");
  if (s != GNN_OK) return s;
  bool ok;
  *ws_bytes = layer_ws_layout(nullptr, 0, *csr, F_in, F_out, &ok).bytes;
  return GNN_OK;
}

extern "C" gnn_status gnn_layer_fwd(const gnn_csr* csr, const gnn_boundary* bnd, const float* H_in,
                                    int64_t ldh, int32_t F_in, const uint16_t* W, int32_t F_out,
                                    int32_t relu, uint32_t seed, uint8_t* packed_ws,
                                    float* meta_ws, uint16_t* Mb, int64_t ldmb, float* H_out,
                                    int64_t ldo, void* ws, size_t ws_bytes, gnn_stream_t stream) {
  GNN_REQUIRE(csr, "gnn_layer_fwd: csr is NULL");
  gnn_status s = check_dims(csr->n, F_in, F_out, "gnn_layer_fwd");
  if (s != GNN_OK) return s;
  if (csr->n == 0) return GNN_OK;
  if ((s = check_mb(Mb, ldmb, F_in, "gnn_layer_fwd")) != GNN_OK) return s;
  GNN_REQUIRE(W && H_out && ldo >= F_out && ldo % 4 == 0 && ((uintptr_t)H_out & 15) == 0,
              "gnn_layer_fwd: bad W or H_out");
  bool ok;
  LayerWs w = layer_ws_layout(ws, ws_bytes, *csr, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_layer_fwd: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  cudaStream_t st = as_stream(stream);
  if (bnd && bnd->n_slots > 0) {
    GNN_REQUIRE(bnd->slot_node && bnd->slot_bits && bnd->slot_off && bnd->F == F_in,
                "gnn_layer_fwd: boundary offsets must be for F_in");
    GNN_REQUIRE(packed_ws && meta_ws && ((uintptr_t)packed_ws & 15) == 0 && ((uintptr_t)meta_ws & 7) == 0,
                "gnn_layer_fwd: packed_ws/meta_ws required with a boundary");
    GNN_REQUIRE(ldh >= F_in && ldh % 4 == 0 && ((uintptr_t)H_in & 15) == 0, "gnn_layer_fwd: bad H_in");
    s = launch_quant_pack_owned(*bnd, H_in, ldh, F_in, seed, packed_ws,
                                reinterpret_cast<float2*>(meta_ws), st);
    if (s != GNN_OK) return s;
  }
  s = gnn_spmm_fwd(csr, bnd, H_in, ldh, F_in, packed_ws, meta_ws, nullptr, 0, Mb, ldmb, w.spmm,
                   spmm_workspace_bytes(*csr, F_in), stream);
  if (s != GNN_OK) return s;
  return dense_fwd_impl(Mb, ldmb, csr->n, F_in, W, F_out, relu, H_out, ldo, w.dense, st);
}

extern "C" gnn_status gnn_layer_bwd(const gnn_csr* csr, const gnn_boundary* bnd,
                                    const float* dH_out, int64_t ldg, const float* H_out,
                                    int64_t ldo, int32_t relu, const uint16_t* Mb, int64_t ldmb,
                                    const uint16_t* W, int32_t F_in, int32_t F_out, uint32_t seed,
                                    uint8_t* packed_ws, float* meta_ws, float* dW, float* dH_in,
                                    int64_t ldh, void* ws, size_t ws_bytes, gnn_stream_t stream) {
  GNN_REQUIRE(csr, "gnn_layer_bwd: csr is NULL");
  gnn_status s = check_dims(csr->n, F_in, F_out, "gnn_layer_bwd");
  if (s != GNN_OK) return s;
  if (csr->n == 0) return GNN_OK;
  bool ok;
  LayerWs w = layer_ws_layout(ws, ws_bytes, *csr, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_layer_bwd: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  GNN_REQUIRE(dW, "gnn_layer_bwd: dW is NULL");
  const int64_t ldm = round_up(F_in, 4);
  s = gnn_dense_bwd(Mb, ldmb, csr->n, F_in, W, F_out, dH_out, ldg, H_out, ldo, relu,
                    dH_in ? w.dM : nullptr, ldm, dW, w.dense.wt, w.dense.bytes, stream);
  if (s != GNN_OK) return s;
  if (!dH_in) return GNN_OK;
  return gnn_spmm_bwd(csr, bnd, w.dM, ldm, F_in, seed, packed_ws, meta_ws, dH_in, ldh, w.spmm,
                      spmm_workspace_bytes(*csr, F_in), stream);
}

// ------------------------------------------------------------------ asynchronous epochs
// `aux` waits for `stream` (the layer's input is ready), runs the quantise
// and pack of this epoch's messages, and `stream` waits for `aux` before the
// call returns, so the overlap stays inside the call.
struct Fork {
  cudaEvent_t ready = nullptr, done = nullptr;
  ~Fork() {
    if (ready) cudaEventDestroy(ready);
    if (done) cudaEventDestroy(done);
  }
};

static gnn_status fork_to(Fork& f, cudaStream_t st, cudaStream_t aux) {
  GNN_CUDA(cudaEventCreateWithFlags(&f.ready, cudaEventDisableTiming));
  GNN_CUDA(cudaEventCreateWithFlags(&f.done, cudaEventDisableTiming));
  GNN_CUDA(cudaEventRecord(f.ready, st));
  GNN_CUDA(cudaStreamWaitEvent(aux, f.ready, 0));
  return GNN_OK;
}

static gnn_status join_from(Fork& f, cudaStream_t st, cudaStream_t aux) {
  GNN_CUDA(cudaEventRecord(f.done, aux));
  GNN_CUDA(cudaStreamWaitEvent(st, f.done, 0));
  return GNN_OK;
}

extern "C" gnn_status gnn_layer_fwd_async(const gnn_csr* csr, const gnn_boundary* bnd,
                                          const float* H_in, int64_t ldh, int32_t F_in,
                                          const uint16_t* W, int32_t F_out, int32_t relu,
                                          uint32_t seed, const uint8_t* packed_prev,
                                          const float* meta_prev, uint8_t* packed_next,
                                          float* meta_next, uint16_t* Mb, int64_t ldmb,
                                          float* H_out, int64_t ldo, void* ws, size_t ws_bytes,
                                          gnn_stream_t stream, gnn_stream_t aux) {
  GNN_REQUIRE(csr && bnd, "gnn_layer_fwd_async: csr and boundary required");
  gnn_status s = check_dims(csr->n, F_in, F_out, "gnn_layer_fwd_async");
  if (s != GNN_OK) return s;
  if (csr->n == 0) return GNN_OK;
  if ((s = check_mb(Mb, ldmb, F_in, "gnn_layer_fwd_async")) != GNN_OK) return s;
  GNN_REQUIRE(W && H_out && ldo >= F_out && ldo % 4 == 0 && ((uintptr_t)H_out & 15) == 0,
              "gnn_layer_fwd_async: bad W or H_out");
  GNN_REQUIRE(bnd->F == F_in, "gnn_layer_fwd_async: boundary offsets must be for F_in");
  GNN_REQUIRE(bnd->n_slots == 0 ||
                  (packed_prev && meta_prev && packed_next && meta_next &&
                   ((uintptr_t)packed_next & 15) == 0 && ((uintptr_t)meta_next & 7) == 0 &&
                   bnd->slot_node && bnd->slot_bits && bnd->slot_off),
              "gnn_layer_fwd_async: message buffers required with a boundary");
  GNN_REQUIRE(ldh >= F_in && ldh % 4 == 0 && H_in && ((uintptr_t)H_in & 15) == 0,
              "gnn_layer_fwd_async: bad H_in");
  GNN_REQUIRE(bnd->n_slots == 0 || (packed_prev != packed_next && meta_prev != meta_next),
              "gnn_layer_fwd_async: the previous and next message buffers must differ");
  bool ok;
  LayerWs w = layer_ws_layout(ws, ws_bytes, *csr, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_layer_fwd_async: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  cudaStream_t st = as_stream(stream), ax = as_stream(aux);
  Fork f;
  if ((s = fork_to(f, st, ax)) != GNN_OK) return s;
  // from here on `stream` always waits for `aux` before returning, error or not
  if (bnd->n_slots > 0)
    s = launch_quant_pack_owned(*bnd, H_in, ldh, F_in, seed, packed_next,
                                reinterpret_cast<float2*>(meta_next), ax);
  if (s == GNN_OK)
    s = gnn_spmm_fwd(csr, bnd, H_in, ldh, F_in, packed_prev, meta_prev, nullptr, 0, Mb, ldmb,
                     w.spmm, spmm_workspace_bytes(*csr, F_in), stream);
  if (s == GNN_OK) s = dense_fwd_impl(Mb, ldmb, csr->n, F_in, W, F_out, relu, H_out, ldo, w.dense, st);
  const gnn_status j = join_from(f, st, ax);
  return s != GNN_OK ? s : j;
}

extern "C" gnn_status gnn_layer_bwd_async(const gnn_csr* csr, const gnn_boundary* bnd,
                                          const float* dH_out, int64_t ldg, const float* H_out,
                                          int64_t ldo, int32_t relu, const uint16_t* Mb,
                                          int64_t ldmb, const uint16_t* W, int32_t F_in,
                                          int32_t F_out, uint32_t seed,
                                          const uint8_t* packed_prev, const float* meta_prev,
                                          uint8_t* packed_next, float* meta_next, float* dW,
                                          float* dH_in, int64_t ldh, void* ws, size_t ws_bytes,
                                          gnn_stream_t stream, gnn_stream_t aux) {
  GNN_REQUIRE(csr && bnd, "gnn_layer_bwd_async: csr and boundary required");
  gnn_status s = check_dims(csr->n, F_in, F_out, "gnn_layer_bwd_async");
  if (s != GNN_OK) return s;
  if (csr->n == 0) return GNN_OK;
  bool ok;
  LayerWs w = layer_ws_layout(ws, ws_bytes, *csr, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_layer_bwd_async: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  GNN_REQUIRE(dW, "gnn_layer_bwd_async: dW is NULL");
  GNN_REQUIRE(!dH_in || bnd->n_slots == 0 || (packed_prev != packed_next && meta_prev != meta_next),
              "gnn_layer_bwd_async: the previous and next message buffers must differ");
  const int64_t ldm = round_up(F_in, 4);
  s = gnn_dense_bwd(Mb, ldmb, csr->n, F_in, W, F_out, dH_out, ldg, H_out, ldo, relu,
                    dH_in ? w.dM : nullptr, ldm, dW, w.dense.wt, w.dense.bytes, stream);
  if (s != GNN_OK || !dH_in) return s;
  cudaStream_t st = as_stream(stream), ax = as_stream(aux);
  Fork f;
  if ((s = fork_to(f, st, ax)) != GNN_OK) return s;
  // from here on `stream` always waits for `aux` before returning, error or not
  s = gnn_halo_quant_pack(bnd, w.dM, ldm, F_in, seed, packed_next, meta_next, aux);
  if (s == GNN_OK)
    s = gnn_spmm_bwd_local(csr, bnd, w.dM, ldm, F_in, packed_prev, meta_prev, dH_in, ldh, w.spmm,
                           spmm_workspace_bytes(*csr, F_in), stream);
  const gnn_status j = join_from(f, st, ax);
  return s != GNN_OK ? s : j;
}

// ------------------------------------------------------------------ transform-first layers
// A (H W) = (A H) W: when F_out < F_in the aggregation (and the message) runs
// at the narrower width F_out.
struct TfWs {
  DenseWs dense;
  float* dz;  // masked upstream gradient, fp32 [n x round_up(F_out, 4)]
  float* dy;  // A^T dz, fp32 [n x round_up(F_out, 4)]
  float* spmm;
  size_t bytes;
};

static TfWs tf_ws_layout(void* base, size_t cap, const gnn_csr& csr, int F_in, int F_out, bool* ok) {
  TfWs w{};
  bool ok1;
  DenseWs probe = dense_ws_layout(nullptr, 0, csr.n, F_in, F_out, &ok1);
  Arena ar(base, cap);
  void* dbase = ar.take_bytes(probe.bytes);
  w.dense = dense_ws_layout(dbase, probe.bytes, csr.n, F_in, F_out, &ok1);
  const size_t ldy = (size_t)round_up(F_out, 4);
  w.dz = ar.take<float>((size_t)csr.n * ldy);
  w.dy = ar.take<float>((size_t)csr.n * ldy);
  const size_t sp = spmm_workspace_bytes(csr, F_out);
  w.spmm = sp ? reinterpret_cast<float*>(ar.take_bytes(sp)) : nullptr;
  w.bytes = ar.used;
  *ok = ar.ok();
  return w;
}

extern "C" gnn_status gnn_layer_tf_workspace(const gnn_csr* csr, int32_t F_in, int32_t F_out,
                                             size_t* ws_bytes) {
  GNN_REQUIRE(csr && ws_bytes, "gnn_layer_tf_workspace: NULL argument");
  gnn_status s = check_dims(csr->n, F_in, F_out, "gnn_layer_tf_workspace");
  if (s != GNN_OK) return s;
  bool ok;
  *ws_bytes = tf_ws_layout(nullptr, 0, *csr, F_in, F_out, &ok).bytes;
  return GNN_OK;
}

extern "C" gnn_status gnn_layer_fwd_tf(const gnn_csr* csr, const gnn_boundary* bnd,
                                       const float* H_in, int64_t ldh, int32_t F_in,
                                       const uint16_t* W, int32_t F_out, int32_t relu,
                                       uint32_t seed, uint8_t* packed_ws, float* meta_ws,
                                       uint16_t* Hb, int64_t ldhb, float* Y, int64_t ldy,
                                       float* H_out, int64_t ldo, void* ws, size_t ws_bytes,
                                       gnn_stream_t stream) {
  GNN_REQUIRE(csr, "gnn_layer_fwd_tf: csr is NULL");
  gnn_status s = check_dims(csr->n, F_in, F_out, "gnn_layer_fwd_tf");
  if (s != GNN_OK) return s;
  if (csr->n == 0) return GNN_OK;
  if ((s = check_mb(Hb, ldhb, F_in, "gnn_layer_fwd_tf")) != GNN_OK) return s;
  GNN_REQUIRE(H_in && ldh >= F_in && ldh % 4 == 0 && ((uintptr_t)H_in & 15) == 0,
              "gnn_layer_fwd_tf: bad H_in");
  GNN_REQUIRE(W && Y && ldy >= round_up(F_out, 4) && ldy % 4 == 0 && ((uintptr_t)Y & 15) == 0,
              "gnn_layer_fwd_tf: bad W or Y");
  GNN_REQUIRE(H_out && ldo >= F_out && ldo % 4 == 0 && ((uintptr_t)H_out & 15) == 0,
              "gnn_layer_fwd_tf: bad H_out");
  bool ok;
  TfWs w = tf_ws_layout(ws, ws_bytes, *csr, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_layer_fwd_tf: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  cudaStream_t st = as_stream(stream);
  // Y = bf16(H_in) W
  if ((s = launch_cast_bf16(csr->n, F_in, H_in, ldh, Hb, ldhb, st)) != GNN_OK) return s;
  if ((s = dense_fwd_impl(Hb, ldhb, csr->n, F_in, W, F_out, 0, Y, ldy, w.dense, st)) != GNN_OK)
    return s;
  // the messages are Y's boundary rows
  if (bnd && bnd->n_slots > 0) {
    GNN_REQUIRE(bnd->slot_node && bnd->slot_bits && bnd->slot_off && bnd->F == F_out,
                "gnn_layer_fwd_tf: boundary offsets must be for F_out");
    GNN_REQUIRE(packed_ws && meta_ws && ((uintptr_t)packed_ws & 15) == 0 && ((uintptr_t)meta_ws & 7) == 0,
                "gnn_layer_fwd_tf: packed_ws/meta_ws required with a boundary");
    s = launch_quant_pack_owned(*bnd, Y, ldy, F_out, seed, packed_ws,
                                reinterpret_cast<float2*>(meta_ws), st);
    if (s != GNN_OK) return s;
  } else if (bnd) {
    GNN_REQUIRE(bnd->F == F_out, "gnn_layer_fwd_tf: boundary offsets must be for F_out");
  }
  // H_out = act(A Y)
  return spmm_fwd_checked(csr, bnd, Y, ldy, F_out, packed_ws, meta_ws, H_out, ldo, nullptr, 0,
                          w.spmm, spmm_workspace_bytes(*csr, F_out), stream, relu);
}

extern "C" gnn_status gnn_layer_bwd_tf(const gnn_csr* csr, const gnn_boundary* bnd,
                                       const float* dH_out, int64_t ldg, const float* H_out,
                                       int64_t ldo, int32_t relu, const uint16_t* Hb,
                                       int64_t ldhb, const uint16_t* W, int32_t F_in,
                                       int32_t F_out, uint32_t seed, uint8_t* packed_ws,
                                       float* meta_ws, float* dW, float* dH_in, int64_t ldh,
                                       void* ws, size_t ws_bytes, gnn_stream_t stream) {
  GNN_REQUIRE(csr, "gnn_layer_bwd_tf: csr is NULL");
  gnn_status s = check_dims(csr->n, F_in, F_out, "gnn_layer_bwd_tf");
  if (s != GNN_OK) return s;
  if (csr->n == 0) return GNN_OK;
  if ((s = check_mb(Hb, ldhb, F_in, "gnn_layer_bwd_tf")) != GNN_OK) return s;
  GNN_REQUIRE(W && dW, "gnn_layer_bwd_tf: W and dW required");
  GNN_REQUIRE(dH_out && ldg >= F_out && ldg % 4 == 0 && ((uintptr_t)dH_out & 15) == 0,
              "gnn_layer_bwd_tf: bad dH_out");
  GNN_REQUIRE(!relu || (H_out && ldo >= F_out && ldo % 4 == 0 && ((uintptr_t)H_out & 15) == 0),
              "gnn_layer_bwd_tf: relu needs H_out");
  GNN_REQUIRE(!dH_in || (ldh >= round_up(F_in, 4) && ldh % 4 == 0 && ((uintptr_t)dH_in & 15) == 0),
              "gnn_layer_bwd_tf: dH_in needs ldh >= round_up(F_in,4), a multiple of 4");
  bool ok;
  TfWs w = tf_ws_layout(ws, ws_bytes, *csr, F_in, F_out, &ok);
  GNN_REQUIRE(ws && ok, "gnn_layer_bwd_tf: workspace too small (%zu < %zu)", ws_bytes, w.bytes);
  cudaStream_t st = as_stream(stream);
  const int64_t ldy = round_up(F_out, 4);
  // dZ = dH_out * 1[H_out > 0]
  const float* dz = dH_out;
  int64_t ldz = ldg;
  if (relu) {
    if ((s = launch_relu_mask_f32(csr->n, F_out, dH_out, ldg, H_out, ldo, w.dz, ldy, st)) != GNN_OK)
      return s;
    dz = w.dz;
    ldz = ldy;
  }
  // dY = A^T dZ with the backward messages at width F_out
  s = gnn_spmm_bwd(csr, bnd, dz, ldz, F_out, seed, packed_ws, meta_ws, w.dy, ldy, w.spmm,
                   spmm_workspace_bytes(*csr, F_out), stream);
  if (s != GNN_OK) return s;
  // dW = Hb^T bf16(dY), dH_in = bf16(dY) W^T
  return dense_bwd_impl(Hb, ldhb, csr->n, F_in, W, F_out, w.dy, ldy, nullptr, 0, 0, dH_in, ldh, dW,
                        w.dense, st);
}
