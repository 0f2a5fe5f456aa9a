/*
 * gnnagg.h -- C ABI of the boundary-quantised GCN aggregation library
 * (libgnnagg.so, CUDA kernels for sm_103a).
 *
 * What it computes is the per-layer data path of distributed full-graph GCN
 * training described in the SYLVIE guide ("SYLVIE: 3D-adaptive and Universal
 * System for Large-scale Graph Neural Network Training"): the normalised
 * aggregation of section 2, the boundary messages of section 3, the
 * stochastic integer quantisation of section 6 and the node-importance widths
 * of sections 7 and 9.  Partitions are contiguous node blocks of one graph on
 * one GPU; a message "exchange" is a buffer that stays in device memory.
 *
 * Conventions shared by every call:
 *   - Every function returns a gnn_status; GNN_OK is 0.  Nothing throws.
 *     gnn_last_error() gives a message for the calling thread's last failure.
 *   - Arrays are device pointers owned by the caller.  The library neither
 *     allocates nor frees them; setup calls take an explicit workspace whose
 *     size the matching *_workspace call reports.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) unless the comment says the call
 *     synchronises.  Argument errors are detected on the host and returned
 *     before anything is launched.
 *   - Feature matrices are row-major fp32 with a row stride `ld` (elements)
 *     that is a multiple of 4 and at least F; rows must be 16-byte aligned.
 *     Output columns F..round_up(F,4)-1 are written as zero; columns beyond
 *     that are not touched.
 *   - Bit widths are 1, 2, 4 or 8 (quantised) or 32 (fp32 passed through,
 *     for testing).  F is 1..1024.
 */
#ifndef GNNAGG_H
#define GNNAGG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gnn_status {
  GNN_OK = 0,
  GNN_ERR_INVALID_ARG = 1, /* a NULL pointer, size, stride or alignment out of range */
  GNN_ERR_UNSUPPORTED = 2, /* a valid request this build does not serve (e.g. F > 1024) */
  GNN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  GNN_ERR_DEVICE_CHECK = 4,/* a device-side check flagged bad data */
  GNN_ERR_TIMEOUT = 5,     /* a bounded device wait gave up */
  GNN_ERR_CAPACITY = 6     /* an output buffer is smaller than the result */
} gnn_status;

typedef void* gnn_stream_t; /* cudaStream_t */

/* Thread-local text of the last failure in this thread ("" if none). */
const char* gnn_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int gnn_version(void);
/* Kernels this process has launched through the library so far. */
unsigned long long gnn_kernel_launches(void);

/* ------------------------------------------------------------------------ */
/* CSR adjacency with GCN normalisation.                                    */
/* ------------------------------------------------------------------------ */
#define GNN_CSR_SYMMETRIZE 1u /* add v->u for every u->v                     */
#define GNN_CSR_DEDUP 2u      /* keep one copy of repeated edges             */
#define GNN_CSR_SELF_LOOPS 4u /* drop given self-loops, add one per node     */
#define GNN_CSR_MEAN 8u       /* GraphSAGE mean: weight 1/d_v, not GCN's     */

/* Row v lists the sources u it aggregates (ascending); val[e] is the GCN
 * weight 1/sqrt(d_v d_u) or, with GNN_CSR_MEAN, the mean weight 1/d_v
 * (SYLVIE guide section 2: GraphSAGE changes the neighbour aggregation),
 * computed in fp64 and rounded to fp32, d = row length including the
 * self-loop.  `symmetric` is 1 when A = A^T (symmetrised GCN weights).  The
 * backward calls need A^T: A itself when symmetric, else val_t, the weights
 * of A^T on the same (symmetrised) pattern. */
typedef struct gnn_csr {
  int32_t n;         /* nodes                                     */
  int32_t symmetric; /* 1 if A = A^T by construction              */
  int64_t nnz;       /* entries, self-loops included              */
  int64_t* rowptr;   /* [n+1]                                     */
  int32_t* col;      /* [nnz]                                     */
  float* val;        /* [nnz]                                     */
  /* Optional load-balancing plan filled by gnn_csr_split (all zero/NULL:
   * none).  Rows with more than split_len entries ("long rows", the hubs of
   * a power-law graph) are cut into pieces of split_len entries that run in
   * parallel; the aggregation calls then keep one partial row per piece in
   * their workspace and add the pieces of a row in piece order.             */
  int32_t split_len;  /* 0 = no plan                                         */
  int32_t n_long;     /* long rows                                           */
  int64_t n_pieces;   /* pieces of all long rows                             */
  int32_t* long_rows; /* [n_long] ascending                                  */
  int64_t* piece_ptr; /* [n_long+1] first piece of long row i                */
  int32_t* piece_row; /* [n_pieces] row of piece p                           */
  int64_t* piece_beg; /* [n_pieces] first entry of piece p                   */
  /* Optional A^T weights (NULL: none).  gnn_csr_build fills a caller buffer
   * [capacity] here for GNN_CSR_MEAN with GNN_CSR_SYMMETRIZE: entry e of row
   * u holds A[col[e]][u] = 1/d_col[e].                                      */
  float* val_t;
} gnn_csr;

/* Workspace bytes for gnn_csr_build with these sizes. */
gnn_status gnn_csr_build_workspace(int32_t n, int64_t n_edges, uint32_t flags,
                                   size_t* ws_bytes);

/* Edge list (src[i] -> dst[i], device int32) to CSR, following the GCN layer
 * of the SYLVIE guide, section 2 (aggregation over N(v) plus v itself with
 * weight 1/sqrt(d_v d_u)).  out->rowptr [n+1], out->col and out->val
 * [capacity] are caller buffers; out->n, out->nnz and out->symmetric are set.
 * Synchronises `stream` (the entry count is data-dependent).  Returns
 * GNN_ERR_CAPACITY, with out->nnz set to the needed count, when capacity is
 * too small.  Endpoints must lie in [0, n). */
gnn_status gnn_csr_build(int32_t n, int64_t n_edges, const int32_t* src,
                         const int32_t* dst, uint32_t flags, int64_t capacity,
                         gnn_csr* out, void* ws, size_t ws_bytes,
                         gnn_stream_t stream);

/* Row-split plan for load balance.  gnn_csr_split_count (synchronises)
 * reports the long rows and pieces for split_len >= 32; the caller allocates
 * long_rows [n_long], piece_ptr [n_long+1], piece_row and piece_beg
 * [n_pieces], sets those pointers, split_len, n_long and n_pieces in `csr`,
 * and gnn_csr_split fills them.  Workspace: gnn_csr_split_workspace. */
gnn_status gnn_csr_split_workspace(const gnn_csr* csr, size_t* ws_bytes);
gnn_status gnn_csr_split_count(const gnn_csr* csr, int32_t split_len, int32_t* n_long,
                               int64_t* n_pieces, void* ws, size_t ws_bytes,
                               gnn_stream_t stream);
gnn_status gnn_csr_split(gnn_csr* csr, void* ws, size_t ws_bytes, gnn_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Partitions, boundary slots and per-node bit widths.                       */
/* ------------------------------------------------------------------------ */
/* Width rule.  A boundary node u (one that some other partition aggregates)
 * gets c_u = #{w in pool : d_w <= d_u}, n = pool size (importance c_u/n: the
 * max-degree node has 1, equal degrees share a value, SYLVIE guide section
 * 7), level = #{i < n_levels-1 : 100*c_u > pct[i]*n}, mask = bits[level],
 * and width min(8, mask * base_bits) (section 9); mask 32 passes through.
 * Nodes outside the pool get 0 (they are never sent).  A top-Q% rule is
 * n_levels=2, pct[0]=100-Q. */
typedef struct gnn_bit_rule {
  int32_t n_levels; /* 1..4                                 */
  int32_t pct[3];   /* ascending thresholds in percent      */
  uint8_t bits[4];  /* 1, 2, 4, 8 or 32 per level           */
} gnn_bit_rule;

/* Partition p holds nodes [part_start[p], part_start[p+1]) with
 * part_start[p] = floor(p*n/P).  A slot s is a pair (q, u): node u is
 * aggregated by some node of partition q != part(u), as the boundary nodes of
 * the SYLVIE guide, section 3.  Slots are ordered by q, then u. */
typedef struct gnn_boundary {
  int32_t P;
  int32_t n;
  int64_t n_slots;      /* S                                                   */
  int64_t nnz_cut;      /* CSR entries whose source lies in another partition  */
  int32_t F;            /* feature width slot_off was computed for             */
  int32_t reserved;
  int64_t* part_start;  /* [P+1]                                               */
  int64_t* send_start;  /* [P+1] first slot received by partition q            */
  int32_t* slot_node;   /* [S] u of slot s                                     */
  int32_t* col_remap;   /* [nnz] each row's entries, local sources first (their
                         * ids, in CSR order), then remote ones as ~s of the
                         * slot (part(row), col), in CSR order                 */
  float* val_remap;     /* [nnz] the GCN weights in the same order             */
  int32_t* local_cnt;   /* [n] local entries at the start of each row          */
  int64_t* slot_rowptr; /* [S+1] backward entries of slot s ...                */
  int32_t* slot_col;    /* [nnz_cut] ... the rows v of q that aggregate u,     */
  float* slot_val;      /* [nnz_cut] ... ascending, with their weights A_vu    */
  int64_t* own_ptr;     /* [n+1] slots whose node is u ...                     */
  int32_t* own_slot;    /* [S]   ... ascending s                               */
  uint8_t* node_bits;   /* [n]                                                 */
  uint8_t* slot_bits;   /* [S] = node_bits[slot_node[s]]                       */
  int64_t* slot_off;    /* [S+1] byte offset of slot s in a message buffer     */
  /* Optional list of slots with more than long_slot_len backward entries
   * (gnn_boundary_long_slots; zero/NULL = none).  Their halo partials are
   * summed by a whole thread block each, in the same fixed order.          */
  int32_t long_slot_len;
  int32_t n_long_slots;
  int32_t* long_slots;  /* [n_long_slots] ascending                          */
  /* [nnz] the A^T weights (csr->val_t) in col_remap order; filled by
   * gnn_boundary_index when both it and csr->val_t are non-NULL, and then
   * used by the backward calls in place of val_remap (NULL: A symmetric).   */
  float* val_remap_t;
  /* Optional visiting order of the backward halo kernel (filled by
   * gnn_boundary_long_slots when non-NULL; NULL = slot order): the slots
   * sorted by their first backward entry v, ties by s.  Slots that read the
   * same gradient rows then run at the same time and share those rows in L2.
   * It changes no result: every slot's sum keeps its own fixed order.      */
  int32_t* halo_order;  /* [n_slots]                                        */
} gnn_boundary;

/* Workspace bytes for gnn_boundary_count / _index / _set_bits on this CSR. */
gnn_status gnn_boundary_workspace(const gnn_csr* csr, int32_t P, size_t* ws_bytes);

/* Number of slots and of cut entries for P partitions.  Synchronises. */
gnn_status gnn_boundary_count(const gnn_csr* csr, int32_t P, int64_t* n_slots,
                              int64_t* nnz_cut, void* ws, size_t ws_bytes,
                              gnn_stream_t stream);

/* Fill every array of `out` (allocated by the caller with the sizes from
 * gnn_boundary_count; out->P, out->n_slots and out->nnz_cut set) and the
 * widths and byte offsets for feature width F.  Follows the SYLVIE guide:
 * section 3 (boundary nodes per receiving partition), section 5 step 1 and
 * section 7 (global in-degree importance, node mask), section 9 (combination
 * with the base width).  Synchronises. */
gnn_status gnn_boundary_index(const gnn_csr* csr, const gnn_bit_rule* rule,
                              uint8_t base_bits, int32_t F, gnn_boundary* out,
                              void* ws, size_t ws_bytes, gnn_stream_t stream);

/* Recompute node_bits, slot_bits and slot_off (for F) after the base width
 * changes (section 8: the base width moves between epochs). */
gnn_status gnn_boundary_set_bits(const gnn_csr* csr, const gnn_bit_rule* rule,
                                 uint8_t base_bits, int32_t F, gnn_boundary* bnd,
                                 void* ws, size_t ws_bytes, gnn_stream_t stream);

/* Long-slot list for load balance of the backward halo partials: the count
 * of slots with more than long_slot_len (>= 32) entries (synchronises), then,
 * with bnd->long_slots allocated and long_slot_len / n_long_slots set, the
 * list itself.  Workspace: gnn_boundary_workspace bytes. */
gnn_status gnn_boundary_long_slots_count(const gnn_boundary* bnd, int32_t long_slot_len,
                                         int32_t* n_long_slots, void* ws, size_t ws_bytes,
                                         gnn_stream_t stream);
gnn_status gnn_boundary_long_slots(gnn_boundary* bnd, void* ws, size_t ws_bytes,
                                   gnn_stream_t stream);
/* gnn_boundary_long_slots also fills bnd->halo_order when it is non-NULL
 * (n_slots int32 entries, caller-allocated). */

/* slot_off[s] = sum_{t<s} rowbytes(slot_bits[t], F), slot_off[S] = total,
 * rowbytes(b,F) = 16*ceil(F*b/128) (b=32: 16*ceil(4F/16)).  Every row starts
 * on a 16-byte boundary.  `ws` needs gnn_slot_offsets_workspace bytes. */
gnn_status gnn_slot_offsets_workspace(int64_t n_slots, size_t* ws_bytes);
gnn_status gnn_slot_offsets(const uint8_t* slot_bits, int64_t n_slots, int32_t F,
                            int64_t* slot_off, void* ws, size_t ws_bytes,
                            gnn_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Hot path.                                                                 */
/* ------------------------------------------------------------------------ */
/* Stochastic integer quantisation and packing of message rows, SYLVIE guide
 * section 6: for row r, x = X[row_idx[r]][0..F) (row_idx NULL: row r), width
 * b = row_bits[r]; mn = min x, mx = max x (a zero stored as +0);
 * scale = (mx-mn)/(2^b-1) (0 if mx == mn, all codes 0);
 * code_j = min(2^b-1, floor((x_j-mn)/scale + u_j)),
 * u_j = (hash32(seed, r, j) >> 8) * 2^-24,
 * hash32(seed,r,j) = fmix32(fmix32(seed ^ fmix32(r)) ^ j) (MurmurHash3's
 * 32-bit finaliser), every step IEEE fp32 round-to-nearest without
 * contraction.  Code j goes to bits [b*(j mod 32/b), +b) of little-endian
 * 32-bit word floor(j*b/32) of the row at packed + row_off[r]; the row is
 * zero-padded to rowbytes(b, F).  meta[2r] = mn, meta[2r+1] = scale.  Width
 * 32 stores the fp32 values and meta (0, 0).  row_off[r] must be a multiple
 * of 16.  The row key r is the slot index, so forward and backward messages
 * of a slot draw from the same stream for equal seeds. */
gnn_status gnn_quant_pack(const float* X, int64_t ldx, int32_t F,
                          const int32_t* row_idx, int64_t n_rows,
                          const uint8_t* row_bits, const int64_t* row_off,
                          uint32_t seed, uint8_t* packed, float* meta,
                          gnn_stream_t stream);

/* The forward messages of every slot of `bnd` -- the bytes
 * gnn_quant_pack(X, ldx, F, bnd->slot_node, bnd->n_slots, bnd->slot_bits,
 * bnd->slot_off, seed, packed, meta) writes -- formed node by node along the
 * owner lists (own_slot): a node sent to k partitions is read, and its min,
 * max, scale and quotients (x - mn) / scale formed, once for its k slots;
 * each slot then draws its codes with its own row key.  SYLVIE guide section
 * 6 (the quantiser) and section 3 (one boundary node, several receiving
 * partitions).  Needs own_slot, slot_node, slot_bits, slot_off; checks as
 * gnn_quant_pack. */
gnn_status gnn_quant_pack_owned(const gnn_boundary* bnd, const float* X, int64_t ldx,
                                int32_t F, uint32_t seed, uint8_t* packed, float* meta,
                                gnn_stream_t stream);

/* The division (x - min) / scale exactly as the quantiser performs it:
 * q[i] = a[i] / b[i] rounded to nearest fp32, for verification against
 * IEEE division.  For 2^-76 <= b <= 2^100 the library forms it from the
 * reciprocal of b and two fused corrections (Markstein's method); a result
 * there is exact whenever it is >= 2^-26, and below 2^-25 otherwise (where
 * the quantiser's code is 0 whatever its last bits).  Other b use the IEEE
 * divide.  Device pointers, n elements each.  The pages have no counterpart:
 * it exists so the division the codes depend on can be tested directly. */
gnn_status gnn_quant_divide(const float* a, const float* b, float* q, int64_t n,
                            gnn_stream_t stream);

/* Receive side of section 6: out[r][j] = scale*code_j + mn (fp32 multiply,
 * then fp32 add; width 32 copies the stored value). */
gnn_status gnn_dequant_unpack(const uint8_t* packed, const float* meta,
                              const int64_t* row_off, const uint8_t* row_bits,
                              int64_t n_rows, int32_t F, float* out, int64_t ldo,
                              gnn_stream_t stream);

/* Forward aggregation, SYLVIE guide sections 2, 3 and 11 (receive, dequantise,
 * aggregate): M[v] = sum_e val[e] * x_e with x_e = H[u] for a source u in
 * v's partition and, for a remote u, the dequantised message of slot
 * (part(v), u) read from packed/meta (as gnn_quant_pack wrote them with
 * bnd->slot_bits and bnd->slot_off).  bnd NULL: plain M = A H.  fp32
 * accumulation in any order.  Mb (optional, may be NULL) receives M rounded
 * to bf16 (nearest-even) with row stride ldmb >= round_up(F, 16); its columns
 * F..round_up(F,16)-1 are written as zero so it can feed the dense
 * transform.  ws/ws_bytes: gnn_spmm_workspace bytes (NULL/0 without a split
 * plan); calls that share a workspace must not overlap on the GPU. */
gnn_status gnn_spmm_fwd(const gnn_csr* csr, const gnn_boundary* bnd,
                        const float* H, int64_t ldh, int32_t F,
                        const uint8_t* packed, const float* meta, float* M,
                        int64_t ldm, uint16_t* Mb, int64_t ldmb, void* ws,
                        size_t ws_bytes, gnn_stream_t stream);

/* Workspace bytes the aggregation calls need for `csr`'s split plan at
 * feature width F: n_pieces * round_up(F, 4) * 4 (0 without a plan). */
gnn_status gnn_spmm_workspace(const gnn_csr* csr, int32_t F, size_t* ws_bytes);

/* gnn_spmm_fwd without a workspace, for callers that cannot allocate device
 * memory while they run (a serving loop whose memory is all reserved at
 * start-up, or a plugin that its host framework gives only input and output
 * pointers).  The pages this library follows have no counterpart: it is an
 * interface convenience.  The split plan's partial rows go to a fixed 32 MiB
 * device array inside the library (n_pieces * round_up(F,4) * 4 bytes must fit,
 * else GNN_ERR_UNSUPPORTED with no launch); every GPU that loads the library
 * holds that array until the process exits.  The first call on a device looks
 * up the array's device address with that device current, so make it before
 * any stream capture.  All calls share the array: calls that overlap on the
 * GPU (other streams, other threads) race.  Arguments and results are as for
 * gnn_spmm_fwd. */
gnn_status gnn_spmm_fwd_noalloc(const gnn_csr* csr, const gnn_boundary* bnd,
                                const float* H, int64_t ldh, int32_t F,
                                const uint8_t* packed, const float* meta, float* M,
                                int64_t ldm, uint16_t* Mb, int64_t ldmb,
                                gnn_stream_t stream);

/* Backward aggregation dH = A^T G for symmetric A (section 3: embedding
 * gradients travel back along the same cross-partition dependencies).  With
 * bnd: each slot s = (q, u) first forms the halo partial
 * P_s = sum over its entries (ascending v) of slot_val * G[v], in fp32 with
 * every product and sum rounded (start +0), and quantises/packs it like
 * gnn_quant_pack (row key s, width slot_bits[s], offsets slot_off) into
 * packed_ws / meta_ws (sizes slot_off[S] bytes and 2S floats); then
 * dH[u] = sum over u's local entries of val * G[v] + sum over the slots u
 * owns of their dequantised partials.  bnd NULL: plain A^T G. */
gnn_status gnn_spmm_bwd(const gnn_csr* csr, const gnn_boundary* bnd,
                        const float* G, int64_t ldg, int32_t F, uint32_t seed,
                        uint8_t* packed_ws, float* meta_ws, float* dH,
                        int64_t ldh, void* ws, size_t ws_bytes,
                        gnn_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Dense transform (tcgen05 tensor cores) and whole layers.                   */
/* ------------------------------------------------------------------------ */
/* bf16 operands are raw bf16 bit patterns (uint16).  W is [F_in][F_out]
 * row-major.  F_out must be a multiple of 16, at most 256.  Products
 * accumulate in fp32. */

/* Workspace bytes for gnn_dense_fwd / gnn_dense_bwd with n rows. */
gnn_status gnn_dense_workspace(int64_t n, int32_t F_in, int32_t F_out, size_t* ws_bytes);

/* The transform of the GCN layer, SYLVIE guide section 2 (z = W h after
 * aggregation, h' = sigma(z)): H_out = act(Mb W), Mb [n][ldmb] bf16 with
 * columns F_in..round_up(F_in,16)-1 zero, act = ReLU if relu else identity.
 * H_out is fp32 [n][ldo], ldo >= F_out. */
gnn_status gnn_dense_fwd(const uint16_t* Mb, int64_t ldmb, int64_t n, int32_t F_in,
                         const uint16_t* W, int32_t F_out, int32_t relu, float* H_out,
                         int64_t ldo, void* ws, size_t ws_bytes, gnn_stream_t stream);

/* Backward of the transform: dZ = dH_out * 1[H_out > 0] (relu) or dH_out,
 * rounded to bf16; dM = dZ W^T (fp32 [n][ldm], may be NULL) and the weight
 * gradient of section 7, dW = Mb^T dZ (fp32 [F_in][F_out]), accumulated over
 * row blocks and added in a fixed order (deterministic). */
gnn_status gnn_dense_bwd(const uint16_t* Mb, int64_t ldmb, int64_t n, int32_t F_in,
                         const uint16_t* W, int32_t F_out, const float* dH_out, int64_t ldg,
                         const float* H_out, int64_t ldo, int32_t relu, float* dM, int64_t ldm,
                         float* dW, void* ws, size_t ws_bytes, gnn_stream_t stream);

/* Workspace bytes for gnn_layer_fwd / gnn_layer_bwd on this CSR. */
gnn_status gnn_layer_workspace(const gnn_csr* csr, int32_t F_in, int32_t F_out, size_t* ws_bytes);

/* One forward GCN layer as in the SYLVIE guide, section 11: quantise and pack
 * the boundary rows of H_in (gnn_quant_pack with bnd's slots, widths and
 * offsets, which must be for F_in), aggregate with dequantised remote rows
 * (gnn_spmm_fwd) into Mb (bf16, kept for the backward), then
 * H_out = act(Mb W).  bnd NULL: plain A H. */
gnn_status gnn_layer_fwd(const gnn_csr* csr, const gnn_boundary* bnd, const float* H_in,
                         int64_t ldh, int32_t F_in, const uint16_t* W, int32_t F_out,
                         int32_t relu, uint32_t seed, uint8_t* packed_ws, float* meta_ws,
                         uint16_t* Mb, int64_t ldmb, float* H_out, int64_t ldo, void* ws,
                         size_t ws_bytes, gnn_stream_t stream);

/* One backward GCN layer: gnn_dense_bwd (dW and dM), then, unless dH_in is
 * NULL (the first layer), the boundary-quantised gnn_spmm_bwd of dM with
 * `seed` into dH_in [n][ldh]. */
gnn_status gnn_layer_bwd(const gnn_csr* csr, const gnn_boundary* bnd, const float* dH_out,
                         int64_t ldg, const float* H_out, int64_t ldo, int32_t relu,
                         const uint16_t* Mb, int64_t ldmb, const uint16_t* W, int32_t F_in,
                         int32_t F_out, uint32_t seed, uint8_t* packed_ws, float* meta_ws,
                         float* dW, float* dH_in, int64_t ldh, void* ws, size_t ws_bytes,
                         gnn_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Asynchronous epochs (SYLVIE guide, section 10: boundary messages one      */
/* epoch stale, their quantisation overlapped with local computation).       */
/* ------------------------------------------------------------------------ */
/* The two halves of gnn_spmm_bwd, for callers that overlap them:
 * gnn_halo_quant_pack forms each slot's fixed-order halo partial of G and
 * quantises/packs it (row key s, `seed`) into packed/meta;
 * gnn_spmm_bwd_local computes dH[u] = sum over u's local entries of
 * val * G[v] + the dequantised messages in packed/meta of the slots u owns.
 * gnn_spmm_bwd(G) equals gnn_halo_quant_pack(G) then gnn_spmm_bwd_local(G)
 * with the same buffers. */
gnn_status gnn_halo_quant_pack(const gnn_boundary* bnd, const float* G, int64_t ldg, int32_t F,
                               uint32_t seed, uint8_t* packed, float* meta, gnn_stream_t stream);
/* Slot-range forms for a rank that holds some partitions of a multi-GPU
 * job (SYLVIE guide, section 5: every worker quantises the boundary rows it
 * owns and sends them; section 11: backward messages return to the owners).
 * gnn_quant_pack_slots quantises and packs the message rows of slots
 * s0..s1-1 only (row X[slot_node[s]], width slot_bits[s], row key s, bytes
 * at packed + slot_off[s], meta[2s..2s+1]): the bytes a full gnn_quant_pack
 * over every slot writes there.  gnn_halo_quant_pack_slots forms the
 * backward messages of slots s0..s1-1 only (bytes as gnn_halo_quant_pack
 * writes them).  Neither touches the rows of other slots.  Checks as
 * gnn_quant_pack / gnn_halo_quant_pack; 0 <= s0 <= s1 (<= n_slots). */
gnn_status gnn_quant_pack_slots(const float* X, int64_t ldx, int32_t F, const int32_t* slot_node,
                                int64_t s0, int64_t s1, const uint8_t* slot_bits,
                                const int64_t* slot_off, uint32_t seed, uint8_t* packed,
                                float* meta, gnn_stream_t stream);
gnn_status gnn_halo_quant_pack_slots(const gnn_boundary* bnd, const float* G, int64_t ldg,
                                     int32_t F, int64_t s0, int64_t s1, uint32_t seed,
                                     uint8_t* packed, float* meta, gnn_stream_t stream);
gnn_status gnn_spmm_bwd_local(const gnn_csr* csr, const gnn_boundary* bnd, const float* G,
                              int64_t ldg, int32_t F, const uint8_t* packed, const float* meta,
                              float* dH, int64_t ldh, void* ws, size_t ws_bytes,
                              gnn_stream_t stream);

/* The backward aggregation with the lower layer's ReLU gate fused into its
 * store: dZ = bf16((A^T G) * 1[H_mask > 0]) (round to nearest even; H_mask
 * NULL: no gate), the gradient at the pre-activation of the layer below in
 * the bf16 layout its dense backward reads (row stride ldz >=
 * round_up(F, 64), columns F..ldz-1 written as zero).  H_mask is that
 * layer's output, i.e. this layer's input.  Messages, workspace and checks as
 * gnn_spmm_bwd; the fp32 sums are those gnn_spmm_bwd stores.  No counterpart
 * on the pages: it fuses the elementwise gate into the producing kernel. */
gnn_status gnn_spmm_bwd_masked(const gnn_csr* csr, const gnn_boundary* bnd, const float* G,
                               int64_t ldg, int32_t F, uint32_t seed, uint8_t* packed_ws,
                               float* meta_ws, const float* H_mask, int64_t ldhm, uint16_t* dZ,
                               int64_t ldz, void* ws, size_t ws_bytes, gnn_stream_t stream);

/* The owner-side half of gnn_spmm_bwd_masked, for callers that form the
 * backward messages themselves (gnn_halo_quant_pack) or time the two halves
 * apart: dZ = bf16((local A^T G + the dequantised messages in packed/meta of
 * the slots each row owns) * 1[H_mask > 0]), as gnn_spmm_bwd_local sums them
 * (SYLVIE guide, section 3: backward gradients return along the forward
 * dependencies; section 11: dequantise, then aggregate).  Layout, workspace
 * and checks as gnn_spmm_bwd_masked; gnn_spmm_bwd_masked(G) equals
 * gnn_halo_quant_pack(G) followed by this call with the same buffers. */
gnn_status gnn_spmm_bwd_local_masked(const gnn_csr* csr, const gnn_boundary* bnd,
                                     const float* G, int64_t ldg, int32_t F,
                                     const uint8_t* packed, const float* meta,
                                     const float* H_mask, int64_t ldhm, uint16_t* dZ,
                                     int64_t ldz, void* ws, size_t ws_bytes,
                                     gnn_stream_t stream);

/* gnn_dense_bwd from a given bf16 dZ (as gnn_spmm_bwd_masked writes it; row
 * stride ldz >= round_up(F_out, 64), columns F_out..ldz-1 zero):
 * dM = dZ W^T and dW = Mb^T dZ.  Either output may be NULL. */
gnn_status gnn_dense_bwd_z(const uint16_t* Mb, int64_t ldmb, int64_t n, int32_t F_in,
                           const uint16_t* W, int32_t F_out, const uint16_t* dZ, int64_t ldz,
                           float* dM, int64_t ldm, float* dW, void* ws, size_t ws_bytes,
                           gnn_stream_t stream);

/* An asynchronous forward layer:/* An asynchronous forward layer: the aggregation uses the messages of the
 * previous epoch (packed_prev/meta_prev, as gnn_quant_pack wrote them from
 * that epoch's H_in), while this epoch's H_in is quantised and packed into
 * packed_next/meta_next on `aux` at the same time.  The call orders `stream`
 * after that work (the next buffers are complete when later work on `stream`
 * runs).  Other arguments as gnn_layer_fwd. */
gnn_status gnn_layer_fwd_async(const gnn_csr* csr, const gnn_boundary* bnd, const float* H_in,
                               int64_t ldh, int32_t F_in, const uint16_t* W, int32_t F_out,
                               int32_t relu, uint32_t seed, const uint8_t* packed_prev,
                               const float* meta_prev, uint8_t* packed_next, float* meta_next,
                               uint16_t* Mb, int64_t ldmb, float* H_out, int64_t ldo, void* ws,
                               size_t ws_bytes, gnn_stream_t stream, gnn_stream_t aux);

/* An asynchronous backward layer: dense backward on `stream`; then the
 * owner-side aggregation into dH_in uses the previous epoch's backward
 * messages (packed_prev/meta_prev) while this epoch's halo partials of dM are
 * quantised and packed into packed_next/meta_next on `aux`. */
gnn_status gnn_layer_bwd_async(const gnn_csr* csr, const gnn_boundary* bnd,
                               const float* dH_out, int64_t ldg, const float* H_out, int64_t ldo,
                               int32_t relu, const uint16_t* Mb, int64_t ldmb,
                               const uint16_t* W, int32_t F_in, int32_t F_out, uint32_t seed,
                               const uint8_t* packed_prev, const float* meta_prev,
                               uint8_t* packed_next, float* meta_next, float* dW, float* dH_in,
                               int64_t ldh, void* ws, size_t ws_bytes, gnn_stream_t stream,
                               gnn_stream_t aux);

/* Transform-first layers.  SYLVIE guide section 2 writes the GCN layer as
 * z_v = sum_u 1/sqrt(d_v d_u) W h_u: the transform may run before the
 * aggregation, A (H W) = (A H) W, and then the aggregation and the boundary
 * messages are F_out wide instead of F_in -- fewer bytes when F_out < F_in.
 *
 * gnn_layer_fwd_tf: Hb = bf16(H_in) (caller buffer [n x ldhb], ldhb >=
 * round_up(F_in, 16), kept for the backward); Y = Hb W on tcgen05 (fp32
 * accumulate, caller buffer [n x ldy], ldy >= round_up(F_out, 4)); Y's
 * boundary rows are quantised and packed (bnd offsets for width F_out, key
 * s, `seed`); H_out = act(A Y) with the dequantised messages for remote
 * sources, fp32.  bnd may be NULL (no partitions).
 *
 * gnn_layer_bwd_tf: dZ = dH_out * 1[H_out > 0] (relu) in fp32; dY = A^T dZ
 * with the backward messages at width F_out (as gnn_spmm_bwd); then
 * dW = Hb^T bf16(dY) and, unless dH_in is NULL, dH_in = bf16(dY) W^T.
 * F_out: a multiple of 16, at most 256; workspace from
 * gnn_layer_tf_workspace. */
gnn_status gnn_layer_tf_workspace(const gnn_csr* csr, int32_t F_in, int32_t F_out,
                                  size_t* ws_bytes);
gnn_status gnn_layer_fwd_tf(const gnn_csr* csr, const gnn_boundary* bnd, const float* H_in,
                            int64_t ldh, int32_t F_in, const uint16_t* W, int32_t F_out,
                            int32_t relu, uint32_t seed, uint8_t* packed_ws, float* meta_ws,
                            uint16_t* Hb, int64_t ldhb, float* Y, int64_t ldy, float* H_out,
                            int64_t ldo, void* ws, size_t ws_bytes, gnn_stream_t stream);
gnn_status gnn_layer_bwd_tf(const gnn_csr* csr, const gnn_boundary* bnd, const float* dH_out,
                            int64_t ldg, const float* H_out, int64_t ldo, int32_t relu,
                            const uint16_t* Hb, int64_t ldhb, const uint16_t* W, int32_t F_in,
                            int32_t F_out, uint32_t seed, uint8_t* packed_ws, float* meta_ws,
                            float* dW, float* dH_in, int64_t ldh, void* ws, size_t ws_bytes,
                            gnn_stream_t stream);

/* Attention aggregator (SYLVIE guide section 2: GAT weights the aggregation
 * by attention coefficients alpha_vu; section 12: one head).  Reading: the
 * single-head graph attention layer on the transformed rows,
 *   Y = bf16(H) W,  s_l = Y a_l,  s_r = Y a_r,
 *   e_vu = LeakyReLU(s_l[v] + s_r[u]) (slope 0.2) over u in N(v) + {v},
 *   alpha_v. = softmax(e_v.) (fp32, expf),  H' = act(sum_u alpha_vu Y_u),
 * where a remote source is seen through its dequantised message Y~_u (its
 * score a_r . Y~_u is formed by the receiver).  The pattern must be
 * symmetrised.
 *
 * gnn_gat_index: position maps for the backward: tpos [nnz] (entry order of
 * the aggregation: col_remap with a boundary, col without) gives, for a local
 * entry of row u reading v, the position of v's entry reading u (-1 for a
 * remote entry); spos [nnz_cut] gives, for each slot-CSR entry (s, v), the
 * position of v's entry reading slot s.  Computed once per graph.
 *
 * gnn_gat_layer_fwd: Hb = bf16(H_in), Y (fp32, ldy >= round_up(F_out, 4)),
 * the messages of Y's boundary rows (offsets for F_out, key s, `seed`), the
 * attention alpha [nnz] (entry order as above) and H_out = act(A_alpha Y).
 *
 * gnn_gat_layer_bwd: dZ = dH_out * 1[H_out > 0] (relu); per entry
 * dalpha = dZ_v . x_u (x the row the forward aggregated: Y_u or the
 * dequantised message of packed_fwd/meta_fwd), g = alpha (dalpha -
 * sum alpha dalpha) LeakyReLU'(e) (written to g_out [nnz] when given).  The
 * backward message of slot s is the fixed-order halo partial
 * sum_v alpha_vs dZ_v (start +0, v ascending, products and sums in fp32)
 * followed by fl(P + fl(r_s a_r)), r_s = sum_v g_vs in entry order, then
 * quantised with key s and `seed` into packed_ws/meta_ws.  dY = the local
 * transposed aggregation + the owned messages + ds_r a_r + ds_l a_l;
 * da_l = sum_v ds_l[v] Y_v, da_r = sum_u ds_r[u] Y_u + sum_s r_s Y~_s;
 * dW = Hb^T bf16(dY) and, unless dH_in is NULL, dH_in = bf16(dY) W^T.
 * Workspace from gnn_gat_workspace (same for both directions). */
gnn_status gnn_gat_index(const gnn_csr* csr, const gnn_boundary* bnd, int64_t* tpos,
                         int64_t* spos, gnn_stream_t stream);
gnn_status gnn_gat_workspace(const gnn_csr* csr, const gnn_boundary* bnd, int32_t F_in,
                             int32_t F_out, size_t* ws_bytes);
gnn_status gnn_gat_layer_fwd(const gnn_csr* csr, const gnn_boundary* bnd, const float* H_in,
                             int64_t ldh, int32_t F_in, const uint16_t* W, int32_t F_out,
                             const float* a_l, const float* a_r, int32_t relu, uint32_t seed,
                             uint8_t* packed, float* meta, uint16_t* Hb, int64_t ldhb, float* Y,
                             int64_t ldy, float* alpha, float* H_out, int64_t ldo, void* ws,
                             size_t ws_bytes, gnn_stream_t stream);
gnn_status gnn_gat_layer_bwd(const gnn_csr* csr, const gnn_boundary* bnd, const int64_t* tpos,
                             const int64_t* spos, const float* dH_out, int64_t ldg,
                             const float* H_out, int64_t ldo, int32_t relu, const uint16_t* Hb,
                             int64_t ldhb, const float* Y, int64_t ldy, const float* alpha,
                             const uint8_t* packed_fwd, const float* meta_fwd, const uint16_t* W,
                             const float* a_l, const float* a_r, int32_t F_in, int32_t F_out,
                             uint32_t seed, uint8_t* packed_ws, float* meta_ws, float* dW,
                             float* da_l, float* da_r, float* dH_in, int64_t ldh, float* g_out,
                             void* ws, size_t ws_bytes, gnn_stream_t stream);

/* Cluster-blocked aggregation (the TorchGT guide's cluster-aware layout --
 * place the node pairs with high locality next to each other -- applied to
 * this aggregation).  The local entries (all entries without a boundary) are
 * cut into T x T tiles of (row block, column block); a tile with at least
 * min_entries entries is dense.  A dense tile's source rows are staged in
 * shared memory, 128 columns at a time, and its entries read them there.
 * Every other entry (sparse tiles, remote entries) forms `residual`, a CSR
 * in the aggregation order (local ids, then ~slot), aggregated by the row
 * kernels first; the tiles are then added in tile order.  Needs symmetric
 * weights (GCN).  T must be 128.
 *
 * Build: gnn_blocked_workspace, gnn_blocked_count (synchronises; sizes),
 * allocate the arrays, then gnn_blocked_build.  A split plan for the
 * residual (gnn_csr_split on `residual`) is optional, as for any CSR.
 * gnn_spmm_fwd_blocked / gnn_spmm_bwd_blocked compute what gnn_spmm_fwd /
 * gnn_spmm_bwd (or gnn_spmm_bwd_masked with dZ) compute, the same messages,
 * the fp32 sums in another order; workspace from gnn_blocked_spmm_workspace.
 * No counterpart on the pages for the layout's use here. */
typedef struct gnn_blocked {
  int32_t T;             /* tile edge: 128                                    */
  int32_t n_rb;          /* row blocks, ceil(n / T)                           */
  int64_t n_tiles;       /* dense tiles                                       */
  int64_t n_entries;     /* entries in dense tiles                            */
  int64_t* rb_tile_ptr;  /* [n_rb+1] first dense tile of each row block      */
  int32_t* tile_cb;      /* [n_tiles] column block                           */
  int64_t* tile_ptr;     /* [n_tiles+1] first entry of each tile             */
  int32_t* tile_rowptr;  /* [n_tiles*(T+1)] a tile's row offsets (relative)  */
  uint8_t* ent_col;      /* [n_entries + 16] column within the block (padded) */
  float* ent_val;        /* [n_entries] weight                               */
  gnn_csr residual;      /* rowptr [n+1], col/val [nnz]; nnz = residual count */
  int32_t* res_local_cnt;/* [n] local residual entries per row (with a boundary) */
} gnn_blocked;

gnn_status gnn_blocked_workspace(const gnn_csr* csr, const gnn_boundary* bnd, int32_t T,
                                 int32_t min_entries, size_t* ws_bytes);
gnn_status gnn_blocked_count(const gnn_csr* csr, const gnn_boundary* bnd, int32_t T,
                             int32_t min_entries, int64_t* n_tiles, int64_t* n_entries,
                             int64_t* n_residual, void* ws, size_t ws_bytes, gnn_stream_t stream);
gnn_status gnn_blocked_build(const gnn_csr* csr, const gnn_boundary* bnd, int32_t T,
                             int32_t min_entries, gnn_blocked* out, void* ws, size_t ws_bytes,
                             gnn_stream_t stream);
gnn_status gnn_blocked_spmm_workspace(const gnn_blocked* bp, int32_t F, size_t* ws_bytes);
gnn_status gnn_spmm_fwd_blocked(const gnn_csr* csr, const gnn_boundary* bnd,
                                const gnn_blocked* bp, const float* H, int64_t ldh, int32_t F,
                                const uint8_t* packed, const float* meta, float* M, int64_t ldm,
                                uint16_t* Mb, int64_t ldmb, void* ws, size_t ws_bytes,
                                gnn_stream_t stream);
/* dH (fp32) and/or dZ = bf16(dH * 1[H_mask > 0]) (H_mask may be NULL). */
gnn_status gnn_spmm_bwd_blocked(const gnn_csr* csr, const gnn_boundary* bnd,
                                const gnn_blocked* bp, const float* G, int64_t ldg, int32_t F,
                                uint32_t seed, uint8_t* packed_ws, float* meta_ws,
                                const float* H_mask, int64_t ldhm, float* dH, int64_t ldh,
                                uint16_t* dZ, int64_t ldz, void* ws, size_t ws_bytes,
                                gnn_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Epoch control (SYLVIE guide, sections 8 and 11).  Host code.              */
/* ------------------------------------------------------------------------ */
#define GNN_LDR_MAX_DELTA 64
/* Coordinator, Quant Orchestrator and Pipeline Adaptor state.  After every
 * epoch, gnn_ldr_update takes the partitions' losses and the epoch time:
 * L_t = mean loss, F_t = lambda F_{t-1} + (1 - lambda) L_t (F_0 = L_0),
 * LDR_t = (F_{t-1} - F_t) / et_t, the descent rate (LDR_0 = 0).  Then, for
 * the next epoch: after the first epoch base_bits = b_min; when t > delta,
 * LDR_t < LDR_{t-delta} doubles base_bits (at most b_max) and makes the next
 * epoch synchronous, otherwise base_bits halves (at least b_min) and the next
 * epoch is asynchronous; for 0 < t <= delta nothing changes.  The sign reading
 * (smaller descent rate = worse) follows the pages' prose. */
typedef struct gnn_ldr_state {
  double lambda;     /* smoothing coefficient (0.9 recommended)       */
  int32_t delta;     /* look-back interval in epochs (5, 10, 20)      */
  int32_t b_min;     /* 1                                             */
  int32_t b_max;     /* 8                                             */
  int32_t t;         /* epochs reported so far                        */
  int32_t base_bits; /* base width for the next epoch                 */
  int32_t async_next;/* 1: run the next epoch asynchronously          */
  double F;          /* smoothed loss after the last report           */
  double ldr[GNN_LDR_MAX_DELTA + 1]; /* last delta+1 LDR values (ring) */
} gnn_ldr_state;

gnn_status gnn_ldr_init(gnn_ldr_state* st, double lambda, int32_t delta, int32_t b_min,
                        int32_t b_max);
gnn_status gnn_ldr_update(gnn_ldr_state* st, const double* partition_loss, int32_t n_parts,
                          double epoch_seconds);

/* Synchronise `stream`, then the whole device (a flag can come from a kernel
 * on another stream, e.g. the aux stream of the asynchronous layers), and
 * report device-side failures (GNN_ERR_CUDA for a CUDA error,
 * GNN_ERR_DEVICE_CHECK / GNN_ERR_TIMEOUT for flags the kernels raised).
 * Clears the flags. */
gnn_status gnn_sync_check(gnn_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GNNAGG_H */
