/*
 * coracle.c -- the oracle's bulk routines in plain C.
 *
 * TEST INFRASTRUCTURE ONLY.  The same definitions as oracle.py, written a
 * second time as straight loops so that full-size message buffers (tens of
 * millions of rows) can be checked and the oracle can be timed on every
 * host core.  It is called only by the test suite and by the benchmark's CPU
 * baseline, never by the GPU library, and shares no code with it.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (oracle/coracle.py).
 * -ffp-contract=off keeps every fp32 multiply and add separately rounded, as
 * the definitions below state; fp32 arithmetic is IEEE round-to-nearest.  The
 * only parallelism is one OpenMP loop over independent rows or slots; each
 * row is computed exactly as the sequential definition reads.
 *
 * Sources (the SYLVIE guide, "SYLVIE: 3D-adaptive and Universal System for
 * Large-scale Graph Neural Network Training"):
 *   section 2  -- the GCN aggregation z_v = sum_{u in N(v)+{v}} w_vu h_u;
 *   section 3  -- boundary messages per receiving partition, and backward
 *                 gradients returned along the same dependencies;
 *   section 6  -- quantisation: scale = (max - min)/(2^b - 1),
 *                 q = stochastic_round((h - min)/scale), h~ = scale*q + min;
 *   section 11 -- quantise, exchange, dequantise, aggregate.
 * Readings where the pages are silent (the same as oracle.py): the hash is
 * MurmurHash3's 32-bit finaliser composed as
 * hash32(seed, s, j) = fmix32(fmix32(seed ^ fmix32(s)) ^ j) with
 * u = (hash32 >> 8) * 2^-24; codes are packed LSB-first into little-endian
 * 32-bit words, rows zero-padded to 16*ceil(F*b/128) bytes; a zero min or max
 * is stored as +0; a constant row has scale 0 and codes 0; halo partial sums
 * run in fp32, entries by ascending v, product and sum each rounded.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- threads */
int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_threads(int t) {
#ifdef _OPENMP
  if (t > 0) omp_set_num_threads(t);
#else
  (void)t;
#endif
}

/* ---------------------------------------------------------------- hashing */
/* MurmurHash3's 32-bit finaliser (Austin Appleby, SMHasher, public domain). */
uint32_t orc_fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

uint32_t orc_hash32(uint32_t seed, uint32_t s, uint32_t j) {
  const uint32_t k = orc_fmix32(seed ^ orc_fmix32(s));
  return orc_fmix32(k ^ j);
}

/* ---------------------------------------------------------------- widths */
int64_t orc_rowbytes(int b, int F) {
  if (b == 32) return 16 * (((int64_t)4 * F + 15) / 16);
  return 16 * (((int64_t)F * b + 127) / 128);
}

/* ---------------------------------------------------------------- quantiser */
/* Quantise one fp32 row x[0..F) with width b and row key `key`, and pack it
 * at `out` (rowbytes(b, F) bytes, zero padding included); meta[0] = min,
 * meta[1] = scale (section 6). */
static void quant_pack_row(const float* x, int F, int b, uint32_t key, uint32_t seed,
                           uint8_t* out, float* meta) {
  const int64_t rb = orc_rowbytes(b, F);
  memset(out, 0, (size_t)rb);
  if (b == 32) {
    memcpy(out, x, (size_t)F * sizeof(float));
    meta[0] = 0.0f;
    meta[1] = 0.0f;
    return;
  }
  float mn = x[0], mx = x[0];
  for (int j = 1; j < F; ++j) {
    if (x[j] < mn) mn = x[j];
    if (x[j] > mx) mx = x[j];
  }
  if (mn == 0.0f) mn = 0.0f; /* -0 becomes +0 */
  if (mx == 0.0f) mx = 0.0f;
  const uint32_t top = (1u << b) - 1u;
  const int flat = !(mx > mn);
  const float scale = flat ? 0.0f : (mx - mn) / (float)top;
  meta[0] = mn;
  meta[1] = scale;
  if (flat) return; /* every code 0 */
  const uint32_t rk = orc_fmix32(seed ^ orc_fmix32(key));
  uint32_t* words = (uint32_t*)out;
  for (int j = 0; j < F; ++j) {
    const float t = (x[j] - mn) / scale;
    const float u = (float)(orc_fmix32(rk ^ (uint32_t)j) >> 8) * 0x1p-24f;
    const float r = floorf(t + u);
    uint32_t q = (uint32_t)r;
    if (q > top) q = top;
    const int64_t bit = (int64_t)j * b;
    words[bit >> 5] |= q << (bit & 31);
  }
}

/* Rows X[row_idx[r]] (row_idx NULL: X[r]) for r < n_rows, width bits[r], row
 * key key0 + r, packed at packed + off[r]; meta[2r], meta[2r+1] = (min,
 * scale).  key0 lets a long list of slots be processed in pieces. */
void orc_quant_pack(const float* X, int64_t ldx, int F, const int32_t* row_idx, int64_t n_rows,
                    const uint8_t* bits, const int64_t* off, uint32_t seed, int64_t key0,
                    uint8_t* packed, float* meta) {
#pragma omp parallel for schedule(dynamic, 1024)
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t src = row_idx ? (int64_t)row_idx[r] : r;
    quant_pack_row(X + src * ldx, F, bits[r], (uint32_t)(key0 + r), seed, packed + off[r],
                   meta + 2 * r);
  }
}

/* Dequantised value j of a packed row: fl(fl(scale * code) + min) (section
 * 6's h~ = scale*q + min, multiply and add each rounded); width 32 stores the
 * fp32 value itself. */
static float dequant(const uint8_t* row, int b, float mn, float scale, int j) {
  if (b == 32) {
    float v;
    memcpy(&v, row + 4 * (int64_t)j, sizeof(float));
    return v;
  }
  const uint32_t* words = (const uint32_t*)row;
  const int64_t bit = (int64_t)j * b;
  const uint32_t q = (words[bit >> 5] >> (bit & 31)) & ((1u << b) - 1u);
  const float p = scale * (float)q;
  return p + mn;
}

/* Backward messages (section 3): for every slot s, the halo copy's partial
 * gradient P_s[j] = sum over the slot's entries e (ascending v) of
 * sval[e] * G[scol[e]][j] in fp32 -- start at +0, each product rounded, then
 * each sum rounded -- quantised with row key key0 + s and packed at off[s]
 * (srp, bits, off and meta may start at slot key0 of a longer list). */
void orc_halo_quant_pack(int64_t S, const int64_t* srp, const int32_t* scol, const float* sval,
                         const float* G, int64_t ldg, int F, const uint8_t* bits,
                         const int64_t* off, uint32_t seed, int64_t key0, uint8_t* packed,
                         float* meta) {
#pragma omp parallel
  {
    float* acc = (float*)malloc((size_t)F * sizeof(float));
#pragma omp for schedule(dynamic, 16)
    for (int64_t s = 0; s < S; ++s) {
      for (int j = 0; j < F; ++j) acc[j] = 0.0f;
      for (int64_t e = srp[s]; e < srp[s + 1]; ++e) {
        const float w = sval[e];
        const float* g = G + (int64_t)scol[e] * ldg;
        for (int j = 0; j < F; ++j) {
          const float p = w * g[j];
          acc[j] = acc[j] + p;
        }
      }
      quant_pack_row(acc, F, bits[s], (uint32_t)(key0 + s), seed, packed + off[s], meta + 2 * s);
    }
    free(acc);
  }
}

/* Forward aggregation (sections 2 and 11) of the output rows rows[i]:
 * M[i][j] = sum over the row's entries of w_e * x_e[j] in fp64, x_e = H[u]
 * for a local source (col_remap[e] = u >= 0) and the dequantised message of
 * slot s = ~col_remap[e] from packed/meta otherwise; T[i][j] = the sum of
 * |w_e * x_e[j]| (the scale of the rounding-error bound). */
void orc_spmm_fwd_rows(const int64_t* rowptr, const int32_t* col_remap, const float* val_remap,
                       const float* H, int64_t ldh, int F, const uint8_t* packed,
                       const float* meta, const uint8_t* slot_bits, const int64_t* slot_off,
                       const int64_t* rows, int64_t n_rows, double* M, double* T) {
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t v = rows[i];
    double* m = M + i * F;
    double* t = T + i * F;
    for (int j = 0; j < F; ++j) m[j] = t[j] = 0.0;
    for (int64_t e = rowptr[v]; e < rowptr[v + 1]; ++e) {
      const double w = (double)val_remap[e];
      const int32_t c = col_remap[e];
      if (c >= 0) {
        const float* h = H + (int64_t)c * ldh;
        for (int j = 0; j < F; ++j) {
          const double p = w * (double)h[j];
          m[j] += p;
          t[j] += fabs(p);
        }
      } else {
        const int64_t s = ~(int64_t)c;
        const uint8_t* row = packed + slot_off[s];
        for (int j = 0; j < F; ++j) {
          const double p = w * (double)dequant(row, slot_bits[s], meta[2 * s], meta[2 * s + 1], j);
          m[j] += p;
          t[j] += fabs(p);
        }
      }
    }
  }
}

/* Backward aggregation (section 3) of the rows rows[i]:
 * dH[i][j] = sum over row u's local entries of wt_e * G[v][j] (wt: the A^T
 * weights in col_remap order; remote entries are skipped, their
 * contribution arrives as messages) + the dequantised backward messages of
 * the slots u owns (own_slot[own_ptr[u] .. own_ptr[u+1])), in fp64; T as in
 * the forward. */
void orc_spmm_bwd_rows(const int64_t* rowptr, const int32_t* col_remap, const float* wt,
                       const float* G, int64_t ldg, int F, const int64_t* own_ptr,
                       const int32_t* own_slot, const uint8_t* packed, const float* meta,
                       const uint8_t* slot_bits, const int64_t* slot_off, const int64_t* rows,
                       int64_t n_rows, double* dH, double* T) {
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t u = rows[i];
    double* d = dH + i * F;
    double* t = T + i * F;
    for (int j = 0; j < F; ++j) d[j] = t[j] = 0.0;
    for (int64_t e = rowptr[u]; e < rowptr[u + 1]; ++e) {
      const int32_t c = col_remap[e];
      if (c < 0) continue;
      const double w = (double)wt[e];
      const float* g = G + (int64_t)c * ldg;
      for (int j = 0; j < F; ++j) {
        const double p = w * (double)g[j];
        d[j] += p;
        t[j] += fabs(p);
      }
    }
    for (int64_t k = own_ptr[u]; k < own_ptr[u + 1]; ++k) {
      const int64_t s = own_slot[k];
      const uint8_t* row = packed + slot_off[s];
      for (int j = 0; j < F; ++j) {
        const double x = (double)dequant(row, slot_bits[s], meta[2 * s], meta[2 * s + 1], j);
        d[j] += x;
        t[j] += fabs(x);
      }
    }
  }
}
