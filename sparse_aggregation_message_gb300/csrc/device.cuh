// Device helpers: hashing, the fp32 quantiser, packing and unpacking of
// message rows held in registers.
//
// Register layout used by every row kernel: a group of G lanes (G a power of
// two, G divides 32) owns one row; lane g of the group holds the 4-element
// chunks c = g + i*G for i < CPL, chunk c covering elements 4c..4c+3.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gnn {

// MurmurHash3's 32-bit finaliser (Appleby, SMHasher, public domain).
__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

// Per-row part of hash32(seed, r, j) = fmix32(fmix32(seed ^ fmix32(r)) ^ j).
__device__ __forceinline__ uint32_t row_key(uint32_t seed, uint32_t r) {
  return fmix32(seed ^ fmix32(r));
}

__device__ __forceinline__ uint32_t group_mask(int G, int lane) {
  return G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
}

__device__ __forceinline__ float elem(const float4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint32_t rowbytes_dev(int b, int F) {
  return b == 32 ? 16u * ((4u * F + 15u) / 16u) : 16u * ((uint32_t)(F * b + 127) / 128u);
}

// The quantiser's true division a / b, correctly rounded, with the
// reciprocal of the row's scale b formed once per row.  Markstein's method
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with y = RN(1/b) and
// a faithful quotient q, the residual r = a - b q is exact and RN(q + r y) is
// RN(a / b).  q0 = RN(a y) is within 1.5 ulp of a/b; one correction makes it
// faithful, the second rounds it correctly.  The identity needs the residuals
// and the reciprocal to stay normal: for 2^-76 <= b <= 2^100 every quotient at
// or above 2^-26 is exact, and a smaller one stays below 2^-25, where the
// stochastic rounding gives code 0 whatever its last bits (t + u < 1 - 2^-25
// for every u <= 1 - 2^-24).  Other b take the IEEE divide.
struct Divisor {
  float b, y;
  bool fast;
};

__device__ __forceinline__ Divisor make_divisor(float b) {
  Divisor d;
  d.b = b;
  d.fast = b >= 0x1p-76f && b <= 0x1p100f;
  d.y = d.fast ? __frcp_rn(b) : 0.f;
  return d;
}

// FAST: the row's divisor is in the reciprocal method's range (d.fast).
template <bool FAST>
__device__ __forceinline__ float div_rn(float a, const Divisor& d) {
  if (!FAST) return __fdiv_rn(a, d.b);
  float q = __fmul_rn(a, d.y);
  q = __fmaf_rn(__fmaf_rn(-d.b, q, a), d.y, q);     // faithful
  return __fmaf_rn(__fmaf_rn(-d.b, q, a), d.y, q);  // correctly rounded
}

// Paired fp32 arithmetic: each lane of a float2 rounded exactly as the
// scalar operation (sm_100's packed FMA/MUL/ADD issue two IEEE operations
// per instruction).  A paired multiply whose result feeds a paired add may be
// contracted into one fused multiply-add by the code generator even with an
// explicit .rn (measured), so they are used only where no multiply feeds an
// add: fused multiply-adds, sums of loaded values, and the quantiser's
// subtract / multiply / fused-correction chain.
__device__ __forceinline__ float2 dup2(float a) { return make_float2(a, a); }

__device__ __forceinline__ unsigned long long pack2(float2 v) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}

__device__ __forceinline__ float2 unpack2(unsigned long long r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}

__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)));
  return unpack2(d);
}

__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)));
  return unpack2(d);
}

__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)), "l"(pack2(c)));
  return unpack2(d);
}

// div_rn on a pair of dividends.
template <bool FAST>
__device__ __forceinline__ float2 div2_rn(float2 a, const Divisor& d) {
  if (!FAST) return make_float2(__fdiv_rn(a.x, d.b), __fdiv_rn(a.y, d.b));
  const float2 y = dup2(d.y), nb = dup2(-d.b);
  float2 q = mul2_rn(a, y);
  q = fma2_rn(fma2_rn(nb, q, a), y, q);     // faithful
  return fma2_rn(fma2_rn(nb, q, a), y, q);  // correctly rounded
}

// The rest of fmix32 after its first step h ^= h >> 16.
__device__ __forceinline__ uint32_t fmix32_tail(uint32_t h) {
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

// Codes of one quantised row at compile-time width B, packed into 32-bit
// words: the 8/B chunks of a word sit on consecutive lanes of the group and
// are OR-ed together with shuffles; zero words pad the row to rowbytes(B, F).
// u_j * 2^24 is an integer below 2^24, so RN(t + u) is formed by one fused
// multiply-add of that integer by 2^-24 (exact) and t.  hash32 of element
// j = 4c + k (k < 4) is fmix32(key ^ j); j and 4c differ only in their two
// low bits, so key ^ j = (key ^ 4c) ^ k and (key ^ j) >> 16 = (key ^ 4c) >> 16,
// and fmix32's first step gives A_c ^ k with A_c formed once per chunk.
template <int G, int CPL, int B>
__device__ __forceinline__ void pack_codes_t(const float4 (&t)[CPL], int F, bool flat, uint32_t key,
                                           uint32_t* __restrict__ words, int gl, uint32_t gmask) {
  constexpr uint32_t TOP = (1u << B) - 1u;
  constexpr int PER_WORD = 8 / B;  // chunks per 32-bit word
  const int nch = (F + 3) >> 2;
  const int slots = (int)(rowbytes_dev(B, F) * 2u) / B;  // chunk slots of the padded row
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = gl + i * G;
    uint32_t part = 0;
    if (c < nch && !flat) {
      // all four codes, then the fields of elements >= F cleared (their
      // quotients come from in-row values, so no element is special-cased)
      const uint32_t kc = key ^ (uint32_t)(4 * c);
      const uint32_t a = kc ^ (kc >> 16);
      const float2 m01 = make_float2(static_cast<float>(fmix32_tail(a) >> 8),
                                     static_cast<float>(fmix32_tail(a ^ 1u) >> 8));
      const float2 m23 = make_float2(static_cast<float>(fmix32_tail(a ^ 2u) >> 8),
                                     static_cast<float>(fmix32_tail(a ^ 3u) >> 8));
      const float2 e24 = dup2(5.9604644775390625e-08f);
      const float2 r01 = fma2_rn(m01, e24, make_float2(t[i].x, t[i].y));
      const float2 r23 = fma2_rn(m23, e24, make_float2(t[i].z, t[i].w));
      // floor(t + u) >= 0 and below 2^24: round down while converting
      part = min(__float2uint_rd(r01.x), TOP) | (min(__float2uint_rd(r01.y), TOP) << B) |
             (min(__float2uint_rd(r23.x), TOP) << (2 * B)) |
             (min(__float2uint_rd(r23.y), TOP) << (3 * B));
      const int nv = F - 4 * c;  // elements of chunk c below F, >= 1
      if (nv < 4) part &= (1u << (B * nv)) - 1u;
    }
    if (PER_WORD > 1) {
      part <<= (c % PER_WORD) * 4 * B;
#pragma unroll
      for (int o = 1; o < PER_WORD; o <<= 1) part |= __shfl_xor_sync(gmask, part, o);
    }
    if (c < slots && (c % PER_WORD) == 0) words[(c * B) >> 3] = part;
  }
}

// The per-row part of the quantiser for the group's row held in v[]
// (elements >= F ignored) at width b < 32: min and max (a zero stored as +0),
// scale = (mx - mn) / (2^b - 1) (0 for a constant row: flat), and the
// quotients t = (x - mn) / scale of every element, correctly rounded.  The
// codes of any row key follow from t alone (pack_codes_t), so a row sent to
// several partitions is prepared once.  All lanes of the group must call.
template <int G, int CPL>
__device__ __forceinline__ void quant_prepare(const float4 (&v)[CPL], int F, int b, int gl,
                                              uint32_t gmask, float4 (&t)[CPL], float& mn_out,
                                              float& scale_out, bool& flat_out) {
  const int nch = (F + 3) >> 2;
  // elements >= F of the last chunk take the chunk's first element: min,
  // max and the codes of the other elements are unchanged by in-row values
  float4 x[CPL];
  float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = gl + i * G;
    x[i] = v[i];
    const int nv = F - 4 * c;
    if (nv < 4) {
      if (nv < 2) x[i].y = x[i].x;
      if (nv < 3) x[i].z = x[i].x;
      x[i].w = x[i].x;
    }
    if (c < nch) {
      // three-input min / max (sm_100+): two instructions per chunk each
      // instead of four (the quantiser is bound by this pipe: measured 0.8%)
      float a, b2;
      asm("min.f32 %0, %1, %2, %3;" : "=f"(a) : "f"(mn), "f"(x[i].x), "f"(x[i].y));
      asm("min.f32 %0, %1, %2, %3;" : "=f"(mn) : "f"(a), "f"(x[i].z), "f"(x[i].w));
      asm("max.f32 %0, %1, %2, %3;" : "=f"(b2) : "f"(mx), "f"(x[i].x), "f"(x[i].y));
      asm("max.f32 %0, %1, %2, %3;" : "=f"(mx) : "f"(b2), "f"(x[i].z), "f"(x[i].w));
    }
  }
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(gmask, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, o));
  }
  if (__float_as_uint(mn) == 0x80000000u) mn = 0.f;  // a zero min/max is stored as +0
  if (__float_as_uint(mx) == 0x80000000u) mx = 0.f;
  const float top = static_cast<float>((1u << b) - 1u);  // exact: 2^b - 1 < 2^24
  const bool flat = !(mx > mn);
  const float scale = flat ? 0.f : __fdiv_rn(__fsub_rn(mx, mn), top);
  const Divisor dv = make_divisor(scale);
  // x - min (as x + (-min): the same IEEE result), then the division
  const float2 nmn = dup2(-mn);
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = gl + i * G;
    t[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < nch && !flat) {
      float2 t01, t23;
      if (dv.fast) {
        t01 = div2_rn<true>(add2_rn(make_float2(x[i].x, x[i].y), nmn), dv);
        t23 = div2_rn<true>(add2_rn(make_float2(x[i].z, x[i].w), nmn), dv);
      } else {
        t01 = div2_rn<false>(add2_rn(make_float2(x[i].x, x[i].y), nmn), dv);
        t23 = div2_rn<false>(add2_rn(make_float2(x[i].z, x[i].w), nmn), dv);
      }
      t[i] = make_float4(t01.x, t01.y, t23.x, t23.y);
    }
  }
  mn_out = mn;
  scale_out = scale;
  flat_out = flat;
}

// Codes of the prepared row t at width b (< 32) with row key `key`, packed
// into the 16-byte aligned row at `words`.
template <int G, int CPL>
__device__ __forceinline__ void pack_codes_b(const float4 (&t)[CPL], int F, int b, bool flat,
                                             uint32_t key, uint32_t* __restrict__ words, int gl,
                                             uint32_t gmask) {
  switch (b) {
    case 1: pack_codes_t<G, CPL, 1>(t, F, flat, key, words, gl, gmask); break;
    case 2: pack_codes_t<G, CPL, 2>(t, F, flat, key, words, gl, gmask); break;
    case 4: pack_codes_t<G, CPL, 4>(t, F, flat, key, words, gl, gmask); break;
    default: pack_codes_t<G, CPL, 8>(t, F, flat, key, words, gl, gmask); break;
  }
}

// Width 32: the row's fp32 values, elements >= F zeroed.
template <int G, int CPL>
__device__ __forceinline__ void store_raw_row(const float4 (&v)[CPL], int F, uint8_t* __restrict__ out,
                                              int gl) {
  const int nch = (F + 3) >> 2;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = gl + i * G;
    if (c < nch) {
      float4 x = v[i];
      const int j0 = 4 * c;
      if (j0 + 1 >= F) x.y = 0.f;
      if (j0 + 2 >= F) x.z = 0.f;
      if (j0 + 3 >= F) x.w = 0.f;
      reinterpret_cast<float4*>(out)[c] = x;
    }
  }
}

template <int G, int CPL, int B, bool FAST>
__device__ __forceinline__ void pack_codes(const float4 (&v)[CPL], int F, float mn, const Divisor& dv,
                                           bool flat, uint32_t key, uint32_t* __restrict__ words,
                                           int gl, uint32_t gmask) {
  constexpr uint32_t TOP = (1u << B) - 1u;
  constexpr int PER_WORD = 8 / B;  // chunks per 32-bit word
  const int nch = (F + 3) >> 2;
  const int slots = (int)(rowbytes_dev(B, F) * 2u) / B;  // chunk slots of the padded row
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = gl + i * G;
    uint32_t part = 0;
    if (c < nch && !flat) {
      // all four codes, then the fields of elements >= F cleared (the caller
      // gives those elements in-row values, so no element is special-cased)
      const uint32_t kc = key ^ (uint32_t)(4 * c);
      const uint32_t a = kc ^ (kc >> 16);
      // x - min (as x + (-min): the same IEEE result), then the division
      const float2 nmn = dup2(-mn);
      const float2 t01 = div2_rn<FAST>(add2_rn(make_float2(v[i].x, v[i].y), nmn), dv);
      const float2 t23 = div2_rn<FAST>(add2_rn(make_float2(v[i].z, v[i].w), nmn), dv);
      const float2 m01 = make_float2(static_cast<float>(fmix32_tail(a) >> 8),
                                     static_cast<float>(fmix32_tail(a ^ 1u) >> 8));
      const float2 m23 = make_float2(static_cast<float>(fmix32_tail(a ^ 2u) >> 8),
                                     static_cast<float>(fmix32_tail(a ^ 3u) >> 8));
      const float2 e24 = dup2(5.9604644775390625e-08f);
      const float2 r01 = fma2_rn(m01, e24, t01), r23 = fma2_rn(m23, e24, t23);
      // floor(t + u) >= 0 and below 2^24: round down while converting
      part = min(__float2uint_rd(r01.x), TOP) | (min(__float2uint_rd(r01.y), TOP) << B) |
             (min(__float2uint_rd(r23.x), TOP) << (2 * B)) |
             (min(__float2uint_rd(r23.y), TOP) << (3 * B));
      const int nv = F - 4 * c;  // elements of chunk c below F, >= 1
      if (nv < 4) part &= (1u << (B * nv)) - 1u;
    }
    if (PER_WORD > 1) {
      part <<= (c % PER_WORD) * 4 * B;
#pragma unroll
      for (int o = 1; o < PER_WORD; o <<= 1) part |= __shfl_xor_sync(gmask, part, o);
    }
    if (c < slots && (c % PER_WORD) == 0) words[(c * B) >> 3] = part;
  }
}

// Quantises the group's row held in v[] (elements >= F ignored) with width b
// and row key `key`, writes the packed row at `out` (16-byte aligned) and
// (mn, scale) at meta (lane 0 of the group).  All lanes of the group must
// call.  Groups of at least 8 lanes (one 1-bit word spans 8 chunks).
template <int G, int CPL>
__device__ __forceinline__ void quantize_pack_row(const float4 (&v)[CPL], int F, int b,
                                                  uint32_t key, uint8_t* __restrict__ out,
                                                  float2* __restrict__ meta, int gl,
                                                  uint32_t gmask) {
  const int nch = (F + 3) >> 2;
  if (b == 32) {
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = gl + i * G;
      if (c < nch) {
        float4 x = v[i];
        const int j0 = 4 * c;
        if (j0 + 1 >= F) x.y = 0.f;
        if (j0 + 2 >= F) x.z = 0.f;
        if (j0 + 3 >= F) x.w = 0.f;
        reinterpret_cast<float4*>(out)[c] = x;
      }
    }
    if (gl == 0) *meta = make_float2(0.f, 0.f);
    return;
  }
  // elements >= F of the last chunk take the chunk's first element: min,
  // max and the codes of the other elements are unchanged by in-row values
  float4 x[CPL];
  float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = gl + i * G;
    x[i] = v[i];
    const int nv = F - 4 * c;
    if (nv < 4) {
      if (nv < 2) x[i].y = x[i].x;
      if (nv < 3) x[i].z = x[i].x;
      x[i].w = x[i].x;
    }
    if (c < nch) {
      // three-input min / max (sm_100+): two instructions per chunk each
      // instead of four (the quantiser is bound by this pipe: measured 0.8%)
      float a, b2;
      asm("min.f32 %0, %1, %2, %3;" : "=f"(a) : "f"(mn), "f"(x[i].x), "f"(x[i].y));
      asm("min.f32 %0, %1, %2, %3;" : "=f"(mn) : "f"(a), "f"(x[i].z), "f"(x[i].w));
      asm("max.f32 %0, %1, %2, %3;" : "=f"(b2) : "f"(mx), "f"(x[i].x), "f"(x[i].y));
      asm("max.f32 %0, %1, %2, %3;" : "=f"(mx) : "f"(b2), "f"(x[i].z), "f"(x[i].w));
    }
  }
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(gmask, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, o));
  }
  if (__float_as_uint(mn) == 0x80000000u) mn = 0.f;  // a zero min/max is stored as +0
  if (__float_as_uint(mx) == 0x80000000u) mx = 0.f;
  const float top = static_cast<float>((1u << b) - 1u);  // exact: 2^b - 1 < 2^24
  const bool flat = !(mx > mn);
  const float scale = flat ? 0.f : __fdiv_rn(__fsub_rn(mx, mn), top);
  uint32_t* words = reinterpret_cast<uint32_t*>(out);
  const Divisor dv = make_divisor(scale);
  if (dv.fast || flat) {
    switch (b) {
      case 1: pack_codes<G, CPL, 1, true>(x, F, mn, dv, flat, key, words, gl, gmask); break;
      case 2: pack_codes<G, CPL, 2, true>(x, F, mn, dv, flat, key, words, gl, gmask); break;
      case 4: pack_codes<G, CPL, 4, true>(x, F, mn, dv, flat, key, words, gl, gmask); break;
      default: pack_codes<G, CPL, 8, true>(x, F, mn, dv, flat, key, words, gl, gmask); break;
    }
  } else {
    switch (b) {
      case 1: pack_codes<G, CPL, 1, false>(x, F, mn, dv, flat, key, words, gl, gmask); break;
      case 2: pack_codes<G, CPL, 2, false>(x, F, mn, dv, flat, key, words, gl, gmask); break;
      case 4: pack_codes<G, CPL, 4, false>(x, F, mn, dv, flat, key, words, gl, gmask); break;
      default: pack_codes<G, CPL, 8, false>(x, F, mn, dv, flat, key, words, gl, gmask); break;
    }
  }
  if (gl == 0) *meta = make_float2(mn, scale);
}

// quantize_pack_row (above) as quant_prepare then pack_codes_t: the same
// bytes; the ring kernel of the backward messages measured faster with it
// (37.8 against 42.1 ms on the R-MAT graph), the per-slot quantiser slower
// (16.3 against 14.2 ms), so each takes its own.
template <int G, int CPL>
__device__ __forceinline__ void quantize_pack_row_split(const float4 (&v)[CPL], int F, int b,
                                                  uint32_t key, uint8_t* __restrict__ out,
                                                  float2* __restrict__ meta, int gl,
                                                  uint32_t gmask) {
  if (b == 32) {
    store_raw_row<G, CPL>(v, F, out, gl);
    if (gl == 0) *meta = make_float2(0.f, 0.f);
    return;
  }
  float4 t[CPL];
  float mn, scale;
  bool flat;
  quant_prepare<G, CPL>(v, F, b, gl, gmask, t, mn, scale, flat);
  pack_codes_b<G, CPL>(t, F, b, flat, key, reinterpret_cast<uint32_t*>(out), gl, gmask);
  if (gl == 0) *meta = make_float2(mn, scale);
}

// A code k < 2^23 as an exact float without a conversion instruction: the
// float whose mantissa field holds k and whose exponent is 23 is 2^23 + k,
// and subtracting 2^23 from it is exact (measured: the forward aggregation
// 2.4% faster than with integer-to-float conversions).
__device__ __forceinline__ float code_to_float(uint32_t k) {
  return __fadd_rn(__uint_as_float(0x4B000000u | k), -8388608.0f);
}

// The 4 dequantised values fl(fl(scale * code) + min) of the codes in the low
// 4b bits of bits4 (width b < 32).
__device__ __forceinline__ float4 dequant4(uint32_t bits4, int b, float mn, float scale) {
  const uint32_t m = (1u << b) - 1u;
  float4 r;
  r.x = __fadd_rn(__fmul_rn(scale, code_to_float(bits4 & m)), mn);
  r.y = __fadd_rn(__fmul_rn(scale, code_to_float((bits4 >> b) & m)), mn);
  r.z = __fadd_rn(__fmul_rn(scale, code_to_float((bits4 >> (2 * b)) & m)), mn);
  r.w = __fadd_rn(__fmul_rn(scale, code_to_float((bits4 >> (3 * b)) & m)), mn);
  return r;
}

// The 4 dequantised values of chunk c of a packed row (width b, meta m).
__device__ __forceinline__ float4 dequant_chunk(const uint8_t* __restrict__ row, int b,
                                                float mn, float scale, int c) {
  if (b == 32) return __ldg(reinterpret_cast<const float4*>(row) + c);
  const uint32_t bitpos = (uint32_t)(4 * c * b);
  const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(row) + (bitpos >> 5));
  const uint32_t bits4 = w >> (bitpos & 31u);
  return dequant4(bits4, b, mn, scale);
}

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& x) {
  const float2 ww = dup2(w);
  const float2 lo = fma2_rn(ww, make_float2(x.x, x.y), make_float2(acc.x, acc.y));
  const float2 hi = fma2_rn(ww, make_float2(x.z, x.w), make_float2(acc.z, acc.w));
  acc = make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ void add4(float4& acc, const float4& x) {
  const float2 lo = add2_rn(make_float2(acc.x, acc.y), make_float2(x.x, x.y));
  const float2 hi = add2_rn(make_float2(acc.z, acc.w), make_float2(x.z, x.w));
  acc = make_float4(lo.x, lo.y, hi.x, hi.y);
}

// acc = fl(acc + fl(w * x)) element by element (product and sum each
// rounded: the fixed-order halo partial sums).  Scalar: the paired multiply
// and add can be contracted into one fused operation by the code generator,
// the scalar _rn forms never are.
__device__ __forceinline__ void mul_add4(float4& acc, float w, const float4& x) {
  acc.x = __fadd_rn(acc.x, __fmul_rn(w, x.x));
  acc.y = __fadd_rn(acc.y, __fmul_rn(w, x.y));
  acc.z = __fadd_rn(acc.z, __fmul_rn(w, x.z));
  acc.w = __fadd_rn(acc.w, __fmul_rn(w, x.w));
}

// 16-byte asynchronous copy global -> shared (cached in L2 only), the commit
// of the copies issued so far as one group, and the wait until at most the N
// newest groups are still in flight.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gsrc)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Stores chunk c of an fp32 row, zeroing elements >= F.
__device__ __forceinline__ void store_chunk_f32(float* __restrict__ row, int c, int F, float4 x) {
  const int j0 = 4 * c;
  if (j0 + 1 >= F) x.y = 0.f;
  if (j0 + 2 >= F) x.z = 0.f;
  if (j0 + 3 >= F) x.w = 0.f;
  reinterpret_cast<float4*>(row)[c] = x;
}

// Stores chunk c of a bf16 row (4 values, 8 bytes), zeroing elements >= F.
__device__ __forceinline__ void store_chunk_bf16(__nv_bfloat16* __restrict__ row, int c, int F,
                                                 float4 x) {
  const int j0 = 4 * c;
  if (j0 >= F) x.x = 0.f;
  if (j0 + 1 >= F) x.y = 0.f;
  if (j0 + 2 >= F) x.z = 0.f;
  if (j0 + 3 >= F) x.w = 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
  uint2 p;
  p.x = *reinterpret_cast<uint32_t*>(&lo);
  p.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(row)[c] = p;
}

}  // namespace gnn
