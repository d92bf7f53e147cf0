/*
 * synth.h - seeded synthetic inputs for the W12 verify path.
 *
 * This module makes test and benchmark INPUTS only: bf16 weight matrices with
 * the per-channel distribution of the verify workloads, bf16 activations,
 * random draft trees and draft tokens.  It holds none of the W12 arithmetic
 * (no window choice, no record packing, no decode, no GEMM).  Both the CPU
 * oracle's callers and the GPU path's callers draw their inputs from here, so
 * the same seed gives the same bf16 bits on either side.
 *
 * Every value is a pure function of (key, counter): the generator is the
 * splitmix64 sequence (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), read at an arbitrary position.  The
 * floating-point steps use only IEEE add, multiply, divide and square root
 * with round-to-nearest-even and no contraction, so host (x86-64, AArch64)
 * and device produce identical bits.  The logarithm and exp2 below are our
 * own short series, written from their Taylor expansions.
 *
 * Weight recipe (per matrix, per output channel n):
 *   s_n = 0.005 * 10^u,  u ~ U(0,1)         (log-uniform in [0.005, 0.05])
 *   w   = bf16_rne(z * s_n),  z ~ N(0,1)     (Marsaglia polar method)
 *   then, from one 32-bit uniform c per element:
 *     c < 0.005  -> outlier:  w * 2^9
 *     c < 0.007  -> exact zero with a random sign
 *     c < 0.008  -> bf16 denormal: random sign, mantissa uniform in 1..127
 * Head recipe (the *_ex calls with outliers = 0): the same without the outliers,
 * for an INT8 head, whose per-channel scale an outlier would set.
 */
#ifndef W12_SYNTH_H
#define W12_SYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYN_HD __host__ __device__ __forceinline__
#else
#define SYN_HD static inline
#endif

#if defined(__CUDA_ARCH__)
#define SYN_MUL(a, b) __fmul_rn((a), (b))
#define SYN_ADD(a, b) __fadd_rn((a), (b))
#define SYN_DIV(a, b) __fdiv_rn((a), (b))
#define SYN_SQRT(a) __fsqrt_rn(a)
#define SYN_F2U(f) __float_as_uint(f)
#define SYN_U2F(u) __uint_as_float(u)
#else
#include <math.h>
#include <string.h>
#define SYN_MUL(a, b) ((a) * (b))
#define SYN_ADD(a, b) ((a) + (b))
#define SYN_DIV(a, b) ((a) / (b))
#define SYN_SQRT(a) sqrtf(a)
SYN_HD uint32_t syn_f2u_host(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
SYN_HD float syn_u2f_host(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
#define SYN_F2U(f) syn_f2u_host(f)
#define SYN_U2F(u) syn_u2f_host(u)
#endif

#define SYN_GAMMA 0x9e3779b97f4a7c15ULL

/* Stream ids inside one matrix key. */
enum { SYN_S_SCALE = 1, SYN_S_CAT = 2, SYN_S_GAUSS = 3, SYN_S_TREE = 4, SYN_S_DRAFT = 5 };

/* splitmix64 output function. */
SYN_HD uint64_t syn_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

/* Element `ctr` of the splitmix64 sequence whose state starts at `key`. */
SYN_HD uint64_t syn_at(uint64_t key, uint64_t ctr) {
  return syn_mix64(key + (ctr + 1ULL) * SYN_GAMMA);
}

/* Key of one tensor: (seed, layer, tensor id) -> 64-bit key. */
SYN_HD uint64_t syn_key(uint64_t seed, uint64_t layer, uint64_t tensor) {
  uint64_t k = syn_mix64(seed + SYN_GAMMA);
  k = syn_mix64(k + layer + SYN_GAMMA);
  return syn_mix64(k + tensor + SYN_GAMMA);
}

SYN_HD uint64_t syn_substream(uint64_t key, uint64_t s) { return syn_mix64(key ^ (s * SYN_GAMMA)); }

/* ln(v) for 0 < v < 1 (normal floats): v = 2^e f, f in [sqrt(1/2), sqrt(2)),
 * ln f = 2 atanh(t), t = (f-1)/(f+1), atanh series to t^9. */
SYN_HD float syn_log(float v) {
  uint32_t u = SYN_F2U(v);
  int e = (int)((u >> 23) & 0xFF) - 127;
  float f = SYN_U2F((u & 0x007FFFFFu) | 0x3F800000u);
  if (f > 1.41421356f) { f = SYN_MUL(f, 0.5f); e += 1; }
  float t = SYN_DIV(SYN_ADD(f, -1.0f), SYN_ADD(f, 1.0f));
  float t2 = SYN_MUL(t, t);
  float p = 0.111111111f;
  p = SYN_ADD(SYN_MUL(p, t2), 0.142857143f);
  p = SYN_ADD(SYN_MUL(p, t2), 0.2f);
  p = SYN_ADD(SYN_MUL(p, t2), 0.333333333f);
  p = SYN_ADD(SYN_MUL(p, t2), 1.0f);
  float lnf = SYN_MUL(SYN_MUL(2.0f, t), p);
  return SYN_ADD(SYN_MUL((float)e, 0.693147181f), lnf);
}

/* 2^y for 0 <= y < 8: 2^floor(y) * exp(frac * ln2), Taylor to degree 9. */
SYN_HD float syn_exp2(float y) {
  int i = (int)y;
  float f = SYN_MUL(SYN_ADD(y, -(float)i), 0.693147181f);
  float term = 1.0f, sum = 1.0f;
  for (int k = 1; k <= 9; ++k) {
    term = SYN_DIV(SYN_MUL(term, f), (float)k);
    sum = SYN_ADD(sum, term);
  }
  return SYN_MUL(sum, SYN_U2F((uint32_t)(127 + i) << 23));
}

/* Signed 23-bit grid value in (-1, 1), exact in binary32. */
SYN_HD float syn_sym23(uint32_t n23) {
  int32_t v = (int32_t)(2u * n23 + 1u) - (int32_t)(1u << 23);
  return SYN_MUL((float)v, 1.1920928955078125e-07f); /* 2^-23 */
}

/* Standard normal, polar method; element `ctr` of the key's stream.  Up to 16
 * attempts; (probability 2e-11 of running out, then 0). */
SYN_HD float syn_normal(uint64_t key, uint64_t ctr) {
  for (uint32_t a = 0; a < 16; ++a) {
    uint64_t r = syn_at(key, ctr * 16ULL + a);
    float x = syn_sym23((uint32_t)(r >> 41));
    float y = syn_sym23((uint32_t)(r >> 18) & 0x7FFFFFu);
    float s = SYN_ADD(SYN_MUL(x, x), SYN_MUL(y, y));
    if (s < 1.0f && s > 0.0f) {
      float m = SYN_SQRT(SYN_DIV(SYN_MUL(-2.0f, syn_log(s)), s));
      return SYN_MUL(x, m);
    }
  }
  return 0.0f;
}

/* binary32 -> bf16 bits, round to nearest even (finite inputs). */
SYN_HD uint16_t syn_bf16_rne(float f) {
  uint32_t u = SYN_F2U(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

SYN_HD float syn_bf16_to_f32(uint16_t h) { return SYN_U2F((uint32_t)h << 16); }

/* Per-channel scale s_n of a weight matrix. */
SYN_HD float syn_channel_scale(uint64_t key, uint64_t n) {
  uint64_t r = syn_at(syn_substream(key, SYN_S_SCALE), n);
  float u = SYN_MUL((float)(uint32_t)(r >> 40), 5.9604644775390625e-08f); /* 2^-24 */
  return SYN_MUL(0.005f, syn_exp2(SYN_MUL(u, 3.32192809f)));              /* 10^u */
}

/* Thresholds on a 32-bit uniform for the injected categories. */
#define SYN_T_OUTLIER 21474836u /* 0.005 * 2^32 */
#define SYN_T_ZERO 30064771u    /* 0.007 * 2^32 */
#define SYN_T_DENORM 34359738u  /* 0.008 * 2^32 */

/* Weight element number e = n*K + k of a matrix, given its channel scale and
 * the matrix's category and Gaussian sub-stream keys.  With outliers == 0 (the
 * head recipe) the elements drawn as outliers keep their plain Gaussian value. */
SYN_HD uint16_t syn_weight_ex(uint64_t key_cat, uint64_t key_gauss, uint64_t e, float scale, int outliers) {
  uint64_t c = syn_at(key_cat, e);
  uint32_t cu = (uint32_t)c;
  uint16_t sign = (uint16_t)(((c >> 32) & 1u) << 15);
  if (cu >= SYN_T_OUTLIER && cu < SYN_T_ZERO) return sign;
  if (cu >= SYN_T_ZERO && cu < SYN_T_DENORM) {
    uint16_t m = (uint16_t)(1u + (uint32_t)(((c >> 33) * 127ULL) >> 31));
    return (uint16_t)(sign | m);
  }
  float z = syn_normal(key_gauss, e);
  uint16_t w = syn_bf16_rne(SYN_MUL(z, scale));
  if (outliers && cu < SYN_T_OUTLIER) w = syn_bf16_rne(SYN_MUL(syn_bf16_to_f32(w), 512.0f));
  return w;
}

SYN_HD uint16_t syn_weight(uint64_t key_cat, uint64_t key_gauss, uint64_t e, float scale) {
  return syn_weight_ex(key_cat, key_gauss, e, scale, 1);
}

/* Activation element: bf16(N(0,1)). */
SYN_HD uint16_t syn_activation(uint64_t key, uint64_t idx) {
  return syn_bf16_rne(syn_normal(syn_substream(key, SYN_S_GAUSS), idx));
}

/* Uniform integer in [0, n) for element idx of a stream (n < 2^32). */
SYN_HD uint32_t syn_below(uint64_t key, uint64_t idx, uint32_t n) {
  uint64_t r = syn_at(key, idx);
  return (uint32_t)(((r >> 32) * (uint64_t)n) >> 32);
}

#endif /* W12_SYNTH_H */
