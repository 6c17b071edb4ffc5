/* Seeded synthetic-input generator: the one piece of code that both the CPU
 * oracle's inputs and the GPU path's inputs come from.
 *
 * It holds none of the MoE method's arithmetic: it only draws random numbers
 * and lays them out as bytes of the input formats (bf16, f32, fp16 fields of
 * the K-quant super-blocks).  The same inline functions are compiled for the
 * host (synth.c) and for the GPU bulk filler (synth_gpu.cu), so the two produce
 * identical bytes wherever only integer and correctly rounded IEEE operations
 * are involved (K-quant blocks, uniform draws, permutations).  Normal draws
 * go through the platform's f64 log/cos and can, in rare cases, differ in one
 * f64 ulp between host and GPU; the bf16 result then differs only when that
 * ulp straddles a bf16 rounding point.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014): the i-th output of the sequence seeded by
 * `key` is mix64(key + (i+1)*GAMMA).  A stream key is derived from
 * (seed, layer, tensor, expert) by chained mix64.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>
#ifndef __CUDACC__
#include <math.h>
#endif

#ifdef __CUDACC__
#define SYN_FN static __host__ __device__ __forceinline__
#else
#define SYN_FN static inline
#endif

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL

/* tensor ids of the stream keys */
enum {
  SYN_T_X = 1,        /* activation rows x, bf16 [m, dim] */
  SYN_T_ROUTER = 2,   /* router weight, bf16 [n_routed, dim] */
  SYN_T_BIAS = 3,     /* router selection bias, f32 [n_routed] */
  SYN_T_W1 = 4,       /* routed gate projection, Q2_K [inter rows][dim/256] */
  SYN_T_W3 = 5,       /* routed up projection, Q2_K */
  SYN_T_W2 = 6,       /* routed down projection, Q3_K [dim rows][inter/256] */
  SYN_T_SH1 = 7,      /* shared expert gate, bf16 [inter, dim] or Q2_K */
  SYN_T_SH3 = 8,      /* shared expert up */
  SYN_T_SH2 = 9,      /* shared expert down, bf16 [dim, inter] or Q3_K */
  SYN_T_OUTLIER = 10, /* permutation choosing the scaled activation rows */
  SYN_T_HOT = 11      /* permutation choosing the hot experts */
};

SYN_FN uint64_t syn_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SYN_FN uint64_t syn_key(uint64_t seed, uint32_t layer, uint32_t tensor, uint32_t expert) {
  uint64_t k = syn_mix64(seed + SYN_GAMMA);
  k = syn_mix64(k ^ ((uint64_t)layer * 0xD1B54A32D192ED03ULL + 1ULL));
  k = syn_mix64(k ^ (((uint64_t)tensor << 32) | (uint64_t)expert));
  return k;
}

SYN_FN uint64_t syn_draw(uint64_t key, uint64_t i) { return syn_mix64(key + (i + 1ULL) * SYN_GAMMA); }

/* exact: a 53-bit integer times a power of two */
SYN_FN double syn_unit(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }

/* lo + (hi - lo) * u with each operation rounded separately (no fused
 * multiply-add on either side) */
SYN_FN double syn_affine(double lo, double hi, double u) {
#ifdef __CUDA_ARCH__
  return __dadd_rn(lo, __dmul_rn(__dadd_rn(hi, -lo), u));
#else
  volatile double span = hi - lo;
  volatile double prod = span * u;
  return lo + prod;
#endif
}

/* f64 -> IEEE binary16, round to nearest even, subnormals and overflow
 * handled.  Integer-only so host and GPU agree bit for bit. */
SYN_FN uint16_t syn_f64_to_f16(double v) {
  union { double d; uint64_t u; } c;
  c.d = v;
  uint64_t b = c.u;
  uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
  int e = (int)((b >> 52) & 0x7FF);
  uint64_t man = b & 0xFFFFFFFFFFFFFULL;
  if (e == 0x7FF) return (uint16_t)(sign | 0x7C00u | (man ? 0x200u : 0u));
  if (e == 0 && man == 0) return sign;
  int ue = e - 1023;                       /* unbiased exponent */
  uint64_t sig = man | (1ULL << 52);       /* 53-bit significand (normals) */
  if (e == 0) return sign;                 /* f64 subnormals underflow to zero */
  int shift;                               /* bits dropped from sig */
  uint16_t hexp;
  if (ue > 15) return (uint16_t)(sign | 0x7C00u);
  if (ue >= -14) { shift = 42; hexp = (uint16_t)(ue + 15); }
  else { shift = 42 + (-14 - ue); hexp = 0; if (shift > 63) return sign; }
  uint64_t kept = sig >> shift;
  uint64_t rem = sig & ((1ULL << shift) - 1ULL);
  uint64_t half = 1ULL << (shift - 1);
  if (rem > half || (rem == half && (kept & 1ULL))) kept += 1ULL;
  uint32_t out;
  if (hexp == 0) {
    out = (uint32_t)kept;                  /* may carry into the smallest normal */
  } else {
    /* kept includes the implicit bit at position 10 */
    out = ((uint32_t)hexp << 10) + (uint32_t)(kept - (1ULL << 10));
  }
  if (out >= 0x7C00u) out = 0x7C00u;
  return (uint16_t)(sign | out);
}

/* f64 -> f32 (C conversion, round to nearest) -> bf16 round to nearest even */
SYN_FN uint16_t syn_f64_to_bf16(double v) {
  union { float f; uint32_t u; } c;
  c.f = (float)v;
  uint32_t b = c.u;
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x7FFFFFu)) return (uint16_t)((b >> 16) | 0x40u);
  uint32_t lsb = (b >> 16) & 1u;
  return (uint16_t)((b + 0x7FFFu + lsb) >> 16);
}

/* One standard normal value from draws 2i and 2i+1 (Box-Muller, cosine branch). */
SYN_FN double syn_normal(uint64_t key, uint64_t i) {
  double u1 = ((double)(syn_draw(key, 2 * i) >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
  double u2 = syn_unit(syn_draw(key, 2 * i + 1));                     /* [0, 1) */
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

/* Byte k of a K-quant block filled from draws: block i takes draws
 * 16*i + (k / 8), byte k % 8 of the little-endian word. */
SYN_FN uint8_t syn_block_byte(uint64_t key, uint64_t block, int k) {
  uint64_t r = syn_draw(key, block * 16ULL + (uint64_t)(k >> 3));
  return (uint8_t)(r >> (8 * (k & 7)));
}

/* Q2_K super-block of 256 weights, 84 bytes: scales[16] qs[64] d dmin.
 * All scale/min nibbles and 2-bit quants uniform; d, dmin ~ U(dlo, dhi) as
 * fp16 (draws 10 and 11 of the block). */
SYN_FN void syn_q2k_block(uint8_t* dst, uint64_t key, uint64_t block, double dlo, double dhi) {
  for (int k = 0; k < 80; ++k) dst[k] = syn_block_byte(key, block, k);
  uint16_t d = syn_f64_to_f16(syn_affine(dlo, dhi, syn_unit(syn_draw(key, block * 16ULL + 10ULL))));
  uint16_t dm = syn_f64_to_f16(syn_affine(dlo, dhi, syn_unit(syn_draw(key, block * 16ULL + 11ULL))));
  dst[80] = (uint8_t)(d & 0xFF); dst[81] = (uint8_t)(d >> 8);
  dst[82] = (uint8_t)(dm & 0xFF); dst[83] = (uint8_t)(dm >> 8);
}

/* Q3_K super-block, 110 bytes: hmask[32] qs[64] scales[12] d.  Every bit of
 * the first 108 bytes uniform (so the 16 six-bit scale codes are uniform on
 * 0..63); d ~ U(dlo, dhi) as fp16 (draw 14 of the block). */
SYN_FN void syn_q3k_block(uint8_t* dst, uint64_t key, uint64_t block, double dlo, double dhi) {
  for (int k = 0; k < 108; ++k) dst[k] = syn_block_byte(key, block, k);
  uint16_t d = syn_f64_to_f16(syn_affine(dlo, dhi, syn_unit(syn_draw(key, block * 16ULL + 14ULL))));
  dst[108] = (uint8_t)(d & 0xFF); dst[109] = (uint8_t)(d >> 8);
}

#endif
