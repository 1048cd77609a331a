/*
 * synth.h -- seeded, counter-based generator for the synthetic inputs of a
 * decode step (random-init BF16 weights and a random BF16 KV cache).
 *
 * This header is the one piece of code that both the CPU oracle and the GPU
 * input-fill kernel compile.  It holds no arithmetic of the decode step
 * itself: it only maps (seed, stream, index) to a BF16 bit pattern, so that
 * either side can regenerate any element of any tensor on demand.
 *
 * Definition (everything below is exact integer arithmetic plus one IEEE-754
 * binary32 multiply, so host and device produce identical bits):
 *
 *   mix(z)       = splitmix64 output function (Steele, Lea, Flood,
 *                  "Fast splittable pseudorandom number generators",
 *                  OOPSLA 2014): z ^= z>>30; z *= 0xbf58476d1ce4e5b9;
 *                  z ^= z>>27; z *= 0x94d049bb133111eb; z ^= z>>31.
 *   key(seed,s)  = mix(seed * G + mix(s + 0x632be59bd9b4e019)),
 *                  G = 0x9e3779b97f4a7c15 (the splitmix64 increment).
 *   draw(key,i)  = mix(key + (i+1)*G), i.e. the (i+1)-th splitmix64 output
 *                  of a generator whose state starts at key.
 *   ih4(r)       = sum of the four 16-bit fields of r minus 131070: an
 *                  Irwin-Hall sum of four discrete uniforms, mean 0,
 *                  standard deviation sqrt((65536^2-1)/3) = 37837.2265...
 *   value        = bf16_rne( (float)ih4(draw(key,i)) * scale ),
 *                  scale = (float)(sigma / 37837.2265...) rounded once.
 *
 * The values are bounded by +-3.46 sigma and have the first two moments of
 * N(0, sigma^2); the decode step's inputs only need "random BF16 of scale
 * sigma", not exact Gaussian tails.
 *
 * FP8 expert weights (the FP8 variant of a model): element i of an expert
 * matrix is the OCP FP8 E4M3 code (1 sign bit, 4 exponent bits biased by
 * 7, 3 mantissa bits, subnormals below 2^-6, largest finite 448) of
 *   ih4(draw(key, i)) * 3.5 * 2^-10          (exact in binary32, |.| < 448)
 * rounded to nearest, ties to even; each output row r of the matrix has
 * one binary32 scale
 *   base * (1 + k * 2^-10),  k = draw(key', r) >> 55  (0 .. 511),
 *   base = (float)(sigma / (37837.2265... * 3.5 * 2^-10)),
 * with key' the key of the scale stream, so row r's weights are
 * e4m3(code) * scale_r, of standard deviation sigma to 1.5 sigma.
 *
 * FP4 expert weights (NVFP4-style): element i is the E2M1 code (1 sign
 * bit, 2 exponent bits biased by 1, 1 mantissa bit: magnitudes 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6) of
 *   ih4(draw(key, i)) * 3 * 2^-16            (exact in binary32, |.| < 6)
 * rounded to nearest, ties to even; two elements per byte, element 2j in the
 * low nibble of byte j.  Each run of 16 elements along a row has an E4M3
 * block scale, code 0x30 | (draw(key_b, blk) >> 61) (0.5 * (1 + m/8)), and
 * each output row the row scale above with
 *   base = (float)(sigma / (37837.2265... * 3 * 2^-16 * 0.71875))
 * (0.71875 is the mean block scale): weight = e2m1 * block scale * row scale.
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define SYNTH_FN static __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GOLDEN 0x9e3779b97f4a7c15ULL
#define SYNTH_IH4_STD 37837.22651061575 /* sqrt((65536^2 - 1) / 3) */

/* Tensor kinds: the stream id of a tensor is (kind, layer, expert). */
enum {
  SYNTH_EMB = 1,   /* token embedding [V][H]                    */
  SYNTH_WQKV = 2,  /* fused q|k|v projection [(nq+2nkv)d][H]     */
  SYNTH_WO = 3,    /* output projection [H][nq d]               */
  SYNTH_WR = 4,    /* router [E][H]                             */
  SYNTH_WG = 5,    /* expert gate [I][H]                        */
  SYNTH_WU = 6,    /* expert up [I][H]                          */
  SYNTH_WD = 7,    /* expert down [H][I]                        */
  SYNTH_WLM = 8,   /* LM head [V][H]                            */
  SYNTH_KPOOL = 9, /* K pool of one layer [pages][nkv][P][d]    */
  SYNTH_VPOOL = 10, /* V pool of one layer [pages][nkv][P][d]   */
  SYNTH_SG = 11,   /* FP8 / FP4 expert gate row scales [I]      */
  SYNTH_SU = 12,   /* FP8 / FP4 expert up row scales [I]        */
  SYNTH_SD = 13,   /* FP8 / FP4 expert down row scales [H]      */
  SYNTH_BG = 14,   /* FP4 expert gate block scales [I][H/16]    */
  SYNTH_BU = 15,   /* FP4 expert up block scales [I][H/16]      */
  SYNTH_BD = 16,   /* FP4 expert down block scales [H][I/16]    */
  SYNTH_GAMMA = 17 /* RMSNorm gains [H]: layer l's input norm is stream
                      (GAMMA, l, 0), the final norm (GAMMA, n_layers, 0) */
};

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

SYNTH_FN uint64_t synth_stream(uint32_t kind, uint32_t layer, uint32_t expert) {
  return ((uint64_t)kind << 48) | ((uint64_t)(layer & 0xffffffu) << 24) | (uint64_t)(expert & 0xffffffu);
}

SYNTH_FN uint64_t synth_key(uint64_t seed, uint64_t stream) {
  return synth_mix64(seed * SYNTH_GOLDEN + synth_mix64(stream + 0x632be59bd9b4e019ULL));
}

SYNTH_FN uint64_t synth_draw(uint64_t key, uint64_t idx) {
  return synth_mix64(key + (idx + 1) * SYNTH_GOLDEN);
}

SYNTH_FN int32_t synth_ih4(uint64_t r) {
  return (int32_t)(r & 0xffffu) + (int32_t)((r >> 16) & 0xffffu) +
         (int32_t)((r >> 32) & 0xffffu) + (int32_t)((r >> 48) & 0xffffu) - 131070;
}

SYNTH_FN uint16_t synth_f32_to_bf16_rne(float f) {
  uint32_t u;
#if defined(__CUDA_ARCH__)
  u = __float_as_uint(f);
#else
  memcpy(&u, &f, sizeof u);
#endif
  /* no NaN or Inf can reach here: |f| <= 131070 * scale */
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* One element: the bf16 bit pattern of element idx of stream key. */
SYNTH_FN uint16_t synth_bf16(uint64_t key, uint64_t idx, float scale) {
  float v = (float)synth_ih4(synth_draw(key, idx)) * scale;
  return synth_f32_to_bf16_rne(v);
}

/* The one rounding of sigma into the per-tensor scale (IEEE double divide,
 * then round-to-nearest-even to binary32), identical on every host. */
SYNTH_FN float synth_scale(double sigma) { return (float)(sigma / SYNTH_IH4_STD); }

SYNTH_FN float synth_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
#if defined(__CUDA_ARCH__)
  f = __uint_as_float(u);
#else
  memcpy(&f, &u, sizeof f);
#endif
  return f;
}

/* ---- RMSNorm gains ---- */

/* Gain idx of stream key: the binary32 with exponent 2^-1 or 2^0 (top bit of
 * the draw) and the draw's low 23 bits as its mantissa, so gains are spread
 * over [0.5, 2) and are built from integer bits only (no rounding). */
SYNTH_FN float synth_gain(uint64_t key, uint64_t idx) {
  const uint64_t r = synth_draw(key, idx);
  const uint32_t bits = ((126u + (uint32_t)(r >> 63)) << 23) | (uint32_t)(r & 0x7fffffu);
  float f;
#if defined(__CUDA_ARCH__)
  f = __uint_as_float(bits);
#else
  memcpy(&f, &bits, sizeof f);
#endif
  return f;
}

/* ---- FP8 expert weights ---- */

#define SYNTH_FP8_STEP 0.00341796875f /* 3.5 * 2^-10: ih4 * step is exact, below 448 */

/* OCP E4M3 code of a finite binary32 of magnitude <= 448, round to nearest
 * even, by integer operations on the bits (no rounding mode involved). */
SYNTH_FN uint8_t synth_f32_to_e4m3_rne(float f) {
  uint32_t u;
#if defined(__CUDA_ARCH__)
  u = __float_as_uint(f);
#else
  memcpy(&u, &f, sizeof u);
#endif
  const uint32_t sign = (u >> 24) & 0x80u;
  const int32_t E = (int32_t)((u >> 23) & 0xffu);
  const uint32_t M = u & 0x7fffffu;
  if (E == 0) return (uint8_t)sign; /* zero or a binary32 subnormal: far below 2^-10 */
  const int32_t e = E - 127;
  uint32_t code;
  if (e >= -6) { /* normal: keep 3 of the 23 mantissa bits */
    uint32_t m = M >> 20, rem = M & 0xfffffu;
    int32_t ee = e;
    if (rem > 0x80000u || (rem == 0x80000u && (m & 1u))) ++m;
    if (m == 8u) {
      m = 0u;
      ++ee;
    }
    code = ((uint32_t)(ee + 7) << 3) | m;
  } else { /* subnormal: multiples of 2^-9 */
    const int32_t sh = 14 - e; /* value * 2^9 = (M | 2^23) >> sh */
    if (sh > 24) return (uint8_t)sign; /* below 2^-10 */
    const uint32_t full = M | 0x800000u;
    uint32_t m = full >> sh;
    const uint32_t rem = full & ((1u << sh) - 1u), half = 1u << (sh - 1);
    if (rem > half || (rem == half && (m & 1u))) ++m;
    code = m; /* m == 8 is the smallest normal, 0x08 */
  }
  return (uint8_t)(sign | code);
}

/* One FP8 expert weight: the E4M3 code of element idx of stream key. */
SYNTH_FN uint8_t synth_fp8(uint64_t key, uint64_t idx) {
  return synth_f32_to_e4m3_rne((float)synth_ih4(synth_draw(key, idx)) * SYNTH_FP8_STEP);
}

/* The base of the row scales (one rounding of sigma / (std * step)). */
SYNTH_FN float synth_fp8_base(double sigma) {
  return (float)(sigma / (SYNTH_IH4_STD * 0.00341796875));
}

/* The scale of output row `row` (stream key of the scale kind). */
SYNTH_FN float synth_row_scale(uint64_t key, uint64_t row, float base) {
  const uint32_t k = (uint32_t)(synth_draw(key, row) >> 55);
  return base * (1.0f + (float)k * 0.0009765625f); /* 1 + k 2^-10 is exact */
}

/* ---- FP4 expert weights ---- */

#define SYNTH_FP4_STEP 4.57763671875e-05f /* 3 * 2^-16: ih4 * step is exact, below 6 */

/* E2M1 code of a finite binary32 of magnitude <= 6, round to nearest even.
 * The midpoints between neighbouring magnitudes are exact in binary32, so
 * the comparisons decide exactly. */
SYNTH_FN uint8_t synth_f32_to_e2m1_rne(float f) {
  const float mid[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
  const uint8_t sign = f < 0.0f ? 8u : 0u;
  const float a = f < 0.0f ? -f : f;
  uint8_t code = 0;
  for (int i = 0; i < 7; ++i) {
    if (a > mid[i]) code = (uint8_t)(i + 1);
    else if (a == mid[i]) code = (uint8_t)((i & 1) ? i + 1 : i); /* the even code */
  }
  return (uint8_t)(sign | code);
}

/* Byte j of an FP4 matrix of stream key: elements 2j (low nibble), 2j+1. */
SYNTH_FN uint8_t synth_fp4_byte(uint64_t key, uint64_t j) {
  const uint8_t lo = synth_f32_to_e2m1_rne((float)synth_ih4(synth_draw(key, 2 * j)) * SYNTH_FP4_STEP);
  const uint8_t hi = synth_f32_to_e2m1_rne((float)synth_ih4(synth_draw(key, 2 * j + 1)) * SYNTH_FP4_STEP);
  return (uint8_t)(lo | (hi << 4));
}

/* The E4M3 block scale of 16-element block blk (stream key of the block kind). */
SYNTH_FN uint8_t synth_fp4_bscale(uint64_t key, uint64_t blk) {
  return (uint8_t)(0x30u | (uint32_t)(synth_draw(key, blk) >> 61));
}

/* The base of the FP4 row scales. */
SYNTH_FN float synth_fp4_base(double sigma) {
  return (float)(sigma / (SYNTH_IH4_STD * 4.57763671875e-05 * 0.71875));
}

#endif /* SYNTH_H */
