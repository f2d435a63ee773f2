/*
 * uq_oracle.c -- plain, slow CPU oracle for the UltraQuant 4-bit KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this code:
 * only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * leg use it.  It shares no code, header, table or constant generator with the
 * CUDA library; each step is written out from the pages' description.
 *
 * Sources (cited by page title and section):
 *   [UQ-review]     "UltraQuant: 4-bit KV Caching for Context-Heavy Agents",
 *                   review at manon006.tistory.com/395, sections 3.1-3.3, 4.2.
 *   [UQ-residency]  "kv-cache-4bit-serving-residency-collapse",
 *                   pheeree.github.io 2026-09-01, body and footnotes 2, 13.
 *   [TQ-guide]      "TurboQuant 완전 정리", juhoplayground.github.io,
 *                   sections on random rotation (RHT) and inner-product
 *                   preservation by orthogonality.
 *
 * Readings taken where the pages are silent (each is listed in the design doc):
 *   R1  rotation = fp32 Sylvester FWHT, stages h = 1,2,4,...,d/2 in that order,
 *       of s (.) x, then times fl32(1/sqrt(d)); s from splitmix64(seed).
 *   R2  scale exponent E = integer nearest to log2(fl32(0.156f * m)).
 *   R3  E2M1 round-to-nearest, ties to even code, saturating at 6; sign = IEEE
 *       sign bit of the rotated value; byte j = code(2j) | code(2j+1) << 4.
 *   R4  query: R1 rotation, then E4M3 RNE satfinite, no per-token scale.
 *   R5  attention on the dequantised values in fp64; output inverse-rotated.
 *   NaN/Inf group -> scale byte 0xFF and zero code bytes.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * -ffp-contract=off matters: the fp32 rotation must not be fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Sign diagonal of the randomised Hadamard transform.                        */
/* [TQ-guide] "RHT = random sign diagonal x Hadamard".  The random signs come */
/* from splitmix64 (Steele, Lea, Flood 2014): output i of the stream seeded    */
/* with `seed` is mix(seed + (i+1) * golden_gamma).                            */
/* ------------------------------------------------------------------------- */
uint64_t uqo_splitmix64(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1u) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* s_i = +1 when bit 63 of output i is 0, else -1. */
void uqo_signs(uint64_t seed, int d, int8_t* s) {
  for (int i = 0; i < d; ++i) s[i] = (uqo_splitmix64(seed, (uint64_t)i) >> 63) ? -1 : 1;
}

/* fl32(1/sqrt(d)), the normalisation of the orthonormal Hadamard transform. */
float uqo_inv_sqrt_d(int d) { return (float)(1.0 / sqrt((double)d)); }

/* ------------------------------------------------------------------------- */
/* R1: forward rotation y = fl32( FWHT_fp32(s .* x) * fl32(1/sqrt d) ).        */
/* [UQ-review] 3.1: keys pass through a Walsh-Hadamard rotation before the     */
/* 32-channel grouping.  The butterfly is the plain Sylvester-order transform. */
/* ------------------------------------------------------------------------- */
void uqo_rotate_fp32(const float* x, int d, const int8_t* s, float* y) {
  float u[1024];
  for (int i = 0; i < d; ++i) u[i] = (s[i] < 0) ? -x[i] : x[i];
  for (int h = 1; h < d; h <<= 1) {
    for (int i = 0; i < d; ++i) {
      if (i & h) continue;
      float a = u[i], b = u[i + h];
      u[i] = a + b;
      u[i + h] = a - b;
    }
  }
  float c = uqo_inv_sqrt_d(d);
  for (int i = 0; i < d; ++i) y[i] = u[i] * c;
}

/* Inverse rotation in fp64: out = s .* (H o) / sqrt(d).  R is orthogonal, so  */
/* its inverse is its transpose ([TQ-guide], inner-product preservation).      */
void uqo_inverse_rotate_f64(const double* o, int d, const int8_t* s, double* out) {
  double u[1024];
  for (int i = 0; i < d; ++i) u[i] = o[i];
  for (int h = 1; h < d; h <<= 1)
    for (int i = 0; i < d; ++i) {
      if (i & h) continue;
      double a = u[i], b = u[i + h];
      u[i] = a + b;
      u[i + h] = a - b;
    }
  double c = 1.0 / sqrt((double)d);
  for (int i = 0; i < d; ++i) out[i] = (double)s[i] * u[i] * c;
}

/* Inverse rotation in fp32, the form the decode's output stage takes:       */
/* out = s .* fl32(FWHT_fp32(o) * fl32(1/sqrt d)), the same ascending-stride  */
/* butterfly as the forward rotation (H is symmetric, so H^T o = H o), each    */
/* output fl32(a+b) / fl32(a-b); the signs last (exact).                       */
void uqo_inverse_rotate_fp32(const float* o, int d, const int8_t* s, float* out) {
  float u[1024];
  for (int i = 0; i < d; ++i) u[i] = o[i];
  for (int h = 1; h < d; h <<= 1) {
    for (int i = 0; i < d; ++i) {
      if (i & h) continue;
      float a = u[i], b = u[i + h];
      u[i] = a + b;
      u[i + h] = a - b;
    }
  }
  float c = uqo_inv_sqrt_d(d);
  for (int i = 0; i < d; ++i) {
    float y = u[i] * c;
    out[i] = (s[i] < 0) ? -y : y;
  }
}

/* ------------------------------------------------------------------------- */
/* R2: UE8M0 scale byte of one 32-channel group.                               */
/* [UQ-review] 3.1/3.3: group absmax m, times the global constant c = 0.156,   */
/* rounded to a power of two; [UQ-review] 3.2: byte = E + 127.                 */
/* mode selects the power-of-two rounding (0 = nearest in log2, the reading    */
/* used by the product; 1 = nearest in linear distance, ties up; 2 = floor;    */
/* 3 = ceil) so that the c sweep can compare them.                             */
/* ------------------------------------------------------------------------- */
int uqo_pow2_exponent(double t, int mode) {
  /* t > 0 and finite.  frexp: t = f * 2^e with f in [0.5, 1), so          */
  /* 2^(e-1) <= t < 2^e.                                                      */
  int e;
  double f = frexp(t, &e);
  int lo = e - 1;                         /* floor(log2 t) */
  int exact = (f == 0.5);
  switch (mode) {
    case 0: /* nearest in log2: round up iff t >= 2^lo * sqrt(2), tested  */
            /* exactly as t^2 >= 2^(2 lo + 1) (t is fp32, t^2 exact in f64) */
      return (t * t >= ldexp(1.0, 2 * lo + 1)) ? lo + 1 : lo;
    case 1: /* nearest in linear distance, ties to the larger power */
      return (t - ldexp(1.0, lo) >= ldexp(1.0, lo + 1) - t) ? lo + 1 : lo;
    case 2: return lo;
    default: return exact ? lo : lo + 1;
  }
}

int uqo_scale_byte(float m, float c, int mode) {
  if (isnan(m) || isinf(m)) return 0xFF;
  float t = c * m; /* fl32(c * m) */
  if (t == 0.0f) return 0;
  int E = uqo_pow2_exponent((double)t, mode);
  int byte = E + 127;
  if (byte < 0) byte = 0;
  if (byte > 254) byte = 254;
  return byte;
}

/* ------------------------------------------------------------------------- */
/* R3: E2M1 code of an exact value r = y * 2^-E.                               */
/* Grid {0, .5, 1, 1.5, 2, 3, 4, 6}; round to nearest, ties to the even code,  */
/* saturating above 6.  Magnitude codes 0..7 are the grid in order; bit 3 is   */
/* the sign.  The thresholds are the midpoints of the grid; at a midpoint the  */
/* code whose mantissa bit is 0 wins (0, 1.0, 1.0, 2, 2, 4, 4 for the seven    */
/* midpoints .25 .75 1.25 1.75 2.5 3.5 5).                                     */
/* ------------------------------------------------------------------------- */
int uqo_e2m1_code(double r) {
  int sign = signbit(r) ? 8 : 0;
  double a = fabs(r);
  int mag;
  if (a <= 0.25) mag = 0;
  else if (a < 0.75) mag = 1;
  else if (a <= 1.25) mag = 2;
  else if (a < 1.75) mag = 3;
  else if (a <= 2.5) mag = 4;
  else if (a < 3.5) mag = 5;
  else if (a <= 5.0) mag = 6;
  else mag = 7;
  return sign | mag;
}

double uqo_e2m1_value(int code) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = mag[code & 7];
  return (code & 8) ? -v : v;
}

/* value = code * 2^(byte-127) ([UQ-review] 3.2; [UQ-residency] body).  The  */
/* byte 0xFF marks a non-finite group and decodes to NaN.                     */
double uqo_fp4_value(int code, int byte) {
  if (byte == 0xFF) return NAN;
  return ldexp(uqo_e2m1_value(code), byte - 127);
}

/* Quantise n_vec rotated vectors of length d (multiple of 32).              */
/* codes: n_vec * d/2 bytes, scales: n_vec * d/32 bytes.                     */
void uqo_quantize_rotated(const float* y, int64_t n_vec, int d, float c, int mode,
                          uint8_t* codes, uint8_t* scales) {
  for (int64_t v = 0; v < n_vec; ++v) {
    const float* yv = y + v * d;
    for (int g = 0; g < d / 32; ++g) {
      const float* yg = yv + 32 * g;
      float m = 0.0f;
      int nonfinite = 0;
      for (int i = 0; i < 32; ++i) {
        if (isnan(yg[i]) || isinf(yg[i])) nonfinite = 1;
        else if (fabsf(yg[i]) > m) m = fabsf(yg[i]);
      }
      int byte = nonfinite ? 0xFF : uqo_scale_byte(m, c, mode);
      scales[v * (d / 32) + g] = (uint8_t)byte;
      for (int i = 0; i < 32; i += 2) {
        int c0 = 0, c1 = 0;
        if (byte != 0xFF) {
          int E = byte - 127;
          c0 = uqo_e2m1_code(ldexp((double)yg[i], -E));
          c1 = uqo_e2m1_code(ldexp((double)yg[i + 1], -E));
        }
        codes[v * (d / 2) + (32 * g + i) / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
}

/* The constant c = 0.156 of [UQ-review] 3.3 / [UQ-residency] footnote 13. */
float uqo_c_constant(void) { return 0.156f; }

/* ------------------------------------------------------------------------- */
/* bf16 helpers (the input tensors of the path are bf16 or fp32).             */
/* ------------------------------------------------------------------------- */
static float bf16_to_f32(uint16_t h) {
  uint32_t b = (uint32_t)h << 16;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

/* Round fp32 to bf16, nearest-even (NaN kept quiet). */
uint16_t uqo_f32_to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((b >> 16) | 0x40);
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}

static void load_row(const void* src, int in_fp32, int64_t row, int d, float* out) {
  if (in_fp32) {
    memcpy(out, (const float*)src + row * d, sizeof(float) * (size_t)d);
  } else {
    const uint16_t* s = (const uint16_t*)src + row * d;
    for (int i = 0; i < d; ++i) out[i] = bf16_to_f32(s[i]);
  }
}

/* Rotate + quantise n vectors (bf16 or fp32 rows). */
/* With a constant c of one's own in R2 (the pages keep one global c and name  */
/* per-layer constants as an open option, [UQ-review] 7.3; the c sweep of     */
/* [UQ-residency] is the objective that picks one).                            */
void uqo_quantize_vectors_c(const void* x, int in_fp32, int64_t n, int d, uint64_t seed, float c,
                            uint8_t* codes, uint8_t* scales) {
  int8_t s[1024];
  float xr[1024], y[1024];
  uqo_signs(seed, d, s);
  for (int64_t v = 0; v < n; ++v) {
    load_row(x, in_fp32, v, d, xr);
    uqo_rotate_fp32(xr, d, s, y);
    uqo_quantize_rotated(y, 1, d, c, 0, codes + v * (d / 2), scales + v * (d / 32));
  }
}

void uqo_quantize_vectors(const void* x, int in_fp32, int64_t n, int d, uint64_t seed,
                          uint8_t* codes, uint8_t* scales) {
  uqo_quantize_vectors_c(x, in_fp32, n, d, seed, uqo_c_constant(), codes, scales);
}

/* ------------------------------------------------------------------------- */
/* Cache byte order of a K row.  A quantised row is a sequence of d/2 code    */
/* bytes, 16 per 32-channel group (natural order above).  In the cache, the   */
/* K row's bytes are interleaved by 4-byte words across the groups: word w    */
/* (bytes 4w..4w+3) of group g is stored at word position (d/32)*w + g, so   */
/* each aligned run of d/8 bytes holds one word of every group.  V rows are   */
/* stored in natural order.  (A layout choice of this library, made so that   */
/* the decode reads the per-group operands with one aligned load; the pages   */
/* state that the cache layout is matched to how the kernel consumes scales,  */
/* [UQ-review] 4.2.)                                                          */
/* ------------------------------------------------------------------------- */
int uqo_kbyte_pos(int j, int d) {
  int g = j / 16, b = j % 16, w = b / 4, k = b % 4;
  return ((d / 32) * w + g) * 4 + k;
}

/* ------------------------------------------------------------------------- */
/* R4: FP8 E4M3 (OCP "FN": bias 7, no inf, max 448, 0x7F NaN).                 */
/* [UQ-review] 3.2: the query is rotated into the key basis, then rounded to   */
/* FP8 E4M3.  Round to nearest by search over the 127 finite non-negative      */
/* values, ties to the code with an even mantissa, saturating at 448.          */
/* ------------------------------------------------------------------------- */
double uqo_e4m3_value(int byte) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

int uqo_e4m3_code(float x) {
  if (isnan(x)) return 0x7F;
  int sign = signbit(x) ? 0x80 : 0;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  int best = 0;
  double bestd = INFINITY;
  for (int code = 0; code <= 0x7E; ++code) {
    double dist = fabs(uqo_e4m3_value(code) - a);
    if (dist < bestd || (dist == bestd && (code & 1) == 0)) {
      best = code;
      bestd = dist;
    }
  }
  return sign | best;
}

/* Rotated, E4M3-rounded query q~ of one head (R4).  q: bf16 row. */
void uqo_query_fp8(const uint16_t* q, int d, uint64_t seed, uint8_t* out) {
  int8_t s[1024];
  float xr[1024], y[1024];
  uqo_signs(seed, d, s);
  for (int i = 0; i < d; ++i) xr[i] = bf16_to_f32(q[i]);
  uqo_rotate_fp32(xr, d, s, y);
  for (int i = 0; i < d; ++i) out[i] = (uint8_t)uqo_e4m3_code(y[i]);
}

/* ------------------------------------------------------------------------- */
/* Paged cache addressing (vLLM convention): slot = page * ps + offset;        */
/* arrays are [num_pages][Hkv][ps][row_bytes].                                 */
/* ------------------------------------------------------------------------- */
static int64_t cache_row(int64_t slot, int h, int Hkv, int ps) {
  int64_t page = slot / ps, off = slot % ps;
  return (page * Hkv + h) * ps + off;
}

/* Quantize-append of T tokens of K and V ([T][Hkv][d], bf16 or fp32) into an */
/* FP4 cache; slots < 0 are skipped.                                          */
void uqo_append_fp4_c(const void* k, const void* v, int in_fp32, int64_t T, const int64_t* slots,
                      int Hkv, int ps, int d, uint64_t seed, float c, uint8_t* kc, uint8_t* ks,
                      uint8_t* vc, uint8_t* vs) {
  size_t esz = in_fp32 ? 4 : 2;
  for (int64_t t = 0; t < T; ++t) {
    if (slots[t] < 0) continue;
    for (int h = 0; h < Hkv; ++h) {
      int64_t src = t * Hkv + h, dst = cache_row(slots[t], h, Hkv, ps);
      const char* kr = (const char*)k + (size_t)src * d * esz;
      const char* vr = (const char*)v + (size_t)src * d * esz;
      uint8_t kn[512];
      uqo_quantize_vectors_c(kr, in_fp32, 1, d, seed, c, kn, ks + dst * (d / 32));
      for (int j = 0; j < d / 2; ++j) kc[dst * (d / 2) + uqo_kbyte_pos(j, d)] = kn[j];
      uqo_quantize_vectors_c(vr, in_fp32, 1, d, seed, c, vc + dst * (d / 2), vs + dst * (d / 32));
    }
  }
}

void uqo_append_fp4(const void* k, const void* v, int in_fp32, int64_t T, const int64_t* slots,
                    int Hkv, int ps, int d, uint64_t seed, uint8_t* kc, uint8_t* ks,
                    uint8_t* vc, uint8_t* vs) {
  uqo_append_fp4_c(k, v, in_fp32, T, slots, Hkv, ps, d, seed, uqo_c_constant(), kc, ks, vc, vs);
}

/* FP8 anchor append: e4m3_RNE_sat(x / scale), unrotated. */
void uqo_append_fp8(const void* k, const void* v, int in_fp32, int64_t T, const int64_t* slots,
                    int Hkv, int ps, int d, float k_scale, float v_scale, uint8_t* k8,
                    uint8_t* v8) {
  float xr[1024];
  for (int64_t t = 0; t < T; ++t) {
    if (slots[t] < 0) continue;
    for (int h = 0; h < Hkv; ++h) {
      int64_t src = t * Hkv + h, dst = cache_row(slots[t], h, Hkv, ps);
      load_row(k, in_fp32, src, d, xr);
      for (int i = 0; i < d; ++i) k8[dst * d + i] = (uint8_t)uqo_e4m3_code(xr[i] / k_scale);
      load_row(v, in_fp32, src, d, xr);
      for (int i = 0; i < d; ++i) v8[dst * d + i] = (uint8_t)uqo_e4m3_code(xr[i] / v_scale);
    }
  }
}

/* BF16 anchor append: bf16 inputs stored as they are, fp32 inputs rounded. */
void uqo_append_bf16(const void* k, const void* v, int in_fp32, int64_t T, const int64_t* slots,
                     int Hkv, int ps, int d, uint16_t* kb, uint16_t* vb) {
  float xr[1024];
  for (int64_t t = 0; t < T; ++t) {
    if (slots[t] < 0) continue;
    for (int h = 0; h < Hkv; ++h) {
      int64_t src = t * Hkv + h, dst = cache_row(slots[t], h, Hkv, ps);
      load_row(k, in_fp32, src, d, xr);
      for (int i = 0; i < d; ++i) kb[dst * d + i] = uqo_f32_to_bf16(xr[i]);
      load_row(v, in_fp32, src, d, xr);
      for (int i = 0; i < d; ++i) vb[dst * d + i] = uqo_f32_to_bf16(xr[i]);
    }
  }
}

/* ------------------------------------------------------------------------- */
/* TQ4: the TurboQuant Q_mse codebook variant ([TQ-guide] "Lloyd-Max 스칼라    */
/* 양자화 (Q_mse)" and "직교성을 이용한 내적 보존").  A row is rotated with R1, */
/* its L2 norm n is stored, and every coordinate of the unit vector y / n is   */
/* replaced by the index of its nearest Lloyd-Max centroid.  The codebook      */
/* (computed from the pdf in oracle/tq.py) comes in as the fp64 centroids      */
/* c_8 < ... < c_15 of the non-negative half (the negative half mirrors).      */
/* Readings:                                                       */
/*   T3  n = sqrt(sum y_i^2) in fp64, stored as fl32(n); u_i = y_i / n in fp64; */
/*       a non-finite n stores NaN and zero codes; n = 0 stores 0 and zero     */
/*       codes (every code decodes to 0 there).                                */
/*   T4  code of u: sign-magnitude nibble, bit 3 set for u < 0, bits 0..2 the  */
/*       rank of the centroid nearest to |u| (ties to the lower rank).         */
/*   T5  q~ = f16(R1 q), round to nearest even.                                */
/* ------------------------------------------------------------------------- */
double uqo_f16_round(float x) {
  if (isnan(x)) return NAN;
  double a = fabs((double)x), r;
  if (a >= 65520.0) {
    r = INFINITY;  /* at and above the midpoint 65504 + 16 ties go to 2^16 */
  } else if (a < ldexp(1.0, -14)) {
    r = nearbyint(a * ldexp(1.0, 24)) * ldexp(1.0, -24);  /* subnormal quantum 2^-24 */
  } else {
    int e;
    frexp(a, &e);                       /* a in [2^(e-1), 2^e) */
    double quantum = ldexp(1.0, e - 11); /* 10 fraction bits */
    r = nearbyint(a / quantum) * quantum;
  }
  return signbit(x) ? -r : r;
}

/* The Euclidean norm of the rotated row, in fp64 (T3). */
double uqo_tq_norm(const float* y, int d) {
  double s = 0.0;
  for (int i = 0; i < d; ++i) s += (double)y[i] * (double)y[i];
  return sqrt(s);
}

/* T4: nearest centroid of u among +-cpos[0..7]. */
int uqo_tq_code(double u, const double* cpos) {
  double a = fabs(u);
  int best = 0;
  for (int k = 1; k < 8; ++k)
    if (fabs(a - cpos[k]) < fabs(a - cpos[best])) best = k;
  return (u < 0.0 ? 8 : 0) | best;
}

double uqo_tq_value(int code, const double* mags) {
  double v = mags[code & 7];
  return (code & 8) ? -v : v;
}

/* Rotate + quantise one row (fp32 values): d/2 code bytes in natural order   */
/* (byte j = code(2j) | code(2j+1) << 4) and the fp32 norm.                    */
void uqo_tq_quantize_row(const float* xr, int d, const int8_t* s, const double* cpos,
                         uint8_t* codes, float* norm) {
  float y[1024];
  uqo_rotate_fp32(xr, d, s, y);
  double n = uqo_tq_norm(y, d);
  if (!isfinite(n) || n == 0.0) {
    memset(codes, 0, (size_t)d / 2);
    *norm = isfinite(n) ? 0.0f : NAN;
    return;
  }
  for (int j = 0; j < d / 2; ++j)
    codes[j] = (uint8_t)(uqo_tq_code((double)y[2 * j] / n, cpos) |
                         (uqo_tq_code((double)y[2 * j + 1] / n, cpos) << 4));
  *norm = (float)n;
}

void uqo_append_tq4(const void* k, const void* v, int in_fp32, int64_t T, const int64_t* slots,
                    int Hkv, int ps, int d, uint64_t seed, const double* cpos, uint8_t* kc,
                    float* kn, uint8_t* vc, float* vn) {
  int8_t s[1024];
  float xr[1024];
  uint8_t row[512];
  uqo_signs(seed, d, s);
  for (int64_t t = 0; t < T; ++t) {
    if (slots[t] < 0) continue;
    for (int h = 0; h < Hkv; ++h) {
      int64_t src = t * Hkv + h, dst = cache_row(slots[t], h, Hkv, ps);
      load_row(k, in_fp32, src, d, xr);
      uqo_tq_quantize_row(xr, d, s, cpos, row, kn + dst);
      for (int j = 0; j < d / 2; ++j) kc[dst * (d / 2) + uqo_kbyte_pos(j, d)] = row[j];
      load_row(v, in_fp32, src, d, xr);
      uqo_tq_quantize_row(xr, d, s, cpos, vc + dst * (d / 2), vn + dst);
    }
  }
}

/* T5: rotated query rounded to f16, as fp64 values. */
void uqo_query_f16(const uint16_t* q, int d, uint64_t seed, double* out) {
  int8_t s[1024];
  float xr[1024], y[1024];
  uqo_signs(seed, d, s);
  for (int i = 0; i < d; ++i) xr[i] = bf16_to_f32(q[i]);
  uqo_rotate_fp32(xr, d, s, y);
  for (int i = 0; i < d; ++i) out[i] = uqo_f16_round(y[i]);
}

/* ------------------------------------------------------------------------- */
/* R5: decode attention in fp64 on the dequantised cache.                      */
/* One query token per sequence; q head h reads kv head h / (Hq/Hkv).          */
/* Logical token j of sequence b lives in page block_table[b][j/ps], slot      */
/* offset j % ps.  logits = sm_scale * <q, k>, softmax with max subtraction,   */
/* o = sum p v.  For the FP4 cache q is the rotated E4M3 query q~ and the      */
/* output is rotated back ([UQ-review] 3.2).  kind: 0 = FP4, 1 = FP8, 2 = BF16,*/
/* 3 = TQ4 (q~ = f16(R1 q), values = codebook value x stored norm, rotated). */
/* ------------------------------------------------------------------------- */
static double kv_value(int kind, int is_k, const uint8_t* codes, const uint8_t* scales, int64_t row,
                       int d, int i, float tensor_scale, const double* tq_mags) {
  if (kind == 0 || kind == 3) {
    int pos = is_k ? uqo_kbyte_pos(i / 2, d) : i / 2;
    int byte = codes[row * (d / 2) + pos];
    int code = (i & 1) ? (byte >> 4) : (byte & 15);
    if (kind == 3) return uqo_tq_value(code, tq_mags) * (double)((const float*)scales)[row];
    return uqo_fp4_value(code, scales[row * (d / 32) + i / 32]);
  }
  if (kind == 1) return uqo_e4m3_value(codes[row * d + i]) * (double)tensor_scale;
  const uint16_t* b = (const uint16_t*)codes;
  return (double)bf16_to_f32(b[row * d + i]);
}

void uqo_decode_ex(int kind, const uint16_t* q, int B, int Hq, int Hkv, int d, int ps,
                   const uint8_t* kc, const uint8_t* ks, const uint8_t* vc, const uint8_t* vs,
                   float k_scale, float v_scale, const int32_t* block_table, int max_pages,
                   const int32_t* seq_lens, double sm_scale, uint64_t seed, const double* tq_mags,
                   double* out) {
  int G = Hq / Hkv;
  if (sm_scale <= 0.0) sm_scale = 1.0 / sqrt((double)d);
  int8_t s[1024];
  uqo_signs(seed, d, s);
  double qd[1024], o[1024];
  for (int b = 0; b < B; ++b) {
    int L = seq_lens[b];
    for (int kvh = 0; kvh < Hkv; ++kvh) {
      if (L <= 0) {
        for (int h = kvh * G; h < (kvh + 1) * G; ++h)
          for (int i = 0; i < d; ++i) out[((int64_t)b * Hq + h) * d + i] = 0.0;
        continue;
      }
      /* dequantised keys and values of this (sequence, kv head), logical order */
      double* K = (double*)malloc(sizeof(double) * (size_t)L * d);
      double* V = (double*)malloc(sizeof(double) * (size_t)L * d);
      double* logit = (double*)malloc(sizeof(double) * (size_t)L);
      for (int j = 0; j < L; ++j) {
        int64_t page = block_table[(int64_t)b * max_pages + j / ps];
        int64_t row = (page * Hkv + kvh) * ps + j % ps;
        for (int i = 0; i < d; ++i) {
          K[(int64_t)j * d + i] = kv_value(kind, 1, kc, ks, row, d, i, k_scale, tq_mags);
          V[(int64_t)j * d + i] = kv_value(kind, 0, vc, vs, row, d, i, v_scale, tq_mags);
        }
      }
      for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
        double* ob = out + ((int64_t)b * Hq + h) * d;
        const uint16_t* qrow = q + ((int64_t)b * Hq + h) * d;
        if (kind == 0) {
          uint8_t q8[1024];
          uqo_query_fp8(qrow, d, seed, q8);
          for (int i = 0; i < d; ++i) qd[i] = uqo_e4m3_value(q8[i]);
        } else if (kind == 3) {
          uqo_query_f16(qrow, d, seed, qd);
        } else {
          for (int i = 0; i < d; ++i) qd[i] = (double)bf16_to_f32(qrow[i]);
        }
        double mx = -INFINITY;
        for (int j = 0; j < L; ++j) {
          double acc = 0.0;
          for (int i = 0; i < d; ++i) acc += qd[i] * K[(int64_t)j * d + i];
          logit[j] = sm_scale * acc;
          if (logit[j] > mx) mx = logit[j]; /* a NaN logit reaches the output via exp */
        }
        double lsum = 0.0;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        for (int j = 0; j < L; ++j) {
          double p = exp(logit[j] - mx);
          lsum += p;
          for (int i = 0; i < d; ++i) o[i] += p * V[(int64_t)j * d + i];
        }
        for (int i = 0; i < d; ++i) o[i] /= lsum;
        if (kind == 0 || kind == 3) uqo_inverse_rotate_f64(o, d, s, ob);
        else memcpy(ob, o, sizeof(double) * (size_t)d);
      }
      free(K);
      free(V);
      free(logit);
    }
  }
}

void uqo_decode(int kind, const uint16_t* q, int B, int Hq, int Hkv, int d, int ps,
                const uint8_t* kc, const uint8_t* ks, const uint8_t* vc, const uint8_t* vs,
                float k_scale, float v_scale, const int32_t* block_table, int max_pages,
                const int32_t* seq_lens, double sm_scale, uint64_t seed, double* out) {
  uqo_decode_ex(kind, q, B, Hq, Hkv, d, ps, kc, ks, vc, vs, k_scale, v_scale, block_table, max_pages,
                seq_lens, sm_scale, seed, NULL, out);
}

/* ------------------------------------------------------------------------- */
/* Array forms used by the tests.                                             */
/* ------------------------------------------------------------------------- */
void uqo_e2m1_codes(const double* r, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)uqo_e2m1_code(r[i]);
}

/* Enumerations for the exhaustive tests: element i is the fp32 value whose   */
/* bit pattern is first + i (the caller keeps first + n - 1 <= 0xFFFFFFFF).   */
/* R3 of that value, read exactly as a double; a NaN pattern gives 0xFF.      */
void uqo_e2m1_codes_bits(uint32_t first, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    uint32_t b = first + (uint32_t)i;
    float f;
    memcpy(&f, &b, 4);
    out[i] = isnan(f) ? 0xFF : (uint8_t)uqo_e2m1_code((double)f);
  }
}

/* R2 with the pages' constant for a group whose absolute maximum is |value|. */
void uqo_scale_bytes_bits(uint32_t first, int64_t n, float c, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    uint32_t b = first + (uint32_t)i;
    float f;
    memcpy(&f, &b, 4);
    out[i] = (uint8_t)uqo_scale_byte(fabsf(f), c, 0);
  }
}

void uqo_e4m3_codes(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)uqo_e4m3_code(x[i]);
}

void uqo_scale_bytes(const float* m, int64_t n, float c, int mode, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)uqo_scale_byte(m[i], c, mode);
}

/* Mean squared reconstruction error of 32-element groups, the objective of  */
/* the constant c ([UQ-residency], c* = argmin_c E[(z - c m q(z/(c m)))^2]).  */
/* mode < 0: continuous scale s = c*m; mode >= 0: s = 2^E with the R2 byte   */
/* rounding of that mode.                                                     */
double uqo_group_mse(const float* y, int64_t n_groups, float c, int mode) {
  double acc = 0.0;
  for (int64_t g = 0; g < n_groups; ++g) {
    const float* yg = y + 32 * g;
    float m = 0.0f;
    for (int i = 0; i < 32; ++i)
      if (fabsf(yg[i]) > m) m = fabsf(yg[i]);
    double s;
    if (m == 0.0f) continue;
    if (mode < 0) s = (double)c * (double)m;
    else s = ldexp(1.0, uqo_scale_byte(m, c, mode) - 127);
    for (int i = 0; i < 32; ++i) {
      double rec = s * uqo_e2m1_value(uqo_e2m1_code((double)yg[i] / s));
      double e = (double)yg[i] - rec;
      acc += e * e;
    }
  }
  return acc / (double)(32 * n_groups);
}
