/*
 * moe_oracle.c -- TEST INFRASTRUCTURE ONLY: the CPU oracle of the routed-expert
 * MoE layer.  Plain, single-threaded, obviously correct; FP64 accumulation.
 *
 * Sources (restated, never copied):
 *   [minnow] "coder543/minnow" README, "Quantization": NVFP4 = E2M1 values,
 *            E4M3 scales per 16, FP32 accumulation; INT4/INT8 = groups of 128
 *            weights with FP16 scales; the optional INT8 activation mode
 *            quantises activations per group, accumulates in INT32 and applies
 *            the scales in FP32; routed experts run fused gate/up/SiLU.
 *   [card]   "LLaDA2.2-flash-minnow" model card, "Checkpoints and precision":
 *            signed INT8 / signed INT4 with one FP16 scale per 128 weights;
 *            NVFP4 weights with an FP32 outer scale per expert matrix and
 *            activations with an FP32 outer scale per input row; W8A8/W4A8
 *            quantise expert inputs to signed INT8 with FP32 scales per 128
 *            values, use INT32 group dot products and combine scaled groups
 *            in FP32; the layer's outputs are BF16 again.
 *
 * Where the pages are silent, the reading taken is stated at the point of
 * use below.
 *
 * Build: plain C11, -ffp-contract=off (no fused multiply-add contraction), no
 * fast-math, so that every float expression rounds as written.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Scalar decoders                                                            */
/* ------------------------------------------------------------------------- */

/* BF16 is the upper half of an IEEE binary32. */
double mnwo_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits; subnormals
 * are fraction * 2^-24.  FP16 scales must be finite. */
int mnwo_fp16_to_double(uint16_t bits, double* out) {
  int s = (bits >> 15) & 1, e = (bits >> 10) & 0x1f, f = bits & 0x3ff;
  double v;
  if (e == 31) return MNWO_E_NONFINITE;
  if (e == 0) v = ldexp((double)f, -24);
  else v = ldexp((double)(1024 + f), e - 25);
  *out = s ? -v : v;
  return MNWO_OK;
}

/* Signed INT4: a two's-complement nibble ([card] "Signed INT4"). */
int mnwo_int4_value(uint8_t nibble) {
  int v = nibble & 0xf;
  return v >= 8 ? v - 16 : v;
}

/* Signed INT8: a two's-complement byte ([card] "Signed INT8"). */
int mnwo_int8_value(uint8_t byte) { return byte >= 128 ? (int)byte - 256 : (int)byte; }

/* E2M1: sign | 2 exponent bits (bias 1) | 1 mantissa bit.  Exponent 0 is
 * subnormal: mantissa * 0.5.  Magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}. */
double mnwo_e2m1_to_double(uint8_t nibble) {
  int s = (nibble >> 3) & 1, e = (nibble >> 1) & 3, m = nibble & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

/* E4M3 (OCP E4M3FN): sign | 4 exponent bits (bias 7) | 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; exponent 0 is subnormal: m/8 * 2^-6. */
int mnwo_e4m3_to_double(uint8_t byte, double* out) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 0xf, m = byte & 7;
  double v;
  if (e == 15 && m == 7) return MNWO_E_NONFINITE;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  *out = s ? -v : v;
  return MNWO_OK;
}

/* ------------------------------------------------------------------------- */
/* Scalar encoders                                                            */
/* ------------------------------------------------------------------------- */

/* Round a finite a >= 0 to the nearest value of a binary format with `mbits`
 * stored mantissa bits and minimum normal exponent `emin` (subnormals below
 * it), ties to the even mantissa.  Exact: every step is a power-of-two scaling
 * or an integer comparison. */
static double round_to_format(double a, int mbits, int emin) {
  int e2;
  double fl, frac, n, quantum;
  if (a == 0.0) return 0.0;
  frexp(a, &e2);           /* a = f * 2^e2, f in [0.5, 1): leading bit at e2-1 */
  e2 -= 1;
  if (e2 < emin) e2 = emin; /* subnormal range shares the emin quantum */
  quantum = ldexp(1.0, e2 - mbits);
  n = a / quantum;          /* exact */
  fl = floor(n);
  frac = n - fl;
  if (frac > 0.5) fl += 1.0;
  else if (frac == 0.5 && fmod(fl, 2.0) != 0.0) fl += 1.0;
  return fl * quantum;
}

uint16_t mnwo_bf16_from_double(double v) {
  /* BF16 keeps 7 mantissa bits and binary32's exponent range (emin -126). */
  double a = fabs(v), r;
  float f;
  uint32_t u;
  if (isnan(v)) return 0x7fc0;
  r = round_to_format(a, 7, -126);
  if (r > 3.38953138925153547590e+38 /* largest finite BF16 */) r = INFINITY;
  f = (float)r; /* exact: r is representable in binary32 */
  u = 0;
  memcpy(&u, &f, sizeof u);
  u >>= 16;
  if (signbit(v)) u |= 0x8000;
  return (uint16_t)u;
}

/* IEEE binary16 encoder: RNE, 10 stored mantissa bits, emin -14 with
 * subnormals below it, overflow to Inf. */
uint16_t mnwo_fp16_from_double(double v) {
  double a = fabs(v), r;
  int e2, code;
  if (isnan(v)) return 0x7e00;
  r = round_to_format(a, 10, -14);
  if (r > 65504.0) code = 0x7c00;
  else if (r < ldexp(1.0, -14)) code = (int)(r / ldexp(1.0, -24)); /* subnormal: m * 2^-24 */
  else {
    double f = frexp(r, &e2);          /* r = f * 2^e2, f in [0.5,1) */
    int m = (int)((2.0 * f - 1.0) * 1024.0);
    code = ((e2 - 1 + 15) << 10) | m;
  }
  return (uint16_t)((signbit(v) ? 0x8000 : 0) | code);
}

/* E4M3 encoder: RNE, saturating to the largest finite magnitude 448.  The
 * sign of the input is kept, also for results that round to zero. */
uint8_t mnwo_e4m3_rn_satfinite(float v) {
  double a = fabs((double)v), r;
  int s = signbit(v) ? 1 : 0, e2, code;
  r = round_to_format(a, 3, -6);
  if (r > 448.0) r = 448.0;
  if (r < ldexp(1.0, -6)) {
    code = (int)(r / ldexp(1.0, -9)); /* subnormal: m * 2^-9 */
  } else {
    double f = frexp(r, &e2);         /* r = f * 2^e2, f in [0.5,1) */
    int m = (int)((2.0 * f - 1.0) * 8.0);
    code = ((e2 - 1 + 7) << 3) | m;
  }
  return (uint8_t)((s << 7) | code);
}

/* E2M1 encoder: RNE, saturating at 6.  A negative input that rounds to zero
 * keeps its sign (code 0x8). */
uint8_t mnwo_e2m1_rn_satfinite(float v) {
  double a = fabs((double)v), r;
  int s = signbit(v) ? 1 : 0, code;
  r = round_to_format(a, 1, 0);
  if (r > 6.0) r = 6.0;
  if (r < 1.0) code = (int)(r / 0.5);             /* 0 or 0.5 */
  else {
    int e2;
    double f = frexp(r, &e2);
    int m = (int)((2.0 * f - 1.0) * 2.0);
    code = ((e2 - 1 + 1) << 1) | m;
  }
  return (uint8_t)((s << 3) | code);
}

/* ------------------------------------------------------------------------- */
/* Dynamic activation quantisers                                              */
/* ------------------------------------------------------------------------- */

static float bf16f(uint16_t b) { return (float)mnwo_bf16_to_double(b); }

/* Round a binary32 to the nearest integer, ties to even. */
static float rne_int(float v) {
  double d = (double)v, fl = floor(d), frac = d - fl;
  if (frac > 0.5) fl += 1.0;
  else if (frac == 0.5 && fmod(fl, 2.0) != 0.0) fl += 1.0;
  return (float)fl;
}

/* [card] W8A8/W4A8 paragraph: inputs become signed INT8 with an FP32 scale per
 * 128 values.  Reading: symmetric absmax scaling, scale = amax / 127 and
 * code = clamp(rne(x / scale), -127, 127), every step one binary32 operation;
 * a group whose amax is 0 gets scale 0 and codes 0. */
int mnwo_quant_int8_g128(const uint16_t* x, int R, int K, int8_t* codes, float* scales) {
  int G, r, g, i;
  if (R < 0 || K <= 0 || K % 128) return MNWO_E_ARG;
  G = K / 128;
  for (r = 0; r < R; ++r) {
    for (g = 0; g < G; ++g) {
      const uint16_t* xs = x + (size_t)r * K + g * 128;
      int8_t* q = codes + (size_t)r * K + g * 128;
      float amax = 0.0f, scale;
      for (i = 0; i < 128; ++i) {
        float a = fabsf(bf16f(xs[i]));
        if (a > amax) amax = a;
      }
      if (amax == 0.0f) {
        scales[(size_t)r * G + g] = 0.0f;
        for (i = 0; i < 128; ++i) q[i] = 0;
        continue;
      }
      scale = amax / 127.0f;
      scales[(size_t)r * G + g] = scale;
      for (i = 0; i < 128; ++i) {
        float t = rne_int(bf16f(xs[i]) / scale);
        if (t > 127.0f) t = 127.0f;
        if (t < -127.0f) t = -127.0f;
        q[i] = (int8_t)t;
      }
    }
  }
  return MNWO_OK;
}

/* [card] NVFP4 row: activations become E2M1 with an E4M3 scale per 16 values
 * and an FP32 outer scale per input row.  Reading (the two-level NVFP4 recipe,
 * binary32 steps):
 *   outer = amax_row / 2688            (2688 = 6 * 448, the largest product)
 *   sb    = e4m3(rn, satfinite)((amax_block / outer) / 6)
 *   d     = float(sb) * outer
 *   code  = e2m1(rn, satfinite)(x / d)
 * A row with outer == 0, or a block with d == 0, gets zero codes (and scale
 * byte 0 where sb is 0). */
int mnwo_quant_nvfp4_g16(const uint16_t* x, int R, int K, uint8_t* codes, uint8_t* sf, float* outer) {
  int r, b, i;
  if (R < 0 || K <= 0 || K % 16) return MNWO_E_ARG;
  for (r = 0; r < R; ++r) {
    const uint16_t* xr = x + (size_t)r * K;
    uint8_t* cr = codes + (size_t)r * (K / 2);
    uint8_t* sr = sf + (size_t)r * (K / 16);
    float amax = 0.0f, o;
    for (i = 0; i < K; ++i) {
      float a = fabsf(bf16f(xr[i]));
      if (a > amax) amax = a;
    }
    o = amax / 2688.0f;
    outer[r] = o;
    memset(cr, 0, (size_t)K / 2);
    memset(sr, 0, (size_t)K / 16);
    if (o == 0.0f) continue;
    for (b = 0; b < K / 16; ++b) {
      float ab = 0.0f, s, d;
      double sbv;
      uint8_t sb;
      for (i = 0; i < 16; ++i) {
        float a = fabsf(bf16f(xr[b * 16 + i]));
        if (a > ab) ab = a;
      }
      s = (ab / o) / 6.0f;
      sb = mnwo_e4m3_rn_satfinite(s);
      sr[b] = sb;
      mnwo_e4m3_to_double(sb, &sbv);
      d = (float)sbv * o;
      if (d == 0.0f) continue;
      for (i = 0; i < 16; ++i) {
        int kk = b * 16 + i;
        uint8_t c = mnwo_e2m1_rn_satfinite(bf16f(xr[kk]) / d);
        cr[kk / 2] |= (uint8_t)((kk & 1) ? (c << 4) : c); /* low nibble = even index */
      }
    }
  }
  return MNWO_OK;
}

/* ------------------------------------------------------------------------- */
/* Permutation                                                                */
/* ------------------------------------------------------------------------- */

/* Assignment a = t*k + j goes to expert ids[a].  counts -> exclusive offsets;
 * position of a = offsets[e] + number of earlier assignments to the same
 * expert (stable in a).  Out-of-range ids are dropped: assign_pos[a] = -1.
 * sorted_assign[pos] = a; unused tail slots hold -1. */
/* Not a step of the pages: the CUDA path's FP16 operand form of a BF16 row
 * (W8A16/W4A16 gate/up on FP16 tensor cores).  A power-of-two factor moves
 * the row's largest magnitude into [2^14, 2^15), so no value overflows FP16
 * and values down to 2^-28 of the maximum stay normal.  The clamp keeps 2^e
 * and 2^-e normal binary32 numbers (every finite BF16 row has e <= 113). */
int mnwo_encode_f16_rows(const uint16_t* x, int R, int K, uint16_t* codes, float* factor) {
  int r, k;
  if (!x || !codes || !factor || R < 0 || K <= 0) return MNWO_E_ARG;
  for (r = 0; r < R; ++r) {
    const uint16_t* row = x + (size_t)r * K;
    double amax = 0.0;
    int e;
    for (k = 0; k < K; ++k) {
      double v = mnwo_bf16_to_double(row[k]);
      if (!isfinite(v)) return MNWO_E_NONFINITE;
      if (fabs(v) > amax) amax = fabs(v);
    }
    if (amax == 0.0) e = -110;
    else {
      frexp(amax, &e);  /* amax = f * 2^e, f in [0.5, 1): floor(log2 amax) = e - 1 */
      e = e - 1 - 14;
      if (e < -110) e = -110;
      if (e > 113) e = 113;
    }
    factor[r] = (float)ldexp(1.0, e);
    for (k = 0; k < K; ++k) codes[(size_t)r * K + k] = mnwo_fp16_from_double(ldexp(mnwo_bf16_to_double(row[k]), -e));
  }
  return MNWO_OK;
}

/* Router: logits by the plain dot product, then the k largest by selection
 * (each pass takes the largest logit not yet chosen; on equal logits the
 * first expert in index order), then a softmax over the chosen logits. */
int mnwo_route(const uint16_t* x, const uint16_t* wr, int T, int H, int E, int k, int32_t* ids, float* w,
               double* logits) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || k > E || !x || !wr || !ids || !w) return MNWO_E_ARG;
  double* l = (double*)malloc(sizeof(double) * (size_t)E);
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  if (!l || !taken) {
    free(l);
    free(taken);
    return MNWO_E_ARG;
  }
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += mnwo_bf16_to_double(x[(size_t)t * H + h]) * mnwo_bf16_to_double(wr[(size_t)e * H + h]);
      l[e] = acc;
      taken[e] = 0;
      if (logits) logits[(size_t)t * E + e] = acc;
    }
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      ids[(size_t)t * k + j] = best;
    }
    const double lmax = l[ids[(size_t)t * k]];
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += exp(l[ids[(size_t)t * k + j]] - lmax);
    for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = (float)(exp(l[ids[(size_t)t * k + j]] - lmax) / sum);
  }
  free(l);
  free(taken);
  return MNWO_OK;
}

int mnwo_permute(const int32_t* ids, int T, int k, int E,
                 int32_t* expert_offsets, int32_t* sorted_assign, int32_t* assign_pos) {
  int P, a, e, dropped = 0;
  int32_t* fill;
  if (T < 0 || k <= 0 || E <= 0) return -1;
  P = T * k;
  for (e = 0; e <= E; ++e) expert_offsets[e] = 0;
  for (a = 0; a < P; ++a) {
    if (ids[a] >= 0 && ids[a] < E) expert_offsets[ids[a] + 1] += 1;
    else dropped += 1;
  }
  for (e = 0; e < E; ++e) expert_offsets[e + 1] += expert_offsets[e];
  fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  if (!fill) return -1;
  for (a = 0; a < P; ++a) sorted_assign[a] = -1;
  for (a = 0; a < P; ++a) {
    int id = ids[a];
    if (id < 0 || id >= E) { assign_pos[a] = -1; continue; }
    assign_pos[a] = expert_offsets[id] + fill[id];
    sorted_assign[assign_pos[a]] = a;
    fill[id] += 1;
  }
  free(fill);
  return dropped;
}

/* ------------------------------------------------------------------------- */
/* Expert blob                                                                */
/* ------------------------------------------------------------------------- */
/* Layout (little-endian), defined by this library since the pages give none:
 *   header, 256 bytes: "MNWB", u32 version=1, u32 wfmt, u32 E, u32 H, u32 I,
 *   u32 group, u32 header_bytes=256, u64 data_offset, u64 expert_stride,
 *   u64 codes_off[3], u64 scales_off[3], u64 outer_off[3], u64 total_bytes,
 *   zero padding, u32 CRC-32 (IEEE 802.3) of bytes [0, 252) at byte 252.
 *   Expert e starts at data_offset + e*expert_stride; its matrices gate [I,H],
 *   up [I,H], down [H,I] are row-major with K (the reduction index) fastest:
 *   BF16: u16 [N][K].  INT8: i8 [N][K] then f16 scales [N][K/128].
 *   INT4: u8 [N][K/2] (even k in the low nibble) then f16 scales [N][K/128].
 *   NVFP4: u8 [N][K/2] (same nibble order), E4M3 scales [N][K/16], f32 outer. */

static uint32_t rd32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
static uint64_t rd64(const uint8_t* p) { return (uint64_t)rd32(p) | ((uint64_t)rd32(p + 4) << 32); }

/* CRC-32 (reflected polynomial 0xEDB88320), bit by bit. */
static uint32_t crc32_ieee(const uint8_t* p, size_t n) {
  uint32_t c = 0xffffffffu;
  size_t i;
  int b;
  for (i = 0; i < n; ++i) {
    c ^= p[i];
    for (b = 0; b < 8; ++b) c = (c & 1) ? (c >> 1) ^ 0xedb88320u : (c >> 1);
  }
  return c ^ 0xffffffffu;
}

static void mat_dims(const mnwo_blob_info* in, int m, int* N, int* K) {
  if (m == MNWO_DOWN) { *N = (int)in->H; *K = (int)in->I; }
  else { *N = (int)in->I; *K = (int)in->H; }
}

int mnwo_blob_parse(const uint8_t* blob, size_t bytes, mnwo_blob_info* in) {
  int m;
  if (!blob || bytes < 256) return MNWO_E_BLOB;
  if (memcmp(blob, "MNWB", 4) != 0 || rd32(blob + 4) != 1 || rd32(blob + 28) != 256) return MNWO_E_BLOB;
  if (crc32_ieee(blob, 252) != rd32(blob + 252)) return MNWO_E_BLOB;
  in->wfmt = rd32(blob + 8);
  in->E = rd32(blob + 12);
  in->H = rd32(blob + 16);
  in->I = rd32(blob + 20);
  in->group = rd32(blob + 24);
  in->data_offset = rd64(blob + 32);
  in->expert_stride = rd64(blob + 40);
  for (m = 0; m < 3; ++m) {
    in->codes_off[m] = rd64(blob + 48 + 8 * m);
    in->scales_off[m] = rd64(blob + 72 + 8 * m);
    in->outer_off[m] = rd64(blob + 96 + 8 * m);
  }
  in->total_bytes = rd64(blob + 120);
  if (in->wfmt > 3 || in->E == 0 || in->H == 0 || in->I == 0) return MNWO_E_BLOB;
  if (in->H % 128 || in->I % 128) return MNWO_E_BLOB;
  if ((in->wfmt == MNWO_FMT_BF16 && in->group != 0) ||
      ((in->wfmt == MNWO_FMT_INT8_G128 || in->wfmt == MNWO_FMT_INT4_G128) && in->group != 128) ||
      (in->wfmt == MNWO_FMT_NVFP4_G16 && in->group != 16))
    return MNWO_E_BLOB;
  if (in->total_bytes > bytes || in->data_offset + (uint64_t)in->E * in->expert_stride > in->total_bytes)
    return MNWO_E_BLOB;
  for (m = 0; m < 3; ++m) {
    int N, K;
    uint64_t cb, sb = 0;
    mat_dims(in, m, &N, &K);
    cb = (uint64_t)N * K * (in->wfmt == MNWO_FMT_BF16 ? 2 : in->wfmt == MNWO_FMT_INT8_G128 ? 1 : 0);
    if (in->wfmt >= MNWO_FMT_INT4_G128) cb = (uint64_t)N * K / 2;
    if (in->codes_off[m] + cb > in->expert_stride) return MNWO_E_BLOB;
    if (in->wfmt == MNWO_FMT_INT8_G128 || in->wfmt == MNWO_FMT_INT4_G128) sb = (uint64_t)N * (K / 128) * 2;
    if (in->wfmt == MNWO_FMT_NVFP4_G16) sb = (uint64_t)N * (K / 16);
    if (in->scales_off[m] + sb > in->expert_stride) return MNWO_E_BLOB;
    if (in->wfmt == MNWO_FMT_NVFP4_G16 && in->outer_off[m] + 4 > in->expert_stride) return MNWO_E_BLOB;
  }
  return MNWO_OK;
}

/* Decoded weight value ([card] precision table):
 *   INT8/INT4: q * fp16 scale of group floor(k/128) of row n;
 *   NVFP4: e2m1 * e4m3 scale of block floor(k/16) of row n * FP32 outer scale
 *          of the matrix (reading: all three factors multiply);
 *   BF16: the value itself. */
int mnwo_weight(const uint8_t* blob, const mnwo_blob_info* in, int e, int m, int n, int k, double* out) {
  int N, K, rc;
  const uint8_t* base = blob + in->data_offset + (uint64_t)e * in->expert_stride;
  const uint8_t* codes = base + in->codes_off[m];
  const uint8_t* scales = base + in->scales_off[m];
  double s, sb;
  mat_dims(in, m, &N, &K);
  switch (in->wfmt) {
    case MNWO_FMT_BF16: {
      const uint8_t* p = codes + ((size_t)n * K + k) * 2;
      *out = mnwo_bf16_to_double((uint16_t)(p[0] | (p[1] << 8)));
      return MNWO_OK;
    }
    case MNWO_FMT_INT8_G128: {
      const uint8_t* sp = scales + ((size_t)n * (K / 128) + k / 128) * 2;
      rc = mnwo_fp16_to_double((uint16_t)(sp[0] | (sp[1] << 8)), &s);
      if (rc) return rc;
      *out = mnwo_int8_value(codes[(size_t)n * K + k]) * s;
      return MNWO_OK;
    }
    case MNWO_FMT_INT4_G128: {
      const uint8_t* sp = scales + ((size_t)n * (K / 128) + k / 128) * 2;
      uint8_t byte = codes[(size_t)n * (K / 2) + k / 2];
      rc = mnwo_fp16_to_double((uint16_t)(sp[0] | (sp[1] << 8)), &s);
      if (rc) return rc;
      *out = mnwo_int4_value((k & 1) ? (byte >> 4) : (byte & 0xf)) * s;
      return MNWO_OK;
    }
    case MNWO_FMT_NVFP4_G16: {
      uint8_t byte = codes[(size_t)n * (K / 2) + k / 2];
      float o;
      memcpy(&o, base + in->outer_off[m], 4);
      rc = mnwo_e4m3_to_double(scales[(size_t)n * (K / 16) + k / 16], &sb);
      if (rc) return rc;
      if (!isfinite(o)) return MNWO_E_NONFINITE;
      *out = mnwo_e2m1_to_double((k & 1) ? (byte >> 4) : (byte & 0xf)) * sb * (double)o;
      return MNWO_OK;
    }
  }
  return MNWO_E_BLOB;
}

/* ------------------------------------------------------------------------- */
/* One expert applied to one row                                              */
/* ------------------------------------------------------------------------- */

/* SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g))  (reading of "SiLU"). */
static double silu(double g) { return g / (1.0 + exp(-g)); }

/* Activation row in one of the three modes, held decoded for the dot products. */
typedef struct {
  int act, K;
  const uint16_t* bf16;                                   /* A16 */
  const uint16_t* f16;                                    /* FP16 rows (factor in outer) */
  const int8_t* q; const float* s;                        /* A8: codes, scales [K/128] */
  const uint8_t* c4; const uint8_t* sf; float outer;      /* A4 */
} act_row;

/* Dot product of an activation row with row n of matrix m of expert e. */
static int row_dot(const uint8_t* blob, const mnwo_blob_info* in, int e, int m, int n,
                   const act_row* a, double* out, int32_t* dots /* nullable, [K/128] */) {
  int k, rc, K = a->K;
  double acc = 0.0, w;
  if (a->act == MNWO_ACT_BF16) {
    for (k = 0; k < K; ++k) {
      rc = mnwo_weight(blob, in, e, m, n, k, &w);
      if (rc) return rc;
      acc += mnwo_bf16_to_double(a->bf16[k]) * w;
    }
  } else if (a->act == MNWO_ACT_F16_ROWS) {
    for (k = 0; k < K; ++k) {
      double v;
      rc = mnwo_weight(blob, in, e, m, n, k, &w);
      if (rc) return rc;
      rc = mnwo_fp16_to_double(a->f16[k], &v);
      if (rc) return rc;
      acc += v * w;
    }
    acc *= (double)a->outer;
  } else if (a->act == MNWO_ACT_INT8_G128) {
    /* INT32 group dot products of the integer codes, each scaled by
     * (weight scale * activation scale) and summed ([card] W8A8 paragraph). */
    const uint8_t* base = blob + in->data_offset + (uint64_t)e * in->expert_stride;
    const uint8_t* codes = base + in->codes_off[m];
    const uint8_t* scales = base + in->scales_off[m];
    int g, G = K / 128;
    for (g = 0; g < G; ++g) {
      long long d = 0;
      double sw;
      const uint8_t* sp = scales + ((size_t)n * G + g) * 2;
      for (k = g * 128; k < g * 128 + 128; ++k) {
        int qw;
        if (in->wfmt == MNWO_FMT_INT8_G128) qw = mnwo_int8_value(codes[(size_t)n * K + k]);
        else {
          uint8_t byte = codes[(size_t)n * (K / 2) + k / 2];
          qw = mnwo_int4_value((k & 1) ? (byte >> 4) : (byte & 0xf));
        }
        d += (long long)a->q[k] * qw;
      }
      if (d > 2147483647LL || d < -2147483648LL) return MNWO_E_ARG; /* cannot happen: |d| <= 128*127*127 */
      if (dots) dots[g] = (int32_t)d;
      rc = mnwo_fp16_to_double((uint16_t)(sp[0] | (sp[1] << 8)), &sw);
      if (rc) return rc;
      acc += (sw * (double)a->s[g]) * (double)d;
    }
  } else {
    /* NVFP4: products of the block-scaled E2M1 values, then both outer scales. */
    const uint8_t* base = blob + in->data_offset + (uint64_t)e * in->expert_stride;
    const uint8_t* codes = base + in->codes_off[m];
    const uint8_t* scales = base + in->scales_off[m];
    float ow;
    memcpy(&ow, base + in->outer_off[m], 4);
    for (k = 0; k < K; ++k) {
      double sbw, sba, vw, va;
      uint8_t bw = codes[(size_t)n * (K / 2) + k / 2], ba = a->c4[k / 2];
      rc = mnwo_e4m3_to_double(scales[(size_t)n * (K / 16) + k / 16], &sbw);
      if (rc) return rc;
      rc = mnwo_e4m3_to_double(a->sf[k / 16], &sba);
      if (rc) return rc;
      vw = mnwo_e2m1_to_double((k & 1) ? (bw >> 4) : (bw & 0xf)) * sbw;
      va = mnwo_e2m1_to_double((k & 1) ? (ba >> 4) : (ba & 0xf)) * sba;
      acc += va * vw;
    }
    acc *= (double)a->outer * (double)ow;
  }
  *out = acc;
  return MNWO_OK;
}

static int mode_ok(uint32_t wfmt, int act) {
  if (act == MNWO_ACT_BF16) return wfmt != MNWO_FMT_NVFP4_G16;
  if (act == MNWO_ACT_INT8_G128) return wfmt == MNWO_FMT_INT8_G128 || wfmt == MNWO_FMT_INT4_G128;
  if (act == MNWO_ACT_NVFP4_G16) return wfmt == MNWO_FMT_NVFP4_G16;
  if (act == MNWO_ACT_F16_ROWS) return wfmt == MNWO_FMT_INT8_G128 || wfmt == MNWO_FMT_INT4_G128;
  return 0;
}

/* One grouped-GEMM output row: GATE_UP writes I values bf16(SiLU(g)*u),
 * DOWN writes H values bf16(dot), GATE / UP write I values bf16(dot) of the
 * gate / up matrix alone (the unfused-activation comparison path). */
static int expert_row(const uint8_t* blob, const mnwo_blob_info* in, int kind, int e,
                      const act_row* a, uint16_t* out, int32_t* dots) {
  int n, rc, N = kind == MNWO_KIND_DOWN ? (int)in->H : (int)in->I;
  int G = a->K / 128;
  for (n = 0; n < N; ++n) {
    double g, u;
    if (kind == MNWO_KIND_GATE_UP) {
      rc = row_dot(blob, in, e, MNWO_GATE, n, a, &g, dots ? dots + (size_t)n * G : NULL);
      if (rc) return rc;
      rc = row_dot(blob, in, e, MNWO_UP, n, a, &u, dots ? dots + (size_t)(N + n) * G : NULL);
      if (rc) return rc;
      out[n] = mnwo_bf16_from_double(silu(g) * u);
    } else {
      const int m = kind == MNWO_KIND_DOWN ? MNWO_DOWN : (kind == MNWO_KIND_GATE ? MNWO_GATE : MNWO_UP);
      rc = row_dot(blob, in, e, m, n, a, &g, dots ? dots + (size_t)n * G : NULL);
      if (rc) return rc;
      out[n] = mnwo_bf16_from_double(g);
    }
  }
  return MNWO_OK;
}

static int gemm_common(const uint8_t* blob, size_t bytes, int kind, int act, const void* a0,
                       const void* a1, const void* a2, const int32_t* offsets, int P,
                       uint16_t* out, int32_t* dots) {
  mnwo_blob_info in;
  int rc, e, p, K, N;
  if ((rc = mnwo_blob_parse(blob, bytes, &in))) return rc;
  if (!mode_ok(in.wfmt, act)) return MNWO_E_MODE;
  if (kind < MNWO_KIND_GATE_UP || kind > MNWO_KIND_UP) return MNWO_E_ARG;
  K = kind == MNWO_KIND_DOWN ? (int)in.I : (int)in.H;
  N = kind == MNWO_KIND_DOWN ? (int)in.H : (int)in.I;
  if (offsets[0] < 0 || offsets[in.E] > P) return MNWO_E_ARG;
  for (e = 0; e < (int)in.E; ++e) {
    if (offsets[e + 1] < offsets[e]) return MNWO_E_ARG;
    for (p = offsets[e]; p < offsets[e + 1]; ++p) {
      act_row r;
      memset(&r, 0, sizeof r);
      r.act = act;
      r.K = K;
      if (act == MNWO_ACT_BF16) r.bf16 = (const uint16_t*)a0 + (size_t)p * K;
      else if (act == MNWO_ACT_F16_ROWS) {
        r.f16 = (const uint16_t*)a0 + (size_t)p * K;
        r.outer = ((const float*)a1)[p];
      } else if (act == MNWO_ACT_INT8_G128) {
        r.q = (const int8_t*)a0 + (size_t)p * K;
        r.s = (const float*)a1 + (size_t)p * (K / 128);
      } else {
        r.c4 = (const uint8_t*)a0 + (size_t)p * (K / 2);
        r.sf = (const uint8_t*)a1 + (size_t)p * (K / 16);
        r.outer = ((const float*)a2)[p];
      }
      rc = expert_row(blob, &in, kind, e, &r, out + (size_t)p * N,
                      dots ? dots + (size_t)p * (kind == MNWO_KIND_GATE_UP ? 2 : 1) * N * (K / 128) : NULL);
      if (rc) return rc;
    }
  }
  return MNWO_OK;
}

int mnwo_gemm_a16(const uint8_t* blob, size_t bytes, int kind, const uint16_t* a,
                  const int32_t* offsets, int P, uint16_t* out) {
  return gemm_common(blob, bytes, kind, MNWO_ACT_BF16, a, NULL, NULL, offsets, P, out, NULL);
}

int mnwo_gemm_a8(const uint8_t* blob, size_t bytes, int kind, const int8_t* a_codes,
                 const float* a_scales, const int32_t* offsets, int P, uint16_t* out, int32_t* dots) {
  return gemm_common(blob, bytes, kind, MNWO_ACT_INT8_G128, a_codes, a_scales, NULL, offsets, P, out, dots);
}

int mnwo_gemm_a4(const uint8_t* blob, size_t bytes, int kind, const uint8_t* a_codes,
                 const uint8_t* a_sf, const float* a_outer, const int32_t* offsets, int P,
                 uint16_t* out) {
  return gemm_common(blob, bytes, kind, MNWO_ACT_NVFP4_G16, a_codes, a_sf, a_outer, offsets, P, out, NULL);
}

int mnwo_gemm_f16rows(const uint8_t* blob, size_t bytes, int kind, const uint16_t* a,
                      const float* factor, const int32_t* offsets, int P, uint16_t* out) {
  return gemm_common(blob, bytes, kind, MNWO_ACT_F16_ROWS, a, factor, NULL, offsets, P, out, NULL);
}

/* The activation of the unfused comparison path: out[i] = bf16(SiLU(g[i]) *
 * u[i]) from BF16 g and u, in FP64. */
void mnwo_silu_mul(const uint16_t* g, const uint16_t* u, size_t n, uint16_t* out) {
  size_t i;
  for (i = 0; i < n; ++i)
    out[i] = mnwo_bf16_from_double(silu(mnwo_bf16_to_double(g[i])) * mnwo_bf16_to_double(u[i]));
}

/* ------------------------------------------------------------------------- */
/* Combine and the whole layer                                                */
/* ------------------------------------------------------------------------- */

/* out[t] = bf16(sum_j w[t,j] * y[assign_pos[t*k+j]]), j ascending, in FP64;
 * dropped assignments (assign_pos < 0) contribute nothing.  The routing
 * weights are used as given (the router is outside the layer). */
void mnwo_combine(const uint16_t* y, const int32_t* assign_pos, const float* w, int T, int k,
                  int H, uint16_t* out) {
  int t, j, c;
  for (t = 0; t < T; ++t) {
    for (c = 0; c < H; ++c) {
      double acc = 0.0;
      for (j = 0; j < k; ++j) {
        int32_t pos = assign_pos[t * k + j];
        if (pos < 0) continue;
        acc += (double)w[t * k + j] * mnwo_bf16_to_double(y[(size_t)pos * H + c]);
      }
      out[(size_t)t * H + c] = mnwo_bf16_from_double(acc);
    }
  }
}

/* The layer for each selected token: for every slot j with a valid expert e,
 * (quantise x in A8/A4) -> h = bf16(SiLU(x.Wg^T) * (x.Wu^T)) -> (quantise h
 * in A8/A4, the same dynamic rule as for x) -> y = bf16(h.Wd^T); then
 * out = bf16(sum_j w_j y_j).  Each token depends only on its own row. */
int mnwo_moe_forward(const uint8_t* blob, size_t bytes, int act, const uint16_t* x,
                     const int32_t* ids, const float* w, int T, int k,
                     const int32_t* rows, int nrows, uint16_t* out) {
  mnwo_blob_info in;
  int rc = 0, i, j, c, H, I;
  uint16_t *h = NULL, *y = NULL;
  int8_t* q8 = NULL;
  float *s8 = NULL, outer = 0.0f;
  uint8_t *c4 = NULL, *sf = NULL;
  double* acc = NULL;
  if ((rc = mnwo_blob_parse(blob, bytes, &in))) return rc;
  if (act == MNWO_ACT_F16_ROWS || !mode_ok(in.wfmt, act)) return MNWO_E_MODE; /* not a layer mode */
  if (T < 0 || k <= 0) return MNWO_E_ARG;
  if (!rows) nrows = T;
  H = (int)in.H;
  I = (int)in.I;
  h = (uint16_t*)malloc(sizeof(uint16_t) * I);
  y = (uint16_t*)malloc(sizeof(uint16_t) * H);
  q8 = (int8_t*)malloc((size_t)(H > I ? H : I));
  s8 = (float*)malloc(sizeof(float) * ((H > I ? H : I) / 128));
  c4 = (uint8_t*)malloc((size_t)(H > I ? H : I) / 2);
  sf = (uint8_t*)malloc((size_t)(H > I ? H : I) / 16);
  acc = (double*)malloc(sizeof(double) * H);
  if (!h || !y || !q8 || !s8 || !c4 || !sf || !acc) { rc = MNWO_E_ARG; goto done; }
  for (i = 0; i < nrows; ++i) {
    int t = rows ? rows[i] : i;
    if (t < 0 || t >= T) { rc = MNWO_E_ARG; goto done; }
    for (c = 0; c < H; ++c) acc[c] = 0.0;
    for (j = 0; j < k; ++j) {
      int e = ids[t * k + j];
      act_row ra;
      if (e < 0 || e >= (int)in.E) continue; /* dropped */
      memset(&ra, 0, sizeof ra);
      ra.act = act;
      ra.K = H;
      if (act == MNWO_ACT_BF16) ra.bf16 = x + (size_t)t * H;
      else if (act == MNWO_ACT_INT8_G128) {
        mnwo_quant_int8_g128(x + (size_t)t * H, 1, H, q8, s8);
        ra.q = q8; ra.s = s8;
      } else {
        mnwo_quant_nvfp4_g16(x + (size_t)t * H, 1, H, c4, sf, &outer);
        ra.c4 = c4; ra.sf = sf; ra.outer = outer;
      }
      if ((rc = expert_row(blob, &in, MNWO_KIND_GATE_UP, e, &ra, h, NULL))) goto done;
      memset(&ra, 0, sizeof ra);
      ra.act = act;
      ra.K = I;
      if (act == MNWO_ACT_BF16) ra.bf16 = h;
      else if (act == MNWO_ACT_INT8_G128) {
        mnwo_quant_int8_g128(h, 1, I, q8, s8);
        ra.q = q8; ra.s = s8;
      } else {
        mnwo_quant_nvfp4_g16(h, 1, I, c4, sf, &outer);
        ra.c4 = c4; ra.sf = sf; ra.outer = outer;
      }
      if ((rc = expert_row(blob, &in, MNWO_KIND_DOWN, e, &ra, y, NULL))) goto done;
      for (c = 0; c < H; ++c) acc[c] += (double)w[t * k + j] * mnwo_bf16_to_double(y[c]);
    }
    for (c = 0; c < H; ++c) out[(size_t)i * H + c] = mnwo_bf16_from_double(acc[c]);
  }
done:
  free(h); free(y); free(q8); free(s8); free(c4); free(sf); free(acc);
  return rc;
}

/* ------------------------------------------------------------------------- */
/* Block attention for prefill (the second workload)                          */
/* ------------------------------------------------------------------------- */

/* [minnow] "Quantization": Block FlashAttention computes prompt attention
 * with the scores kept on chip; this is the result it computes, written out
 * directly.  For each selected token t of sequence b and query head h (kv
 * head g = h / (Hq / Hkv)):
 *   s_j = scale * sum_c q[b,t,h,c] * k[b,j,g,c]   for every allowed key j,
 *   out[b,t,h,:] = sum_j exp(s_j - max s) v[b,j,g,:] / sum_j exp(s_j - max s),
 * key j allowed iff j < T and j / blk <= t / blk (the block-causal mask of a
 * block-diffusion model's prompt: blk = 1 is causal, blk >= T bidirectional).
 * Everything in FP64 from the BF16 inputs.  q, out: [B, T, Hq, d]; k, v:
 * [B, T, Hkv, d]; rows (nullable) lists flat token indices b*T + t, and out
 * then holds [nrows, Hq, d]. */
int mnwo_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int T, int Hq, int Hkv,
                   int d, int blk, double scale, const int32_t* rows, int nrows, double* out) {
  int i, h, j, c;
  double *s = NULL, *qd = NULL;
  if (B <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || blk <= 0 || Hq % Hkv) return MNWO_E_ARG;
  if (!rows) nrows = B * T;
  s = (double*)malloc(sizeof(double) * T);
  qd = (double*)malloc(sizeof(double) * d);
  if (!s || !qd) { free(s); free(qd); return MNWO_E_ARG; }
  for (i = 0; i < nrows; ++i) {
    const int flat = rows ? rows[i] : i;
    int b, t, kmax;
    long long km;
    if (flat < 0 || flat >= B * T) { free(s); free(qd); return MNWO_E_ARG; }
    b = flat / T;
    t = flat % T;
    km = ((long long)(t / blk) + 1) * blk; /* keys 0 .. kmax-1 are allowed */
    kmax = km > T ? T : (int)km;
    for (h = 0; h < Hq; ++h) {
      const int g = h / (Hq / Hkv);
      double m = -INFINITY, l = 0.0;
      double* o = out + ((size_t)i * Hq + h) * d;
      for (c = 0; c < d; ++c) qd[c] = mnwo_bf16_to_double(q[(((size_t)b * T + t) * Hq + h) * d + c]);
      for (j = 0; j < kmax; ++j) {
        const uint16_t* kr = k + (((size_t)b * T + j) * Hkv + g) * d;
        double acc = 0.0;
        for (c = 0; c < d; ++c) acc += qd[c] * mnwo_bf16_to_double(kr[c]);
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
      }
      for (c = 0; c < d; ++c) o[c] = 0.0;
      for (j = 0; j < kmax; ++j) {
        const uint16_t* vr = v + (((size_t)b * T + j) * Hkv + g) * d;
        const double p = exp(s[j] - m);
        l += p;
        for (c = 0; c < d; ++c) o[c] += p * mnwo_bf16_to_double(vr[c]);
      }
      for (c = 0; c < d; ++c) o[c] /= l;
    }
  }
  free(s);
  free(qd);
  return 0;
}
