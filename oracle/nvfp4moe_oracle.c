/*
 * nvfp4moe_oracle.c -- plain, slow, obviously correct CPU restatement of the
 * NVFP4 mixture-of-experts expert computation at decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker that the CUDA path is
 * compared against.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load it.  It shares no code, header, table or
 * helper with the CUDA library: every table below is built here from the
 * format definitions, and every step is written in the order the method
 * states it, with no blocking, fusion or reordering.
 *
 * Sources (page titles and sections of the reference pages):
 *  - "The Benchmark That Confirmed the Ceiling: NVFP4 Cutlass on sm_120",
 *    section "The NVFP4 Pivot": NVFP4 = FP4 E2M1 values, group-16 E4M3 block
 *    scales; W4A16 (FP4 -> BF16 dequantise, BF16 MMA) versus native FP4xFP4.
 *  - "The 2x Gap: Diagnosing Suboptimal FP4 GEMM Kernels on Blackwell SM120",
 *    section "Discovering the sgl_kernel Alternative": a scaled FP4 GEMM takes
 *    (a, b, block_scale_a, block_scale_b, alpha) -- i.e. per-block scales on
 *    both operands plus one per-tensor coefficient; section "The Investigation
 *    So Far": routed top-8 of 256 experts, ~16 tokens per expert.
 *  - "The Benchmark That Confirmed the Ceiling: NVFP4 Cutlass on sm_120",
 *    sections "The Optimization Hierarchy" and "The NVFP4 Pivot": the stock checkpoint is
 *    MXFP4 -- group-32 blocks with UE8M0 (power-of-two) scales.
 *  - "The 24% Ceiling: Diagnosing the Limits of NVFP4 Quantization on
 *    Blackwell SM120 GPUs", section "The Core Insight": W4A16 keeps the
 *    activations in BF16, W4A4 quantises them to FP4 as well.
 *  - "Native FP4 Is Slower Than Emulated FP4 ...", section 1: routed experts
 *    (512 experts, 22 active per token); NVFP4 as FP4 weights with FP8
 *    activations (the W4A8 mode).
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes of the repository):
 *  - E2M1 and E4M3 are the standard OCP "MX" element/scale encodings: E2M1
 *    magnitudes {0,.5,1,1.5,2,3,4,6}; E4M3 "FN" (bias 7, no infinity, max 448,
 *    0x7F/0xFF = NaN).
 *  - Two-level scaling: per-tensor FP32 decode scale S = amax(|x|)/(6*448),
 *    block scale = E4M3(RNE, satfinite) of (amax_block/6)/S, element code =
 *    E2M1(RNE, satfinite) of x / (E4M3value * S).  Every one of these steps is
 *    a single IEEE fp32 operation, because a quantised code is an integer
 *    decision and both sides must take it in the same precision.
 *  - Ties to even, sign of zero kept (-0.1 -> code 0x8), S == 0 or a zero
 *    block decode scale gives scale code 0 and element code 0.
 *  - Packing: two E2M1 codes per byte, element 2i in the low nibble; block
 *    scales stored linearly as [rows, cols/16].
 *  - MXFP4 (the group-32, UE8M0 format the pages name as the stock
 *    checkpoint's): the OCP MX conversion -- shared exponent
 *    floor(log2(amax_block)) - 2 (E2M1's largest magnitude is 1.5 * 2^2),
 *    clamped to the UE8M0 range, elements E2M1(RNE, satfinite) of x / 2^E;
 *    an all-zero block takes the smallest scale.  No per-tensor scale.
 *    Scales stored linearly as [rows, cols/32].
 *  - FP8 activations (W4A8): E4M3 "FN" codes with one fp32 per-tensor decode
 *    scale, S = amax/448 (dynamic, for x) or a caller-given static S (for
 *    h); code = E4M3(RNE, satfinite) of x / S, sign kept.
 *  - Router: top-k by logit, ties to the lower expert id, descending order;
 *    weights = softmax over the k selected logits (fp64 here).
 *  - Permutation: stable by (expert, token).
 *  - Gate/up order: G[:, 0:I] = gate, G[:, I:2I] = up; SwiGLU h = silu(g)*u.
 *  - Storage roundings mirrored: G fp32, h fp32 before requantisation (or
 *    fp32 then BF16 in W4A16), Y fp32, out fp32.  All dot products and sums
 *    accumulate in fp64.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fopenmp
 * (no fast-math: IEEE division and no FMA contraction are required).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Format tables                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1 magnitudes indexed by the 3 low bits of a code (OCP MX element
 * format FP4 E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int code) {
  code &= 15;
  double m = E2M1_MAG[code & 7];
  return (code & 8) ? -m : m;
}

/* E4M3 "FN" decode straight from the field definition. */
double orc_e4m3_value(int code) {
  code &= 0xFF;
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);          /* subnormal: m/8 * 2^(1-7) */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal */
  return sign ? -v : v;
}

/* Round a non-negative fp32 value to the nearest finite E4M3 value, ties to
 * the code with an even mantissa LSB, saturating at 448.  Brute force over
 * all finite non-negative codes (0x00..0x7E, monotone in value). */
int orc_e4m3_encode(float bf) {
  double b = (double)bf;
  if (!(b >= 0.0)) return 0;      /* negative or NaN never occurs; map to 0 */
  if (b >= 448.0) return 0x7E;    /* satfinite */
  int best = 0;
  double bestd = fabs(b - orc_e4m3_value(0));
  for (int c = 1; c <= 0x7E; ++c) {
    double d = fabs(b - orc_e4m3_value(c));
    if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bestd = d;
    }
  }
  return best;
}

/* Round an fp32 value to the nearest E2M1 magnitude (ties to the even
 * code), saturating at 6; the sign bit is copied from the input even when
 * the magnitude rounds to zero. */
int orc_e2m1_encode(float q) {
  int neg = signbit(q) ? 1 : 0;
  double a = fabs((double)q);
  int best;
  if (a >= 6.0) {
    best = 7;
  } else {
    best = 0;
    double bestd = fabs(a - E2M1_MAG[0]);
    for (int c = 1; c < 8; ++c) {
      double d = fabs(a - E2M1_MAG[c]);
      if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
        best = c;
        bestd = d;
      }
    }
  }
  return best | (neg << 3);
}

/* fp32 -> bf16 with round-to-nearest-even: pick the nearer of the two bf16
 * neighbours (truncation and truncation + 1 ulp), ties to the even one.
 * Returns the bf16 value widened back to fp32. Finite inputs only. */
float orc_round_bf16(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  uint32_t lo_bits = u & 0xFFFF0000u;
  uint32_t hi_bits = lo_bits + 0x00010000u;  /* next bf16 away from zero */
  float lo, hi;
  memcpy(&lo, &lo_bits, 4);
  memcpy(&hi, &hi_bits, 4);
  double dl = fabs((double)v - (double)lo);
  double dh = fabs((double)v - (double)hi);
  if (dl < dh) return lo;
  if (dh < dl) return hi;
  return ((lo_bits >> 16) & 1u) ? hi : lo;  /* tie: even mantissa LSB */
}

/* ------------------------------------------------------------------------ */
/* NVFP4 quantisation                                                       */
/* ------------------------------------------------------------------------ */

static float f32_abs(float v) { return v < 0.0f ? -v : (v == 0.0f ? 0.0f : v); }

/* Per-tensor decode scale: S = fp32(amax(|x|)) / 2688 (one fp32 division). */
float orc_tensor_scale(const float* x, int64_t rows, int64_t cols, int64_t ld) {
  float amax = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      float a = f32_abs(x[r * ld + c]);
      if (a > amax) amax = a;
    }
  return amax / 2688.0f;
}

/* Quantise one 16-element block with decode scale S.  Writes the scale code
 * and 16 element codes (one per entry of `ecodes`). */
void orc_quantize_block(const float* xb, float S, uint8_t* scode, uint8_t* ecodes) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = f32_abs(xb[i]);
    if (a > amax) amax = a;
  }
  if (S == 0.0f) {
    *scode = 0;
    for (int i = 0; i < 16; ++i) ecodes[i] = 0;
    return;
  }
  float b = (amax / 6.0f) / S;               /* two fp32 divisions, in order */
  int sc = orc_e4m3_encode(b);
  float d = (float)orc_e4m3_value(sc) * S;   /* fp32 multiply */
  *scode = (uint8_t)sc;
  if (d == 0.0f) {
    for (int i = 0; i < 16; ++i) ecodes[i] = 0;
    return;
  }
  for (int i = 0; i < 16; ++i) {
    float q = xb[i] / d;                     /* fp32 IEEE division */
    ecodes[i] = (uint8_t)orc_e2m1_encode(q);
  }
}

/* Quantise x [rows, cols] (row stride ld, fp32 holding the input values) to
 * NVFP4: codes [rows, cols/2] (low nibble = even element), scales
 * [rows, cols/16].  dynamic != 0: S = amax/2688 is computed and written to
 * *S; otherwise *S is read. cols must be a multiple of 16. */
void orc_quantize(const float* x, int64_t rows, int64_t cols, int64_t ld, int dynamic, float* S,
                  uint8_t* codes, uint8_t* scales) {
  if (dynamic) *S = orc_tensor_scale(x, rows, cols, ld);
  float s = *S;
  int64_t nb = cols / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      uint8_t ec[16];
      uint8_t sc;
      orc_quantize_block(x + r * ld + b * 16, s, &sc, ec);
      scales[r * nb + b] = sc;
      for (int i = 0; i < 8; ++i)
        codes[r * (cols / 2) + b * 8 + i] = (uint8_t)(ec[2 * i] | (ec[2 * i + 1] << 4));
    }
  }
}

/* Decoded value of element (r, c) without the per-tensor scale:
 * e2m1(code) * e4m3(block scale).  Exact in fp64. */
static double dec_elem(const uint8_t* codes, const uint8_t* scales, int64_t cols, int64_t r, int64_t c) {
  uint8_t byte = codes[r * (cols / 2) + c / 2];
  int code = (c & 1) ? (byte >> 4) : (byte & 15);
  return orc_e2m1_value(code) * orc_e4m3_value(scales[r * (cols / 16) + c / 16]);
}

/* Full dequantisation to fp64 including the per-tensor scale. */
void orc_dequantize(const uint8_t* codes, const uint8_t* scales, float S, int64_t rows, int64_t cols,
                    double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = dec_elem(codes, scales, cols, r, c) * (double)S;
}

/* ------------------------------------------------------------------------ */
/* MXFP4 quantisation (OCP MX: E2M1 elements, one UE8M0 scale per 32)      */
/* ------------------------------------------------------------------------ */

/* UE8M0 decode: an unsigned 8-bit exponent, value 2^(code - 127); code 0xFF
 * is NaN. */
double orc_ue8m0_value(int code) {
  code &= 0xFF;
  if (code == 0xFF) return NAN;
  return ldexp(1.0, code - 127);
}

/* Quantise one 32-element block to MXFP4.  The shared exponent is
 * E = floor(log2(amax)) - 2, where 2 is the exponent of E2M1's largest
 * magnitude (6 = 1.5 * 2^2); E is clamped to the UE8M0 range [-127, 127],
 * and an all-zero block takes E = -127.  Scale code = E + 127.  Element
 * code = E2M1(RNE, satfinite, sign kept) of q = x / 2^E, where q is the fp32
 * value nearest the exact quotient (a power-of-two scaling: exact unless q is
 * subnormal).  Magnitudes in [6, 8) * 2^E saturate to 6. */
void orc_mx_quantize_block(const float* xb, uint8_t* scode, uint8_t* ecodes) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    float a = f32_abs(xb[i]);
    if (a > amax) amax = a;
  }
  int E;
  if (amax == 0.0f) {
    E = -127;
  } else {
    int p;
    frexp((double)amax, &p); /* amax = m * 2^p, m in [0.5, 1): floor(log2 amax) = p - 1 */
    E = (p - 1) - 2;
  }
  if (E < -127) E = -127;
  if (E > 127) E = 127;
  *scode = (uint8_t)(E + 127);
  for (int i = 0; i < 32; ++i) {
    float q = (float)ldexp((double)xb[i], -E); /* exact in fp64, one rounding to fp32 */
    ecodes[i] = (uint8_t)orc_e2m1_encode(q);
  }
}

/* Quantise x [rows, cols] (row stride ld) to MXFP4: codes [rows, cols/2]
 * (low nibble = even element), scales [rows, cols/32].  cols must be a
 * multiple of 32. */
void orc_mx_quantize(const float* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes, uint8_t* scales) {
  int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      uint8_t ec[32];
      uint8_t sc;
      orc_mx_quantize_block(x + r * ld + b * 32, &sc, ec);
      scales[r * nb + b] = sc;
      for (int i = 0; i < 16; ++i)
        codes[r * (cols / 2) + b * 16 + i] = (uint8_t)(ec[2 * i] | (ec[2 * i + 1] << 4));
    }
  }
}

/* Decoded MXFP4 element (r, c): e2m1(code) * 2^(scale - 127).  Exact in
 * fp64. */
static double dec_elem_mx(const uint8_t* codes, const uint8_t* scales, int64_t cols, int64_t r, int64_t c) {
  uint8_t byte = codes[r * (cols / 2) + c / 2];
  int code = (c & 1) ? (byte >> 4) : (byte & 15);
  return orc_e2m1_value(code) * orc_ue8m0_value(scales[r * (cols / 32) + c / 32]);
}

void orc_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) out[r * cols + c] = dec_elem_mx(codes, scales, cols, r, c);
}

/* ------------------------------------------------------------------------ */
/* Router and permutation                                                   */
/* ------------------------------------------------------------------------ */
/* FP8 (E4M3) activations with a per-tensor scale (W4A8)                    */
/* ------------------------------------------------------------------------ */

/* "NVFP4 means FP4 weights with FP8 activations" ("Native FP4 Is Slower Than
 * Emulated FP4", section 1).  Reading: an activation is one E4M3 "FN" code
 * times one fp32 per-tensor decode scale S, the same two-level idea as the
 * NVFP4 tensor scale with E4M3's largest value 448 in place of 6 * 448:
 *   S = fp32(amax(|x|)) / 448          (one fp32 division; dynamic scale)
 *   code = sign | E4M3(RNE, satfinite) of |x / S|  (x / S one fp32 division)
 * The sign bit is copied from x / S even when the magnitude rounds to zero
 * (-0.1 * 2^-9 * S encodes as 0x80).  S == 0 gives all codes 0.
 * value = e4m3(code) * S. */
int orc_fp8_encode(float q) {
  int neg = signbit(q) ? 1 : 0;
  return orc_e4m3_encode(fabsf(q)) | (neg << 7);
}

float orc_fp8_tensor_scale(const float* x, int64_t rows, int64_t cols, int64_t ld) {
  float amax = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      float a = f32_abs(x[r * ld + c]);
      if (a > amax) amax = a;
    }
  return amax / 448.0f;
}

/* x [rows, cols] (row stride ld) -> codes [rows, cols] (one byte each).
 * dynamic != 0: S = amax / 448 is computed and written to *S; otherwise *S
 * is read. */
void orc_fp8_quantize(const float* x, int64_t rows, int64_t cols, int64_t ld, int dynamic, float* S,
                      uint8_t* codes) {
  if (dynamic) *S = orc_fp8_tensor_scale(x, rows, cols, ld);
  float s = *S;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      codes[r * cols + c] = (s == 0.0f) ? 0 : (uint8_t)orc_fp8_encode(x[r * ld + c] / s);
}

/* ------------------------------------------------------------------------ */

/* Router logits, the step before routing ("The 2x Gap: Diagnosing Suboptimal
 * FP4 GEMM Kernels on Blackwell SM120", section "The Investigation So Far":
 * each token goes to 8 of 256 experts chosen from these scores):
 *   logits[t, e] = sum_h x[t, h] * w[e, h]
 * x [T, H] and w [E, H] hold bf16 values widened to fp32; the sum is fp64
 * and the result is stored as fp32 (the GPU's storage type). */
void orc_router_logits(const float* x, const float* w, int T, int H, int E, float* logits) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h) acc += (double)x[(int64_t)t * H + h] * (double)w[(int64_t)e * H + h];
      logits[(int64_t)t * E + e] = (float)acc;
    }
}

/* Top-k selection by repeated arg-max (strict >, so ties go to the lower
 * expert id), then softmax over the k selected logits in fp64. */
void orc_route(const float* logits, int T, int E, int k, int32_t* ids, double* w) {
  char* taken = (char*)malloc((size_t)E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;
      }
      taken[best] = 1;
      ids[t * k + j] = best;
    }
    double lmax = (double)l[ids[t * k]];
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += exp((double)l[ids[t * k + j]] - lmax);
    for (int j = 0; j < k; ++j) w[t * k + j] = exp((double)l[ids[t * k + j]] - lmax) / sum;
  }
  free(taken);
}

/* Stable counting sort of the T*k (token, slot) pairs by expert.
 * offsets[E+1] = exclusive prefix sum of per-expert counts; perm[r] = source
 * token of permuted row r; inv[t*k+j] = permuted row of pair (t, j). */
void orc_permute(const int32_t* ids, int T, int E, int k, int32_t* offsets, int32_t* perm, int32_t* inv) {
  int32_t* cursor = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int e = 0; e <= E; ++e) offsets[e] = 0;
  for (int i = 0; i < T * k; ++i) offsets[ids[i] + 1] += 1;
  for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = ids[t * k + j];
      int r = offsets[e] + cursor[e]++;
      perm[r] = t;
      inv[t * k + j] = r;
    }
  free(cursor);
}

/* ------------------------------------------------------------------------ */
/* Grouped GEMM                                                             */
/* ------------------------------------------------------------------------ */

/* W4A4: out[r, n] = S_a * S_w[e(r)] * sum_k dec(a[r,k]) * dec(w[e(r), n, k]),
 * fp64 accumulation.  a: codes [R, K/2], scales [R, K/16]; w: codes
 * [E, N, K/2], scales [E, N, K/16] (linear layout); out fp64 [R, N]. */
void orc_grouped_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales, float S_a,
                           const uint8_t* w_codes, const uint8_t* w_scales, const float* w_S,
                           const int32_t* offsets, int E, int N, int K, double* out) {
  int R = offsets[E];
  double* adq = (double*)malloc(sizeof(double) * (size_t)R * (size_t)K);
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < K; ++c) adq[r * K + c] = dec_elem(a_codes, a_scales, K, r, c);
  for (int e = 0; e < E; ++e) {
    int r0 = offsets[e], r1 = offsets[e + 1];
    if (r1 <= r0) continue;
    const uint8_t* wc = w_codes + (int64_t)e * N * (K / 2);
    const uint8_t* ws = w_scales + (int64_t)e * N * (K / 16);
    double alpha = (double)S_a * (double)w_S[e];
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
      double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
      for (int64_t c = 0; c < K; ++c) wrow[c] = dec_elem(wc, ws, K, n, c);
      for (int r = r0; r < r1; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) acc += adq[(int64_t)r * K + c] * wrow[c];
        out[(int64_t)r * N + n] = acc * alpha;
      }
      free(wrow);
    }
  }
  free(adq);
}

/* W4A16: as above but the activation is the exact BF16 value (given as the
 * fp32 widening of a bf16 number) and only the weight is NVFP4. */
void orc_grouped_gemm_w4a16(const float* a, const uint8_t* w_codes, const uint8_t* w_scales,
                            const float* w_S, const int32_t* offsets, int E, int N, int K, double* out) {
  for (int e = 0; e < E; ++e) {
    int r0 = offsets[e], r1 = offsets[e + 1];
    if (r1 <= r0) continue;
    const uint8_t* wc = w_codes + (int64_t)e * N * (K / 2);
    const uint8_t* ws = w_scales + (int64_t)e * N * (K / 16);
    double alpha = (double)w_S[e];
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
      double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
      for (int64_t c = 0; c < K; ++c) wrow[c] = dec_elem(wc, ws, K, n, c);
      for (int r = r0; r < r1; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) acc += (double)a[(int64_t)r * K + c] * wrow[c];
        out[(int64_t)r * N + n] = acc * alpha;
      }
      free(wrow);
    }
  }
}

/* MXFP4 x MXFP4: out[r, n] = sum_k dec(a[r,k]) * dec(w[e(r), n, k]), fp64
 * accumulation, no per-tensor coefficient.  a: codes [R, K/2], scales
 * [R, K/32]; w: codes [E, N, K/2], scales [E, N, K/32]; out fp64 [R, N]. */
void orc_grouped_gemm_mx(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* w_codes,
                         const uint8_t* w_scales, const int32_t* offsets, int E, int N, int K, double* out) {
  int R = offsets[E];
  double* adq = (double*)malloc(sizeof(double) * (size_t)R * (size_t)K);
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < K; ++c) adq[r * K + c] = dec_elem_mx(a_codes, a_scales, K, r, c);
  for (int e = 0; e < E; ++e) {
    int r0 = offsets[e], r1 = offsets[e + 1];
    if (r1 <= r0) continue;
    const uint8_t* wc = w_codes + (int64_t)e * N * (K / 2);
    const uint8_t* ws = w_scales + (int64_t)e * N * (K / 32);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
      double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
      for (int64_t c = 0; c < K; ++c) wrow[c] = dec_elem_mx(wc, ws, K, n, c);
      for (int r = r0; r < r1; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) acc += adq[(int64_t)r * K + c] * wrow[c];
        out[(int64_t)r * N + n] = acc;
      }
      free(wrow);
    }
  }
  free(adq);
}

/* W4A8: out[r, n] = S_a * S_w[e(r)] * sum_k e4m3(a[r,k]) * dec(w[e(r), n, k]),
 * fp64 accumulation.  a: FP8 codes [R, K]; w as for W4A4; out fp64 [R, N]. */
void orc_grouped_gemm_w4a8(const uint8_t* a_codes, float S_a, const uint8_t* w_codes, const uint8_t* w_scales,
                           const float* w_S, const int32_t* offsets, int E, int N, int K, double* out) {
  int R = offsets[E];
  double* adq = (double*)malloc(sizeof(double) * (size_t)R * (size_t)K);
  for (int64_t i = 0; i < (int64_t)R * K; ++i) adq[i] = orc_e4m3_value(a_codes[i]);
  for (int e = 0; e < E; ++e) {
    int r0 = offsets[e], r1 = offsets[e + 1];
    if (r1 <= r0) continue;
    const uint8_t* wc = w_codes + (int64_t)e * N * (K / 2);
    const uint8_t* ws = w_scales + (int64_t)e * N * (K / 16);
    double alpha = (double)S_a * (double)w_S[e];
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
      double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
      for (int64_t c = 0; c < K; ++c) wrow[c] = dec_elem(wc, ws, K, n, c);
      for (int r = r0; r < r1; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) acc += adq[(int64_t)r * K + c] * wrow[c];
        out[(int64_t)r * N + n] = acc * alpha;
      }
      free(wrow);
    }
  }
  free(adq);
}

/* ------------------------------------------------------------------------ */
/* SwiGLU, requantisation, combine                                          */
/* ------------------------------------------------------------------------ */

/* h[r, i] = silu(g) * u with g = G[r, i], u = G[r, I + i], silu(x) = x/(1+e^-x),
 * evaluated in fp64 from the stored fp32 G. */
void orc_swiglu(const float* G, int64_t R, int64_t I, double* h) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t i = 0; i < I; ++i) {
      double g = (double)G[r * 2 * I + i];
      double u = (double)G[r * 2 * I + I + i];
      h[r * I + i] = g / (1.0 + exp(-g)) * u;
    }
}

/* Combine: out[t, n] = sum_j w[t, j] * Y[inv[t, j], n] (fp64 sum). */
void orc_combine(const float* Y, const int32_t* inv, const double* w, int T, int k, int64_t H, double* out) {
  for (int t = 0; t < T; ++t)
    for (int64_t n = 0; n < H; ++n) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += w[t * k + j] * (double)Y[(int64_t)inv[t * k + j] * H + n];
      out[(int64_t)t * H + n] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* Full MoE layer, two independent restatements                             */
/* ------------------------------------------------------------------------ */

/* One layer forward, step by step as the path defines it:
 *   route -> permute -> (W4A4: quantise x, dynamic S) -> gather ->
 *   gate_up grouped GEMM (G stored fp32) -> SwiGLU (h stored fp32) ->
 *   (W4A4: requantise h with the static S_h | W4A16: round h to bf16) ->
 *   down grouped GEMM (Y stored fp32) -> weighted combine (out fp64).
 * mode 0 = W4A4, 1 = W4A16, 2 = MXFP4 weights and activations (x quantised
 * and h requantised per 32-element block with UE8M0 scales; the per-tensor
 * scales w13_S, w2_S, S_h and S_x do not exist in this format and are not
 * read; hq_scales_o then holds R * I/32 bytes), 3 = W4A8 (NVFP4 weights; x
 * quantised to FP8 E4M3 with the dynamic per-tensor scale, h requantised to
 * FP8 with the static decode scale S_h; hq_codes_o then holds R * I bytes,
 * hq_scales_o is not written).
 * x is [T, H] (bf16 values widened to fp32).
 * S_x_in: NULL = the dynamic per-tensor scale of these T rows; otherwise the
 * scale of a larger tensor these rows were taken from (to check a sample of
 * tokens of a big batch, the scale must be the whole batch's).
 * Optional intermediate outputs may be NULL. */
void orc_moe_layer(int mode, const float* x, const float* logits, int T, int H, int I, int E, int k,
                   const uint8_t* w13_codes, const uint8_t* w13_scales, const float* w13_S,
                   const uint8_t* w2_codes, const uint8_t* w2_scales, const float* w2_S, float S_h,
                   const float* S_x_in, double* out, int32_t* ids_o, double* w_o, int32_t* offsets_o, int32_t* perm_o,
                   int32_t* inv_o, float* S_x_o, uint8_t* hq_codes_o, uint8_t* hq_scales_o, float* h32_o) {
  int R = T * k;
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
  double* w = (double*)malloc(sizeof(double) * (size_t)R);
  int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
  int32_t* inv = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
  double* G64 = (double*)malloc(sizeof(double) * (size_t)R * 2 * I);
  float* G32 = (float*)malloc(sizeof(float) * (size_t)R * 2 * I);
  double* h64 = (double*)malloc(sizeof(double) * (size_t)R * I);
  float* h32 = (float*)malloc(sizeof(float) * (size_t)R * I);
  double* Y64 = (double*)malloc(sizeof(double) * (size_t)R * H);
  float* Y32 = (float*)malloc(sizeof(float) * (size_t)R * H);
  float S_x = 0.0f;

  orc_route(logits, T, E, k, ids, w);
  orc_permute(ids, T, E, k, offsets, perm, inv);

  if (mode == 3) {
    uint8_t* xc = (uint8_t*)malloc((size_t)T * H);
    uint8_t* ac = (uint8_t*)malloc((size_t)R * H);
    if (S_x_in) S_x = *S_x_in;
    orc_fp8_quantize(x, T, H, H, S_x_in ? 0 : 1, &S_x, xc);
    for (int r = 0; r < R; ++r) memcpy(ac + (int64_t)r * H, xc + (int64_t)perm[r] * H, (size_t)H);
    orc_grouped_gemm_w4a8(ac, S_x, w13_codes, w13_scales, w13_S, offsets, E, 2 * I, H, G64);
    free(xc); free(ac);
  } else if (mode == 2) {
    uint8_t* xc = (uint8_t*)malloc((size_t)T * H / 2);
    uint8_t* xs = (uint8_t*)malloc((size_t)T * H / 32);
    uint8_t* ac = (uint8_t*)malloc((size_t)R * H / 2);
    uint8_t* as = (uint8_t*)malloc((size_t)R * H / 32);
    orc_mx_quantize(x, T, H, H, xc, xs);
    for (int r = 0; r < R; ++r) {
      memcpy(ac + (int64_t)r * H / 2, xc + (int64_t)perm[r] * H / 2, (size_t)H / 2);
      memcpy(as + (int64_t)r * H / 32, xs + (int64_t)perm[r] * H / 32, (size_t)H / 32);
    }
    orc_grouped_gemm_mx(ac, as, w13_codes, w13_scales, offsets, E, 2 * I, H, G64);
    free(xc); free(xs); free(ac); free(as);
  } else if (mode == 0) {
    uint8_t* xc = (uint8_t*)malloc((size_t)T * H / 2);
    uint8_t* xs = (uint8_t*)malloc((size_t)T * H / 16);
    uint8_t* ac = (uint8_t*)malloc((size_t)R * H / 2);
    uint8_t* as = (uint8_t*)malloc((size_t)R * H / 16);
    if (S_x_in) S_x = *S_x_in;
    orc_quantize(x, T, H, H, S_x_in ? 0 : 1, &S_x, xc, xs);
    for (int r = 0; r < R; ++r) {
      memcpy(ac + (int64_t)r * H / 2, xc + (int64_t)perm[r] * H / 2, (size_t)H / 2);
      memcpy(as + (int64_t)r * H / 16, xs + (int64_t)perm[r] * H / 16, (size_t)H / 16);
    }
    orc_grouped_gemm_w4a4(ac, as, S_x, w13_codes, w13_scales, w13_S, offsets, E, 2 * I, H, G64);
    free(xc); free(xs); free(ac); free(as);
  } else {
    float* ax = (float*)malloc(sizeof(float) * (size_t)R * H);
    for (int r = 0; r < R; ++r) memcpy(ax + (int64_t)r * H, x + (int64_t)perm[r] * H, sizeof(float) * (size_t)H);
    orc_grouped_gemm_w4a16(ax, w13_codes, w13_scales, w13_S, offsets, E, 2 * I, H, G64);
    free(ax);
  }
  for (int64_t i = 0; i < (int64_t)R * 2 * I; ++i) G32[i] = (float)G64[i];
  orc_swiglu(G32, R, I, h64);
  for (int64_t i = 0; i < (int64_t)R * I; ++i) h32[i] = (float)h64[i];

  if (mode == 3) {
    uint8_t* hc = (uint8_t*)malloc((size_t)R * I);
    float sh = S_h;
    orc_fp8_quantize(h32, R, I, I, 0, &sh, hc);
    orc_grouped_gemm_w4a8(hc, sh, w2_codes, w2_scales, w2_S, offsets, E, H, I, Y64);
    if (hq_codes_o) memcpy(hq_codes_o, hc, (size_t)R * I);
    free(hc);
  } else if (mode == 2) {
    uint8_t* hc = (uint8_t*)malloc((size_t)R * I / 2);
    uint8_t* hs = (uint8_t*)malloc((size_t)R * I / 32);
    orc_mx_quantize(h32, R, I, I, hc, hs);
    orc_grouped_gemm_mx(hc, hs, w2_codes, w2_scales, offsets, E, H, I, Y64);
    if (hq_codes_o) memcpy(hq_codes_o, hc, (size_t)R * I / 2);
    if (hq_scales_o) memcpy(hq_scales_o, hs, (size_t)R * I / 32);
    free(hc); free(hs);
  } else if (mode == 0) {
    uint8_t* hc = (uint8_t*)malloc((size_t)R * I / 2);
    uint8_t* hs = (uint8_t*)malloc((size_t)R * I / 16);
    float sh = S_h;
    orc_quantize(h32, R, I, I, 0, &sh, hc, hs);
    orc_grouped_gemm_w4a4(hc, hs, sh, w2_codes, w2_scales, w2_S, offsets, E, H, I, Y64);
    if (hq_codes_o) memcpy(hq_codes_o, hc, (size_t)R * I / 2);
    if (hq_scales_o) memcpy(hq_scales_o, hs, (size_t)R * I / 16);
    free(hc); free(hs);
  } else {
    float* hb = (float*)malloc(sizeof(float) * (size_t)R * I);
    for (int64_t i = 0; i < (int64_t)R * I; ++i) hb[i] = orc_round_bf16(h32[i]);
    orc_grouped_gemm_w4a16(hb, w2_codes, w2_scales, w2_S, offsets, E, H, I, Y64);
    free(hb);
  }
  for (int64_t i = 0; i < (int64_t)R * H; ++i) Y32[i] = (float)Y64[i];
  orc_combine(Y32, inv, w, T, k, H, out);

  if (ids_o) memcpy(ids_o, ids, sizeof(int32_t) * (size_t)R);
  if (w_o) memcpy(w_o, w, sizeof(double) * (size_t)R);
  if (offsets_o) memcpy(offsets_o, offsets, sizeof(int32_t) * (size_t)(E + 1));
  if (perm_o) memcpy(perm_o, perm, sizeof(int32_t) * (size_t)R);
  if (inv_o) memcpy(inv_o, inv, sizeof(int32_t) * (size_t)R);
  if (S_x_o) *S_x_o = S_x;
  if (h32_o) memcpy(h32_o, h32, sizeof(float) * (size_t)R * I);
  free(ids); free(w); free(offsets); free(perm); free(inv);
  free(G64); free(G32); free(h64); free(h32); free(Y64); free(Y32);
}

/* Second restatement used only to pin the first: no permutation, no grouped
 * GEMM, no gather.  For each token and each of its k experts, dequantise the
 * token row and the expert's weight rows, run the dense fp64 loops, and add
 * the weighted result.  Same storage roundings as orc_moe_layer. */
void orc_moe_layer_naive(int mode, const float* x, const float* logits, int T, int H, int I, int E, int k,
                         const uint8_t* w13_codes, const uint8_t* w13_scales, const float* w13_S,
                         const uint8_t* w2_codes, const uint8_t* w2_scales, const float* w2_S, float S_h,
                         const float* S_x_in, double* out) {
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
  orc_route(logits, T, E, k, ids, w);
  double* xd = (double*)malloc(sizeof(double) * (size_t)T * H);
  if (mode == 3) {
    uint8_t* xc = (uint8_t*)malloc((size_t)T * H);
    float S_x = S_x_in ? *S_x_in : 0.0f;
    orc_fp8_quantize(x, T, H, H, S_x_in ? 0 : 1, &S_x, xc);
    for (int64_t i = 0; i < (int64_t)T * H; ++i) xd[i] = orc_e4m3_value(xc[i]) * (double)S_x;
    free(xc);
  } else if (mode == 2) {
    uint8_t* xc = (uint8_t*)malloc((size_t)T * H / 2);
    uint8_t* xs = (uint8_t*)malloc((size_t)T * H / 32);
    orc_mx_quantize(x, T, H, H, xc, xs);
    orc_mx_dequantize(xc, xs, T, H, xd);
    free(xc); free(xs);
  } else if (mode == 0) {
    uint8_t* xc = (uint8_t*)malloc((size_t)T * H / 2);
    uint8_t* xs = (uint8_t*)malloc((size_t)T * H / 16);
    float S_x = S_x_in ? *S_x_in : 0.0f;
    orc_quantize(x, T, H, H, S_x_in ? 0 : 1, &S_x, xc, xs);
    orc_dequantize(xc, xs, S_x, T, H, xd);
    free(xc); free(xs);
  } else {
    for (int64_t i = 0; i < (int64_t)T * H; ++i) xd[i] = (double)x[i];
  }
  for (int64_t i = 0; i < (int64_t)T * H; ++i) out[i] = 0.0;
#pragma omp parallel for schedule(dynamic)
  for (int t = 0; t < T; ++t) {
    float* h32 = (float*)malloc(sizeof(float) * (size_t)I);
    double* hd = (double*)malloc(sizeof(double) * (size_t)I);
    for (int j = 0; j < k; ++j) {
      int e = ids[t * k + j];
      const int mx = mode == 2;
      const int sb = mx ? 32 : 16; /* elements per block scale */
      const uint8_t* c13 = w13_codes + (int64_t)e * 2 * I * (H / 2);
      const uint8_t* s13 = w13_scales + (int64_t)e * 2 * I * (H / sb);
      const uint8_t* c2 = w2_codes + (int64_t)e * H * (I / 2);
      const uint8_t* s2 = w2_scales + (int64_t)e * H * (I / sb);
      const double S13 = mx ? 1.0 : (double)w13_S[e];
      const double S2 = mx ? 1.0 : (double)w2_S[e];
      for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
          const double wg = mx ? dec_elem_mx(c13, s13, H, i, c) : dec_elem(c13, s13, H, i, c);
          const double wu = mx ? dec_elem_mx(c13, s13, H, I + i, c) : dec_elem(c13, s13, H, I + i, c);
          g += xd[(int64_t)t * H + c] * wg * S13;
          u += xd[(int64_t)t * H + c] * wu * S13;
        }
        float g32 = (float)g, u32 = (float)u;
        double hv = (double)g32 / (1.0 + exp(-(double)g32)) * (double)u32;
        h32[i] = (float)hv;
      }
      if (mx) {
        uint8_t hsc;
        uint8_t ec[32];
        for (int b = 0; b < I / 32; ++b) {
          orc_mx_quantize_block(h32 + b * 32, &hsc, ec);
          for (int q = 0; q < 32; ++q) hd[b * 32 + q] = orc_e2m1_value(ec[q]) * orc_ue8m0_value(hsc);
        }
      } else if (mode == 3) {
        for (int i = 0; i < I; ++i)
          hd[i] = S_h == 0.0f ? 0.0 : orc_e4m3_value(orc_fp8_encode(h32[i] / S_h)) * (double)S_h;
      } else if (mode == 0) {
        uint8_t hsc;
        uint8_t ec[16];
        for (int b = 0; b < I / 16; ++b) {
          orc_quantize_block(h32 + b * 16, S_h, &hsc, ec);
          for (int q = 0; q < 16; ++q)
            hd[b * 16 + q] = orc_e2m1_value(ec[q]) * orc_e4m3_value(hsc) * (double)S_h;
        }
      } else {
        for (int i = 0; i < I; ++i) hd[i] = (double)orc_round_bf16(h32[i]);
      }
      for (int n = 0; n < H; ++n) {
        double y = 0.0;
        for (int i = 0; i < I; ++i) y += hd[i] * (mx ? dec_elem_mx(c2, s2, I, n, i) : dec_elem(c2, s2, I, n, i)) * S2;
        float y32 = (float)y;
        out[(int64_t)t * H + n] += w[t * k + j] * (double)y32;
      }
    }
    free(h32);
    free(hd);
  }
  free(ids); free(w); free(xd);
}

/* Threads the oracle runs with (OpenMP), for reporting. */
int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
