/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for NVFP4 block quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or constant with the
 * CUDA library; it is written from the method's definitions, step by step.
 *
 * Citation keys used below (page title, then the part of the page):
 *   [FOS-01]  "SOAR 周冠军笔记 07 | 香草小张：NVFP4 量化改进与推测解码实践"
 *             (openbmb.cn blog), section "01 问题背景": the FP4 E2M1 value set
 *             {0, ±0.5, ±1, ±1.5, ±2, ±3, ±4, ±6}, largest magnitude 6.
 *   [FOS-02]  same page, section "02 FourOverSix": scale_m4 = fp8(scale_m6*1.5);
 *             the dequant MSE of both candidates; keep m4 iff mse_m4 < mse_m6.
 *   [SOAR-Q]  "SOAR: Scale Optimization for Accurate Reconstruction in NVFP4
 *             Quantization" (july-h5kf3.github.io notes), the NVFP4 quantizer
 *             display equation: alpha = max|X| / (M_FP4 * M_FP8) with
 *             M_FP4 = 6, M_FP8 = 448; Delta_i = Q_E4M3(max|X_i| / (alpha*6));
 *             the piecewise FP4 rounding of X / (alpha*Delta).
 *   [SOAR-DQ] same page, dequantization equation: Xhat * (alpha*Delta).
 *   [SOAR-OBJ] same page, CJSO objective: min sum_i ||W_i - Q_i alpha Delta_i||^2.
 *   [SOAR-A]  same page, closed form for the global scale alpha*.
 *   [SOAR-D]  same page, closed form for each block scale Delta_i*.
 *   [SOAR-SCHED] same page, CJSO schedule paragraph: start from the max rule,
 *             update alpha and Delta_i by the closed forms, re-quantize Q
 *             after every update.
 *   [SOAR-DEC] same page, decoupled objective (Delta^q in R, Delta^d in FP8)
 *             and its search: Delta^d from CJSO, Delta^q = Delta^d at start;
 *             Delta^q scaled by [0.5, 1.5] in steps of 0.01; Delta^d limited to
 *             the two nearest E4M3 values; keep the pair of least error.
 *
 * Readings taken where the pages are silent:
 *   R1  block = 16 consecutive elements of one row (row-major [rows, cols]).
 *   R2  E2M1 rounding ties go to the even code (round-half-even inside each
 *       piece of the [SOAR-Q] formula); magnitudes above 6 saturate to 6; the
 *       sign bit of a code is the sign bit of the input element.
 *   R3  E4M3 is the OCP E4M3FN format (bias 7, subnormals, max 448, no inf);
 *       rounding is nearest-even and saturates at 448.
 *   R4  fp32 evaluation of the quantizer, one rounding per written operation:
 *       s = fl(alpha*Delta), v = fl(|x| / s) (IEEE division);
 *       Delta_i = e4m3(fl(amax_i / fl(alpha*6))); alpha = fl(amax / 2688).
 *   R5  per-block sums P = sum |x| q and R = sum q^2 are the exact sums rounded
 *       once to fp32 (for in-range inputs they are exact in fp32).
 *   R6  the MSE comparisons of [FOS-02] and [SOAR-DEC] drop the common term
 *       sum x^2 and the 1/16: err - sum x^2 = s*(s*R - 2P), evaluated as
 *       g = fl(s * fma(s, R, -2P)) in fp32.
 *   R7  a block whose dequant scale fl(alpha*Delta) is zero has all code
 *       magnitudes 0 (and P = R = 0).
 *   R8  CJSO: alpha* = sum_i Delta_i P_i / sum_i Delta_i^2 R_i (the printed
 *       form has alpha where Delta_i belongs), both sums exact (128-bit fixed
 *       point), each rounded once to double, the quotient taken in double and
 *       rounded to fp32; Delta_i* = e4m3(fl(P_i / fl(alpha R_i))),
 *       Delta_i kept when R_i = 0; one iteration = alpha step, re-quantize,
 *       Delta step, re-quantize; T = 0 is the max rule.
 *   R9  decoupled: m_k = fl32((50+k)/100), k = 0..100; Delta^q = fl(Delta^d0*m_k);
 *       the two Delta^d candidates are the largest E4M3 value <= Delta^q and
 *       the smallest E4M3 value >= Delta^q (448 when Delta^q > 448); the first
 *       strict minimum of g in the order (k ascending, lower before upper)
 *       wins; alpha is not refitted after the search.
 *   R10 dequantized output is bf16_rne(fl(q * fl(alpha*Delta))).
 *   R12 the W4A16 product (the consumer of the codes) multiplies the R10
 *       bf16 weights by bf16 activations; the oracle sums in double.
 *   R13 the tensor-core scale layout (tiles of 128 x 4 scales, 32 x 16
 *       interleave inside a tile) is the one block-scaled matrix multiplies
 *       read; the pages give none.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC ... -lm -lpthread
 * (-ffp-contract=off: every float operation written here is rounded once,
 * no silent fusing; fmaf() is written out where a fused operation is meant).
 */
#include <fenv.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define BLOCK 16

enum { MODE_MAX = 0, MODE_FOUR_OVER_SIX = 1, MODE_CJSO = 2, MODE_CJSO_DECOUPLED = 3 };

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* [FOS-01] the eight E2M1 magnitudes, indexed by the 3 low bits of a code. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static double rne(double t) { return nearbyint(t); } /* FE_TONEAREST: ties to even */

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static int f32_signbit(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (int)(u >> 31);
}

/* [SOAR-Q] piecewise FP4 rounding, reading R2: a >= 0 -> magnitude code 0..7.
 *   |x| < 2      : (1/2) * round(2x)
 *   2 <= |x| <= 4: round(x)
 *   4 <= |x| <= 6: 2 * round(x/2)       (above 6: saturate to 6)          */
static int e2m1_mag_code(double a) {
  double q;
  if (isnan(a)) return 0;
  if (a < 2.0)
    q = 0.5 * rne(2.0 * a);
  else if (a <= 4.0)
    q = rne(a);
  else
    q = 2.0 * rne(0.5 * a);
  if (q > 6.0) q = 6.0;
  for (int c = 0; c < 8; ++c)
    if (E2M1_MAG[c] == q) return c;
  return 0; /* unreachable: q is always on the grid */
}

/* Reading R3: value of an E4M3FN code (bias 7; exponent field 0 = subnormal). */
static double e4m3_value(int code) {
  int sgn = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return sgn ? -v : v;
}

/* Reading R3: nearest-even E4M3FN code of r >= 0, saturating at 448 (0x7E). */
static int e4m3_code(double r) {
  if (!(r > 0.0)) return 0;
  if (r >= 448.0) return 0x7E;
  if (r < 0x1p-6) return (int)rne(r * 512.0); /* subnormal step 2^-9; 8 -> 2^-6 */
  int e = ilogb(r);                           /* r in [2^e, 2^(e+1)) */
  double t = rne(ldexp(r, 3 - e));            /* 8..16; 16 carries into e */
  int code = ((e + 7) << 3) + (int)(t - 8.0);
  return code > 0x7E ? 0x7E : code;
}

/* Largest E4M3 code (0..0x7E) whose value is <= r (r >= 0). Binary search
 * over the positive codes, whose values increase with the code. */
static int e4m3_floor_code(double r) {
  int lo = 0, hi = 0x7E;
  if (e4m3_value(hi) <= r) return hi;
  while (hi - lo > 1) { /* value(lo) <= r < value(hi) */
    int mid = (lo + hi) / 2;
    if (e4m3_value(mid) <= r) lo = mid; else hi = mid;
  }
  return lo;
}

/* Smallest E4M3 code whose value is >= r; 0x7E (448) when r > 448. */
static int e4m3_ceil_code(double r) {
  int lo = 0, hi = 0x7E;
  if (r <= 0.0) return 0;
  if (r > e4m3_value(hi)) return hi;
  while (hi - lo > 1) { /* value(lo) < r <= value(hi) */
    int mid = (lo + hi) / 2;
    if (e4m3_value(mid) < r) lo = mid; else hi = mid;
  }
  return hi;
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs). */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* One block                                                           */
/* ------------------------------------------------------------------ */

/* [SOAR-Q] Q_i = Q_fp4(W_i / (alpha*Delta)) under readings R4, R5, R7.
 * Writes 16 magnitude codes; P = sum |x| q, R = sum q^2. */
static void quant_block(const float *x, float alpha, float delta, uint8_t *mag,
                        float *P, float *R) {
  float s = alpha * delta;
  double p = 0.0, rr = 0.0;
  if (s == 0.0f) {
    memset(mag, 0, BLOCK);
    *P = 0.0f;
    *R = 0.0f;
    return;
  }
  for (int j = 0; j < BLOCK; ++j) {
    float v = fabsf(x[j]) / s;
    int c = e2m1_mag_code((double)v);
    double q = E2M1_MAG[c];
    mag[j] = (uint8_t)c;
    p += fabs((double)x[j]) * q;
    rr += q * q;
  }
  *P = (float)p;
  *R = (float)rr;
}

/* Reading R6: error of a candidate minus the common sum x^2. */
static float cand_err(float s, float P, float R) { return s * fmaf(s, R, -2.0f * P); }

static void load_block(const uint16_t *w, int64_t b, float *x) {
  for (int j = 0; j < BLOCK; ++j) x[j] = bf16_to_f32(w[b * BLOCK + j]);
}

static float block_amax(const float *x) {
  float m = 0.0f;
  for (int j = 0; j < BLOCK; ++j) m = fmaxf(m, fabsf(x[j]));
  return m;
}

/* Codes with sign (reading R2), two per byte, even element in the low nibble. */
static void pack_codes(const float *x, const uint8_t *mag, uint8_t *out8) {
  for (int j = 0; j < BLOCK; j += 2) {
    int lo = mag[j] | (f32_signbit(x[j]) << 3);
    int hi = mag[j + 1] | (f32_signbit(x[j + 1]) << 3);
    out8[j / 2] = (uint8_t)(lo | (hi << 4));
  }
}

/* ------------------------------------------------------------------ */
/* Tensor-level state and passes                                       */
/* ------------------------------------------------------------------ */

typedef struct {
  const uint16_t *w;
  int64_t nblocks;
  float alpha;
  float six_alpha;  /* fl(alpha*6), reading R4 */
  uint8_t *dcode;   /* per block E4M3 code */
  float *P, *R;     /* per block sums */
  uint8_t *m4;      /* FourOverSix: 1 if the M=4 scale was kept (may be NULL) */
  uint8_t *codes;   /* packed output, nblocks*8 (may be NULL) */
  const int64_t *sample; /* decoupled: blocks to search (NULL = all) */
  int64_t nsample;
  uint8_t *out_codes;    /* decoupled output, per sample */
  uint8_t *out_scales;
  int phase;
  int write_codes;
} ctx_t;

typedef struct {
  ctx_t *c;
  int64_t b0, b1;
} job_t;

enum { PH_MAX = 0, PH_FOS, PH_CJSO_ITER, PH_DECOUPLED };

/* [SOAR-Q] max rule for one block: Delta_i = e4m3(amax_i / (alpha*6)). */
static int max_rule_code(const ctx_t *c, const float *x) {
  if (c->alpha == 0.0f) return 0;
  return e4m3_code((double)(block_amax(x) / c->six_alpha));
}

static void do_block_max(ctx_t *c, int64_t b, uint8_t *out8) {
  float x[BLOCK];
  uint8_t mag[BLOCK];
  load_block(c->w, b, x);
  int d = max_rule_code(c, x);
  quant_block(x, c->alpha, (float)e4m3_value(d), mag, &c->P[b], &c->R[b]);
  c->dcode[b] = (uint8_t)d;
  if (out8) pack_codes(x, mag, out8);
}

/* [FOS-02] FourOverSix: Delta4 = e4m3(1.5*Delta6); keep Delta4 iff its dequant
 * error is strictly smaller (reading R6 for the error). */
static void do_block_fos(ctx_t *c, int64_t b, uint8_t *out8) {
  float x[BLOCK];
  uint8_t mag6[BLOCK], mag4[BLOCK];
  float P6, R6, P4, R4;
  load_block(c->w, b, x);
  int d6 = max_rule_code(c, x);
  float delta6 = (float)e4m3_value(d6);
  int d4 = e4m3_code((double)(delta6 * 1.5f));
  float delta4 = (float)e4m3_value(d4);
  quant_block(x, c->alpha, delta6, mag6, &P6, &R6);
  quant_block(x, c->alpha, delta4, mag4, &P4, &R4);
  float g6 = cand_err(c->alpha * delta6, P6, R6);
  float g4 = cand_err(c->alpha * delta4, P4, R4);
  int use4 = g4 < g6;
  c->dcode[b] = (uint8_t)(use4 ? d4 : d6);
  c->P[b] = use4 ? P4 : P6;
  c->R[b] = use4 ? R4 : R6;
  if (c->m4) c->m4[b] = (uint8_t)use4;
  if (out8) pack_codes(x, use4 ? mag4 : mag6, out8);
}

/* [SOAR-D] + [SOAR-SCHED], reading R8: with alpha fixed, re-quantize with the
 * current Delta_i, take the closed-form Delta_i*, round it to E4M3 and
 * re-quantize again. */
static void do_block_cjso(ctx_t *c, int64_t b, uint8_t *out8) {
  float x[BLOCK];
  uint8_t mag[BLOCK];
  float P, R;
  load_block(c->w, b, x);
  int d = c->dcode[b];
  quant_block(x, c->alpha, (float)e4m3_value(d), mag, &P, &R);
  if (R > 0.0f) {
    float t = P / (c->alpha * R);
    d = e4m3_code((double)t);
  }
  quant_block(x, c->alpha, (float)e4m3_value(d), mag, &c->P[b], &c->R[b]);
  c->dcode[b] = (uint8_t)d;
  if (out8) pack_codes(x, mag, out8);
}

/* [SOAR-DEC], reading R9: 101 quantization scales x 2 stored scales. */
static void do_block_decoupled(ctx_t *c, int64_t si) {
  int64_t b = c->sample ? c->sample[si] : si;
  float x[BLOCK];
  uint8_t mag[BLOCK], best_mag[BLOCK];
  float P, R;
  load_block(c->w, b, x);
  int d0 = c->dcode[b];
  float delta0 = (float)e4m3_value(d0);
  int best_d = d0;
  memset(best_mag, 0, BLOCK);
  if (c->alpha * delta0 != 0.0f) {
    float best_g = INFINITY;
    for (int k = 0; k <= 100; ++k) {
      float m = (float)((50 + k) / 100.0);
      float dq = delta0 * m;
      quant_block(x, c->alpha, dq, mag, &P, &R);
      int cand[2] = {e4m3_floor_code((double)dq), e4m3_ceil_code((double)dq)};
      for (int h = 0; h < 2; ++h) {
        float sd = c->alpha * (float)e4m3_value(cand[h]);
        float g = cand_err(sd, P, R);
        if (g < best_g) {
          best_g = g;
          best_d = cand[h];
          memcpy(best_mag, mag, BLOCK);
        }
      }
    }
  }
  pack_codes(x, best_mag, c->out_codes + si * 8);
  c->out_scales[si] = (uint8_t)best_d;
}

static void *run_job(void *arg) {
  job_t *j = (job_t *)arg;
  ctx_t *c = j->c;
  for (int64_t b = j->b0; b < j->b1; ++b) {
    uint8_t *out8 = c->write_codes ? c->codes + b * 8 : NULL;
    switch (c->phase) {
      case PH_MAX: do_block_max(c, b, out8); break;
      case PH_FOS: do_block_fos(c, b, out8); break;
      case PH_CJSO_ITER: do_block_cjso(c, b, out8); break;
      default: do_block_decoupled(c, b); break;
    }
  }
  return NULL;
}

/* Runs one pass over n items on nthreads threads (contiguous ranges). The
 * per-item work is independent, so the result does not depend on nthreads. */
static void run_pass(ctx_t *c, int phase, int64_t n, int nthreads) {
  c->phase = phase;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n) nthreads = n > 0 ? (int)n : 1;
  job_t jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].c = c;
    jobs[t].b0 = n * t / nthreads;
    jobs[t].b1 = n * (t + 1) / nthreads;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, run_job, &jobs[t]);
  run_job(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* [SOAR-Q] alpha = max|X| / (6*448). */
static float tensor_alpha(const uint16_t *w, int64_t n) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(bf16_to_f32(w[i])));
  return amax / 2688.0f;
}

static void set_alpha(ctx_t *c, float alpha) {
  c->alpha = alpha;
  c->six_alpha = alpha * 6.0f;
}

/* A nonnegative 128-bit integer -> the nearest double (ties to even). */
static double u128_to_double(unsigned __int128 v) {
  int h = 127;
  if (v == 0) return 0.0;
  while (!((v >> h) & 1)) --h; /* the highest set bit */
  if (h < 53) return (double)(uint64_t)v;
  int drop = h - 52; /* bits below a 53-bit significand */
  unsigned __int128 top = v >> drop;
  unsigned __int128 rem = v - (top << drop);
  unsigned __int128 half = (unsigned __int128)1 << (drop - 1);
  if (rem > half || (rem == half && (top & 1))) top += 1; /* may become 2^53: still exact */
  return ldexp((double)(uint64_t)top, drop);
}

/* [SOAR-A], reading R8: alpha* = sum_i Delta_i P_i / sum_i Delta_i^2 R_i from the
 * current Delta_i, P_i, R_i.  Both sums are formed exactly (so the order of the
 * blocks does not matter), as nonnegative 128-bit integers:
 *   Delta_i^2 R_i = M^2 R4 * 2^-20 exactly, with Delta_i = M * 2^-9 and R_i = R4 / 4;
 *   Delta_i P_i = M mP * 2^(e - 33), with P_i = mP * 2^(e - 24) (mP < 2^24),
 *   counted in units of 2^U, U = (biased exponent of the alpha the P_i were
 *   computed with) - 127 - 48; a term's bits below 2^U would be dropped (for
 *   inputs in range there are none: every P_i is a multiple of about
 *   2^(exponent of alpha - 33)).
 * Each sum is rounded once to double, the quotient is taken in double and
 * rounded to fp32.  Returns alpha_old if the denominator is 0. */
static float alpha_step(const ctx_t *c, float alpha_old) {
  uint32_t abits;
  memcpy(&abits, &alpha_old, 4);
  const int U = (int)((abits >> 23) & 0xFFu) - 127 - 48;
  unsigned __int128 num = 0, den = 0;
  for (int64_t b = 0; b < c->nblocks; ++b) {
    const uint64_t M = (uint64_t)ldexp(e4m3_value(c->dcode[b]), 9); /* Delta = M * 2^-9, exactly */
    const uint64_t R4 = (uint64_t)(c->R[b] * 4.0f);                  /* R = R4 / 4, exactly */
    den += (unsigned __int128)(M * M) * R4;
    if (c->P[b] > 0.0f && M > 0) {
      int e;
      const float f = frexpf(c->P[b], &e); /* P = f 2^e, f in [0.5, 1) */
      const uint64_t mP = (uint64_t)ldexpf(f, 24);
      const unsigned __int128 t = (unsigned __int128)(M * mP);
      const int sh = e - 33 - U;
      num += sh >= 0 ? t << sh : t >> -sh;
    }
  }
  if (den == 0) return alpha_old;
  const double nd = ldexp(u128_to_double(num), U);
  const double dd = ldexp(u128_to_double(den), -20);
  return (float)(nd / dd);
}

static int check_args(const uint16_t *w, int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0 || cols % BLOCK != 0) return 1;
  if (rows * cols > 0 && !w) return 1;
  return 0;
}

/* Full quantization. codes: rows*cols/2 bytes; scales: rows*cols/16 bytes.
 * m4_flags (optional, FourOverSix): 1 per block where the M=4 scale was kept.
 * Returns 0 on success, 1 on invalid arguments, 2 if out of memory. */
int oracle_quantize(const uint16_t *w, int64_t rows, int64_t cols, int mode, int iters,
                    uint8_t *codes, uint8_t *scales, float *alpha_out, uint8_t *m4_flags,
                    int nthreads) {
  if (check_args(w, rows, cols) || mode < 0 || mode > 3 || !alpha_out) return 1;
  if ((mode == MODE_CJSO || mode == MODE_CJSO_DECOUPLED) && (iters < 0 || iters > 64)) return 1;
  if (fegetround() != FE_TONEAREST) return 1;
  int64_t n = rows * cols, nb = n / BLOCK;
  ctx_t c;
  memset(&c, 0, sizeof c);
  c.w = w;
  c.nblocks = nb;
  c.dcode = (uint8_t *)malloc(nb > 0 ? (size_t)nb : 1);
  c.P = (float *)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
  c.R = (float *)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
  if (!c.dcode || !c.P || !c.R) {
    free(c.dcode); free(c.P); free(c.R);
    return 2;
  }
  set_alpha(&c, tensor_alpha(w, n));
  c.codes = codes;
  c.m4 = m4_flags;
  int T = (mode == MODE_CJSO || mode == MODE_CJSO_DECOUPLED) ? iters : 0;
  int rc = 0;
  if (mode == MODE_FOUR_OVER_SIX) {
    c.write_codes = 1;
    run_pass(&c, PH_FOS, nb, nthreads);
  } else {
    c.write_codes = (mode == MODE_MAX) || (mode == MODE_CJSO && T == 0);
    run_pass(&c, PH_MAX, nb, nthreads);
    for (int t = 1; t <= T; ++t) {
      set_alpha(&c, alpha_step(&c, c.alpha));
      c.write_codes = (mode == MODE_CJSO && t == T);
      run_pass(&c, PH_CJSO_ITER, nb, nthreads);
    }
    if (mode == MODE_CJSO_DECOUPLED) {
      c.sample = NULL;
      c.nsample = nb;
      c.out_codes = codes;
      c.out_scales = (uint8_t *)malloc(nb > 0 ? (size_t)nb : 1);
      if (!c.out_scales) {
        rc = 2;
      } else {
        run_pass(&c, PH_DECOUPLED, nb, nthreads);
        memcpy(c.dcode, c.out_scales, (size_t)nb);
        free(c.out_scales);
      }
    }
  }
  if (rc == 0) {
    memcpy(scales, c.dcode, (size_t)nb);
    *alpha_out = c.alpha;
  }
  free(c.dcode); free(c.P); free(c.R);
  return rc;
}

/* Same method, but the per-block outputs are produced only for the listed
 * blocks (codes: nsample*8 bytes, scales: nsample bytes, in list order).
 * Everything that couples blocks (alpha, the CJSO iterations) still runs over
 * the whole tensor; only the final per-block pass is restricted.  For MAX,
 * FourOverSix and decoupled CJSO the final pass is the expensive part. */
int oracle_quantize_sampled(const uint16_t *w, int64_t rows, int64_t cols, int mode, int iters,
                            const int64_t *sample, int64_t nsample, uint8_t *codes,
                            uint8_t *scales, float *alpha_out, int nthreads) {
  if (check_args(w, rows, cols) || mode < 0 || mode > 3 || !alpha_out || nsample < 0) return 1;
  if ((mode == MODE_CJSO || mode == MODE_CJSO_DECOUPLED) && (iters < 0 || iters > 64)) return 1;
  if (fegetround() != FE_TONEAREST) return 1;
  int64_t n = rows * cols, nb = n / BLOCK;
  for (int64_t i = 0; i < nsample; ++i)
    if (sample[i] < 0 || sample[i] >= nb) return 1;
  ctx_t c;
  memset(&c, 0, sizeof c);
  c.w = w;
  c.nblocks = nb;
  c.dcode = (uint8_t *)calloc(nb > 0 ? (size_t)nb : 1, 1);
  c.P = (float *)calloc(nb > 0 ? (size_t)nb : 1, sizeof(float));
  c.R = (float *)calloc(nb > 0 ? (size_t)nb : 1, sizeof(float));
  if (!c.dcode || !c.P || !c.R) {
    free(c.dcode); free(c.P); free(c.R);
    return 2;
  }
  set_alpha(&c, tensor_alpha(w, n));
  int T = (mode == MODE_CJSO || mode == MODE_CJSO_DECOUPLED) ? iters : 0;
  if (mode == MODE_CJSO || mode == MODE_CJSO_DECOUPLED) {
    run_pass(&c, PH_MAX, nb, nthreads);
    for (int t = 1; t <= T; ++t) {
      set_alpha(&c, alpha_step(&c, c.alpha));
      run_pass(&c, PH_CJSO_ITER, nb, nthreads);
    }
  }
  if (mode == MODE_CJSO_DECOUPLED) {
    c.sample = sample;
    c.nsample = nsample;
    c.out_codes = codes;
    c.out_scales = scales;
    run_pass(&c, PH_DECOUPLED, nsample, nthreads);
  } else {
    /* one block at a time, final pass only */
    for (int64_t i = 0; i < nsample; ++i) {
      int64_t b = sample[i];
      if (mode == MODE_MAX) do_block_max(&c, b, codes + i * 8);
      else if (mode == MODE_FOUR_OVER_SIX) do_block_fos(&c, b, codes + i * 8);
      else { /* CJSO: recompute the last block state for output */
        float x[BLOCK];
        uint8_t mag[BLOCK];
        float P, R;
        load_block(w, b, x);
        quant_block(x, c.alpha, (float)e4m3_value(c.dcode[b]), mag, &P, &R);
        pack_codes(x, mag, codes + i * 8);
      }
      scales[i] = c.dcode[b];
    }
  }
  *alpha_out = c.alpha;
  free(c.dcode); free(c.P); free(c.R);
  return 0;
}

/* [SOAR-DQ], reading R10. out: rows*cols bf16 bit patterns. */
int oracle_dequantize(const uint8_t *codes, const uint8_t *scales, float alpha, int64_t rows,
                      int64_t cols, uint16_t *out) {
  if (rows < 0 || cols < 0 || cols % BLOCK != 0) return 1;
  int64_t n = rows * cols;
  for (int64_t i = 0; i < n; ++i) {
    int code = (codes[i / 2] >> (4 * (i & 1))) & 0xF;
    float q = (float)E2M1_MAG[code & 7];
    if (code & 8) q = -q;
    float s = alpha * (float)e4m3_value(scales[i / BLOCK]);
    out[i] = f32_to_bf16_rne(q * s);
  }
  return 0;
}

/* Reconstruction MSE in double: (1/N) sum (x - q * fl(alpha*Delta))^2. */
double oracle_mse(const uint16_t *w, const uint8_t *codes, const uint8_t *scales, float alpha,
                  int64_t n) {
  double acc = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    int code = (codes[i / 2] >> (4 * (i & 1))) & 0xF;
    double q = E2M1_MAG[code & 7];
    if (code & 8) q = -q;
    double s = (double)(alpha * (float)e4m3_value(scales[i / BLOCK]));
    double e = (double)bf16_to_f32(w[i]) - q * s;
    acc += e * e;
  }
  return n > 0 ? acc / (double)n : 0.0;
}

/* Per-block squared error sum in double, for block-level invariants. */
void oracle_block_sse(const uint16_t *w, const uint8_t *codes, const uint8_t *scales,
                      float alpha, int64_t nblocks, double *out) {
  for (int64_t b = 0; b < nblocks; ++b) {
    double s = (double)(alpha * (float)e4m3_value(scales[b]));
    double acc = 0.0;
    for (int j = 0; j < BLOCK; ++j) {
      int64_t i = b * BLOCK + j;
      int code = (codes[i / 2] >> (4 * (i & 1))) & 0xF;
      double q = E2M1_MAG[code & 7];
      if (code & 8) q = -q;
      double e = (double)bf16_to_f32(w[i]) - q * s;
      acc += e * e;
    }
    out[b] = acc;
  }
}

/* CJSO trace for the monotonicity pin: MSE (double, with the exact product
 * alpha*Delta) after the max-rule start and, per iteration, after the alpha
 * step, the re-quantization, the Delta step and the second re-quantization.
 * trace must hold 1 + 4*iters doubles. */
static double state_mse(const uint16_t *w, int64_t nb, const uint8_t *mags, const uint8_t *dcode,
                        double alpha) {
  double acc = 0.0;
  for (int64_t b = 0; b < nb; ++b) {
    double s = alpha * e4m3_value(dcode[b]);
    for (int j = 0; j < BLOCK; ++j) {
      double x = fabs((double)bf16_to_f32(w[b * BLOCK + j]));
      double e = x - E2M1_MAG[mags[b * BLOCK + j]] * s;
      acc += e * e;
    }
  }
  return acc;
}

int oracle_cjso_trace(const uint16_t *w, int64_t rows, int64_t cols, int iters, double *trace,
                      float *alphas) {
  if (check_args(w, rows, cols) || iters < 0 || iters > 64) return 1;
  int64_t n = rows * cols, nb = n / BLOCK;
  uint8_t *mags = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
  ctx_t c;
  memset(&c, 0, sizeof c);
  c.w = w;
  c.nblocks = nb;
  c.dcode = (uint8_t *)malloc(nb > 0 ? (size_t)nb : 1);
  c.P = (float *)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
  c.R = (float *)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
  if (!mags || !c.dcode || !c.P || !c.R) {
    free(mags); free(c.dcode); free(c.P); free(c.R);
    return 2;
  }
  set_alpha(&c, tensor_alpha(w, n));
  float x[BLOCK];
  for (int64_t b = 0; b < nb; ++b) {
    load_block(w, b, x);
    int d = max_rule_code(&c, x);
    c.dcode[b] = (uint8_t)d;
    quant_block(x, c.alpha, (float)e4m3_value(d), mags + b * BLOCK, &c.P[b], &c.R[b]);
  }
  int k = 0;
  trace[k++] = state_mse(w, nb, mags, c.dcode, c.alpha);
  if (alphas) alphas[0] = c.alpha;
  for (int t = 1; t <= iters; ++t) {
    set_alpha(&c, alpha_step(&c, c.alpha));
    if (alphas) alphas[t] = c.alpha;
    trace[k++] = state_mse(w, nb, mags, c.dcode, c.alpha);
    for (int64_t b = 0; b < nb; ++b) {
      load_block(w, b, x);
      quant_block(x, c.alpha, (float)e4m3_value(c.dcode[b]), mags + b * BLOCK, &c.P[b], &c.R[b]);
    }
    trace[k++] = state_mse(w, nb, mags, c.dcode, c.alpha);
    for (int64_t b = 0; b < nb; ++b)
      if (c.R[b] > 0.0f) c.dcode[b] = (uint8_t)e4m3_code((double)(c.P[b] / (c.alpha * c.R[b])));
    trace[k++] = state_mse(w, nb, mags, c.dcode, c.alpha);
    for (int64_t b = 0; b < nb; ++b) {
      load_block(w, b, x);
      quant_block(x, c.alpha, (float)e4m3_value(c.dcode[b]), mags + b * BLOCK, &c.P[b], &c.R[b]);
    }
    trace[k++] = state_mse(w, nb, mags, c.dcode, c.alpha);
  }
  free(mags); free(c.dcode); free(c.P); free(c.R);
  return 0;
}

/* ---------------- element-wise access for the format pins ---------------- */

/* E2M1 code (sign | magnitude) of each fp32 value (reading R2). */
void oracle_e2m1_encode(const float *v, int64_t n, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = (uint8_t)(e2m1_mag_code(fabs((double)v[i])) | (f32_signbit(v[i]) << 3));
}

/* E4M3 code of each fp32 value >= 0 (nearest even, saturating; reading R3). */
void oracle_e4m3_encode(const float *v, int64_t n, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)e4m3_code((double)v[i]);
}

void oracle_e4m3_floor_ceil(const float *v, int64_t n, uint8_t *lo, uint8_t *hi) {
  for (int64_t i = 0; i < n; ++i) {
    lo[i] = (uint8_t)e4m3_floor_code((double)v[i]);
    hi[i] = (uint8_t)e4m3_ceil_code((double)v[i]);
  }
}

double oracle_e2m1_value(int code) {
  double q = E2M1_MAG[code & 7];
  return (code & 8) ? -q : q;
}

double oracle_e4m3_value(int code) { return e4m3_value(code & 0xFF); }

/* The 128-bit integer hi * 2^64 + lo rounded to the nearest double. */
double oracle_u128_to_double(uint64_t hi, uint64_t lo) {
  return u128_to_double(((unsigned __int128)hi << 64) | lo);
}

void oracle_bf16_round(const float *v, int64_t n, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(v[i]);
}

/* Per-block diagnostics of the quantizer with a given alpha and E4M3 code:
 * P, R (fp32, reading R5) and the exact double sum of |x| q, to pin R5. */
void oracle_block_sums(const uint16_t *w, int64_t nblocks, float alpha, const uint8_t *dcodes,
                       float *P, float *R, double *P_exact) {
  for (int64_t b = 0; b < nblocks; ++b) {
    float x[BLOCK];
    uint8_t mag[BLOCK];
    load_block(w, b, x);
    quant_block(x, alpha, (float)e4m3_value(dcodes[b]), mag, &P[b], &R[b]);
    double p = 0.0;
    for (int j = 0; j < BLOCK; ++j) p += fabs((double)x[j]) * E2M1_MAG[mag[j]];
    P_exact[b] = p;
  }
}

/* ---------------- consumer: W4A16 matrix-vector product ---------------- */

/* y[b][r] = sum_c What[r][c] * x[b][c] in double, What = the dequantized
 * bf16 weights of [SOAR-DQ] under reading R10 (the form a W4A16 kernel
 * consumes), x bf16 [batch][cols]; y double [batch][rows].  Reading R12:
 * the product consumes the dequantized weights rounded to bf16, exactly as
 * oracle_dequantize writes them. */
int oracle_gemv(const uint8_t *codes, const uint8_t *scales, float alpha, int64_t rows, int64_t cols,
                const uint16_t *x, int batch, double *y) {
  if (rows < 0 || cols < 0 || cols % BLOCK != 0 || batch < 1) return 1;
  for (int64_t r = 0; r < rows; ++r) {
    for (int b = 0; b < batch; ++b) {
      double acc = 0.0;
      for (int64_t c = 0; c < cols; ++c) {
        int64_t i = r * cols + c;
        int code = (codes[i / 2] >> (4 * (i & 1))) & 0xF;
        float q = (float)E2M1_MAG[code & 7];
        if (code & 8) q = -q;
        float s = alpha * (float)e4m3_value(scales[i / BLOCK]);
        double w = (double)bf16_to_f32(f32_to_bf16_rne(q * s));
        acc += w * (double)bf16_to_f32(x[(int64_t)b * cols + c]);
      }
      y[(int64_t)b * rows + r] = acc;
    }
  }
  return 0;
}

/* ---------------- scale layout for block-scaled tensor-core GEMMs ---------------- */

/* Reading R13 (the pages store the E4M3 scales but give no layout): the
 * layout block-scaled tensor-core matrix multiplies read.  The scale matrix
 * [rows, kb] (kb = cols/16) is padded with zeros to multiples of 128 rows and
 * 4 columns and cut into tiles of 128 x 4; tiles are stored one after the
 * other, the column tile varying fastest; inside a tile, the scale of tile
 * row r (0..127) and tile column c (0..3) sits at byte
 * (r mod 32) * 16 + (r div 32) * 4 + c.  out: round_up(rows,128) *
 * round_up(kb,4) bytes. */
int64_t oracle_swizzled_size(int64_t rows, int64_t kb) {
  return ((rows + 127) / 128 * 128) * ((kb + 3) / 4 * 4);
}

int oracle_swizzle_scales(const uint8_t *scales, int64_t rows, int64_t kb, uint8_t *out) {
  if (rows < 0 || kb < 0) return 1;
  int64_t ct = (kb + 3) / 4;
  memset(out, 0, (size_t)oracle_swizzled_size(rows, kb));
  for (int64_t i = 0; i < rows; ++i) {
    for (int64_t k = 0; k < kb; ++k) {
      int64_t tile = (i / 128) * ct + k / 4;
      int64_t r = i % 128, c = k % 4;
      out[tile * 512 + (r % 32) * 16 + (r / 32) * 4 + c] = scales[i * kb + k];
    }
  }
  return 0;
}
