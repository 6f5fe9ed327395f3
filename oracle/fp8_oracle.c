/*
 * fp8_oracle.c -- plain CPU reference for the FP8 linear-layer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only users of this file.  It shares no code,
 * header, table or constant generator with the CUDA library; the CUDA
 * library never loads it.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math (see oracle/build.py), so
 * every float operation written below rounds exactly once, in the type it is
 * written in (fp32 where the method works in fp32, fp64 for the GEMM).
 *
 * What it computes, with the passages it follows:
 *
 *  - E4M3FN decode / encode (1 sign, 4 exponent bits with bias 7, 3 mantissa
 *    bits, no infinities, S.1111.111 = NaN, largest finite 448).  Encoding
 *    rounds to nearest, ties to even, and saturates to +-448; NaN becomes +448
 *    the way the sanitizing clamp does in sglang PR #33533 ("[JIT]
 *    per_token_group_quant: fix the fp16 UE8M0 multiplier overflow ...",
 *    Modifications section 1).  A tie such as 168.0 rounds to 160, 168 plus
 *    one fp32 ulp to 176 (same PR, Motivation).
 *
 *  - per-token group quant (same PR, section 1 and the commit notes on the
 *    compile-time floor): per group of g consecutive elements of a row,
 *      amax = max |v| over the group's non-NaN elements,  a = max(amax, 1e-10),
 *      s = fl32(a / 448),  mult = fl32(448 / a)      (IEEE division),
 *      UE8M0: e = biased exponent of s (+1 if its mantissa is non-zero),
 *             s = 2^(e-127), mult = 2^(127-e)       (power of two),
 *      q = E4M3(fl32(v * mult)).
 *    The multiply is always fp32, so an fp16 input never sees the
 *    448/1e-10 multiplier overflow that the PR fixes.
 *    NaN inputs: the PR says only that a NaN reaching the encoder's clamp
 *    becomes +448; it does not say how the group absmax treats a NaN.  The
 *    reading taken here leaves NaN elements out of the absmax (infinities are
 *    kept), so a stray NaN does not poison the scale of its whole group.
 *
 *  - fused SiLU(gate)*up in front of the quant (same PR, section 2): silu(g) =
 *    g / (1 + exp(-g)) with a plain IEEE divide.  exp is the Cody-Waite
 *    reduced, degree-7 Taylor method written out in exp_cw7 below; it is a
 *    fixed sequence of IEEE fp32 operations so that a GPU that performs the
 *    same sequence reproduces it bit for bit.
 *
 *  - int8 group quant, the third output format of the same kernel family
 *    (same PR, "Verified": fp32 / ue8m0 / int8 scale formats): the same steps
 *    with 127 in place of 448, fp32 scales s = fl32(a / 127), multiplier
 *    fl32(127 / a), and q = int8(v * mult) after the same sanitizing clamp
 *    (NaN -> +127, then [-128, 127]) and rounding to nearest, ties to even.
 *    The pages print no int8 rounding rule; ties-to-even is the reading taken.
 *
 *  - scaled FP8 GEMM (sglang PR #34318 "Route large SM90 row/column-scaled
 *    FP8 GEMMs to Torch", Summary; prhub summary of sglang PR #33148,
 *    "Features and motivation"): D[m,n] = out(a_s * b_s * sum_k A[m,k] B[n,k]
 *    (+ bias[n])).  The sum is accumulated in fp64, which is exact: every
 *    E4M3 value is an integer times 2^-9, so every product is an integer
 *    times 2^-18 of at most 2^17.6 magnitude, and for K <= 2^15 every partial
 *    sum stays below 2^33 * 2^18 = 2^51 < 2^53 ulps.  The result is scaled in
 *    fp64 and rounded once to bf16 / fp16 (round to nearest even).
 *
 *  - block scales (sglang PR #44861, duplicate check: it names the block /
 *    MXFP8 GEMM of PR #42865 without detail; the layout here is the plainest
 *    one): A carries one scale per row and 128-wide K block, B one per
 *    128 x 128 block, and out = sum over K blocks g of
 *    a_s[m,g] * b_s[n/128, g] * partial_g.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------ */
/* E4M3FN                                                               */
/* ------------------------------------------------------------------ */

/* Value of an E4M3FN code, straight from its bit fields. */
static double e4m3_value(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 0x7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);            /* subnormal: (m/8) * 2^(1-7) */
  else
    v = ldexp(8.0 + (double)m, e - 10);  /* normal: (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

void oracle_decode_e4m3(const uint8_t* c, double* out, int64_t n) {
  double lut[256];
  for (int i = 0; i < 256; ++i) lut[i] = e4m3_value((uint8_t)i);
  for (int64_t i = 0; i < n; ++i) out[i] = lut[c[i]];
}

/* Code of a non-negative value r that lies exactly on the E4M3 grid. */
static uint8_t e4m3_code_of_grid_value(double r) {
  if (r == 0.0) return 0;
  if (r < ldexp(1.0, -6)) return (uint8_t)(r / ldexp(1.0, -9)); /* subnormal: m */
  int e2;
  frexp(r, &e2);                         /* r in [2^(e2-1), 2^e2) */
  int e = e2 - 1 + 7;                    /* biased exponent */
  int m = (int)(r / ldexp(1.0, e2 - 4)) - 8;
  return (uint8_t)((e << 3) | m);
}

/* Round-to-nearest-even E4M3FN encode with saturation to +-448. */
static uint8_t e4m3_encode(float x) {
  if (isnan(x)) return 0x7E;             /* the clamp turns NaN into +448 */
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  /* spacing of the E4M3 grid around a */
  double q;
  if (a < ldexp(1.0, -6)) {
    q = ldexp(1.0, -9);                  /* subnormal spacing */
  } else {
    int e2;
    frexp(a, &e2);
    q = ldexp(1.0, e2 - 4);              /* 3 mantissa bits: 2^(E-3), E = e2-1 */
  }
  double k = nearbyint(a / q);           /* a/q is exact; ties go to even k */
  return sign | e4m3_code_of_grid_value(k * q);
}

void oracle_encode_e4m3(const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------ */
/* bf16 / fp16 rounding from fp64 (round to nearest even, overflow to inf)  */
/* ------------------------------------------------------------------ */

/* Round |v| to a binary format with `mbits` explicit mantissa bits, minimum
 * normal exponent emin and maximum exponent emax.  Returns the rounded
 * magnitude (possibly +inf). */
static double round_binary(double a, int mbits, int emin, int emax) {
  if (a == 0.0) return 0.0;
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;                        /* a in [2^E, 2^(E+1)) */
  if (E < emin) E = emin;                /* subnormal range: fixed spacing */
  double q = ldexp(1.0, E - mbits);
  double r = nearbyint(a / q) * q;
  if (r >= ldexp(1.0, emax + 1)) return INFINITY;
  return r;
}

static uint16_t pack_binary16(int sign, double r, int mbits, int emin, int bias) {
  uint16_t s = sign ? 0x8000 : 0;
  if (isinf(r)) return s | (uint16_t)(((2 * bias + 1) << mbits));
  if (r == 0.0) return s;
  if (r < ldexp(1.0, emin)) return s | (uint16_t)(r / ldexp(1.0, emin - mbits));
  int e2;
  frexp(r, &e2);
  int E = e2 - 1;
  uint32_t m = (uint32_t)(r / ldexp(1.0, E - mbits)) - (1u << mbits);
  return s | (uint16_t)(((E + bias) << mbits) | m);
}

static uint16_t bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  double r = round_binary(fabs(v), 7, -126, 127);
  return pack_binary16(signbit(v), r, 7, -126, 127);
}

static uint16_t fp16_from_double(double v) {
  if (isnan(v)) return 0x7E00;
  double r = round_binary(fabs(v), 10, -14, 15);
  return pack_binary16(signbit(v), r, 10, -14, 15);
}

void oracle_round_bf16(const double* v, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_from_double(v[i]);
}

void oracle_round_fp16(const double* v, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = fp16_from_double(v[i]);
}

/* bf16 / fp16 bits -> fp32 (exact). */
static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static float fp16_to_float(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 31) v = m ? NAN : INFINITY;
  else if (e == 0) v = ldexp((double)m, -24);
  else v = ldexp(1024.0 + (double)m, e - 25);
  return (float)(s ? -v : v);            /* exact: fp16 values are fp32 values */
}

static float load_x(const uint16_t* x, int dtype, int64_t i) {
  return dtype == 0 ? bf16_to_float(x[i]) : fp16_to_float(x[i]);
}

/* ------------------------------------------------------------------ */
/* exp and SiLU in fp32                                                  */
/* ------------------------------------------------------------------ */

/* Power of two 2^k for k in [-126, 127], built from its bit pattern. */
static float pow2f_exact(int k) {
  uint32_t u = (uint32_t)(k + 127) << 23;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* exp(x) in fp32 by Cody-Waite range reduction and a Taylor polynomial:
 *   n = rint(x * log2(e)),  r = x - n*ln2 (ln2 split into a 16-bit head,
 *   so n*head is exact, and an fp32 tail), exp(r) = sum_{k<=7} r^k/k!
 *   by Horner's rule with fused multiply-adds, and exp(x) = exp(r) * 2^n
 *   applied as two exact power-of-two factors.  |r| <= 0.347, so the
 *   truncated term r^8/8! is below 0.2 ulp. */
static float exp_cw7(float x) {
  if (isnan(x)) return x;
  if (x > 89.0f) return INFINITY;
  if (x < -104.0f) return 0.0f;
  const float log2e = 1.44269502162933349609375f;  /* fl32(1/ln 2) */
  const float ln2_hi = 0.693145751953125f;          /* floor(ln2 * 2^16) / 2^16 */
  const float ln2_lo = 1.428606765330187e-06f;      /* fl32(ln2 - ln2_hi) */
  float n = rintf(x * log2e);
  float r = fmaf(-n, ln2_hi, x);
  r = fmaf(-n, ln2_lo, r);
  float p = 1.0f / 5040.0f;
  p = fmaf(p, r, 1.0f / 720.0f);
  p = fmaf(p, r, 1.0f / 120.0f);
  p = fmaf(p, r, 1.0f / 24.0f);
  p = fmaf(p, r, 1.0f / 6.0f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  int ni = (int)n;
  int n1 = ni / 2;                       /* truncating division */
  int n2 = ni - n1;
  return (p * pow2f_exact(n1)) * pow2f_exact(n2);
}

static float silu_f32(float g) {
  float e = exp_cw7(-g);
  float d = 1.0f + e;
  return g / d;
}

void oracle_exp_f32(const float* x, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = exp_cw7(x[i]);
}

void oracle_silu_f32(const float* x, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = silu_f32(x[i]);
}

/* ------------------------------------------------------------------ */
/* per-token group quant                                                 */
/* ------------------------------------------------------------------ */

/* Canonical outputs, one entry per (row, group):
 *   q      [M, K]  E4M3 codes
 *   s      [M, G]  the scale as fp32 (a/448, or 2^(e-127) under UE8M0)
 *   e      [M, G]  the UE8M0 exponent byte (0 when ue8m0 == 0)
 * Laying the scales out (row / column major, packing) is left to the
 * caller, which does it with plain indexing.
 * x is [M, K] (fuse == 0) or [M, 2K] with gate = x[:, :K], up = x[:, K:]. */
/* One step of the group absmax: |v| joins the maximum unless v is a NaN.  Every
   NaN is skipped, quiet or signaling; C's fmaxf may return NaN for a signaling
   operand (IEEE 754-2008 maxNum), which would make the result depend on where
   the NaN sits in the group. */
static float absmax_step(float amax, float v) {
  if (isnan(v)) return amax;
  float a = fabsf(v);
  return a > amax ? a : amax;
}

int oracle_group_quant(const uint16_t* x, int x_dtype, int64_t M, int64_t K, int64_t group,
                       int fuse_silu_mul, int ue8m0, uint8_t* q, float* s, uint8_t* e) {
  if (group <= 0 || K % group != 0) return -1;
  int64_t G = K / group;
  int64_t ldx = fuse_silu_mul ? 2 * K : K;
  float* v = (float*)malloc(sizeof(float) * (size_t)group);
  if (!v) return -2;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t g = 0; g < G; ++g) {
      /* step 1: load (and SiLU(gate) * up) */
      for (int64_t i = 0; i < group; ++i) {
        int64_t k = g * group + i;
        if (fuse_silu_mul) {
          float gate = load_x(x, x_dtype, m * ldx + k);
          float up = load_x(x, x_dtype, m * ldx + K + k);
          v[i] = silu_f32(gate) * up;
        } else {
          v[i] = load_x(x, x_dtype, m * ldx + k);
        }
      }
      /* step 2: group absmax and the floor */
      float amax = 0.0f;
      for (int64_t i = 0; i < group; ++i) amax = absmax_step(amax, v[i]);
      float a = fmaxf(amax, 1e-10f);
      /* step 3: scale and multiplier */
      float sc = a / 448.0f;
      float mult;
      uint8_t eb = 0;
      if (ue8m0) {
        uint32_t bits;
        memcpy(&bits, &sc, 4);
        int be = (int)((bits >> 23) & 0xFF);
        int ex = be + ((bits & 0x7FFFFF) != 0);
        sc = pow2f_exact(ex - 127);
        mult = pow2f_exact(127 - ex);
        eb = (uint8_t)ex;
      } else {
        mult = 448.0f / a;
      }
      /* step 4: encode */
      for (int64_t i = 0; i < group; ++i) q[m * K + g * group + i] = e4m3_encode(v[i] * mult);
      s[m * G + g] = sc;
      e[m * G + g] = eb;
    }
  }
  free(v);
  return 0;
}

/* int8 code of an fp32 value: NaN -> +127 (the clamp's min(v, 127) comes
   first), clamp to [-128, 127], round to nearest with ties to even. */
static int8_t i8_encode(float x) {
  if (isnan(x)) return 127;
  double c = (double)x;
  if (c > 127.0) c = 127.0;
  if (c < -128.0) c = -128.0;
  double f = floor(c), r = c - f;
  double n = f;
  if (r > 0.5 || (r == 0.5 && fmod(f, 2.0) != 0.0)) n = f + 1.0;
  return (int8_t)n;
}

void oracle_encode_i8(const float* x, int8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = i8_encode(x[i]);
}

int oracle_group_quant_int8(const uint16_t* x, int x_dtype, int64_t M, int64_t K, int64_t group,
                            int fuse_silu_mul, int8_t* q, float* s) {
  if (group <= 0 || K % group != 0) return -1;
  int64_t G = K / group;
  int64_t ldx = fuse_silu_mul ? 2 * K : K;
  float* v = (float*)malloc(sizeof(float) * (size_t)group);
  if (!v) return -2;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t g = 0; g < G; ++g) {
      for (int64_t i = 0; i < group; ++i) {
        int64_t k = g * group + i;
        if (fuse_silu_mul)
          v[i] = silu_f32(load_x(x, x_dtype, m * ldx + k)) * load_x(x, x_dtype, m * ldx + K + k);
        else
          v[i] = load_x(x, x_dtype, m * ldx + k);
      }
      float amax = 0.0f;
      for (int64_t i = 0; i < group; ++i) amax = absmax_step(amax, v[i]);
      float a = fmaxf(amax, 1e-10f);
      float mult = 127.0f / a;
      for (int64_t i = 0; i < group; ++i) q[m * K + g * group + i] = i8_encode(v[i] * mult);
      s[m * G + g] = a / 127.0f;
    }
  }
  free(v);
  return 0;
}

/* ------------------------------------------------------------------ */
/* scaled FP8 GEMM                                                       */
/* ------------------------------------------------------------------ */

typedef struct {
  const uint8_t* A; int64_t lda;
  const uint8_t* B; int64_t ldb;
  int64_t M, N, K;
  const float* a_scale; int a_mode; int64_t a_ld;  /* a_mode: 0 scalar, 1 row, 2 group row-major, 3 group col-major,
                                                      4 group UE8M0 bytes packed four per int32, col-major */
  const float* b_scale; int b_mode;                /* b_mode: 0 scalar, 1 column, 2 per 128 x 128 block */
  int64_t b_ld;                                    /* block scales per row of blocks (K / 128) */
  const uint16_t* bias;                            /* bf16 [N] or NULL */
  int out_dtype;                                   /* 0 bf16, 1 fp16 */
  const int64_t* rows; int64_t n_rows;             /* rows to compute (NULL: all) */
  uint16_t* out;                                   /* [n_rows, N] */
  double* exact;                                   /* [n_rows, N] or NULL */
  double* sumabs;                                  /* [n_rows, N] or NULL */
  const double* lut;
  int64_t r0, r1;
} gemm_job;

static double a_scale_at(const gemm_job* j, int64_t m, int64_t g) {
  switch (j->a_mode) {
    case 0: return (double)j->a_scale[0];
    case 1: return (double)j->a_scale[m];
    case 2: return (double)j->a_scale[m * j->a_ld + g];
    case 3: return (double)j->a_scale[g * j->a_ld + m];
    default: {
      /* UE8M0: byte g % 4 of word (g / 4, m) stands for the fp32 scale
         2^(byte - 127) (same PR, Modifications 3: the fp32 form of a UE8M0
         scale is 2^(e-127)).  Every byte is taken by that formula and the value
         rounded to fp32, the type the scales have everywhere else: byte 0 is the
         subnormal 2^-127, byte 255 (2^128) overflows to +inf. */
      const uint32_t* w = (const uint32_t*)j->a_scale;
      uint32_t e = (w[(g / 4) * j->a_ld + m] >> (8 * (g % 4))) & 0xFFu;
      return (double)ldexpf(1.0f, (int)e - 127);
    }
  }
}

static double b_block_scale_at(const gemm_job* j, int64_t n, int64_t g) {
  return (double)j->b_scale[(n / 128) * j->b_ld + g];
}

static void* gemm_rows(void* arg) {
  const gemm_job* j = (const gemm_job*)arg;
  const double* lut = j->lut;
  const int64_t group = 128;
  for (int64_t r = j->r0; r < j->r1; ++r) {
    int64_t m = j->rows ? j->rows[r] : r;
    const uint8_t* a = j->A + m * j->lda;
    for (int64_t n = 0; n < j->N; ++n) {
      const uint8_t* b = j->B + n * j->ldb;
      double bs = j->b_mode == 0 ? (double)j->b_scale[0] : (j->b_mode == 1 ? (double)j->b_scale[n] : 1.0);
      double val, sabs = 0.0;
      if (j->a_mode <= 1) {
        double acc = 0.0;
        for (int64_t k = 0; k < j->K; ++k) {
          double p = lut[a[k]] * lut[b[k]];
          acc += p;
          sabs += fabs(p);
        }
        double as = a_scale_at(j, m, 0);
        val = acc * as * bs;
        sabs = sabs * fabs(as * bs);
      } else {
        /* per-group A scales: sum over groups of a_s[m,g] * (sum over the group) */
        double tot = 0.0;
        for (int64_t g = 0; g * group < j->K; ++g) {
          double acc = 0.0, gabs = 0.0;
          for (int64_t k = g * group; k < (g + 1) * group && k < j->K; ++k) {
            double p = lut[a[k]] * lut[b[k]];
            acc += p;
            gabs += fabs(p);
          }
          double as = a_scale_at(j, m, g);
          if (j->b_mode == 2) as *= b_block_scale_at(j, n, g);  /* exact: fp32 x fp32 fits fp64 */
          tot += as * acc;
          sabs += fabs(as) * gabs;
        }
        val = tot * bs;
        sabs = sabs * fabs(bs);
      }
      if (j->bias) val += (double)bf16_to_float(j->bias[n]);
      int64_t o = r * j->N + n;
      j->out[o] = j->out_dtype == 0 ? bf16_from_double(val) : fp16_from_double(val);
      if (j->exact) j->exact[o] = val;
      if (j->sumabs) j->sumabs[o] = sabs;
    }
  }
  return NULL;
}

int oracle_gemm(const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb, int64_t M, int64_t N,
                int64_t K, const float* a_scale, int a_mode, int64_t a_ld, const float* b_scale,
                int b_mode, const uint16_t* bias, int out_dtype, const int64_t* rows, int64_t n_rows,
                uint16_t* out, double* exact, double* sumabs, int nthreads) {
  if (b_mode == 2 && a_mode < 2) return -3;  /* block B scales go with per-group A scales */
  double lut[256];
  for (int i = 0; i < 256; ++i) lut[i] = e4m3_value((uint8_t)i);
  if (!rows) n_rows = M;
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n_rows) nthreads = n_rows > 0 ? (int)n_rows : 1;
  gemm_job base = {A, lda, B, ldb, M, N, K, a_scale, a_mode, a_ld, b_scale, b_mode, (K + 127) / 128, bias,
                   out_dtype, rows, n_rows, out, exact, sumabs, lut, 0, 0};
  gemm_job* jobs = (gemm_job*)malloc(sizeof(gemm_job) * (size_t)nthreads);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!jobs || !th) { free(jobs); free(th); return -2; }
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = base;
    jobs[t].r0 = n_rows * t / nthreads;
    jobs[t].r1 = n_rows * (t + 1) / nthreads;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, gemm_rows, &jobs[t]);
  gemm_rows(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
  return nthreads;
}

int oracle_num_threads(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }
