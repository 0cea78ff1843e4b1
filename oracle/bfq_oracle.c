/*
 * bfq_oracle.c — plain, slow, obviously-correct CPU oracle for block-scaled
 * FP8 (W8A8) quantization and GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant
 * generator with the CUDA library; it is written from the definitions on the
 * pages it cites:
 *
 *   [vLLM-29546]  "[Perf] Deepgemm fused layout kernel for activations"
 *                 (vLLM PR #29546): Purpose section (scales packed into a
 *                 uint32 early, inside the quant kernel) and the review thread
 *                 (packed UE8M0 int32 scales vs. the GEMM's E8M0 flag).
 *   [vLLM-19885]  "[EP+DP] Optimize the little operations in the DeepGEMM +
 *                 DeepEP low latency case" (vLLM PR #19885): Summary, item 2
 *                 (fused silu-mul-quant that neither loads nor computes
 *                 padded tokens).
 *   [vLLM-19111]  "[Kernel] Integrate batched/masked deepgemm kernel"
 *                 (vLLM PR #19111): Summary of Changes (masked grouped GEMM
 *                 m_grouped_gemm_fp8_fp8_bf16_nt_masked, 128x128 blocks).
 *   [DG-bench]    "vLLM DeepGEMM FP8 Block GEMM 基准测试" (pgsm.cn article on
 *                 benchmarks/kernels/deepgemm): §4.1 (per_token_group_quant_fp8
 *                 with column-major TMA-aligned scales, per_block_cast_to_fp8
 *                 with amax / fp8_max and UE8M0 ceil-to-power-of-two),
 *                 §4.2 (block-scaled GEMM: per-K-block dot times a_s * b_s),
 *                 §4.3 (metric formulas).
 *
 * Readings where the pages are silent:
 *   - e4m3 is the OCP "fn" variant (bias 7, max 448, no inf, S.1111.111 = NaN);
 *     conversion is round-to-nearest, ties to the even code, saturating to
 *     +-448 ("satfinite"); NaN converts to 0x7F.
 *   - group scale s = fl32(max(amax, eps) / 448) with eps = 1e-10, IEEE fp32
 *     division; the quantized value is e4m3(fl32(x / s)) (division, not a
 *     reciprocal multiply).
 *   - UE8M0 scale = the smallest power of two >= s (eps applied first).
 *   - packed word for row r, word w holds the biased exponents of groups
 *     4w..4w+3, group 4w in the least significant byte; missing groups of a
 *     partial last word are 0.
 *   - scale arrays are column-major: element (row r, column c) at c*ld + r.
 *   - silu(g) = g / (1 + exp(-g)) in fp32, y = silu(g) * u in fp32, y is not
 *     rounded to bf16 before it is quantized; gate is the first half of the
 *     row, up the second half.  exp is the fp32 function bfq-exp defined
 *     below (Cody-Waite reduction + degree-7 Taylor polynomial), because a
 *     quantized code is decided by it and both implementations must take that
 *     decision in the same arithmetic.
 *   - 128x128 weight blocks use the same rule as the 1x128 activation groups.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -o _bfq_oracle.so
 *        bfq_oracle.c -lm      (no fast-math: every fp32 op is IEEE).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_FMT_F32 0          /* fp32 scales, column-major [G][ld]          */
#define ORC_FMT_F32_POW2 1     /* fp32 power-of-two (UE8M0 value) scales     */
#define ORC_FMT_UE8M0_PACKED 2 /* int32 words, 4 exponents each, [W][ld]     */

static const float ORC_FP8_MAX = 448.0f;
static const float ORC_EPS = 1e-10f;

/* ------------------------------------------------------------------------ */
/* bf16 / fp32 bit views                                                     */
/* ------------------------------------------------------------------------ */
static float orc_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static float orc_f32_from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ------------------------------------------------------------------------ */
/* OCP FP8 E4M3 ("fn") — decode is the format's definition                   */
/* ------------------------------------------------------------------------ */
double orc_e4m3_decode(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN; /* the only NaN pattern (per sign) */
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

static double orc_mag_table[127]; /* magnitudes of codes 0x00..0x7E, ascending */
static int orc_tables_ready = 0;

static void orc_init_tables(void) {
  if (orc_tables_ready) return;
  for (int c = 0; c < 127; ++c) orc_mag_table[c] = orc_e4m3_decode((uint8_t)c);
  orc_tables_ready = 1;
}

/* Nearest representable magnitude, ties to the even code, saturate at 448. */
uint8_t orc_e4m3_encode(float v) {
  orc_init_tables();
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= orc_mag_table[126]) return sign | 126; /* satfinite: +-448 */
  /* largest code c with mag[c] <= a (binary search over the sorted table) */
  int lo = 0, hi = 126;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (orc_mag_table[mid] <= a) lo = mid; else hi = mid;
  }
  int c = lo;
  if (orc_mag_table[c] == a) return sign | (uint8_t)c;
  /* compare 2a with mag[c] + mag[c+1]: both sides exact in double */
  double twice = 2.0 * a, mid = orc_mag_table[c] + orc_mag_table[c + 1];
  int pick;
  if (twice < mid) pick = c;
  else if (twice > mid) pick = c + 1;
  else pick = (c % 2 == 0) ? c : c + 1; /* tie: even code (mantissa lsb 0) */
  return sign | (uint8_t)pick;
}

/* ------------------------------------------------------------------------ */
/* Group scale (1x128 activations, 128x128 weights): s = max(amax,eps)/448   */
/* ------------------------------------------------------------------------ */
static float orc_group_scale(float amax) {
  float a = amax > ORC_EPS ? amax : ORC_EPS;
  return a / ORC_FP8_MAX; /* IEEE fp32 division */
}

/* Smallest power of two >= s (s positive, normal).  frexp gives
 * s = f * 2^e with f in [0.5, 1); s is a power of two iff f == 0.5. */
static float orc_ceil_pow2(float s) {
  int e;
  float f = frexpf(s, &e);
  if (f == 0.5f) return s;
  return ldexpf(1.0f, e);
}

/* Biased UE8M0 exponent byte of a positive power of two p (p = 2^(byte-127)). */
static uint8_t orc_ue8m0_byte(float p) {
  int e;
  (void)frexpf(p, &e);           /* p = 0.5 * 2^e  =>  p = 2^(e-1) */
  return (uint8_t)(e - 1 + 127);
}

/* Quantize one group of n fp32 values (n <= 128).  Writes the n codes and
 * returns the fp32 scale actually used (pow2-rounded when pow2 != 0). */
static float orc_quant_group(const float* v, int n, int pow2, uint8_t* q) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  float s = orc_group_scale(amax);
  if (pow2) s = orc_ceil_pow2(s);
  for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(v[i] / s);
  return s;
}

static void orc_store_scale(int fmt, void* scales, int64_t ld, int64_t r, int64_t g,
                            float s) {
  if (fmt == ORC_FMT_UE8M0_PACKED) {
    uint32_t* w = (uint32_t*)scales + (g / 4) * ld + r;
    uint32_t byte = orc_ue8m0_byte(s);
    int shift = 8 * (int)(g % 4);
    *w = (*w & ~(0xFFu << shift)) | (byte << shift);
  } else {
    ((float*)scales)[g * ld + r] = s;
  }
}

/* Per-token-group quant of a bf16 activation matrix x[M][ld_x] (first K
 * columns used).  q is [M][K] row-major; scales column-major with leading
 * dimension scale_ld >= M ([DG-bench] §4.1 "column-major, TMA-aligned";
 * [vLLM-29546] Purpose: packed 4 per uint32). Returns 0, or -1 on bad args. */
int orc_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ld_x, int fmt, uint8_t* q,
              void* scales, int64_t scale_ld) {
  if (K % 128 != 0 || scale_ld < M || ld_x < K) return -1;
  for (int64_t r = 0; r < M; ++r) {
    float buf[128];
    int64_t G = K / 128;
    if (fmt == ORC_FMT_UE8M0_PACKED)
      for (int64_t w = 0; w < (G + 3) / 4; ++w) ((uint32_t*)scales)[w * scale_ld + r] = 0u;
    for (int64_t g = 0; g < G; ++g) {
      for (int i = 0; i < 128; ++i) buf[i] = orc_bf16_to_f32(x[r * ld_x + g * 128 + i]);
      float s = orc_quant_group(buf, 128, fmt != ORC_FMT_F32, q + r * K + g * 128);
      orc_store_scale(fmt, scales, scale_ld, r, g, s);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* bfq-exp: fp32 exp by Cody-Waite range reduction and a Taylor polynomial.  */
/*   n = rint(x * log2(e)),  r = (x - n*ln2_hi) - n*ln2_lo,                  */
/*   exp(r) ~ sum_{k=0..7} r^k / k!  (Horner, fused multiply-adds),          */
/*   exp(x) = exp(r) * 2^n, the power applied as two exact factors.          */
/* ln2_hi = 0x1.62e4p-1 (15 significant bits), ln2_lo = fl32(ln2 - ln2_hi).   */
/* Inputs below -88 return 0, above 89 return +inf, NaN propagates.          */
/* ------------------------------------------------------------------------ */
static float orc_pow2i(int k) { /* 2^k for -126 <= k <= 127 */
  return orc_f32_from_bits((uint32_t)(k + 127) << 23);
}

float orc_expf(float x) {
  if (isnan(x)) return x;
  if (x < -88.0f) return 0.0f;
  if (x > 89.0f) return INFINITY;
  const float log2e = 0x1.715476p+0f;
  const float ln2_hi = 0x1.62e4p-1f;
  const float ln2_lo = 0x1.7f7d1cp-20f;
  float n = rintf(x * log2e);
  float r = fmaf(-n, ln2_hi, x);
  r = fmaf(-n, ln2_lo, r);
  float p = 0x1.a01a02p-13f;        /* 1/7! */
  p = fmaf(p, r, 0x1.6c16c2p-10f);  /* 1/6! */
  p = fmaf(p, r, 0x1.111112p-7f);   /* 1/5! */
  p = fmaf(p, r, 0x1.555556p-5f);   /* 1/4! */
  p = fmaf(p, r, 0x1.555556p-3f);   /* 1/3! */
  p = fmaf(p, r, 0.5f);             /* 1/2! */
  p = fmaf(p, r, 1.0f);             /* 1/1! */
  p = fmaf(p, r, 1.0f);             /* 1/0! */
  int k = (int)n;
  int k1 = k / 2;
  int k2 = k - k1;
  return (p * orc_pow2i(k1)) * orc_pow2i(k2);
}

/* silu(g) = g / (1 + exp(-g)), fp32 ([vLLM-19885] Summary item 2). */
float orc_silu(float g) { return g / (1.0f + orc_expf(-g)); }

/* Fused silu-and-mul + group quant over a masked batch
 * ([vLLM-19885] Summary item 2; [vLLM-19111] masked per-expert layout).
 * x: [E][T][2I] bf16, gate = cols [0,I), up = cols [I,2I).
 * Row r of expert e is processed iff r < counts[e]; other rows of q and of
 * the scales are not touched.  q: [E][T][I]; scales: [E][cols][scale_ld]
 * with cols = I/128 (fp32 formats) or ceil(I/512) (packed). */
int orc_silu_mul_quant(const uint16_t* x, int64_t E, int64_t T, int64_t I,
                       const int32_t* counts, int fmt, uint8_t* q, void* scales,
                       int64_t scale_ld) {
  if (I % 128 != 0 || scale_ld < T) return -1;
  int64_t G = I / 128;
  int64_t cols = (fmt == ORC_FMT_UE8M0_PACKED) ? (G + 3) / 4 : G;
  float buf[128];
  for (int64_t e = 0; e < E; ++e) {
    int64_t cnt = counts[e];
    if (cnt < 0) cnt = 0;
    if (cnt > T) cnt = T;
    void* sc = (fmt == ORC_FMT_UE8M0_PACKED)
                   ? (void*)((uint32_t*)scales + e * cols * scale_ld)
                   : (void*)((float*)scales + e * cols * scale_ld);
    for (int64_t r = 0; r < cnt; ++r) {
      const uint16_t* xr = x + (e * T + r) * (2 * I);
      uint8_t* qr = q + (e * T + r) * I;
      if (fmt == ORC_FMT_UE8M0_PACKED)
        for (int64_t w = 0; w < cols; ++w) ((uint32_t*)sc)[w * scale_ld + r] = 0u;
      for (int64_t g = 0; g < G; ++g) {
        for (int i = 0; i < 128; ++i) {
          float gate = orc_bf16_to_f32(xr[g * 128 + i]);
          float up = orc_bf16_to_f32(xr[I + g * 128 + i]);
          buf[i] = orc_silu(gate) * up;
        }
        float s = orc_quant_group(buf, 128, fmt != ORC_FMT_F32, qr + g * 128);
        orc_store_scale(fmt, sc, scale_ld, r, g, s);
      }
    }
  }
  return 0;
}

/* 128x128 block weight quant ([DG-bench] §4.1, per_block_cast_to_fp8):
 * w: [N][K] bf16 -> wq [N][K] e4m3, sw [ceil(N/128)][K/128] fp32
 * (power-of-two values when pow2 != 0).  A partial last row-block uses only
 * its rows < N. */
int orc_weight_block_quant(const uint16_t* w, int64_t N, int64_t K, int pow2, uint8_t* wq,
                           float* sw) {
  if (K % 128 != 0) return -1;
  int64_t NB = (N + 127) / 128, KB = K / 128;
  for (int64_t nb = 0; nb < NB; ++nb) {
    int64_t n0 = nb * 128, n1 = n0 + 128 < N ? n0 + 128 : N;
    for (int64_t kb = 0; kb < KB; ++kb) {
      float amax = 0.0f;
      for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
          float a = fabsf(orc_bf16_to_f32(w[n * K + k]));
          if (a > amax) amax = a;
        }
      float s = orc_group_scale(amax);
      if (pow2) s = orc_ceil_pow2(s);
      sw[nb * KB + kb] = s;
      for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
          wq[n * K + k] = orc_e4m3_encode(orc_bf16_to_f32(w[n * K + k]) / s);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Block-scaled GEMM ([DG-bench] §4.2):                                      */
/*   C[m,n] = sum_b sA[m,b] * sW[n/128,b] * sum_{k in block b} a[m,k] w[n,k] */
/* The inner block dot is exact in fp64 (products of two e4m3 values are    */
/* multiples of 2^-18 below 2^18; a 128-term sum stays below 2^25, so 43    */
/* bits suffice).  The scaled block partials are accumulated in fp64.       */
/* ------------------------------------------------------------------------ */
static double orc_act_scale(const void* sa, int fmt, int64_t ld, int64_t m, int64_t b) {
  if (fmt == ORC_FMT_UE8M0_PACKED) {
    uint32_t word = ((const uint32_t*)sa)[(b / 4) * ld + m];
    int byte = (int)((word >> (8 * (b % 4))) & 0xFF);
    return ldexp(1.0, byte - 127);
  }
  return (double)((const float*)sa)[b * ld + m];
}

/* Rows rows[0..nrows) of C = A * W^T.  aq [M][K], wq [N][K] e4m3 row-major,
 * sa column-major (ld = sa_ld), sw [ceil(N/128)][K/128] fp32.  out is
 * [nrows][N] fp64. */
int orc_gemm_rows(const uint8_t* aq, const void* sa, int fmt_a, int64_t sa_ld,
                  const uint8_t* wq, const float* sw, int64_t M, int64_t N, int64_t K,
                  const int64_t* rows, int64_t nrows, double* out) {
  if (K % 128 != 0) return -1;
  orc_init_tables();
  double dec[256];
  for (int c = 0; c < 256; ++c) dec[c] = orc_e4m3_decode((uint8_t)c);
  int64_t KB = K / 128;
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = rows[i];
    if (m < 0 || m >= M) return -1;
    const uint8_t* a = aq + m * K;
    for (int64_t n = 0; n < N; ++n) {
      const uint8_t* w = wq + n * K;
      double acc = 0.0;
      for (int64_t b = 0; b < KB; ++b) {
        double dot = 0.0;
        for (int64_t k = b * 128; k < b * 128 + 128; ++k) dot += dec[a[k]] * dec[w[k]];
        double s = orc_act_scale(sa, fmt_a, sa_ld, m, b) * (double)sw[(n / 128) * KB + b];
        acc += dot * s;
      }
      out[i * N + n] = acc;
    }
  }
  return 0;
}

/* Masked grouped GEMM ([vLLM-19111]: per-expert valid-row count).
 * aq [E][T][K], sa per expert [E][cols][sa_ld], wq [E][N][K],
 * sw [E][ceil(N/128)][K/128]; out [E][T][N] fp64, rows r >= counts[e]
 * are not written. */
int orc_gemm_masked(const uint8_t* aq, const void* sa, int fmt_a, int64_t sa_ld,
                    const uint8_t* wq, const float* sw, const int32_t* counts, int64_t E,
                    int64_t T, int64_t N, int64_t K, double* out) {
  if (K % 128 != 0) return -1;
  int64_t KB = K / 128;
  int64_t cols = (fmt_a == ORC_FMT_UE8M0_PACKED) ? (KB + 3) / 4 : KB;
  int64_t NB = (N + 127) / 128;
  for (int64_t e = 0; e < E; ++e) {
    int64_t cnt = counts[e];
    if (cnt < 0) cnt = 0;
    if (cnt > T) cnt = T;
    const void* sae = (fmt_a == ORC_FMT_UE8M0_PACKED)
                          ? (const void*)((const uint32_t*)sa + e * cols * sa_ld)
                          : (const void*)((const float*)sa + e * cols * sa_ld);
    for (int64_t r = 0; r < cnt; ++r) {
      int rc = orc_gemm_rows(aq + e * T * K, sae, fmt_a, sa_ld, wq + e * N * K,
                             sw + e * NB * KB, T, N, K, &r, 1, out + (e * T + r) * N);
      if (rc) return rc;
    }
  }
  return 0;
}
