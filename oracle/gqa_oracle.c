/*
 * gqa_oracle.c -- plain FP64 CPU definition of single-token grouped-query
 * decode attention over a KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity oracle for the CUDA
 * library in gqa_decode_attention_sm_gb300/.  It shares no code, header,
 * table or constant with that library, and only tests/, the smoke check in
 * __graft_entry__.py and the CPU-baseline leg of bench.py may load it.
 *
 * Sources (the pages this oracle restates):
 *   [FI]  "FlashInfer sm110_gqa_decode" article (cf-1.com), sections
 *         "Input contract" (q [batch,32,128], kv [batch,2,8,capacity,128],
 *         K plane 0 / V plane 1, lengths in [1,capacity] read only on the
 *         device), "Convenience API" (q_scale and the softmax scale
 *         q_scale/sqrt(128); the grouped view of q in 8 groups of 4
 *         consecutive heads: query heads 4g..4g+3 share KV head g).
 *   [FP8] "FP8 KV cache port on Jetson AGX Thor" blog (kipfel.ltd),
 *         section 1, patch 2: the e4m3 tile is promoted before the dot
 *         product, scores are multiplied by k_scale, the normalised output
 *         by v_scale; patch 1 item 5: the cache bytes are reinterpreted as
 *         float8_e4m3fn, not converted.
 *   [ORIN] "Qwen3-VL official BF16 on Jetson Orin (SM87)" docs, section
 *         "INT8 KV cache (kv_mode)": the cache kept as int8 codes, each
 *         (position, KV head) row with its own bf16 scale; section "Decode
 *         weight quantization": symmetric int8, the scale amax/127.
 *   [TU]  "FreeToken-Kai on Turing" notes, change 7: below Ampere every key
 *         of the range is scored first and one ordinary softmax runs over
 *         all of them, with no running maximum.  This oracle takes that
 *         two-pass form.
 *
 * Definition computed for every requested (b, h):
 *   g   = h / 4                                  (grouped view, [FI])
 *   L   = seq_lens[b], 1 <= L <= capacity        (slots >= L are never read)
 *   K_t = dec(kv[b,0,g,t,:]) * k_scale,  V_t = dec(kv[b,1,g,t,:]) * v_scale
 *   s_t = (q_scale / sqrt(128)) * sum_d dec(q[b,h,d]) * K_t[d]
 *   w_t = exp(s_t - max_u s_u)
 *   out = sum_t w_t V_t / sum_t w_t,  rounded once, FP64 -> fp16/bf16, RNE.
 * Verify window (q_len = T > 1, [FP8] section 2, MTP draft tokens): q is
 * [batch, T, 32, 128]; query token j sits at position L - T + j and attends
 * slots [0, L - T + j], i.e. the definition above with L_j = L - T + 1 + j.
 * For the INT8 cache ([ORIN]) dec(kv[b,p,g,t,d]) = code * scale[b,p,g,t], the
 * int8 code times the bf16 scale of that (plane, KV head, position) row.
 * For fp16/bf16 KV, k_scale = v_scale = 1.  Multiplying V by v_scale before
 * the weighted sum equals multiplying the normalised output by v_scale in
 * exact arithmetic ([FP8]).
 *
 * Number formats are decoded from their definitions, not from any library:
 *   binary16 (IEEE 754): 1 sign, 5 exponent (bias 15), 10 fraction bits.
 *   bfloat16: the upper 16 bits of IEEE 754 binary32 (bias 127, 7 fraction).
 *   float8 e4m3fn (OCP FP8): 1 sign, 4 exponent (bias 7), 3 fraction bits,
 *   no infinities, S.1111.111 is NaN, largest finite 448.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread (no fast-math).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_I8 = 3 };

enum {
  ORC_OK = 0,
  ORC_EINVAL = 1,   /* bad argument (null pointer, unknown type, size) */
  ORC_ELENGTH = 2,  /* a requested row has a length outside [1, capacity] */
  ORC_ENOMEM = 3
};

#define ORC_HQ 32
#define ORC_HKV 8
#define ORC_D 128

/* ---------------------------------------------------------------- decode */

double orc_decode_f16(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0x1f) v = m ? NAN : INFINITY;
  else if (e == 0) v = ldexp((double)m, -24);           /* subnormal: m * 2^(1-15-10) */
  else v = ldexp((double)(1024 + m), e - 25);           /* (1 + m/2^10) * 2^(e-15) */
  return s ? -v : v;
}

double orc_decode_bf16(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 7) & 0xff, m = h & 0x7f;
  double v;
  if (e == 0xff) v = m ? NAN : INFINITY;
  else if (e == 0) v = ldexp((double)m, -133);          /* m * 2^(1-127-7) */
  else v = ldexp((double)(128 + m), e - 134);           /* (1 + m/2^7) * 2^(e-127) */
  return s ? -v : v;
}

double orc_decode_e4m3(uint8_t b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 0xf, m = b & 0x7;
  double v;
  if (e == 0xf && m == 0x7) v = NAN;                    /* the only NaN encoding */
  else if (e == 0) v = ldexp((double)m, -9);            /* m * 2^(1-7-3) */
  else v = ldexp((double)(8 + m), e - 10);              /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* ----------------------------------------------------------------- round */

/* Round x to the nearest value of a binary format with `frac` fraction bits,
 * minimum normal exponent `emin` and maximum finite value `maxf`, ties to
 * even, and return the encoded bits.  The quantum (spacing of representable
 * values around |x|) is a power of two, so x / quantum is exact in double and
 * rint() (default rounding mode: nearest, ties to even) does the rounding. */
static uint16_t orc_round_generic(double x, int frac, int emin, int ebits, double maxf) {
  const int bias = (1 << (ebits - 1)) - 1;
  const uint16_t sign = signbit(x) ? (uint16_t)(1u << (frac + ebits)) : 0;
  const uint16_t exp_all = (uint16_t)(((1u << ebits) - 1) << frac);
  if (isnan(x)) return (uint16_t)(exp_all | (1u << (frac - 1)));     /* quiet NaN */
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | exp_all);
  int e;
  frexp(a, &e);                  /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
  int unbiased = e - 1;
  if (unbiased < emin) unbiased = emin;                 /* subnormal range */
  double quantum = ldexp(1.0, unbiased - frac);
  double r = rint(a / quantum) * quantum;               /* exact */
  if (r > maxf) return (uint16_t)(sign | exp_all);      /* overflow -> inf */
  if (r == 0.0) return sign;
  frexp(r, &e);
  unbiased = e - 1;
  if (unbiased < emin) {                                /* subnormal encoding */
    uint32_t m = (uint32_t)(r / ldexp(1.0, emin - frac));
    return (uint16_t)(sign | m);
  }
  uint32_t m = (uint32_t)(r / ldexp(1.0, unbiased - frac)) - (1u << frac);
  return (uint16_t)(sign | ((uint32_t)(unbiased + bias) << frac) | m);
}

uint16_t orc_round_f16(double x) {
  return orc_round_generic(x, 10, -14, 5, 65504.0);
}

uint16_t orc_round_bf16(double x) {
  return orc_round_generic(x, 7, -126, 8, ldexp(255.0, 120)); /* (2 - 2^-7) * 2^127 */
}

/* Array forms of the two functions above (one call instead of one per value). */
void orc_decode_array(const void* in, int fmt, size_t n, double* out) {
  for (size_t i = 0; i < n; ++i) {
    if (fmt == ORC_I8) out[i] = (double)((const int8_t*)in)[i];
    else if (fmt == ORC_E4M3) out[i] = orc_decode_e4m3(((const uint8_t*)in)[i]);
    else if (fmt == ORC_F16) out[i] = orc_decode_f16(((const uint16_t*)in)[i]);
    else out[i] = orc_decode_bf16(((const uint16_t*)in)[i]);
  }
}

void orc_round_array(const double* in, size_t n, int fmt, uint16_t* out) {
  for (size_t i = 0; i < n; ++i)
    out[i] = fmt == ORC_F16 ? orc_round_f16(in[i]) : orc_round_bf16(in[i]);
}

/* ------------------------------------------------------------- attention */

typedef struct {
  const void* q;
  int q_type;
  const void* kv;
  int kv_type;
  const uint16_t* kv_scales;  /* ORC_I8: bf16 bits [B,2,8,C]; else NULL */
  const int32_t* lens;
  int batch, capacity, q_len;
  double q_scale, k_scale, v_scale;
  const int32_t* rows;  /* (b*q_len + j)*32 + h */
  int n_rows;
  double* out_f64;      /* [n_rows][128] */
  uint16_t* out_bits;   /* [n_rows][128] or NULL */
  int out_type;
  int n_threads;
  int thread_index;
  int status;
} orc_job;

static double orc_elem(const void* base, int type, size_t i) {
  if (type == ORC_I8) return (double)((const int8_t*)base)[i];
  if (type == ORC_E4M3) return orc_decode_e4m3(((const uint8_t*)base)[i]);
  uint16_t h = ((const uint16_t*)base)[i];
  return type == ORC_F16 ? orc_decode_f16(h) : orc_decode_bf16(h);
}

/* One output row: the plain two-pass softmax of [TU] over slots [0, L). */
static int orc_row(const orc_job* j, int r, double* s) {
  const int bh = j->rows[r];
  const int bq = bh / ORC_HQ, h = bh % ORC_HQ;   /* bq = b * q_len + query token */
  const int b = bq / j->q_len, qt = bq % j->q_len;
  const int g = h / (ORC_HQ / ORC_HKV);
  const int len = j->lens[b];
  if (len < j->q_len || len > j->capacity) return ORC_ELENGTH;
  const int L = len - j->q_len + 1 + qt;         /* causal within the window */
  const size_t C = (size_t)j->capacity;
  const size_t q_off = ((size_t)bq * ORC_HQ + h) * ORC_D;
  const size_t k_off = (((size_t)b * 2 + 0) * ORC_HKV + g) * C * ORC_D;
  const size_t v_off = (((size_t)b * 2 + 1) * ORC_HKV + g) * C * ORC_D;
  const double scale = j->q_scale / sqrt((double)ORC_D);

  double qd[ORC_D];
  for (int d = 0; d < ORC_D; ++d) qd[d] = orc_elem(j->q, j->q_type, q_off + d);

  /* pass 1: every score, and their maximum */
  /* one scale per (plane, KV head, position) row for the INT8 cache */
  const size_t ks_off = (((size_t)b * 2 + 0) * ORC_HKV + g) * C;
  const size_t vs_off = (((size_t)b * 2 + 1) * ORC_HKV + g) * C;
  double m = -INFINITY;
  for (int t = 0; t < L; ++t) {
    const double row_k = j->kv_type == ORC_I8 ? orc_decode_bf16(j->kv_scales[ks_off + t]) : 1.0;
    double dot = 0.0;
    for (int d = 0; d < ORC_D; ++d) {
      double k = orc_elem(j->kv, j->kv_type, k_off + (size_t)t * ORC_D + d) * row_k * j->k_scale;
      dot += qd[d] * k;
    }
    s[t] = scale * dot;
    if (s[t] > m) m = s[t];
  }
  /* pass 2: weights, their sum, and the weighted sum of value rows */
  double acc[ORC_D];
  for (int d = 0; d < ORC_D; ++d) acc[d] = 0.0;
  double denom = 0.0;
  for (int t = 0; t < L; ++t) {
    double w = exp(s[t] - m);
    denom += w;
    const double row_v = j->kv_type == ORC_I8 ? orc_decode_bf16(j->kv_scales[vs_off + t]) : 1.0;
    for (int d = 0; d < ORC_D; ++d) {
      double v = orc_elem(j->kv, j->kv_type, v_off + (size_t)t * ORC_D + d) * row_v * j->v_scale;
      acc[d] += w * v;
    }
  }
  for (int d = 0; d < ORC_D; ++d) {
    double o = acc[d] / denom;
    j->out_f64[(size_t)r * ORC_D + d] = o;
    if (j->out_bits)
      j->out_bits[(size_t)r * ORC_D + d] =
          j->out_type == ORC_F16 ? orc_round_f16(o) : orc_round_bf16(o);
  }
  return ORC_OK;
}

static void* orc_worker(void* arg) {
  orc_job* j = (orc_job*)arg;
  double* s = (double*)malloc(sizeof(double) * (size_t)(j->capacity > 0 ? j->capacity : 1));
  if (!s) { j->status = ORC_ENOMEM; return NULL; }
  for (int r = j->thread_index; r < j->n_rows; r += j->n_threads) {
    int st = orc_row(j, r, s);
    if (st != ORC_OK) { j->status = st; break; }
  }
  free(s);
  return NULL;
}

/* Compute the rows listed in `rows` (each (b*q_len + j)*32 + h; NULL = all
 * batch*q_len*32 rows in order) with `n_threads` POSIX threads.  q is
 * [batch, q_len, 32, 128]; lengths must lie in [q_len, capacity].  kv_scales: bf16 bit patterns
 * [batch,2,8,capacity] for kv_type ORC_I8 (int8 codes), ignored otherwise.  Returns ORC_OK or an error code;
 * on ORC_ELENGTH nothing about the other rows is promised. */
int orc_gqa_decode(const void* q, int q_type, const void* kv, int kv_type,
                   const uint16_t* kv_scales, const int32_t* lens, int batch, int capacity,
                   int q_len, double q_scale, double k_scale, double v_scale,
                   const int32_t* rows, int n_rows,
                   double* out_f64, uint16_t* out_bits, int out_type, int n_threads) {
  if (!q || !kv || !lens || !out_f64 || batch < 1 || capacity < 1 || q_len < 1) return ORC_EINVAL;
  if ((q_type != ORC_F16 && q_type != ORC_BF16) ||
      (kv_type != ORC_F16 && kv_type != ORC_BF16 && kv_type != ORC_E4M3 && kv_type != ORC_I8) ||
      (kv_type == ORC_I8 && !kv_scales) ||
      (out_type != ORC_F16 && out_type != ORC_BF16))
    return ORC_EINVAL;
  int32_t* all = NULL;
  if (!rows) {
    n_rows = batch * q_len * ORC_HQ;
    all = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_rows);
    if (!all) return ORC_ENOMEM;
    for (int i = 0; i < n_rows; ++i) all[i] = i;
    rows = all;
  }
  for (int i = 0; i < n_rows; ++i)
    if (rows[i] < 0 || rows[i] >= batch * q_len * ORC_HQ) { free(all); return ORC_EINVAL; }
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n_rows) n_threads = n_rows > 0 ? n_rows : 1;

  orc_job* jobs = (orc_job*)calloc((size_t)n_threads, sizeof(orc_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  if (!jobs || !tids) { free(jobs); free(tids); free(all); return ORC_ENOMEM; }
  for (int t = 0; t < n_threads; ++t) {
    orc_job j = {q, q_type, kv, kv_type, kv_scales, lens, batch, capacity, q_len, q_scale, k_scale, v_scale,
                 rows, n_rows, out_f64, out_bits, out_type, n_threads, t, ORC_OK};
    jobs[t] = j;
  }
  int started = 0;
  for (int t = 1; t < n_threads; ++t) {
    if (pthread_create(&tids[t], NULL, orc_worker, &jobs[t]) != 0) break;
    started = t;
  }
  orc_worker(&jobs[0]);
  /* threads that failed to start: run their share here */
  for (int t = started + 1; t < n_threads; ++t) orc_worker(&jobs[t]);
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
  int status = ORC_OK;
  for (int t = 0; t < n_threads; ++t)
    if (jobs[t].status != ORC_OK) status = jobs[t].status;
  free(jobs);
  free(tids);
  free(all);
  return status;
}

/* ------------------------------------------------------------ K/V append */

/* The step before decode ("Qwen3-VL official BF16 on Jetson Thor (SM110)"
 * docs, "Runtime architecture": fused kernels that normalise Q and K,
 * rotate them and write the cache;
 * decode graphs keyed by (cache_pos, rope_pos)).  For one new token per batch
 * row b, each query head and each KV head vector x of 128:
 *   y_d  = x_d / sqrt(mean_e(x_e^2) + eps) * w_d            (RMS norm, weight w)
 *   a_i  = pos[b] * theta^(-i/64), i = 0..63                 (rotary angles)
 *   z_i      = y_i cos a_i - y_{i+64} sin a_i                (rotate-half RoPE)
 *   z_{i+64} = y_{i+64} cos a_i + y_i sin a_i
 * q heads use w = q_norm_w, k heads k_norm_w; v is copied unchanged.  Output
 * is FP64 (the caller rounds or quantises).  x, w are given as FP64 values. */
void orc_norm_rope(const double* x, const double* w, int pos, double eps, double theta, double* z) {
  double ss = 0.0;
  for (int d = 0; d < ORC_D; ++d) ss += x[d] * x[d];
  const double r = 1.0 / sqrt(ss / ORC_D + eps);
  double y[ORC_D];
  for (int d = 0; d < ORC_D; ++d) y[d] = x[d] * r * w[d];
  const int half = ORC_D / 2;
  for (int i = 0; i < half; ++i) {
    const double a = (double)pos * pow(theta, -(double)i / half);
    const double c = cos(a), s = sin(a);
    z[i] = y[i] * c - y[i + half] * s;
    z[i + half] = y[i + half] * c + y[i] * s;
  }
}
