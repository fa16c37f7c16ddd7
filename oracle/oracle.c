/*
 * oracle.c -- plain, slow, double-precision CPU oracle for the decoder-step
 * attention path of an encoder-decoder speech recogniser.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg load
 * it.  It shares no source, header, table or helper with the CUDA library;
 * it has its own binary16 codec, its own RMSNorm, RoPE and softmax.
 *
 * Every function computes the plain definition of its step, in double, in
 * the order the definition states.  Threads (pthreads) only split independent
 * (sequence, head) work items; they never change the order of any sum.
 *
 * Sources followed (web pages, cited by title and section):
 *  - "wavo 0.1.0, src/whisper/decoder.rs": `Buffers` doc (a cache row is K then
 *    V of all heads, as f16), `Decoder::record_step` (pack k,v into row `pos`,
 *    then attend over pos+1 rows; cross attend over all frames).
 *  - "Nest whisper-tiny, src/lib.linnet": `Attention.attend` (scores scaled by
 *    rsqrt(D/Heads)), `DecoderLayer.step` (write_at then a mask slots<=pos),
 *    `DecoderLayer.cross` (no mask), `DecoderLayer.prefill` (write_span at 0,
 *    causal mask).
 *  - "mlx-bun whisper.ts": `WhisperKvCache.rearrange` (take along the batch
 *    axis), `#attention` (k/v keep their own batch: beams share a broadcast
 *    encoder output; precise softmax; additive causal mask).
 *  - "transcribe.cpp qwen3_asr/decoder.h", header comment: per-head Q/K RMSNorm
 *    weight*rsqrt(mean(x^2)+eps)*x with eps 1e-6 after projection and before
 *    RoPE, NeoX (rotate_half) RoPE at freq_base 1e6, GQA 16 Q / 8 KV heads of
 *    128; `StepBuildBatched` (position = n_past, K/V written at row n_past,
 *    mask hides positions > n_past); `PrefillBuildBatched` (positions 0..T-1,
 *    K/V into rows [0,T), shared causal mask).
 *
 * Layout conventions (shared with the library only by specification):
 *  - f16 values are IEEE binary16 bit patterns in uint16_t.
 *  - A cache row holds 2*Hkv*hd f16: K of KV heads 0..Hkv-1, then V of KV
 *    heads 0..Hkv-1; head h sits at offset h*hd inside its half.
 *  - Query head h reads KV head h / (Hq/Hkv).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* threads: a plain parallel-for over independent work items                 */
/* ------------------------------------------------------------------------ */

static int g_threads = 1;

int orc_set_threads(int n) {
  g_threads = n < 1 ? 1 : n;
  return g_threads;
}

int orc_get_threads(void) { return g_threads; }

typedef void (*orc_item_fn)(void* ctx, int64_t item);

typedef struct {
  orc_item_fn fn;
  void* ctx;
  int64_t n_items;
  int tid, nthreads;
} orc_job;

static void* orc_worker(void* arg) {
  orc_job* j = (orc_job*)arg;
  for (int64_t i = j->tid; i < j->n_items; i += j->nthreads) j->fn(j->ctx, i);
  return NULL;
}

static void orc_parallel_for(int64_t n_items, orc_item_fn fn, void* ctx) {
  int nt = g_threads;
  if (nt > n_items) nt = (int)(n_items > 0 ? n_items : 1);
  if (nt <= 1) {
    for (int64_t i = 0; i < n_items; ++i) fn(ctx, i);
    return;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nt);
  orc_job* jobs = (orc_job*)malloc(sizeof(orc_job) * nt);
  for (int t = 0; t < nt; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].n_items = n_items;
    jobs[t].tid = t;
    jobs[t].nthreads = nt;
    pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
  }
  for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
}

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 codec (own implementation)                              */
/* ------------------------------------------------------------------------ */

/* binary16 bits -> double, exact.  Layout: 1 sign bit, 5 exponent bits (bias
 * 15), 10 fraction bits.  Exponent 0 is zero/subnormal (m * 2^-24), exponent
 * 31 is inf/NaN, otherwise (1024 + m) * 2^(e - 25). */
double orc_f16_to_f64(uint16_t h) {
  int s = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);
  return s ? -v : v;
}

/* Round half to even of a non-negative double to an integer value. */
static double orc_round_half_even(double q) {
  double fl = floor(q);
  double fr = q - fl;
  if (fr > 0.5) return fl + 1.0;
  if (fr < 0.5) return fl;
  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* double -> binary16 bits, IEEE round-to-nearest-even, overflow to +-inf.
 * Applied to a float argument (exactly representable in double) this is the
 * single rounding float -> half. */
uint16_t orc_f64_to_f16(double x) {
  uint16_t sign = (uint16_t)(signbit(x) ? 0x8000 : 0);
  double a = fabs(x);
  if (isnan(x)) return (uint16_t)(sign | 0x7e00);
  /* The largest finite half is 65504 = (2 - 2^-10) * 2^15; the midpoint to
   * the next step (65536, not representable) is 65520, which ties to even,
   * i.e. upward, so everything >= 65520 becomes infinity. */
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: units of 2^-24; a result of 1024 units is the
     * smallest normal, whose bit pattern is exactly 1024 (0x0400). */
    double q = orc_round_half_even(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)q);
  }
  int k;
  (void)frexp(a, &k); /* a = f * 2^k, f in [0.5, 1) => a in [2^(k-1), 2^k) */
  int E = k - 1;      /* unbiased exponent */
  double q = orc_round_half_even(ldexp(a, 10 - E)); /* in [1024, 2048] */
  if (q >= 2048.0) {
    q = 1024.0;
    E += 1;
  }
  if (E + 15 >= 31) return (uint16_t)(sign | 0x7c00);
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)q - 1024));
}

uint16_t orc_f32_to_f16(float x) { return orc_f64_to_f16((double)x); }

void orc_f16_decode_array(const uint16_t* h, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f64(h[i]);
}

void orc_f32_encode_array(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
}

void orc_f64_encode_array(const double* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_f16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Attention of one query over L cached rows: the plain definition           */
/* ------------------------------------------------------------------------ */

/* z_j = scale * sum_d q_d K_j[d]  (j < L);  p = softmax(z);
 * out_d = sum_j p_j V_j[d].
 * k0 / v0 point at row 0's K / V segment of the head; consecutive rows are
 * row_stride f16 apart.  Softmax as its definition with the maximum
 * subtracted first (exp(z - m) / sum exp(z - m) equals exp(z) / sum exp(z)).
 * Scratch z must hold L doubles. */
void orc_attend_one(const double* q, const uint16_t* k0, const uint16_t* v0, int64_t row_stride,
                    int L, int hd, double scale, double* z, double* out) {
  double m = -INFINITY;
  for (int j = 0; j < L; ++j) {
    const uint16_t* kj = k0 + (int64_t)j * row_stride;
    double dot = 0.0;
    for (int d = 0; d < hd; ++d) dot += q[d] * orc_f16_to_f64(kj[d]);
    z[j] = scale * dot;
    if (z[j] > m) m = z[j];
  }
  double den = 0.0;
  for (int j = 0; j < L; ++j) {
    z[j] = exp(z[j] - m);
    den += z[j];
  }
  for (int d = 0; d < hd; ++d) out[d] = 0.0;
  for (int j = 0; j < L; ++j) {
    const uint16_t* vj = v0 + (int64_t)j * row_stride;
    double p = z[j] / den;
    for (int d = 0; d < hd; ++d) out[d] += p * orc_f16_to_f64(vj[d]);
  }
}

/* ------------------------------------------------------------------------ */
/* a1: K/V append                                                            */
/* ------------------------------------------------------------------------ */

/* wavo record_step packs the new token's k and v (floats) into cache row
 * `pos` as f16; lib.linnet DecoderLayer.step does write_at(self_k/self_v,
 * pos).  Row slot[b] of sequence b becomes f16(k_b) || f16(v_b).
 * Sequences with slot outside [0, capacity) are skipped; the count of skipped
 * sequences is returned. */
int orc_kv_append(const float* k, const float* v, int64_t src_row_stride, uint16_t* cache,
                  int64_t seq_stride, const int32_t* slot, int B, int kv_heads, int head_dim,
                  int capacity) {
  int64_t half = (int64_t)kv_heads * head_dim;
  int skipped = 0;
  for (int b = 0; b < B; ++b) {
    int s = slot[b];
    if (s < 0 || s >= capacity) {
      ++skipped;
      continue;
    }
    uint16_t* row = cache + (int64_t)b * seq_stride + (int64_t)s * 2 * half;
    for (int64_t i = 0; i < half; ++i) row[i] = orc_f32_to_f16(k[(int64_t)b * src_row_stride + i]);
    for (int64_t i = 0; i < half; ++i)
      row[half + i] = orc_f32_to_f16(v[(int64_t)b * src_row_stride + i]);
  }
  return skipped;
}

/* ------------------------------------------------------------------------ */
/* a2 / a3: self- and cross-attention of one new token per sequence          */
/* ------------------------------------------------------------------------ */

typedef struct {
  const float* q;
  int64_t q_stride;
  const uint16_t* kv;
  int64_t src_stride;
  const int32_t* src_of_seq; /* NULL: source = sequence */
  const int32_t* lens;       /* NULL: every source has L_fixed rows */
  int L_fixed, n_src, max_rows;
  int q_heads, kv_heads, head_dim;
  double scale;
  double* out; /* [B][q_heads*head_dim] */
  int* bad;    /* per sequence: 1 if skipped */
} orc_decode_ctx;

static void orc_decode_item(void* vctx, int64_t item) {
  orc_decode_ctx* c = (orc_decode_ctx*)vctx;
  int b = (int)(item / c->q_heads);
  int h = (int)(item % c->q_heads);
  int hd = c->head_dim;
  double* o = c->out + ((int64_t)b * c->q_heads + h) * hd;
  int src = c->src_of_seq ? c->src_of_seq[b] : b;
  int L = c->lens ? c->lens[b] : c->L_fixed;
  if (src < 0 || src >= c->n_src || L < 1 || L > c->max_rows) {
    for (int d = 0; d < hd; ++d) o[d] = 0.0;
    c->bad[b] = 1;
    return;
  }
  int kvh = h / (c->q_heads / c->kv_heads);
  int64_t row = 2LL * c->kv_heads * hd;
  const uint16_t* base = c->kv + (int64_t)src * c->src_stride;
  double* q = (double*)malloc(sizeof(double) * hd);
  double* z = (double*)malloc(sizeof(double) * L);
  for (int d = 0; d < hd; ++d) q[d] = (double)c->q[(int64_t)b * c->q_stride + (int64_t)h * hd + d];
  orc_attend_one(q, base + (int64_t)kvh * hd, base + (int64_t)c->kv_heads * hd + (int64_t)kvh * hd,
                 row, L, hd, c->scale, z, o);
  free(q);
  free(z);
}

static int orc_count_bad(const int* bad, int B) {
  int n = 0;
  for (int b = 0; b < B; ++b) n += bad[b] != 0;
  return n;
}

/* Causal self-attention of the new token: wavo `attend(q, own, pos+1)`;
 * lib.linnet DecoderLayer.step masks slots > pos.  lens[b] counts the keys the
 * token attends, its own included (rows [0, lens[b]) of sequence b).  MHA:
 * one KV head per query head.  Returns the number of skipped sequences
 * (lens outside [1, capacity]); their output is 0. */
int orc_self_attn_step(const float* q, int64_t q_stride, const uint16_t* cache, int64_t seq_stride,
                       const int32_t* lens, int B, int heads, int head_dim, int capacity,
                       double scale, double* out) {
  int* bad = (int*)calloc(B > 0 ? B : 1, sizeof(int));
  orc_decode_ctx c = {q, q_stride, cache, seq_stride, NULL, lens, 0, B, capacity,
                      heads, heads, head_dim, scale, out, bad};
  orc_parallel_for((int64_t)B * heads, orc_decode_item, &c);
  int n = orc_count_bad(bad, B);
  free(bad);
  return n;
}

/* Cross-attention over the encoder's cached K/V: wavo `attend(q, cross,
 * frames)`; lib.linnet DecoderLayer.cross uses no mask.  Sequence b reads the
 * rows of group[b] (mlx-bun #attention: beams attend one broadcast encoder
 * output).  Returns the number of skipped sequences (group outside [0,G)). */
int orc_cross_attn_step(const float* q, int64_t q_stride, const uint16_t* cross,
                        int64_t group_stride, const int32_t* group, int B, int G, int heads,
                        int head_dim, int frames, double scale, double* out) {
  int* bad = (int*)calloc(B > 0 ? B : 1, sizeof(int));
  orc_decode_ctx c = {q, q_stride, cross, group_stride, group, NULL, frames, G, frames,
                      heads, heads, head_dim, scale, out, bad};
  orc_parallel_for((int64_t)B * heads, orc_decode_item, &c);
  int n = orc_count_bad(bad, B);
  free(bad);
  return n;
}

/* ------------------------------------------------------------------------ */
/* a5: per-head RMSNorm + NeoX RoPE + GQA step                               */
/* ------------------------------------------------------------------------ */

/* transcribe.cpp decoder.h: RMSNorm is weight * rsqrt(mean(x^2) + eps) * x,
 * over head_dim for the per-head Q/K norm. */
void orc_rmsnorm(const double* x, const double* w, double eps, int n, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) y[i] = w[i] * (x[i] * r);
}

/* NeoX-style rotary embedding (rotate_half) at position pos: frequency
 * theta_i = base^(-2i/hd) for i in [0, hd/2); the pair (i, i + hd/2) turns by
 * the angle pos*theta_i:
 *   y_i        = x_i cos - x_{i+hd/2} sin
 *   y_{i+hd/2} = x_{i+hd/2} cos + x_i sin            */
void orc_rope_neox(const double* x, int hd, double pos, double base, double* y) {
  int half = hd / 2;
  for (int i = 0; i < half; ++i) {
    double theta = pow(base, -2.0 * i / hd);
    double a = pos * theta;
    double c = cos(a), s = sin(a);
    y[i] = x[i] * c - x[i + half] * s;
    y[i + half] = x[i + half] * c + x[i] * s;
  }
}

typedef struct {
  const float* q;
  const uint16_t* cache;
  int64_t seq_stride;
  const int32_t* n_past;
  const double* wq;
  double eps, base, scale;
  int q_heads, kv_heads, head_dim, capacity;
  double* out;
  const int* bad;
} orc_gqa_ctx;

static void orc_gqa_item(void* vctx, int64_t item) {
  orc_gqa_ctx* c = (orc_gqa_ctx*)vctx;
  int b = (int)(item / c->q_heads);
  int h = (int)(item % c->q_heads);
  int hd = c->head_dim;
  double* o = c->out + ((int64_t)b * c->q_heads + h) * hd;
  if (c->bad[b]) {
    for (int d = 0; d < hd; ++d) o[d] = 0.0;
    return;
  }
  int p = c->n_past[b];
  int L = p + 1;
  double* x = (double*)malloc(sizeof(double) * hd);
  double* xn = (double*)malloc(sizeof(double) * hd);
  double* qr = (double*)malloc(sizeof(double) * hd);
  double* z = (double*)malloc(sizeof(double) * L);
  for (int d = 0; d < hd; ++d) x[d] = (double)c->q[((int64_t)b * c->q_heads + h) * hd + d];
  orc_rmsnorm(x, c->wq, c->eps, hd, xn);
  orc_rope_neox(xn, hd, (double)p, c->base, qr);
  int kvh = h / (c->q_heads / c->kv_heads);
  int64_t row = 2LL * c->kv_heads * hd;
  const uint16_t* base = c->cache + (int64_t)b * c->seq_stride;
  orc_attend_one(qr, base + (int64_t)kvh * hd, base + (int64_t)c->kv_heads * hd + (int64_t)kvh * hd,
                 row, L, hd, c->scale, z, o);
  free(x);
  free(xn);
  free(qr);
  free(z);
}

/* One Qwen3-ASR-style decode step (decoder.h StepBuildBatched): for sequence
 * b at position p = n_past[b]:
 *   k^ = RoPE(RMSNorm(k_new, w_k), p), v = v_new  -> cache row p = f16(k^)||f16(v)
 *   q^ = RoPE(RMSNorm(q, w_q), p)                 (kept in double, not rounded)
 *   out = attention of q^ over rows [0, p] (keys up to and including p).
 * q: [B][q_heads*hd], k_new / v_new: [B][kv_heads*hd].  Sequences with
 * n_past outside [0, capacity) are skipped (output 0, cache untouched). */
int orc_gqa_step(const float* q, const float* k_new, const float* v_new, const float* q_norm_w,
                 const float* k_norm_w, double eps, double rope_base, const int32_t* n_past,
                 uint16_t* cache, int64_t seq_stride, int capacity, int B, int q_heads,
                 int kv_heads, int head_dim, double scale, double* out) {
  int hd = head_dim;
  double* wq = (double*)malloc(sizeof(double) * hd);
  double* wk = (double*)malloc(sizeof(double) * hd);
  double* x = (double*)malloc(sizeof(double) * hd);
  double* xn = (double*)malloc(sizeof(double) * hd);
  double* xr = (double*)malloc(sizeof(double) * hd);
  int* bad = (int*)calloc(B > 0 ? B : 1, sizeof(int));
  for (int d = 0; d < hd; ++d) {
    wq[d] = q_norm_w[d];
    wk[d] = k_norm_w[d];
  }
  int64_t half = (int64_t)kv_heads * hd;
  for (int b = 0; b < B; ++b) {
    int p = n_past[b];
    if (p < 0 || p >= capacity) {
      bad[b] = 1;
      continue;
    }
    uint16_t* row = cache + (int64_t)b * seq_stride + (int64_t)p * 2 * half;
    for (int h = 0; h < kv_heads; ++h) {
      for (int d = 0; d < hd; ++d) x[d] = (double)k_new[(int64_t)b * half + (int64_t)h * hd + d];
      orc_rmsnorm(x, wk, eps, hd, xn);
      orc_rope_neox(xn, hd, (double)p, rope_base, xr);
      for (int d = 0; d < hd; ++d) row[(int64_t)h * hd + d] = orc_f64_to_f16(xr[d]);
      for (int d = 0; d < hd; ++d)
        row[half + (int64_t)h * hd + d] = orc_f32_to_f16(v_new[(int64_t)b * half + (int64_t)h * hd + d]);
    }
  }
  orc_gqa_ctx c = {q, cache, seq_stride, n_past, wq, eps, rope_base, scale,
                   q_heads, kv_heads, hd, capacity, out, bad};
  orc_parallel_for((int64_t)B * q_heads, orc_gqa_item, &c);
  int n = orc_count_bad(bad, B);
  free(wq);
  free(wk);
  free(x);
  free(xn);
  free(xr);
  free(bad);
  return n;
}

/* ------------------------------------------------------------------------ */
/* a6: beam reorder                                                          */
/* ------------------------------------------------------------------------ */

/* mlx-bun WhisperKvCache.rearrange: keep rows `indices` of every layer's
 * self K/V (take along the batch axis) into a new array.  Here the cache of
 * beam b becomes the history of beam idx[b]: the lens_src[idx[b]] - 1 rows
 * written before the coming step's token, in every one of n_layers layers
 * (layer l of sequence s starts at s*seq_stride + l*layer_stride).  lens_dst[b]
 * = lens_src[idx[b]].  Beams with idx outside [0,B) or a source length outside
 * [1, capacity] are skipped with lens_dst[b] = 0.  Returns the skip count. */
int orc_kv_rearrange(const uint16_t* src, uint16_t* dst, int64_t seq_stride, int64_t layer_stride,
                     int n_layers, int row_elems, int capacity, const int32_t* idx,
                     const int32_t* lens_src, int32_t* lens_dst, int B) {
  int skipped = 0;
  for (int b = 0; b < B; ++b) {
    int s = idx[b];
    if (s < 0 || s >= B || lens_src[s] < 1 || lens_src[s] > capacity) {
      lens_dst[b] = 0;
      ++skipped;
      continue;
    }
    int64_t n = (int64_t)(lens_src[s] - 1) * row_elems;
    for (int l = 0; l < n_layers; ++l) {
      const uint16_t* from = src + (int64_t)s * seq_stride + (int64_t)l * layer_stride;
      uint16_t* to = dst + (int64_t)b * seq_stride + (int64_t)l * layer_stride;
      for (int64_t i = 0; i < n; ++i) to[i] = from[i];
    }
    lens_dst[b] = lens_src[s];
  }
  return skipped;
}

/* ------------------------------------------------------------------------ */
/* a7 / a8: batched prefill (norm + RoPE + cache write, causal attention)     */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t* qhat; /* [B][T][q_heads*hd] f16, normed + roped + rounded */
  const uint16_t* cache;
  int64_t seq_stride;
  int B, T, q_heads, kv_heads, head_dim;
  double scale;
  double* out; /* [B][T][q_heads*hd] */
} orc_prefill_ctx;

static void orc_prefill_item(void* vctx, int64_t item) {
  orc_prefill_ctx* c = (orc_prefill_ctx*)vctx;
  int hd = c->head_dim;
  int b = (int)(item / c->q_heads);
  int h = (int)(item % c->q_heads);
  int kvh = h / (c->q_heads / c->kv_heads);
  int64_t row = 2LL * c->kv_heads * hd;
  const uint16_t* base = c->cache + (int64_t)b * c->seq_stride;
  double* q = (double*)malloc(sizeof(double) * hd);
  double* z = (double*)malloc(sizeof(double) * c->T);
  for (int t = 0; t < c->T; ++t) {
    const uint16_t* qh = c->qhat + (((int64_t)b * c->T + t) * c->q_heads + h) * hd;
    for (int d = 0; d < hd; ++d) q[d] = orc_f16_to_f64(qh[d]);
    double* o = c->out + (((int64_t)b * c->T + t) * c->q_heads + h) * hd;
    /* causal: query t sees keys 0..t */
    orc_attend_one(q, base + (int64_t)kvh * hd, base + (int64_t)c->kv_heads * hd + (int64_t)kvh * hd,
                   row, t + 1, hd, c->scale, z, o);
  }
  free(q);
  free(z);
}

/* Prefill preparation (decoder.h build_prefill_graph_batched: positions
 * 0..T-1, K/V into rows [0, T)): every prompt position t in [0,T) of every
 * sequence gets q^ = f16(RoPE(RMSNorm(q, w_q), t)) and
 * k^ = f16(RoPE(RMSNorm(k, w_k), t)); cache row t = k^ || v (v copied as
 * given).  q, k, v are f16 [B][T][H*hd]; qhat receives q^ [B][T][Hq*hd].
 * The f16 rounding of q^ and k^ is part of the definition here because they
 * are the f16 matrix operands.  Returns 0, or -1 if T > capacity. */
int orc_prefill_prep(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const float* q_norm_w, const float* k_norm_w, double eps, double rope_base,
                     int B, int T, int q_heads, int kv_heads, int head_dim, uint16_t* cache,
                     int64_t seq_stride, int capacity, uint16_t* qhat) {
  if (T > capacity) return -1;
  int hd = head_dim;
  int64_t qw = (int64_t)q_heads * hd, kw = (int64_t)kv_heads * hd;
  double* wq = (double*)malloc(sizeof(double) * hd);
  double* wk = (double*)malloc(sizeof(double) * hd);
  double* x = (double*)malloc(sizeof(double) * hd);
  double* xn = (double*)malloc(sizeof(double) * hd);
  double* xr = (double*)malloc(sizeof(double) * hd);
  for (int d = 0; d < hd; ++d) {
    wq[d] = q_norm_w[d];
    wk[d] = k_norm_w[d];
  }
  for (int b = 0; b < B; ++b) {
    for (int t = 0; t < T; ++t) {
      for (int h = 0; h < q_heads; ++h) {
        const uint16_t* src = q + ((int64_t)b * T + t) * qw + (int64_t)h * hd;
        for (int d = 0; d < hd; ++d) x[d] = orc_f16_to_f64(src[d]);
        orc_rmsnorm(x, wq, eps, hd, xn);
        orc_rope_neox(xn, hd, (double)t, rope_base, xr);
        uint16_t* dq = qhat + ((int64_t)b * T + t) * qw + (int64_t)h * hd;
        for (int d = 0; d < hd; ++d) dq[d] = orc_f64_to_f16(xr[d]);
      }
      uint16_t* row = cache + (int64_t)b * seq_stride + (int64_t)t * 2 * kw;
      for (int h = 0; h < kv_heads; ++h) {
        const uint16_t* src = k + ((int64_t)b * T + t) * kw + (int64_t)h * hd;
        for (int d = 0; d < hd; ++d) x[d] = orc_f16_to_f64(src[d]);
        orc_rmsnorm(x, wk, eps, hd, xn);
        orc_rope_neox(xn, hd, (double)t, rope_base, xr);
        for (int d = 0; d < hd; ++d) row[(int64_t)h * hd + d] = orc_f64_to_f16(xr[d]);
      }
      const uint16_t* vs = v + ((int64_t)b * T + t) * kw;
      for (int64_t i = 0; i < kw; ++i) row[kw + i] = vs[i];
    }
  }
  free(wq);
  free(wk);
  free(x);
  free(xn);
  free(xr);
  return 0;
}

/* Batched prefill (decoder.h build_prefill_graph_batched; lib.linnet
 * DecoderLayer.prefill): orc_prefill_prep, then causal attention of q^ at
 * position t over cache rows [0, t] for every t, sequence and query head.
 * qhat_out (may be NULL) receives q^.  Returns 0, or -1 if T > capacity. */
int orc_prefill_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const float* q_norm_w, const float* k_norm_w, double eps, double rope_base,
                     int B, int T, int q_heads, int kv_heads, int head_dim, double scale,
                     uint16_t* cache, int64_t seq_stride, int capacity, double* out,
                     uint16_t* qhat_out) {
  if (T > capacity) return -1;
  int64_t qw = (int64_t)q_heads * head_dim;
  uint16_t* qhat = qhat_out ? qhat_out : (uint16_t*)malloc(sizeof(uint16_t) * (size_t)B * T * qw);
  orc_prefill_prep(q, k, v, q_norm_w, k_norm_w, eps, rope_base, B, T, q_heads, kv_heads,
                   head_dim, cache, seq_stride, capacity, qhat);
  orc_prefill_ctx c = {qhat, cache, seq_stride, B, T, q_heads, kv_heads, head_dim, scale, out};
  orc_parallel_for((int64_t)B * q_heads, orc_prefill_item, &c);
  if (!qhat_out) free(qhat);
  return 0;
}

/* Causal attention only, for a sample of query positions of one (b, head):
 * queries q^ given as f16 rows (already normed, roped, rounded), keys/values
 * from the cache rows.  Used to check single outputs of a large prefill. */
void orc_prefill_attn_rows(const uint16_t* qhat_rows, const int32_t* t_of_row, int n_rows,
                           const uint16_t* seq_cache, int q_heads, int kv_heads, int head_dim,
                           int head, double scale, double* out) {
  int hd = head_dim;
  int kvh = head / (q_heads / kv_heads);
  int64_t row = 2LL * kv_heads * hd;
  double* q = (double*)malloc(sizeof(double) * hd);
  int maxT = 0;
  for (int i = 0; i < n_rows; ++i)
    if (t_of_row[i] + 1 > maxT) maxT = t_of_row[i] + 1;
  double* z = (double*)malloc(sizeof(double) * (maxT > 0 ? maxT : 1));
  for (int i = 0; i < n_rows; ++i) {
    for (int d = 0; d < hd; ++d) q[d] = orc_f16_to_f64(qhat_rows[(int64_t)i * hd + d]);
    orc_attend_one(q, seq_cache + (int64_t)kvh * hd,
                   seq_cache + (int64_t)kv_heads * hd + (int64_t)kvh * hd, row, t_of_row[i] + 1,
                   hd, scale, z, out + (int64_t)i * hd);
  }
  free(q);
  free(z);
}

/* ------------------------------------------------------------------------ */
/* Next rows: MHA prompt prefill with per-sequence lengths, and the         */
/* encoder's unmasked self-attention                                        */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* lens;
  int B, T, heads, head_dim, causal;
  double scale;
  double* out;
} orc_mha_ctx;

static void orc_mha_item(void* vctx, int64_t item) {
  orc_mha_ctx* c = (orc_mha_ctx*)vctx;
  int hd = c->head_dim;
  int b = (int)(item / c->heads);
  int h = (int)(item % c->heads);
  int L = c->lens ? c->lens[b] : c->T;
  int64_t row = (int64_t)c->heads * hd; /* q, k, v rows: all heads of one position */
  const uint16_t* kb = c->k + (int64_t)b * c->T * row + (int64_t)h * hd;
  const uint16_t* vb = c->v + (int64_t)b * c->T * row + (int64_t)h * hd;
  double* q = (double*)malloc(sizeof(double) * hd);
  double* z = (double*)malloc(sizeof(double) * (L > 0 ? L : 1));
  for (int t = 0; t < L; ++t) {
    const uint16_t* qt = c->q + ((int64_t)b * c->T + t) * row + (int64_t)h * hd;
    for (int d = 0; d < hd; ++d) q[d] = orc_f16_to_f64(qt[d]);
    double* o = c->out + ((int64_t)b * c->T + t) * row + (int64_t)h * hd;
    /* causal: query t sees keys 0..t; unmasked: every real key 0..L-1 */
    orc_attend_one(q, kb, vb, row, c->causal ? t + 1 : L, hd, c->scale, z, o);
  }
  free(q);
  free(z);
}

/* Multi-head attention of the positions of a batch of sequences among
 * themselves, with the f16 q, k, v as the matrix operands:
 *  - causal = 1: the decoder's prompt prefill ("Nest whisper-tiny,
 *    src/lib.linnet", DecoderLayer.prefill: the S prompt tokens' keys and
 *    values go to cache rows [0, S) and they attend causally among
 *    themselves);
 *  - causal = 0: the encoder's self-attention (EncoderLayer.forward: every
 *    audio frame attends to every other, padding included, no mask).
 * q, k, v: f16 [B][T][heads*hd].  lens[b] (NULL: T for every sequence) is
 * the number of real positions of sequence b ("transcribe.cpp,
 * decoder.h", PrefillBuildBatched: prompts of up to T_prompt_max tokens,
 * each with its own last real position): query t < lens[b] attends keys
 * j < lens[b] (j <= t when causal); out rows t >= lens[b] are not written.
 * cache (may be NULL): rows [0, lens[b]) of sequence b receive k || v, the
 * row layout of the decoder's self cache.  Returns the number of sequences
 * skipped for a length outside [0, T], or -1 if T > capacity. */
int orc_mha_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* lens,
                 int B, int T, int heads, int head_dim, double scale, int causal, uint16_t* cache,
                 int64_t seq_stride, int capacity, double* out) {
  if (cache && T > capacity) return -1;
  int bad = 0;
  int32_t* L = (int32_t*)malloc(sizeof(int32_t) * (B > 0 ? B : 1));
  for (int b = 0; b < B; ++b) {
    int lb = lens ? lens[b] : T;
    if (lb < 0 || lb > T) {
      ++bad;
      lb = 0;
    }
    L[b] = lb;
  }
  int64_t row = (int64_t)heads * head_dim;
  if (cache) {
    for (int b = 0; b < B; ++b) {
      for (int t = 0; t < L[b]; ++t) {
        uint16_t* dst = cache + (int64_t)b * seq_stride + (int64_t)t * 2 * row;
        const uint16_t* ks = k + ((int64_t)b * T + t) * row;
        const uint16_t* vs = v + ((int64_t)b * T + t) * row;
        for (int64_t i = 0; i < row; ++i) {
          dst[i] = ks[i];
          dst[row + i] = vs[i];
        }
      }
    }
  }
  orc_mha_ctx c = {q, k, v, L, B, T, heads, head_dim, causal, scale, out};
  orc_parallel_for((int64_t)B * heads, orc_mha_item, &c);
  free(L);
  return bad;
}

/* ------------------------------------------------------------------------ */
/* Next row: the cross K/V fill                                             */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t* enc;
  const uint16_t* w;
  const float* bias_v;
  int frames, d;
  uint16_t* cross;
  int64_t group_stride;
} orc_fill_ctx;

static void orc_fill_item(void* vctx, int64_t item) {
  orc_fill_ctx* c = (orc_fill_ctx*)vctx;
  int d = c->d;
  int64_t g = item / c->frames;
  int t = (int)(item % c->frames);
  const uint16_t* e = c->enc + (g * c->frames + t) * (int64_t)d;
  uint16_t* row = c->cross + g * c->group_stride + (int64_t)t * 2 * d;
  double* x = (double*)malloc(sizeof(double) * d);
  for (int k = 0; k < d; ++k) x[k] = orc_f16_to_f64(e[k]);
  for (int n = 0; n < 2 * d; ++n) {
    const uint16_t* wn = c->w + (int64_t)n * d;
    double acc = 0.0;
    for (int k = 0; k < d; ++k) acc += x[k] * orc_f16_to_f64(wn[k]);
    if (n >= d) acc += (double)c->bias_v[n - d]; /* k has no bias */
    row[n] = orc_f64_to_f16(acc);
  }
  free(x);
}

/* The cross-attention K and V of one layer from the encoder output
 * ("wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_cross: a GEMM of
 * the encoder rows with the layer's [k | v] weight and a bias epilogue,
 * then a pack to f16 cache rows; Decoder::load: the bias of k is zero, v
 * has its own; "Nest whisper-tiny, src/lib.linnet", DecoderLayer.listen).
 *   cross row t of group g = f16(enc[g][t] . W^T + [0 | bias_v]),
 *   i.e. element n is sum_k enc[g][t][k] * W[n][k] (+ bias_v[n - d] for
 *   n >= d): the first d elements are K of all heads, the last d are V.
 * enc: f16 [G][frames][d]; W: f16 [2d][d] (row n makes output column n);
 * bias_v: fp32 [d]; cross: f16 [G][group_stride], rows of 2d. */
void orc_cross_kv_fill(const uint16_t* enc, const uint16_t* w, const float* bias_v, int G,
                       int frames, int d, uint16_t* cross, int64_t group_stride) {
  orc_fill_ctx c = {enc, w, bias_v, frames, d, cross, group_stride};
  orc_parallel_for((int64_t)G * frames, orc_fill_item, &c);
}

/* ------------------------------------------------------------------------ */
/* Next row: the dense steps of a decoder layer around the attention         */
/* ------------------------------------------------------------------------ */

/* LayerNorm of one row of K values ("Nest whisper-tiny, src/lib.linnet",
 * LayerNorm: torch.nn.LayerNorm's definition with its default eps 1e-5):
 *   mean = sum_k x_k / K,  var = sum_k (x_k - mean)^2 / K  (biased),
 *   y_k = (x_k - mean) / sqrt(var + eps) * g_k + b_k. */
void orc_layer_norm(const float* x, int64_t K, const float* g, const float* b, double eps,
                    double* y) {
  double mean = 0.0;
  for (int64_t k = 0; k < K; ++k) mean += (double)x[k];
  mean /= (double)K;
  double var = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    double dx = (double)x[k] - mean;
    var += dx * dx;
  }
  var /= (double)K;
  double inv = 1.0 / sqrt(var + eps);
  for (int64_t k = 0; k < K; ++k) y[k] = ((double)x[k] - mean) * inv * (double)g[k] + (double)b[k];
}

/* GELU in its error-function form (Whisper's config asks for `gelu`, the
 * exact one; "Nest whisper-tiny, src/lib.linnet" uses gelu_erf):
 *   gelu(v) = v * Phi(v) = v / 2 * (1 + erf(v / sqrt(2))). */
double orc_gelu_erf(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }

/* SiLU, the gate of the SwiGLU MLP ("transcribe.cpp,
 * src/arch/qwen3_asr/decoder.h", header comment: down_proj(silu(gate_proj(x))
 * * up_proj(x))): silu(v) = v * sigmoid(v) = v / (1 + e^-v). */
double orc_silu(double v) { return v / (1.0 + exp(-v)); }

typedef struct {
  const float* x;
  int64_t x_stride;
  int K, N;
  int norm; /* 0 none, 1 LayerNorm, 2 RMSNorm */
  const float* ln_g;
  const float* ln_b;
  double eps;
  int act; /* 0 none, 1 SwiGLU input */
  const double* w; /* decoded weights [N][K] */
  const float* bias;
  int mode;
  double* y;
  int64_t y_stride;
} orc_linear_ctx;

static void orc_linear_item(void* vctx, int64_t m) {
  orc_linear_ctx* c = (orc_linear_ctx*)vctx;
  const float* xm = c->x + m * c->x_stride;
  double* a = (double*)malloc(sizeof(double) * c->K);
  if (c->norm == 1) {
    orc_layer_norm(xm, c->K, c->ln_g, c->ln_b, c->eps, a);
  } else if (c->norm == 2) {
    double* xd = (double*)malloc(sizeof(double) * c->K);
    double* wd = (double*)malloc(sizeof(double) * c->K);
    for (int k = 0; k < c->K; ++k) {
      xd[k] = (double)xm[k];
      wd[k] = (double)c->ln_g[k];
    }
    orc_rmsnorm(xd, wd, c->eps, c->K, a);
    free(xd);
    free(wd);
  } else if (c->act == 1) {
    for (int k = 0; k < c->K; ++k) a[k] = orc_silu((double)xm[k]) * (double)xm[c->K + k];
  } else {
    for (int k = 0; k < c->K; ++k) a[k] = (double)xm[k];
  }
  double* ym = c->y + m * c->y_stride;
  for (int n = 0; n < c->N; ++n) {
    const double* wn = c->w + (int64_t)n * c->K;
    double v = 0.0;
    for (int k = 0; k < c->K; ++k) v += a[k] * wn[k];
    if (c->bias) v += (double)c->bias[n];
    if (c->mode == 1) {
      ym[n] += v; /* Residual(1.0): added onto what y holds */
    } else if (c->mode == 2) {
      ym[n] = orc_gelu_erf(v);
    } else {
      ym[n] = v;
    }
  }
  free(a);
}

/* One dense step of a decoder layer ("wavo 0.1.0, src/whisper/decoder.rs",
 * Decoder::record_step: `layer_norm` into y, then `gemv` of y with a weight
 * and one of the epilogues Bias, Residual(1.0) or Gelu; "transcribe.cpp,
 * src/arch/qwen3_asr/decoder.h", header comment: pre-norm RMSNorm and the
 * SwiGLU MLP):
 *   a_m = LayerNorm(x_m; ln_g, ln_b, eps) (norm 1), RMSNorm(x_m; ln_g, eps)
 *         (norm 2), silu(x_m[0..K)) * x_m[K..2K) (act 1, no norm), else x_m;
 *   v_mn = sum_k a_mk * W[n][k] + bias_n  (bias may be NULL: 0);
 *   mode 0: y_mn = v_mn;  mode 1: y_mn = y_mn + v_mn;  mode 2: y_mn = gelu(v_mn).
 * x: fp32 [M][x_stride] (K used); W: f16 [N][K] (row n makes output n);
 * y: double [M][y_stride].  The activations are used as their fp32 values
 * (the pages' buffers are f32); every sum is in double. */
void orc_linear(const float* x, int64_t x_stride, int M, int K, int norm, const float* ln_g,
                const float* ln_b, double eps, int act, const uint16_t* w, int N, const float* bias,
                int mode, double* y, int64_t y_stride) {
  double* wd = (double*)malloc(sizeof(double) * (size_t)N * (size_t)K);
  for (int64_t i = 0; i < (int64_t)N * K; ++i) wd[i] = orc_f16_to_f64(w[i]);
  orc_linear_ctx c = {x, x_stride, K, N, norm, ln_g, ln_b, eps, act, wd, bias, mode, y, y_stride};
  orc_parallel_for(M, orc_linear_item, &c);
  free(wd);
}
