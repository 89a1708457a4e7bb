/*
 * gqa_oracle.c -- plain, slow, fp64 CPU oracle for grouped-query attention
 * over a KV cache (head_dim 128, 32 query heads, 8 KV heads).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant generator
 * with the CUDA library: every format below is decoded from its published bit
 * definition, and every attention result is the textbook softmax written out.
 *
 * Sources (page titles of the material this library restates):
 *  - "NVIDIA SM110 GPU를 위한 실험적인 FP16 GQA 디코드 커널 추가" (FlashInfer
 *    PR #5052 analysis), section 1 (the sm110_gqa_decode API docstring:
 *    q [batch,32,128], kv [batch,2,8,capacity,128], int32 sequence_lengths,
 *    the caller's q_scale in front of the usual 1/sqrt(128) factor),
 *    section 2 (fixed 32/8/128 configuration) and section 3 (the SDPA
 *    comparator with enable_gqa=True, scale 1/sqrt(128)).
 *  - "GB300 NVFP4 Context Attention: scale slot 조기 반납과 8단 packed K/V
 *    ring" (FlashInfer PR #9177 analysis), introduction: FP8-E4M3 query and
 *    output, NVFP4 K/V pages with E4M3 block scales dequantised to E4M3,
 *    head dim 128, bottom-right causal mask, HND page layout.
 *
 * Readings taken where the pages are silent:
 *  - GQA head mapping: query head h reads KV head h / 4 (contiguous groups,
 *    the enable_gqa convention of the SDPA comparator).
 *  - A decode length of 0 yields a zero row; lengths are clamped to
 *    [0, capacity].
 *  - E2M1 nibble order: element 2i sits in the low nibble of byte i.
 *  - Block scale layout: sf[page, kv_head, slot, d / 16], same HND order as
 *    the data.
 *  - Dequantisation target: the exact product e2m1(code) * e4m3(scale) is
 *    rounded to E4M3, round-to-nearest-even, saturating at +-448.
 *  - Context attention scale: q_scale / sqrt(128), as for decode.  The output
 *    is O / out_scale (the caller dequantises with out = out_fp8 * out_scale).
 *    A query row that sees no key yields a zero row.
 *
 * Threading: work is split over independent (row, head) items with pthreads;
 * each item is computed start to finish by one thread with no blocking or
 * reordering of its arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_HQ 32
#define ORACLE_HKV 8
#define ORACLE_D 128
#define ORACLE_PAGE 64

/* ------------------------------------------------------------------------ */
/* Number formats, decoded from their bit definitions.                      */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 mantissa bits. */
double oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0x1f) {
    v = (m == 0) ? INFINITY : NAN;
  } else if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-14 * 2^-10 */
  } else {
    v = ldexp(1.0 + (double)m / 1024.0, e - 15);
  }
  return sign ? -v : v;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; no infinities; S.1111.111 is NaN; largest finite 448; subnormals
 * m * 2^-9. */
double oracle_e4m3_to_f64(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xf;
  int m = c & 0x7;
  double v;
  if (e == 0xf && m == 0x7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)m, -9);
  } else {
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  return sign ? -v : v;
}

/* OCP FP4 E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0
 * is subnormal with value m * 0.5.  Gives {0, 0.5, 1, 1.5, 2, 3, 4, 6}. */
double oracle_e2m1_to_f64(uint8_t nib) {
  int sign = (nib >> 3) & 1;
  int e = (nib >> 1) & 0x3;
  int m = nib & 0x1;
  double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
  return sign ? -v : v;
}

/* Round a non-negative double that is a multiple of 1/2 or finer to the
 * nearest integer, ties to even. */
static double round_half_even(double y) {
  double f = floor(y);
  double r = y - f;
  if (r > 0.5) return f + 1.0;
  if (r < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* Encode to E4M3 with round-to-nearest-even, saturating finite values to
 * +-448 (the "satfinite" behaviour); NaN maps to the positive NaN code. */
uint8_t oracle_f64_to_e4m3_rne_sat(double x) {
  if (isnan(x)) return 0x7f;
  uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80 : 0x00;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7e; /* E=15, M=6 -> 448 */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: units of 2^-9 */
    double k = round_half_even(a * 512.0);
    if (k >= 8.0) return sign | 0x08; /* rounds up into 2^-6, E=1, M=0 */
    return sign | (uint8_t)k;
  }
  int e2;
  double fr = frexp(a, &e2); /* a = fr * 2^e2, fr in [0.5, 1) */
  int e = e2 - 1;            /* a = (2 fr) * 2^e, 2 fr in [1, 2) */
  double m8 = round_half_even((2.0 * fr - 1.0) * 8.0);
  if (m8 >= 8.0) {
    m8 = 0.0;
    e += 1;
  }
  int E = e + 7;
  if (E > 15 || (E == 15 && m8 > 6.0)) return sign | 0x7e; /* saturate */
  return sign | (uint8_t)((E << 3) | (int)m8);
}

/* ------------------------------------------------------------------------ */
/* Thread pool helper: run fn(i, ctx) for i in [0, n) over nthreads.          */
/* ------------------------------------------------------------------------ */

typedef void (*item_fn)(int64_t i, void* ctx);
typedef struct {
  item_fn fn;
  void* ctx;
  int64_t n;
  int64_t next;
  pthread_mutex_t mu;
} pool_t;

static void* pool_worker(void* arg) {
  pool_t* p = (pool_t*)arg;
  for (;;) {
    pthread_mutex_lock(&p->mu);
    int64_t i = p->next++;
    pthread_mutex_unlock(&p->mu);
    if (i >= p->n) break;
    p->fn(i, p->ctx);
  }
  return NULL;
}

static void run_items(int64_t n, int nthreads, item_fn fn, void* ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  pool_t p;
  p.fn = fn;
  p.ctx = ctx;
  p.n = n;
  p.next = 0;
  pthread_mutex_init(&p.mu, NULL);
  if (nthreads == 1) {
    pool_worker(&p);
  } else {
    pthread_t th[512];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
      if (pthread_create(&th[t], NULL, pool_worker, &p) == 0) started++;
      else break;
    }
    if (started == 0) pool_worker(&p);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  }
  pthread_mutex_destroy(&p.mu);
}

/* Value of every binary16 code, filled once from oracle_f16_to_f64. */
static double f16_table[65536];
static pthread_once_t f16_once = PTHREAD_ONCE_INIT;
static void f16_table_init(void) {
  for (int i = 0; i < 65536; ++i) f16_table[i] = oracle_f16_to_f64((uint16_t)i);
}

/* ------------------------------------------------------------------------ */
/* FP16 GQA single-token decode.                                             */
/*   out[b,h,:] = sum_t softmax_t(s) V[b,g,t,:],                             */
/*   s_t = (q[b,h,:] . K[b,g,t,:]) * q_scale / sqrt(128),  g = h / 4,        */
/*   t < len_b,  K = kv[b,0], V = kv[b,1].                                   */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t* q;
  const uint16_t* kv;
  const int32_t* seq_lens;
  int64_t cap;
  double q_scale;
  const int64_t* items; /* pairs (b, h); NULL means all b*32 in order */
  double* out;          /* [n_items, 128] */
} decode_ctx;

static void decode_item(int64_t i, void* vctx) {
  decode_ctx* c = (decode_ctx*)vctx;
  int64_t b, h;
  if (c->items) {
    b = c->items[2 * i];
    h = c->items[2 * i + 1];
  } else {
    b = i / ORACLE_HQ;
    h = i % ORACLE_HQ;
  }
  int64_t g = h / (ORACLE_HQ / ORACLE_HKV);
  double* o = c->out + i * ORACLE_D;
  int64_t len = c->seq_lens[b];
  if (len < 0) len = 0;
  if (len > c->cap) len = c->cap;
  for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
  if (len == 0) return;

  double qv[ORACLE_D];
  const uint16_t* qrow = c->q + (b * ORACLE_HQ + h) * ORACLE_D;
  for (int d = 0; d < ORACLE_D; ++d) qv[d] = f16_table[qrow[d]];
  const double scale = c->q_scale / sqrt((double)ORACLE_D);

  /* kv[b, kv_index, g, t, d] */
  const int64_t slab = c->cap * ORACLE_D;
  const uint16_t* K = c->kv + ((b * 2 + 0) * ORACLE_HKV + g) * slab;
  const uint16_t* V = c->kv + ((b * 2 + 1) * ORACLE_HKV + g) * slab;

  double* s = (double*)malloc(sizeof(double) * (size_t)len);
  double mx = -INFINITY;
  for (int64_t t = 0; t < len; ++t) {
    double acc = 0.0;
    for (int d = 0; d < ORACLE_D; ++d) acc += qv[d] * f16_table[K[t * ORACLE_D + d]];
    s[t] = acc * scale;
    if (s[t] > mx) mx = s[t];
  }
  double l = 0.0;
  for (int64_t t = 0; t < len; ++t) {
    s[t] = exp(s[t] - mx);
    l += s[t];
  }
  for (int64_t t = 0; t < len; ++t) {
    double p = s[t] / l;
    for (int d = 0; d < ORACLE_D; ++d) o[d] += p * f16_table[V[t * ORACLE_D + d]];
  }
  free(s);
}

/* q: [B,32,128] f16 bits; kv: [B,2,8,cap,128] f16 bits; seq_lens: [B].
 * items: NULL (all rows, out [B,32,128]) or n_items pairs (b,h) (out
 * [n_items,128]).  Returns 0. */
int oracle_gqa_decode(const uint16_t* q, const uint16_t* kv, const int32_t* seq_lens, int64_t B,
                      int64_t cap, double q_scale, const int64_t* items, int64_t n_items,
                      double* out, int nthreads) {
  pthread_once(&f16_once, f16_table_init);
  decode_ctx c = {q, kv, seq_lens, cap, q_scale, items, out};
  int64_t n = items ? n_items : B * ORACLE_HQ;
  run_items(n, nthreads, decode_item, &c);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* NVFP4 paged K/V -> E4M3 dequantisation.                                   */
/* Token t of sequence b lives in page block_table[b, t / 64], slot t % 64.   */
/* fp4 pages: [num_pages, 8, 64, 64] bytes (two E2M1 codes per byte, element  */
/* 2i in the low nibble); scale pages: [num_pages, 8, 64, 8] E4M3, one scale  */
/* per 16 consecutive head-dim elements.                                     */
/* ------------------------------------------------------------------------ */

static uint8_t dequant_one(const uint8_t* fp4, const uint8_t* sf, int64_t page, int64_t g,
                           int64_t slot, int d) {
  const int64_t row = (page * ORACLE_HKV + g) * ORACLE_PAGE + slot;
  uint8_t byte = fp4[row * (ORACLE_D / 2) + d / 2];
  uint8_t nib = (d % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
  double scale = oracle_e4m3_to_f64(sf[row * (ORACLE_D / 16) + d / 16]);
  return oracle_f64_to_e4m3_rne_sat(oracle_e2m1_to_f64(nib) * scale);
}

/* out: [B, max_kv, 8, 128] E4M3 codes; token t of seq b for t < kv_lens[b],
 * zero bytes beyond.  Returns 0. */
int oracle_dequant_pages(const uint8_t* fp4, const uint8_t* sf, const int32_t* block_table,
                         int64_t max_pages_per_seq, const int32_t* kv_lens, int64_t B,
                         int64_t max_kv, uint8_t* out) {
  memset(out, 0, (size_t)(B * max_kv * ORACLE_HKV * ORACLE_D));
  for (int64_t b = 0; b < B; ++b) {
    int64_t len = kv_lens[b];
    if (len > max_kv) len = max_kv;
    for (int64_t t = 0; t < len; ++t) {
      int64_t page = block_table[b * max_pages_per_seq + t / ORACLE_PAGE];
      int64_t slot = t % ORACLE_PAGE;
      for (int64_t g = 0; g < ORACLE_HKV; ++g)
        for (int d = 0; d < ORACLE_D; ++d)
          out[((b * max_kv + t) * ORACLE_HKV + g) * ORACLE_D + d] =
              dequant_one(fp4, sf, page, g, slot, d);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* NVFP4 paged context attention, bottom-right causal.                       */
/* Step 1 dequantises every page a sequence uses to E4M3 (dequant_one).      */
/* Step 2, for sequence b with q_len = qo_indptr[b+1]-qo_indptr[b], kv_len:   */
/* query i (0-based within b) sees key j iff j <= kv_len - q_len + i.         */
/*   s_j = (q_e4m3[r,h,:] . Kq[b,g,j,:]) * q_scale / sqrt(128)               */
/*   O   = sum_j softmax_j(s) Vq[b,g,j,:];  result = O / out_scale.           */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint8_t* q;
  double q_scale;
  const uint8_t* kq; /* [B, max_kv, 8, 128] E4M3 codes */
  const uint8_t* vq;
  int64_t max_kv;
  const int32_t* qo_indptr;
  const int32_t* kv_lens;
  int64_t B;
  double out_scale;
  const double* e4m3; /* value of each E4M3 code */
  const int64_t* items; /* pairs (row, h); NULL means every row and head */
  double* out;
} ctx_ctx;

static void ctx_item(int64_t i, void* vctx) {
  ctx_ctx* c = (ctx_ctx*)vctx;
  int64_t r, h;
  if (c->items) {
    r = c->items[2 * i];
    h = c->items[2 * i + 1];
  } else {
    r = i / ORACLE_HQ;
    h = i % ORACLE_HQ;
  }
  double* o = c->out + i * ORACLE_D;
  for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
  /* which sequence holds row r */
  int64_t b = -1;
  for (int64_t bb = 0; bb < c->B; ++bb)
    if (r >= c->qo_indptr[bb] && r < c->qo_indptr[bb + 1]) {
      b = bb;
      break;
    }
  if (b < 0) return;
  const int64_t q_len = c->qo_indptr[b + 1] - c->qo_indptr[b];
  const int64_t kv_len = c->kv_lens[b];
  const int64_t qi = r - c->qo_indptr[b];
  int64_t n_vis = kv_len - q_len + qi + 1; /* keys j = 0 .. kv_len-q_len+qi */
  if (n_vis > kv_len) n_vis = kv_len;
  if (n_vis <= 0) return;
  const int64_t g = h / (ORACLE_HQ / ORACLE_HKV);

  double qv[ORACLE_D];
  for (int d = 0; d < ORACLE_D; ++d) qv[d] = c->e4m3[c->q[(r * ORACLE_HQ + h) * ORACLE_D + d]];
  const double scale = c->q_scale / sqrt((double)ORACLE_D);

  double* s = (double*)malloc(sizeof(double) * (size_t)n_vis);
  double mx = -INFINITY;
  for (int64_t j = 0; j < n_vis; ++j) {
    const uint8_t* krow = c->kq + ((b * c->max_kv + j) * ORACLE_HKV + g) * ORACLE_D;
    double acc = 0.0;
    for (int d = 0; d < ORACLE_D; ++d) acc += qv[d] * c->e4m3[krow[d]];
    s[j] = acc * scale;
    if (s[j] > mx) mx = s[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < n_vis; ++j) {
    s[j] = exp(s[j] - mx);
    l += s[j];
  }
  for (int64_t j = 0; j < n_vis; ++j) {
    const uint8_t* vrow = c->vq + ((b * c->max_kv + j) * ORACLE_HKV + g) * ORACLE_D;
    double p = s[j] / l;
    for (int d = 0; d < ORACLE_D; ++d) o[d] += p * c->e4m3[vrow[d]];
  }
  for (int d = 0; d < ORACLE_D; ++d) o[d] /= c->out_scale;
  free(s);
}

/* q: [total_q,32,128] E4M3 codes.  items: NULL (out [total_q,32,128]) or
 * n_items pairs (row, h) (out [n_items,128]).  Returns 0, or -1 when the
 * dequantised pages do not fit in host memory. */
int oracle_nvfp4_paged_ctx_attn(const uint8_t* q, double q_scale, const uint8_t* k_fp4,
                                const uint8_t* k_sf, const uint8_t* v_fp4, const uint8_t* v_sf,
                                const int32_t* block_table, int64_t max_pages_per_seq,
                                const int32_t* qo_indptr, const int32_t* kv_lens, int64_t B,
                                double out_scale, const int64_t* items, int64_t n_items,
                                double* out, int nthreads) {
  int64_t max_kv = 0;
  for (int64_t b = 0; b < B; ++b)
    if (kv_lens[b] > max_kv) max_kv = kv_lens[b];
  if (max_kv < 1) max_kv = 1;
  size_t bytes = (size_t)(B * max_kv * ORACLE_HKV * ORACLE_D);
  uint8_t* kq = (uint8_t*)malloc(bytes);
  uint8_t* vq = (uint8_t*)malloc(bytes);
  if (!kq || !vq) {
    free(kq);
    free(vq);
    return -1;
  }
  oracle_dequant_pages(k_fp4, k_sf, block_table, max_pages_per_seq, kv_lens, B, max_kv, kq);
  oracle_dequant_pages(v_fp4, v_sf, block_table, max_pages_per_seq, kv_lens, B, max_kv, vq);
  double e4m3[256];
  for (int code = 0; code < 256; ++code) e4m3[code] = oracle_e4m3_to_f64((uint8_t)code);
  ctx_ctx c = {q,       q_scale, kq,        vq,   max_kv, qo_indptr, kv_lens,
               B,       out_scale, e4m3,    items, out};
  int64_t n = items ? n_items : (int64_t)qo_indptr[B] * ORACLE_HQ;
  run_items(n, nthreads, ctx_item, &c);
  free(kq);
  free(vq);
  return 0;
}
