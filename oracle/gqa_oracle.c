/*
 * gqa_oracle.c -- plain, slow, fp64 CPU oracle for causal grouped-query
 * attention of new query rows against a KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's product path links,
 * loads or calls this file. It is compiled by oracle/build.py and used by the
 * tests, by __graft_entry__.smoke() and by the CPU-baseline leg of bench.py.
 * It shares no source with the CUDA path: no header, no helper, no table.
 *
 * What it computes (the definition, written out with no blocking, no fusion
 * and no online softmax):
 *
 *   For batch b, query row i, query head h:
 *     kvh = h / (H / Hkv)                      (kopitiam-runtime src/attention.rs,
 *                                              `repeat_kv_heads` doc: query head g
 *                                              reads KV head g / group_size)
 *     p   = position of row i                  (kopitiam-runtime src/attention.rs,
 *                                              `causal_mask` doc: row i sits at
 *                                              position_offset + i)
 *     s_j = scale * sum_c q[b,i,h,c] * K_b(j, kvh, c)      for j = 0..p
 *     out[b,i,h,:] = sum_j exp(s_j - max s) V_b(j, kvh, :) / sum_j exp(s_j - max s)
 *                                             (kopitiam-runtime src/attention.rs,
 *                                              `attention_forward`: scores, mask,
 *                                              softmax over keys, probs @ V)
 *   Keys j > p take no part (their weight is exactly zero: the mask is -inf,
 *   kopitiam-runtime src/attention.rs, test `masked_logits_are_exactly_negative_infinity`).
 *
 *   `scale` is the sole multiplier on q.k (frink-models src/decoder/attn_block.rs
 *   applies `attention_scale` to q before the kernel; frink-models src/mla/mod.rs
 *   passes an explicit `scale`). The caller passes 1/sqrt(d_k) for the plain
 *   kopitiam form, which divides by sqrt(head_dim).
 *
 *   K/V row addressing:
 *     contiguous  K_b(j,kvh,:) = k[b, kvh, j, :]   (head-major [B, Hkv, max_len, d],
 *                                                   kopitiam's per-layer [n_kv, seq, d])
 *     paged       K_b(j,kvh,:) = pool[table[b][j / bs], kvh, j % bs, :]
 *                                                  (frink-models src/decoder/attn_block.rs,
 *                                                   `push_and_attend_row`: paging changes
 *                                                   where rows live and nothing else)
 *
 *   Interleaved RoPE (frink-models src/mla/mod.rs, module doc point 2 and
 *   `rotate_pe`: ggml NORM layout, adjacent pairs). The pages print no formula;
 *   the reading used: for pair t < rot_dim/2 of the rotated slice starting at
 *   rot_offset, w_t = theta^(-2t/rot_dim), a = pos * w_t,
 *     x'[2t]   = x[2t] cos a - x[2t+1] sin a
 *     x'[2t+1] = x[2t] sin a + x[2t+1] cos a.
 *
 *   Paged append (frink-models src/decoder/attn_block.rs, `push_and_attend_row`:
 *   the row's position is read before the push, then the row is pushed, then
 *   the sequence attends over everything it holds): with p = seq_lens_in[b],
 *   rotate q[b] (every head) and k_new[b] (every KV head) at position p, write
 *   k and v to pool[table[b][p / bs], kvh, p % bs, :], set seq_lens_out[b] = p+1.
 *
 * Element storage: f32, bf16 (raw 16-bit pattern) or f64. Every value is
 * widened to double exactly; all arithmetic is in double. Stores into an f32
 * or bf16 buffer round to nearest-even (the bf16 rounding is done here, from
 * its definition, not by any library routine).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };
enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_BAD_INDEX = 2, ORC_NO_MEMORY = 3 };

/* ---- element access ---------------------------------------------------- */

double orc_bf16_bits_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16; /* bf16 is the top half of an IEEE binary32 */
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, binary32 exponent
 * range), ties to even, and return the 16-bit pattern. */
uint16_t orc_double_to_bf16_bits(double x) {
  if (isnan(x)) return 0x7fc0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double ax = fabs(x);
  if (isinf(x)) return sign | 0x7f80;
  if (ax == 0.0) return sign;
  int e;
  (void)frexp(ax, &e);          /* ax = m * 2^e, m in [0.5, 1) */
  int shift = e - 8;            /* keep 8 significant bits: grid spacing 2^(e-8) */
  if (shift < -133) shift = -133; /* below the normal range the grid is 2^-133 */
  double r = nearbyint(ldexp(ax, -shift)); /* current mode: nearest, ties to even */
  double y = ldexp(r, shift);
  if (y >= 0x1p128) return sign | 0x7f80; /* overflow to infinity */
  float f = (float)y; /* exact: y has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)((u >> 16) & 0x7fff);
}

static double ld(const void* base, size_t i, int et) {
  switch (et) {
    case ORC_F32: return (double)((const float*)base)[i];
    case ORC_BF16: return orc_bf16_bits_to_double(((const uint16_t*)base)[i]);
    default: return ((const double*)base)[i];
  }
}

static void st(void* base, size_t i, int et, double x) {
  switch (et) {
    case ORC_F32: ((float*)base)[i] = (float)x; break;
    case ORC_BF16: ((uint16_t*)base)[i] = orc_double_to_bf16_bits(x); break;
    default: ((double*)base)[i] = x; break;
  }
}

/* ---- key/value row sources ----------------------------------------------- */

typedef struct {
  int paged;             /* 0: contiguous [B, Hkv, max_len, d]; 1: paged pool */
  const void* k;
  const void* v;
  int max_len;           /* contiguous: rows per (b, kvh) */
  const int32_t* tables; /* paged: [B, mbps] */
  int mbps, bs, num_blocks;
  int Hkv, dk, dv, et;
} kv_source;

/* Flat index of element c of row j of (b, kvh) in a buffer of row width d. */
static size_t row_index(const kv_source* s, int b, int kvh, int j, int d, int c) {
  if (!s->paged)
    return (((size_t)b * s->Hkv + kvh) * s->max_len + j) * (size_t)d + c;
  int32_t blk = s->tables[(size_t)b * s->mbps + j / s->bs];
  return (((size_t)blk * s->Hkv + kvh) * s->bs + (j % s->bs)) * (size_t)d + c;
}

/* Check every block-table entry a sequence of n rows uses. */
static int check_rows(const kv_source* s, int b, int n) {
  if (!s->paged) return n <= s->max_len ? ORC_OK : ORC_BAD_INDEX;
  if (n > s->mbps * s->bs) return ORC_BAD_INDEX;
  for (int j = 0; j < n; j += s->bs) {
    int32_t blk = s->tables[(size_t)b * s->mbps + j / s->bs];
    if (blk < 0 || blk >= s->num_blocks) return ORC_BAD_INDEX;
  }
  return ORC_OK;
}

/* One query vector (already widened) against keys 0..n-1: the definition. */
static void attend(const double* qv, const kv_source* s, int b, int kvh, int n, double scale,
                   double* out, double* w) {
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    double dot = 0.0;
    for (int c = 0; c < s->dk; ++c) dot += qv[c] * ld(s->k, row_index(s, b, kvh, j, s->dk, c), s->et);
    w[j] = scale * dot;
    if (w[j] > m) m = w[j];
  }
  double den = 0.0;
  for (int j = 0; j < n; ++j) {
    w[j] = exp(w[j] - m);
    den += w[j];
  }
  for (int c = 0; c < s->dv; ++c) {
    double num = 0.0;
    for (int j = 0; j < n; ++j) num += w[j] * ld(s->v, row_index(s, b, kvh, j, s->dv, c), s->et);
    out[c] = num / den;
  }
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Shared driver: rows (b, i, h) with q row at q + ((b*seq_q + i)*H + h)*dk and
 * visible key count n(b, i) = base_len[b] - seq_q + i + 1. */
static int run_rows(const void* q, const kv_source* s, const int32_t* base_len, double* out, int B,
                    int seq_q, int H, double scale, int nthreads) {
  if (B < 0 || seq_q < 0 || H <= 0 || s->Hkv <= 0 || H % s->Hkv != 0 || s->dk <= 0 || s->dv <= 0)
    return ORC_BAD_ARG;
  const int G = H / s->Hkv;
  int maxn = 0;
  for (int b = 0; b < B; ++b) {
    int n = base_len[b];
    if (n < seq_q || n < 1) return ORC_BAD_ARG;
    int rc = check_rows(s, b, n);
    if (rc != ORC_OK) return rc;
    if (n > maxn) maxn = n;
  }
  set_threads(nthreads);
  const long total = (long)B * seq_q * H;
  int failed = 0;
#pragma omp parallel
  {
    double* qv = (double*)malloc(sizeof(double) * (size_t)s->dk);
    double* w = (double*)malloc(sizeof(double) * (size_t)(maxn > 0 ? maxn : 1));
    if (!qv || !w) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (long r = 0; r < total; ++r) {
        int h = (int)(r % H);
        int i = (int)((r / H) % seq_q);
        int b = (int)(r / ((long)H * seq_q));
        int kvh = h / G;
        int n = base_len[b] - seq_q + i + 1; /* keys 0..position of row i */
        for (int c = 0; c < s->dk; ++c) qv[c] = ld(q, (size_t)r * s->dk + c, s->et);
        attend(qv, s, b, kvh, n, scale, out + (size_t)r * s->dv, w);
      }
    }
    free(qv);
    free(w);
  }
  return failed ? ORC_NO_MEMORY : ORC_OK;
}

/* ---- public entry points --------------------------------------------------- */

/* Causal prefill: q [B, seq_q, H, dk], k [B, Hkv, seq_kv_max, dk], v [.., dv],
 * offsets [B] (NULL = 0), out f64 [B, seq_q, H, dv]. Row i of batch b sees
 * keys 0..=offsets[b] + i. */
int oracle_prefill_causal(const void* q, const void* k, const void* v, double* out, int B, int seq_q,
                          int seq_kv_max, const int32_t* offsets, int H, int Hkv, int dk, int dv,
                          double scale, int et, int nthreads) {
  kv_source s = {0, k, v, seq_kv_max, NULL, 0, 0, 0, Hkv, dk, dv, et};
  int32_t* base = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
  if (!base) return ORC_NO_MEMORY;
  for (int b = 0; b < B; ++b) {
    int off = offsets ? offsets[b] : 0;
    if (off < 0) {
      free(base);
      return ORC_BAD_ARG;
    }
    base[b] = off + seq_q; /* keys present after this pass's rows */
  }
  int rc = run_rows(q, &s, base, out, B, seq_q, H, scale, nthreads);
  free(base);
  return rc;
}

/* Decode against contiguous caches: q [B, H, dk], k [B, Hkv, max_len, dk],
 * v [B, Hkv, max_len, dv], seq_lens[b] = rows present, the query's own row
 * included (query position = seq_lens[b] - 1). out f64 [B, H, dv]. */
int oracle_decode_contig(const void* q, const void* k, const void* v, const int32_t* seq_lens,
                         double* out, int B, int max_len, int H, int Hkv, int dk, int dv, double scale,
                         int et, int nthreads) {
  kv_source s = {0, k, v, max_len, NULL, 0, 0, 0, Hkv, dk, dv, et};
  return run_rows(q, &s, seq_lens, out, B, 1, H, scale, nthreads);
}

/* Decode against a paged pool: pools [num_blocks, Hkv, bs, d], tables
 * [B, mbps] (row j of sequence b lives in block tables[b][j / bs], slot j % bs). */
int oracle_decode_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* tables,
                        const int32_t* seq_lens, double* out, int B, int mbps, int num_blocks, int bs,
                        int H, int Hkv, int dk, int dv, double scale, int et, int nthreads) {
  if (bs <= 0 || mbps <= 0) return ORC_BAD_ARG;
  kv_source s = {1, k_pool, v_pool, 0, tables, mbps, bs, num_blocks, Hkv, dk, dv, et};
  return run_rows(q, &s, seq_lens, out, B, 1, H, scale, nthreads);
}

/* ---- the arms of the attention row ------------------------------------------
 *
 * frink-models src/decoder/attn_block.rs, `push_and_attend_row`: one kernel
 * serves plain, windowed, softcapped and sink-bearing layers, and takes ALiBi
 * slopes too (`causal_gqa_attention_row(..., window, sinks, softcap, alibi)` and
 * `causal_gqa_attention_paged_sinks(...)`). The pages print no formula for the
 * arms; the readings used here:
 *   window W > 0   the query at position p sees keys j with p - W < j <= p
 *                  (W keys, its own included);
 *   softcap c > 0  s_j <- c * tanh(s_j / c), on the scaled score;
 *   ALiBi slope a  s_j <- s_j + a_h * (j - p)  (zero for the query's own key,
 *                  falling off with distance);
 *   sink z         one more term exp(z_h - m) in the softmax denominator and
 *                  none in the numerator, m = max(max_j s_j, z_h).
 * Order: scale, softcap, ALiBi, then the causal and window mask, then the
 * softmax with the sink.
 */
static void attend_arms(const double* qv, const kv_source* s, int b, int kvh, int p, int lo, double scale,
                        double softcap, const double* sink, double slope, double* out, double* w) {
  double m = sink ? *sink : -INFINITY;
  for (int j = lo; j <= p; ++j) {
    double dot = 0.0;
    for (int c = 0; c < s->dk; ++c) dot += qv[c] * ld(s->k, row_index(s, b, kvh, j, s->dk, c), s->et);
    double sj = scale * dot;
    if (softcap > 0.0) sj = softcap * tanh(sj / softcap);
    sj += slope * (double)(j - p);
    w[j - lo] = sj;
    if (sj > m) m = sj;
  }
  double total = sink ? exp(*sink - m) : 0.0;
  for (int j = lo; j <= p; ++j) {
    w[j - lo] = exp(w[j - lo] - m);
    total += w[j - lo];
  }
  for (int c = 0; c < s->dv; ++c) {
    double num = 0.0;
    for (int j = lo; j <= p; ++j) num += w[j - lo] * ld(s->v, row_index(s, b, kvh, j, s->dv, c), s->et);
    out[c] = num / total;
  }
}

/* Query rows against contiguous caches with the arms: q [B, seq_q, H, dk],
 * k [B, Hkv, max_len, dk], v [B, Hkv, max_len, dv]; base_len[b] = keys present
 * after this pass's rows, so row i sits at position base_len[b] - seq_q + i
 * (decode: seq_q = 1, base_len = seq_lens). window <= 0: none; softcap <= 0:
 * none; sinks, slopes: [H] or NULL. out f64 [B, seq_q, H, dv]. */
int oracle_attention_arms(const void* q, const void* k, const void* v, const int32_t* base_len, double* out,
                          int B, int seq_q, int max_len, int H, int Hkv, int dk, int dv, double scale,
                          int window, double softcap, const double* sinks, const double* slopes, int et,
                          int nthreads) {
  if (B < 0 || seq_q < 1 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || dk <= 0 || dv <= 0) return ORC_BAD_ARG;
  kv_source s = {0, k, v, max_len, NULL, 0, 0, 0, Hkv, dk, dv, et};
  for (int b = 0; b < B; ++b) {
    int n = base_len[b];
    if (n < seq_q || n < 1) return ORC_BAD_ARG;
    if (check_rows(&s, b, n) != ORC_OK) return ORC_BAD_INDEX;
  }
  const int G = H / Hkv;
  set_threads(nthreads);
  const long total = (long)B * seq_q * H;
  int failed = 0;
#pragma omp parallel
  {
    double* qv = (double*)malloc(sizeof(double) * (size_t)dk);
    double* w = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    if (!qv || !w) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (long r = 0; r < total; ++r) {
        int h = (int)(r % H);
        int i = (int)((r / H) % seq_q);
        int b = (int)(r / ((long)H * seq_q));
        int pos = base_len[b] - seq_q + i;
        int lo = (window > 0 && pos - window + 1 > 0) ? pos - window + 1 : 0;
        for (int c = 0; c < dk; ++c) qv[c] = ld(q, (size_t)r * dk + c, et);
        attend_arms(qv, &s, b, h / G, pos, lo, scale, softcap, sinks ? sinks + h : NULL, slopes ? slopes[h] : 0.0,
                    out + (size_t)r * dv, w);
      }
    }
    free(qv);
    free(w);
  }
  return failed ? ORC_NO_MEMORY : ORC_OK;
}

/* Interleaved RoPE in place on x [B, T, heads, d] stored as `et`; positions
 * [B, T]. The rotated slice is x[..., rot_offset : rot_offset + rot_dim]. */
int oracle_rope_interleaved(void* x, const int32_t* positions, int B, int T, int heads, int d,
                            int rot_offset, int rot_dim, double theta, int et) {
  if (rot_dim <= 0 || rot_dim % 2 || rot_offset < 0 || rot_offset + rot_dim > d || theta <= 0.0)
    return ORC_BAD_ARG;
  for (int b = 0; b < B; ++b)
    for (int t = 0; t < T; ++t) {
      double pos = (double)positions[(size_t)b * T + t];
      for (int h = 0; h < heads; ++h) {
        size_t row = (((size_t)b * T + t) * heads + h) * (size_t)d + rot_offset;
        for (int pr = 0; pr < rot_dim / 2; ++pr) {
          double w = pow(theta, -2.0 * pr / rot_dim);
          double a = pos * w;
          double x0 = ld(x, row + 2 * pr, et), x1 = ld(x, row + 2 * pr + 1, et);
          st(x, row + 2 * pr, et, x0 * cos(a) - x1 * sin(a));
          st(x, row + 2 * pr + 1, et, x0 * sin(a) + x1 * cos(a));
        }
      }
    }
  return ORC_OK;
}

/* Paged append of one new row per sequence: q [B, H, dk] and k_new [B, Hkv, dk]
 * rotated at p = seq_lens_in[b] (theta <= 0: no rotation), k/v written into the
 * pools, seq_lens_out[b] = p + 1 (may alias seq_lens_in). All buffers are `et`. */
int oracle_kv_append_paged(void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                           const int32_t* tables, const int32_t* seq_lens_in, int32_t* seq_lens_out,
                           int B, int mbps, int num_blocks, int bs, int H, int Hkv, int dk, int dv,
                           double theta, int rot_offset, int rot_dim, int et) {
  if (bs <= 0 || mbps <= 0 || Hkv <= 0 || H % Hkv) return ORC_BAD_ARG;
  for (int b = 0; b < B; ++b) {
    int p = seq_lens_in[b];
    if (p < 0 || p >= mbps * bs) return ORC_BAD_INDEX;
    int32_t blk = tables[(size_t)b * mbps + p / bs];
    if (blk < 0 || blk >= num_blocks) return ORC_BAD_INDEX;
  }
  double* row = (double*)malloc(sizeof(double) * (size_t)(dk > dv ? dk : dv));
  void* tmp = malloc(sizeof(double) * (size_t)(dk > dv ? dk : dv));
  if (!row || !tmp) {
    free(row);
    free(tmp);
    return ORC_NO_MEMORY;
  }
  for (int b = 0; b < B; ++b) {
    int p = seq_lens_in[b];
    int32_t pos = p;
    int32_t blk = tables[(size_t)b * mbps + p / bs];
    for (int h = 0; h < H && theta > 0.0; ++h) {
      /* the query row of this step, every head, rotated in place at position p */
      size_t off = ((size_t)b * H + h) * (size_t)dk;
      for (int c = 0; c < dk; ++c) ((double*)tmp)[c] = ld(q, off + c, et);
      oracle_rope_interleaved(tmp, &pos, 1, 1, 1, dk, rot_offset, rot_dim, theta, ORC_F64);
      for (int c = 0; c < dk; ++c) st(q, off + c, et, ((double*)tmp)[c]);
    }
    for (int kvh = 0; kvh < Hkv; ++kvh) {
      size_t src_k = ((size_t)b * Hkv + kvh) * (size_t)dk;
      for (int c = 0; c < dk; ++c) row[c] = ld(k_new, src_k + c, et);
      if (theta > 0.0) oracle_rope_interleaved(row, &pos, 1, 1, 1, dk, rot_offset, rot_dim, theta, ORC_F64);
      size_t dst_k = (((size_t)blk * Hkv + kvh) * bs + p % bs) * (size_t)dk;
      for (int c = 0; c < dk; ++c) st(k_pool, dst_k + c, et, row[c]);
      size_t src_v = ((size_t)b * Hkv + kvh) * (size_t)dv;
      size_t dst_v = (((size_t)blk * Hkv + kvh) * bs + p % bs) * (size_t)dv;
      for (int c = 0; c < dv; ++c) st(v_pool, dst_v + c, et, ld(v_new, src_v + c, et));
    }
    seq_lens_out[b] = p + 1;
  }
  free(row);
  free(tmp);
  return ORC_OK;
}
