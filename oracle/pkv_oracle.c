/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for the paged KV-cache write and
 * PagedAttention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the package smoke check and the bench's CPU-baseline
 * leg do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (sources, by page title and section):
 *
 *  [book]   "Implémentation du cœur du moteur d'inférence haute performance vLLM"
 *           (AiReadCodeBooks), ch. 5 "slot_mapping et la block table" and ch. 6
 *           ("Structure des métadonnées", "Flux des paramètres du chemin
 *           non-cascadé", "Branche de masque", "Écriture du KV cache").
 *  [gpuhub] "Khám phá vLLM: Giải phẫu hệ thống suy luận LLM thông lượng cao",
 *           note under "KV cache manager" and "allocate_slots" step 1.
 *
 *  - KV write ([book] ch. 6 "Écriture du KV cache"; ch. 5 on the -1 padding of
 *    slot_mapping): every new token t whose slot is >= 0 has its K and V rows
 *    copied, bit for bit, into cache row `slot`; slots < 0 are padding and
 *    skipped.  Caches are [num_blocks, block_size, num_kv_heads, head_size], so
 *    row `slot` is block slot / block_size, offset slot % block_size.
 *
 *  - Attention ([book] ch. 6 "Structure des métadonnées" and "Flux des
 *    paramètres"): sequence s owns the query rows query_start_loc[s] ..
 *    query_start_loc[s+1]-1 and context_lens[s] keys (history plus this step's
 *    new tokens: the varlen kernel's seqused_k = seq_lens).  Key p of sequence s
 *    lives in physical block block_tables[s][p / block_size] at offset
 *    p % block_size.  Query j of a chunk of q_s queries sits at absolute
 *    position L_s - q_s + j ([book] ch. 6 "Branche de masque") and sees the
 *    keys p <= that position.  Exact scaled-dot-product attention in fp64:
 *        x_p = scale * sum_d q[d] K_p[d],   w_p = exp(x_p - max_p x_p),
 *        out = sum_p w_p V_p / sum_p w_p.
 *    GQA: query head hq reads kv head hq / (num_q_heads / num_kv_heads)
 *    (contiguous groups; the pages do not state the mapping).
 *
 *  - Sliding window ([book] ch. 2 "FullAttentionSpec", ch. 4 §4.1 null block,
 *    ch. 6 "Flux des paramètres": causal window (w, 0)): with window W > 0 the
 *    query at position pos sees only keys pos - W < p <= pos (W keys including
 *    itself); block-table entries wholly before that range are never read (they
 *    may hold the null block).  W = 0 means no window.
 *
 *  - FP8 KV cache ([book] ch. 6 "Matrice de capacités": fp8 cache dtypes;
 *    "Flux des paramètres": descales shaped (num_sequences, num_kv_heads)):
 *    the cache holds e4m3 codes (sign, 4 exponent bits with bias 7, 3 mantissa
 *    bits; exponent 0 is subnormal; S.1111.111 is NaN; no infinities; largest
 *    finite 448).  Writing stores encode(k / k_scale[h]) with the division in
 *    fp32, rounding to the nearest code (ties to the even code) and clamping
 *    magnitudes above 448 to 448.  Attention reads K = decode(code) *
 *    k_descale[s][h] and V = decode(code) * v_descale[s][h].
 *
 *  - Partial state and merge (the split buffer of [book] ch. 6 "build() étape
 *    par étape", fourth step, and merge_attn_states in the ch. 6 sequence
 *    diagram): a key range yields (m, l, acc) = (max x, sum e^(x-m),
 *    sum e^(x-m) V); several ranges merge to
 *        out = sum_i e^(m_i - M) acc_i / sum_i e^(m_i - M) l_i,  M = max_i m_i.
 *
 * Sequence-level metadata errors (context length <= 0 while the sequence has
 * queries, more queries than keys, or more keys than its block-table row holds)
 * give zero output rows and status 1.  A block id outside [0, num_blocks) gives
 * status 2 and NaN rows: the output of such a sequence is unspecified.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_FP8 = 2 };

typedef struct {
  const void *q;              /* [num_tokens, num_q_heads, head_size] */
  const void *k_cache;        /* [num_blocks, block_size, num_kv_heads, head_size] */
  const void *v_cache;        /* same */
  const int32_t *block_tables;   /* [num_seqs, bt_stride] */
  const int32_t *context_lens;   /* [num_seqs] */
  const int32_t *query_start_loc;/* [num_seqs + 1] */
  int64_t bt_stride;
  int32_t num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks;
  int32_t dtype;              /* ORC_F32 or ORC_BF16 */
  double scale;
  int32_t window;             /* sliding window W (keys per query), 0 = none */
  const float *k_descale;     /* ORC_FP8 caches: [num_seqs, num_kv_heads] */
  const float *v_descale;
} orc_problem;

/* e4m3 code -> value, straight from the format's definition. */
double orc_e4m3_decode(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);          /* subnormal */
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* value -> e4m3 code: the nearest of the 127 finite magnitudes (ties to the
 * code with an even last bit), sign kept (so -0 stays -0), magnitudes above
 * 448 clamped to 448, NaN to 0x7F.  A plain search over every code. */
uint8_t orc_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a > 448.0) a = 448.0;
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    const double err = fabs(orc_e4m3_decode((uint8_t)c) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

/* One stored element, widened exactly to double.  bf16 is the top half of an
 * IEEE binary32, so shifting its 16 bits up and reinterpreting is exact. */
static double orc_load(const void *base, int64_t idx, int32_t dtype) {
  float f;
  if (dtype == ORC_FP8) return orc_e4m3_decode(((const uint8_t *)base)[idx]);
  if (dtype == ORC_F32) {
    memcpy(&f, (const char *)base + idx * 4, 4);
  } else {
    uint16_t h;
    uint32_t u;
    memcpy(&h, (const char *)base + idx * 2, 2);
    u = ((uint32_t)h) << 16;
    memcpy(&f, &u, 4);
  }
  return (double)f;
}

/* KV write.  Returns the number of tokens whose slot was past the pool (those
 * are skipped, like padding). */
int64_t orc_write(const void *k, const void *v, const int64_t *slot_mapping,
                  int64_t num_tokens, void *k_cache, void *v_cache,
                  int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                  int32_t head_size, int32_t elem_bytes) {
  const int64_t row = (int64_t)num_kv_heads * head_size * elem_bytes;
  int64_t bad = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;                       /* padding */
    if (slot >= num_blocks * block_size) { ++bad; continue; }
    const int64_t blk = slot / block_size, off = slot % block_size;
    const int64_t dst = (blk * block_size + off) * row;
    memcpy((char *)k_cache + dst, (const char *)k + t * row, (size_t)row);
    memcpy((char *)v_cache + dst, (const char *)v + t * row, (size_t)row);
  }
  return bad;
}

/* FP8 KV write: every element of row t of k/v (bf16 bits) divided in fp32 by
 * its kv head's scale and encoded; rows with slot < 0 skipped.  Returns the
 * number of out-of-range slots. */
int64_t orc_write_fp8(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                      int64_t num_tokens, uint8_t *k_cache, uint8_t *v_cache,
                      int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                      int32_t head_size, const float *k_scale, const float *v_scale) {
  const int64_t row = (int64_t)num_kv_heads * head_size;
  int64_t bad = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * block_size) { ++bad; continue; }
    for (int64_t i = 0; i < row; ++i) {
      const int32_t h = (int32_t)(i / head_size);
      uint32_t uk = ((uint32_t)k[t * row + i]) << 16, uv = ((uint32_t)v[t * row + i]) << 16;
      float fk, fv;
      memcpy(&fk, &uk, 4);
      memcpy(&fv, &uv, 4);
      const float qk = fk / k_scale[h];   /* fp32 division, round to nearest */
      const float qv = fv / v_scale[h];
      k_cache[slot * row + i] = orc_e4m3_encode(qk);
      v_cache[slot * row + i] = orc_e4m3_encode(qv);
    }
  }
  return bad;
}

/* Checks sequence s's metadata.  0 = fine, 1 = metadata error. */
static int orc_check_seq(const orc_problem *P, int32_t s, int32_t *q_len, int32_t *L) {
  const int32_t q0 = P->query_start_loc[s], q1 = P->query_start_loc[s + 1];
  *q_len = q1 - q0;
  *L = P->context_lens[s];
  if (*q_len < 0) return 1;
  if (*q_len == 0) return 0;
  if (*L <= 0 || *q_len > *L) return 1;
  if ((int64_t)*L > P->bt_stride * P->block_size) return 1;
  return 0;
}

/* Unnormalised softmax state of query row j of sequence s, head hq, over the
 * visible keys with p in [p_lo, p_hi).  m = max x (or -inf when no key is in
 * range), l = sum exp(x - m), acc[d] = sum exp(x - m) V[d].
 * Returns 0, 1 (metadata error) or 2 (block id out of range). */
int orc_row_state(const orc_problem *P, int32_t s, int32_t hq, int32_t j,
                  int64_t p_lo, int64_t p_hi, double *m_out, double *l_out,
                  double *acc) {
  int32_t q_len, L;
  const int32_t D = P->head_size, Hkv = P->num_kv_heads;
  const int32_t G = P->num_q_heads / P->num_kv_heads;
  const int32_t kvh = hq / G;
  int st = orc_check_seq(P, s, &q_len, &L);
  for (int32_t d = 0; d < D; ++d) acc[d] = 0.0;
  *m_out = -INFINITY;
  *l_out = 0.0;
  if (st) return st;
  if (j < 0 || j >= q_len) return 1;
  const int64_t pos = (int64_t)L - q_len + j;      /* absolute query position */
  int64_t hi = p_hi < pos + 1 ? p_hi : pos + 1;    /* causal: keys p <= pos */
  int64_t lo = p_lo < 0 ? 0 : p_lo;
  if (P->window > 0 && lo < pos - P->window + 1) lo = pos - P->window + 1;  /* window */
  if (hi <= lo) return 0;

  const int64_t t = P->query_start_loc[s] + j;
  const int64_t qbase = (t * P->num_q_heads + hq) * D;
  /* q is bf16 when the cache is fp8 */
  const int32_t qtype = P->dtype == ORC_FP8 ? ORC_BF16 : P->dtype;
  const double kd = P->dtype == ORC_FP8 ? (double)P->k_descale[(int64_t)s * Hkv + kvh] : 1.0;
  const double vd = P->dtype == ORC_FP8 ? (double)P->v_descale[(int64_t)s * Hkv + kvh] : 1.0;
  double *x = (double *)malloc(sizeof(double) * (size_t)(hi - lo));
  int64_t *row = (int64_t *)malloc(sizeof(int64_t) * (size_t)(hi - lo));
  int status = 0;
  double m = -INFINITY;
  for (int64_t p = lo; p < hi; ++p) {
    const int32_t blk = P->block_tables[(int64_t)s * P->bt_stride + p / P->block_size];
    if (blk < 0 || blk >= P->num_blocks) { status = 2; break; }
    const int64_t slot = (int64_t)blk * P->block_size + p % P->block_size;
    const int64_t kbase = (slot * Hkv + kvh) * D;
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d)
      dot += orc_load(P->q, qbase + d, qtype) * (orc_load(P->k_cache, kbase + d, P->dtype) * kd);
    x[p - lo] = P->scale * dot;
    row[p - lo] = kbase;
    if (x[p - lo] > m) m = x[p - lo];
  }
  if (status == 0) {
    double l = 0.0;
    for (int64_t p = lo; p < hi; ++p) {
      const double w = exp(x[p - lo] - m);
      l += w;
      for (int32_t d = 0; d < D; ++d)
        acc[d] += w * (orc_load(P->v_cache, row[p - lo] + d, P->dtype) * vd);
    }
    *m_out = m;
    *l_out = l;
  } else {
    for (int32_t d = 0; d < D; ++d) acc[d] = NAN;
    *m_out = NAN;
    *l_out = NAN;
  }
  free(x);
  free(row);
  return status;
}

/* Merge n partial states (m_i, l_i, acc_i[D]) into a normalised output row. */
void orc_merge(int32_t n, const double *m, const double *l, const double *acc,
               int32_t D, double *out) {
  double M = -INFINITY, den = 0.0;
  for (int32_t i = 0; i < n; ++i) if (m[i] > M) M = m[i];
  for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
  if (M == -INFINITY) return;                 /* no key anywhere: zero row */
  for (int32_t i = 0; i < n; ++i) {
    if (m[i] == -INFINITY) continue;
    const double w = exp(m[i] - M);
    den += w * l[i];
    for (int32_t d = 0; d < D; ++d) out[d] += w * acc[(int64_t)i * D + d];
  }
  for (int32_t d = 0; d < D; ++d) out[d] /= den;
}

/* Full attention for every query row.  out: [num_tokens, num_q_heads, head_size]
 * fp64 (rows of tokens that belong to no sequence are left untouched).
 * seq_status[s] receives 0/1/2 as above.  Returns the number of sequences with a
 * non-zero status.  nthreads <= 0 lets OpenMP choose. */
int32_t orc_attention(const orc_problem *P, double *out, int32_t *seq_status,
                      int32_t nthreads) {
  const int32_t S = P->num_seqs, Hq = P->num_q_heads, D = P->head_size;
  int64_t nrows = 0;
  for (int32_t s = 0; s < S; ++s) {
    int32_t q_len, L;
    seq_status[s] = orc_check_seq(P, s, &q_len, &L);
    if (q_len > 0) nrows += q_len;
  }
  /* Flatten (row, head) work items so OpenMP balances across them. */
  int64_t *item_seq = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nrows > 0 ? nrows : 1));
  int64_t *item_j = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nrows > 0 ? nrows : 1));
  int64_t r = 0;
  for (int32_t s = 0; s < S; ++s) {
    const int32_t q_len = P->query_start_loc[s + 1] - P->query_start_loc[s];
    for (int32_t j = 0; j < q_len; ++j) { item_seq[r] = s; item_j[r] = j; ++r; }
  }
  const int64_t nitems = nrows * Hq;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  #pragma omp parallel
  {
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    #pragma omp for schedule(dynamic, 4)
    for (int64_t it = 0; it < nitems; ++it) {
      const int32_t s = (int32_t)item_seq[it / Hq];
      const int32_t j = (int32_t)item_j[it / Hq];
      const int32_t hq = (int32_t)(it % Hq);
      const int64_t t = P->query_start_loc[s] + j;
      double *o = out + (t * Hq + hq) * D;
      double m, l;
      const int st = orc_row_state(P, s, hq, j, 0, INT64_MAX, &m, &l, acc);
      if (st == 1) {
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
      } else if (st == 2) {
        for (int32_t d = 0; d < D; ++d) o[d] = NAN;
        seq_status[s] = 2;   /* benign race: every writer stores 2 */
      } else {
        for (int32_t d = 0; d < D; ++d) o[d] = (l > 0.0) ? acc[d] / l : 0.0;
      }
    }
    free(acc);
  }
  free(item_seq);
  free(item_j);
  int32_t nbad = 0;
  for (int32_t s = 0; s < S; ++s) nbad += seq_status[s] != 0;
  return nbad;
}

/* Threads OpenMP would use (for reporting the CPU baseline's core count). */
int32_t orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
