/*
 * pattn_ref.c -- float64 CPU oracle for paged variable-length attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline / reference arm load it.
 * It shares no code, header or table with the CUDA library and must never be
 * used as a fallback for it.
 *
 * What it computes (pages: "[vLLM] FlashAttention" -- FlashAttentionBackend
 * get_kv_cache_shape, FlashAttentionImpl, FlashAttentionMetadata;
 * "[vLLM] other attention backends" -- TritonAttentionMetadata;
 * "RBLN Attention modes" -- overview, Full Attention, Sliding-Window Attention):
 *
 *   For request r: q_len = qsl[r+1]-qsl[r], s = seq_lens[r],
 *   ctx = s - q_len (seq_len = context_len + query_len).
 *   Query row i of r sits at position p = ctx + i.  Head h reads KV head
 *   g = h / (num_heads / num_kv_heads) (contiguous GQA groups).
 *   Key k (0 <= k < s) lives in physical block block_table[r][k / bs],
 *   slot k % bs of the cache laid out as [2][num_blocks][bs][num_kv_heads][d]
 *   (index 0 = K, 1 = V).
 *   k is visible iff (causal == 0 or k <= p) and (window <= 0 or p - k < window).
 *   score_k = scale * sum_j q_j K_kj, m = max score, w_k = exp(score_k - m),
 *   out = sum_k w_k V_k / sum_k w_k, lse = m + ln(sum_k w_k).
 *
 * Attention sinks (optional, one logit per query head): the pages name them
 * only in the RBLN kernel-selection rule ("Full Attention", choice between
 * naive and flash attention) and give no formula.  The reading taken here is
 * a learned logit sink_h that joins the softmax normaliser as one more term
 * with no value: with m = max(max_k score_k, sink_h),
 *   out = sum_k w_k V_k / (exp(sink_h - m) + sum_k w_k),
 *   lse = m + ln(exp(sink_h - m) + sum_k w_k).
 * sink_h is in the units of score (natural log, not multiplied by scale).
 * sink_h = -inf is the same as no sink.
 *
 * This is the "naive attention" of the RBLN overview: scores over the valid
 * tokens, softmax, product with V -- with the causal mask of its Full
 * Attention section and the window of its SWA section.  The FlashAttention
 * page states that the tiled online-softmax method is exact, so the tiled
 * CUDA kernels must reach this result up to rounding.
 *
 * DiffKV layout (head_size_v > 0): "[vLLM] other attention backends",
 * FlashAttention DiffKV, lets V have its own head size head_size_v and says
 * the cache is then asymmetric, without giving its shape.  The reading taken:
 * one tensor [num_blocks][block_size][num_kv_heads][head_size + head_size_v],
 * each row holding the token's K (head_size elements) then its V (head_size_v
 * elements); scores use the head_size elements of q and K, the output has
 * head_size_v elements.
 *
 * Split mode (num_splits > 1) is the RBLN "flash attention" reading: the
 * visible keys are cut into partitions of whole KV blocks, each partition
 * gives (o_p, lse_p) by the same definition, and the partitions are merged
 * with lse = ln sum_p exp(lse_p), out = sum_p exp(lse_p - lse) o_p.  It exists
 * so the test suite can check that merging is exact (split == unsplit).
 *
 * Inputs are converted to double exactly: bf16 by a 16-bit shift into an IEEE
 * single; fp8 e4m3 by the OCP FP8 / "FP8 Formats for Deep Learning"
 * (Micikevicius et al., 2022) definition -- sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, subnormals at exponent 0, no infinities, S.1111.111 = NaN --
 * then multiplied by the per-tensor fp32 scale promoted to double.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REF_OK 0
#define REF_ERR_ARG 1
#define REF_ERR_METADATA 2
#define REF_ERR_NOMEM 3

/* bf16 -> double: the bf16 bits are the high half of an IEEE single. */
double pattn_ref_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16 -> double, from the format definition: sign, 5 exponent bits
 * with bias 15, 10 mantissa bits; exponent 0 holds subnormals (m * 2^-24),
 * exponent 31 infinities (m = 0) and NaNs. */
double pattn_ref_f16_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  double mag;
  if (e == 0x1F) return m ? NAN : (sign ? -INFINITY : INFINITY);
  if (e == 0)
    mag = ldexp((double)m, -24);
  else
    mag = ldexp(1.0 + (double)m / 1024.0, e - 15);
  return sign ? -mag : mag;
}

/* e4m3 (OCP "E4M3FN") -> double, from the format definition. */
double pattn_ref_e4m3_to_double(uint8_t b) {
  int sign = (b >> 7) & 1;
  int e = (b >> 3) & 0xF;
  int m = b & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN; /* S.1111.111 */
  if (e == 0)
    mag = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

typedef struct {
  const uint16_t* q;
  const void* kv;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int num_seqs, max_blocks_per_seq, num_blocks;
  double scale;
  int num_heads, num_kv_heads, head_size, block_size;
  int head_size_v; /* elements of a V row (== head_size unless diffkv) */
  int diffkv;      /* cache in the DiffKV layout */
  int window, causal, kv_dtype;
  double k_scale, v_scale;
  const int32_t* row_token;
  const int32_t* row_head;
  int64_t n_rows;
  int num_splits;
  double* out;
  double* lse;
  const float* sinks; /* [num_heads] or NULL */
  atomic_llong next_row;
  atomic_int error;
  int max_seq;
} job_t;

/* Element (kv_index, block, slot, g, j) of the cache, as double. */
static double cache_elem(const job_t* jb, int kv_index, int block, int slot, int g, int j) {
  int64_t idx;
  if (jb->diffkv)
    idx = (((int64_t)block * jb->block_size + slot) * jb->num_kv_heads + g) *
              (jb->head_size + jb->head_size_v) + (kv_index ? jb->head_size + j : j);
  else
    idx = ((((int64_t)kv_index * jb->num_blocks + block) * jb->block_size + slot) *
               jb->num_kv_heads + g) * jb->head_size + j;
  if (jb->kv_dtype == 0) return pattn_ref_bf16_to_double(((const uint16_t*)jb->kv)[idx]);
  if (jb->kv_dtype == 2) return pattn_ref_f16_to_double(((const uint16_t*)jb->kv)[idx]);
  return pattn_ref_e4m3_to_double(((const uint8_t*)jb->kv)[idx]) *
         (kv_index == 0 ? jb->k_scale : jb->v_scale);
}

static int find_request(const job_t* jb, int t) {
  for (int r = 0; r < jb->num_seqs; ++r)
    if (jb->qsl[r] <= t && t < jb->qsl[r + 1]) return r;
  return -1;
}

static int key_visible(const job_t* jb, int k, int p) {
  if (jb->causal && k > p) return 0;
  if (jb->window > 0 && p - k >= jb->window) return 0;
  return 1;
}

/*
 * Attention of one query row over the visible keys in [k_begin, k_end), with
 * the sink logit `sink` in the normaliser (-inf: none).  Writes the
 * normalised output to o[d] and returns lse (-inf if no key is visible and
 * there is no sink, with o = 0).  scores[] has room for s doubles.
 */
static double attend_range(const job_t* jb, int r, const double* qv, int g, int p,
                           int k_begin, int k_end, double sink, double* scores, double* o) {
  const int d = jb->head_size, dv = jb->head_size_v, bs = jb->block_size;
  const int32_t* bt = jb->block_table + (int64_t)r * jb->max_blocks_per_seq;
  double m = -INFINITY;
  int any = 0;
  for (int j = 0; j < dv; ++j) o[j] = 0.0;
  for (int k = k_begin; k < k_end; ++k) {
    if (!key_visible(jb, k, p)) continue;
    int blk = bt[k / bs], slot = k % bs;
    double dot = 0.0;
    for (int j = 0; j < d; ++j) dot += qv[j] * cache_elem(jb, 0, blk, slot, g, j);
    scores[k] = jb->scale * dot;
    if (!any || scores[k] > m) m = scores[k];
    any = 1;
  }
  const int has_sink = sink > -INFINITY;
  if (!any && !has_sink) return -INFINITY;
  if (has_sink && (!any || sink > m)) m = sink;
  double denom = has_sink ? exp(sink - m) : 0.0;
  for (int k = k_begin; k < k_end; ++k) {
    if (!key_visible(jb, k, p)) continue;
    int blk = bt[k / bs], slot = k % bs;
    double w = exp(scores[k] - m);
    denom += w;
    for (int j = 0; j < dv; ++j) o[j] += w * cache_elem(jb, 1, blk, slot, g, j);
  }
  for (int j = 0; j < dv; ++j) o[j] /= denom;
  return m + log(denom);
}

static int row_compute(job_t* jb, int64_t row, double* scores, double* qv, double* part) {
  const int d = jb->head_size, dv = jb->head_size_v, bs = jb->block_size;
  int t = jb->row_token[row], h = jb->row_head[row];
  if (h < 0 || h >= jb->num_heads) return REF_ERR_ARG;
  int r = find_request(jb, t);
  if (r < 0) return REF_ERR_METADATA;
  int q_len = jb->qsl[r + 1] - jb->qsl[r];
  int s = jb->seq_lens[r];
  if (q_len > s || s > jb->max_blocks_per_seq * bs) return REF_ERR_METADATA;
  for (int k = 0; k < s; k += bs) {
    int blk = jb->block_table[(int64_t)r * jb->max_blocks_per_seq + k / bs];
    if (blk < 0 || blk >= jb->num_blocks) return REF_ERR_METADATA;
  }
  int ctx = s - q_len, i = t - jb->qsl[r], p = ctx + i;
  int g = h / (jb->num_heads / jb->num_kv_heads);
  for (int j = 0; j < d; ++j)
  {
    const uint16_t bits = jb->q[((int64_t)t * jb->num_heads + h) * d + j];
    qv[j] = jb->kv_dtype == 2 ? pattn_ref_f16_to_double(bits) : pattn_ref_bf16_to_double(bits);
  }
  double* o = jb->out + row * dv;
  const double sink = jb->sinks ? (double)jb->sinks[h] : -INFINITY;

  if (jb->num_splits <= 1) {
    jb->lse[row] = attend_range(jb, r, qv, g, p, 0, s, sink, scores, o);
    return REF_OK;
  }

  /* Split mode: the visible keys span blocks [b_lo, b_hi); cut them into
     num_splits runs of ceil(nblk / num_splits) whole blocks each. */
  int k_lo = -1, k_hi = -1;
  for (int k = 0; k < s; ++k)
    if (key_visible(jb, k, p)) {
      if (k_lo < 0) k_lo = k;
      k_hi = k + 1;
    }
  for (int j = 0; j < dv; ++j) o[j] = 0.0;
  if (k_lo < 0) {
    jb->lse[row] = sink;  /* the sink alone (or -inf) */
    return REF_OK;
  }
  int b_lo = k_lo / bs, b_hi = (k_hi + bs - 1) / bs, nblk = b_hi - b_lo;
  int per = (nblk + jb->num_splits - 1) / jb->num_splits;
  /* Each partition gives (o_p, lse_p) by the plain definition (no sink); then
     merge, the sink entering the merge as one more term with no output. */
  double* lse_p = part + (int64_t)jb->num_splits * dv;
  double lse_max = -INFINITY;
  for (int sp = 0; sp < jb->num_splits; ++sp) {
    int kb = (b_lo + sp * per) * bs, ke = (b_lo + (sp + 1) * per) * bs;
    if (kb > s) kb = s;
    if (ke > s) ke = s;
    lse_p[sp] = (kb < ke) ? attend_range(jb, r, qv, g, p, kb, ke, -INFINITY, scores,
                                         part + (int64_t)sp * dv)
                          : -INFINITY;
    if (lse_p[sp] > lse_max) lse_max = lse_p[sp];
  }
  if (sink > lse_max) lse_max = sink;
  double sum = 0.0;
  for (int sp = 0; sp < jb->num_splits; ++sp)
    if (lse_p[sp] > -INFINITY) sum += exp(lse_p[sp] - lse_max);
  if (sink > -INFINITY) sum += exp(sink - lse_max);
  double lse = lse_max + log(sum);
  for (int sp = 0; sp < jb->num_splits; ++sp) {
    if (!(lse_p[sp] > -INFINITY)) continue;
    double wgt = exp(lse_p[sp] - lse);
    for (int j = 0; j < dv; ++j) o[j] += wgt * part[(int64_t)sp * dv + j];
  }
  jb->lse[row] = lse;
  return REF_OK;
}

static void* worker(void* arg) {
  job_t* jb = (job_t*)arg;
  int nsp = jb->num_splits > 1 ? jb->num_splits : 1;
  double* scores = (double*)malloc(sizeof(double) * (size_t)(jb->max_seq + 1));
  double* qv = (double*)malloc(sizeof(double) * (size_t)jb->head_size);
  double* part = (double*)malloc(sizeof(double) * (size_t)(jb->head_size_v + 1) * (size_t)nsp);
  if (!scores || !qv || !part) {
    atomic_store(&jb->error, REF_ERR_NOMEM);
  } else {
    for (;;) {
      int64_t row = atomic_fetch_add(&jb->next_row, 1);
      if (row >= jb->n_rows || atomic_load(&jb->error)) break;
      int rc = row_compute(jb, row, scores, qv, part);
      if (rc) atomic_store(&jb->error, rc);
    }
  }
  free(scores);
  free(qv);
  free(part);
  return NULL;
}

/*
 * Attention for an explicit list of (token, head) rows.
 *   q          bf16 bits [num_tokens][num_heads][head_size]
 *   kv_cache   [2][num_blocks][block_size][num_kv_heads][head_size], or with
 *              head_size_v > 0 the DiffKV layout
 *              [num_blocks][block_size][num_kv_heads][head_size + head_size_v],
 *              bf16 bits (kv_dtype 0), e4m3 bytes (kv_dtype 1) or f16 bits
 *              (kv_dtype 2, where q is f16 too; else q is bf16)
 *   kv_scale   {k_scale, v_scale}; read only for kv_dtype 1
 *   out        [n_rows][head_size_v, or head_size] doubles, lse [n_rows] doubles
 *   sinks      [num_heads] sink logits, or NULL for none
 *   head_size_v  0: the standard layout; > 0: the DiffKV layout (16-bit K/V)
 * Returns 0, or REF_ERR_* (bad arguments, metadata, or memory).
 */
int pattn_ref_rows(const void* q, const void* kv_cache, const int32_t* block_table,
                   const int32_t* seq_lens, const int32_t* query_start_loc, int num_seqs,
                   int max_blocks_per_seq, int num_blocks, float scale, int num_heads,
                   int num_kv_heads, int head_size, int block_size, int window, int causal,
                   int kv_dtype, const float* kv_scale, const int32_t* row_token,
                   const int32_t* row_head, int64_t n_rows, int num_splits, int num_threads,
                   double* out, double* lse, const float* sinks, int head_size_v) {
  if (!q || !kv_cache || !block_table || !seq_lens || !query_start_loc || !out || !lse)
    return REF_ERR_ARG;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_size <= 0 ||
      block_size <= 0 || num_seqs < 0 || kv_dtype < 0 || kv_dtype > 2 ||
      (kv_dtype == 1 && !kv_scale) || head_size_v < 0 || (head_size_v > 0 && kv_dtype == 1))
    return REF_ERR_ARG;
  if (n_rows == 0) return REF_OK;
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.q = (const uint16_t*)q;
  jb.kv = kv_cache;
  jb.block_table = block_table;
  jb.seq_lens = seq_lens;
  jb.qsl = query_start_loc;
  jb.num_seqs = num_seqs;
  jb.max_blocks_per_seq = max_blocks_per_seq;
  jb.num_blocks = num_blocks;
  jb.scale = (double)scale;
  jb.num_heads = num_heads;
  jb.num_kv_heads = num_kv_heads;
  jb.head_size = head_size;
  jb.diffkv = head_size_v > 0;
  jb.head_size_v = head_size_v > 0 ? head_size_v : head_size;
  jb.block_size = block_size;
  jb.window = window;
  jb.causal = causal;
  jb.kv_dtype = kv_dtype;
  jb.k_scale = kv_dtype == 1 ? (double)kv_scale[0] : 1.0;
  jb.v_scale = kv_dtype == 1 ? (double)kv_scale[1] : 1.0;
  jb.row_token = row_token;
  jb.row_head = row_head;
  jb.n_rows = n_rows;
  jb.num_splits = num_splits;
  jb.out = out;
  jb.lse = lse;
  jb.sinks = sinks;
  atomic_init(&jb.next_row, 0);
  atomic_init(&jb.error, 0);
  jb.max_seq = 0;
  for (int r = 0; r < num_seqs; ++r)
    if (seq_lens[r] > jb.max_seq) jb.max_seq = seq_lens[r];

  if (num_threads < 1) num_threads = 1;
  if (num_threads > 256) num_threads = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 1; i < num_threads; ++i) {
    if (pthread_create(&th[started], NULL, worker, &jb) != 0) break;
    ++started;
  }
  worker(&jb);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  return atomic_load(&jb.error);
}

/* ------------------------------------------------------------------ cache write */

/*
 * fp32 -> e4m3 byte (OCP "E4M3FN"), from the format definition: round to the
 * nearest representable value, ties to the even code (mantissa LSB 0), with
 * saturation -- magnitudes at or above the largest finite value 448, and
 * infinities, give +-448 -- and NaN giving the NaN code S.1111.111.  The
 * finite codes 0x00..0x7E are scanned in order of magnitude (they are
 * monotonic in it): slow and plain.
 */
uint8_t pattn_ref_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  const int sign = signbit(x) ? 1 : 0;
  const double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)((sign << 7) | 0x7E);
  int lo = 0; /* largest code whose magnitude is <= a */
  for (int c = 0; c <= 0x7E; ++c)
    if (pattn_ref_e4m3_to_double((uint8_t)c) <= a) lo = c;
  const double below = a - pattn_ref_e4m3_to_double((uint8_t)lo);
  const double above = pattn_ref_e4m3_to_double((uint8_t)(lo + 1)) - a;
  int c;
  if (below < above)
    c = lo;
  else if (above < below)
    c = lo + 1;
  else
    c = (lo & 1) ? lo + 1 : lo;
  return (uint8_t)((sign << 7) | c);
}

/*
 * KV-cache write, the step that fills the cache attention reads ("[vLLM]
 * FlashAttention", FlashAttentionMetadata.slot_mapping and the PagedAttention
 * point of its "why this design" list; the cache-write kernel of the DiffKV
 * backend in "[vLLM] other attention backends").  Token t with slot
 * s = slot_mapping[t] >= 0 writes its key and value rows of every KV head to
 * cache[0 or 1][s / bs][s % bs][h][0..d): bf16 bits as they are, or for an
 * e4m3 cache the byte e4m3(x / scale) of the fp32 quotient (x the bf16 value,
 * scale the K or V per-tensor scale), rounded as pattn_ref_e4m3_encode does.
 * A negative slot writes nothing.  A slot at or beyond num_blocks * bs writes
 * nothing and makes the call return REF_ERR_METADATA.  key and value are bf16
 * bits [T][Hkv][d]; the cache is updated in place.
 */
int pattn_ref_reshape_and_cache(const uint16_t* key, const uint16_t* value, void* kv_cache,
                                const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                int head_size, int block_size, int num_blocks, int kv_dtype,
                                float k_scale, float v_scale) {
  if (!key || !value || !kv_cache || !slot_mapping || num_tokens < 0 || num_kv_heads <= 0 ||
      head_size <= 0 || block_size <= 0 || num_blocks < 0 || kv_dtype < 0 || kv_dtype > 2)
    return REF_ERR_ARG;
  int err = REF_OK;
  const int64_t pool = (int64_t)num_blocks * block_size;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    if (s >= pool) {
      err = REF_ERR_METADATA;
      continue;
    }
    const int64_t blk = s / block_size, slot = s % block_size;
    for (int kv = 0; kv < 2; ++kv) {
      const uint16_t* src = kv ? value : key;
      const float sc = kv ? v_scale : k_scale;
      for (int h = 0; h < num_kv_heads; ++h)
        for (int j = 0; j < head_size; ++j) {
          const uint16_t bits = src[((int64_t)t * num_kv_heads + h) * head_size + j];
          const int64_t dst =
              ((((int64_t)kv * num_blocks + blk) * block_size + slot) * num_kv_heads + h) *
                  head_size + j;
          if (kv_dtype != 1) {  /* 16-bit cache: the bits as they are */
            ((uint16_t*)kv_cache)[dst] = bits;
          } else {
            const float x = (float)pattn_ref_bf16_to_double(bits);
            const float q = x / sc;
            ((uint8_t*)kv_cache)[dst] = pattn_ref_e4m3_encode(q);
          }
        }
    }
  }
  return err;
}

/*
 * KV-cache write for the DiffKV layout ("[vLLM] other attention backends",
 * FlashAttention DiffKV, which has its own cache-write kernel for its
 * asymmetric cache).  Token t with slot s = slot_mapping[t] >= 0 writes, for
 * every KV head h, its key row (head_size elements) and then its value row
 * (head_size_v elements) to cache row [s / bs][s % bs][h] of
 * [num_blocks][block_size][num_kv_heads][head_size + head_size_v]: 16-bit
 * bits as they are.  A negative slot writes nothing; a slot at or beyond
 * num_blocks * bs writes nothing and makes the call return REF_ERR_METADATA.
 * key is [T][Hkv][head_size] and value [T][Hkv][head_size_v], 16-bit bits.
 */
int pattn_ref_reshape_and_cache_diffkv(const uint16_t* key, const uint16_t* value,
                                       uint16_t* kv_cache, const int64_t* slot_mapping,
                                       int num_tokens, int num_kv_heads, int head_size,
                                       int head_size_v, int block_size, int num_blocks) {
  if (!key || !value || !kv_cache || !slot_mapping || num_tokens < 0 || num_kv_heads <= 0 ||
      head_size <= 0 || head_size_v <= 0 || block_size <= 0 || num_blocks < 0)
    return REF_ERR_ARG;
  int err = REF_OK;
  const int64_t pool = (int64_t)num_blocks * block_size;
  const int width = head_size + head_size_v;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t sl = slot_mapping[t];
    if (sl < 0) continue;
    if (sl >= pool) {
      err = REF_ERR_METADATA;
      continue;
    }
    for (int h = 0; h < num_kv_heads; ++h) {
      uint16_t* row = kv_cache + ((sl / block_size * block_size + sl % block_size) *
                                      num_kv_heads + h) * (int64_t)width;
      for (int j = 0; j < head_size; ++j)
        row[j] = key[((int64_t)t * num_kv_heads + h) * head_size + j];
      for (int j = 0; j < head_size_v; ++j)
        row[head_size + j] = value[((int64_t)t * num_kv_heads + h) * head_size_v + j];
    }
  }
  return err;
}
