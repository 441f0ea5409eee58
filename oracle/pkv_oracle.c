/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header, table or constant with the CUDA
 * library; the two meet only through seeded inputs.
 *
 * What each routine computes, and the passage of the source pages it follows:
 *
 *  - orc_reshape_and_cache: the slot write.  "PagedAttention por dentro"
 *    (section "La tabla de páginas (block table)") says a new token goes to
 *    the free position of the sequence's last block; a slot is the flat
 *    index block_id * block_size + offset.  Plain scatter, with the element
 *    converted to the cache's type.
 *  - orc_gather_kv: the block-table gather.  "La despensa por casilleros"
 *    (section "El mecanismo: bloques, block table y el gather del kernel"):
 *    walk a sequence's physical blocks in logical order and read K and V as
 *    if they were contiguous.
 *  - orc_copy_blocks: whole-block copies between pools.  "PagedAttention
 *    por dentro" (sections "Copy-on-write para sampling paralelo" and
 *    "Evicción y preemption: qué hace cuando el pool se agota", the swap
 *    strategy) and "La despensa por casilleros" (section "Prefix caching:
 *    compartir casilleros con copy-on-write"): a shared block is copied for
 *    the branch about to write it; a preempted sequence's blocks move to
 *    host memory and back.  A plain byte copy per pair.
 *  - orc_paged_attention_decode: the decode attention definition,
 *    softmax(q . K^T * scale) . V over every cached token of the sequence,
 *    the current one included ("Optimización de Inferencia LLM", section
 *    "El Cuello de Botella de Atención del que Nadie Habla", and "Capítulo 2",
 *    section "Qué guarda realmente el KV cache").  Query head qh reads kv
 *    head qh / (Hq / Hkv) (grouped-query sharing, "KV cache: la memoria de
 *    trabajo", section "Trucos para que el cuaderno sea más fino").  With a
 *    sliding window the sum runs only over the window's last tokens and the
 *    attention sinks, the first tokens ("PagedAttention por dentro",
 *    sections "Sliding window attention" and "StreamingLLM (Xiao et al.,
 *    2024): los attention sinks").
 *  - orc_paged_attention_multi: the same attention for several query tokens
 *    per sequence, a prefill chunk or the tokens a speculative step
 *    verifies.  "PagedAttention por dentro" (section "Chunked prefill
 *    integrado con paged KV": prefill chunks and decode tokens attend the
 *    same paged cache in one step) and "Componentes Internos de Servicio de
 *    vLLM" (section "Chunked prefill protege la cola del TTFT": fixed-size
 *    chunks, 512 tokens by default).  The chunk's tokens are the sequence's
 *    last positions, written to the cache first, and each attends the
 *    positions up to its own (prefill attention is causal; the pages do
 *    not spell out the mask, this is the plain reading).
 *  - orc_partition_attention / orc_split_kv_reduce: the same attention
 *    restricted to fixed token partitions, and the log-sum-exp merge of the
 *    partitions.  The pages do not describe a split; this is the plain
 *    algebra of a softmax over a union of disjoint token sets.
 *  - fp8 e4m3: the OCP 8-bit floating point E4M3 definition (1 sign bit,
 *    4 exponent bits with bias 7, 3 mantissa bits, no infinities, the single
 *    NaN pattern S.1111.111, maximum finite 448), encoded with round to
 *    nearest, ties to even, and saturation of finite overflow to +-448.
 *  - bf16: the upper 16 bits of an IEEE binary32, encoded with round to
 *    nearest, ties to even.
 *
 * Readings taken where the pages are silent: a negative slot is skipped; a
 * sequence of length 0 yields a zero output row; the fp8 scale is one
 * per-tensor factor shared by K and V (stored = e4m3(x / kv_scale) with the
 * division done in binary32, real value = code * kv_scale).
 *
 * Floating point: every attention quantity is double precision.  Only the
 * cache writes use binary32 arithmetic, because the cache types are defined
 * from binary32 inputs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_FP8_E4M3 = 2 };
enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_RANGE = 2, ORC_ERR_NOMEM = 3 };

/* ------------------------------------------------------------------ */
/* Element types                                                       */
/* ------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static uint32_t bits_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
}

double orc_bf16_decode(uint16_t b) { return (double)f32_from_bits((uint32_t)b << 16); }

/* binary32 -> bf16, round to nearest, ties to even.  The kept part is the
 * upper half of the word; the dropped half decides the rounding. */
uint16_t orc_bf16_encode(float x) {
  uint32_t u = bits_from_f32(x);
  if (isnan(x)) return (uint16_t)((u >> 16) | 0x0040u); /* stay a quiet NaN */
  uint32_t kept = u >> 16;
  uint32_t dropped = u & 0xFFFFu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

/* Value of an E4M3 code, straight from the format definition. */
double orc_fp8_e4m3_decode(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6); /* subnormal: 0.mmm * 2^(1-7) */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* binary32 -> E4M3, round to nearest with ties to the even code, finite
 * overflow (and infinity) saturated to the largest finite magnitude 448.
 * The non-negative finite codes 0x00..0x7E are increasing in value, so the
 * neighbours of |x| are found by a walk over that ordered list and the tie
 * is broken by the code's least significant bit (the mantissa's). */
uint8_t orc_fp8_e4m3_encode(float x) {
  if (isnan(x)) return (uint8_t)(signbit(x) ? 0xFF : 0x7F);
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int lo = 0; /* largest code whose value is <= a */
  while (lo + 1 <= 0x7E && orc_fp8_e4m3_decode((uint8_t)(lo + 1)) <= a) ++lo;
  double vlo = orc_fp8_e4m3_decode((uint8_t)lo);
  if (vlo == a) return (uint8_t)(sign | lo);
  int hi = lo + 1; /* exists because a < 448 */
  double vhi = orc_fp8_e4m3_decode((uint8_t)hi);
  double mid = 0.5 * (vlo + vhi); /* exact: both have 4 significant bits */
  int pick;
  if (a < mid)
    pick = lo;
  else if (a > mid)
    pick = hi;
  else
    pick = (lo & 1) ? hi : lo;
  return (uint8_t)(sign | pick);
}

static size_t elem_size(int dtype) {
  switch (dtype) {
    case ORC_F32: return 4;
    case ORC_BF16: return 2;
    case ORC_FP8_E4M3: return 1;
    default: return 0;
  }
}

/* Read element i of a typed array as a binary32 value (exact for all three
 * types except fp8, which is never a source type here). */
static float load_as_f32(const void* base, int dtype, size_t i) {
  if (dtype == ORC_F32) return ((const float*)base)[i];
  return f32_from_bits((uint32_t)((const uint16_t*)base)[i] << 16);
}

/* Read element i of a cache as a double, fp8 codes multiplied by kv_scale. */
static double load_cache_f64(const void* base, int dtype, size_t i, double kv_scale) {
  switch (dtype) {
    case ORC_F32: return (double)((const float*)base)[i];
    case ORC_BF16: return orc_bf16_decode(((const uint16_t*)base)[i]);
    default: return orc_fp8_e4m3_decode(((const uint8_t*)base)[i]) * kv_scale;
  }
}

static void store_cache(void* base, int dtype, size_t i, float x, float kv_scale) {
  switch (dtype) {
    case ORC_F32: ((float*)base)[i] = x; break;
    case ORC_BF16: ((uint16_t*)base)[i] = orc_bf16_encode(x); break;
    default: ((uint8_t*)base)[i] = orc_fp8_e4m3_encode(x / kv_scale); break;
  }
}

/* ------------------------------------------------------------------ */
/* Cache write and gather                                              */
/* ------------------------------------------------------------------ */

/* k, v: [num_tokens, num_kv_heads, head_dim] of src_dtype (f32 or bf16).
 * caches: [num_blocks, num_kv_heads, block_size, head_dim] of cache_dtype.
 * slot_mapping[t] = block_id * block_size + offset, negative = skip. */
int orc_reshape_and_cache(const void* k, const void* v, int src_dtype, int num_tokens,
                          int num_kv_heads, int head_dim, void* k_cache, void* v_cache,
                          int cache_dtype, int num_blocks, int block_size,
                          const int64_t* slot_mapping, float kv_scale) {
  if (src_dtype != ORC_F32 && src_dtype != ORC_BF16) return ORC_ERR_ARG;
  if (elem_size(cache_dtype) == 0 || block_size <= 0 || head_dim <= 0) return ORC_ERR_ARG;
  for (int t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t blk = slot / block_size, off = slot % block_size;
    if (blk >= num_blocks) return ORC_ERR_RANGE;
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int i = 0; i < head_dim; ++i) {
        size_t src = ((size_t)t * num_kv_heads + h) * head_dim + i;
        size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim + i;
        store_cache(k_cache, cache_dtype, dst, load_as_f32(k, src_dtype, src), kv_scale);
        store_cache(v_cache, cache_dtype, dst, load_as_f32(v, src_dtype, src), kv_scale);
      }
    }
  }
  return ORC_OK;
}

/* Contiguous copy of each sequence's cached tokens:
 * k_out[cu_seq_lens[s] + p][h][:] = k_cache[block_tables[s][p / bs]][h][p % bs][:]. */
int orc_gather_kv(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                  int cache_dtype, int num_blocks, int num_kv_heads, int block_size,
                  int head_dim, const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* seq_lens, const int64_t* cu_seq_lens, int num_seqs) {
  size_t es = elem_size(cache_dtype);
  if (es == 0) return ORC_ERR_ARG;
  size_t row = (size_t)head_dim * es;
  for (int s = 0; s < num_seqs; ++s) {
    for (int p = 0; p < seq_lens[s]; ++p) {
      int j = p / block_size, off = p % block_size;
      if (j >= max_blocks_per_seq) return ORC_ERR_RANGE;
      int32_t blk = block_tables[(size_t)s * max_blocks_per_seq + j];
      if (blk < 0 || blk >= num_blocks) return ORC_ERR_RANGE;
      for (int h = 0; h < num_kv_heads; ++h) {
        size_t src = (((size_t)blk * num_kv_heads + h) * block_size + off) * row;
        size_t dst = (((size_t)cu_seq_lens[s] + p) * num_kv_heads + h) * row;
        memcpy((char*)k_out + dst, (const char*)k_cache + src, row);
        memcpy((char*)v_out + dst, (const char*)v_cache + src, row);
      }
    }
  }
  return ORC_OK;
}

/* Whole-block copies between pools (copy-on-write of a shared block, swap
 * to host memory and back): for each pair (src, dst), block src of both
 * source caches replaces block dst of both destination caches.  A block of
 * one cache is num_kv_heads * block_size * head_dim contiguous elements.
 * The pairs are applied in order; an id outside its pool stops the call
 * with ORC_ERR_RANGE before anything of that pair is written. */
int orc_copy_blocks(void* k_dst, void* v_dst, int dst_blocks, const void* k_src, const void* v_src,
                    int src_blocks, int cache_dtype, int num_kv_heads, int block_size, int head_dim,
                    const int64_t* pairs, int num_pairs) {
  size_t es = elem_size(cache_dtype);
  if (es == 0) return ORC_ERR_ARG;
  size_t blk = (size_t)num_kv_heads * block_size * head_dim * es;
  for (int i = 0; i < num_pairs; ++i) {
    int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) return ORC_ERR_RANGE;
    memcpy((char*)k_dst + (size_t)dst * blk, (const char*)k_src + (size_t)src * blk, blk);
    memcpy((char*)v_dst + (size_t)dst * blk, (const char*)v_src + (size_t)src * blk, blk);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Attention                                                           */
/* ------------------------------------------------------------------ */

typedef struct {
  /* problem */
  const void* q;
  int q_dtype;
  const void* k_cache;
  const void* v_cache;
  int cache_dtype;
  int num_blocks, num_kv_heads, block_size, head_dim;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  int num_seqs, num_q_heads;
  double scale, kv_scale;
  /* partition mode (partition_tokens > 0) writes partials instead of out */
  int partition_tokens, max_partitions;
  double* out;    /* [B, Hq, d] */
  double* o_part; /* [B, Hq, P, d] */
  double* m_part; /* [B, Hq, P] */
  double* l_part; /* [B, Hq, P] */
  /* sliding window (window > 0): a sequence of length L attends only its
   * first `sinks` tokens and its last `window` tokens */
  int window, sinks;
  /* multi-token queries (q_start != NULL): sequence s has the query tokens
   * q_start[s] .. q_start[s+1]-1 of q [total, Hq, d]; out is [total, Hq, d] */
  const int32_t* q_start;
  /* work distribution over (sequence, kv head) pairs */
  int next_unit;
  pthread_mutex_t lock;
  int status;
} orc_job;

/* Is token p of a sequence of length L attended?  Without a window every
 * p < L is.  With one, only the first `sinks` tokens (attention sinks) and
 * the last `window` tokens are ("PagedAttention por dentro", sections
 * "Sliding window attention" and "StreamingLLM (Xiao et al., 2024): los
 * attention sinks"). */
static int attended(const orc_job* jb, int L, int p) {
  if (p < 0 || p >= L) return 0;
  if (jb->window <= 0 || L <= jb->window) return 1;
  return p < jb->sinks || p >= L - jb->window;
}

/* Copy sequence s, kv head h into contiguous fp64 K and V ([L][d]) through
 * the block table: logical token p lives in physical block table[p / bs] at
 * offset p % bs.  Tokens that are not attended are left zero and their
 * blocks are never looked at (an engine frees the blocks that fell out of
 * the window). */
static int gather_f64(const orc_job* jb, int s, int h, int L, double* K, double* V) {
  const int d = jb->head_dim, bs = jb->block_size;
  for (int p = 0; p < L; ++p) {
    if (!attended(jb, L, p)) {
      for (int i = 0; i < d; ++i) K[(size_t)p * d + i] = V[(size_t)p * d + i] = 0.0;
      continue;
    }
    int j = p / bs, off = p % bs;
    if (j >= jb->max_blocks_per_seq) return ORC_ERR_RANGE;
    int32_t blk = jb->block_tables[(size_t)s * jb->max_blocks_per_seq + j];
    if (blk < 0 || blk >= jb->num_blocks) return ORC_ERR_RANGE;
    size_t base = (((size_t)blk * jb->num_kv_heads + h) * bs + off) * d;
    for (int i = 0; i < d; ++i) {
      K[(size_t)p * d + i] = load_cache_f64(jb->k_cache, jb->cache_dtype, base + i, jb->kv_scale);
      V[(size_t)p * d + i] = load_cache_f64(jb->v_cache, jb->cache_dtype, base + i, jb->kv_scale);
    }
  }
  return ORC_OK;
}

/* softmax(scale * q . K[t]) . V over the attended tokens t in [t0, t1)
 * (keep[t] != 0); returns the normalised output in o, the largest scaled
 * score in *m_out and the sum of exp(score - max) in *l_out.  With no token
 * attended: o = 0, m = -inf, l = 0. */
static void attend_f64(const double* qv, const double* K, const double* V, const unsigned char* keep,
                       int t0, int t1, int d, double scale, double* o, double* m_out, double* l_out,
                       double* w) {
  double m = -INFINITY;
  for (int t = t0; t < t1; ++t) {
    if (!keep[t]) continue;
    double dot = 0.0;
    for (int i = 0; i < d; ++i) dot += qv[i] * K[(size_t)t * d + i];
    w[t - t0] = scale * dot;
    if (w[t - t0] > m) m = w[t - t0];
  }
  double l = 0.0;
  for (int t = t0; t < t1; ++t) {
    if (!keep[t]) continue;
    w[t - t0] = exp(w[t - t0] - m);
    l += w[t - t0];
  }
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  for (int t = t0; t < t1; ++t) {
    if (!keep[t]) continue;
    for (int i = 0; i < d; ++i) o[i] += w[t - t0] * V[(size_t)t * d + i];
  }
  if (l > 0.0)
    for (int i = 0; i < d; ++i) o[i] /= l;
  *m_out = m;
  *l_out = l;
}

/* Multi-token queries of one (sequence, kv head): the T query tokens of the
 * sequence are its last T positions; query token i sits at position
 * L - T + i and attends positions 0 .. L - T + i, itself included (the causal
 * mask inside the chunk). */
static int run_unit_multi(orc_job* jb, int s, int h, int L, const double* K, const double* V,
                          double* qv, double* w, unsigned char* keep) {
  const int d = jb->head_dim;
  const int g = jb->num_q_heads / jb->num_kv_heads;
  const int q0 = jb->q_start[s], T = jb->q_start[s + 1] - q0;
  if (T < 0 || T > L) return ORC_ERR_RANGE;
  for (int p = 0; p < L; ++p) keep[p] = 1;
  for (int i = 0; i < T; ++i) {
    const int pos = L - T + i;
    for (int qh = h * g; qh < (h + 1) * g; ++qh) {
      size_t qbase = ((size_t)(q0 + i) * jb->num_q_heads + qh) * d;
      for (int c = 0; c < d; ++c) qv[c] = (double)load_as_f32(jb->q, jb->q_dtype, qbase + c);
      double m, l;
      attend_f64(qv, K, V, keep, 0, pos + 1, d, jb->scale, jb->out + qbase, &m, &l, w);
    }
  }
  return ORC_OK;
}

static int run_unit(orc_job* jb, int unit, double* K, double* V, double* qv, double* w,
                    unsigned char* keep) {
  const int d = jb->head_dim;
  const int g = jb->num_q_heads / jb->num_kv_heads;
  const int s = unit / jb->num_kv_heads, h = unit % jb->num_kv_heads;
  const int L = jb->seq_lens[s];
  if (L < 0) return ORC_ERR_RANGE;
  int rc = gather_f64(jb, s, h, L, K, V);
  if (rc != ORC_OK) return rc;
  if (jb->q_start) return run_unit_multi(jb, s, h, L, K, V, qv, w, keep);
  for (int p = 0; p < L; ++p) keep[p] = (unsigned char)attended(jb, L, p);
  for (int qh = h * g; qh < (h + 1) * g; ++qh) {
    size_t qbase = ((size_t)s * jb->num_q_heads + qh) * d;
    for (int i = 0; i < d; ++i) qv[i] = (double)load_as_f32(jb->q, jb->q_dtype, qbase + i);
    if (jb->partition_tokens <= 0) {
      double* o = jb->out + qbase;
      if (L == 0) {
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        continue;
      }
      double m, l;
      attend_f64(qv, K, V, keep, 0, L, d, jb->scale, o, &m, &l, w);
    } else {
      const int P = jb->partition_tokens;
      for (int p = 0; p < jb->max_partitions; ++p) {
        size_t pi = ((size_t)s * jb->num_q_heads + qh) * jb->max_partitions + p;
        double* o = jb->o_part + pi * d;
        int t0 = p * P, t1 = (p + 1) * P < L ? (p + 1) * P : L;
        if (t0 >= t1) { /* empty partition: the neutral element of the merge */
          for (int i = 0; i < d; ++i) o[i] = 0.0;
          jb->m_part[pi] = -INFINITY;
          jb->l_part[pi] = 0.0;
          continue;
        }
        attend_f64(qv, K, V, keep, t0, t1, d, jb->scale, o, &jb->m_part[pi], &jb->l_part[pi], w);
      }
    }
  }
  return ORC_OK;
}

static int max_len(const orc_job* jb) {
  int mx = 1;
  for (int s = 0; s < jb->num_seqs; ++s)
    if (jb->seq_lens[s] > mx) mx = jb->seq_lens[s];
  return mx;
}

static void* worker(void* arg) {
  orc_job* jb = (orc_job*)arg;
  const int d = jb->head_dim;
  const size_t L = (size_t)max_len(jb);
  double* K = (double*)malloc(L * d * sizeof(double));
  double* V = (double*)malloc(L * d * sizeof(double));
  double* qv = (double*)malloc((size_t)d * sizeof(double));
  double* w = (double*)malloc(L * sizeof(double));
  unsigned char* keep = (unsigned char*)malloc(L);
  int rc = (K && V && qv && w && keep) ? ORC_OK : ORC_ERR_NOMEM;
  const int units = jb->num_seqs * jb->num_kv_heads;
  while (rc == ORC_OK) {
    pthread_mutex_lock(&jb->lock);
    int u = jb->next_unit++;
    pthread_mutex_unlock(&jb->lock);
    if (u >= units) break;
    rc = run_unit(jb, u, K, V, qv, w, keep);
  }
  if (rc != ORC_OK) {
    pthread_mutex_lock(&jb->lock);
    jb->status = rc;
    jb->next_unit = units; /* stop the others */
    pthread_mutex_unlock(&jb->lock);
  }
  free(K);
  free(V);
  free(qv);
  free(w);
  free(keep);
  return NULL;
}

static int run_job(orc_job* jb, int num_threads) {
  if (jb->num_kv_heads <= 0 || jb->num_q_heads % jb->num_kv_heads != 0) return ORC_ERR_ARG;
  if (elem_size(jb->cache_dtype) == 0 || (jb->q_dtype != ORC_F32 && jb->q_dtype != ORC_BF16))
    return ORC_ERR_ARG;
  if (num_threads < 1) num_threads = 1;
  jb->next_unit = 0;
  jb->status = ORC_OK;
  pthread_mutex_init(&jb->lock, NULL);
  if (num_threads == 1) {
    worker(jb);
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)num_threads);
    if (!th) return ORC_ERR_NOMEM;
    for (int i = 0; i < num_threads; ++i) pthread_create(&th[i], NULL, worker, jb);
    for (int i = 0; i < num_threads; ++i) pthread_join(th[i], NULL);
    free(th);
  }
  pthread_mutex_destroy(&jb->lock);
  return jb->status;
}

/* out: [num_seqs, num_q_heads, head_dim] doubles.  window > 0: each
 * sequence attends only its first `sinks` and last `window` tokens. */
int orc_paged_attention_decode_window(double* out, const void* q, int q_dtype, int num_seqs,
                                      int num_q_heads, const void* k_cache, const void* v_cache,
                                      int cache_dtype, int num_blocks, int num_kv_heads,
                                      int block_size, int head_dim, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* seq_lens, double scale,
                                      double kv_scale, int window, int sinks, int num_threads) {
  if (window < 0 || sinks < 0) return ORC_ERR_ARG;
  orc_job jb;
  memset(&jb, 0, sizeof jb);
  jb.q = q;
  jb.q_dtype = q_dtype;
  jb.k_cache = k_cache;
  jb.v_cache = v_cache;
  jb.cache_dtype = cache_dtype;
  jb.num_blocks = num_blocks;
  jb.num_kv_heads = num_kv_heads;
  jb.block_size = block_size;
  jb.head_dim = head_dim;
  jb.block_tables = block_tables;
  jb.max_blocks_per_seq = max_blocks_per_seq;
  jb.seq_lens = seq_lens;
  jb.num_seqs = num_seqs;
  jb.num_q_heads = num_q_heads;
  jb.scale = scale;
  jb.kv_scale = kv_scale;
  jb.window = window;
  jb.sinks = sinks;
  jb.out = out;
  return run_job(&jb, num_threads);
}

int orc_paged_attention_decode(double* out, const void* q, int q_dtype, int num_seqs,
                               int num_q_heads, const void* k_cache, const void* v_cache,
                               int cache_dtype, int num_blocks, int num_kv_heads, int block_size,
                               int head_dim, const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* seq_lens, double scale, double kv_scale,
                               int num_threads) {
  return orc_paged_attention_decode_window(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache,
                                           cache_dtype, num_blocks, num_kv_heads, block_size, head_dim,
                                           block_tables, max_blocks_per_seq, seq_lens, scale, kv_scale,
                                           0, 0, num_threads);
}

/* Per-partition attention: partition p of sequence s covers tokens
 * [p * partition_tokens, (p + 1) * partition_tokens) clipped to seq_lens[s].
 * o_part [B, Hq, P, d] (normalised within the partition), m_part and l_part
 * [B, Hq, P] (largest scaled score, sum of exp(score - m)).  An empty
 * partition gets o = 0, m = -inf, l = 0. */
int orc_partition_attention(double* o_part, double* m_part, double* l_part, const void* q,
                            int q_dtype, int num_seqs, int num_q_heads, const void* k_cache,
                            const void* v_cache, int cache_dtype, int num_blocks,
                            int num_kv_heads, int block_size, int head_dim,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* seq_lens, double scale, double kv_scale,
                            int partition_tokens, int max_partitions, int num_threads) {
  if (partition_tokens <= 0 || max_partitions <= 0) return ORC_ERR_ARG;
  orc_job jb;
  memset(&jb, 0, sizeof jb);
  jb.q = q;
  jb.q_dtype = q_dtype;
  jb.k_cache = k_cache;
  jb.v_cache = v_cache;
  jb.cache_dtype = cache_dtype;
  jb.num_blocks = num_blocks;
  jb.num_kv_heads = num_kv_heads;
  jb.block_size = block_size;
  jb.head_dim = head_dim;
  jb.block_tables = block_tables;
  jb.max_blocks_per_seq = max_blocks_per_seq;
  jb.seq_lens = seq_lens;
  jb.num_seqs = num_seqs;
  jb.num_q_heads = num_q_heads;
  jb.scale = scale;
  jb.kv_scale = kv_scale;
  jb.partition_tokens = partition_tokens;
  jb.max_partitions = max_partitions;
  jb.o_part = o_part;
  jb.m_part = m_part;
  jb.l_part = l_part;
  return run_job(&jb, num_threads);
}

/* Log-sum-exp merge of the partitions that hold at least one token
 * (the first ceil(seq_len / partition_tokens) of them):
 *   M = max_p m_p,  w_p = l_p * exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
 * A sequence of length 0 gets a zero row. */
int orc_split_kv_reduce(double* out, const double* o_part, const double* m_part,
                        const double* l_part, const int32_t* seq_lens, int num_seqs,
                        int num_q_heads, int head_dim, int partition_tokens, int max_partitions) {
  if (partition_tokens <= 0) return ORC_ERR_ARG;
  for (int s = 0; s < num_seqs; ++s) {
    int L = seq_lens[s];
    if (L < 0) return ORC_ERR_RANGE;
    int np = (L + partition_tokens - 1) / partition_tokens;
    if (np > max_partitions) return ORC_ERR_RANGE;
    for (int qh = 0; qh < num_q_heads; ++qh) {
      size_t row = (size_t)s * num_q_heads + qh;
      double* o = out + row * head_dim;
      for (int i = 0; i < head_dim; ++i) o[i] = 0.0;
      if (np == 0) continue;
      double M = -INFINITY;
      for (int p = 0; p < np; ++p)
        if (m_part[row * max_partitions + p] > M) M = m_part[row * max_partitions + p];
      double den = 0.0;
      for (int p = 0; p < np; ++p) {
        size_t pi = row * max_partitions + p;
        double wp = l_part[pi] * exp(m_part[pi] - M);
        den += wp;
        for (int i = 0; i < head_dim; ++i) o[i] += wp * o_part[pi * head_dim + i];
      }
      for (int i = 0; i < head_dim; ++i) o[i] /= den;
    }
  }
  return ORC_OK;
}

/* Paged attention of several query tokens per sequence (chunked prefill,
 * the verification step of speculative decoding).  Sequence s has the
 * query tokens q_start[s] .. q_start[s+1]-1 of q [total, Hq, d]; they are
 * the sequence's last T = q_start[s+1] - q_start[s] positions, already in
 * the cache, and query token i attends positions 0 .. seq_lens[s] - T + i
 * (causal inside the chunk).  out: [total, Hq, d] doubles.  T = 1 for every
 * sequence is decode. */
int orc_paged_attention_multi(double* out, const void* q, int q_dtype, const int32_t* q_start,
                              int num_seqs, int num_q_heads, const void* k_cache, const void* v_cache,
                              int cache_dtype, int num_blocks, int num_kv_heads, int block_size,
                              int head_dim, const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* seq_lens, double scale, double kv_scale, int num_threads) {
  if (!q_start || q_start[0] != 0) return ORC_ERR_ARG;
  for (int s = 0; s < num_seqs; ++s)
    if (q_start[s + 1] < q_start[s]) return ORC_ERR_ARG;
  orc_job jb;
  memset(&jb, 0, sizeof jb);
  jb.q = q;
  jb.q_dtype = q_dtype;
  jb.q_start = q_start;
  jb.k_cache = k_cache;
  jb.v_cache = v_cache;
  jb.cache_dtype = cache_dtype;
  jb.num_blocks = num_blocks;
  jb.num_kv_heads = num_kv_heads;
  jb.block_size = block_size;
  jb.head_dim = head_dim;
  jb.block_tables = block_tables;
  jb.max_blocks_per_seq = max_blocks_per_seq;
  jb.seq_lens = seq_lens;
  jb.num_seqs = num_seqs;
  jb.num_q_heads = num_q_heads;
  jb.scale = scale;
  jb.kv_scale = kv_scale;
  jb.out = out;
  return run_job(&jb, num_threads);
}
