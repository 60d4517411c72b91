/*
 * pd_oracle.c -- plain, slow fp64 CPU oracle for ragged attention over a paged
 * KV cache and for the KV-cache append / pack / unpack copies.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker, not the product: only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library; the two meet
 * only in the seeded inputs both consume.
 *
 * What it computes (the definition, written out; no tiling, splitting, online
 * softmax or any other reordering):
 *
 *   Perplexity, "Disaggregated prefill and decode" (2025), section "Prefill vs
 *   Decode performance": attention of every request runs over the kv_len tokens
 *   held in its KV cache; a decode request brings one new token (qo_len = 1), a
 *   prefill request brings many (large qo_len).
 *   Same post, section "Sharded KV cache transfers" and its figure on NHD and
 *   HND layouts: inside a page the HND layout puts the head index before the
 *   token index, so page p holds [Hkv][page_size][head_dim].
 *   The NHD layout of the same figure puts the token first: page p holds
 *   [page_size][Hkv][head_dim]. Every function takes the layout of its pools.
 *   Same post, section "Qwen3-Coder": the model uses grouped-query attention,
 *   several query heads sharing one KV head.
 *
 *   For request r, query row i in [0, qo_len), query head h, KV head
 *   g = h / (Hq / Hkv) (contiguous groups), logical key j in [0, kv_len):
 *     page  = page_indices[page_indptr[r] + j / page_size], slot = j % page_size
 *     k_j   = k_pool[page][g][slot][:] (HND) or k_pool[page][slot][g][:] (NHD),
 *             v_j likewise
 *     s_j   = scale * <q_i,h , k_j>      for j <= kv_len - qo_len + i (causal,
 *             the new rows are the last qo_len positions), every j otherwise;
 *             masked keys get s_j = -inf
 *     m     = max_j s_j,  l = sum_j exp(s_j - m)
 *     o     = sum_j exp(s_j - m) v_j / l,     lse = m + ln(l)   (natural log)
 *   A row with no allowed key returns o = 0 and lse = -inf.
 *
 *   Append (same post, section "KV Messenger": a layer's page copies start as
 *   soon as the model has appended that layer's KV entries): new token i of
 *   request r (n_r new tokens) sits at logical position kv_len[r] - n_r + i.
 *
 *   Pack / unpack (same post, "Sharded KV cache transfers": pages are copied
 *   between a prefiller and a decoder, and pages are split or rebuilt when the
 *   two sides differ): request r's KV of all layers is gathered into one
 *   contiguous block laid out [layer][K,V][Hkv][kv_len][head_dim]; unpack
 *   scatters that block into a pool with its own page size and page table.
 *
 * Inputs are the exact fp32 or bf16 values the GPU receives, widened to fp64.
 * Built with -DORACLE_MUTANT=n, one deliberate mistake is planted (tests show
 * that the pins catch each one); the default build has none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_HND = 0, ORACLE_NHD = 1 };

/* element offset of (page, kv head g, slot, dim 0) in one pool:
 * HND [page][Hkv][P][D], NHD [page][P][Hkv][D] */
static int64_t pool_offset(int layout, int64_t page, int g, int slot, int hkv, int p, int d) {
#if ORACLE_MUTANT == 12
  layout = ORACLE_HND; /* planted: an NHD pool read as HND */
#endif
  if (layout == ORACLE_NHD) return ((page * p + slot) * (int64_t)hkv + g) * d;
  return ((page * hkv + g) * (int64_t)p + slot) * d;
}

/* one stored element (fp32 or bf16 bit pattern) widened to fp64 */
static double elem(const void *base, int64_t idx, int dtype) {
  if (dtype == ORACLE_BF16) {
    uint32_t u = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
  }
  return (double)((const float *)base)[idx];
}

typedef struct {
  int32_t batch, hq, hkv, d, p, dtype, causal, layout;
  double scale;
  const int32_t *qo_indptr, *kv_len, *page_indptr, *page_indices;
  const void *q, *k_pool, *v_pool;
} attn_args;

/* element offset of (page, kv head g, slot, dim 0) in the pools of a */
static int64_t kv_offset(const attn_args *a, int64_t page, int g, int slot) {
  return pool_offset(a->layout, page, g, slot, a->hkv, a->p, a->d);
}

/* physical page holding logical token j of request r */
static int64_t page_of(const attn_args *a, int r, int64_t j) {
#if ORACLE_MUTANT == 5
  return a->page_indices[a->page_indptr[r] + j / a->p];
#else
  return a->page_indices[a->page_indptr[r] + j / a->p];
#endif
}

static int slot_of(const attn_args *a, int64_t j) {
#if ORACLE_MUTANT == 5
  return (int)((j % a->p) ^ 1); /* planted: neighbouring slots swapped */
#else
  return (int)(j % a->p);
#endif
}

/* the attention of one (request r, query row i, query head h); s holds kv_len doubles */
static void attend_row(const attn_args *a, int r, int i, int h, double *o, double *lse, double *s) {
  const int qo_len = a->qo_indptr[r + 1] - a->qo_indptr[r];
  const int n = a->kv_len[r];
  const int group = a->hq / a->hkv;
#if ORACLE_MUTANT == 2
  const int g = h % a->hkv; /* planted: interleaved instead of contiguous groups */
#else
  const int g = h / group;
#endif
  const int64_t row = (int64_t)a->qo_indptr[r] + i;
  const int64_t q_off = (row * a->hq + h) * a->d;
#if ORACLE_MUTANT == 3
  const int64_t last = a->causal ? (int64_t)n - qo_len + i - 1 : (int64_t)n - 1; /* planted: off by one */
#elif ORACLE_MUTANT == 4
  const int64_t last = a->causal ? (int64_t)i : (int64_t)n - 1; /* planted: top-left alignment */
#else
  const int64_t last = a->causal ? (int64_t)n - qo_len + i : (int64_t)n - 1;
#endif
#if ORACLE_MUTANT == 1
  const double scale = 1.0; /* planted: scale dropped */
#else
  const double scale = a->scale;
#endif
  (void)group;

  /* scores */
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    if (j > last) {
      s[j] = -INFINITY;
      continue;
    }
    const int64_t k_off = kv_offset(a, page_of(a, r, j), g, slot_of(a, j));
    double dot = 0.0;
    for (int dd = 0; dd < a->d; ++dd)
      dot += elem(a->q, q_off + dd, a->dtype) * elem(a->k_pool, k_off + dd, a->dtype);
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }
  for (int dd = 0; dd < a->d; ++dd) o[dd] = 0.0;
  if (m == -INFINITY) { /* no allowed key */
    *lse = -INFINITY;
    return;
  }
  /* softmax weights and the weighted sum of values */
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    if (s[j] == -INFINITY) continue; /* exp(-inf) = 0 adds nothing */
    const double w = exp(s[j] - m);
    l += w;
#if ORACLE_MUTANT == 7
    const void *vsrc = a->k_pool; /* planted: values read from the key pool */
#else
    const void *vsrc = a->v_pool;
#endif
    const int64_t v_off = kv_offset(a, page_of(a, r, j), g, slot_of(a, j));
    for (int dd = 0; dd < a->d; ++dd) o[dd] += w * elem(vsrc, v_off + dd, a->dtype);
  }
  for (int dd = 0; dd < a->d; ++dd) o[dd] /= l;
#if ORACLE_MUTANT == 6
  *lse = m + log2(l); /* planted: base-2 logarithm */
#else
  *lse = m + log(l);
#endif
}

static int check_attn(const attn_args *a) {
  if (a->batch < 0 || a->hq <= 0 || a->hkv <= 0 || a->d <= 0 || a->p <= 0) return -1;
  if (a->layout != ORACLE_HND && a->layout != ORACLE_NHD) return -1;
  if (a->hq % a->hkv != 0) return -1;
  for (int r = 0; r < a->batch; ++r) {
    const int qo = a->qo_indptr[r + 1] - a->qo_indptr[r];
    const int n = a->kv_len[r];
    if (qo < 0 || n < 0) return -1;
    if (a->causal && qo > n) return -1;
    const int64_t pages = a->page_indptr[r + 1] - a->page_indptr[r];
    if (pages * a->p < n) return -1;
  }
  return 0;
}

static int threads_of(int nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/*
 * Every output row. o: fp64 [total_qo][hq][d]; lse: fp64 [total_qo][hq].
 * One task per (request, query head); OpenMP spreads the tasks over nthreads
 * (<= 0: the OpenMP default). Returns 0, or -1 for inconsistent sizes.
 */
int oracle_attention(int32_t batch, const int32_t *qo_indptr, const int32_t *kv_len,
                     const int32_t *page_indptr, const int32_t *page_indices, int32_t hq,
                     int32_t hkv, int32_t d, int32_t p, int32_t dtype, double scale,
                     int32_t causal, int32_t layout, const void *q, const void *k_pool,
                     const void *v_pool, double *o, double *lse, int32_t nthreads) {
  attn_args a = {batch, hq, hkv, d, p, dtype, causal, layout, scale, qo_indptr, kv_len,
                 page_indptr, page_indices, q, k_pool, v_pool};
  if (check_attn(&a)) return -1;
  int max_n = 1;
  for (int r = 0; r < batch; ++r)
    if (kv_len[r] > max_n) max_n = kv_len[r];
  const int64_t tasks = (int64_t)batch * hq;
  int err = 0;
#pragma omp parallel num_threads(threads_of(nthreads))
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)max_n);
    if (!s) {
#pragma omp atomic write
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t t = 0; t < tasks; ++t) {
        const int r = (int)(t / hq), h = (int)(t % hq);
        const int qo_len = qo_indptr[r + 1] - qo_indptr[r];
        for (int i = 0; i < qo_len; ++i) {
          const int64_t row = (int64_t)qo_indptr[r] + i;
          attend_row(&a, r, i, h, o + (row * hq + h) * d, lse + row * hq + h, s);
        }
      }
      free(s);
    }
  }
  return err ? -2 : 0;
}

/*
 * Selected outputs only: for each k < n_sel, the query row sel_row[k] (a global
 * row of q) and query head sel_head[k]. o: fp64 [n_sel][d]; lse: fp64 [n_sel].
 */
int oracle_attention_rows(int32_t batch, const int32_t *qo_indptr, const int32_t *kv_len,
                          const int32_t *page_indptr, const int32_t *page_indices, int32_t hq,
                          int32_t hkv, int32_t d, int32_t p, int32_t dtype, double scale,
                          int32_t causal, int32_t layout, const void *q, const void *k_pool,
                          const void *v_pool, int64_t n_sel, const int32_t *sel_row,
                          const int32_t *sel_head, double *o, double *lse, int32_t nthreads) {
  attn_args a = {batch, hq, hkv, d, p, dtype, causal, layout, scale, qo_indptr, kv_len,
                 page_indptr, page_indices, q, k_pool, v_pool};
  if (check_attn(&a)) return -1;
  int max_n = 1;
  for (int r = 0; r < batch; ++r)
    if (kv_len[r] > max_n) max_n = kv_len[r];
  int err = 0;
#pragma omp parallel num_threads(threads_of(nthreads))
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)max_n);
    if (!s) {
#pragma omp atomic write
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t k = 0; k < n_sel; ++k) {
        /* request owning the row: last r with qo_indptr[r] <= row */
        int r = 0;
        while (r + 1 < batch && qo_indptr[r + 1] <= sel_row[k]) ++r;
        const int i = sel_row[k] - qo_indptr[r];
        if (i < 0 || i >= qo_indptr[r + 1] - qo_indptr[r] || sel_head[k] < 0 || sel_head[k] >= hq) {
#pragma omp atomic write
          err = 1;
          continue;
        }
        attend_row(&a, r, i, sel_head[k], o + k * d, lse + k, s);
      }
      free(s);
    }
  }
  return err ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Byte copies: append, pack, unpack. es = bytes per element.                 */
/* ------------------------------------------------------------------------- */

/* byte offset of (page, head, slot) in one layer's pool */
static int64_t pool_row_bytes(int layout, int64_t page, int h, int slot, int hkv, int p, int d, int es) {
  return pool_offset(layout, page, h, slot, hkv, p, d) * es;
}

static int layout_ok(int32_t layout) { return layout == ORACLE_HND || layout == ORACLE_NHD; }

/*
 * Append: new-token row idx (request r's token i, idx = new_indptr[r] + i) of
 * k_new / v_new ([total_new][hkv][d]) goes to logical position
 * kv_len[r] - n_r + i of request r's pages. Returns -1 on an inconsistent table.
 */
int oracle_kv_append(int32_t batch, const int32_t *new_indptr, const int32_t *kv_len,
                     const int32_t *page_indptr, const int32_t *page_indices, int32_t num_pages,
                     int32_t hkv, int32_t d, int32_t p, int32_t es, int32_t layout,
                     const void *k_new, const void *v_new, void *k_pool, void *v_pool) {
  const int64_t row_bytes = (int64_t)d * es;
  if (!layout_ok(layout)) return -1;
  for (int r = 0; r < batch; ++r) {
    const int n_new = new_indptr[r + 1] - new_indptr[r];
    if (n_new < 0 || n_new > kv_len[r]) return -1;
    for (int i = 0; i < n_new; ++i) {
#if ORACLE_MUTANT == 10
      const int64_t t = (int64_t)kv_len[r] - n_new + (n_new - 1 - i); /* planted: reversed */
#else
      const int64_t t = (int64_t)kv_len[r] - n_new + i;
#endif
      const int64_t pi = page_indptr[r] + t / p;
      if (pi >= page_indptr[r + 1]) return -1;
      const int64_t page = page_indices[pi];
      if (page < 0 || page >= num_pages) return -1;
      const int slot = (int)(t % p);
      const int64_t src_row = (int64_t)new_indptr[r] + i;
      for (int h = 0; h < hkv; ++h) {
        const int64_t src = (src_row * hkv + h) * row_bytes;
        const int64_t dst = pool_row_bytes(layout, page, h, slot, hkv, p, d, es);
        memcpy((char *)k_pool + dst, (const char *)k_new + src, (size_t)row_bytes);
        memcpy((char *)v_pool + dst, (const char *)v_new + src, (size_t)row_bytes);
      }
    }
  }
  return 0;
}

/* byte offset of (layer, K or V, head, token) inside one request's packed block */
static int64_t packed_row_bytes(int layer, int kv, int h, int64_t t, int64_t n, int hkv, int d, int es) {
#if ORACLE_MUTANT == 8
  return ((((int64_t)layer * 2 + kv) * n + t) * hkv + h) * d * es; /* planted: token before head */
#else
  return ((((int64_t)layer * 2 + kv) * hkv + h) * n + t) * d * es;
#endif
}

/*
 * Pack: for every request r, layer, K/V, head h and token t < kv_len[r]:
 *   dst[dst_offsets[r] + packed(layer, kv, h, t)] = pool_layer,kv[page(r, t)][h][t % p]
 * ([page(r, t)][t % p][h] for NHD pools)
 * where layer l's pools start at k_pool / v_pool + l * layer_stride bytes.
 */
/*
 * Head range (same post, "Sharded KV cache transfers": when prefiller and
 * decoder shard the heads differently, pages are split or rebuilt): pack and
 * unpack move heads [head_begin, head_begin + head_count) of a pool holding hkv
 * heads; the block then holds head_count heads, [layer][K,V][head_count][kv_len]
 * [head_dim]. The full range (0, hkv) is the plain handoff.
 */
static int head_range_ok(int32_t hkv, int32_t head_begin, int32_t head_count) {
  return head_begin >= 0 && head_count >= 1 && head_begin + head_count <= hkv;
}

/* pool head that packed head h of the range maps to */
static int pool_head(int32_t head_begin, int h) {
#if ORACLE_MUTANT == 11
  (void)head_begin;
  return h; /* planted: the range's offset into the pool is dropped */
#else
  return head_begin + h;
#endif
}

int oracle_kv_pack(int32_t batch, const int32_t *kv_len, const int32_t *page_indptr,
                   const int32_t *page_indices, int32_t num_pages, int32_t num_layers,
                   int64_t layer_stride, int32_t hkv, int32_t head_begin, int32_t head_count, int32_t d,
                   int32_t p, int32_t es, int32_t layout, const void *k_pool, const void *v_pool,
                   void *dst, const int64_t *dst_offsets) {
  const int64_t row_bytes = (int64_t)d * es;
  if (!head_range_ok(hkv, head_begin, head_count) || !layout_ok(layout)) return -1;
  for (int r = 0; r < batch; ++r) {
    const int64_t n = kv_len[r];
    if ((int64_t)(page_indptr[r + 1] - page_indptr[r]) * p < n) return -1;
    for (int layer = 0; layer < num_layers; ++layer)
      for (int kv = 0; kv < 2; ++kv) {
        const char *pool = (const char *)(kv ? v_pool : k_pool) + (int64_t)layer * layer_stride;
        for (int h = 0; h < head_count; ++h)
          for (int64_t t = 0; t < n; ++t) {
            const int64_t page = page_indices[page_indptr[r] + t / p];
            if (page < 0 || page >= num_pages) return -1;
            const int64_t src =
                pool_row_bytes(layout, page, pool_head(head_begin, h), (int)(t % p), hkv, p, d, es);
            const int64_t out = dst_offsets[r] + packed_row_bytes(layer, kv, h, t, n, head_count, d, es);
            memcpy((char *)dst + out, pool + src, (size_t)row_bytes);
          }
      }
  }
  return 0;
}

/*
 * Unpack: the inverse of pack into a pool with its own page size p and page
 * table; only slots of tokens t < kv_len[r] are written.
 */
int oracle_kv_unpack(int32_t batch, const int32_t *kv_len, const int32_t *page_indptr,
                     const int32_t *page_indices, int32_t num_pages, int32_t num_layers,
                     int64_t layer_stride, int32_t hkv, int32_t head_begin, int32_t head_count, int32_t d,
                     int32_t p, int32_t es, int32_t layout, const void *src, const int64_t *src_offsets,
                     void *k_pool, void *v_pool) {
  const int64_t row_bytes = (int64_t)d * es;
  if (!head_range_ok(hkv, head_begin, head_count) || !layout_ok(layout)) return -1;
  for (int r = 0; r < batch; ++r) {
    const int64_t n = kv_len[r];
    if ((int64_t)(page_indptr[r + 1] - page_indptr[r]) * p < n) return -1;
    for (int layer = 0; layer < num_layers; ++layer)
      for (int kv = 0; kv < 2; ++kv) {
#if ORACLE_MUTANT == 9
        char *pool = (char *)(kv ? k_pool : v_pool) + (int64_t)layer * layer_stride; /* planted: K and V swapped */
#else
        char *pool = (char *)(kv ? v_pool : k_pool) + (int64_t)layer * layer_stride;
#endif
        for (int h = 0; h < head_count; ++h)
          for (int64_t t = 0; t < n; ++t) {
            const int64_t page = page_indices[page_indptr[r] + t / p];
            if (page < 0 || page >= num_pages) return -1;
            const int slot = (int)(t % p);
            const int64_t dst = pool_row_bytes(layout, page, pool_head(head_begin, h), slot, hkv, p, d, es);
            const int64_t in = src_offsets[r] + packed_row_bytes(layer, kv, h, t, n, head_count, d, es);
            memcpy(pool + dst, (const char *)src + in, (size_t)row_bytes);
          }
      }
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* MLA decode over a paged latent cache.                                      */
/* ------------------------------------------------------------------------- */

/*
 * Perplexity, "Disaggregated prefill and decode" (2025), section
 * "Disaggregated Deployments", "DeepSeek-R1": multi-head latent attention
 * compresses the KV heads of a token into one latent vector that every query
 * head reads, so the cache holds one vector per token and is never split by
 * head. The pages give no formula; the reading taken is MLA's published
 * decode form with the up-projections folded into q and o: the stored row of
 * token j is c_j = [c_j^kv (d_c values) | k_j^rope (d_r values)], the query of
 * head h is a row of d_c + d_r values, and
 *   s_j = scale * <q_h, c_j>          over all d_c + d_r values
 *   o_h = sum_j softmax(s)_j c_j^kv   over the first d_c values only
 *   lse = m + ln(sum_j exp(s_j - m)).
 * Pool: [num_pages][p][d_c + d_r]; page of token j as for attention. One query
 * row per request; a request with no key gives o = 0, lse = -inf.
 */
static void mla_row(int32_t r, int32_t h, const int32_t *kv_len, const int32_t *page_indptr,
                    const int32_t *page_indices, int32_t hq, int32_t d_c, int32_t d_r, int32_t p,
                    int32_t dtype, double scale, const void *q, const void *kv_pool, double *o,
                    double *lse, double *s) {
  const int32_t w = d_c + d_r;
  const int64_t n = kv_len[r];
  const int64_t q_off = ((int64_t)r * hq + h) * w;
#if ORACLE_MUTANT == 13
  const int32_t score_dims = d_c; /* planted: the rope part left out of the scores */
#else
  const int32_t score_dims = w;
#endif
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    const int64_t page = page_indices[page_indptr[r] + j / p];
    const int64_t c_off = (page * p + j % p) * w;
    double dot = 0.0;
    for (int dd = 0; dd < score_dims; ++dd)
      dot += elem(q, q_off + dd, dtype) * elem(kv_pool, c_off + dd, dtype);
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }
  for (int dd = 0; dd < d_c; ++dd) o[dd] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    const double wt = exp(s[j] - m);
    l += wt;
    const int64_t page = page_indices[page_indptr[r] + j / p];
    const int64_t c_off = (page * p + j % p) * w;
    for (int dd = 0; dd < d_c; ++dd) o[dd] += wt * elem(kv_pool, c_off + dd, dtype);
  }
  for (int dd = 0; dd < d_c; ++dd) o[dd] /= l;
  *lse = m + log(l);
}

/*
 * All (request, head) pairs when sel_req is NULL (o: [batch][hq][d_c], lse:
 * [batch][hq]); else the n_sel pairs (sel_req[k], sel_head[k]) (o: [n_sel][d_c],
 * lse: [n_sel]). Returns 0, or -1 for inconsistent sizes.
 */
int oracle_mla_decode(int32_t batch, const int32_t *kv_len, const int32_t *page_indptr,
                      const int32_t *page_indices, int32_t hq, int32_t d_c, int32_t d_r, int32_t p,
                      int32_t dtype, double scale, const void *q, const void *kv_pool, int64_t n_sel,
                      const int32_t *sel_req, const int32_t *sel_head, double *o, double *lse,
                      int32_t nthreads) {
  if (batch < 0 || hq <= 0 || d_c <= 0 || d_r < 0 || p <= 0) return -1;
  int max_n = 1;
  for (int r = 0; r < batch; ++r) {
    if (kv_len[r] < 0 || (int64_t)(page_indptr[r + 1] - page_indptr[r]) * p < kv_len[r]) return -1;
    if (kv_len[r] > max_n) max_n = kv_len[r];
  }
  const int64_t tasks = sel_req != NULL ? n_sel : (int64_t)batch * hq;
  int err = 0;
#pragma omp parallel num_threads(threads_of(nthreads))
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)max_n);
    if (!s) {
#pragma omp atomic write
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t t = 0; t < tasks; ++t) {
        const int r = sel_req != NULL ? sel_req[t] : (int)(t / hq);
        const int h = sel_req != NULL ? sel_head[t] : (int)(t % hq);
        if (r < 0 || r >= batch || h < 0 || h >= hq) {
#pragma omp atomic write
          err = 1;
          continue;
        }
        mla_row(r, h, kv_len, page_indptr, page_indices, hq, d_c, d_r, p, dtype, scale, q, kv_pool,
                o + t * d_c, lse + t, s);
      }
      free(s);
    }
  }
  return err ? -1 : 0;
}

int oracle_num_threads(int32_t nthreads) { return threads_of(nthreads); }

int oracle_mutant(void) { return ORACLE_MUTANT; }
