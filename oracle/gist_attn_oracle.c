/*
 * gist_attn_oracle.c -- plain, slow fp64 CPU oracle for attention of a short
 * block of new tokens against a read-only cached KV segment.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or constant generator with the CUDA library; neither
 * side includes or links the other.
 *
 * Sources (cited by page title and section throughout):
 *   [Gist page]   "把 item 压成 KV：gist 能不能用在相关性任务上" (liam.page, 2026-10-30)
 *   [Suffix page] icman.com.cn news 64898, suffix KV-cache reuse and attention-aware
 *                 eviction; its numbered sections 1-7
 *   [KV page]     "为什么自回归推理缓存 KV，而不缓存历史 Q？" (mcfzz.com notes)
 *
 * What is computed (the plain definition, written out; no blocking, fusion or
 * reordering):
 *   [Gist page, "在线的一次 attention"]: per layer, K = cat(G_item, K_new),
 *   V = cat(G_item, V_new), X = attn(Q, K, V), with the new tokens numbered
 *   after the k cached positions, causal inside the new block, nothing written
 *   back.  [KV page, "Reusable-state"]: o_t = softmax(q_t K^T / sqrt(d_k)) V.
 *   [Gist page, "收益有多大：存储"]: G is stored per KV head; with GQA each KV
 *   head serves a contiguous group of Hq/Hkv query heads.
 *   [Gist page, "论文做了什么"]: optionally the gist mask (tokens after the gist
 *   no longer see the prompt), and the store of each layer's K/V at the gist
 *   positions as an item's cache entry.
 *   [Suffix page, §2 and the end of §5]: optionally an fp8 (E4M3) cached
 *   segment with one scale per (block, layer, K|V, KV head).
 *   [KV page, "Reusable-state"]: the append of the decode step's k_t, v_t.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - RoPE is the rotate-half form on pairs (j, j + d/2) with
 *     theta_j = rope_theta^(-2j/d); the pages only say RoPE depends on the
 *     position difference ([Gist page, "在线的一次 attention"]).
 *   - Positions are 0-based: new token i sits at pos_offset[p] + i; when no
 *     pos_offset array is given it is the number of cached positions, i.e. the
 *     query follows the cached segment.  Cached K is stored already rotated.
 *   - A new token attends to every cached key and to new keys i' <= i,
 *     including its own (the decode step's K_{<=t} = [K_{<t}; k_t]).
 *
 * Every input bf16 value is taken as its 16-bit pattern and widened exactly to
 * double; all arithmetic is double; the output is double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ORA_PLANT (default 0) compiles one deliberate mistake into a separate test
 * build, so the pin tests can show that each mistake is caught.  The default
 * build has none: every "#if ORA_PLANT == n" below is then dead code. */
#ifndef ORA_PLANT
#define ORA_PLANT 0
#endif

typedef struct {
  int32_t num_pairs;       /* P: pairs (or sequences for decode)            */
  int32_t n_new;           /* l: new tokens per pair                        */
  int32_t num_q_heads;     /* Hq                                            */
  int32_t num_kv_heads;    /* Hkv                                           */
  int32_t head_dim;        /* d                                             */
  int32_t block_len;       /* cached positions per pool block               */
  int32_t blocks_per_pair; /* cached blocks per pair                        */
  int32_t num_blocks;      /* pool extent                                   */
  int32_t num_layers;      /* L, layers held by the pool                    */
  int32_t layer;           /* layer this call reads                         */
  double rope_theta;       /* RoPE base                                     */
  double softmax_scale;    /* 0 -> 1/sqrt(d)                                */
  int32_t prerotated;      /* 1: q and k_new arrive rotated at their positions
                              (by the projection that made them): no RoPE here */
} ora_dims;

enum { ORA_OK = 0, ORA_BAD_ARG = -1, ORA_BAD_BLOCK = -2, ORA_NO_MEM = -3 };

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an IEEE
 * binary32, so shifting it into place gives the same real number. */
double ora_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* FP8 E4M3 (the "fn" variant: no infinities) widened exactly to double:
 * sign s, 4-bit exponent e (bias 7), 3-bit mantissa m.  e = 0 is subnormal,
 * (m / 8) * 2^-6; e = 15 with m = 7 is NaN; otherwise (1 + m / 8) * 2^(e - 7).
 * [Suffix page, §2 and the end of §5]: a KV cache of 1-byte elements. */
double ora_e4m3_to_f64(uint8_t v) {
  const int sgn = v >> 7, e = (v >> 3) & 15, m = v & 7;
  double x;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) x = ldexp((double)m / 8.0, -6);
  else x = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sgn ? -x : x;
}

/* RoPE, rotate-half form: for j < d/2 the pair (x[j], x[j+d/2]) is turned by
 * the angle pos * theta^(-2j/d).  Only position differences survive in the
 * dot product q.k ([Gist page, "在线的一次 attention"], second remark). */
void ora_rope(const double* x, int d, double pos, double theta, double* y) {
  int half = d / 2;
  for (int j = 0; j < half; ++j) {
    double freq = pow(theta, -2.0 * (double)j / (double)d);
    double a = pos * freq;
    double c = cos(a), s = sin(a);
    double x0 = x[j], x1 = x[j + half];
#if ORA_PLANT == 1 /* wrong rotation sign */
    y[j] = x0 * c + x1 * s;
    y[j + half] = x1 * c - x0 * s;
#else
    y[j] = x0 * c - x1 * s;
    y[j + half] = x1 * c + x0 * s;
#endif
  }
}

/* Byte counts of the cache.
 * [Gist page, "先看复用结构" and "收益有多大：存储"]: one position holds
 * 2 x L x H x h numbers (K and V, every layer, every KV head), b bytes each. */
int64_t ora_kv_bytes_per_position(int64_t L, int64_t Hkv, int64_t d, int64_t b) {
  return 2 * L * Hkv * d * b;
}
/* [Gist page, "在线的一次 attention"]: a compressed item keeps 2 x L x k x H x h
 * elements. */
int64_t ora_kv_bytes_per_item(int64_t L, int64_t Hkv, int64_t d, int64_t k, int64_t b) {
  return k * ora_kv_bytes_per_position(L, Hkv, d, b);
}
/* [KV page, "Memory"]: M_KV = 2 B L T h_kv d_h b. */
int64_t ora_kv_bytes_batch(int64_t B, int64_t L, int64_t T, int64_t Hkv, int64_t d, int64_t b) {
  return 2 * B * L * T * Hkv * d * b;
}

/* Element offsets of the layouts shared with the caller. */
static size_t off_q(const ora_dims* D, int p, int i, int h) {
  return (((size_t)p * D->n_new + i) * D->num_q_heads + h) * D->head_dim;
}
static size_t off_kvnew(const ora_dims* D, int p, int i, int g) {
  return (((size_t)p * D->n_new + i) * D->num_kv_heads + g) * D->head_dim;
}
/* pool[num_blocks][L][2][Hkv][block_len][d]; kv = 0 for K, 1 for V */
static size_t off_pool(const ora_dims* D, int blk, int kv, int g, int t) {
  size_t r = (size_t)blk;
#if ORA_PLANT == 7 /* always reads layer 0 */
  r = r * D->num_layers + 0;
#else
  r = r * D->num_layers + D->layer;
#endif
  r = r * 2 + kv;
  r = r * D->num_kv_heads + g;
  r = r * D->block_len + t;
  return r * D->head_dim;
}

typedef struct {
  const ora_dims* D;
  int f64_inputs;        /* 0: q/k_new/v_new/pool are bf16 bit patterns; 1: doubles */
  const void *q, *k_new, *v_new, *pool;
  const float* kv_scale; /* non-NULL: pool holds E4M3 bytes, one scale per
                            (block, layer, K|V, KV head); value = e4m3 * scale */
  const int32_t *item_ids, *block_table, *pos_offset;
  const int32_t* gist_start; /* NULL, or [P]: first prompt-free key of the gist mask */
  int32_t gist_len;          /* k, the gist length of the gist mask              */
  const int32_t* pairs; /* which pairs to compute; NULL = all */
  int32_t n_pairs_out;
  double* out;          /* [n_pairs_out][l][Hq][d]                         */
  double* weights;      /* optional [n_pairs_out][l][Hq][C+l], zeros where masked */
  int32_t first, last;  /* this worker's slice of [0, n_pairs_out)          */
  int status;
} ora_job;

/* Input element idx of array a, widened to double. */
static double elem(const ora_job* J, const void* a, size_t idx) {
  if (J->f64_inputs) return ((const double*)a)[idx];
  return ora_bf16_to_f64(((const uint16_t*)a)[idx]);
}

/* Cached element e of row t of (block, layer, kv, KV head g). */
static double pool_elem(const ora_job* J, int blk, int kv, int g, int t, int e) {
  const ora_dims* D = J->D;
  size_t idx = off_pool(D, blk, kv, g, t) + e;
  if (J->kv_scale) {
    size_t sidx = (((size_t)blk * D->num_layers + D->layer) * 2 + kv) * D->num_kv_heads + g;
    return ora_e4m3_to_f64(((const uint8_t*)J->pool)[idx]) * (double)J->kv_scale[sidx];
  }
  return elem(J, J->pool, idx);
}

static int32_t block_of(const ora_job* J, int p, int b) {
  const ora_dims* D = J->D;
  if (J->block_table) return J->block_table[(size_t)p * D->blocks_per_pair + b];
  return J->item_ids[p];
}

/* One (item, query) pair, all heads, all new tokens. */
static int attend_pair(const ora_job* J, int p, double* out_p, double* w_p) {
  const ora_dims* D = J->D;
  const int l = D->n_new, Hq = D->num_q_heads, Hkv = D->num_kv_heads, d = D->head_dim;
  const int G = Hq / Hkv;
  const int C = D->blocks_per_pair * D->block_len;
  const int nk = C + l;
#if ORA_PLANT == 4 /* scale dropped */
  const double scale = 1.0;
#else
  const double scale = D->softmax_scale > 0.0 ? D->softmax_scale : 1.0 / sqrt((double)d);
#endif
#if ORA_PLANT == 5 /* new tokens numbered from 0, ignoring the cached positions */
  const double pos0 = 0.0;
#else
  const double pos0 = J->pos_offset ? (double)J->pos_offset[p] : (double)C;
#endif

  double* keys = malloc(sizeof(double) * (size_t)nk * d);
  double* vals = malloc(sizeof(double) * (size_t)nk * d);
  double* s = malloc(sizeof(double) * (size_t)nk);
  double* x = malloc(sizeof(double) * (size_t)d);
  double* qr = malloc(sizeof(double) * (size_t)d);
  int rc = ORA_OK;
  if (!keys || !vals || !s || !x || !qr) { rc = ORA_NO_MEM; goto done; }

  for (int g = 0; g < Hkv; ++g) {
    /* Cached rows, in block-table order, exactly as stored (K already rotated). */
    for (int b = 0; b < D->blocks_per_pair; ++b) {
      int32_t blk = block_of(J, p, b);
      if (blk < 0 || blk >= D->num_blocks) { rc = ORA_BAD_BLOCK; goto done; }
      for (int t = 0; t < D->block_len; ++t) {
        int kappa = b * D->block_len + t;
        for (int e = 0; e < d; ++e) {
          keys[(size_t)kappa * d + e] = pool_elem(J, blk, 0, g, t, e);
          vals[(size_t)kappa * d + e] = pool_elem(J, blk, 1, g, t, e);
        }
      }
    }
    /* New rows: K rotated at its own position, V as given. */
    for (int i = 0; i < l; ++i) {
      for (int e = 0; e < d; ++e) x[e] = elem(J, J->k_new, off_kvnew(D, p, i, g) + e);
      if (D->prerotated)
        memcpy(&keys[(size_t)(C + i) * d], x, sizeof(double) * (size_t)d);
      else
        ora_rope(x, d, pos0 + i, D->rope_theta, &keys[(size_t)(C + i) * d]);
      for (int e = 0; e < d; ++e)
        vals[(size_t)(C + i) * d + e] = elem(J, J->v_new, off_kvnew(D, p, i, g) + e);
    }
    for (int h = g * G; h < (g + 1) * G; ++h) {
      for (int i = 0; i < l; ++i) {
#if ORA_PLANT == 3 /* interleaved instead of contiguous head groups */
        int hq = (h % G) * Hkv + g;
#else
        int hq = h;
#endif
        for (int e = 0; e < d; ++e) x[e] = elem(J, J->q, off_q(D, p, i, hq) + e);
        if (D->prerotated)
          memcpy(qr, x, sizeof(double) * (size_t)d);
        else
          ora_rope(x, d, pos0 + i, D->rope_theta, qr);
#if ORA_PLANT == 2 /* not causal inside the new block */
        int n = C + l;
#elif ORA_PLANT == 6 /* a token does not see its own key */
        int n = C + i;
#else
        int n = C + i + 1; /* every cached key, then new keys 0..i */
#endif
        /* [Gist page, "论文做了什么"]: under the gist mask a token after the
         * gist (index C + i >= start + k) no longer sees the prompt before it. */
        int lo = 0;
#if ORA_PLANT != 9 /* gist mask ignored: post-gist tokens still see the prompt */
        if (J->gist_start && C + i >= J->gist_start[p] + J->gist_len) lo = J->gist_start[p];
#endif
        double m = -INFINITY;
        for (int j = lo; j < n; ++j) {
          double acc = 0.0;
          for (int e = 0; e < d; ++e) acc += qr[e] * keys[(size_t)j * d + e];
          s[j] = scale * acc;
          if (s[j] > m) m = s[j];
        }
        double denom = 0.0;
        for (int j = lo; j < n; ++j) { s[j] = exp(s[j] - m); denom += s[j]; }
        double* o = out_p + ((size_t)i * Hq + h) * d;
        for (int e = 0; e < d; ++e) {
          double acc = 0.0;
#if ORA_PLANT == 8 /* keys used as values */
          for (int j = lo; j < n; ++j) acc += s[j] * keys[(size_t)j * d + e];
#else
          for (int j = lo; j < n; ++j) acc += s[j] * vals[(size_t)j * d + e];
#endif
          o[e] = acc / denom;
        }
        if (w_p) {
          double* w = w_p + ((size_t)i * Hq + h) * nk;
          for (int j = 0; j < nk; ++j) w[j] = (j >= lo && j < n) ? s[j] / denom : 0.0;
        }
      }
    }
  }
done:
  free(keys); free(vals); free(s); free(x); free(qr);
  return rc;
}

static void* worker(void* arg) {
  ora_job* J = (ora_job*)arg;
  const ora_dims* D = J->D;
  size_t per_pair_out = (size_t)D->n_new * D->num_q_heads * D->head_dim;
  size_t per_pair_w = (size_t)D->n_new * D->num_q_heads *
                      ((size_t)D->blocks_per_pair * D->block_len + D->n_new);
  for (int32_t r = J->first; r < J->last; ++r) {
    int p = J->pairs ? J->pairs[r] : r;
    int rc = attend_pair(J, p, J->out + (size_t)r * per_pair_out,
                         J->weights ? J->weights + (size_t)r * per_pair_w : NULL);
    if (rc != ORA_OK) { J->status = rc; break; }
  }
  return NULL;
}

static int dims_ok(const ora_dims* D) {
  if (!D) return 0;
  if (D->num_pairs < 0 || D->n_new < 1 || D->head_dim < 2 || (D->head_dim & 1)) return 0;
  if (D->num_q_heads < 1 || D->num_kv_heads < 1 || D->num_q_heads % D->num_kv_heads) return 0;
  if (D->block_len < 0 || D->blocks_per_pair < 0 || D->num_layers < 1) return 0;
  if (D->layer < 0 || D->layer >= D->num_layers) return 0;
  return 1;
}

/*
 * Attention output for the listed pairs (all pairs when `pairs` is NULL).
 * Layouts (row-major, element counts):
 *   q       [P][l][Hq][d]      pre-RoPE
 *   k_new   [P][l][Hkv][d]     pre-RoPE
 *   v_new   [P][l][Hkv][d]
 *   pool    [num_blocks][L][2][Hkv][block_len][d], K rows already rotated
 *   item_ids [P] (one block per pair) or block_table [P][blocks_per_pair]
 *   pos_offset [P] or NULL
 *   out     [n_pairs_out][l][Hq][d]  double
 *   weights [n_pairs_out][l][Hq][C + l] double or NULL
 * Returns 0, or a negative code (bad argument, block id out of range, no memory).
 */
static int run_attn(int f64_inputs, const void* q, const void* k_new, const void* v_new,
                    const void* pool, const float* kv_scale, const int32_t* item_ids,
                    const int32_t* block_table,
                    const int32_t* pos_offset, const int32_t* gist_start, int32_t gist_len,
                    const int32_t* pairs, int32_t n_pairs_out,
                    double* out, double* weights, const ora_dims* D, int32_t num_threads) {
  if (!dims_ok(D) || !out) return ORA_BAD_ARG;
  if (gist_start) {
    if (gist_len < 0) return ORA_BAD_ARG;
    for (int p = 0; p < D->num_pairs; ++p)
      if (gist_start[p] < 0) return ORA_BAD_ARG;
  }
  int C = D->blocks_per_pair * D->block_len;
  if (C > 0 && (!pool || (!item_ids && !block_table))) return ORA_BAD_ARG;
  if (C > 0 && !block_table && D->blocks_per_pair != 1) return ORA_BAD_ARG;
  if (!q || !k_new || !v_new) return ORA_BAD_ARG;
  if (!pairs) n_pairs_out = D->num_pairs;
  if (n_pairs_out <= 0) return ORA_OK;
  if (num_threads < 1) num_threads = 1;
  if (num_threads > n_pairs_out) num_threads = n_pairs_out;

  ora_job* jobs = calloc((size_t)num_threads, sizeof(ora_job));
  pthread_t* th = calloc((size_t)num_threads, sizeof(pthread_t));
  if (!jobs || !th) { free(jobs); free(th); return ORA_NO_MEM; }
  for (int t = 0; t < num_threads; ++t) {
    ora_job* J = &jobs[t];
    J->D = D; J->f64_inputs = f64_inputs; J->kv_scale = kv_scale; J->q = q; J->k_new = k_new; J->v_new = v_new; J->pool = pool;
    J->item_ids = item_ids; J->block_table = block_table; J->pos_offset = pos_offset;
    J->gist_start = gist_start; J->gist_len = gist_len;
    J->pairs = pairs; J->n_pairs_out = n_pairs_out; J->out = out; J->weights = weights;
    J->first = (int32_t)((int64_t)n_pairs_out * t / num_threads);
    J->last = (int32_t)((int64_t)n_pairs_out * (t + 1) / num_threads);
    J->status = ORA_OK;
  }
  char* created = calloc((size_t)num_threads, 1);
  if (!created) { free(jobs); free(th); return ORA_NO_MEM; }
  for (int t = 1; t < num_threads; ++t)
    created[t] = pthread_create(&th[t], NULL, worker, &jobs[t]) == 0;
  worker(&jobs[0]);
  for (int t = 1; t < num_threads; ++t) {
    if (created[t]) pthread_join(th[t], NULL);
    else worker(&jobs[t]); /* no thread available: run that slice here */
  }
  free(created);
  int rc = ORA_OK;
  for (int t = 0; t < num_threads; ++t)
    if (jobs[t].status < 0) rc = jobs[t].status;
  free(jobs); free(th);
  return rc;
}

int ora_gist_attn(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                  const uint16_t* pool, const int32_t* item_ids, const int32_t* block_table,
                  const int32_t* pos_offset, const int32_t* pairs, int32_t n_pairs_out,
                  double* out, double* weights, const ora_dims* D, int32_t num_threads) {
  return run_attn(0, q, k_new, v_new, pool, NULL, item_ids, block_table, pos_offset, NULL, 0,
                  pairs, n_pairs_out, out, weights, D, num_threads);
}

/* The same computation with the cached segment stored as E4M3 bytes and one
 * fp32 scale per (block, layer, K|V, KV head), kv_scale[num_blocks][L][2][Hkv];
 * q, k_new, v_new stay bf16. */
int ora_gist_attn_fp8kv(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                        const uint8_t* pool, const float* kv_scale, const int32_t* item_ids,
                        const int32_t* block_table, const int32_t* pos_offset,
                        const int32_t* pairs, int32_t n_pairs_out, double* out, double* weights,
                        const ora_dims* D, int32_t num_threads) {
  if (!kv_scale && D && D->blocks_per_pair * D->block_len > 0) return ORA_BAD_ARG;
  return run_attn(0, q, k_new, v_new, pool, kv_scale, item_ids, block_table, pos_offset, NULL, 0,
                  pairs, n_pairs_out, out, weights, D, num_threads);
}

/* The same computation on double inputs (same layouts), for multi-layer pins
 * whose later layers see activations that are not bf16 values. */
int ora_gist_attn_f64(const double* q, const double* k_new, const double* v_new,
                      const double* pool, const int32_t* item_ids, const int32_t* block_table,
                      const int32_t* pos_offset, const int32_t* pairs, int32_t n_pairs_out,
                      double* out, double* weights, const ora_dims* D, int32_t num_threads) {
  return run_attn(1, q, k_new, v_new, pool, NULL, item_ids, block_table, pos_offset, NULL, 0,
                  pairs, n_pairs_out, out, weights, D, num_threads);
}

/*
 * The same computation under the gist mask ([Gist page, "论文做了什么"]): the
 * keys of pair p are numbered kappa = 0 .. C + l - 1 over [cached; new]; the
 * prompt is kappa < gist_start[p] and the gist the next gist_len keys; a token
 * whose own index C + i lies after the gist sees only keys kappa >= gist_start[p]
 * (and, as always, kappa <= C + i).  With C = 0 and new tokens
 * [prompt; gist; rest] this is the training forward of one whole sequence;
 * over [prompt; gist] alone it is the plain causal mask (the offline
 * compression pass).  gist_start[p] >= 0, gist_len >= 0.
 */
int ora_gist_attn_masked(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                         const uint16_t* pool, const int32_t* item_ids,
                         const int32_t* block_table, const int32_t* pos_offset,
                         const int32_t* gist_start, int32_t gist_len, const int32_t* pairs,
                         int32_t n_pairs_out, double* out, double* weights, const ora_dims* D,
                         int32_t num_threads) {
  if (!gist_start) return ORA_BAD_ARG;
  return run_attn(0, q, k_new, v_new, pool, NULL, item_ids, block_table, pos_offset, gist_start,
                  gist_len, pairs, n_pairs_out, out, weights, D, num_threads);
}

/*
 * The cached segment each pair reads, copied bit for bit:
 *   dst[p][g][kv][kappa][e] = pool[block(p, kappa / block_len)][layer][kv][g][kappa % block_len][e]
 * for kappa < blocks_per_pair * block_len.  A pair with an out-of-range block
 * id gets all-zero rows and the call returns ORA_BAD_BLOCK.
 */
int ora_gather(const uint16_t* pool, const int32_t* item_ids, const int32_t* block_table,
               uint16_t* dst, const ora_dims* D) {
  if (!dims_ok(D) || !pool || !dst || (!item_ids && !block_table)) return ORA_BAD_ARG;
  ora_job J;
  memset(&J, 0, sizeof J);
  J.D = D; J.item_ids = item_ids; J.block_table = block_table;
  const int C = D->blocks_per_pair * D->block_len, d = D->head_dim;
  int rc = ORA_OK;
  for (int p = 0; p < D->num_pairs; ++p) {
    int bad = 0;
    for (int b = 0; b < D->blocks_per_pair; ++b) {
      int32_t blk = block_of(&J, p, b);
      if (blk < 0 || blk >= D->num_blocks) bad = 1;
    }
    for (int g = 0; g < D->num_kv_heads; ++g)
      for (int kv = 0; kv < 2; ++kv)
        for (int kappa = 0; kappa < C; ++kappa) {
          uint16_t* row = dst + ((((size_t)p * D->num_kv_heads + g) * 2 + kv) * C + kappa) * d;
          if (bad) { memset(row, 0, sizeof(uint16_t) * d); continue; }
          int32_t blk = block_of(&J, p, kappa / D->block_len);
          memcpy(row, pool + off_pool(D, blk, kv, g, kappa % D->block_len), sizeof(uint16_t) * d);
        }
    if (bad) rc = ORA_BAD_BLOCK;
  }
  return rc;
}

/*
 * The decode step's append ([KV page, "Reusable-state"]: K_{<=t} = [K_{<t}; k_t],
 * the new K/V are appended to every layer's cache): for each sequence p and KV
 * head g, row slot[p] of the sequence's cache -- block block_table[p][slot /
 * block_len], row slot % block_len, at `layer` -- receives k_new rotated at
 * position pos_offset[p] (NULL: slot[p]) and rounded to bf16 (nearest even),
 * and v_new unchanged.  The pool is bf16 bits [num_blocks][L][2][Hkv][block_len][d].
 * Returns ORA_BAD_BLOCK (writing nothing for that sequence) on an out-of-range
 * block id or slot.
 */
static uint16_t f64_to_bf16_rne(double v) {
  float f = (float)v; /* exact enough: the bf16 rounding below decides */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)(u >> 16); /* inf / nan */
  /* round the double directly: the nearest bf16 to v, ties to even */
  double a = fabs(v);
  if (a == 0.0) return (uint16_t)(signbit(v) ? 0x8000u : 0u);
  int e;
  frexp(a, &e);                    /* a = m * 2^e, m in [0.5, 1) */
  int q = e - 8;                   /* bf16 keeps 8 significant bits */
  if (q < -133) q = -133;          /* subnormal spacing 2^-133 */
  double ulp = ldexp(1.0, q);
  double n = a / ulp, fl = floor(n), r = n - fl;
  if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
  float rf = (float)(fl * ulp);
  memcpy(&u, &rf, sizeof u);
  u >>= 16;
  return (uint16_t)(signbit(v) ? (u | 0x8000u) : u);
}

int ora_kv_append(const uint16_t* k_new, const uint16_t* v_new, uint16_t* pool,
                  const int32_t* block_table, const int32_t* slot, const int32_t* pos_offset,
                  const ora_dims* D) {
  if (!dims_ok(D) || !k_new || !v_new || !pool || !block_table || !slot) return ORA_BAD_ARG;
  const int d = D->head_dim, Hkv = D->num_kv_heads;
  double* x = malloc(sizeof(double) * (size_t)d);
  double* y = malloc(sizeof(double) * (size_t)d);
  if (!x || !y) { free(x); free(y); return ORA_NO_MEM; }
  int rc = ORA_OK;
  for (int p = 0; p < D->num_pairs; ++p) {
    int s = slot[p];
    if (s < 0 || s >= D->blocks_per_pair * D->block_len) { rc = ORA_BAD_BLOCK; continue; }
    int32_t blk = block_table[(size_t)p * D->blocks_per_pair + s / D->block_len];
    if (blk < 0 || blk >= D->num_blocks) { rc = ORA_BAD_BLOCK; continue; }
    double pos = pos_offset ? (double)pos_offset[p] : (double)s;
    for (int g = 0; g < Hkv; ++g) {
      size_t src = ((size_t)p * Hkv + g) * d; /* one new token: [P][1][Hkv][d] */
      for (int e = 0; e < d; ++e) x[e] = ora_bf16_to_f64(k_new[src + e]);
      ora_rope(x, d, pos, D->rope_theta, y);
      uint16_t* krow = pool + off_pool(D, blk, 0, g, s % D->block_len);
      uint16_t* vrow = pool + off_pool(D, blk, 1, g, s % D->block_len);
      for (int e = 0; e < d; ++e) {
        krow[e] = f64_to_bf16_rne(y[e]);
        vrow[e] = v_new[src + e];
      }
    }
  }
  free(x); free(y);
  return rc;
}

/*
 * Stores a compressed item ([Gist page, "论文做了什么" and "在线的一次 attention"]:
 * after the offline pass over [prompt; gist] each layer keeps the K/V at the
 * k gist positions as the item's cache entry).  For pair p (one sequence of
 * n_new tokens) and KV head g, rows first_row[p] + t, t < block_len (= k), of
 * k_new / v_new go to block item_ids[p] at `layer`:
 *   pool[blk][layer][0][g][t] = bf16_rne(R(k_new[p][first_row[p] + t][g]) at
 *                               position (store_pos ? store_pos[p] : 0) + t)
 *   pool[blk][layer][1][g][t] = v_new[p][first_row[p] + t][g]
 * A pair whose rows fall outside [0, n_new) or whose block id is out of range
 * writes nothing and the call returns ORA_BAD_BLOCK.
 */
int ora_kv_store(const uint16_t* k_new, const uint16_t* v_new, uint16_t* pool,
                 const int32_t* item_ids, const int32_t* first_row, const int32_t* store_pos,
                 const ora_dims* D) {
  if (!dims_ok(D) || !k_new || !v_new || !pool || !item_ids || !first_row) return ORA_BAD_ARG;
  const int d = D->head_dim, Hkv = D->num_kv_heads, k = D->block_len, l = D->n_new;
  double* x = malloc(sizeof(double) * (size_t)d);
  double* y = malloc(sizeof(double) * (size_t)d);
  if (!x || !y) { free(x); free(y); return ORA_NO_MEM; }
  int rc = ORA_OK;
  for (int p = 0; p < D->num_pairs; ++p) {
    int r0 = first_row[p];
    int32_t blk = item_ids[p];
    if (r0 < 0 || r0 > l - k || blk < 0 || blk >= D->num_blocks) { rc = ORA_BAD_BLOCK; continue; }
    double pos0 = store_pos ? (double)store_pos[p] : 0.0;
    for (int g = 0; g < Hkv; ++g) {
      for (int t = 0; t < k; ++t) {
        size_t src = (((size_t)p * l + r0 + t) * Hkv + g) * d;
        for (int e = 0; e < d; ++e) x[e] = ora_bf16_to_f64(k_new[src + e]);
        ora_rope(x, d, pos0 + t, D->rope_theta, y);
        uint16_t* krow = pool + off_pool(D, blk, 0, g, t);
        uint16_t* vrow = pool + off_pool(D, blk, 1, g, t);
        for (int e = 0; e < d; ++e) {
          krow[e] = f64_to_bf16_rne(y[e]);
          vrow[e] = v_new[src + e];
        }
      }
    }
  }
  free(x); free(y);
  return rc;
}
