/*
 * pa_oracle.c -- plain fp64 CPU oracle for paged multi-token attention.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test suite, the smoke check and the
 * benchmark's CPU-baseline leg, never by the library's product path. It shares
 * nothing with the CUDA sources. Every step below is the plain definition from
 * the pages, written out with no tiling, fusion or online softmax:
 *
 *   "PagedAttention" wiki page, "Mathematical formulation":
 *       a_ij = exp(q_i.k_j / sqrt(d)) / sum_{t<=i} exp(q_i.k_t / sqrt(d))
 *       o_i  = sum_{j<=i} a_ij v_j
 *     (the page's text lost the square root; scale = 1/sqrt(D) is the reading).
 *     The block form over K_j = (k_{(j-1)B+1} .. k_{jB}) is oracle_attention_blockwise.
 *   vLLM post (devpress), "1. overall architecture", worked example: a token at
 *     position p of a sequence lives in slot block_table[p / B] * B + p % B.
 *   same post, "2.1 parallel sampling": copy-on-write copies a whole block.
 *   Pensieve summary, "unified prefill and generation" and the multi-token
 *     kernel description: the query rows are the last query_len tokens of the
 *     context and each attends causally to every earlier token.
 *
 * A masked key gets probability zero (Pensieve's "set to 0" of the upper
 * triangle is read as zero weight, not a zero score).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -pthread pa_oracle.c -lm
 * ORACLE_MUTATION (default 0) plants one known mistake; only the test that
 * checks that the pins catch planted mistakes builds a non-zero value.
 */
#include "pa_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

static _Thread_local char g_err[256];

static int fail(const char* msg) {
  snprintf(g_err, sizeof g_err, "%s", msg);
  return -1;
}

const char* oracle_last_error(void) { return g_err; }

double oracle_bf16_to_double(uint16_t bits) {
  /* A bf16 value is the top half of an IEEE binary32 value. */
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------------------- slots */

int oracle_slot_mapping(const int32_t* block_table, int32_t num_seqs, int32_t max_blocks,
                        int32_t block_size, int32_t num_blocks, const int32_t* seq_ids,
                        const int32_t* positions, int64_t n, int64_t* slots_out) {
  if (block_size <= 0 || max_blocks <= 0 || num_blocks <= 0) return fail("bad sizes");
  for (int64_t t = 0; t < n; ++t) {
    int32_t s = seq_ids[t];
    int32_t p = positions[t];
    if (s < 0 || s >= num_seqs) return fail("seq id out of range");
    if (p < 0) { slots_out[t] = -1; continue; }
    int32_t logical = p / block_size;
    if (logical >= max_blocks) return fail("position beyond the block table");
    int32_t phys = block_table[(int64_t)s * max_blocks + logical];
    if (phys < 0 || phys >= num_blocks) return fail("block id out of range");
#if ORACLE_MUTATION == 5
    slots_out[t] = (int64_t)logical * block_size + p % block_size; /* planted: ignores the table */
#else
    slots_out[t] = (int64_t)phys * block_size + p % block_size;
#endif
  }
  return 0;
}

/* ---------------------------------------------------------------- write */

int oracle_write_kv(const uint16_t* k_new, const uint16_t* v_new, const int64_t* slot_mapping,
                    int64_t n_new, uint16_t* k_pool, uint16_t* v_pool, int32_t num_blocks,
                    int32_t block_size, int32_t Hkv, int32_t D) {
  if (num_blocks <= 0 || block_size <= 0 || Hkv <= 0 || D <= 0) return fail("bad sizes");
  int64_t n_slots = (int64_t)num_blocks * block_size;
  int64_t row = (int64_t)Hkv * D; /* values of one token in one pool */
  unsigned char* seen = (unsigned char*)calloc((size_t)n_slots, 1);
  if (!seen) return fail("out of memory");
  for (int64_t t = 0; t < n_new; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= n_slots) { free(seen); return fail("slot out of range"); }
    if (seen[slot]) { free(seen); return fail("duplicate slot"); }
    seen[slot] = 1;
  }
  free(seen);
  for (int64_t t = 0; t < n_new; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    memcpy(k_pool + slot * row, k_new + t * row, (size_t)row * sizeof(uint16_t));
#if ORACLE_MUTATION == 8
    memcpy(v_pool + slot * row, k_new + t * row, (size_t)row * sizeof(uint16_t)); /* planted */
#else
    memcpy(v_pool + slot * row, v_new + t * row, (size_t)row * sizeof(uint16_t));
#endif
  }
  return 0;
}

/* ---------------------------------------------------------------- copy */

int oracle_copy_blocks(uint16_t* k_pool, uint16_t* v_pool, const int32_t* src, const int32_t* dst,
                       int32_t n_pairs, int32_t num_blocks, int32_t block_size, int32_t Hkv,
                       int32_t D) {
  if (num_blocks <= 0 || block_size <= 0 || Hkv <= 0 || D <= 0 || n_pairs < 0)
    return fail("bad sizes");
  for (int32_t i = 0; i < n_pairs; ++i) {
    if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks)
      return fail("block id out of range");
    for (int32_t j = 0; j < n_pairs; ++j) {
      if (j != i && dst[j] == dst[i]) return fail("duplicate destination block");
      if (src[j] == dst[i]) return fail("destination block is also a source");
    }
  }
  int64_t blk = (int64_t)block_size * Hkv * D;
  for (int32_t i = 0; i < n_pairs; ++i) {
    memcpy(k_pool + (int64_t)dst[i] * blk, k_pool + (int64_t)src[i] * blk,
           (size_t)blk * sizeof(uint16_t));
#if ORACLE_MUTATION != 6
    memcpy(v_pool + (int64_t)dst[i] * blk, v_pool + (int64_t)src[i] * blk,
           (size_t)blk * sizeof(uint16_t));
#endif
  }
  return 0;
}

/* ---------------------------------------------------------------- attention */

typedef struct {
  const uint16_t* q;
  int32_t Hq, D, Hkv, block_size, max_blocks;
  const uint16_t *k_pool, *v_pool;
  const int32_t* block_table;
  const int32_t *context_lens, *query_lens;
  const int64_t* row_seq;    /* sequence of each row of q */
  const int64_t* row_first;  /* first row of that sequence */
  const int64_t* rows;       /* rows to compute (NULL = all) */
  int64_t n_rows;
  double scale;
  double* out;
  int32_t n_threads, thread_id;
  int32_t max_ctx;
  int status;
} att_job;

/* One output vector O[r, h, :] from the definition. */
static void attend_one(const att_job* j, int64_t r, int32_t h, double* x, double* o) {
  const int32_t D = j->D, B = j->block_size;
  int64_t s = j->row_seq[r];
  int32_t L = j->context_lens[s], ql = j->query_lens[s];
  int32_t i = (int32_t)(r - j->row_first[s]);
  int32_t g = j->Hq / j->Hkv;
#if ORACLE_MUTATION == 2
  int32_t p = i; /* planted: top-left aligned mask */
  (void)L; (void)ql;
#else
  int32_t p = L - ql + i; /* absolute position of this query token */
#endif
#if ORACLE_MUTATION == 3
  int32_t kvh = h % j->Hkv; /* planted: interleaved head map */
#else
  int32_t kvh = h / g;
#endif
  const uint16_t* qv = j->q + (r * j->Hq + h) * (int64_t)D;
  const int32_t* bt = j->block_table + s * (int64_t)j->max_blocks;
#if ORACLE_MUTATION == 4
  int32_t last = p - 1; /* planted: excludes the query's own key */
#elif ORACLE_MUTATION == 7
  int32_t last = L - 1; /* planted: no causal mask */
#else
  int32_t last = p; /* keys 0..p are visible */
#endif
  double m = -INFINITY;
  for (int32_t t = 0; t <= last; ++t) {
    int64_t slot = (int64_t)bt[t / B] * B + t % B;
    const uint16_t* kv = j->k_pool + (slot * j->Hkv + kvh) * (int64_t)D;
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d)
      dot += oracle_bf16_to_double(qv[d]) * oracle_bf16_to_double(kv[d]);
    x[t] = dot * j->scale;
    if (x[t] > m) m = x[t];
  }
  double denom = 0.0;
  for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
  for (int32_t t = 0; t <= last; ++t) {
    double w = exp(x[t] - m);
    denom += w;
    int64_t slot = (int64_t)bt[t / B] * B + t % B;
    const uint16_t* vv = j->v_pool + (slot * j->Hkv + kvh) * (int64_t)D;
    for (int32_t d = 0; d < D; ++d) o[d] += w * oracle_bf16_to_double(vv[d]);
  }
  for (int32_t d = 0; d < D; ++d) o[d] = (last >= 0) ? o[d] / denom : 0.0;
}

static void* att_worker(void* arg) {
  att_job* j = (att_job*)arg;
  double* x = (double*)malloc(sizeof(double) * (size_t)(j->max_ctx > 0 ? j->max_ctx : 1));
  if (!x) { j->status = -1; return NULL; }
  int64_t n_tasks = j->n_rows * j->Hq;
  for (int64_t task = j->thread_id; task < n_tasks; task += j->n_threads) {
    int64_t k = task / j->Hq;
    int32_t h = (int32_t)(task % j->Hq);
    int64_t r = j->rows ? j->rows[k] : k;
    attend_one(j, r, h, x, j->out + (k * j->Hq + h) * (int64_t)j->D);
  }
  free(x);
  return NULL;
}

/* Shared argument checks and row -> sequence tables. */
static int check_and_index(int64_t total_q, int32_t Hq, int32_t D, int32_t num_blocks,
                           int32_t block_size, int32_t Hkv, const int32_t* block_table,
                           int32_t max_blocks, const int32_t* context_lens,
                           const int32_t* query_lens, int32_t num_seqs, int64_t** row_seq,
                           int64_t** row_first, int32_t* max_ctx) {
  if (Hq <= 0 || Hkv <= 0 || D <= 0 || block_size <= 0 || num_blocks <= 0 || num_seqs < 0 ||
      max_blocks <= 0)
    return fail("bad sizes");
  if (Hq % Hkv) return fail("Hq must be a multiple of Hkv");
  int64_t sum_q = 0;
  *max_ctx = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t L = context_lens[s], ql = query_lens[s];
    if (L < 0 || ql < 0 || ql > L) return fail("need 0 <= query_len <= context_len");
    if ((int64_t)(L + block_size - 1) / block_size > max_blocks)
      return fail("context longer than the block table");
    for (int32_t b = 0; b < (L + block_size - 1) / block_size; ++b) {
      int32_t phys = block_table[(int64_t)s * max_blocks + b];
      if (phys < 0 || phys >= num_blocks) return fail("block id out of range");
    }
    sum_q += ql;
    if (L > *max_ctx) *max_ctx = L;
  }
  if (sum_q != total_q) return fail("total_q != sum(query_lens)");
  *row_seq = (int64_t*)malloc(sizeof(int64_t) * (size_t)(total_q > 0 ? total_q : 1));
  *row_first = (int64_t*)malloc(sizeof(int64_t) * (size_t)(num_seqs > 0 ? num_seqs : 1));
  if (!*row_seq || !*row_first) return fail("out of memory");
  int64_t r = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    (*row_first)[s] = r;
    for (int32_t i = 0; i < query_lens[s]; ++i) (*row_seq)[r++] = s;
  }
  return 0;
}

int oracle_attention(const uint16_t* q, int64_t total_q, int32_t Hq, int32_t D,
                     const uint16_t* k_pool, const uint16_t* v_pool, int32_t num_blocks,
                     int32_t block_size, int32_t Hkv, const int32_t* block_table,
                     int32_t max_blocks, const int32_t* context_lens,
                     const int32_t* query_lens, int32_t num_seqs, double scale,
                     const int64_t* rows, int64_t n_rows, int32_t n_threads, double* out) {
  int64_t *row_seq = NULL, *row_first = NULL;
  int32_t max_ctx = 0;
  int rc = check_and_index(total_q, Hq, D, num_blocks, block_size, Hkv, block_table, max_blocks,
                           context_lens, query_lens, num_seqs, &row_seq, &row_first, &max_ctx);
  if (rc) { free(row_seq); free(row_first); return rc; }
  if (rows) {
    for (int64_t k = 0; k < n_rows; ++k)
      if (rows[k] < 0 || rows[k] >= total_q) {
        free(row_seq); free(row_first);
        return fail("row index out of range");
      }
  } else {
    n_rows = total_q;
  }
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
#if ORACLE_MUTATION == 1
  scale = 1.0 / (double)D; /* planted: the square root dropped */
#endif
  if (n_threads <= 0) n_threads = 1;
  att_job* jobs = (att_job*)calloc((size_t)n_threads, sizeof(att_job));
  pthread_t* th = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  if (!jobs || !th) { free(jobs); free(th); free(row_seq); free(row_first); return fail("oom"); }
  for (int32_t t = 0; t < n_threads; ++t) {
    att_job* j = &jobs[t];
    j->q = q; j->Hq = Hq; j->D = D; j->Hkv = Hkv; j->block_size = block_size;
    j->max_blocks = max_blocks; j->k_pool = k_pool; j->v_pool = v_pool;
    j->block_table = block_table; j->context_lens = context_lens; j->query_lens = query_lens;
    j->row_seq = row_seq; j->row_first = row_first; j->rows = rows; j->n_rows = n_rows;
    j->scale = scale; j->out = out; j->n_threads = n_threads; j->thread_id = t;
    j->max_ctx = max_ctx; j->status = 0;
  }
  if (n_threads == 1) {
    att_worker(&jobs[0]);
  } else {
    for (int32_t t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, att_worker, &jobs[t]);
    for (int32_t t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
  }
  rc = 0;
  for (int32_t t = 0; t < n_threads; ++t)
    if (jobs[t].status) rc = fail("out of memory in a worker");
  free(jobs); free(th); free(row_seq); free(row_first);
  return rc;
}

/* ---------------------------------------------------------------- block form */

int oracle_attention_blockwise(const uint16_t* q, int64_t total_q, int32_t Hq, int32_t D,
                               const uint16_t* k_pool, const uint16_t* v_pool,
                               int32_t num_blocks, int32_t block_size, int32_t Hkv,
                               const int32_t* block_table, int32_t max_blocks,
                               const int32_t* context_lens, const int32_t* query_lens,
                               int32_t num_seqs, double scale, double* out) {
  int64_t *row_seq = NULL, *row_first = NULL;
  int32_t max_ctx = 0;
  int rc = check_and_index(total_q, Hq, D, num_blocks, block_size, Hkv, block_table, max_blocks,
                           context_lens, query_lens, num_seqs, &row_seq, &row_first, &max_ctx);
  if (rc) { free(row_seq); free(row_first); return rc; }
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
  const int32_t B = block_size, g = Hq / Hkv;
  int32_t nb_max = (max_ctx + B - 1) / B;
  /* score vector of every block, A[j][0..B-1]; masked entries carry no weight */
  double* A = (double*)malloc(sizeof(double) * (size_t)(nb_max > 0 ? nb_max : 1) * B);
  if (!A) { free(row_seq); free(row_first); return fail("out of memory"); }
  for (int64_t r = 0; r < total_q; ++r) {
    int64_t s = row_seq[r];
    int32_t p = context_lens[s] - query_lens[s] + (int32_t)(r - row_first[s]);
    int32_t nblk = p / B + 1; /* ceil((p + 1) / B): blocks that hold keys 0..p */
    const int32_t* bt = block_table + s * (int64_t)max_blocks;
    for (int32_t h = 0; h < Hq; ++h) {
      const uint16_t* qv = q + (r * Hq + h) * (int64_t)D;
      int32_t kvh = h / g;
      double m = -INFINITY;
      /* K_j q_i for every block j: one vector of B scores per block */
      for (int32_t jb = 0; jb < nblk; ++jb) {
        const uint16_t* Kj = k_pool + ((int64_t)bt[jb] * B * Hkv) * D;
        for (int32_t u = 0; u < B; ++u) {
          int32_t t = jb * B + u;
          if (t > p) { A[jb * B + u] = -INFINITY; continue; }
          const uint16_t* kv = Kj + ((int64_t)u * Hkv + kvh) * D;
          double dot = 0.0;
          for (int32_t d = 0; d < D; ++d)
            dot += oracle_bf16_to_double(qv[d]) * oracle_bf16_to_double(kv[d]);
          A[jb * B + u] = dot * scale;
          if (A[jb * B + u] > m) m = A[jb * B + u];
        }
      }
      /* normalise over the concatenation of the block score vectors */
      double denom = 0.0;
      for (int32_t e = 0; e < nblk * B; ++e) {
        A[e] = (A[e] == -INFINITY) ? 0.0 : exp(A[e] - m);
        denom += A[e];
      }
      /* o_i = sum_j V_j^T A_ij */
      double* o = out + (r * Hq + h) * (int64_t)D;
      for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
      for (int32_t jb = 0; jb < nblk; ++jb) {
        const uint16_t* Vj = v_pool + ((int64_t)bt[jb] * B * Hkv) * D;
        for (int32_t u = 0; u < B; ++u) {
          double a = A[jb * B + u] / denom;
          if (a == 0.0) continue;
          const uint16_t* vv = Vj + ((int64_t)u * Hkv + kvh) * D;
          for (int32_t d = 0; d < D; ++d) o[d] += a * oracle_bf16_to_double(vv[d]);
        }
      }
    }
  }
  free(A); free(row_seq); free(row_first);
  return 0;
}
