/*
 * HSTU fused attention forward: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker, not the product: only the
 * tests, the smoke check and the benchmark's CPU-baseline leg load it. It shares
 * no code, header or constant with the CUDA library.
 *
 * Source: "RecOps Running Case Documentation" (gitcode.com/Ascend/RecSDK,
 * docs/en/rec_ops/hstu_v1_forward.md).
 *   - Introduction to the HSTU_V1 Forward Operator: the operator chains, in this
 *     order, the QK matrix multiplication, the SiLU activation, the scaling, the
 *     mask application and the multiplication with V.
 *   - Feature table, "Attention mechanism": S = Q*K^T, P = silu(S), O = P*V.
 *   - Feature table, "GQA": several query heads share one key/value head.
 *   - Feature table, "Relative attention bias": optional rab [b, n, s, s].
 *   - Feature table, "Support causal mask": built from num_context, num_targets
 *     and target_group_size, any of which may be absent.
 *   - Inputs and Outputs table: jagged [s_b, N, D] layout with seq_offsets [B+1];
 *     mask_type 0 = built-in lower-triangular (causal) mask, 2 = no mask, 3 = custom
 *     mask passed in as mask [B, N, S, S] of q's type;
 *     silu_scale defaults to 1/max_seq_len; target_group_size 0 = no target
 *     mask; alpha = "alpha scaling parameter".
 *
 * Readings taken where the page is silent (each also listed in the design notes):
 *   - alpha multiplies Q*K^T only; rab is added after it, before SiLU.
 *   - rab is indexed by local positions: rab[b, h, i, j], row stride max_seqlen.
 *   - Feature table, "Support for rab broadcasting": rab may be [b, 1, s, s]; its one
 *     plane per sequence is then added for every query head.
 *   - GQA head map: kv head = h / (Nq / Nk) (contiguous groups).
 *   - Causal mask with H = (g > 0) ? max(L - nt, 0) : L (history length):
 *       valid(i, j) = (j <= i && j < H)                       causal over history
 *                  || (i < nc && j < H)                       context rows see all history
 *                  || (g > 0 && i >= H && j >= H && j <= i
 *                      && (i - H) / g == (j - H) / g)         targets: own group, causal
 *                  || (g == 0 && j <= i)                      no target mask: plain causal
 *   - A masked entry of P is exactly 0 (select, not multiply).
 *   - Custom mask (mask_type 3): every key of the sequence is a candidate and P is
 *     multiplied by mask[b, h, i, j] after the SiLU and the scaling (the chain's order);
 *     a 0/1 mask selects exactly like the built-in one.
 *   - Different query and key lengths (Inputs and Outputs table: seq_offsets_q,
 *     seq_offsets_k, max_seq_len_q, max_seq_len_k, is_delta_qk): sequence b has Lq query
 *     rows and Lk >= Lq keys, and the queries are the last Lq tokens of the sequence:
 *     query row i sits at position p = Lk - Lq + i. The mask, the rab row and the custom
 *     mask row are taken at p (with L = Lk); rab and mask are [B, N, Sk, Sk],
 *     Sk = max_seq_len_k. So a call with fewer queries computes exactly the last Lq rows
 *     of the call with all Lk queries.
 *   - KV cache (Inputs and Outputs table: kv_cache [num_pages, 2, page_size, N, D],
 *     page_offsets [B+1], page_ids, last_page_len [B]; feature table "Page"): the cache
 *     holds the history of each sequence. Its keys are the rows of pages
 *     page_ids[page_offsets[b]], ..., page_ids[page_offsets[b+1] - 1] in that order
 *     (plane 0 of a page holds K, plane 1 holds V), every page full except the last, which
 *     holds last_page_len[b] rows; the new k/v rows of the call follow the history. So
 *     Lk = (pages - 1) * page_size + last_page_len[b] + (new k rows), or just the new rows
 *     when the sequence has no pages.
 *
 * Pinned by tests/test_oracle_pins.py: closed forms (L = 1, silu(ln 3) = 0.75 ln 3,
 * silu(x) - silu(-x) = x), the dense equal-length case against torch.matmul and
 * torch.nn.functional.silu in fp64, hand-written 0/1 mask matrices, and the
 * invariants (Q = 0 gives 0, causal locality, GQA = replicated MHA, batch
 * permutation, V = ones); the key side by the identities "fewer queries = the last rows
 * of the call with all queries" and "paged keys = the same keys passed contiguously"
 * (bit for bit), and a Q = 0 closed form through a cache. The alpha/rab positions, the
 * mask semantics and the query alignment are readings of a silent page: parity of those
 * readings is unpinned by the page.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MASK_CAUSAL 0 /* "0: built-in lower triangular mask" */
#define ORACLE_MASK_NONE 2   /* "2: do not use a mask" */
#define ORACLE_MASK_CUSTOM 3 /* "3: use a custom mask ... the user must pass in the mask" */

/* The mask predicate (reading above). Returns 1 when query row i may attend key j. */
int hstu_oracle_valid(int64_t i, int64_t j, int64_t L, int mask_type, int64_t nc,
                      int64_t nt, int64_t g) {
  if (i < 0 || j < 0 || i >= L || j >= L) return 0;
  /* no mask, or a custom mask: every key of the sequence is a candidate (a custom mask
     acts through its values, step 4 of the forward) */
  if (mask_type == ORACLE_MASK_NONE || mask_type == ORACLE_MASK_CUSTOM) return 1;
  int64_t H = L;
  if (g > 0) {
    H = L - nt;
    if (H < 0) H = 0;
  }
  if (j <= i && j < H) return 1;
  if (i < nc && j < H) return 1;
  if (g > 0 && i >= H && j >= H && j <= i && (i - H) / g == (j - H) / g) return 1;
  if (g == 0 && j <= i) return 1;
  return 0;
}

/* silu(x) = x * sigmoid(x) = x / (1 + exp(-x)). */
static double silu(double x) { return x / (1.0 + exp(-x)); }

typedef struct {
  const double *q, *k, *v, *rab;
  const double *mask; /* custom mask [B, Nq, Sk, Sk] (mask_type 3) */
  const int64_t *seq_offsets, *num_context, *num_targets;
  const int64_t *seq_offsets_k; /* offsets of the k/v rows, or NULL: those of q */
  const double *kv_cache;       /* [num_pages, 2, page_size, Nk, D] or NULL */
  const int64_t *page_offsets, *page_ids, *last_page_len;
  int64_t page_size;
  int64_t B, Nq, Nk, D, max_seqlen; /* max_seqlen: Sk, the row length of rab and mask */
  int64_t rab_heads; /* rab planes per sequence: Nq, or 1 (broadcast to every head) */
  int mask_type;
  int64_t g;
  double alpha, silu_scale;
  double *out;
  /* row mode: rows[3*r + {0,1,2}] = (b, h, i); out_rows is [nrows, D] */
  const int64_t *rows;
  int64_t nrows;
  double *out_rows;
  int64_t next; /* work counter, taken with an atomic add */
} job_t;

/* Cached history length of sequence b (0 without a cache). */
static int64_t history_len(const job_t *J, int64_t b) {
  if (!J->kv_cache) return 0;
  const int64_t pages = J->page_offsets[b + 1] - J->page_offsets[b];
  return pages > 0 ? (pages - 1) * J->page_size + J->last_page_len[b] : 0;
}

/* Number of new k/v rows of sequence b. */
static int64_t new_kv_len(const job_t *J, int64_t b) {
  const int64_t *so = J->seq_offsets_k ? J->seq_offsets_k : J->seq_offsets;
  return so[b + 1] - so[b];
}

/* Key (plane 0) or value (plane 1) row of key position j of sequence b, head hk. */
static const double *kv_row(const job_t *J, int64_t b, int64_t hk, int64_t j, int plane) {
  const int64_t hist = history_len(J, b);
  if (j < hist) {
    const int64_t page = J->page_ids[J->page_offsets[b] + j / J->page_size];
    const int64_t row = j % J->page_size;
    return J->kv_cache + (((page * 2 + plane) * J->page_size + row) * J->Nk + hk) * J->D;
  }
  const int64_t *so = J->seq_offsets_k ? J->seq_offsets_k : J->seq_offsets;
  return (plane ? J->v : J->k) + ((so[b] + (j - hist)) * J->Nk + hk) * J->D;
}

/* One output row: out[t0 + i, h, :] for sequence b, query head h, local query row i. */
static void one_row(const job_t *J, int64_t b, int64_t h, int64_t i, double *o) {
  const int64_t t0 = J->seq_offsets[b];
  const int64_t Lq = J->seq_offsets[b + 1] - t0;
  const int64_t L = history_len(J, b) + new_kv_len(J, b); /* keys of the sequence */
  const int64_t pos = L - Lq + i; /* position of the query in the sequence */
  const int64_t D = J->D;
  const int64_t G = J->Nq / J->Nk;
  const int64_t hk = h / G;
  const int64_t nc = J->num_context ? J->num_context[b] : 0;
  const int64_t nt = J->num_targets ? J->num_targets[b] : 0;
  const double *qi = J->q + ((t0 + i) * J->Nq + h) * D;
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < L; ++j) {
    const double *kj = kv_row(J, b, hk, j, 0);
    const double *vj = kv_row(J, b, hk, j, 1);
    /* 1. QK matrix multiplication */
    double s = 0.0;
    for (int64_t d = 0; d < D; ++d) s += qi[d] * kj[d];
    /* alpha on Q*K^T, then the relative attention bias */
    double x = J->alpha * s;
    if (J->rab) {
      const int64_t plane = b * J->rab_heads + (J->rab_heads == 1 ? 0 : h);
      x += J->rab[(plane * J->max_seqlen + pos) * J->max_seqlen + j];
    }
    /* 2. SiLU activation */
    double p = silu(x);
    /* 3. scaling */
    p *= J->silu_scale;
    /* 4. mask application: the built-in mask selects; a custom mask multiplies P by
       mask[b, h, i, j] (a 0/1 mask selects the same way) */
    if (!hstu_oracle_valid(pos, j, L, J->mask_type, nc, nt, J->g)) p = 0.0;
    if (J->mask_type == ORACLE_MASK_CUSTOM)
      p *= J->mask[((b * J->Nq + h) * J->max_seqlen + pos) * J->max_seqlen + j];
    /* 5. matrix multiplication with V */
    for (int64_t d = 0; d < D; ++d) o[d] += p * vj[d];
  }
}

static void *worker_units(void *arg) {
  job_t *J = (job_t *)arg;
  const int64_t units = J->B * J->Nq;
  for (;;) {
    int64_t u = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
    if (u >= units) break;
    const int64_t b = u / J->Nq, h = u % J->Nq;
    const int64_t t0 = J->seq_offsets[b];
    const int64_t Lq = J->seq_offsets[b + 1] - t0;
    for (int64_t i = 0; i < Lq; ++i) one_row(J, b, h, i, J->out + ((t0 + i) * J->Nq + h) * J->D);
  }
  return NULL;
}

static void *worker_rows(void *arg) {
  job_t *J = (job_t *)arg;
  for (;;) {
    int64_t r = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
    if (r >= J->nrows) break;
    one_row(J, J->rows[3 * r], J->rows[3 * r + 1], J->rows[3 * r + 2], J->out_rows + r * J->D);
  }
  return NULL;
}

static int run_pool(job_t *J, void *(*fn)(void *), int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads == 1) {
    fn(J);
    return 0;
  }
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return -1;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, fn, J) != 0) break;
    ++started;
  }
  if (started == 0) fn(J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  return 0;
}

static int check_args(int64_t B, int64_t Nq, int64_t Nk, int64_t D, int mask_type) {
  if (B < 0 || Nq <= 0 || Nk <= 0 || D <= 0) return -1;
  if (Nq % Nk != 0) return -1;
  if (mask_type != ORACLE_MASK_CAUSAL && mask_type != ORACLE_MASK_NONE &&
      mask_type != ORACLE_MASK_CUSTOM)
    return -1;
  return 0;
}

/* The key side: a page table that names pages outside the cache or a last page length
 * outside [1, page_size], or a sequence with more queries than keys, is rejected. */
static int check_kv(const job_t *J, int64_t num_pages) {
  if (J->kv_cache && J->page_size <= 0) return -1;
  for (int64_t b = 0; b < J->B; ++b) {
    if (J->kv_cache) {
      const int64_t pages = J->page_offsets[b + 1] - J->page_offsets[b];
      if (pages < 0) return -1;
      if (pages > 0 && (J->last_page_len[b] < 1 || J->last_page_len[b] > J->page_size))
        return -1;
      for (int64_t x = 0; x < pages; ++x) {
        const int64_t id = J->page_ids[J->page_offsets[b] + x];
        if (id < 0 || id >= num_pages) return -1;
      }
    }
    const int64_t Lq = J->seq_offsets[b + 1] - J->seq_offsets[b];
    if (Lq < 0 || new_kv_len(J, b) < 0 || Lq > history_len(J, b) + new_kv_len(J, b)) return -1;
  }
  return 0;
}

static void set_kv(job_t *J, const int64_t *seq_offsets_k, const double *kv_cache,
                   const int64_t *page_offsets, const int64_t *page_ids,
                   const int64_t *last_page_len, int64_t page_size) {
  J->seq_offsets_k = seq_offsets_k;
  J->kv_cache = kv_cache;
  J->page_offsets = page_offsets;
  J->page_ids = page_ids;
  J->last_page_len = last_page_len;
  J->page_size = page_size;
}

/*
 * Whole forward. q [T, Nq, D], k/v [Tk, Nk, D], rab [B, rab_heads, S, S] or NULL
 * (rab_heads = Nq, or 1 for a plane shared by all heads), mask [B, Nq, S, S] (custom
 * mask, mask_type 3 only) or NULL, S = max_seqlen (the key-side bound Sk),
 * seq_offsets [B+1] (queries), num_context/num_targets [B] or NULL; out [T, Nq, D].
 * Key side: seq_offsets_k [B+1] (new k/v rows; NULL = seq_offsets), and kv_cache
 * [num_pages, 2, page_size, Nk, D] with page_offsets [B+1], page_ids, last_page_len [B]
 * (kv_cache NULL = no history).
 * Rows of out outside every sequence are left untouched. Returns 0 or -1.
 */
int hstu_oracle_fwd(const double *q, const double *k, const double *v,
                    const int64_t *seq_offsets, int64_t B, int64_t Nq, int64_t Nk,
                    int64_t D, const double *rab, int64_t rab_heads, const double *mask,
                    int64_t max_seqlen, const int64_t *seq_offsets_k, const double *kv_cache,
                    int64_t num_pages, const int64_t *page_offsets, const int64_t *page_ids,
                    const int64_t *last_page_len, int64_t page_size,
                    const int64_t *num_context,
                    const int64_t *num_targets, int mask_type, int64_t target_group_size,
                    double alpha, double silu_scale, double *out, int nthreads) {
  if (check_args(B, Nq, Nk, D, mask_type)) return -1;
  if (rab && rab_heads != 1 && rab_heads != Nq) return -1;
  if ((mask_type == ORACLE_MASK_CUSTOM) != (mask != NULL)) return -1;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.seq_offsets = seq_offsets; J.B = B;
  set_kv(&J, seq_offsets_k, kv_cache, page_offsets, page_ids, last_page_len, page_size);
  if (check_kv(&J, num_pages)) return -1;
  J.q = q; J.k = k; J.v = v; J.rab = rab; J.mask = mask;
  J.seq_offsets = seq_offsets; J.num_context = num_context; J.num_targets = num_targets;
  J.B = B; J.Nq = Nq; J.Nk = Nk; J.D = D; J.max_seqlen = max_seqlen; J.rab_heads = rab_heads;
  J.mask_type = mask_type; J.g = target_group_size;
  J.alpha = alpha; J.silu_scale = silu_scale; J.out = out;
  return run_pool(&J, worker_units, nthreads);
}

/* Selected rows only: rows[3r..3r+2] = (b, h, i); out_rows [nrows, D]. */
int hstu_oracle_fwd_rows(const double *q, const double *k, const double *v,
                         const int64_t *seq_offsets, int64_t B, int64_t Nq, int64_t Nk,
                         int64_t D, const double *rab, int64_t rab_heads,
                         const double *mask, int64_t max_seqlen,
                         const int64_t *seq_offsets_k, const double *kv_cache,
                         int64_t num_pages, const int64_t *page_offsets,
                         const int64_t *page_ids, const int64_t *last_page_len,
                         int64_t page_size,
                         const int64_t *num_context, const int64_t *num_targets,
                         int mask_type, int64_t target_group_size, double alpha,
                         double silu_scale, const int64_t *rows, int64_t nrows,
                         double *out_rows, int nthreads) {
  if (check_args(B, Nq, Nk, D, mask_type)) return -1;
  if (rab && rab_heads != 1 && rab_heads != Nq) return -1;
  if ((mask_type == ORACLE_MASK_CUSTOM) != (mask != NULL)) return -1;
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
    if (b < 0 || b >= B || h < 0 || h >= Nq || i < 0 ||
        i >= seq_offsets[b + 1] - seq_offsets[b])
      return -1;
  }
  job_t J;
  memset(&J, 0, sizeof(J));
  J.seq_offsets = seq_offsets; J.B = B;
  set_kv(&J, seq_offsets_k, kv_cache, page_offsets, page_ids, last_page_len, page_size);
  if (check_kv(&J, num_pages)) return -1;
  J.q = q; J.k = k; J.v = v; J.rab = rab; J.mask = mask;
  J.seq_offsets = seq_offsets; J.num_context = num_context; J.num_targets = num_targets;
  J.B = B; J.Nq = Nq; J.Nk = Nk; J.D = D; J.max_seqlen = max_seqlen; J.rab_heads = rab_heads;
  J.mask_type = mask_type; J.g = target_group_size;
  J.alpha = alpha; J.silu_scale = silu_scale;
  J.rows = rows; J.nrows = nrows; J.out_rows = out_rows;
  return run_pool(&J, worker_rows, nthreads);
}

/* Number of (query head, i, j) triples with valid(i, j): sum over b of Nq * #valid. */
int64_t hstu_oracle_count_valid(const int64_t *seq_offsets, int64_t B, int64_t Nq,
                                const int64_t *num_context, const int64_t *num_targets,
                                int mask_type, int64_t target_group_size) {
  int64_t total = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t L = seq_offsets[b + 1] - seq_offsets[b];
    const int64_t nc = num_context ? num_context[b] : 0;
    const int64_t nt = num_targets ? num_targets[b] : 0;
    int64_t c = 0;
    for (int64_t i = 0; i < L; ++i)
      for (int64_t j = 0; j < L; ++j)
        c += hstu_oracle_valid(i, j, L, mask_type, nc, nt, target_group_size);
    total += c * Nq;
  }
  return total;
}

/* Mask-aware pair count with per-sequence query and key lengths: sum over b of
 * Nq * #{(i, j) : i < lq[b], j < lk[b], valid(lk[b] - lq[b] + i, j, lk[b])}. */
int64_t hstu_oracle_count_valid_kv(const int64_t *lq, const int64_t *lk, int64_t B, int64_t Nq,
                                   const int64_t *num_context, const int64_t *num_targets,
                                   int mask_type, int64_t target_group_size) {
  int64_t total = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t nc = num_context ? num_context[b] : 0;
    const int64_t nt = num_targets ? num_targets[b] : 0;
    int64_t c = 0;
    for (int64_t i = 0; i < lq[b]; ++i)
      for (int64_t j = 0; j < lk[b]; ++j)
        c += hstu_oracle_valid(lk[b] - lq[b] + i, j, lk[b], mask_type, nc, nt,
                               target_group_size);
    total += c * Nq;
  }
  return total;
}
