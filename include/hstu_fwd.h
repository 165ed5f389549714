/*
 * hstu_fwd.h — C ABI of the GB300 (sm_103a) HSTU fused attention forward.
 *
 * The operation ("RecOps Running Case Documentation", gitcode.com/Ascend/RecSDK,
 * docs/en/rec_ops/hstu_v1_forward.md):
 *   - Introduction to the HSTU_V1 Forward Operator: one fused operator chains the
 *     QK matrix multiplication, the SiLU activation, the scaling, the mask and the
 *     multiplication with V.
 *   - Feature table: S = Q*K^T, P = silu(S), O = P*V; MHA and GQA (query heads
 *     map many-to-one onto key/value heads); jagged sequences; fp32/fp16/bf16;
 *     optional relative attention bias rab [b, n, s, s]; no mask or a causal mask
 *     built from num_context, num_targets and target_group_size.
 *   - Inputs and Outputs table: argument layouts, mask_type codes, the silu_scale
 *     default 1/max_seq_len, alpha, and "empty input: the operator does not run";
 *     seq_offsets_q / seq_offsets_k / max_seq_len_k / is_delta_qk (query and key
 *     lengths may differ) and kv_cache / page_offsets / page_ids / last_page_len (the
 *     paged KV cache of the feature table's "Page" row): see hstu_fwd_run_kv.
 *
 * For every sequence b (L = seq_offsets[b+1] - seq_offsets[b], t0 = seq_offsets[b]),
 * query head h (kv head hk = h / (Nq / Nk)), row i < L and column d < D:
 *
 *   x_ij = alpha * sum_d q[t0+i, h, d] * k[t0+j, hk, d]  (+ rab[b, h, i, j])
 *   out[t0+i, h, d] = silu_scale * sum_{j < L, valid(i,j)} silu(x_ij) * v[t0+j, hk, d]
 *
 * with silu(x) = x / (1 + exp(-x)). The page does not place alpha or rab in the
 * formula; this library multiplies Q*K^T by alpha and adds rab after it. The
 * causal predicate valid(i, j) (the page names its inputs but does not spell it
 * out) is, with H = (g > 0) ? max(L - nt, 0) : L:
 *   (j <= i && j < H) || (i < nc && j < H)
 *   || (g > 0 && i >= H && j >= H && j <= i && (i - H) / g == (j - H) / g)
 *   || (g == 0 && j <= i)
 * nc = num_context[b] (0 when absent), nt = num_targets[b] (0 when absent),
 * g = target_group_size. mask_type NONE makes every (i, j) with i, j < L valid.
 *
 * Ownership: the caller owns every tensor. All tensor arguments of
 * hstu_fwd_run are DEVICE pointers to contiguous, 16-byte aligned memory on the
 * plan's device. The plan owns a small device workspace (work list, error word),
 * allocated by hstu_fwd_create and freed by hstu_fwd_destroy.
 *
 * Errors are returned as hstu_status codes; nothing aborts, throws or traps.
 * Asynchronous errors found on the device (invalid seq_offsets, a pipeline wait
 * that ran past its time limit) are recorded in the plan's error word and read
 * with hstu_fwd_get_error.
 */
#ifndef HSTU_FWD_H_
#define HSTU_FWD_H_

#if defined(__GNUC__)
#define HSTU_API __attribute__((visibility("default")))
#else
#define HSTU_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HSTU_OK = 0,
  HSTU_ERR_INVALID_ARG = 1,  /* null pointer, bad size or alignment, bad descriptor */
  HSTU_ERR_UNSUPPORTED = 2,  /* valid on the page but not built here (see each field) */
  HSTU_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  HSTU_ERR_TIMEOUT = 4,      /* a device pipeline wait ran past its limit (error word) */
  HSTU_ERR_DEVICE_CHECK = 5  /* the device rejected the inputs (error word) */
} hstu_status;

/* Element type of q, k, v, rab and out (Inputs and Outputs table: "the type must
 * match q"; the output "same as q"). HSTU_FP8_E4M3 (feature table, "FP8 quantization
 * types"): q, k, v and the KV cache hold FP8 E4M3 bytes, either a plain cast or scaled
 * copies with descale factors (desc.descale, hstu_fwd_run_fp8); both products run on
 * 8-bit tensor cores with fp32 accumulation, P is rounded to E4M3 (saturating) for the
 * second one, and out is bf16. rab (has_rab, no key side) is bf16 [B, Nq or 1, S, S] and
 * is added in fp32; a custom mask (no key side, not together with rab) is bf16 and
 * multiplies P in fp32 before its E4M3 rounding. Head dims 16 to 128 in steps of 16; not
 * on the allocation-free entry point. */
typedef enum { HSTU_F32 = 0, HSTU_F16 = 1, HSTU_BF16 = 2, HSTU_FP8_E4M3 = 3 } hstu_dtype;

/* Granularity of the FP8 descale factors (feature table, "FP8 quantization types": cast,
 * per-tensor, per-batch, per-head, per-block). The value of an element is its descale
 * factor times the stored E4M3 value. Factor arrays are fp32 (hstu_fwd_descale):
 *   CAST    no factors (every factor 1)
 *   TENSOR  q [1], k [1], v [1]
 *   BATCH   q [B], k [B], v [B]: one factor per sequence
 *   HEAD    q [B, Nq], k [B, Nk], v [B, Nk]: per sequence and head
 *   BLOCK   q [B, ceil(max_seqlen / 128), Nq], k and v [B, ceil(Sk / 128), Nk]: per
 *           sequence, head and block of 128 query rows (q) or 128 key positions (k, v),
 *           counted from the sequence's first query row / first key (cached history
 *           included); Sk is the key bound (max_seqlen_k, else max_seqlen).
 * BLOCK factors of v scale P before its E4M3 rounding relative to the largest |factor| of
 * the sequence's v blocks, so blocks whose factors are far below that largest one lose
 * precision to E4M3's subnormal range. */
typedef enum {
  HSTU_DESCALE_CAST = 0,
  HSTU_DESCALE_TENSOR = 1,
  HSTU_DESCALE_BATCH = 2,
  HSTU_DESCALE_HEAD = 3,
  HSTU_DESCALE_BLOCK = 4
} hstu_descale_granularity;

/* Tensor layout (Inputs and Outputs table, layout): "jagged" q [T, Nq, D] with
 * seq_offsets, or "normal" q [B, S, Nq, D] where every sequence has S = max_seqlen
 * tokens (the same memory as jagged with seq_offsets[b] = b * S, T = B * S). */
typedef enum { HSTU_LAYOUT_JAGGED = 0, HSTU_LAYOUT_NORMAL = 1 } hstu_layout;

/* mask_type codes of the Inputs and Outputs table. UPPER ("currently not
 * supported" on the page) is rejected with HSTU_ERR_UNSUPPORTED. */
typedef enum {
  HSTU_MASK_CAUSAL = 0, /* built-in lower-triangular mask with context/targets */
  HSTU_MASK_UPPER = 1,
  HSTU_MASK_NONE = 2,   /* bidirectional: no mask */
  HSTU_MASK_CUSTOM = 3  /* mask [B, Nq, S, S] passed to hstu_fwd_run_masked (or, together
                           with rab, to hstu_fwd_run_args): P is multiplied by mask[b, h, i, j]
                           after the SiLU and the scaling; no context or target counts. With
                           rab (has_rab): head dims up to 128 on the 16-bit path
                           (HSTU_ERR_UNSUPPORTED otherwise) */
} hstu_mask_type;

/* Device error word values (hstu_fwd_get_error). */
enum {
  HSTU_DEVERR_NONE = 0,
  HSTU_DEVERR_OFFSETS = 1,  /* seq_offsets not increasing from >= 0, last > total_tokens,
                               or a length above max_seqlen: nothing was written */
  HSTU_DEVERR_TIMEOUT = 2   /* a pipeline wait gave up; out is incomplete */
};

typedef struct {
  int dtype;             /* hstu_dtype */
  int batch;             /* B in [0, 2^20]; 0 = empty input, run does nothing */
  int num_heads_q;       /* Nq >= 0; 0 = empty input */
  int num_heads_kv;      /* Nk >= 1, Nq % Nk == 0 (Inputs and Outputs table, k) */
  int head_dim;          /* D: f16/bf16 need a multiple of 16 in [16, 512] (above 256: no
                            rab, custom mask or key side), FP8 one in [16, 128]; f32 needs
                            1 <= D <= 256 */
  int max_seqlen;        /* S in [1, 131072]: bound on every L; rab is [B, Nq, S, S];
                            for rab with f16/bf16, S must be a multiple of 8 */
  int index_is_int64;    /* 1: seq_offsets/num_context/num_targets are int64, 0: int32 */
  int mask_type;         /* hstu_mask_type: CAUSAL or NONE */
  int target_group_size; /* g >= 0; 0 = no target mask (causal only) */
  int has_rab;           /* 1: rab is passed to every run */
  int has_num_context;   /* 1: num_context [B] is passed to every run */
  int has_num_targets;   /* 1: num_targets [B] is passed to every run */
  int watchdog_ms;       /* limit of one device pipeline wait; 0 = 1000 ms. Test aid: a
                            bf16/fp16/FP8 plan created while the environment holds
                            HSTU_TEST_STALL=k never signals its K tiles, so every run
                            ends through this limit with HSTU_DEVERR_TIMEOUT */
  int layout;            /* hstu_layout; 0 = jagged */
  int rab_heads;         /* bias planes per sequence: 0 or Nq for rab [B, Nq, S, S]; 1 for
                            rab [B, 1, S, S], one plane added for every query head (feature
                            table, "Support for rab broadcasting") */
  int is_delta_qk;       /* 1: the new k/v rows have offsets of their own (seq_offsets_k of
                            hstu_fwd_kv); jagged layout only */
  int max_seqlen_k;      /* Sk, bound on the keys of a sequence (history + new rows) and the
                            S of rab / mask when is_delta_qk or page_size is set (0 = use
                            max_seqlen); must be 0 otherwise. max_seqlen then bounds the
                            query rows of a sequence */
  int page_size;         /* 0, or the rows of one KV-cache page: 32, 128 or 256 (Inputs and
                            Outputs table, kv_cache); jagged layout only */
  int descale;           /* hstu_descale_granularity; FP8 plans only (0 otherwise). Plans
                            with a value other than CAST run through hstu_fwd_run_fp8 */
  int reserved;          /* must be 0 */
} hstu_fwd_desc;

/*
 * Key side of hstu_fwd_run_kv (Inputs and Outputs table: seq_offsets_k, kv_cache,
 * page_offsets, page_ids, last_page_len). Index arrays are int32 or int64 per
 * desc.index_is_int64; all pointers are DEVICE pointers.
 */
typedef struct {
  const void* seq_offsets_k;  /* [B+1] new k/v rows of each sequence (desc.is_delta_qk = 1),
                                 increasing, seq_offsets_k[B] <= total_tokens_k; NULL when
                                 is_delta_qk = 0: the new k/v rows are the query rows */
  long long total_tokens_k;   /* rows of k and v (is_delta_qk = 1; ignored otherwise, when k
                                 and v have total_tokens rows). With 0, k and v may be NULL */
  const void* kv_cache;       /* [num_pages, 2, page_size, Nk, D] of the plan's dtype, 16-byte
                                 aligned: plane 0 of a page holds K rows, plane 1 V rows.
                                 NULL iff desc.page_size = 0. Rows past a sequence's last
                                 valid row must hold finite values (they are multiplied by 0) */
  long long num_pages;
  const void* page_offsets;   /* [B+1] the pages of sequence b are page_ids[page_offsets[b]
                                 .. page_offsets[b+1]), in order */
  const void* page_ids;       /* [page_offsets[B]] values in [0, num_pages) */
  const void* last_page_len;  /* [B] rows of the last page, in [1, page_size] (unused for a
                                 sequence without pages) */
} hstu_fwd_kv;

typedef struct hstu_fwd_plan hstu_fwd_plan; /* opaque */

/* Validate desc for the current CUDA device, allocate the plan's workspace.
 * *plan is set on HSTU_OK only. */
HSTU_API hstu_status hstu_fwd_create(const hstu_fwd_desc* desc, hstu_fwd_plan** plan);

/*
 * Enqueue one forward on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   q    [T, Nq, D]        k, v [T, Nk, D]       out [T, Nq, D]   (dtype of the plan)
 *   seq_offsets [B+1]      increasing from 0, seq_offsets[B] <= T; for the normal layout
 *                          NULL, and T must be B * S (q is [B, S, Nq, D])
 *   rab  [B, Nq, S, S] (or [B, 1, S, S] with desc.rab_heads = 1) or NULL (must be
 *        non-NULL iff desc.has_rab)
 *   num_context, num_targets [B] or NULL (non-NULL iff the desc flags say so)
 *   total_tokens = T, the row count of q, k, v and out.
 * Rows of out that belong to no sequence are not written. silu_scale is used as
 * given (the Python layer supplies 1/max_seqlen when the caller passes none).
 * Asynchronous: no allocation, no synchronisation. One plan must not be used by
 * two runs that may execute at the same time (it holds one work list).
 * Returns HSTU_OK with nothing enqueued when B, Nq or T is 0.
 *
 * Stream order (every entry point that takes a plan): the run's first kernel, the
 * work-list build, is launched with programmatic dependent launch. It reads the index
 * arrays (seq_offsets, num_context, num_targets and the key side's seq_offsets_k,
 * page_offsets, page_ids, last_page_len) while the kernel before it on the stream may
 * still run, and it completes only after that kernel; every other input is read after
 * that. A kernel that does not trigger its dependents early (no
 * cudaTriggerProgrammaticLaunchCompletion / griddepcontrol.launch_dependents): every
 * PyTorch kernel, and this library's forward kernel, which writes no index array, has
 * completed before the build starts. A kernel that does trigger early and writes those
 * arrays after its trigger must not directly precede a run: put another stream operation
 * between them.
 */
HSTU_API hstu_status hstu_fwd_run(hstu_fwd_plan* plan, const void* q, const void* k, const void* v,
                         const void* seq_offsets, const void* rab, const void* num_context,
                         const void* num_targets, long long total_tokens, float alpha,
                         float silu_scale, void* out, void* stream);

/*
 * Enqueue one forward of a plan created with mask_type HSTU_MASK_CUSTOM ("3: use a
 * custom mask; the user must define and pass in the mask", Inputs and Outputs table).
 *   mask [B, Nq, S, S] of the plan's dtype, 16-byte aligned; every other argument as
 *   for hstu_fwd_run (no rab, num_context or num_targets). Every key j < L of a
 *   sequence is a candidate and P(i, j) is multiplied by mask[b, h, i, j]; a 0/1 mask
 *   selects. Returns HSTU_ERR_INVALID_ARG for a plan of another mask type or one with
 *   has_rab (which runs through hstu_fwd_run_args), and hstu_fwd_run does for a CUSTOM
 *   plan.
 */
HSTU_API hstu_status hstu_fwd_run_masked(hstu_fwd_plan* plan, const void* q, const void* k,
                                         const void* v, const void* seq_offsets,
                                         const void* mask, long long total_tokens, float alpha,
                                         float silu_scale, void* out, void* stream);

/*
 * Enqueue one forward whose queries and keys may differ (plans with is_delta_qk or
 * page_size set; any plan accepts kv = NULL, which is hstu_fwd_run / hstu_fwd_run_masked).
 * For sequence b: Lq = seq_offsets[b+1] - seq_offsets[b] query rows (q and out rows
 * from seq_offsets[b]); the keys are the cached history, hist = (pages - 1) * page_size +
 * last_page_len[b] rows from the pages (0 without pages or cache), followed by the new
 * k/v rows; Lk = hist + new rows, Lq <= Lk <= Sk, Lq <= max_seqlen. Query row i sits at
 * key position p = Lk - Lq + i (the queries are the last Lq tokens): the mask is
 * valid(p, j) over L = Lk and the rab / custom-mask row is p. rab_or_mask is rab
 * [B, Nq or 1, Sk, Sk] for plans with has_rab, the mask [B, Nq, Sk, Sk] for CUSTOM plans,
 * else NULL. Other arguments as for hstu_fwd_run. Invalid offsets or page tables (a
 * page id outside the cache, last_page_len outside [1, page_size], Lq > Lk, a length
 * above its bound) are reported through the error word (HSTU_DEVERR_OFFSETS) and leave
 * out unwritten.
 */
HSTU_API hstu_status hstu_fwd_run_kv(hstu_fwd_plan* plan, const void* q, const void* k,
                                     const void* v, const void* seq_offsets,
                                     const hstu_fwd_kv* kv, const void* rab_or_mask,
                                     const void* num_context, const void* num_targets,
                                     long long total_tokens, float alpha, float silu_scale,
                                     void* out, void* stream);

/*
 * Every input of one forward, for hstu_fwd_run_args: the general entry point, the only one
 * that takes a custom mask together with rab. Pointers as for hstu_fwd_run / _kv / _fp8;
 * NULL for what the plan does not use.
 */
typedef struct hstu_fwd_descale hstu_fwd_descale;
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const void* seq_offsets;
  const hstu_fwd_kv* kv;            /* key side (plans with is_delta_qk or page_size) */
  const void* rab;                  /* plans with has_rab */
  const void* mask;                 /* plans with mask_type CUSTOM */
  const void* num_context;
  const void* num_targets;
  const hstu_fwd_descale* descale;  /* FP8 plans whose descale is not CAST */
  long long total_tokens;
  float alpha;
  float silu_scale;
} hstu_fwd_args;

/* Enqueue one forward with every input in `args` (see hstu_fwd_args). A CUSTOM plan with
 * has_rab adds rab[b, h, i, j] before the SiLU and multiplies P by mask[b, h, i, j] after
 * it. Returns HSTU_ERR_INVALID_ARG when an input the plan needs is missing or one it does
 * not take is given. */
HSTU_API hstu_status hstu_fwd_run_args(hstu_fwd_plan* plan, const hstu_fwd_args* args,
                                       void* stream);

/* Descale factor arrays of hstu_fwd_run_fp8 / hstu_fwd_run_args: DEVICE pointers to fp32, 4-byte aligned, of
 * the lengths that desc.descale gives (hstu_descale_granularity). */
struct hstu_fwd_descale {
  const float* q;
  const float* k;
  const float* v;
};

/*
 * Enqueue one forward of an FP8 E4M3 plan with descale factors (feature table, "FP8
 * quantization types"): x_ij = alpha * (qd q_i) . (kd k_j) (+ rab), and v_j is vd v_j,
 * with qd, kd, vd the factors of desc.descale's granularity for row i and key j.
 * kv as for hstu_fwd_run_kv (NULL for a plan without a key side), rab as for hstu_fwd_run
 * (bf16; not with a key side), other arguments as for hstu_fwd_run. descale may be NULL
 * only for a CAST plan. Returns HSTU_ERR_INVALID_ARG for a plan that is not FP8 or has
 * mask_type CUSTOM (hstu_fwd_run_args takes a mask with descales), and hstu_fwd_run /
 * hstu_fwd_run_kv do for an FP8 plan whose granularity is not CAST.
 */
HSTU_API hstu_status hstu_fwd_run_fp8(hstu_fwd_plan* plan, const void* q, const void* k,
                                      const void* v, const void* seq_offsets,
                                      const hstu_fwd_kv* kv, const void* rab,
                                      const void* num_context, const void* num_targets,
                                      const hstu_fwd_descale* descale, long long total_tokens,
                                      float alpha, float silu_scale, void* out, void* stream);

/* Free the workspace. NULL is accepted. Waits for the plan's last run to complete first
 * (an event recorded on that run's stream; other streams and plans are not waited for). */
HSTU_API hstu_status hstu_fwd_destroy(hstu_fwd_plan* plan);

/* Wait for the plan's last run to complete (an event recorded on that run's stream, not a
 * device-wide synchronisation), read the plan's device error word into *device_error
 * (HSTU_DEVERR_*), and clear it. Returns HSTU_ERR_DEVICE_CHECK or HSTU_ERR_TIMEOUT when
 * the word was set, else HSTU_OK. */
HSTU_API hstu_status hstu_fwd_get_error(hstu_fwd_plan* plan, int* device_error);

/* Kernel launches one hstu_fwd_run enqueues for this plan (for launch accounting). */
HSTU_API hstu_status hstu_fwd_launches_per_run(const hstu_fwd_plan* plan, int* launches);

/* Host-side count of the mask-aware work: sum over sequences of Nq * #valid(i, j),
 * from HOST arrays seq_offsets [B+1] (NULL for the normal layout: every length is S)
 * and optional num_context / num_targets [B]
 * (int32 or int64 per desc.index_is_int64). 4 * D * pairs is the useful flop
 * count of one run. */
HSTU_API hstu_status hstu_fwd_count_pairs(const hstu_fwd_desc* desc, const void* seq_offsets_host,
                                 const void* num_context_host, const void* num_targets_host,
                                 long long* pairs);

/* hstu_fwd_count_pairs for hstu_fwd_run_kv calls, from HOST arrays: seq_offsets [B+1]
 * (queries), seq_offsets_k [B+1] or NULL (new k/v rows = query rows), page_offsets [B+1]
 * and last_page_len [B] or NULL (no cache); pairs = sum over sequences of
 * Nq * #{(i, j): i < Lq, j < Lk, valid(Lk - Lq + i, j)}. */
HSTU_API hstu_status hstu_fwd_count_pairs_kv(const hstu_fwd_desc* desc,
                                             const void* seq_offsets_host,
                                             const void* seq_offsets_k_host,
                                             const void* page_offsets_host,
                                             const void* last_page_len_host,
                                             const void* num_context_host,
                                             const void* num_targets_host, long long* pairs);

/*
 * Same forward as hstu_fwd_run, without a plan and without allocating anything.
 * The source pages have no counterpart to this entry point: it exists for callers
 * that cannot call cudaMalloc, such as a plugin that its host framework only hands
 * input and output buffers, a runtime whose memory pool has already reserved all
 * device memory, or a latency-critical path that must not pay for cudaMalloc's
 * implicit device synchronisation.
 *   - The work list lives in a fixed device array inside the library (about 64 KB,
 *     held by every GPU that loads the library until the process exits). It has room
 *     for batch * ceil(max_seqlen / 128) <= 16384 entries; larger descriptors return
 *     HSTU_ERR_UNSUPPORTED without launching anything.
 *   - Arguments, layouts and ownership are those of hstu_fwd_run; desc is validated
 *     like hstu_fwd_create validates it, on every call. Descriptors with is_delta_qk or
 *     page_size set, mask_type CUSTOM or dtype HSTU_FP8_E4M3 return
 *     HSTU_ERR_UNSUPPORTED.
 *   - The first call on a device (with that device current) looks up the array's
 *     device address and configures the kernels for that device; make that first
 *     call before any stream capture.
 *   - All calls share the one array: calls whose kernels may overlap on the GPU
 *     (different streams without ordering, several host threads) race and produce
 *     wrong results. Serialise them.
 *   - Nothing detected on the device is reported back: invalid seq_offsets leave out
 *     unwritten, and a pipeline wait that runs past its limit (HSTU_DEVERR_TIMEOUT on a
 *     plan) leaves out partly written, while the call still returns HSTU_OK. Use a plan
 *     and hstu_fwd_get_error when such errors must be seen.
 */
HSTU_API hstu_status hstu_fwd_run_noalloc(const hstu_fwd_desc* desc, const void* q, const void* k,
                                          const void* v, const void* seq_offsets, const void* rab,
                                          const void* num_context, const void* num_targets,
                                          long long total_tokens, float alpha, float silu_scale,
                                          void* out, void* stream);

/*
 * Pipeline trace of the plan's forward kernels (tooling; the source pages have no
 * counterpart). Only a library built with -DHSTU_TRACE=1 records one: there every
 * bf16/fp16/FP8 plan owns a 40 MB device buffer of four launch slots (run r of the plan
 * records into slot r % 4) into which selected threads of each CTA stamp pipeline events
 * (event kind, tile or item counter, SM clock). This call waits for the plan's last run,
 * copies min(bytes, 40 MB) of the buffer to the HOST memory at `host`, and clears it. Returns HSTU_ERR_UNSUPPORTED from ordinary builds and
 * for fp32 plans; HSTU_ERR_INVALID_ARG for a NULL plan or host pointer.
 */
HSTU_API hstu_status hstu_fwd_trace_read(hstu_fwd_plan* plan, void* host, long long bytes);

/* Static description of a status code. */
HSTU_API const char* hstu_status_string(hstu_status status);

#ifdef __cplusplus
}
#endif

#endif /* HSTU_FWD_H_ */
