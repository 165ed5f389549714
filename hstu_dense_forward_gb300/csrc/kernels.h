// Launch interface between the host planner (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hstu {

// Everything a forward kernel reads besides the tensor maps. Device pointers.
struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* rab;          // [B, Nq, S, S] or nullptr
  void* out;
  const void* seq_offsets;  // [B+1]
  const void* num_context;  // [B] or nullptr
  const void* num_targets;  // [B] or nullptr
  const uint32_t* work;     // work list: packed (b, m-tile), heaviest first
  const int* work_count;    // number of list entries
  int* next_item;           // dynamic scheduling counter (reset by the work-list builder)
  int* err;                 // device error word (HSTU_DEVERR_*)
  long long total_tokens;   // T
  long long timeout_ns;     // limit of one pipeline wait
  int index64;              // index tensors are int64
  int B, Nq, Nk, D, S;      // batch, heads, head dim, max_seqlen
  int mask_type, g;         // mask code, target group size
  int dense;                // normal layout: sequence b is tokens [b * S, (b + 1) * S)
  int rab_bcast;            // rab [B, 1, S, S]: one bias plane for every query head
  int rab_is_mask;          // the rab stream carries a custom mask [B, Nq, S, S]: P is
                            // multiplied by it after the SiLU instead of rab being added
                            // before (mask_type is then NONE for the tile geometry)
  const void* mask;         // a custom mask [B, Nq, S, S] given together with rab (rab in
                            // `rab`, rab_is_mask 0, mask_type NONE), or nullptr
  float alpha, silu_scale;
  // Key side. The keys of sequence b are its cached history (page_offsets != nullptr)
  // followed by its new k/v rows: rows [seq_offsets_k[b], seq_offsets_k[b + 1]) of k and v,
  // or, with seq_offsets_k == nullptr, the rows of its queries. The Lq queries are the last
  // Lq of the Lk key positions. S bounds Lk (and is the row length of rab), Sq bounds Lq.
  const void* seq_offsets_k;  // [B+1] or nullptr
  const void* page_offsets;   // [B+1] or nullptr (no cache)
  const void* page_ids;       // [page_offsets[B]]
  const void* last_page_len;  // [B]
  const void* kv_cache;       // [num_pages, 2, page_size, Nk, D]
  long long total_tokens_k;   // rows of k and v
  long long num_pages;
  int page_size;
  int Sq;
  int fp8;                    // q, k, v (and the cache) are FP8 E4M3; out is bf16
  int test_stall;             // watchdog test (plans created with HSTU_TEST_STALL=k): the K
                              // producer signals nothing, so the first score product's wait
                              // runs out and the kernel takes its timeout path
  unsigned long long* trace;  // pipeline trace buffer (builds with HSTU_TRACE=1), or nullptr
  // rab added by the tensor core (head dims up to 64, bf16/fp16, no key side): the kernel
  // variant that multiplies the rab tile by a diagonal operand holding rab_ident, the 16-bit
  // pattern of 1/alpha in the input type (set by the host when 1/alpha is finite there)
  int rab_mma;
  unsigned rab_ident;
  // FP8 descale factors (an element's value is its factor times the stored E4M3 value):
  // device fp32 arrays indexed by ds_index; ds_mode 0 is the plain cast (no arrays)
  const float* q_ds;
  const float* k_ds;
  const float* v_ds;
  int ds_mode;  // 0 cast, 1 per tensor, 2 per sequence, 3 per sequence and head, 4 per block
  int ds_qb;    // 128-row query blocks per sequence (ceil(Sq / 128)), mode 4
  int ds_kb;    // 128-position key blocks per sequence (ceil(S / 128)), mode 4
};

// FP8 kernels hold kP8Scale * P (E4M3) for the second product; silu_scale is divided by it.
constexpr float kP8Scale = 16.0f;

__host__ __device__ inline long long load_index(const void* p, long long i, int is64) {
  return is64 ? static_cast<const long long*>(p)[i] : static_cast<const int*>(p)[i];
}

// First token of sequence b: from seq_offsets (jagged layout) or b * S (normal layout).
__host__ __device__ inline long long seq_start(const FwdParams& p, long long b) {
  return p.dense ? b * p.S : load_index(p.seq_offsets, b, p.index64);
}

// Query and key geometry of sequence b (after the work-list builder has validated it).
struct SeqKV {
  long long tq;    // first query row
  long long tk;    // first new k/v row
  long long po;    // first page_ids entry of the sequence
  long long Lq;    // query rows
  long long hist;  // cached keys: positions [0, hist)
  long long Lk;    // keys: hist + new rows; query row i sits at position Lk - Lq + i
};

__host__ __device__ inline SeqKV seq_kv(const FwdParams& p, long long b) {
  SeqKV s;
  s.tq = seq_start(p, b);
  s.Lq = seq_start(p, b + 1) - s.tq;
  long long nk = s.Lq;
  s.tk = s.tq;
  if (p.seq_offsets_k) {
    s.tk = load_index(p.seq_offsets_k, b, p.index64);
    nk = load_index(p.seq_offsets_k, b + 1, p.index64) - s.tk;
  }
  s.po = 0;
  s.hist = 0;
  if (p.page_offsets) {
    s.po = load_index(p.page_offsets, b, p.index64);
    const long long pages = load_index(p.page_offsets, b + 1, p.index64) - s.po;
    if (pages > 0)
      s.hist = (pages - 1) * p.page_size + load_index(p.last_page_len, b, p.index64);
  }
  s.Lk = s.hist + nk;
  return s;
}

// rab plane of (sequence b, query head h): [B, Nq, S, S], or [B, 1, S, S] broadcast.
__host__ __device__ inline long long rab_plane(const FwdParams& p, long long b, int h) {
  return p.rab_bcast ? b : b * p.Nq + h;
}

// Scheduler: validates seq_offsets and writes the work list (one CTA).
cudaError_t launch_build_worklist(const FwdParams& p, uint32_t* work, int* work_count,
                                  int tile_m, cudaStream_t stream,
                                  bool pdl);

// fp32 path on CUDA cores.
size_t simt_smem_bytes(int D);
cudaError_t simt_prepare();
cudaError_t launch_fwd_simt(const FwdParams& p, int grid, cudaStream_t stream, bool pdl);

// bf16 / fp16 tensor-core path (tcgen05, TMA, TMEM).
struct TcMaps {
  CUtensorMap q, k, v, rab, out, cache, mask;  // (mask: a custom mask beside rab)
};
bool tc_supported_dim(int D);
int tc_kernel_dim(int D);     // head dim of the kernel variant that runs D (32/64/128/256)
int tc_swizzle_bytes(int D, int elem_bytes);  // row width of one TMA box / UMMA swizzle atom
int tc_out_box_cols(int D);   // columns of one output store box (32 rows each)
int tc_rab_box_rows();        // rows of one rab / custom-mask load box (64 columns each)
int tc_v_box_rows(int D);     // rows of one V load box (64 for the 512 kernel, else 128)
// elem: 0 f16, 1 bf16, 2 FP8 E4M3; rab: 0 none, 1 rab, 2 custom mask, 3 custom mask and
// rab; kv: the key-side variant (own k/v offsets, KV cache)
cudaError_t tc_prepare(int D, int elem, int rab, int kv, int ds = 0);  // ds: FP8 descale mode
// The variant that adds rab with the tensor core exists for these (rab = 1: rab, not a
// custom mask; no key side; bf16 / fp16; head dim 32 or 64).
bool rab_mma_dim(int D, int elem, int rab, int kv);
cudaError_t launch_fwd_tc(const FwdParams& p, const TcMaps& maps, int bf16, int grid,
                          cudaStream_t stream, bool pdl);

}  // namespace hstu
