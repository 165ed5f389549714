// C ABI and host planner of the HSTU forward: descriptor validation, workspace,
// TMA tensor maps, kernel selection and launch. See include/hstu_fwd.h for the
// contract of every entry point.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <cmath>
#include <initializer_list>
#include <mutex>

#include "../../include/hstu_fwd.h"
#include "common.cuh"
#include "kernels.h"
#include "trace.cuh"

using hstu::FwdParams;
using hstu::TcMaps;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct hstu_fwd_plan {
  hstu_fwd_desc desc;
  int device;
  int num_sms;
  int grid;            // CTAs of the forward kernel
  bool tensor_cores;   // bf16/fp16 tcgen05 path (else the fp32 CUDA-core path)
  // Two work lists used by alternate runs, so that a run's work-list build can overlap the
  // end of the previous run's forward kernel: list b at d_work + b * work_cap, its entry
  // count at d_count[4 * b] and its claim counter at d_count[4 * b + 2].
  uint32_t* d_work;    // 2 x work_cap entries
  size_t work_cap;     // B * ceil(S / 128)
  int* d_count;
  int* d_err;          // device error word (d_count[1])
  int parity;          // work list of the next run
  int test_stall;      // HSTU_TEST_STALL=k at create: the watchdog test mode
  long long timeout_ns;
  // tensor maps of the last run, re-encoded when a pointer or a row count changes
  TcMaps maps;
  const void* map_ptrs[7];
  long long map_T, map_Tk, map_pages;
  bool maps_valid;
  unsigned long long* d_trace;  // pipeline trace buffer (builds with HSTU_TRACE=1 only)
  long long runs;               // runs enqueued (selects the trace slot)
  // Completion of the plan's last run (recorded on the run's stream) and a private
  // non-blocking stream: get_error and destroy wait for the plan's own work only.
  cudaEvent_t done;
  cudaStream_t aux;
};

extern "C" {

const char* hstu_status_string(hstu_status s) {
  switch (s) {
    case HSTU_OK: return "ok";
    case HSTU_ERR_INVALID_ARG: return "invalid argument";
    case HSTU_ERR_UNSUPPORTED: return "unsupported configuration";
    case HSTU_ERR_CUDA: return "CUDA runtime error";
    case HSTU_ERR_TIMEOUT: return "device pipeline wait timed out";
    case HSTU_ERR_DEVICE_CHECK: return "device rejected the inputs";
  }
  return "unknown status";
}

// seq_offsets for the jagged layout; none for the normal layout, whose token count is
// fixed (B sequences of S tokens).
static bool layout_args_ok(const hstu_fwd_desc& d, const void* seq_offsets,
                           long long total_tokens) {
  if (d.layout == HSTU_LAYOUT_NORMAL)
    return seq_offsets == nullptr && total_tokens == (long long)d.batch * d.max_seqlen;
  return seq_offsets != nullptr;
}

// The key side differs from the queries (own offsets or a KV cache).
static bool key_side(const hstu_fwd_desc& d) { return d.is_delta_qk || d.page_size; }

// rab goes through the tensor core (S accumulates the rab tile times a diagonal operand of
// c = 1/alpha) when that kernel variant exists for the call and c is a finite, normal value
// of the input type; its 16-bit pattern is the diagonal. Otherwise the epilogue adds rab.
static void set_rab_mode(FwdParams& p, const hstu_fwd_desc& d, bool is_mask) {
  p.rab_mma = 0;
  p.rab_ident = 0;
  const int elem = d.dtype == HSTU_FP8_E4M3 ? 2 : (d.dtype == HSTU_BF16 ? 1 : 0);
  if (!p.rab || d.dtype == HSTU_F32 ||
      !hstu::rab_mma_dim(d.head_dim, elem, is_mask ? 2 : 1, key_side(d) ? 1 : 0))
    return;
  if (!(p.alpha != 0.0f) || !std::isfinite(p.alpha)) return;
  const float c = 1.0f / p.alpha;
  float back;
  uint16_t bits;
  if (d.dtype == HSTU_BF16) {
    const __nv_bfloat16 b = __float2bfloat16_rn(c);
    back = __bfloat162float(b);
    memcpy(&bits, &b, 2);
  } else {
    const __half h = __float2half_rn(c);
    back = __half2float(h);
    memcpy(&bits, &h, 2);
  }
  if (!std::isfinite(back) || std::fabs(back) < (d.dtype == HSTU_BF16 ? 1.17549435e-38f
                                                                      : 6.103515625e-05f))
    return;
  p.rab_mma = 1;
  p.rab_ident = bits;
}

// Bound on the keys of a sequence, and the S of rab and of a custom mask.
static int key_bound(const hstu_fwd_desc& d) {
  return key_side(d) && d.max_seqlen_k > 0 ? d.max_seqlen_k : d.max_seqlen;
}

static hstu_status validate_desc(const hstu_fwd_desc* d) {
  if (!d) return HSTU_ERR_INVALID_ARG;
  if (d->reserved) return HSTU_ERR_INVALID_ARG;
  if (d->descale < HSTU_DESCALE_CAST || d->descale > HSTU_DESCALE_BLOCK ||
      (d->descale != HSTU_DESCALE_CAST && d->dtype != HSTU_FP8_E4M3))
    return HSTU_ERR_INVALID_ARG;
  // flags are 0 or 1
  for (int f : {d->is_delta_qk, d->index_is_int64, d->has_rab, d->has_num_context,
                d->has_num_targets})
    if (f != 0 && f != 1) return HSTU_ERR_INVALID_ARG;
  if (d->page_size != 0 && d->page_size != 32 && d->page_size != 128 && d->page_size != 256)
    return HSTU_ERR_INVALID_ARG;  // Inputs and Outputs table: page_size in {32, 128, 256}
  if (d->max_seqlen_k < 0 || d->max_seqlen_k > hstu::kMaxMTiles * hstu::kTileM ||
      (!key_side(*d) && d->max_seqlen_k != 0))
    return HSTU_ERR_INVALID_ARG;
  if (key_side(*d) && d->layout != HSTU_LAYOUT_JAGGED) return HSTU_ERR_UNSUPPORTED;
  if (d->layout != HSTU_LAYOUT_JAGGED && d->layout != HSTU_LAYOUT_NORMAL)
    return HSTU_ERR_INVALID_ARG;
  if (d->rab_heads != 0 && d->rab_heads != 1 && d->rab_heads != d->num_heads_q)
    return HSTU_ERR_INVALID_ARG;
  if (d->dtype != HSTU_F32 && d->dtype != HSTU_F16 && d->dtype != HSTU_BF16 &&
      d->dtype != HSTU_FP8_E4M3)
    return HSTU_ERR_INVALID_ARG;
  if (d->batch < 0 || d->batch > (1 << 20)) return HSTU_ERR_INVALID_ARG;
  if (d->num_heads_q < 0 || d->num_heads_kv < 1) return HSTU_ERR_INVALID_ARG;
  if (d->num_heads_q % d->num_heads_kv != 0) return HSTU_ERR_INVALID_ARG;
  if (d->head_dim < 1) return HSTU_ERR_INVALID_ARG;
  if (d->max_seqlen < 1 || d->max_seqlen > hstu::kMaxMTiles * hstu::kTileM)
    return HSTU_ERR_INVALID_ARG;
  if (d->target_group_size < 0 || d->watchdog_ms < 0) return HSTU_ERR_INVALID_ARG;
  if (d->mask_type == HSTU_MASK_UPPER) return HSTU_ERR_UNSUPPORTED;  // "currently not supported"
  if (d->mask_type != HSTU_MASK_CAUSAL && d->mask_type != HSTU_MASK_NONE &&
      d->mask_type != HSTU_MASK_CUSTOM)
    return HSTU_ERR_INVALID_ARG;
  if (d->mask_type == HSTU_MASK_CUSTOM) {
    // the mask replaces the built-in one (no context / target counts); it streams through
    // the rab path, so rab and a custom mask together are not built
    if (d->has_num_context || d->has_num_targets || (d->rab_heads && !d->has_rab))
      return HSTU_ERR_INVALID_ARG;
    // with rab: one ring slot holds a rab and a mask tile (head dims up to 128)
    if (d->has_rab && d->dtype != HSTU_F32 &&
        (!hstu::tc_supported_dim(d->head_dim) || d->head_dim > 128))
      return HSTU_ERR_UNSUPPORTED;
    if (d->dtype != HSTU_F32 && key_bound(*d) % 8 != 0) return HSTU_ERR_UNSUPPORTED;
  }
  if (d->dtype == HSTU_FP8_E4M3) {
    // FP8 E4M3 inputs: head dims up to 128; bf16 rab or a bf16 custom mask (one of them)
    // without a key side
    if (!hstu::tc_supported_dim(d->head_dim) || d->head_dim > 128) return HSTU_ERR_UNSUPPORTED;
    if (d->mask_type == HSTU_MASK_CUSTOM && (d->has_rab || key_side(*d)))
      return HSTU_ERR_UNSUPPORTED;
    if (d->has_rab && (key_side(*d) || key_bound(*d) % 8 != 0)) return HSTU_ERR_UNSUPPORTED;
  } else if (d->dtype == HSTU_F32) {
    if (d->head_dim > 256) return HSTU_ERR_UNSUPPORTED;
  } else {
    if (!hstu::tc_supported_dim(d->head_dim)) return HSTU_ERR_UNSUPPORTED;
    if (d->has_rab && key_bound(*d) % 8 != 0) return HSTU_ERR_UNSUPPORTED;
    // head dims above 256 (the 512 kernel): built-in masks only, no rab or key side
    if (d->head_dim > 256 && (d->has_rab || d->mask_type == HSTU_MASK_CUSTOM || key_side(*d)))
      return HSTU_ERR_UNSUPPORTED;
  }
  return HSTU_OK;
}

hstu_status hstu_fwd_create(const hstu_fwd_desc* desc, hstu_fwd_plan** plan) {
  if (!plan) return HSTU_ERR_INVALID_ARG;
  *plan = nullptr;
  hstu_status st = validate_desc(desc);
  if (st != HSTU_OK) return st;
  hstu_fwd_plan* P = new hstu_fwd_plan();
  memset(P, 0, sizeof(*P));
  P->desc = *desc;
  P->timeout_ns = (long long)(desc->watchdog_ms > 0 ? desc->watchdog_ms : 1000) * 1000000ll;
  // Watchdog test mode (tensor-core plans): the kernel's K producer signals nothing, so a
  // pipeline wait runs out after watchdog_ms and the run reports HSTU_ERR_TIMEOUT.
  const char* stall = getenv("HSTU_TEST_STALL");
  P->test_stall = stall && stall[0] == 'k' && stall[1] == 0 ? 1 : 0;
  P->tensor_cores = desc->dtype != HSTU_F32;
  cudaError_t e = cudaGetDevice(&P->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, P->device);
  if (e == cudaSuccess) {
    if (P->tensor_cores) {
      int major = 0, minor = 0;
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, P->device);
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, P->device);
      if (major != 10 || minor != 3 || !encode_fn()) {
        delete P;
        return HSTU_ERR_UNSUPPORTED;
      }
      // kernel variant: 0 no rab, 1 rab, 2 custom mask (streamed like rab)
      e = hstu::tc_prepare(desc->head_dim,
                           desc->dtype == HSTU_FP8_E4M3 ? 2 : (desc->dtype == HSTU_BF16 ? 1 : 0),
                           desc->mask_type == HSTU_MASK_CUSTOM ? (desc->has_rab ? 3 : 2)
                                                                : (desc->has_rab ? 1 : 0),
                           key_side(*desc) ? 1 : 0, desc->descale);
      P->grid = P->num_sms;
    } else {
      e = hstu::simt_prepare();
      P->grid = P->num_sms * (desc->head_dim <= 64 ? 4 : (desc->head_dim <= 128 ? 2 : 1));
    }
  }
  const size_t mtiles = (size_t)hstu::ceil_div(desc->max_seqlen, hstu::kTileM);
  const size_t entries = (size_t)(desc->batch > 0 ? desc->batch : 1) * mtiles;
  P->work_cap = entries;
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&P->done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&P->aux, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaMalloc(&P->d_work, 2 * entries * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMalloc(&P->d_count, 8 * sizeof(int));
  if (e == cudaSuccess) {
    P->d_err = P->d_count + 1;
    e = cudaMemsetAsync(P->d_count, 0, 8 * sizeof(int), P->aux);
  }
#if HSTU_TRACE
  if (e == cudaSuccess && P->tensor_cores)
    e = cudaMalloc(&P->d_trace, hstu::trace::kBufferWords * sizeof(unsigned long long));
  if (e == cudaSuccess && P->d_trace)
    e = cudaMemsetAsync(P->d_trace, 0, hstu::trace::kBufferWords * sizeof(unsigned long long),
                        P->aux);
#endif
  // the workspace is zeroed before any run can be enqueued on another stream
  if (e == cudaSuccess) e = cudaStreamSynchronize(P->aux);
  if (e == cudaSuccess) e = cudaEventRecord(P->done, P->aux);  // "no run yet" is complete
  if (e != cudaSuccess) {
    cudaFree(P->d_work);
    cudaFree(P->d_count);
    cudaFree(P->d_trace);
    if (P->done) cudaEventDestroy(P->done);
    if (P->aux) cudaStreamDestroy(P->aux);
    delete P;
    return HSTU_ERR_CUDA;
  }
  *plan = P;
  return HSTU_OK;
}

static bool encode3d(CUtensorMap* m, CUtensorMapDataType ty, const void* base, uint64_t d0,
                     uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1,
                     uint32_t b2, CUtensorMapSwizzle swz) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, ty, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool encode4d(CUtensorMap* m, CUtensorMapDataType ty, const void* base,
                     const uint64_t (&dims)[4], const uint64_t (&strides)[3],
                     const uint32_t (&box)[4], CUtensorMapSwizzle swz) {
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
  const cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, ty, 4, const_cast<void*>(base), d, st, b, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps: q and out over T rows, k and v over Tk rows (at least one row is mapped: a
// call without new k/v rows never loads them), rab [planes, Sk, Sk], and the KV cache
// [num_pages, 2, page_size, Nk, D] as 4-D (D, Nk, page_size, 2 * num_pages).
static hstu_status make_maps(hstu_fwd_plan* P, const void* q, const void* k, const void* v,
                             const void* rab, const void* out, long long T, long long Tk,
                             const void* cache, long long num_pages, const void* mask) {
  const void* ptrs[7] = {q, k, v, rab, out, cache, mask};
  if (P->maps_valid && P->map_T == T && P->map_Tk == Tk && P->map_pages == num_pages &&
      memcmp(ptrs, P->map_ptrs, sizeof(ptrs)) == 0)
    return HSTU_OK;
  const hstu_fwd_desc& d = P->desc;
  const bool fp8 = d.dtype == HSTU_FP8_E4M3;
  // q, k, v and the cache: E4M3 bytes (FP8 plans) or 16-bit; out is 16-bit (bf16 for FP8)
  const CUtensorMapDataType ty = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : d.dtype == HSTU_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapDataType oty = d.dtype == HSTU_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t eb = fp8 ? 1 : 2;
  const int swb = hstu::tc_swizzle_bytes(d.head_dim, (int)eb);
  const CUtensorMapSwizzle swz = swb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : swb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
  const uint32_t epc = (uint32_t)(swb / eb);
  const uint32_t oc = (uint32_t)hstu::tc_out_box_cols(d.head_dim);
  const uint64_t D = (uint64_t)d.head_dim, Nq = (uint64_t)d.num_heads_q,
                 Nk = (uint64_t)d.num_heads_kv;
  bool ok = encode3d(&P->maps.q, ty, q, D, Nq, (uint64_t)T, D * eb, Nq * D * eb, epc, 1,
                     hstu::kTileM, swz) &&
            encode3d(&P->maps.k, ty, k ? k : (cache ? cache : q), D, Nk, (uint64_t)(Tk > 0 ? Tk : 1),
                     D * eb, Nk * D * eb, epc, 1, hstu::kTileN, swz) &&
            encode3d(&P->maps.v, ty, v ? v : (cache ? cache : q), D, Nk, (uint64_t)(Tk > 0 ? Tk : 1),
                     D * eb, Nk * D * eb, epc, 1, (uint32_t)hstu::tc_v_box_rows(d.head_dim), swz) &&
            encode3d(&P->maps.out, oty, out, D, Nq, (uint64_t)T, D * 2, Nq * D * 2, oc, 1, 32,
                     oc * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                     : oc * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                     : oc * 2 == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                    : CU_TENSOR_MAP_SWIZZLE_NONE);
  if (ok && rab) {
    const uint64_t S = (uint64_t)key_bound(d);
    // rab of FP8 plans is bf16
    ok = encode3d(&P->maps.rab, fp8 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : ty, rab, S, S, (uint64_t)d.batch * (d.rab_heads == 1 ? 1 : Nq),
                  S * 2, S * S * 2, 64,
                  hstu::tc_rab_box_rows(), 1, CU_TENSOR_MAP_SWIZZLE_128B);
  } else if (ok) {
    P->maps.rab = P->maps.q;  // unused by the kernel
  }
  if (ok && mask) {  // a custom mask beside rab: [B * Nq, S, S] like a rab of Nq planes
    const uint64_t S = (uint64_t)key_bound(d);
    ok = encode3d(&P->maps.mask, ty, mask, S, S, (uint64_t)d.batch * Nq, S * 2, S * S * 2, 64,
                  hstu::tc_rab_box_rows(), 1, CU_TENSOR_MAP_SWIZZLE_128B);
  } else if (ok) {
    P->maps.mask = P->maps.q;  // unused by the kernel
  }
  if (ok && cache) {
    const uint64_t ps = (uint64_t)d.page_size;
    const uint64_t dims[4] = {D, Nk, ps, 2 * (uint64_t)num_pages};
    const uint64_t strides[3] = {D * eb, Nk * D * eb, ps * Nk * D * eb};
    const uint32_t box[4] = {epc, 1, (uint32_t)(ps < 128 ? ps : 128), 1};
    ok = encode4d(&P->maps.cache, ty, cache, dims, strides, box, swz);
  } else if (ok) {
    P->maps.cache = P->maps.q;  // unused by the kernel
  }
  if (!ok) {
    P->maps_valid = false;
    return HSTU_ERR_INVALID_ARG;
  }
  memcpy(P->map_ptrs, ptrs, sizeof(ptrs));
  P->map_T = T;
  P->map_Tk = Tk;
  P->map_pages = num_pages;
  P->maps_valid = true;
  return HSTU_OK;
}

// The key-side arguments a plan needs: none (kv NULL) for a plain plan; seq_offsets_k with
// is_delta_qk; the cache and its page table with page_size.
static bool kv_args_ok(const hstu_fwd_desc& d, const hstu_fwd_kv* kv) {
  if (!key_side(d)) return kv == nullptr;
  if (!kv) return false;
  if (d.is_delta_qk) {
    if (!kv->seq_offsets_k || kv->total_tokens_k < 0 || kv->total_tokens_k > 0x7fffffffll)
      return false;
  } else if (kv->seq_offsets_k) {
    return false;
  }
  if (d.page_size) {
    if (!kv->kv_cache || !kv->page_offsets || !kv->page_ids || !kv->last_page_len ||
        kv->num_pages < 1 || kv->num_pages > (1ll << 30) || !aligned16(kv->kv_cache))
      return false;
  } else if (kv->kv_cache || kv->page_offsets || kv->page_ids || kv->last_page_len) {
    return false;
  }
  return true;
}

// One forward. `rab` carries the relative attention bias, or the custom mask when
// is_mask (plans of mask_type CUSTOM). `kv` describes the key side (NULL: the keys are the
// query rows of k and v).
static hstu_status run_impl(hstu_fwd_plan* P, const void* q, const void* k, const void* v,
                            const void* seq_offsets, const hstu_fwd_kv* kv, const void* rab,
                            bool is_mask, const void* num_context, const void* num_targets,
                            long long total_tokens, float alpha, float silu_scale, void* out,
                            void* stream, const hstu_fwd_descale* ds = nullptr,
                            const void* mask_with_rab = nullptr) {
  const hstu_fwd_desc& d = P->desc;
  // a CUSTOM plan with has_rab takes both (rab in `rab`, the mask in mask_with_rab)
  const bool both = d.mask_type == HSTU_MASK_CUSTOM && d.has_rab;
  if (both && is_mask) return HSTU_ERR_INVALID_ARG;
  if (!both && mask_with_rab) return HSTU_ERR_INVALID_ARG;
  if (both && !mask_with_rab && d.batch > 0 && d.num_heads_q > 0 && total_tokens > 0)
    return HSTU_ERR_INVALID_ARG;
  if (d.descale != HSTU_DESCALE_CAST) {  // factor arrays: present, fp32-aligned
    if (!ds || !ds->q || !ds->k || !ds->v) return HSTU_ERR_INVALID_ARG;
    for (const float* f : {ds->q, ds->k, ds->v})
      if (reinterpret_cast<uintptr_t>(f) % 4 != 0) return HSTU_ERR_INVALID_ARG;
  }
  if (total_tokens < 0 || total_tokens > 0x7fffffffll) return HSTU_ERR_INVALID_ARG;
  if (!kv_args_ok(d, kv)) return HSTU_ERR_INVALID_ARG;
  if (d.batch == 0 || d.num_heads_q == 0 || total_tokens == 0) return HSTU_OK;  // empty input
  const long long Tk = d.is_delta_qk ? kv->total_tokens_k : total_tokens;
  const bool kv_rows = Tk > 0;  // k and v are read only when there are new rows
  if (!q || !out || !layout_args_ok(d, seq_offsets, total_tokens) ||
      (kv_rows && (!k || !v)))
    return HSTU_ERR_INVALID_ARG;
  if ((rab != nullptr) != (is_mask || d.has_rab != 0)) return HSTU_ERR_INVALID_ARG;
  if (mask_with_rab && !aligned16(mask_with_rab)) return HSTU_ERR_INVALID_ARG;
  if ((num_context != nullptr) != (d.has_num_context != 0)) return HSTU_ERR_INVALID_ARG;
  if ((num_targets != nullptr) != (d.has_num_targets != 0)) return HSTU_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (rab && !aligned16(rab)))
    return HSTU_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != P->device) return HSTU_ERR_INVALID_ARG;
  const void* cache = d.page_size ? kv->kv_cache : nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  FwdParams p = {};
  p.q = q;
  p.k = k;
  p.v = v;
  p.rab = rab;
  p.out = out;
  p.seq_offsets = seq_offsets;
  p.num_context = num_context;
  p.num_targets = num_targets;
  const int b = P->parity;
  P->parity ^= 1;
  p.work = P->d_work + b * P->work_cap;
  p.work_count = P->d_count + 4 * b;
  p.next_item = P->d_count + 4 * b + 2;
  p.err = P->d_err;
  p.total_tokens = total_tokens;
  p.timeout_ns = P->timeout_ns;
  p.index64 = d.index_is_int64 ? 1 : 0;
  p.B = d.batch;
  p.Nq = d.num_heads_q;
  p.Nk = d.num_heads_kv;
  p.D = d.head_dim;
  p.S = key_bound(d);
  p.Sq = d.max_seqlen;
  p.total_tokens_k = Tk;
  if (d.is_delta_qk) p.seq_offsets_k = kv->seq_offsets_k;
  if (d.page_size) {
    p.kv_cache = kv->kv_cache;
    p.page_offsets = kv->page_offsets;
    p.page_ids = kv->page_ids;
    p.last_page_len = kv->last_page_len;
    p.num_pages = kv->num_pages;
    p.page_size = d.page_size;
  }
  p.mask_type = is_mask ? hstu::kMaskNone : d.mask_type;  // a custom mask: every key a candidate
  p.g = d.mask_type == HSTU_MASK_CAUSAL ? d.target_group_size : 0;
  p.dense = d.layout == HSTU_LAYOUT_NORMAL ? 1 : 0;
  p.rab_bcast = d.rab_heads == 1 ? 1 : 0;
  p.rab_is_mask = is_mask ? 1 : 0;
  p.mask = mask_with_rab;
  if (both) p.mask_type = hstu::kMaskNone;  // the mask decides: every key a candidate
  p.alpha = alpha;
  p.silu_scale = silu_scale;
  p.fp8 = d.dtype == HSTU_FP8_E4M3 ? 1 : 0;
  p.test_stall = P->test_stall;
  if (d.descale != HSTU_DESCALE_CAST) {
    p.q_ds = ds->q;
    p.k_ds = ds->k;
    p.v_ds = ds->v;
    p.ds_mode = d.descale;
    p.ds_qb = hstu::ceil_div(d.max_seqlen, hstu::kTileM);
    p.ds_kb = hstu::ceil_div(key_bound(d), hstu::kTileN);
  }
  set_rab_mode(p, d, is_mask);
#if HSTU_TRACE
  // run r of the plan records into launch slot r % kSlots
  if (P->d_trace) p.trace = P->d_trace + (size_t)(P->runs % hstu::trace::kSlots) * hstu::trace::kSlotWords;
  ++P->runs;
#endif
  if (p.fp8) p.silu_scale = silu_scale / hstu::kP8Scale;  // the kernel's P carries kP8Scale

  if (P->tensor_cores) {
    hstu_status ms = make_maps(P, q, k, v, rab, out, total_tokens, Tk, cache,
                               d.page_size ? kv->num_pages : 0, mask_with_rab);
    if (ms != HSTU_OK) return ms;
  }
  if (hstu::launch_build_worklist(p, P->d_work + b * P->work_cap, P->d_count + 4 * b,
                                  hstu::kTileM, st, true) != cudaSuccess)
    return HSTU_ERR_CUDA;
  cudaError_t e = P->tensor_cores
                      ? hstu::launch_fwd_tc(p, P->maps, d.dtype == HSTU_BF16, P->grid, st, true)
                      : hstu::launch_fwd_simt(p, P->grid, st, true);
  if (e == cudaSuccess) e = cudaEventRecord(P->done, st);
  return e == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

hstu_status hstu_fwd_run(hstu_fwd_plan* P, const void* q, const void* k, const void* v,
                         const void* seq_offsets, const void* rab, const void* num_context,
                         const void* num_targets, long long total_tokens, float alpha,
                         float silu_scale, void* out, void* stream) {
  if (!P || P->desc.mask_type == HSTU_MASK_CUSTOM || P->desc.descale != HSTU_DESCALE_CAST)
    return HSTU_ERR_INVALID_ARG;
  return run_impl(P, q, k, v, seq_offsets, nullptr, rab, false, num_context, num_targets,
                  total_tokens, alpha, silu_scale, out, stream);
}

hstu_status hstu_fwd_run_args(hstu_fwd_plan* P, const hstu_fwd_args* a, void* stream) {
  if (!P || !a) return HSTU_ERR_INVALID_ARG;
  const hstu_fwd_desc& d = P->desc;
  const bool custom = d.mask_type == HSTU_MASK_CUSTOM;
  if (!custom && a->mask) return HSTU_ERR_INVALID_ARG;
  if (custom && (a->num_context || a->num_targets)) return HSTU_ERR_INVALID_ARG;
  if (d.descale == HSTU_DESCALE_CAST && a->descale) return HSTU_ERR_INVALID_ARG;
  if (custom && !d.has_rab) {  // the mask streams where rab would
    if (a->rab) return HSTU_ERR_INVALID_ARG;
    if (!a->mask && d.batch > 0 && d.num_heads_q > 0 && a->total_tokens > 0)
      return HSTU_ERR_INVALID_ARG;
    return run_impl(P, a->q, a->k, a->v, a->seq_offsets, a->kv, a->mask, true, nullptr, nullptr,
                    a->total_tokens, a->alpha, a->silu_scale, a->out, stream, a->descale);
  }
  return run_impl(P, a->q, a->k, a->v, a->seq_offsets, a->kv, a->rab, false, a->num_context,
                  a->num_targets, a->total_tokens, a->alpha, a->silu_scale, a->out, stream,
                  a->descale, custom ? a->mask : nullptr);
}

hstu_status hstu_fwd_run_fp8(hstu_fwd_plan* P, const void* q, const void* k, const void* v,
                             const void* seq_offsets, const hstu_fwd_kv* kv, const void* rab,
                             const void* num_context, const void* num_targets,
                             const hstu_fwd_descale* descale, long long total_tokens,
                             float alpha, float silu_scale, void* out, void* stream) {
  // (a CUSTOM plan takes its mask through hstu_fwd_run_masked or hstu_fwd_run_args)
  if (!P || P->desc.dtype != HSTU_FP8_E4M3 || P->desc.mask_type == HSTU_MASK_CUSTOM)
    return HSTU_ERR_INVALID_ARG;
  return run_impl(P, q, k, v, seq_offsets, kv, rab, false, num_context, num_targets,
                  total_tokens, alpha, silu_scale, out, stream, descale);
}

hstu_status hstu_fwd_run_kv(hstu_fwd_plan* P, const void* q, const void* k, const void* v,
                            const void* seq_offsets, const hstu_fwd_kv* kv,
                            const void* rab_or_mask, const void* num_context,
                            const void* num_targets, long long total_tokens, float alpha,
                            float silu_scale, void* out, void* stream) {
  if (!P || P->desc.descale != HSTU_DESCALE_CAST) return HSTU_ERR_INVALID_ARG;
  const bool custom = P->desc.mask_type == HSTU_MASK_CUSTOM;
  if (custom && (num_context || num_targets)) return HSTU_ERR_INVALID_ARG;
  if (custom && !rab_or_mask && P->desc.batch > 0 && P->desc.num_heads_q > 0 && total_tokens > 0)
    return HSTU_ERR_INVALID_ARG;
  return run_impl(P, q, k, v, seq_offsets, kv, rab_or_mask, custom, num_context, num_targets,
                  total_tokens, alpha, silu_scale, out, stream);
}

hstu_status hstu_fwd_run_masked(hstu_fwd_plan* P, const void* q, const void* k, const void* v,
                                const void* seq_offsets, const void* mask,
                                long long total_tokens, float alpha, float silu_scale,
                                void* out, void* stream) {
  if (!P || P->desc.mask_type != HSTU_MASK_CUSTOM) return HSTU_ERR_INVALID_ARG;
  if (!mask && P->desc.batch > 0 && P->desc.num_heads_q > 0 && total_tokens > 0)
    return HSTU_ERR_INVALID_ARG;
  return run_impl(P, q, k, v, seq_offsets, nullptr, mask, true, nullptr, nullptr, total_tokens,
                  alpha, silu_scale, out, stream);
}

hstu_status hstu_fwd_destroy(hstu_fwd_plan* P) {
  if (!P) return HSTU_OK;
  // the plan's last run (and with it every earlier one: runs of a plan never overlap)
  // has finished with the workspace
  cudaEventSynchronize(P->done);
  cudaStreamSynchronize(P->aux);
  cudaFree(P->d_work);
  cudaFree(P->d_count);
  cudaFree(P->d_trace);
  cudaEventDestroy(P->done);
  cudaStreamDestroy(P->aux);
  delete P;
  return HSTU_OK;
}

hstu_status hstu_fwd_trace_read(hstu_fwd_plan* P, void* host, long long bytes) {
  if (!P || !host || bytes < 0) return HSTU_ERR_INVALID_ARG;
  if (!P->d_trace) return HSTU_ERR_UNSUPPORTED;  // not a tracing build, or an fp32 plan
#if HSTU_TRACE
  const size_t all = hstu::trace::kBufferWords * sizeof(unsigned long long);
  const size_t n = (size_t)bytes < all ? (size_t)bytes : all;
  if (cudaEventSynchronize(P->done) != cudaSuccess ||
      cudaMemcpyAsync(host, P->d_trace, n, cudaMemcpyDeviceToHost, P->aux) != cudaSuccess ||
      cudaMemsetAsync(P->d_trace, 0, all, P->aux) != cudaSuccess ||
      cudaStreamSynchronize(P->aux) != cudaSuccess)
    return HSTU_ERR_CUDA;
#endif
  return HSTU_OK;
}

hstu_status hstu_fwd_get_error(hstu_fwd_plan* P, int* device_error) {
  if (!P || !device_error) return HSTU_ERR_INVALID_ARG;
  // wait for the plan's last run only (not the whole device), then read and clear the
  // word on the plan's private stream
  if (cudaEventSynchronize(P->done) != cudaSuccess) return HSTU_ERR_CUDA;
  int w = 0;
  if (cudaMemcpyAsync(&w, P->d_err, sizeof(int), cudaMemcpyDeviceToHost, P->aux) != cudaSuccess ||
      cudaMemsetAsync(P->d_err, 0, sizeof(int), P->aux) != cudaSuccess ||
      cudaStreamSynchronize(P->aux) != cudaSuccess)
    return HSTU_ERR_CUDA;
  *device_error = w;
  if (w == HSTU_DEVERR_TIMEOUT) return HSTU_ERR_TIMEOUT;
  if (w != HSTU_DEVERR_NONE) return HSTU_ERR_DEVICE_CHECK;
  return HSTU_OK;
}

hstu_status hstu_fwd_launches_per_run(const hstu_fwd_plan* P, int* launches) {
  if (!P || !launches) return HSTU_ERR_INVALID_ARG;
  *launches = 2;  // work-list builder + forward kernel
  return HSTU_OK;
}

hstu_status hstu_fwd_count_pairs(const hstu_fwd_desc* d, const void* seq_offsets_host,
                                 const void* num_context_host, const void* num_targets_host,
                                 long long* pairs) {
  if (!d || !pairs) return HSTU_ERR_INVALID_ARG;
  const bool normal = d->layout == HSTU_LAYOUT_NORMAL;
  if (normal ? seq_offsets_host != nullptr : (d->batch > 0 && !seq_offsets_host))
    return HSTU_ERR_INVALID_ARG;
  if (d->mask_type != HSTU_MASK_CAUSAL && d->mask_type != HSTU_MASK_NONE &&
      d->mask_type != HSTU_MASK_CUSTOM)
    return HSTU_ERR_UNSUPPORTED;
  const int is64 = d->index_is_int64 ? 1 : 0;
  const int g = d->mask_type == HSTU_MASK_CAUSAL ? d->target_group_size : 0;
  // a custom mask makes every (i, j) of the sequence a computed pair
  const int mt = d->mask_type == HSTU_MASK_CUSTOM ? HSTU_MASK_NONE : d->mask_type;
  long long total = 0;
  for (int b = 0; b < d->batch; ++b) {
    const long long t0 = normal ? (long long)b * d->max_seqlen
                                : hstu::load_index(seq_offsets_host, b, is64);
    const long long L =
        (normal ? (long long)(b + 1) * d->max_seqlen : hstu::load_index(seq_offsets_host, b + 1, is64)) - t0;
    if (L < 0 || L > d->max_seqlen) return HSTU_ERR_INVALID_ARG;
    const long long nc = num_context_host ? hstu::load_index(num_context_host, b, is64) : 0;
    const long long nt = num_targets_host ? hstu::load_index(num_targets_host, b, is64) : 0;
    const hstu::SeqGeom s = hstu::make_geom((int)L, nc, nt, g, mt);
    long long c = 0;
    for (int i = 0; i < (int)L; ++i) {
      const hstu::RowRange r = hstu::row_range(s, i, mt);
      c += r.hist_end;
      if (r.grp_hi >= r.grp_lo) c += r.grp_hi - r.grp_lo + 1;
    }
    total += c * d->num_heads_q;
  }
  *pairs = total;
  return HSTU_OK;
}

hstu_status hstu_fwd_count_pairs_kv(const hstu_fwd_desc* d, const void* seq_offsets_host,
                                    const void* seq_offsets_k_host,
                                    const void* page_offsets_host,
                                    const void* last_page_len_host,
                                    const void* num_context_host, const void* num_targets_host,
                                    long long* pairs) {
  if (!d || !pairs) return HSTU_ERR_INVALID_ARG;
  if (d->batch > 0 && !seq_offsets_host) return HSTU_ERR_INVALID_ARG;
  if (d->layout != HSTU_LAYOUT_JAGGED) return HSTU_ERR_UNSUPPORTED;
  if ((page_offsets_host != nullptr) != (last_page_len_host != nullptr)) return HSTU_ERR_INVALID_ARG;
  if (page_offsets_host && d->page_size <= 0) return HSTU_ERR_INVALID_ARG;
  if (d->mask_type != HSTU_MASK_CAUSAL && d->mask_type != HSTU_MASK_NONE &&
      d->mask_type != HSTU_MASK_CUSTOM)
    return HSTU_ERR_UNSUPPORTED;
  const int is64 = d->index_is_int64 ? 1 : 0;
  const int g = d->mask_type == HSTU_MASK_CAUSAL ? d->target_group_size : 0;
  const int mt = d->mask_type == HSTU_MASK_CUSTOM ? HSTU_MASK_NONE : d->mask_type;
  const long long Sk = key_bound(*d);
  long long total = 0;
  for (int b = 0; b < d->batch; ++b) {
    const long long Lq = hstu::load_index(seq_offsets_host, b + 1, is64) -
                         hstu::load_index(seq_offsets_host, b, is64);
    long long Lk = seq_offsets_k_host ? hstu::load_index(seq_offsets_k_host, b + 1, is64) -
                                            hstu::load_index(seq_offsets_k_host, b, is64)
                                      : Lq;
    if (page_offsets_host) {
      const long long pages = hstu::load_index(page_offsets_host, b + 1, is64) -
                              hstu::load_index(page_offsets_host, b, is64);
      if (pages < 0) return HSTU_ERR_INVALID_ARG;
      if (pages > 0) {
        const long long last = hstu::load_index(last_page_len_host, b, is64);
        if (last < 1 || last > d->page_size || pages > Sk) return HSTU_ERR_INVALID_ARG;
        Lk += (pages - 1) * d->page_size + last;
      }
    }
    if (Lq < 0 || Lq > d->max_seqlen || Lk < Lq || Lk > Sk) return HSTU_ERR_INVALID_ARG;
    const long long nc = num_context_host ? hstu::load_index(num_context_host, b, is64) : 0;
    const long long nt = num_targets_host ? hstu::load_index(num_targets_host, b, is64) : 0;
    const hstu::SeqGeom s = hstu::make_geom((int)Lk, nc, nt, g, mt);
    long long c = 0;
    for (int i = (int)(Lk - Lq); i < (int)Lk; ++i) {
      const hstu::RowRange r = hstu::row_range(s, i, mt);
      c += r.hist_end;
      if (r.grp_hi >= r.grp_lo) c += r.grp_hi - r.grp_lo + 1;
    }
    total += c * d->num_heads_q;
  }
  *pairs = total;
  return HSTU_OK;
}

// ---------------------------------------------------------------------------
// Entry point that allocates nothing: the work list lives in this file-scope device
// array instead of a plan's cudaMalloc'ed workspace. Layout (32-bit words):
// [0] entry count, [1] device error word, [2] scheduling counter, [64 ..] work-list entries.
// ---------------------------------------------------------------------------
#define HSTU_NOALLOC_MAX_ENTRIES 16384  // (sequence, 128-row query tile) pairs
static __device__ __align__(256) uint32_t g_noalloc_scratch[64 + HSTU_NOALLOC_MAX_ENTRIES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
uint32_t* g_noalloc_ptr[kMaxDevices];   // device address of the array, per device
int g_noalloc_sms[kMaxDevices];
uint32_t g_noalloc_prepared[kMaxDevices];  // kernel variants configured (bit per variant)

// Per-device set-up, run by the first call on each device with that device current.
cudaError_t noalloc_setup(int dev, const hstu_fwd_desc& d, uint32_t** scratch, int* sms) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&g_noalloc_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<uint32_t*>(ptr);
  }
  // shared-memory opt-in of the kernel variant this descriptor uses
  int bit = 0;
  if (d.dtype != HSTU_F32) {
    const int kd = hstu::tc_kernel_dim(d.head_dim);
    const int di = kd == 32 ? 0 : kd == 64 ? 1 : kd == 128 ? 2 : kd == 256 ? 3 : 4;
    bit = 1 + di * 4 + (d.dtype == HSTU_BF16 ? 2 : 0) + (d.has_rab ? 1 : 0);
  }
  if (!(g_noalloc_prepared[dev] & (1u << bit))) {
    cudaError_t e = d.dtype == HSTU_F32
                        ? hstu::simt_prepare()
                        : hstu::tc_prepare(d.head_dim, d.dtype == HSTU_BF16, d.has_rab ? 1 : 0, 0);
    if (e != cudaSuccess) return e;
    g_noalloc_prepared[dev] |= 1u << bit;
  }
  *scratch = g_noalloc_ptr[dev];
  *sms = g_noalloc_sms[dev];
  return cudaSuccess;
}
}  // namespace

hstu_status hstu_fwd_run_noalloc(const hstu_fwd_desc* desc, const void* q, const void* k,
                                 const void* v, const void* seq_offsets, const void* rab,
                                 const void* num_context, const void* num_targets,
                                 long long total_tokens, float alpha, float silu_scale, void* out,
                                 void* stream) {
  hstu_status st = validate_desc(desc);
  if (st != HSTU_OK) return st;
  const hstu_fwd_desc& d = *desc;
  if (total_tokens < 0 || total_tokens > 0x7fffffffll) return HSTU_ERR_INVALID_ARG;
  if (d.batch == 0 || d.num_heads_q == 0 || total_tokens == 0) return HSTU_OK;  // empty input
  if ((long long)d.batch * hstu::ceil_div(d.max_seqlen, hstu::kTileM) > HSTU_NOALLOC_MAX_ENTRIES)
    return HSTU_ERR_UNSUPPORTED;  // work list larger than the static scratch array
  if (d.mask_type == HSTU_MASK_CUSTOM) return HSTU_ERR_UNSUPPORTED;  // hstu_fwd_run_masked only
  if (d.dtype == HSTU_FP8_E4M3) return HSTU_ERR_UNSUPPORTED;          // plans only
  if (key_side(d)) return HSTU_ERR_UNSUPPORTED;                       // hstu_fwd_run_kv only
  if (!q || !k || !v || !out || !layout_args_ok(d, seq_offsets, total_tokens))
    return HSTU_ERR_INVALID_ARG;
  if ((rab != nullptr) != (d.has_rab != 0)) return HSTU_ERR_INVALID_ARG;
  if ((num_context != nullptr) != (d.has_num_context != 0)) return HSTU_ERR_INVALID_ARG;
  if ((num_targets != nullptr) != (d.has_num_targets != 0)) return HSTU_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (rab && !aligned16(rab)))
    return HSTU_ERR_INVALID_ARG;
  const bool tc = d.dtype != HSTU_F32;
  if (tc && !encode_fn()) return HSTU_ERR_UNSUPPORTED;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HSTU_ERR_CUDA;
  if (tc) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return HSTU_ERR_UNSUPPORTED;
  }
  uint32_t* scratch = nullptr;
  int sms = 0;
  if (noalloc_setup(dev, d, &scratch, &sms) != cudaSuccess) return HSTU_ERR_CUDA;
  cudaStream_t st_ = static_cast<cudaStream_t>(stream);

  FwdParams p = {};
  p.q = q;
  p.k = k;
  p.v = v;
  p.rab = rab;
  p.out = out;
  p.seq_offsets = seq_offsets;
  p.num_context = num_context;
  p.num_targets = num_targets;
  p.work = scratch + 64;
  p.work_count = reinterpret_cast<int*>(scratch);
  p.err = reinterpret_cast<int*>(scratch) + 1;
  p.next_item = reinterpret_cast<int*>(scratch) + 2;
  p.total_tokens = total_tokens;
  p.timeout_ns = (long long)(d.watchdog_ms > 0 ? d.watchdog_ms : 1000) * 1000000ll;
  p.index64 = d.index_is_int64 ? 1 : 0;
  p.B = d.batch;
  p.Nq = d.num_heads_q;
  p.Nk = d.num_heads_kv;
  p.D = d.head_dim;
  p.S = d.max_seqlen;
  p.Sq = d.max_seqlen;
  p.mask_type = d.mask_type;
  p.g = d.mask_type == HSTU_MASK_CAUSAL ? d.target_group_size : 0;
  p.dense = d.layout == HSTU_LAYOUT_NORMAL ? 1 : 0;
  p.rab_bcast = d.rab_heads == 1 ? 1 : 0;
  p.alpha = alpha;
  p.silu_scale = silu_scale;
  set_rab_mode(p, d, false);

  TcMaps maps;
  if (tc) {
    const CUtensorMapDataType ty =
        d.dtype == HSTU_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int swb = hstu::tc_swizzle_bytes(d.head_dim, 2);
    const CUtensorMapSwizzle swz = swb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : swb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    const uint32_t epc = (uint32_t)(swb / 2);
    const uint32_t oc = (uint32_t)hstu::tc_out_box_cols(d.head_dim);
    const uint64_t D = (uint64_t)d.head_dim, Nq = (uint64_t)d.num_heads_q,
                   Nk = (uint64_t)d.num_heads_kv, T = (uint64_t)total_tokens;
    bool ok = encode3d(&maps.q, ty, q, D, Nq, T, D * 2, Nq * D * 2, epc, 1, hstu::kTileM, swz) &&
              encode3d(&maps.k, ty, k, D, Nk, T, D * 2, Nk * D * 2, epc, 1, hstu::kTileN, swz) &&
              encode3d(&maps.v, ty, v, D, Nk, T, D * 2, Nk * D * 2, epc, 1,
                       (uint32_t)hstu::tc_v_box_rows(d.head_dim), swz) &&
              encode3d(&maps.out, ty, out, D, Nq, T, D * 2, Nq * D * 2, oc, 1, 32,
                       oc * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                       : oc * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                       : oc * 2 == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                      : CU_TENSOR_MAP_SWIZZLE_NONE);
    if (ok && rab) {
      const uint64_t S = (uint64_t)d.max_seqlen;
      ok = encode3d(&maps.rab, ty, rab, S, S, (uint64_t)d.batch * (d.rab_heads == 1 ? 1 : Nq),
                    S * 2, S * S * 2, 64,
                    hstu::tc_rab_box_rows(), 1, CU_TENSOR_MAP_SWIZZLE_128B);
    } else if (ok) {
      maps.rab = maps.q;  // unused by the kernel
    }
    maps.cache = maps.q;  // no KV cache on this entry point
    if (!ok) return HSTU_ERR_INVALID_ARG;
  }
  // the error word keeps the previous call's value: clear it (the count is rewritten)
  if (cudaMemsetAsync(p.err, 0, sizeof(int), st_) != cudaSuccess) return HSTU_ERR_CUDA;
  // one work list: the build must not overlap a previous call (no programmatic launch)
  if (hstu::launch_build_worklist(p, scratch + 64, reinterpret_cast<int*>(scratch),
                                  hstu::kTileM, st_, false) != cudaSuccess)
    return HSTU_ERR_CUDA;
  const int grid = tc ? sms : sms * (d.head_dim <= 64 ? 4 : (d.head_dim <= 128 ? 2 : 1));
  cudaError_t e = tc ? hstu::launch_fwd_tc(p, maps, d.dtype == HSTU_BF16, grid, st_, true)
                     : hstu::launch_fwd_simt(p, grid, st_, true);
  return e == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

}  // extern "C"
