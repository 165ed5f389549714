// FP8 E4M3 variants of the tensor-core forward kernel (feature table, "FP8 quantization
// types"): q, k and v arrive as E4M3, both products run as tcgen05 kind::f8f6f4 with fp32
// accumulation (P rounded to E4M3 for the second), O is written as bf16. Head dims up to
// 128; with or without a key side. This unit holds the plain-cast kernels (F8 = 1); the
// kernels with descale factors (F8 = 2) are in fwd_tc_f8_ds.cu, those with bf16 rab (added
// by the epilogue) in fwd_tc_f8_rab.cu, those with a bf16 custom mask in fwd_tc_f8_mask.cu.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

namespace {
// (the 16-bit companion type of an FP8 kernel, out and rab, is bf16)
template <bool KV>
cudaError_t dispatch_f8_dim(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                            bool pdl, bool prepare) {
  switch (tc_kernel_dim(p.D)) {
    case 32: return prepare ? prepare_one<32, true, 0, false, KV, 1>() : launch_one<32, true, 0, false, KV, 1>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, true, 0, false, KV, 1>() : launch_one<64, true, 0, false, KV, 1>(p, m, grid, st, pdl);
    case 128: return prepare ? prepare_one<128, true, 0, false, KV, 1>() : launch_one<128, true, 0, false, KV, 1>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t dispatch_f8(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st, bool pdl,
                        bool prepare) {
  const bool kv = p.seq_offsets_k != nullptr || p.page_offsets != nullptr;
  if (p.rab && p.rab_is_mask)
    return kv ? cudaErrorInvalidValue : dispatch_f8_mask(p, m, grid, st, pdl, prepare);
  if (p.rab) return kv ? cudaErrorInvalidValue : dispatch_f8_rab(p, m, grid, st, pdl, prepare);
  if (p.ds_mode) return dispatch_f8_ds(p, m, grid, st, pdl, prepare);
  return kv ? dispatch_f8_dim<true>(p, m, grid, st, pdl, prepare)
            : dispatch_f8_dim<false>(p, m, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
