// FP8 E4M3 variants of the tensor-core forward kernel (feature table, "FP8 quantization
// types: cast"): q, k and v arrive as E4M3, both products run as tcgen05 kind::f8f6f4 with
// fp32 accumulation (P rounded to E4M3 for the second), O is written as bf16. Head dims
// 32, 64, 128; no rab or custom mask; with or without a key side.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

namespace {
template <bool KV>
cudaError_t dispatch_f8_dim(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                            bool pdl, bool prepare) {
  switch (tc_kernel_dim(p.D)) {
    case 32: return prepare ? prepare_one<32, false, false, false, KV, true>() : launch_one<32, false, false, false, KV, true>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, false, false, false, KV, true>() : launch_one<64, false, false, false, KV, true>(p, m, grid, st, pdl);
    case 128: return prepare ? prepare_one<128, false, false, false, KV, true>() : launch_one<128, false, false, false, KV, true>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t dispatch_f8(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st, bool pdl,
                        bool prepare) {
  const bool kv = p.seq_offsets_k != nullptr || p.page_offsets != nullptr;
  return kv ? dispatch_f8_dim<true>(p, m, grid, st, pdl, prepare)
            : dispatch_f8_dim<false>(p, m, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
