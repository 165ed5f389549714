// Key-side variants (own k/v offsets, KV cache) for a custom mask together with rab: each
// rab ring slot holds the rab tile and the mask tile of one key visit, both taken at the
// key positions of the item's queries. Head dims up to 128.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

namespace {
template <bool BF16>
cudaError_t one_type(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st, bool pdl,
                     bool prepare) {
  switch (tc_kernel_dim(p.D)) {
    case 32: return prepare ? prepare_one<32, BF16, 3, true, true>() : launch_one<32, BF16, 3, true, true>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, BF16, 3, true, true>() : launch_one<64, BF16, 3, true, true>(p, m, grid, st, pdl);
    case 128: return prepare ? prepare_one<128, BF16, 3, true, true>() : launch_one<128, BF16, 3, true, true>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t dispatch_kv_mask_rab(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                                 cudaStream_t st, bool pdl, bool prepare) {
  return bf16 ? one_type<true>(p, m, grid, st, pdl, prepare)
              : one_type<false>(p, m, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
