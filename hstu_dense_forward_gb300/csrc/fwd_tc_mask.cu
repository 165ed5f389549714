// Custom-mask (mask_type 3) variants of the tensor-core forward kernel: the rab stream
// carries the mask tiles and the epilogue multiplies P by them after the SiLU.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

namespace {
template <bool BF16>
cudaError_t dispatch_mask_d(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                            bool pdl, bool prepare) {
  switch (p.D) {
    case 32: return prepare ? prepare_one<32, BF16, true, true>() : launch_one<32, BF16, true, true>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, BF16, true, true>() : launch_one<64, BF16, true, true>(p, m, grid, st, pdl);
    case 128: return prepare ? prepare_one<128, BF16, true, true>() : launch_one<128, BF16, true, true>(p, m, grid, st, pdl);
    case 256: return prepare ? prepare_one<256, BF16, true, true>() : launch_one<256, BF16, true, true>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t dispatch_mask(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                          cudaStream_t st, bool pdl, bool prepare) {
  return bf16 ? dispatch_mask_d<true>(p, m, grid, st, pdl, prepare)
              : dispatch_mask_d<false>(p, m, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
