// FP8 E4M3 variants with a custom mask (mask_type 3): the bf16 mask tiles stream through
// the rab ring and the epilogue multiplies P by them in fp32 before its E4M3 rounding.
// Head dims up to 128, no key side, no rab; plain cast or descale factors.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

namespace {
template <int F8>
cudaError_t dim_mask(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st, bool pdl,
                     bool prepare) {
  switch (tc_kernel_dim(p.D)) {
    case 32: return prepare ? prepare_one<32, true, 1, true, false, F8>() : launch_one<32, true, 1, true, false, F8>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, true, 1, true, false, F8>() : launch_one<64, true, 1, true, false, F8>(p, m, grid, st, pdl);
    case 128: return prepare ? prepare_one<128, true, 1, true, false, F8>() : launch_one<128, true, 1, true, false, F8>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t dispatch_f8_mask(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                             bool pdl, bool prepare) {
  return p.ds_mode ? dim_mask<2>(p, m, grid, st, pdl, prepare)
                   : dim_mask<1>(p, m, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
