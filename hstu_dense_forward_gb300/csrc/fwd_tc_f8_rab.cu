// FP8 E4M3 variants with rab: the bf16 rab tiles stream through the rab ring and the
// epilogue adds rab / 2 to the fp32 SiLU argument, as in the 16-bit kernels. Head dims up
// to 128, no key side; plain cast or descale factors.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

namespace {
template <int F8>
cudaError_t dim_rab(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st, bool pdl,
                    bool prepare) {
  switch (tc_kernel_dim(p.D)) {
    case 32: return prepare ? prepare_one<32, true, 1, false, false, F8>() : launch_one<32, true, 1, false, false, F8>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, true, 1, false, false, F8>() : launch_one<64, true, 1, false, false, F8>(p, m, grid, st, pdl);
    case 128: return prepare ? prepare_one<128, true, 1, false, false, F8>() : launch_one<128, true, 1, false, false, F8>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

// plain cast (F8 = 1) or descale factors (F8 = 2)
cudaError_t dispatch_f8_rab(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                            bool pdl, bool prepare) {
  return p.ds_mode ? dim_rab<2>(p, m, grid, st, pdl, prepare)
                   : dim_rab<1>(p, m, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
