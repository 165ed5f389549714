// Custom-mask (mask_type 3) variants of the tensor-core forward kernel: the rab stream
// carries the mask tiles and the epilogue multiplies P by them after the SiLU.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

cudaError_t dispatch_mask(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                          cudaStream_t st, bool pdl, bool prepare) {
  return dispatch_type<true, true, false>(p, m, bf16, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
