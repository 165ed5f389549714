// Key-side variants of the tensor-core forward kernel with a custom mask (mask_type 3).
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

cudaError_t dispatch_kv_mask(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                             cudaStream_t st, bool pdl, bool prepare) {
  return dispatch_type<true, true, true>(p, m, bf16, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
