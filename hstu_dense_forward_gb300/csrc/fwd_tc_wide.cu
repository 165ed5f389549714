// Head dims 272 to 512 (Inputs and Outputs table: v's D up to 512): the kernel built for
// 512 computes S over every column of q and k and O over one half (256 columns) of v per
// work item, so each 128-row tile is two items. bf16 / fp16; causal or no mask with
// context and target counts; no rab, custom mask or key side.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

cudaError_t dispatch_wide(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                          cudaStream_t st, bool pdl, bool prepare) {
  if (bf16)
    return prepare ? prepare_one<512, true, 0, false, false>()
                   : launch_one<512, true, 0, false, false>(p, m, grid, st, pdl);
  return prepare ? prepare_one<512, false, 0, false, false>()
                 : launch_one<512, false, 0, false, false>(p, m, grid, st, pdl);
}

}  // namespace tc
}  // namespace hstu
