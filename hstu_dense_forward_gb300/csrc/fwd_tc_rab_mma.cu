// Variants of the tensor-core forward kernel that add rab with the tensor core (head dims
// 32 and 64, bf16 / fp16, no key side): the score products accumulate the rab tile times a
// diagonal operand of 1/alpha, and the epilogue is that of the plain kernel.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

namespace {
template <bool BF16>
cudaError_t one_type(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st, bool pdl,
                     bool prepare) {
  switch (tc_kernel_dim(p.D)) {
    case 32: return prepare ? prepare_one<32, BF16, 2, false, false>() : launch_one<32, BF16, 2, false, false>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, BF16, 2, false, false>() : launch_one<64, BF16, 2, false, false>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t dispatch_rab_mma(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                             cudaStream_t st, bool pdl, bool prepare) {
  return bf16 ? one_type<true>(p, m, grid, st, pdl, prepare)
              : one_type<false>(p, m, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
