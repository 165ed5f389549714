// FP8 E4M3 variants with descale factors (F8 = 2): the epilogue folds the q and k factors
// of each item (or, with per-block factors, of each key tile) into the SiLU argument's
// factor and the v factors into P or the output scale. Kept apart from the plain-cast
// kernels, which read no factors. Head dims up to 128, with or without a key side.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

namespace {
template <bool KV>
cudaError_t dim_ds(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st, bool pdl,
                   bool prepare) {
  switch (tc_kernel_dim(p.D)) {
    case 32: return prepare ? prepare_one<32, true, 0, false, KV, 2>() : launch_one<32, true, 0, false, KV, 2>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, true, 0, false, KV, 2>() : launch_one<64, true, 0, false, KV, 2>(p, m, grid, st, pdl);
    case 128: return prepare ? prepare_one<128, true, 0, false, KV, 2>() : launch_one<128, true, 0, false, KV, 2>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t dispatch_f8_ds(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                           bool pdl, bool prepare) {
  const bool kv = p.seq_offsets_k != nullptr || p.page_offsets != nullptr;
  return kv ? dim_ds<true>(p, m, grid, st, pdl, prepare) : dim_ds<false>(p, m, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
