// Instantiations and launch of the tensor-core forward kernel (the custom-mask variants
// are instantiated in fwd_tc_mask.cu, a translation unit of their own).
#include "fwd_tc_launch.cuh"

namespace hstu {

namespace {

template <int D, bool BF16, bool RAB>
cudaError_t prepare_one() {
  return tc::prepare_one<D, BF16, RAB, false>();
}

template <int D, bool BF16, bool RAB>
cudaError_t launch_one(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t stream,
                       bool pdl) {
  return tc::launch_one<D, BF16, RAB, false>(p, m, grid, stream, pdl);
}

template <bool BF16, bool RAB>
cudaError_t dispatch_d(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st, bool pdl,
                       bool prepare) {
  switch (p.D) {
    case 32: return prepare ? prepare_one<32, BF16, RAB>() : launch_one<32, BF16, RAB>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, BF16, RAB>() : launch_one<64, BF16, RAB>(p, m, grid, st, pdl);
    case 128: return prepare ? prepare_one<128, BF16, RAB>() : launch_one<128, BF16, RAB>(p, m, grid, st, pdl);
    case 256: return prepare ? prepare_one<256, BF16, RAB>() : launch_one<256, BF16, RAB>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t dispatch(const FwdParams& p, const TcMaps& m, int bf16, int grid, cudaStream_t st,
                     bool pdl, bool prepare) {
  if (p.rab_is_mask) return tc::dispatch_mask(p, m, bf16, grid, st, pdl, prepare);
  const bool rab = p.rab != nullptr;
  if (bf16) return rab ? dispatch_d<true, true>(p, m, grid, st, pdl, prepare)
                       : dispatch_d<true, false>(p, m, grid, st, pdl, prepare);
  return rab ? dispatch_d<false, true>(p, m, grid, st, pdl, prepare)
             : dispatch_d<false, false>(p, m, grid, st, pdl, prepare);
}

}  // namespace

bool tc_supported_dim(int D) { return D == 32 || D == 64 || D == 128 || D == 256; }

int tc_swizzle_bytes(int D) { return D * 2 >= 128 ? 128 : D * 2; }

int tc_out_box_cols(int D) { return D / tc::kEpiWG; }

cudaError_t tc_prepare(int D, int bf16, int rab) {
  FwdParams p = {};
  p.D = D;
  p.rab = rab ? reinterpret_cast<const void*>(1) : nullptr;
  p.rab_is_mask = rab == 2 ? 1 : 0;
  TcMaps m = {};
  return dispatch(p, m, bf16, 0, nullptr, false, true);
}

cudaError_t launch_fwd_tc(const FwdParams& p, const TcMaps& maps, int bf16, int grid,
                          cudaStream_t stream, bool pdl) {
  return dispatch(p, maps, bf16, grid, stream, pdl, false);
}

}  // namespace hstu
