// Key-side variants of the tensor-core forward kernel (no rab / rab): the queries are the
// last tokens of longer key sequences whose keys are a paged cached history followed by
// new k/v rows with offsets of their own.
#include "fwd_tc_launch.cuh"

namespace hstu {
namespace tc {

cudaError_t dispatch_kv(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                        cudaStream_t st, bool pdl, bool prepare) {
  return p.rab ? dispatch_type<true, false, true>(p, m, bf16, grid, st, pdl, prepare)
               : dispatch_type<false, false, true>(p, m, bf16, grid, st, pdl, prepare);
}

}  // namespace tc
}  // namespace hstu
