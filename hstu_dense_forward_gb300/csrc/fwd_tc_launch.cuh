// Launch helpers of the tensor-core forward kernel, shared by the translation units that
// instantiate its variants (fwd_tc.cu: no rab / rab; fwd_tc_mask.cu: custom mask).
#pragma once
#include "fwd_tc.cuh"

namespace hstu {
namespace tc {

template <int D, bool BF16, bool RAB, bool MASK>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(fwd_tc_kernel<D, BF16, RAB, MASK>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, RAB>::SMEM_BYTES);
}

template <int D, bool BF16, bool RAB, bool MASK>
cudaError_t launch_one(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t stream,
                       bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D, RAB>::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_tc_kernel<D, BF16, RAB, MASK>, m.q, m.k, m.v, m.rab, m.out,
                            m.cache, p);
}

// Custom-mask variants (fwd_tc_mask.cu): prepare (shared-memory opt-in) or launch.
cudaError_t dispatch_mask(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                          cudaStream_t st, bool pdl, bool prepare);

}  // namespace tc
}  // namespace hstu
