// Launch helpers of the tensor-core forward kernel, shared by the translation units that
// instantiate its variants (fwd_tc.cu: no rab / rab; fwd_tc_mask.cu: custom mask;
// fwd_tc_kv.cu and fwd_tc_kv_mask.cu: the same with a key side of its own).
#pragma once
#include "fwd_tc.cuh"

namespace hstu {
namespace tc {

template <int D, bool BF16, int RAB, bool MASK, bool KV, int F8 = 0>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(fwd_tc_kernel<D, BF16, RAB, MASK, KV, F8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, RAB, F8>::SMEM_BYTES);
}

template <int D, bool BF16, int RAB, bool MASK, bool KV, int F8 = 0>
cudaError_t launch_one(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t stream,
                       bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg<D, RAB, F8>::THREADS);
  cfg.dynamicSmemBytes = Cfg<D, RAB, F8>::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_tc_kernel<D, BF16, RAB, MASK, KV, F8>, m.q, m.k, m.v, m.rab, m.out,
                            m.cache, m.mask, p);
}

// Prepare (shared-memory opt-in) or launch one variant, chosen by head dim and type.
template <bool BF16, int RAB, bool MASK, bool KV>
cudaError_t dispatch_dim(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                         bool pdl, bool prepare) {
  switch (tc_kernel_dim(p.D)) {
    case 32: return prepare ? prepare_one<32, BF16, RAB, MASK, KV>() : launch_one<32, BF16, RAB, MASK, KV>(p, m, grid, st, pdl);
    case 64: return prepare ? prepare_one<64, BF16, RAB, MASK, KV>() : launch_one<64, BF16, RAB, MASK, KV>(p, m, grid, st, pdl);
    case 128: return prepare ? prepare_one<128, BF16, RAB, MASK, KV>() : launch_one<128, BF16, RAB, MASK, KV>(p, m, grid, st, pdl);
    case 256: return prepare ? prepare_one<256, BF16, RAB, MASK, KV>() : launch_one<256, BF16, RAB, MASK, KV>(p, m, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int RAB, bool MASK, bool KV>
cudaError_t dispatch_type(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                          cudaStream_t st, bool pdl, bool prepare) {
  return bf16 ? dispatch_dim<true, RAB, MASK, KV>(p, m, grid, st, pdl, prepare)
              : dispatch_dim<false, RAB, MASK, KV>(p, m, grid, st, pdl, prepare);
}

// Head dims above 256 (fwd_tc_wide.cu): the 512 kernel, no rab, mask tiles or key side.
cudaError_t dispatch_wide(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                          cudaStream_t st, bool pdl, bool prepare);

// rab added by the tensor core (fwd_tc_rab_mma.cu): head dims 32 and 64, no key side.
cudaError_t dispatch_rab_mma(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                             cudaStream_t st, bool pdl, bool prepare);

// Custom-mask variants (fwd_tc_mask.cu): prepare (shared-memory opt-in) or launch.
cudaError_t dispatch_mask(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                          cudaStream_t st, bool pdl, bool prepare);
// A custom mask together with rab (fwd_tc_mask_rab.cu; with a key side fwd_tc_kv_mask_rab.cu):
// head dims up to 128.
cudaError_t dispatch_mask_rab(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                              cudaStream_t st, bool pdl, bool prepare);
cudaError_t dispatch_kv_mask_rab(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                                 cudaStream_t st, bool pdl, bool prepare);

// FP8 E4M3 variants (fwd_tc_f8.cu): head dims up to 128, with or without a key side; with
// rab (fwd_tc_f8_rab.cu) or a custom mask (fwd_tc_f8_mask.cu) without a key side.
cudaError_t dispatch_f8(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st, bool pdl,
                        bool prepare);
cudaError_t dispatch_f8_rab(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                            bool pdl, bool prepare);
// FP8 with a custom mask (fwd_tc_f8_mask.cu): no key side, no rab
cudaError_t dispatch_f8_mask(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                             bool pdl, bool prepare);
// FP8 with descale factors (fwd_tc_f8_ds.cu; fwd_tc_f8_rab.cu with rab): F8 = 2 kernels
cudaError_t dispatch_f8_ds(const FwdParams& p, const TcMaps& m, int grid, cudaStream_t st,
                           bool pdl, bool prepare);

// Key-side variants (fwd_tc_kv.cu, fwd_tc_kv_mask.cu): own k/v offsets and / or a KV cache.
cudaError_t dispatch_kv(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                        cudaStream_t st, bool pdl, bool prepare);
cudaError_t dispatch_kv_mask(const FwdParams& p, const TcMaps& m, int bf16, int grid,
                             cudaStream_t st, bool pdl, bool prepare);

}  // namespace tc
}  // namespace hstu
