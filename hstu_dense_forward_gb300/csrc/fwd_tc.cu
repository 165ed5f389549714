// Instantiations and launch of the tensor-core forward kernel: the plain variants here;
// the custom-mask variants (fwd_tc_mask.cu), the key-side variants (fwd_tc_kv.cu,
// fwd_tc_kv_mask.cu) and the FP8 variants (fwd_tc_f8.cu) are instantiated in translation
// units of their own.
#include "fwd_tc_launch.cuh"

namespace hstu {

namespace {

// A call with its own k/v offsets or a KV cache takes the key-side variants.
bool key_side(const FwdParams& p) { return p.seq_offsets_k != nullptr || p.page_offsets != nullptr; }

cudaError_t dispatch(const FwdParams& p, const TcMaps& m, int bf16, int grid, cudaStream_t st,
                     bool pdl, bool prepare) {
  if (p.fp8) return tc::dispatch_f8(p, m, grid, st, pdl, prepare);
  if (tc_kernel_dim(p.D) == 512) return tc::dispatch_wide(p, m, bf16, grid, st, pdl, prepare);
  if (key_side(p))
    return p.mask ? tc::dispatch_kv_mask_rab(p, m, bf16, grid, st, pdl, prepare)
           : p.rab_is_mask ? tc::dispatch_kv_mask(p, m, bf16, grid, st, pdl, prepare)
                           : tc::dispatch_kv(p, m, bf16, grid, st, pdl, prepare);
  if (p.rab_is_mask) return tc::dispatch_mask(p, m, bf16, grid, st, pdl, prepare);
  if (p.mask) return tc::dispatch_mask_rab(p, m, bf16, grid, st, pdl, prepare);
  if (p.rab && p.rab_mma) return tc::dispatch_rab_mma(p, m, bf16, grid, st, pdl, prepare);
  return p.rab ? tc::dispatch_type<1, false, false>(p, m, bf16, grid, st, pdl, prepare)
               : tc::dispatch_type<0, false, false>(p, m, bf16, grid, st, pdl, prepare);
}

}  // namespace

// Every multiple of 16 up to 512 runs on the kernel built for the next of 32, 64, 128, 256,
// 512: the tensor maps keep the true head dim (rows of D elements) with boxes of the
// kernel's, so TMA loads fill the extra columns of q, k and v with zeros (Q K^T is
// unchanged, the extra O columns are 0) and TMA stores clip them; direct stores skip them.
bool tc_supported_dim(int D) { return D % 16 == 0 && D >= 16 && D <= 512; }

int tc_kernel_dim(int D) {
  return D <= 32 ? 32 : (D <= 64 ? 64 : (D <= 128 ? 128 : (D <= 256 ? 256 : 512)));
}

int tc_swizzle_bytes(int D, int elem_bytes) {
  const int k = tc_kernel_dim(D);
  return k * elem_bytes >= 128 ? 128 : k * elem_bytes;
}

int tc_out_box_cols(int D) {  // a warpgroup's O staging box (head dims up to 128; the larger
                              // ones store O rows directly and never read this map)
  const int k = tc_kernel_dim(D);
  return k == 32 ? tc::Cfg<32, 0>::OC : k == 64 ? tc::Cfg<64, 0>::OC : k == 128 ? tc::Cfg<128, 0>::OC : 64;
}

int tc_rab_box_rows() { return tc::kRabBoxRows; }

int tc_v_box_rows(int D) { return tc_kernel_dim(D) == 512 ? tc::Cfg<512, 0, 0>::VROWS : kTileN; }

cudaError_t tc_prepare(int D, int elem, int rab, int kv, int ds) {
  FwdParams p = {};
  p.D = D;
  p.ds_mode = ds;  // (FP8: the plain-cast or the descaled kernels)
  p.fp8 = elem == 2 ? 1 : 0;
  const int bf16 = elem == 1 ? 1 : 0;
  p.rab = rab ? reinterpret_cast<const void*>(1) : nullptr;
  p.rab_is_mask = rab == 2 ? 1 : 0;
  p.mask = rab == 3 ? reinterpret_cast<const void*>(1) : nullptr;
  p.seq_offsets_k = kv ? reinterpret_cast<const void*>(1) : nullptr;  // selects the variant only
  TcMaps m = {};
  cudaError_t e = dispatch(p, m, bf16, 0, nullptr, false, true);
  if (e == cudaSuccess && rab_mma_dim(D, elem, rab, kv)) {
    p.rab_mma = 1;  // runs whose 1/alpha is finite in the input type take this variant
    e = dispatch(p, m, bf16, 0, nullptr, false, true);
  }
  return e;
}

bool rab_mma_dim(int D, int elem, int rab, int kv) {
  return rab == 1 && !kv && elem != 2 && tc_kernel_dim(D) <= 64;
}

cudaError_t launch_fwd_tc(const FwdParams& p, const TcMaps& maps, int bf16, int grid,
                          cudaStream_t stream, bool pdl) {
  return dispatch(p, maps, bf16, grid, stream, pdl, false);
}

}  // namespace hstu
