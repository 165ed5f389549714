// fp32 HSTU forward on CUDA cores (FFMA, fp32 accumulation, SiLU through expf).
//
// "RecOps Running Case Documentation", feature table: floating-point types
// FP32, FP16 and BF16 are all supported by the operator. fp32 keeps full
// precision here: a TF32 tensor-core product (10-bit mantissa) cannot stay within
// 1e-5 of the fp64 result relative to max|O|, so this path uses FFMA.
//
// One CTA (256 threads) takes one half (64 query rows) of a 128-row work item of
// the shared work list, for one query head, and walks the key/value tiles of 64
// rows the mask leaves reachable:
//   S = Q_tile * K_tile^T (4x4 outputs per thread), x = alpha*S (+ rab),
//   P = silu(x) masked -> shared memory, O += P * V_tile (registers),
// then writes silu_scale * O for the rows inside the sequence.
#include "../../include/hstu_fwd.h"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace hstu {

namespace {

constexpr int BM = 64;       // query rows per CTA
constexpr int BN = 64;       // key rows per step
constexpr int kThreads = 256;
constexpr int kMaxD = 256;
constexpr int kMaxU = kMaxD / 16;  // output columns per thread / 16

__global__ void __launch_bounds__(kThreads) fwd_simt_f32_kernel(const FwdParams p) {
  ptx::grid_dependency_wait();  // the work list comes from the previous launch
  ptx::grid_dependents_launch();  // after the wait: see the work-list builder
  extern __shared__ float sm[];
  const int D = p.D;
  const int ldk = D + 1;  // padded rows: threads of one warp read different K rows
  float* Qs = sm;                  // [BM][D]
  float* Ks = Qs + BM * D;         // [BN][D+1]
  float* Vs = Ks + BN * ldk;       // [BN][D]
  float* Ps = Vs + BN * D;         // [BM][BN+1]
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

  const float* q = static_cast<const float*>(p.q);
  const float* k = static_cast<const float*>(p.k);
  const float* v = static_cast<const float*>(p.v);
  const float* rab = static_cast<const float*>(p.rab);
  float* out = static_cast<float*>(p.out);
  const int G = p.Nq / p.Nk;
  const long long total = (long long)(*p.work_count) * p.Nq * 2;

  for (long long w = blockIdx.x; w < total; w += gridDim.x) {
    const int half = (int)(w & 1);
    const long long it = w >> 1;
    const int h = (int)(it % p.Nq);
    const uint32_t e = p.work[it / p.Nq];
    const int b = item_b(e);
    const SeqKV kv = seq_kv(p, b);
    const long long t0 = kv.tq;
    const int Lq = (int)kv.Lq, L = (int)kv.Lk, hist = (int)kv.hist;
    const int off = L - Lq;  // key position of query row 0
    const int m0 = item_mt(e) * kTileM + half * BM;
    if (m0 >= Lq) continue;
    const long long nc = p.num_context ? load_index(p.num_context, b, p.index64) : 0;
    const long long nt = p.num_targets ? load_index(p.num_targets, b, p.index64) : 0;
    const SeqGeom s = make_geom(L, nc, nt, p.g, p.mask_type);
    const int kv_end = kv_end_for_rows(s, off + m0, BM, p.mask_type);
    const int hk = h / G;
    const float* cache = static_cast<const float*>(p.kv_cache);

    __syncthreads();  // previous item finished with the shared tiles
    for (int x = threadIdx.x; x < BM * D; x += kThreads) {
      const int r = x / D, d = x - r * D;
      Qs[x] = (m0 + r < Lq) ? q[((t0 + m0 + r) * p.Nq + h) * D + d] : 0.f;
    }
    float acc[4][kMaxU];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int u = 0; u < kMaxU; ++u) acc[a][u] = 0.f;

    for (int n0 = 0; n0 < kv_end; n0 += BN) {
      __syncthreads();  // previous step finished with Ks/Vs/Ps
      for (int x = threadIdx.x; x < BN * D; x += kThreads) {
        const int r = x / D, d = x - r * D;
        const int pos = n0 + r;  // key position
        float kx = 0.f, vx = 0.f;
        if (pos < hist) {  // cached history: page row pos % page_size
          const long long page =
              load_index(p.page_ids, kv.po + pos / p.page_size, p.index64);
          const long long g =
              ((page * 2 * p.page_size + pos % p.page_size) * p.Nk + hk) * D + d;
          kx = cache[g];
          vx = cache[g + (long long)p.page_size * p.Nk * D];
        } else if (pos < L) {  // new rows
          const long long g = ((kv.tk + pos - hist) * p.Nk + hk) * D + d;
          kx = k[g];
          vx = v[g];
        }
        Ks[r * ldk + d] = kx;
        Vs[x] = vx;
      }
      __syncthreads();
      // S for rows ty + 16a, columns tx + 16c
      float sc[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[a][c] = 0.f;
      for (int d = 0; d < D; ++d) {
        float qa[4], kb[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) qa[a] = Qs[(ty + 16 * a) * D + d];
#pragma unroll
        for (int c = 0; c < 4; ++c) kb[c] = Ks[(tx + 16 * c) * ldk + d];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) sc[a][c] = fmaf(qa[a], kb[c], sc[a][c]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int r = ty + 16 * a;
        const int i = off + m0 + r;  // key position of the query row
        const RowRange rr = row_range(s, i, p.mask_type);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int j = n0 + tx + 16 * c;
          float x = p.alpha * sc[a][c];
          const bool ok = (m0 + r < Lq) && (j < L) && valid_in_range(rr, j);
          const float t = (rab != nullptr && ok) ? rab[(rab_plane(p, b, h) * p.S + i) * p.S + j]
                                                 : 0.f;
          if (!p.rab_is_mask) x += t;  // relative attention bias before the SiLU
          float pv = x / (1.0f + expf(-x));
          if (p.rab_is_mask) pv *= t;  // custom mask after it
          if (p.mask != nullptr && ok)  // (a custom mask given together with rab)
            pv *= static_cast<const float*>(p.mask)[(((long long)b * p.Nq + h) * p.S + i) * p.S + j];
          Ps[r * (BN + 1) + tx + 16 * c] = ok ? pv : 0.f;
        }
      }
      __syncthreads();
      // O rows ty + 16a, columns tx + 16u
      for (int j = 0; j < BN; ++j) {
        float pa[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) pa[a] = Ps[(ty + 16 * a) * (BN + 1) + j];
#pragma unroll
        for (int u = 0; u < kMaxU; ++u) {
          const int d = tx + 16 * u;
          if (d < D) {
            const float vv = Vs[j * D + d];
#pragma unroll
            for (int a = 0; a < 4; ++a) acc[a][u] = fmaf(pa[a], vv, acc[a][u]);
          }
        }
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = m0 + ty + 16 * a;
      if (i >= Lq) continue;
#pragma unroll
      for (int u = 0; u < kMaxU; ++u) {
        const int d = tx + 16 * u;
        if (d < D) out[((t0 + i) * p.Nq + h) * D + d] = p.silu_scale * acc[a][u];
      }
    }
  }
}

}  // namespace

size_t simt_smem_bytes(int D) {
  return sizeof(float) * ((size_t)BM * D + (size_t)BN * (D + 1) + (size_t)BN * D +
                          (size_t)BM * (BN + 1));
}

cudaError_t simt_prepare() {
  return cudaFuncSetAttribute(fwd_simt_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)simt_smem_bytes(kMaxD));
}

cudaError_t launch_fwd_simt(const FwdParams& p, int grid, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = simt_smem_bytes(p.D);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_simt_f32_kernel, p);
}

}  // namespace hstu
