// bf16 / fp16 HSTU forward on the 5th-generation tensor cores (sm_103a).
//
// Operation ("RecOps Running Case Documentation", feature table and Inputs and
// Outputs table): per sequence, query head and 128-row query tile,
//   S = Q K^T, x = alpha*S (+ rab), P = silu(x) masked, O = P V, out = silu_scale*O.
// HSTU has no softmax, so there is no running max or rescaling: O is a plain sum
// over key tiles and key tiles the mask removes entirely are never visited.
//
// CTA layout (persistent, one CTA per SM, 320 threads):
//   warps 0-7  epilogue: two warpgroups; each thread owns one query row (TMEM lane)
//              and half of the 128 key columns of every S tile. It reads S from
//              TMEM, applies alpha, rab, SiLU (as h + h*tanh(h), h = x/2, one MUFU
//              op per element) and the mask, and writes P (bf16/fp16) back to TMEM.
//              At the end of a work item it reads O, scales, converts and stores.
//   warp 8     producer: TMA loads of the Q tile, the K/V ring and the rab ring.
//   warp 9     MMA issuer (one thread) and TMEM owner:
//                S(t)  = Q K(t)^T   tcgen05.mma  A = Q (smem), B = K (smem, K-major)
//                O    += P(t) V(t)  tcgen05.mma  A = P (TMEM),  B = V (smem, MN-major)
//              S(t+1) is issued before O += P(t) V(t), so the tensor cores compute the
//              next scores while the epilogue works on the current ones.
// TMEM (512 columns): S double buffer at columns 0 and 128, O at 256 (D columns),
// P double buffer after O (D <= 128) or written over the S buffer it came from
// (D = 256, where O takes all remaining columns).
//
// Every mbarrier wait is bounded (FwdParams::timeout_ns): on expiry the CTA
// records HSTU_DEVERR_TIMEOUT, all roles leave their loops, the MMA queue is
// drained, TMEM is freed and the kernel returns.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "../../include/hstu_fwd.h"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace hstu {
namespace tc {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr uint32_t kTmemCols = 512;

template <int D, bool RAB>
struct Cfg {
  static_assert(D == 32 || D == 64 || D == 128 || D == 256, "head_dim");
  static constexpr int SWB = (D * 2 >= 128) ? 128 : D * 2;  // bytes per swizzled row
  static constexpr uint32_t SWZ = (SWB == 128) ? 2u : (SWB == 64 ? 4u : 6u);
  static constexpr int EPC = SWB / 2;          // elements per column block
  static constexpr int NCB = D / EPC;          // column blocks per tile row
  static constexpr int CB_BYTES = 128 * SWB;   // one column block of a 128-row tile
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int RAB_BYTES = 128 * 128 * 2;
  static constexpr int NQ = (D <= 64) ? 2 : ((D == 128 && !RAB) ? 2 : 1);
  static constexpr int NS = (D <= 64) ? 4 : (D == 128 ? 2 : 1);
  static constexpr int NR = RAB ? ((D == 256) ? 1 : 2) : 0;
  static constexpr bool P_ALIAS = (D == 256);
  // TMEM columns
  static constexpr uint32_t S_COL0 = 0, O_COL = 256;
  static constexpr uint32_t P_COL0 = O_COL + D;  // used when !P_ALIAS
  // shared memory map (offsets from a 1024-aligned base)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
  static constexpr int OFF_R = OFF_V + NS * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_R + NR * RAB_BYTES;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int SMEM_USED = OFF_BAR + BAR_BYTES;
  // keep one CTA per SM (TMEM is allocated whole)
  static constexpr int SMEM_BYTES = (SMEM_USED + 1024 < 120 * 1024) ? 120 * 1024 : SMEM_USED + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(!P_ALIAS || D == 256, "alias only when O fills the spare TMEM");
  static_assert(P_ALIAS || P_COL0 + 128 <= kTmemCols, "TMEM map");
};

// Barrier block layout (uint64 each).
struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t r_full[2], r_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_full, o_empty, drain;
  uint32_t tmem_base;
  volatile int abort;
};
static_assert(sizeof(Bars) <= 1024, "barrier block");

// One work item, decoded identically by every role.
struct Item {
  int b, h, hk, L, m0, n_kv;
  long long t0;
  SeqGeom geom;
};

__device__ __forceinline__ bool decode_item(const FwdParams& p, long long idx, Item& it) {
  const uint32_t e = p.work[idx / p.Nq];
  it.h = (int)(idx % p.Nq);
  it.hk = it.h / (p.Nq / p.Nk);
  it.b = item_b(e);
  it.m0 = item_mt(e) * kTileM;
  it.t0 = load_index(p.seq_offsets, it.b, p.index64);
  it.L = (int)(load_index(p.seq_offsets, it.b + 1, p.index64) - it.t0);
  const long long nc = p.num_context ? load_index(p.num_context, it.b, p.index64) : 0;
  const long long nt = p.num_targets ? load_index(p.num_targets, it.b, p.index64) : 0;
  it.geom = make_geom(it.L, nc, nt, p.g, p.mask_type);
  it.n_kv = ceil_div(kv_end_for_rows(it.geom, it.m0, kTileM, p.mask_type), kTileN);
  return true;
}

// k-th item of this CTA: snake order over the (heaviest-first) list, so that
// every CTA gets a mix of long and short items.
__device__ __forceinline__ long long item_index(int k) {
  const long long G = gridDim.x;
  const long long c = (k & 1) ? (G - 1 - blockIdx.x) : blockIdx.x;
  return (long long)k * G + c;
}

// Bounded wait. Returns false when this CTA is aborting (own timeout or another role's).
__device__ __forceinline__ bool wait_bar(Bars* bars, uint64_t* bar, uint32_t parity,
                                         const FwdParams& p) {
  const uint32_t a = ptx::smem_u32(bar);
  if (ptx::mbar_try_wait(a, parity)) return true;
  const uint64_t start = ptx::globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(a, parity)) return true;
    if ((n & 31u) == 0) {
      if (bars->abort) return false;
      if ((long long)(ptx::globaltimer_ns() - start) > p.timeout_ns) {
        bars->abort = 1;
        atomicCAS(p.err, HSTU_DEVERR_NONE, HSTU_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait by every lane of a warp, with a warp-uniform result: the lanes leave
// together, so the .sync.aligned tcgen05 loads/stores that follow stay converged.
__device__ __forceinline__ bool warp_wait(Bars* bars, uint64_t* bar, uint32_t parity,
                                          const FwdParams& p) {
  const bool ok = wait_bar(bars, bar, parity, p);
  return __all_sync(0xffffffffu, ok);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(v);
  } else {
    __half2 v = *reinterpret_cast<__half2*>(&w);
    return __half22float2(v);
  }
}

// ------------------------------------------------------------------ producer
template <int D, bool RAB>
__device__ void producer(const FwdParams& p, Bars* bars, uint8_t* smem, const CUtensorMap* tq,
                         const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tr,
                         long long total) {
  using C = Cfg<D, RAB>;
  uint32_t q_it = 0, kv_it = 0, r_it = 0;
  const uint32_t sbase = ptx::smem_u32(smem);
  for (int k = 0;; ++k) {
    const long long idx = item_index(k);
    if (idx >= total) break;
    Item it;
    decode_item(p, idx, it);
    // Q tile
    {
      const int s = q_it % C::NQ;
      if (!wait_bar(bars, &bars->q_empty[s], ((q_it / C::NQ) & 1) ^ 1, p)) return;
      const uint32_t full = ptx::smem_u32(&bars->q_full[s]);
      ptx::mbar_arrive_expect_tx(full, C::TILE_BYTES);
      const uint32_t dst = sbase + C::OFF_Q + s * C::TILE_BYTES;
#pragma unroll
      for (int cb = 0; cb < C::NCB; ++cb)
        ptx::tma_load_3d(dst + cb * C::CB_BYTES, tq, full, cb * C::EPC, it.h,
                         (int)(it.t0 + it.m0));
      ++q_it;
    }
    for (int j = 0; j < it.n_kv; ++j) {
      const int s = kv_it % C::NS;
      const uint32_t ph = ((kv_it / C::NS) & 1) ^ 1;
      const int row = (int)(it.t0 + j * kTileN);
      if (!wait_bar(bars, &bars->k_empty[s], ph, p)) return;
      {
        const uint32_t full = ptx::smem_u32(&bars->k_full[s]);
        ptx::mbar_arrive_expect_tx(full, C::TILE_BYTES);
        const uint32_t dst = sbase + C::OFF_K + s * C::TILE_BYTES;
#pragma unroll
        for (int cb = 0; cb < C::NCB; ++cb)
          ptx::tma_load_3d(dst + cb * C::CB_BYTES, tk, full, cb * C::EPC, it.hk, row);
      }
      if constexpr (RAB) {
        const int rs = r_it % C::NR;
        if (!wait_bar(bars, &bars->r_empty[rs], ((r_it / C::NR) & 1) ^ 1, p)) return;
        const uint32_t full = ptx::smem_u32(&bars->r_full[rs]);
        ptx::mbar_arrive_expect_tx(full, C::RAB_BYTES);
        const uint32_t dst = sbase + C::OFF_R + rs * C::RAB_BYTES;
        const int plane = it.b * p.Nq + it.h;
        ptx::tma_load_3d(dst, tr, full, j * kTileN, it.m0, plane);
        ptx::tma_load_3d(dst + C::RAB_BYTES / 2, tr, full, j * kTileN + 64, it.m0, plane);
        ++r_it;
      }
      if (!wait_bar(bars, &bars->v_empty[s], ph, p)) return;
      {
        const uint32_t full = ptx::smem_u32(&bars->v_full[s]);
        ptx::mbar_arrive_expect_tx(full, C::TILE_BYTES);
        const uint32_t dst = sbase + C::OFF_V + s * C::TILE_BYTES;
#pragma unroll
        for (int cb = 0; cb < C::NCB; ++cb)
          ptx::tma_load_3d(dst + cb * C::CB_BYTES, tv, full, cb * C::EPC, it.hk, row);
      }
      ++kv_it;
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
template <int D, bool BF16, bool RAB>
__device__ void mma_issuer(const FwdParams& p, Bars* bars, uint8_t* smem, uint32_t tmem,
                           long long total) {
  using C = Cfg<D, RAB>;
  constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16 ? 1u : 0u, 128, kTileN, 0);
  constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16 ? 1u : 0u, 128, D, 1);
  const uint32_t sbase = ptx::smem_u32(smem);
  uint32_t q_it = 0, k_it = 0, v_it = 0, t = 0, u = 0;

  // S(t) = Q K^T into S buffer t % 2
  auto issue_s = [&](int qs) -> bool {
    const uint32_t sb = t & 1;
    if (C::P_ALIAS && t >= 2) {  // P(t-2) lives in this S buffer until PV(t-2) is done
      if (!wait_bar(bars, &bars->pv_done[sb], ((t >> 1) & 1) ^ 1, p)) return false;
    }
    const int ks = k_it % C::NS;
    if (!wait_bar(bars, &bars->k_full[ks], (k_it / C::NS) & 1, p)) return false;
    ptx::tc_fence_after();
    const uint32_t qa = sbase + C::OFF_Q + qs * C::TILE_BYTES;
    const uint32_t ka = sbase + C::OFF_K + ks * C::TILE_BYTES;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk * 16 / C::EPC) * C::CB_BYTES + ((kk * 16) % C::EPC) * 2;
      const uint64_t ad = ptx::smem_desc(qa + off, 16, 8 * C::SWB, C::SWZ);
      const uint64_t bd = ptx::smem_desc(ka + off, 16, 8 * C::SWB, C::SWZ);
      ptx::mma_ss(tmem + C::S_COL0 + sb * 128, ad, bd, IDESC_S, kk > 0 ? 1u : 0u);
    }
    ptx::mma_commit(ptx::smem_u32(&bars->s_full[sb]));
    ptx::mma_commit(ptx::smem_u32(&bars->k_empty[ks]));
    ++k_it;
    return true;
  };

  for (int k = 0;; ++k) {
    const long long idx = item_index(k);
    if (idx >= total) break;
    Item it;
    decode_item(p, idx, it);
    const int qs = q_it % C::NQ;
    if (!wait_bar(bars, &bars->q_full[qs], (q_it / C::NQ) & 1, p)) goto done;
    const uint32_t t_first = t;
    if (!issue_s(qs)) goto done;
    for (int j = 0; j < it.n_kv; ++j) {
      const uint32_t tj = t_first + j;  // tile whose P is consumed now
      t = tj + 1;                       // next S to issue
      if (j + 1 < it.n_kv) {
        if (!issue_s(qs)) goto done;
      }
      if (j + 1 == it.n_kv) ptx::mma_commit(ptx::smem_u32(&bars->q_empty[qs]));
      // O += P(tj) V(tj)
      const uint32_t sb = tj & 1;
      if (!wait_bar(bars, &bars->p_full[sb], (tj >> 1) & 1, p)) goto done;
      const int vs = v_it % C::NS;
      if (!wait_bar(bars, &bars->v_full[vs], (v_it / C::NS) & 1, p)) goto done;
      if (j == 0) {
        if (!wait_bar(bars, &bars->o_empty, (u & 1) ^ 1, p)) goto done;
      }
      ptx::tc_fence_after();
      const uint32_t va = sbase + C::OFF_V + vs * C::TILE_BYTES;
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk) {
        uint32_t pcol;
        if constexpr (C::P_ALIAS)
          pcol = C::S_COL0 + sb * 128 + (kk >> 2) * 64 + (kk & 3) * 8;
        else
          pcol = C::P_COL0 + sb * 64 + kk * 8;
        const uint64_t bd = ptx::smem_desc(va + kk * 16 * C::SWB, C::CB_BYTES, 8 * C::SWB, C::SWZ);
        ptx::mma_ts(tmem + C::O_COL, tmem + pcol, bd, IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
      }
      ptx::mma_commit(ptx::smem_u32(&bars->v_empty[vs]));
      ptx::mma_commit(ptx::smem_u32(&bars->pv_done[sb]));
      ++v_it;
    }
    t = t_first + it.n_kv;
    ptx::mma_commit(ptx::smem_u32(&bars->o_full));
    ++q_it;
    ++u;
  }
done:
  // Drain: every MMA issued above has finished before TMEM can be released.
  ptx::mma_commit(ptx::smem_u32(&bars->drain));
  {
    const uint32_t a = ptx::smem_u32(&bars->drain);
    const uint64_t start = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(a, 0)) {
      if ((long long)(ptx::globaltimer_ns() - start) > p.timeout_ns) {
        bars->abort = 1;
        atomicCAS(p.err, HSTU_DEVERR_NONE, HSTU_DEVERR_TIMEOUT);
        break;
      }
    }
  }
}

// ------------------------------------------------------------------ epilogue
template <int D, bool BF16, bool RAB>
__device__ void epilogue(const FwdParams& p, Bars* bars, uint8_t* smem, uint32_t tmem,
                         long long total, int warp, int lane) {
  using C = Cfg<D, RAB>;
  using T16 = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  const int wg = warp >> 2;                // column half of S, column half of O
  const int quarter = warp & 3;            // TMEM lane quarter
  const int r = quarter * 32 + lane;       // query row within the tile
  const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
  const float half_alpha = 0.5f * p.alpha;
  uint32_t t = 0, u = 0, r_it = 0;
  T16* out = static_cast<T16*>(p.out);

  for (int k = 0;; ++k) {
    const long long idx = item_index(k);
    if (idx >= total) break;
    Item it;
    decode_item(p, idx, it);
    const int i = it.m0 + r;
    const RowRange rr = row_range(it.geom, i, p.mask_type);
    for (int j = 0; j < it.n_kv; ++j, ++t) {
      const uint32_t sb = t & 1;
      if (!warp_wait(bars, &bars->s_full[sb], (t >> 1) & 1, p)) return;
      ptx::tc_fence_after();
      const uint8_t* rab_row = nullptr;
      int rs = 0;
      if constexpr (RAB) {
        rs = r_it % C::NR;
        if (!warp_wait(bars, &bars->r_full[rs], (r_it / C::NR) & 1, p)) return;
        rab_row = smem + C::OFF_R + rs * C::RAB_BYTES + wg * (C::RAB_BYTES / 2) + r * 128;
      }
      if constexpr (!C::P_ALIAS) {  // P buffer sb is free once PV(t-2) is done
        if (t >= 2 && !warp_wait(bars, &bars->pv_done[sb], ((t >> 1) & 1) ^ 1, p)) return;
      }
      const int n0 = j * kTileN;
      const bool full = tile_all_valid(it.geom, it.m0, kTileM, n0, kTileN, p.mask_type);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col = wg * 64 + c * 32;  // first S column of this chunk
        uint32_t sv[32];
        ptx::tmem_ld32(tmem + lane_off + C::S_COL0 + sb * 128 + col, sv);
        float x[32];
        if constexpr (RAB) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = (c * 4 + q4) ^ (r & 7);  // 128-byte TMA swizzle
            const uint4 w = *reinterpret_cast<const uint4*>(rab_row + chunk * 16);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 rb = unpack2<BF16>(ww[e]);
              x[q4 * 8 + 2 * e] = fmaf(__uint_as_float(sv[q4 * 8 + 2 * e]), half_alpha, 0.5f * rb.x);
              x[q4 * 8 + 2 * e + 1] =
                  fmaf(__uint_as_float(sv[q4 * 8 + 2 * e + 1]), half_alpha, 0.5f * rb.y);
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(sv[e]) * half_alpha;
        }
        // silu(2h) = 2h * sigmoid(2h) = h * (1 + tanh(h)), h = x/2
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = fmaf(x[e], ptx::tanh_approx(x[e]), x[e]);
        if (!full) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!valid_in_range(rr, n0 + col + e)) x[e] = 0.f;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack2<BF16>(x[2 * e], x[2 * e + 1]);
        uint32_t pcol;
        if constexpr (C::P_ALIAS)
          pcol = C::S_COL0 + sb * 128 + wg * 64 + c * 16;
        else
          pcol = C::P_COL0 + sb * 64 + wg * 32 + c * 16;
        ptx::tmem_st16(tmem + lane_off + pcol, pk);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars->p_full[sb]));
      if constexpr (RAB) {
        ptx::mbar_arrive(ptx::smem_u32(&bars->r_empty[rs]));
        ++r_it;
      }
    }
    // output tile
    if (!warp_wait(bars, &bars->o_full, u & 1, p)) return;
    ptx::tc_fence_after();
    constexpr int HALF = D / 2;
    constexpr int CH = HALF < 32 ? HALF : 32;
    const bool row_ok = i < it.L;
    T16* orow = out + ((it.t0 + i) * p.Nq + it.h) * (long long)D + wg * HALF;
#pragma unroll
    for (int c0 = 0; c0 < HALF; c0 += CH) {
      const uint32_t taddr = tmem + lane_off + C::O_COL + wg * HALF + c0;
      uint32_t pk[CH / 2];
      if constexpr (CH == 32) {
        uint32_t ov[32];
        ptx::tmem_ld32(taddr, ov);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack2<BF16>(__uint_as_float(ov[2 * e]) * p.silu_scale,
                              __uint_as_float(ov[2 * e + 1]) * p.silu_scale);
      } else {
        uint32_t ov[16];
        ptx::tmem_ld16(taddr, ov);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          pk[e] = pack2<BF16>(__uint_as_float(ov[2 * e]) * p.silu_scale,
                              __uint_as_float(ov[2 * e + 1]) * p.silu_scale);
      }
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
        for (int v4 = 0; v4 < CH / 8; ++v4)
          dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
      }
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(ptx::smem_u32(&bars->o_empty));
    ++u;
  }
}

// ------------------------------------------------------------------ kernel
template <int D, bool BF16, bool RAB>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r,
                  const FwdParams p) {
  using C = Cfg<D, RAB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == kProducerWarp && lane == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->q_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->q_empty[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->r_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->r_empty[s]), kEpiThreads);
      ptx::mbar_init(ptx::smem_u32(&bars->s_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->p_full[s]), kEpiThreads);
      ptx::mbar_init(ptx::smem_u32(&bars->pv_done[s]), 1);
    }
    for (int s = 0; s < 4; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->k_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->k_empty[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->v_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->v_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->o_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->o_empty), kEpiThreads);
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    bars->abort = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    if (RAB) ptx::prefetch_tmap(&tm_r);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // The work list is written by the launch before this one.
  ptx::grid_dependency_wait();
  const long long total = (long long)(*p.work_count) * p.Nq;

  if (warp < kEpiWarps) {
    epilogue<D, BF16, RAB>(p, bars, smem, tmem, total, warp, lane);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer<D, RAB>(p, bars, smem, &tm_q, &tm_k, &tm_v, &tm_r, total);
  } else if (warp == kMmaWarp) {
    if (lane == 0) mma_issuer<D, BF16, RAB>(p, bars, smem, tmem, total);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (bars->abort) {
    // Let TMA copies that were issued but never consumed land before the CTA exits.
    const uint64_t start = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - start < 200000ull) {
    }
  }
  ptx::tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tc
}  // namespace hstu
