// bf16 / fp16 / FP8 E4M3 HSTU forward on the 5th-generation tensor cores (sm_103a).
//
// Operation ("RecOps Running Case Documentation", feature table and Inputs and
// Outputs table): per sequence, query head and 128-row query tile,
//   S = Q K^T, x = alpha*S (+ rab), P = silu(x) masked (x custom mask), O = P V,
//   out = silu_scale*O.
// HSTU has no softmax, so there is no running max or rescaling: O is a plain sum
// over key tiles and key tiles the mask removes entirely are never visited.
//
// CTA layout (persistent, one CTA per SM, 704 threads):
//   warps 0-15 epilogue: four warpgroups; each thread owns one query row (TMEM lane)
//              and a quarter of the 128 key columns of every S tile (for D >= 256: two
//              groups of two warpgroups take alternate tiles, half the columns each). It
//              reads S from TMEM, applies alpha, rab, SiLU (as h + h*tanh(h), h = x/2, in
//              fp32, one MUFU op per element), the mask and a custom mask, and writes P
//              (16-bit, or E4M3) back to TMEM. An item's O is read, scaled, converted and
//              stored (TMA from a staging block, or row stores) after P of the next item's
//              first tile.
//   warps 16, 18, 19, 21  producers: TMA loads of the K ring, the V ring, the Q tiles
//              and the rab (and custom-mask) ring, one thread each; the Q producer also
//              claims and decodes the work items (heaviest first; CTA i starts with item i).
//   warp 17    TMEM owner; one thread issues S(t) = Q K(t)^T (tcgen05.mma, A = Q and
//              B = K from smem, K-major) as soon as its S buffer is free, followed by the
//              rab products when the tensor core adds rab (RAB = 2).
//   warp 20    one thread issues O += P(t) V(t) (tcgen05.mma, A = P from TMEM, B = V
//              from smem, MN-major) as soon as P(t) is written. Two issuers keep a
//              thread stalled on tensor-pipe back-pressure from delaying the other
//              product. D >= 256 uses one issuer (see mma_serial_issuer).
// TMEM (512 columns): two S buffers of 128 columns from column 0, O after them (D columns,
// 256 for the head-dim-512 kernel, which computes one half of O per item) and, for
// D <= 128, two P buffers of 64 columns after O. An S buffer is handed back as soon as
// the epilogue has loaded it, so S(t + 2) is computed while the epilogue works on tile t.
// For D >= 256 P(t) is written over the columns of S(t) already read, and S(t + 2) waits
// for PV(t) to have read P(t).
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
#include "trace.cuh"

namespace hstu {
namespace tc {

// Warp roles: the epilogue warpgroups come first (their count is set per head dim by Cfg),
// then six warps of one working thread each, in this order after them.
enum : int {
  kRoleProducerK = 0,  // K and rab loads
  kRoleMma = 1,        // score products (and, with P over S, every product)
  kRoleProducerV = 2,  // V loads
  kRoleProducerQ = 3,  // Q loads, item claims
  kRolePv = 4,         // issues O += P V
  kRoleRab = 5,        // rab loads
  kRoleWarps = 6
};
constexpr uint32_t kTmemCols = 512;
// A rab / custom-mask tile (128 rows x 128 keys, 16-bit) arrives as boxes of 32 rows x 64
// keys; boxes whose keys every one of their rows has masked are not loaded (rab only).
constexpr int kRabBoxRows = 32;
// FP8 kernels round kP8Scale * P to E4M3 (the host divides silu_scale by kP8Scale):
// 16 keeps P values down to 2^-10 in the normal range and saturates only above P = 28.

// F8: q, k, v are FP8 E4M3 (one byte each); the products run as tcgen05 kind::f8f6f4 with
// P rounded to E4M3; O is written as bf16. F8 = 1: the plain cast (every descale factor 1,
// nothing read); F8 = 2: descale factors of any granularity (FwdParams::ds_mode).
// RAB: 0 no rab; 1 rab (or a custom mask) read from shared memory by the epilogue; 3 rab
// and a custom mask, one tile of each per ring slot, both read by the epilogue; 2 rab
// added to S by the tensor core: for each 16-key step k of the tile, S[:, 16k:16k+16] +=
// R[:, 16k:16k+16] (c I16) with the rab tile R as the A operand and a 16 x 16 diagonal B of
// c = 1/alpha, so that alpha*S = alpha Q K^T + rab and the epilogue is that of the plain
// kernel (head dims up to 64; eight M128 N16 K16 products per tile).
template <int D, int RAB, int F8 = 0>
struct Cfg {
  static_assert(D == 32 || D == 64 || D == 128 || D == 256 || D == 512, "head_dim");
  // WIDE (D = 512): an item computes S over all 512 columns of q and k but O over one half
  // (256 columns) of v and out; the two halves of a tile are two items. Q stays resident
  // (128 KB), K streams as 64-column chunks through a ring of four, V as two 64-key halves
  // of 256 columns through a one-slot ring; P is written over S as for D = 256. No rab,
  // mask tiles, key side or FP8.
  static constexpr bool WIDE = D == 512;
  static_assert(!WIDE || (!RAB && !F8), "head_dim 512: no rab or FP8");
  static constexpr int DV = WIDE ? 256 : D;  // O columns of one item
  static_assert(!F8 || (D <= 128 && RAB <= 1), "fp8: head_dim <= 128, rab in the epilogue");
  static constexpr bool RM = RAB == 2;        // rab by the tensor core
  static constexpr bool TWO = RAB == 3;       // rab and custom-mask tiles
  static constexpr bool EPI_RAB = RAB == 1 || TWO;  // rab / mask tiles read by the epilogue
  static_assert(!TWO || D <= 128, "rab with a custom mask: head_dim <= 128");
  static_assert(!RM || D <= 64, "rab by the tensor core: head_dim <= 64");
  static constexpr int EB = F8 ? 1 : 2;                     // bytes per q / k / v element
  static constexpr int SWB = (D * EB >= 128) ? 128 : D * EB;  // bytes per swizzled row
  static constexpr uint32_t SWZ = (SWB == 128) ? 2u : (SWB == 64 ? 4u : 6u);
  static constexpr int EPC = SWB / EB;         // elements per column block
  static constexpr int NCB = D / EPC;          // column blocks per tile row
  static constexpr int CB_BYTES = 128 * SWB;   // one column block of a 128-row tile
  static constexpr int TILE_BYTES = 128 * D * EB;
  static constexpr int O_TILE_BYTES = 128 * DV * 2;  // O is 16-bit
  static constexpr int K_SLOT = WIDE ? CB_BYTES : TILE_BYTES;  // one K ring slot
  static constexpr int VROWS = WIDE ? 64 : 128;                // keys of one V ring slot
  static constexpr int V_TILE = VROWS * DV * EB;               // one V slot (DV columns)
  static constexpr int V_CB = VROWS * SWB;                     // one of its column blocks
  static constexpr int NCBV = DV / EPC;                        // its column blocks
  static constexpr int KS = F8 ? 32 : 16;      // K elements of one MMA (32 bytes)
  static constexpr int PW = F8 ? 32 : 64;      // TMEM columns of one P buffer (128 keys)
  static constexpr int RAB_BYTES = 128 * 128 * 2;
  static constexpr int NQ = (D <= 64) ? 2 : ((D == 128 && !RAB) ? 2 : 1);
  // K and V ring depths. With rab at D = 64 the K ring is the deeper one: a K tile's load is
  // requested when the product two tiles back completes, which is too late under the rab
  // stream's HBM load (measured 1.2% faster than two K and two V slots, and than two K,
  // two V and four rab slots)
  static constexpr int NK = D == 32 ? 4 : (D == 64 ? (RAB ? 3 : 4) : (D == 128 ? 2 : (WIDE ? 4 : 1)));
  static constexpr int NV = WIDE ? 1 : ((D == 64 && RAB) ? 2 : NK);
  // rab tiles stream from HBM once each: the deeper the ring, the more bytes in flight
  // (with a custom mask beside rab a slot holds both tiles and the ring is shallower)
  static constexpr int NR = TWO ? (D == 32 ? 2 : 1)
                                : RAB ? (D == 32 ? 4 : (D == 64 ? 3 : (D == 128 ? 2 : 1))) : 0;
  static constexpr int RSLOT = (TWO ? 2 : 1) * RAB_BYTES;  // one ring slot
  // RM: the 16 x 16 diagonal B operand, K-major rows of 64 bytes (64-byte swizzle)
  static constexpr int IDENT_BYTES = RM ? 16 * 64 : 0;
  // O is staged in shared memory and written by TMA in the kernels without a rab / mask
  // stream (head dims up to 128). With one, each thread writes its row directly: the rab
  // workload's short items make the staging's proxy fence and store issue a larger share
  // of every item (measured 1.7 % faster at D = 64 with rab).
  static constexpr bool STAGE = !RAB && D <= 128;
  // Epilogue warpgroups. Four for D <= 128: a thread then takes one 32-column chunk of each
  // tile, and more warps hide more of the chain's latency (two warpgroups measured 10-28 %
  // slower there). Two for D >= 256, whose two epilogue groups are then one warpgroup each
  // with four chunks a thread: 1.8 % faster at D = 256 and 0.7 % at D = 512, and a 448-thread
  // CTA leaves up to 144 registers a thread.
  static constexpr int EPI_WG = D >= 256 ? 2 : 4;
  static constexpr int EPI_WARPS = 4 * EPI_WG;
  static constexpr int THREADS = (EPI_WARPS + kRoleWarps) * 32;
  static constexpr int PRODUCER_WARP = EPI_WARPS + kRoleProducerK;
  static constexpr int MMA_WARP = EPI_WARPS + kRoleMma;
  static constexpr int V_PRODUCER_WARP = EPI_WARPS + kRoleProducerV;
  static constexpr int Q_PRODUCER_WARP = EPI_WARPS + kRoleProducerQ;
  static constexpr int PV_WARP = EPI_WARPS + kRolePv;
  static constexpr int RAB_WARP = EPI_WARPS + kRoleRab;
  static constexpr int OC = DV / EPI_WG;             // O columns per epilogue warpgroup
  static constexpr int OSWB = OC * 2;                // O staging row bytes (swizzle span)
  static constexpr int WARP_STAGE = 32 * OC * 2;     // one warp's O block in shared memory
  // Epilogue groups. With two, the epilogue warps form two groups of two warpgroups and
  // group g takes the S tiles t with t % 2 == g (S and P buffer g), so that one group
  // computes while the other waits for its next tile; that pays for D >= 256, whose longer
  // products leave the epilogue waiting. With one, all four warpgroups work on every tile.
  static constexpr int EPI_GROUPS = D >= 256 ? 2 : 1;
  static constexpr int GROUP_WARPS = EPI_WARPS / EPI_GROUPS;
  static constexpr int COLS_PER_WG = kTileN / (EPI_WG / EPI_GROUPS);  // S columns per tile
  // TMEM (512 columns). For D <= 128, P has two buffers of its own and S two buffers; an
  // S buffer is released as soon as the epilogue has loaded it, so the next score products
  // overlap the epilogue. O has two accumulators where they fit beside them (D <= 64), one
  // for D = 128 (two there would leave one S buffer, which measured slower: it holds the
  // score products back). For D >= 256 (O takes 256 columns) P is written over the S
  // buffer it came from and one thread issues all MMAs.
  static constexpr bool P_SEP = (D <= 128);
  static constexpr bool SERIAL = !P_SEP;
  static constexpr int NPB = 2;             // P buffers (P_SEP), P over S otherwise
  // O accumulators: two where TMEM has room for them next to two S buffers (D <= 64), so
  // that an item's first PV product does not wait for the previous item's O to be drained
  static constexpr int NO = (P_SEP && 2 * 128 + 2 * D + NPB * PW <= (int)kTmemCols) ? 2 : 1;
  static constexpr int NSB_FIT = (int)(kTmemCols - NO * DV - (P_SEP ? NPB * PW : 0)) / 128;
  static constexpr int NSB = NSB_FIT < 2 ? NSB_FIT : 2;  // S buffers
  // TMEM columns
  static constexpr uint32_t S_COL0 = 0, O_COL0 = NSB * 128;
  static constexpr uint32_t P_COL0 = O_COL0 + NO * DV;  // P buffers of PW columns (P_SEP only)
  // shared memory map (offsets from a 1024-aligned base)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NK * K_SLOT;
  static constexpr int OFF_R = OFF_V + NV * V_TILE;
  static constexpr int OFF_I = OFF_R + NR * RSLOT;  // diagonal B operand (RM)
  static constexpr int OFF_O = OFF_I + (RM ? 1024 : 0);   // (a 1024-byte swizzle atom)
  static constexpr int OFF_BAR = OFF_O + (STAGE ? O_TILE_BYTES : 0);
  static constexpr int BAR_BYTES = 1024;
  static constexpr int SMEM_USED = OFF_BAR + BAR_BYTES;
  // keep one CTA per SM (TMEM is allocated whole)
  static constexpr int SMEM_BYTES = (SMEM_USED + 1024 < 120 * 1024) ? 120 * 1024 : SMEM_USED + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(NSB >= 1 && P_COL0 + (P_SEP ? NPB * PW : 0) <= kTmemCols, "TMEM map");
  static_assert(SERIAL ? NSB == NPB : true, "P over S: P buffer = S buffer");
};

// One work item, decoded once (by the Q producer) and read by every role.
struct Item {
  int b, h, hk, m0, n_kv;
  int tq, Lq;      // first query row of the sequence, query rows
  int tk, hist;    // first new k/v row, cached keys (key positions [0, hist))
  int off;         // key position of query row 0 (Lk - Lq)
  int split;       // key tile visited twice (cached part, new part), or -1
  union {
    int po;        // first page_ids entry of the sequence (key side)
    int half;      // O half of a head dim 512 item (no key side)
  };
  SeqGeom geom;    // over the Lk keys
};

constexpr int kInfoDepth = 8;                   // decoded items kept in shared memory
// item readers: epilogue warps, the MMA issuer(s), K and V producers, the rab producer
template <bool SERIAL, int RAB, int EPI_WARPS>
constexpr int info_readers() { return EPI_WARPS + (SERIAL ? 3 : 4) + (RAB ? 1 : 0); }

// Barrier block layout.
struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t r_full[4], r_empty[4];
  uint64_t s_full[3], p_full[3], pv_done[3], s_free[2];
  uint64_t o_full[2], o_empty[2], drain;
  uint64_t info_full[kInfoDepth], info_empty[kInfoDepth];
  Item info[kInfoDepth];
  uint32_t tmem_base;
  volatile int abort;
};
static_assert(sizeof(Bars) <= 1024, "barrier block");

// KV: the kernel variant for key sides that differ from the queries (own k/v offsets, a
// KV cache); without it the keys are the query rows and the decomposition folds away.
// WIDE: items 2i and 2i + 1 are the two O halves of item i of the plain numbering.
template <bool KV, bool WIDE = false>
__device__ __forceinline__ bool decode_item(const FwdParams& p, long long idx, Item& it) {
  int half = 0;
  if constexpr (WIDE) {
    half = (int)(idx & 1);
    idx >>= 1;
  }
  const uint32_t e = p.work[idx / p.Nq];
  it.h = (int)(idx % p.Nq);
  it.hk = it.h / (p.Nq / p.Nk);
  it.b = item_b(e);
  it.m0 = item_mt(e) * kTileM;
  if constexpr (!KV) {
    const long long t0 = seq_start(p, it.b);
    it.tq = it.tk = (int)t0;
    it.Lq = (int)(seq_start(p, it.b + 1) - t0);
    it.hist = it.off = 0;
    it.po = 0;
    if constexpr (WIDE) it.half = half;
    it.split = -1;
    const long long nc = p.num_context ? load_index(p.num_context, it.b, p.index64) : 0;
    const long long nt = p.num_targets ? load_index(p.num_targets, it.b, p.index64) : 0;
    it.geom = make_geom(it.Lq, nc, nt, p.g, p.mask_type);
    it.n_kv = ceil_div(kv_end_for_rows(it.geom, it.m0, kTileM, p.mask_type), kTileN);
    return true;
  }
  const SeqKV kv = seq_kv(p, it.b);
  it.tq = (int)kv.tq;
  it.Lq = (int)kv.Lq;
  it.tk = (int)kv.tk;
  it.hist = (int)kv.hist;
  it.po = (int)kv.po;
  it.off = (int)(kv.Lk - kv.Lq);
  const long long nc = p.num_context ? load_index(p.num_context, it.b, p.index64) : 0;
  const long long nt = p.num_targets ? load_index(p.num_targets, it.b, p.index64) : 0;
  it.geom = make_geom((int)kv.Lk, nc, nt, p.g, p.mask_type);
  it.split = split_tile(it.hist, (int)kv.Lk);
  it.n_kv = key_visits(kv_end_for_rows(it.geom, it.off + it.m0, kTileM, p.mask_type), it.split);
  return true;
}


// Pause between two tries of a wait, per role (a pausing thread issues no instructions).
// Measured: pauses of 128 ns for the producers and 32 ns for the MMA issuers cost more
// (later products) than the issue slots they free, so none is taken.
constexpr uint32_t kNapProducer = 0, kNapIssuer = 0, kNapNone = 0;  // nanoseconds

// Bounded wait. Returns false when this CTA is aborting (own timeout or another role's).
// try_wait suspends the thread in hardware until the phase completes or a short system
// limit passes; the abort flag and the clock are checked every 16 tries only.
template <uint32_t NAP = kNapProducer>
__device__ __forceinline__ bool wait_bar(Bars* bars, uint64_t* bar, uint32_t parity,
                                         const FwdParams& p) {
  const uint32_t a = ptx::smem_u32(bar);
  if (ptx::mbar_try_wait(a, parity)) return true;
  const uint64_t start = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if constexpr (NAP > 0) __nanosleep(NAP);
    if (ptx::mbar_try_wait(a, parity)) return true;
    if ((i & 15u) == 0) {
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
  const bool ok = wait_bar<kNapNone>(bars, bar, parity, p);
  return __all_sync(0xffffffffu, ok);
}

// Item ring: the Q producer decodes item k (global loads of the work list and the
// sequence metadata) and publishes it in slot k % kInfoDepth; every other role
// reads it from shared memory, so no role waits on those loads at an item start.
__device__ __forceinline__ bool put_item(Bars* bars, int k, const Item& it, const FwdParams& p) {
  const int s = k % kInfoDepth;
  if (!wait_bar(bars, &bars->info_empty[s], ((k / kInfoDepth) & 1) ^ 1, p)) return false;
  bars->info[s] = it;
  ptx::mbar_arrive(ptx::smem_u32(&bars->info_full[s]));
  return true;
}

// Single-thread reader.
template <uint32_t NAP = kNapProducer>
__device__ __forceinline__ bool get_item(Bars* bars, int k, Item& it, const FwdParams& p) {
  const int s = k % kInfoDepth;
  if (!wait_bar<NAP>(bars, &bars->info_full[s], (k / kInfoDepth) & 1, p)) return false;
  it = bars->info[s];
  ptx::mbar_arrive(ptx::smem_u32(&bars->info_empty[s]));
  return true;
}

// Bits e (0..31) set where column base + e is valid for the row (RowRange intervals).
__device__ __forceinline__ uint32_t low_bits(int n) {  // n lowest bits, n clamped to [0, 32]
  return n <= 0 ? 0u : (n >= 32 ? 0xffffffffu : ((1u << n) - 1u));
}
__device__ __forceinline__ uint32_t chunk_mask(const RowRange& r, int base) {
  const uint32_t hist = low_bits(r.hist_end - base);
  const uint32_t grp = low_bits(r.grp_hi - base + 1) & ~low_bits(r.grp_lo - base);
  return r.grp_lo <= r.grp_hi ? (hist | grp) : hist;
}
// Bits e set where tile column cc + e lies in the visit's column range [clo, chi).
__device__ __forceinline__ uint32_t cols_mask(const KeyTile& kt, int cc) {
  return low_bits(kt.chi - cc) & ~low_bits(kt.clo - cc);
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

// A packed 16-bit pair as two fp32 values (exact).
template <bool BF16>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
  if constexpr (BF16) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  } else {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = f.x;
    hi = f.y;
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t fma2(uint32_t a, uint32_t b, uint32_t c) {
  if constexpr (BF16)
    return ptx::fma_bf16x2(a, b, c);
  else
    return ptx::fma_f16x2(a, b, c);
}

// ------------------------------------------------------------------ producers
// Three producer threads in separate warps stream Q, K (+ rab) and V, so that no
// load waits behind the release of another ring's slot. With two Q buffers the Q
// producer runs up to two work items ahead; with one, it prefetches the next
// item's Q tile into L2 so that the load after the slot frees hits in L2.
template <int D, int RAB, bool KV, int F8>
__device__ void producer_q(const FwdParams& p, Bars* bars, uint8_t* smem, const CUtensorMap* tq,
                           long long total) {
  using C = Cfg<D, RAB, F8>;
  uint32_t q_it = 0;
  const uint32_t sbase = ptx::smem_u32(smem);
  // Items are claimed dynamically from the heaviest-first list: CTA i starts with item i,
  // later items take one atomic each. With a single Q buffer the next item is claimed one
  // early so that its Q tile can be prefetched into L2.
  auto claim = [&]() -> long long { return (long long)gridDim.x + atomicAdd(p.next_item, 1); };
  long long idx = blockIdx.x;
  for (int k = 0;; ++k) {
    Item it;
    if (idx >= total) {  // no work left: publish the end marker
      it.n_kv = -1;
      put_item(bars, k, it, p);
      return;
    }
    decode_item<KV, C::WIDE>(p, idx, it);
    HSTU_TRACE_EV(p, trace::kRoleQ, trace::kItem, idx);
    if (!put_item(bars, k, it, p)) return;
    long long nidx = -1;
    if (C::NQ == 1) {
      nidx = claim();
      if (nidx < total) {
        Item nx;
        decode_item<KV, C::WIDE>(p, nidx, nx);
#pragma unroll
        for (int cb = 0; cb < C::NCB; ++cb)
          ptx::tma_prefetch_3d(tq, cb * C::EPC, nx.h, nx.tq + nx.m0);
      }
    }
    const int s = q_it % C::NQ;
    if (!wait_bar(bars, &bars->q_empty[s], ((q_it / C::NQ) & 1) ^ 1, p)) return;
    const uint32_t full = ptx::smem_u32(&bars->q_full[s]);
    ptx::mbar_arrive_expect_tx(full, C::TILE_BYTES);
    const uint32_t dst = sbase + C::OFF_Q + s * C::TILE_BYTES;
#pragma unroll
    for (int cb = 0; cb < C::NCB; ++cb)
      ptx::tma_load_3d(dst + cb * C::CB_BYTES, tq, full, cb * C::EPC, it.h, it.tq + it.m0);
    HSTU_TRACE_EV(p, trace::kRoleQ, trace::kLoad, k);
    ++q_it;
    idx = C::NQ == 1 ? nidx : claim();
  }
}

// Pages of the KV cache behind one cached key tile (x, positions [128x, 128x + 128), with
// 128x < hist): one page of >= 128 rows, or four pages of 32 rows. Slots past the sequence's
// last page repeat the last page: their rows lie beyond the history, where P is 0.
struct TilePages {
  int id[4];
};

__device__ __forceinline__ TilePages tile_pages(const FwdParams& p, const Item& it, int x) {
  TilePages t;
  const int npages = ceil_div(it.hist, p.page_size);
  if (p.page_size >= kTileN) {
    t.id[0] = (int)load_index(p.page_ids, it.po + (x * kTileN) / p.page_size, p.index64);
  } else {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int slot = min(x * 4 + m, npages - 1);
      t.id[m] = (int)load_index(p.page_ids, it.po + slot, p.index64);
    }
  }
  return t;
}

// One K or V tile (plane 0 or 1) of key visit j into shared memory at dst: from the
// cache pages when the visit's rows are cached, else rows tk + 128x - hist .. of k / v
// (rows before the sequence's first new row belong to the cached part of a split tile
// and meet P = 0 there).
template <int D, int RAB, int F8>
__device__ __forceinline__ void load_kv_tile(const FwdParams& p, const Item& it, int j,
                                             const TilePages& pg, const CUtensorMap* tnew,
                                             const CUtensorMap* tcache, int plane, uint32_t dst,
                                             uint32_t full) {
  using C = Cfg<D, RAB, F8>;
  const KeyTile kt = key_tile(j, it.split, it.hist);
  if (!kt.cached) {
    const int row = it.tk + kt.x * kTileN - it.hist;
#pragma unroll
    for (int cb = 0; cb < C::NCB; ++cb)
      ptx::tma_load_3d(dst + cb * C::CB_BYTES, tnew, full, cb * C::EPC, it.hk, row);
  } else if (p.page_size >= kTileN) {
    const int r0 = (kt.x * kTileN) % p.page_size;
#pragma unroll
    for (int cb = 0; cb < C::NCB; ++cb)
      ptx::tma_load_4d(dst + cb * C::CB_BYTES, tcache, full, cb * C::EPC, it.hk, r0,
                       2 * pg.id[0] + plane);
  } else {  // four pages of 32 rows
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int cb = 0; cb < C::NCB; ++cb)
        ptx::tma_load_4d(dst + cb * C::CB_BYTES + m * 32 * C::SWB, tcache, full, cb * C::EPC,
                         it.hk, 0, 2 * pg.id[m] + plane);
  }
}

template <int D, int RAB, bool KV, int F8>
__device__ void producer_k(const FwdParams& p, Bars* bars, uint8_t* smem, const CUtensorMap* tk,
                           const CUtensorMap* tc, long long total) {
  using C = Cfg<D, RAB, F8>;
  uint32_t k_it = 0;
  const uint32_t sbase = ptx::smem_u32(smem);
  if (p.test_stall) return;  // watchdog test: no K tile is ever signalled
  for (int k = 0;; ++k) {
    Item it;
    if (!get_item(bars, k, it, p) || it.n_kv < 0) return;
    if constexpr (C::WIDE) {  // 64-column chunks of each K tile, one ring slot each
      for (int j = 0; j < it.n_kv; ++j)
        for (int cb = 0; cb < C::NCB; ++cb) {
          const int s = k_it % C::NK;
          if (!wait_bar(bars, &bars->k_empty[s], ((k_it / C::NK) & 1) ^ 1, p)) return;
          const uint32_t full = ptx::smem_u32(&bars->k_full[s]);
          ptx::mbar_arrive_expect_tx(full, C::K_SLOT);
          ptx::tma_load_3d(sbase + C::OFF_K + s * C::K_SLOT, tk, full, cb * C::EPC, it.hk,
                           it.tq + j * kTileN);
          ++k_it;
        }
      continue;
    }
    for (int j = 0; j < it.n_kv; ++j) {
      const int s = k_it % C::NK;
      // page ids are read before the wait for the slot, which hides their latency
      TilePages pg = {};
      if constexpr (KV) {
        const KeyTile kt = key_tile(j, it.split, it.hist);
        if (kt.cached) pg = tile_pages(p, it, kt.x);
      }
      if (!wait_bar(bars, &bars->k_empty[s], ((k_it / C::NK) & 1) ^ 1, p)) return;
      HSTU_TRACE_EV(p, trace::kRoleK, trace::kLoad, k_it);
      const uint32_t full = ptx::smem_u32(&bars->k_full[s]);
      ptx::mbar_arrive_expect_tx(full, C::TILE_BYTES);
      const uint32_t dst = sbase + C::OFF_K + s * C::TILE_BYTES;
      if constexpr (KV) {
        load_kv_tile<D, RAB, F8>(p, it, j, pg, tk, tc, 0, dst, full);
      } else {
#pragma unroll
        for (int cb = 0; cb < C::NCB; ++cb)
          ptx::tma_load_3d(dst + cb * C::CB_BYTES, tk, full, cb * C::EPC, it.hk,
                           it.tq + j * kTileN);
      }
      ++k_it;
    }
  }
}

// rab tiles of every S tile, in tile order, on their own thread: the rab ring is released
// by the epilogue (late in a tile), and waiting for it must not hold back the K loads.
// A tile is loaded as up to eight boxes of 32 rows x 64 keys (a 128-byte swizzled column
// block of 128 rows takes four); with rab (not a custom mask, which is multiplied into P)
// a box is skipped when its rows lie beyond the item's queries or every key of it is at or
// beyond the end of what its rows may see (diagonal and ragged tiles): its entries are all
// masked, and the epilogue sets a masked entry's h to 0 after adding rab.
template <int D, int RAB, bool MASK, bool KV, int F8>
__device__ void producer_r(const FwdParams& p, Bars* bars, uint8_t* smem, const CUtensorMap* tr,
                           const CUtensorMap* tm, long long total) {
  using C = Cfg<D, RAB, F8>;
  constexpr int STRIPS = kTileM / kRabBoxRows;
  constexpr uint32_t BOX_BYTES = kRabBoxRows * 128;
  uint32_t r_it = 0;
  const uint32_t sbase = ptx::smem_u32(smem);
  for (int k = 0;; ++k) {
    Item it;
    if (!get_item(bars, k, it, p) || it.n_kv < 0) return;
    const int plane = (int)rab_plane(p, it.b, it.h);
    const int row = (KV ? it.off : 0) + it.m0;  // key position of the item's first query row
    // key end of each row strip (keys at or beyond it are masked for all of its rows)
    int strip_end[STRIPS];
#pragma unroll
    for (int st = 0; st < STRIPS; ++st)
      strip_end[st] = it.m0 + st * kRabBoxRows >= it.Lq
                          ? 0
                          : kv_end_for_rows(it.geom, row + st * kRabBoxRows, kRabBoxRows,
                                            p.mask_type);
    for (int j = 0; j < it.n_kv; ++j) {
      const int rs = r_it % C::NR;
      if (!wait_bar(bars, &bars->r_empty[rs], ((r_it / C::NR) & 1) ^ 1, p)) return;
      const uint32_t full = ptx::smem_u32(&bars->r_full[rs]);
      const uint32_t dst = sbase + C::OFF_R + rs * C::RSLOT;
      // rows: the key positions of the item's queries; columns: the visit's key tile
      const KeyTile kt = KV ? key_tile(j, it.split, it.hist) : KeyTile{j, 0, kTileN, false};
      const int n0 = kt.x * kTileN;
      uint32_t need = 0;  // bit st * 2 + cb: box of row strip st, column block cb
#pragma unroll
      for (int st = 0; st < STRIPS; ++st)
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          const bool used = MASK || (strip_end[st] > n0 + 64 * cb && kt.clo < 64 * cb + 64 &&
                                     kt.chi > 64 * cb);
          need |= (used ? 1u : 0u) << (st * 2 + cb);
        }
      ptx::mbar_arrive_expect_tx(full, (__popc(need) + (C::TWO ? 2 * STRIPS : 0)) * BOX_BYTES);
#pragma unroll
      for (int st = 0; st < STRIPS; ++st)
#pragma unroll
        for (int cb = 0; cb < 2; ++cb)
          if (need & (1u << (st * 2 + cb)))
            ptx::tma_load_3d(dst + cb * (C::RAB_BYTES / 2) + st * BOX_BYTES, tr, full,
                             n0 + 64 * cb, row + st * kRabBoxRows, plane);
      if constexpr (C::TWO) {  // the custom-mask tile behind the rab tile (every box)
        const int mplane = it.b * p.Nq + it.h;
#pragma unroll
        for (int st = 0; st < STRIPS; ++st)
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
            ptx::tma_load_3d(dst + C::RAB_BYTES + cb * (C::RAB_BYTES / 2) + st * BOX_BYTES, tm,
                             full, n0 + 64 * cb, row + st * kRabBoxRows, mplane);
      }
      ++r_it;
    }
  }
}

template <int D, int RAB, bool KV, int F8>
__device__ void producer_v(const FwdParams& p, Bars* bars, uint8_t* smem, const CUtensorMap* tv,
                           const CUtensorMap* tc, long long total) {
  using C = Cfg<D, RAB, F8>;
  uint32_t v_it = 0;
  const uint32_t sbase = ptx::smem_u32(smem);
  for (int k = 0;; ++k) {
    Item it;
    if (!get_item(bars, k, it, p) || it.n_kv < 0) return;
    for (int j = 0; j < it.n_kv; ++j) {
      const int s = v_it % C::NV;
      TilePages pg = {};
      if constexpr (KV) {
        const KeyTile kt = key_tile(j, it.split, it.hist);
        if (kt.cached) pg = tile_pages(p, it, kt.x);
      }
      if (!wait_bar(bars, &bars->v_empty[s], ((v_it / C::NV) & 1) ^ 1, p)) return;
      HSTU_TRACE_EV(p, trace::kRoleV, trace::kLoad, v_it);
      const uint32_t full = ptx::smem_u32(&bars->v_full[s]);
      ptx::mbar_arrive_expect_tx(full, C::V_TILE);
      const uint32_t dst = sbase + C::OFF_V + s * C::V_TILE;
      if constexpr (KV) {
        load_kv_tile<D, RAB, F8>(p, it, j, pg, tv, tc, 1, dst, full);
      } else if constexpr (C::WIDE) {
        // the first 64 keys of the tile (the map's box is 64 rows); the second half below
#pragma unroll
        for (int cb = 0; cb < C::NCBV; ++cb)
          ptx::tma_load_3d(dst + cb * C::V_CB, tv, full, it.half * C::DV + cb * C::EPC, it.hk,
                           it.tq + j * kTileN);
        ++v_it;
        const int s2 = v_it % C::NV;
        if (!wait_bar(bars, &bars->v_empty[s2], ((v_it / C::NV) & 1) ^ 1, p)) return;
        const uint32_t full2 = ptx::smem_u32(&bars->v_full[s2]);
        ptx::mbar_arrive_expect_tx(full2, C::V_TILE);
        const uint32_t dst2 = sbase + C::OFF_V + s2 * C::V_TILE;
#pragma unroll
        for (int cb = 0; cb < C::NCBV; ++cb)
          ptx::tma_load_3d(dst2 + cb * C::V_CB, tv, full2, it.half * C::DV + cb * C::EPC, it.hk,
                           it.tq + j * kTileN + C::VROWS);
      } else {
#pragma unroll
        for (int cb = 0; cb < C::NCBV; ++cb)
          ptx::tma_load_3d(dst + cb * C::CB_BYTES, tv, full, cb * C::EPC, it.hk,
                           it.tq + j * kTileN);
      }
      ++v_it;
    }
  }
}

// ------------------------------------------------------------------ MMA issuers
// Two threads issue tcgen05.mma: one the score products S(t) = Q K(t)^T, the other
// the accumulations O += P(t) V(t). An issuing thread stalls while the tensor pipe is
// busy; with one issuer per product neither waits behind the other, and the next
// scores are issued the moment their S buffer is free.

// Both issuers end by waiting until their own MMAs have completed (TMEM is freed after).
__device__ __forceinline__ void mma_drain(Bars* bars, const FwdParams& p) {
  ptx::mma_commit(ptx::smem_u32(&bars->drain));
  const uint32_t a = ptx::smem_u32(&bars->drain);
  const uint64_t start = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait_sleep(a, 0, 20000u)) {
    if ((long long)(ptx::globaltimer_ns() - start) > p.timeout_ns) {
      bars->abort = 1;
      atomicCAS(p.err, HSTU_DEVERR_NONE, HSTU_DEVERR_TIMEOUT);
      break;
    }
  }
}

// Single issuer, used when P is written over its S buffer (D = 256): there S(t+2)
// can only start after PV(t) has read P(t), so the two products form one chain and
// are issued in that order: S(t0), S(t0+1), then per tile PV(t), S(t+2).
template <int D, bool BF16, int RAB, int F8>
__device__ void mma_serial_issuer(const FwdParams& p, Bars* bars, uint8_t* smem, uint32_t tmem,
                                  long long total) {
  using C = Cfg<D, RAB, F8>;
  constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16 ? 1u : 0u, 128, kTileN, 0);
  constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16 ? 1u : 0u, 128, C::DV, 1);
  const uint32_t sbase = ptx::smem_u32(smem);
  uint32_t q_it = 0, k_it = 0, v_it = 0, u = 0, t_base = 0;
  auto issue_s = [&](uint32_t t, int qs) -> bool {
    const uint32_t sb = t % C::NSB;
    if (t >= C::NSB && !wait_bar<kNapIssuer>(bars, &bars->pv_done[sb], ((t / C::NSB) & 1) ^ 1, p))
      return false;
    if constexpr (C::WIDE) {  // S = sum over the 64-column chunks of Q_c K_c^T
      const uint32_t qa = sbase + C::OFF_Q + qs * C::TILE_BYTES;
      for (int cb = 0; cb < C::NCB; ++cb) {
        const int ks = k_it % C::NK;
        if (!wait_bar<kNapIssuer>(bars, &bars->k_full[ks], (k_it / C::NK) & 1, p)) return false;
        ptx::tc_fence_after();
        const uint32_t ka = sbase + C::OFF_K + ks * C::K_SLOT;
#pragma unroll
        for (int kk = 0; kk < C::EPC / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc(qa + cb * C::CB_BYTES + kk * 32, 16, 8 * C::SWB, C::SWZ);
          const uint64_t bd = ptx::smem_desc(ka + kk * 32, 16, 8 * C::SWB, C::SWZ);
          ptx::mma_ss(tmem + C::S_COL0 + sb * 128, ad, bd, IDESC_S, (cb > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&bars->k_empty[ks]));
        ++k_it;
      }
      ptx::mma_commit(ptx::smem_u32(&bars->s_full[sb]));
      return true;
    }
    const int ks = k_it % C::NK;
    if (!wait_bar<kNapIssuer>(bars, &bars->k_full[ks], (k_it / C::NK) & 1, p)) return false;
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
  auto issue_pv = [&](uint32_t t, bool first) -> bool {
    const uint32_t sb = t % C::NSB;
    if (first && !wait_bar<kNapIssuer>(bars, &bars->o_empty[0], (u & 1) ^ 1, p)) return false;
    // one V slot holds VROWS keys: the tile's 128 keys in one slot, or (WIDE) two halves
    for (int k0 = 0; k0 < kTileN; k0 += C::VROWS) {
      const int vs = v_it % C::NV;
      if (!wait_bar<kNapIssuer>(bars, &bars->v_full[vs], (v_it / C::NV) & 1, p)) return false;
      ptx::tc_fence_after();
      const uint32_t va = sbase + C::OFF_V + vs * C::V_TILE;
#pragma unroll
      for (int kk = 0; kk < C::VROWS / 16; ++kk) {
        const int key = k0 + 16 * kk;  // first key of this K = 16 step
        const uint32_t pcol = C::S_COL0 + sb * 128 + (key / C::COLS_PER_WG) * C::COLS_PER_WG +
                              (key % C::COLS_PER_WG) / 2;
        const uint64_t bd = ptx::smem_desc(va + kk * 16 * C::SWB, C::V_CB, 8 * C::SWB, C::SWZ);
        ptx::mma_ts(tmem + C::O_COL0, tmem + pcol, bd, IDESC_O, (!first || key > 0) ? 1u : 0u);
      }
      ptx::mma_commit(ptx::smem_u32(&bars->v_empty[vs]));
      ++v_it;
    }
    ptx::mma_commit(ptx::smem_u32(&bars->pv_done[sb]));
    return true;
  };
  for (int k = 0;; ++k) {
    Item it;
    if (!get_item<kNapIssuer>(bars, k, it, p) || it.n_kv < 0) break;
    const int qs = q_it % C::NQ;
    if (!wait_bar<kNapIssuer>(bars, &bars->q_full[qs], (q_it / C::NQ) & 1, p)) break;
    const int n = it.n_kv;
    bool ok = issue_s(t_base, qs) && (n < 2 || issue_s(t_base + 1, qs));
    if (ok && n <= 2) ptx::mma_commit(ptx::smem_u32(&bars->q_empty[qs]));
    for (int j = 0; j < n && ok; ++j) {
      const uint32_t t = t_base + j;
      ok = wait_bar<kNapIssuer>(bars, &bars->p_full[t % C::NSB], (t / C::NSB) & 1, p) && issue_pv(t, j == 0);
      if (ok && j + 2 < n) {
        ok = issue_s(t + 2, qs);
        if (ok && j + 3 == n) ptx::mma_commit(ptx::smem_u32(&bars->q_empty[qs]));
      }
    }
    if (!ok) break;
    t_base += n;
    ptx::mma_commit(ptx::smem_u32(&bars->o_full[0]));
    ++q_it;
    ++u;
  }
  mma_drain(bars, p);
}

template <int D, bool BF16, int RAB, int F8>
__device__ void mma_s_issuer(const FwdParams& p, Bars* bars, uint8_t* smem, uint32_t tmem,
                             long long total) {
  using C = Cfg<D, RAB, F8>;
  // kind::f16: A/B format 0 = f16, 1 = bf16; kind::f8f6f4: format 0 = E4M3
  constexpr uint32_t IDESC_S = ptx::idesc_f16((BF16 && !F8) ? 1u : 0u, 128, kTileN, 0);
  const uint32_t sbase = ptx::smem_u32(smem);
  uint32_t q_it = 0, k_it = 0, t = 0;
  // RM: the rab tile of S(t) (A, K-major, 128-byte swizzle) against the 16 x 16 diagonal
  // operand (K-major, 64-byte swizzle), one M128 N16 K16 product per 16 keys
  const uint64_t id0 = C::RM ? ptx::smem_desc(sbase + C::OFF_I, 16, 8 * 64, 4) : 0;
  constexpr uint32_t IDESC_R = ptx::idesc_f16((BF16 && !F8) ? 1u : 0u, 128, 16, 0);
  for (int k = 0;; ++k) {
    Item it;
    if (!get_item<kNapIssuer>(bars, k, it, p) || it.n_kv < 0) break;
    const int qs = q_it % C::NQ;
    if (!wait_bar<kNapIssuer>(bars, &bars->q_full[qs], (q_it / C::NQ) & 1, p)) break;
    const uint64_t ad0 =
        ptx::smem_desc(sbase + C::OFF_Q + qs * C::TILE_BYTES, 16, 8 * C::SWB, C::SWZ);
    bool ok = true;
    for (int j = 0; j < it.n_kv && ok; ++j, ++t) {
      const uint32_t sb = t % C::NSB;
      const int ks = k_it % C::NK;
      // S buffer sb is free once the epilogue has loaded S(t - NSB) into registers; both
      // conditions are tested at once, and only one found unmet is waited for
      uint64_t* sfree = &bars->s_free[sb];
      uint64_t* kfull = &bars->k_full[ks];
      const uint32_t sf_par = ((t / C::NSB) & 1) ^ 1, kf_par = (k_it / C::NK) & 1;
      const uint32_t ready = ptx::mbar_test2(ptx::smem_u32(sfree), sf_par, ptx::smem_u32(kfull),
                                             kf_par);
      if (!(ready & 1u) && t >= C::NSB && !wait_bar<kNapIssuer>(bars, sfree, sf_par, p)) {
        ok = false;
        break;
      }
      if (!(ready & 2u) && !wait_bar<kNapIssuer>(bars, kfull, kf_par, p)) { ok = false; break; }
      HSTU_TRACE_EV(p, trace::kRoleS, trace::kIssue, t);
      ptx::tc_fence_after();
      const uint64_t bd0 =
          ptx::smem_desc(sbase + C::OFF_K + ks * C::TILE_BYTES, 16, 8 * C::SWB, C::SWZ);
#pragma unroll
      for (int kk = 0; kk < D / C::KS; ++kk) {  // K steps of 32 bytes
        const int e = kk * C::KS;
        const uint32_t off = (e / C::EPC) * C::CB_BYTES + (e % C::EPC) * C::EB;
        const uint64_t ad = ptx::desc_add(ad0, off);
        const uint64_t bd = ptx::desc_add(bd0, off);
        if constexpr (F8)
          ptx::mma_ss_f8(tmem + C::S_COL0 + sb * 128, ad, bd, IDESC_S, kk > 0 ? 1u : 0u);
        else
          ptx::mma_ss(tmem + C::S_COL0 + sb * 128, ad, bd, IDESC_S, kk > 0 ? 1u : 0u);
      }
      if constexpr (C::RM) {
        // S[:, 16k:16k+16] += R[:, 16k:16k+16] (c I16) for the eight 16-key steps k
        const int rs = t % C::NR;
        if (!wait_bar<kNapIssuer>(bars, &bars->r_full[rs], (t / C::NR) & 1, p)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint64_t rd0 = ptx::smem_desc(sbase + C::OFF_R + rs * C::RAB_BYTES, 16, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          const uint32_t off = (kk / 4) * (C::RAB_BYTES / 2) + (kk % 4) * 32;
          ptx::mma_ss(tmem + C::S_COL0 + sb * 128 + 16 * kk, ptx::desc_add(rd0, off), id0,
                      IDESC_R, 1u);
        }
        ptx::mma_commit(ptx::smem_u32(&bars->r_empty[rs]));
      }
      ptx::mma_commit(ptx::smem_u32(&bars->s_full[sb]));
      ptx::mma_commit(ptx::smem_u32(&bars->k_empty[ks]));
      if (j + 1 == it.n_kv) ptx::mma_commit(ptx::smem_u32(&bars->q_empty[qs]));
      ++k_it;
    }
    if (!ok) break;
    ++q_it;
  }
  mma_drain(bars, p);
}

template <int D, bool BF16, int RAB, int F8>
__device__ void mma_pv_issuer(const FwdParams& p, Bars* bars, uint8_t* smem, uint32_t tmem,
                              long long total) {
  using C = Cfg<D, RAB, F8>;
  constexpr uint32_t IDESC_O = ptx::idesc_f16((BF16 && !F8) ? 1u : 0u, 128, D, 1);
  const uint32_t sbase = ptx::smem_u32(smem);
  uint32_t v_it = 0, t = 0, u = 0;
  for (int k = 0;; ++k) {
    Item it;
    if (!get_item<kNapIssuer>(bars, k, it, p) || it.n_kv < 0) break;
    bool ok = true;
    for (int j = 0; j < it.n_kv; ++j, ++t) {
      const uint32_t pb = t % C::NPB;  // P buffer
      const uint32_t ob = u % C::NO;   // O accumulator of this item
      const int vs = v_it % C::NV;
      uint64_t* pfull = &bars->p_full[pb];
      uint64_t* vfull = &bars->v_full[vs];
      const uint32_t pf_par = (t / C::NPB) & 1, vf_par = (v_it / C::NV) & 1;
      const uint32_t ready = ptx::mbar_test2(ptx::smem_u32(pfull), pf_par, ptx::smem_u32(vfull),
                                             vf_par);
      if (!(ready & 1u) && !wait_bar<kNapIssuer>(bars, pfull, pf_par, p)) { ok = false; break; }
      if (!(ready & 2u) && !wait_bar<kNapIssuer>(bars, vfull, vf_par, p)) { ok = false; break; }
      if (j == 0 && !wait_bar<kNapIssuer>(bars, &bars->o_empty[ob], ((u / C::NO) & 1) ^ 1, p)) {
        ok = false;
        break;
      }
      HSTU_TRACE_EV(p, trace::kRolePV, trace::kIssue, t);
      ptx::tc_fence_after();
      const uint64_t bd0 = ptx::smem_desc(sbase + C::OFF_V + vs * C::TILE_BYTES, C::CB_BYTES,
                                          8 * C::SWB, C::SWZ);
#pragma unroll
      for (int kk = 0; kk < kTileN / C::KS; ++kk) {
        // keys [KS*kk, KS*kk + KS) are packed in P columns [8kk, 8kk + 8) (2 or 4 per column)
        const uint32_t pcol = C::P_COL0 + pb * C::PW + kk * 8;
        const uint64_t bd = ptx::desc_add(bd0, kk * C::KS * C::SWB);
        if constexpr (F8)
          ptx::mma_ts_f8(tmem + C::O_COL0 + ob * D, tmem + pcol, bd, IDESC_O,
                         (j > 0 || kk > 0) ? 1u : 0u);
        else
          ptx::mma_ts(tmem + C::O_COL0 + ob * D, tmem + pcol, bd, IDESC_O,
                      (j > 0 || kk > 0) ? 1u : 0u);
      }
      ptx::mma_commit(ptx::smem_u32(&bars->v_empty[vs]));
      ptx::mma_commit(ptx::smem_u32(&bars->pv_done[pb]));
      ++v_it;
    }
    if (!ok) break;
    ptx::mma_commit(ptx::smem_u32(&bars->o_full[u % C::NO]));
    ++u;
  }
  mma_drain(bars, p);
}

// ------------------------------------------------------------------ epilogue
// Warp w of warpgroup wg = w / 4 reads TMEM lanes 32*(w % 4) .. +31 (one query row per
// thread) and S columns [32*wg, 32*wg + 32) of every tile; it writes the 16 packed P
// columns of those keys and, at the end of an item, O columns [wg*D/4, (wg+1)*D/4).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, uint32_t (&r)[8]) {
  ptx::tmem_ld8(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, uint32_t (&r)[16]) {
  ptx::tmem_ld16(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&r)[32]) {
  ptx::tmem_ld32(taddr, r);
}

// Every lane of the warp arrives once, after its own part (and its tcgen05 fence): one
// warp instruction and no divergent branch; the barrier counts 32 arrivals per warp.
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
  (void)lane;
  ptx::mbar_arrive(ptx::smem_u32(bar));
}

// Byte offset of a 16-byte chunk inside a TMA box written with SWB-byte swizzling
// (the 16-byte chunk index is XORed with the row index within each swizzle atom).
template <int SWB>
__device__ __forceinline__ uint32_t swizzle(uint32_t o) {
  if constexpr (SWB <= 16) {
    return o;  // one chunk per row: no swizzle
  } else {
    constexpr uint32_t mask = SWB == 128 ? 0x70u : (SWB == 64 ? 0x30u : 0x10u);
    return o ^ ((o >> 3) & mask);
  }
}

// FP8 descale factor of (sequence b, block blk, head h) for the granularity p.ds_mode (one
// factor; one per sequence; per sequence and head; per sequence, 128-row block and head,
// with nb blocks per sequence and n heads).
__device__ __forceinline__ long long ds_index(const FwdParams& p, int b, int blk, int h, int nb,
                                              int n) {
  if (p.ds_mode == 1) return 0;
  if (p.ds_mode == 2) return b;
  if (p.ds_mode == 3) return (long long)b * n + h;
  return ((long long)b * nb + blk) * n + h;
}

// The v factor of an item's output: its v descale (one per item below block granularity),
// or the largest |v descale| over the sequence's key blocks, relative to which the
// epilogue scales P for each key tile (block granularity). 1 for the plain cast.
__device__ __forceinline__ float item_v_scale(const FwdParams& p, const Item& it) {
  if (p.ds_mode == 0) return 1.f;
  if (p.ds_mode < 4) return __ldg(p.v_ds + ds_index(p, it.b, 0, it.hk, p.ds_kb, p.Nk));
  float m = 0.f;
  for (int x = 0; x * kTileN < it.geom.L; ++x)
    m = fmaxf(m, fabsf(__ldg(p.v_ds + ds_index(p, it.b, x, it.hk, p.ds_kb, p.Nk))));
  return m;
}

template <int D, bool BF16, int RAB, bool MASK, bool KV, int F8>
__device__ void epilogue(const FwdParams& p, Bars* bars, uint8_t* smem, uint32_t tmem,
                         const CUtensorMap* tm_o, long long total, int warp, int lane) {
  using C = Cfg<D, RAB, F8>;
  constexpr bool OUT_BF16 = BF16 || F8;  // O type (FP8 inputs give bf16 out)
  using T16 = typename std::conditional<OUT_BF16, __nv_bfloat16, __half>::type;
  constexpr int OC = C::OC;                  // O columns per warpgroup
  constexpr int OCH = OC < 32 ? OC : 32;     // O columns per TMEM load
  const int wg = warp >> 2;
  const int quarter = warp & 3;              // TMEM lane quarter
  const int r = quarter * 32 + lane;         // query row within the tile
  const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
  constexpr int WG_PER_GROUP = C::EPI_WG / C::EPI_GROUPS;
  const int group = wg / WG_PER_GROUP;  // takes the S tiles t with t % EPI_GROUPS == group
  const int col = (wg % WG_PER_GROUP) * C::COLS_PER_WG;  // first S column of this warpgroup
  const float half_alpha = 0.5f * p.alpha;
  uint32_t t = 0, u = 0;
  T16* out = static_cast<T16*>(p.out);
  int prev_slot = -1;  // item ring slot of the item whose O is still in TMEM
  // Output of a finished item: read this warpgroup's O columns chunk by chunk, scale,
  // stage (or store), release O, then write the staged block. Called after P of the next
  // item's first tile has been written, so that the epilogue is not idle while the item's
  // last accumulation completes. The item stays in its ring slot until this returns.
  auto drain = [&](int slot) -> bool {
    if (lane == 0 && (warp == 0 || warp == C::EPI_WARPS - 1))
      HSTU_TRACE_EV(p, warp == 0 ? trace::kRoleEpi : trace::kRoleEpiB, trace::kDrainBeg, slot);
    const Item& pit = bars->info[slot];
    const int pi = pit.m0 + r;  // query row within the sequence
    float osc = p.silu_scale;   // (FP8: times the item's v factor)
    if constexpr (F8 == 2) osc *= item_v_scale(p, pit);
    const uint32_t ob = u % C::NO;  // the item's O accumulator
    if (!warp_wait(bars, &bars->o_full[ob], (u / C::NO) & 1, p)) return false;
    ptx::tc_fence_after();
    uint8_t* stage = smem + C::OFF_O + warp * C::WARP_STAGE;
    if constexpr (C::STAGE) {
      if (lane == 0) ptx::bulk_wait_read0();  // this warp's previous store has read it
      __syncwarp();
    }
    // rows of out hold p.D elements (the kernel's D for a padded head dim is larger; its
    // extra columns are not stored)
    const int oc0 = (C::WIDE ? pit.half * C::DV : 0) + wg * OC;  // first out column
    T16* orow = out + (((long long)pit.tq + pi) * p.Nq + pit.h) * (long long)p.D + oc0;
#pragma unroll
    for (int c0 = 0; c0 < OC; c0 += OCH) {
      uint32_t part[OCH];
      tmem_ld<OCH>(tmem + lane_off + C::O_COL0 + ob * C::DV + wg * OC + c0, part);
      if constexpr (OC == OCH) {
        // the whole O slice is in registers: hand the accumulator back before converting
        ptx::tc_fence_before();
        warp_arrive(&bars->o_empty[ob], lane);
      }
#pragma unroll
      for (int v4 = 0; v4 < OCH / 8; ++v4) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float o0, o1;
          ptx::mul_f32x2(o0, o1, __uint_as_float(part[v4 * 8 + 2 * e]),
                         __uint_as_float(part[v4 * 8 + 2 * e + 1]), osc, osc);
          w[e] = pack2<OUT_BF16>(o0, o1);
        }
        if constexpr (C::STAGE) {
          // this warp's 32-row x (D/4)-column block in the TMA box layout: swizzled 16-byte
          // chunks, conflict-free for one row per lane
          *reinterpret_cast<uint4*>(stage + swizzle<C::OSWB>(lane * OC * 2 + c0 * 2 + v4 * 16)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        } else if (pi < pit.Lq && oc0 + c0 + v4 * 8 < p.D) {
          reinterpret_cast<uint4*>(orow + c0)[v4] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    if constexpr (OC != OCH) {
      ptx::tc_fence_before();
      warp_arrive(&bars->o_empty[ob], lane);
    }
    ++u;
    if constexpr (C::STAGE) {
      // one TMA store when all 32 rows of the block lie inside the sequence; a block that
      // crosses the end of the sequence is stored row by row
      const int row0 = pit.m0 + quarter * 32;
      if (row0 + 32 <= pit.Lq) {
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && oc0 < p.D) {  // (a slice wholly beyond a padded head dim: none)
          ptx::tma_store_3d(tm_o, ptx::smem_u32(stage), wg * OC, pit.h, pit.tq + row0);
          ptx::bulk_commit();
        }
      } else if (pi < pit.Lq) {
#pragma unroll
        for (int v4 = 0; v4 < OC / 8; ++v4)
          if (oc0 + v4 * 8 < p.D)
            reinterpret_cast<uint4*>(orow)[v4] = *reinterpret_cast<const uint4*>(
                stage + swizzle<C::OSWB>(lane * OC * 2 + v4 * 16));
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->info_empty[slot]));
    if (lane == 0 && (warp == 0 || warp == C::EPI_WARPS - 1))
      HSTU_TRACE_EV(p, warp == 0 ? trace::kRoleEpi : trace::kRoleEpiB, trace::kDrainEnd, slot);
    return true;
  };

  for (int k = 0;; ++k) {
    // the item is released by drain() once its O has been written
    const int slot = k % kInfoDepth;
    if (!warp_wait(bars, &bars->info_full[slot], (k / kInfoDepth) & 1, p)) return;
    const Item it = bars->info[slot];
    if (it.n_kv < 0) break;  // end marker
    if (lane == 0 && (warp == 0 || warp == C::EPI_WARPS - 1))
      HSTU_TRACE_EV(p, warp == 0 ? trace::kRoleEpi : trace::kRoleEpiB, trace::kItem, k);
    const int m0p = (KV ? it.off : 0) + it.m0;  // key position of the item's first query row
    const int i = m0p + r;                      // and of this thread's row
    const RowRange rr = row_range(it.geom, i, p.mask_type);
    // without a key side, the key tiles that need no mask are a prefix of the item's tiles
    const int n_full = KV ? 0 : full_tiles(it.geom, m0p, kTileM, kTileN, p.mask_type);
    // FP8 descales: alpha * qd * kd folds into the SiLU argument's factor, vd into P (block
    // granularity: per key tile, relative to the item's v factor) or the output scale
    float ha_item = half_alpha, qds = 1.f, p8_per_v = kP8Scale;
    if constexpr (F8 == 2) {
      {
        qds = __ldg(p.q_ds + ds_index(p, it.b, it.m0 / kTileM, it.h, p.ds_qb, p.Nq));
        if (p.ds_mode < 4) {
          ha_item = half_alpha * qds * __ldg(p.k_ds + ds_index(p, it.b, 0, it.hk, p.ds_kb, p.Nk));
        } else {
          const float vm = item_v_scale(p, it);
          p8_per_v = vm > 0.f ? kP8Scale / vm : 0.f;
        }
      }
    }
    int gtile = 0;  // tiles of this item processed by this group
    for (int j = 0; j < it.n_kv; ++j, ++t) {
      if ((int)(t % C::EPI_GROUPS) != group) continue;  // the other group's tile
      const uint32_t sb = t % C::NSB;  // S buffer (== group with two epilogue groups)
      if (!warp_wait(bars, &bars->s_full[sb], (t / C::NSB) & 1, p)) return;
      if (lane == 0 && (warp == 0 || warp == C::EPI_WARPS - 1))
        HSTU_TRACE_EV(p, warp == 0 ? trace::kRoleEpi : trace::kRoleEpiB, trace::kSReady, t);
      ptx::tc_fence_after();
      KeyTile kt;
      if constexpr (KV) {
        kt = key_tile(j, it.split, it.hist);
      } else {
        kt.x = j;
        kt.clo = 0;
        kt.chi = kTileN;
        kt.cached = false;
      }
      const int n0 = kt.x * kTileN;
      float ha = ha_item, p8 = kP8Scale;
      if constexpr (F8 == 2) {
        if (p.ds_mode == 4) {
          const long long ki = ds_index(p, it.b, kt.x, it.hk, p.ds_kb, p.Nk);
          ha = half_alpha * qds * __ldg(p.k_ds + ki);
          p8 = p8_per_v * __ldg(p.v_ds + ki);
        }
      }
      bool full;
      if constexpr (KV)
        full = kt.clo == 0 && kt.chi == kTileN &&
               tile_all_valid(it.geom, m0p, kTileM, n0, kTileN, p.mask_type);
      else
        full = j < n_full;
      const uint8_t* rab_row = nullptr;
      int rs = 0;
      if constexpr (C::EPI_RAB) {
        rs = t % C::NR;  // one rab tile per S tile, in tile order
        // With two epilogue groups and a one-tile rab ring (D = 256) the rab slot alternates
        // between the groups, so a group reaching tile t may find r_full two phases behind,
        // where a parity wait cannot tell phase t from phase t - 2: it first waits until
        // the other group has released tile t - 1 (r_full is then at phase t at most).
        if constexpr (C::NR < C::EPI_GROUPS) {
          if (t >= 1 &&
              !warp_wait(bars, &bars->r_empty[(t - 1) % C::NR], ((t - 1) / C::NR) & 1, p))
            return;
        }
        if (!warp_wait(bars, &bars->r_full[rs], (t / C::NR) & 1, p)) return;
        rab_row = smem + C::OFF_R + rs * C::RSLOT + r * 128;
      }
#pragma unroll 1
      for (int c = 0; c < C::COLS_PER_WG / 32; ++c) {  // 32-column chunks, one after the other
        const int cc = col + c * 32;  // first S column of this 32-column chunk
        uint32_t sv[32];
        ptx::tmem_ld32(tmem + lane_off + C::S_COL0 + sb * 128 + cc, sv);
        if (C::P_SEP && c + 1 == C::COLS_PER_WG / 32) {  // all of this warp's S columns loaded
          ptx::tc_fence_before();
          warp_arrive(&bars->s_free[sb], lane);
        }
        // h = alpha*s/2 (+ rab/2) in fp32, and silu(2h) = 2h*sigmoid(2h) = h + h*tanh(h): one
        // special-function op per element (tanh.approx.f32), products and sums on packed
        // fp32 pairs, P rounded once to the 16-bit type (or to E4M3). A masked entry gets
        // h = 0, so its P is silu(0) = 0.
        float h[32];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          ptx::mul_f32x2(h[e], h[e + 1], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]),
                         ha, ha);
        uint32_t mw[16];  // custom-mask pairs (MASK)
        if constexpr (C::EPI_RAB) {
          // rab / custom-mask tile: two 64-column TMA boxes of 128 rows x 128 bytes with
          // 128-byte swizzle, read conflict-free (one row per lane)
          const uint8_t* box = rab_row + (cc >> 6) * (C::RAB_BYTES / 2);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = (((cc & 63) >> 3) + q4) ^ (r & 7);
            const uint4 w = *reinterpret_cast<const uint4*>(box + chunk * 16);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c2 = q4 * 4 + e;  // pair index: columns 2*c2, 2*c2 + 1
              if constexpr (MASK && !C::TWO) {
                mw[c2] = ww[e];
              } else {
                float r0, r1;
                unpack2<BF16>(ww[e], r0, r1);
                ptx::fma_f32x2(h[2 * c2], h[2 * c2 + 1], r0, r1, 0.5f, 0.5f, h[2 * c2],
                               h[2 * c2 + 1]);
              }
            }
          }
          if constexpr (C::TWO) {  // the custom-mask tile, behind the rab tile in the slot
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int chunk = (((cc & 63) >> 3) + q4) ^ (r & 7);
              const uint4 w = *reinterpret_cast<const uint4*>(box + C::RAB_BYTES + chunk * 16);
              mw[q4 * 4 + 0] = w.x;
              mw[q4 * 4 + 1] = w.y;
              mw[q4 * 4 + 2] = w.z;
              mw[q4 * 4 + 3] = w.w;
            }
          }
        }
        if (!full) {
          // valid columns of this row form [0, hist_end) U [grp_lo, grp_hi]: as a bit mask
          // over the 32 columns of the chunk
          uint32_t m = chunk_mask(rr, n0 + cc);
          if constexpr (KV) m &= cols_mask(kt, cc);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!(m & (1u << e))) h[e] = 0.f;
        }
        uint32_t pk[16];  // 16-bit P pairs, or (F8) E4M3 P quads in pk[0..7]
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float t0 = ptx::tanh_approx(h[2 * e]), t1 = ptx::tanh_approx(h[2 * e + 1]);
          float p0, p1;
          if constexpr (F8) {
            // p8 * P = (p8 * h) * tanh(h) + p8 * h with p8 = kP8Scale (a power of two, so
            // that typical values stay in E4M3's normal range), times vd / max vd for block
            // descales
            float s0, s1;
            ptx::mul_f32x2(s0, s1, h[2 * e], h[2 * e + 1], p8, p8);
            ptx::fma_f32x2(p0, p1, s0, s1, t0, t1, s0, s1);
            if constexpr (MASK) {  // custom mask (bf16) applied before the E4M3 rounding
              float m0, m1;
              unpack2<true>(mw[e], m0, m1);
              ptx::mul_f32x2(p0, p1, p0, p1, m0, m1);
            }
            const uint32_t q = ptx::cvt_e4m3x2_f32(p0, p1);  // keys 2e, 2e + 1
            if (e & 1)
              pk[e >> 1] |= q << 16;
            else
              pk[e >> 1] = q;
          } else {
            ptx::fma_f32x2(p0, p1, h[2 * e], h[2 * e + 1], t0, t1, h[2 * e], h[2 * e + 1]);
            pk[e] = pack2<BF16>(p0, p1);
            // custom mask: P times the mask pair (adding -0 keeps the product exact)
            if constexpr (MASK) pk[e] = fma2<BF16>(pk[e], mw[e], 0x80008000u);
          }
        }
        uint32_t pcol;
        if constexpr (C::P_SEP) {
          // P buffer t % NPB is free once PV(t - NPB) has read it
          const uint32_t pb = t % C::NPB;
          if (c == 0 && t >= C::NPB &&
              !warp_wait(bars, &bars->pv_done[pb], ((t / C::NPB) & 1) ^ 1, p))
            return;
          pcol = C::P_COL0 + pb * C::PW + cc / (C::PW == 64 ? 2 : 4);
        } else {
          pcol = C::S_COL0 + sb * 128 + col + c * 16;  // over S columns already read
        }
        if constexpr (F8) {
          // P rounded to E4M3 (saturating), four keys per TMEM column, lowest key in the
          // low byte: the A operand of the kind::f8f6f4 product
          uint32_t p8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) p8[e] = pk[e];
          ptx::tmem_st8(tmem + lane_off + pcol, p8);
        } else {
          ptx::tmem_st16(tmem + lane_off + pcol, pk);
        }
      }
      if constexpr (C::EPI_RAB) warp_arrive(&bars->r_empty[rs], lane);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      warp_arrive(&bars->p_full[t % C::NPB], lane);
      if (lane == 0 && (warp == 0 || warp == C::EPI_WARPS - 1))
        HSTU_TRACE_EV(p, warp == 0 ? trace::kRoleEpi : trace::kRoleEpiB, trace::kPDone, t);
      // this group's part of the previous item's O, after the group's first tile of this
      // item (P of a whole tile behind the item's last accumulation, which has finished
      // by then), or at the group's last tile of the item
      ++gtile;
      if (prev_slot >= 0 && (gtile == 1 || j + C::EPI_GROUPS >= it.n_kv)) {
        if (!drain(prev_slot)) return;
        prev_slot = -1;
      }
    }
    // a group with no tile in this item drains the previous one here
    if (prev_slot >= 0 && !drain(prev_slot)) return;
    prev_slot = slot;
  }
  if (prev_slot >= 0 && !drain(prev_slot)) return;
  if (C::STAGE && lane == 0) ptx::bulk_wait0();  // this warp's last TMA store is complete
}

// ------------------------------------------------------------------ kernel
// MASK: the rab stream carries a custom mask (multiplied into P after the SiLU).
template <int D, bool BF16, int RAB, bool MASK = false, bool KV = false, int F8 = 0>
__global__ void __launch_bounds__(Cfg<D, RAB, F8>::THREADS, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r,
                  const __grid_constant__ CUtensorMap tm_o,
                  const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_m,
                  const FwdParams p) {
  using C = Cfg<D, RAB, F8>;
  static_assert(C::NQ <= (int)(sizeof(Bars::q_full) / sizeof(uint64_t)) &&
                    C::NK <= (int)(sizeof(Bars::k_full) / sizeof(uint64_t)) &&
                    C::NV <= (int)(sizeof(Bars::v_full) / sizeof(uint64_t)) &&
                    C::NR <= (int)(sizeof(Bars::r_full) / sizeof(uint64_t)),
                "ring depths exceed the barrier arrays");
  static_assert(C::NSB % C::EPI_GROUPS == 0, "S buffers per epilogue group");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == C::PRODUCER_WARP && lane == 0) {
#define HSTU_INIT_ALL(arr, count)                                       \
  for (int s = 0; s < (int)(sizeof(bars->arr) / sizeof(uint64_t)); ++s) \
    ptx::mbar_init(ptx::smem_u32(&bars->arr[s]), (count));
    // every lane of the epilogue group that owns an S / P buffer arrives on s_free, p_full
    // and r_empty (and every epilogue lane on o_empty)
    HSTU_INIT_ALL(s_free, C::GROUP_WARPS * 32)
    HSTU_INIT_ALL(s_full, 1)
    HSTU_INIT_ALL(p_full, C::GROUP_WARPS * 32)
    HSTU_INIT_ALL(pv_done, 1)
    HSTU_INIT_ALL(q_full, 1)
    HSTU_INIT_ALL(q_empty, 1)
    HSTU_INIT_ALL(r_full, 1)
    // rab slots are released by the epilogue lanes, or (RM) by the score issuer's commit
    HSTU_INIT_ALL(r_empty, C::RM ? 1 : C::GROUP_WARPS * 32)
    HSTU_INIT_ALL(k_full, 1)
    HSTU_INIT_ALL(k_empty, 1)
    HSTU_INIT_ALL(v_full, 1)
    HSTU_INIT_ALL(v_empty, 1)
    HSTU_INIT_ALL(o_full, 1)
    HSTU_INIT_ALL(o_empty, C::EPI_WARPS * 32)
#undef HSTU_INIT_ALL
    HSTU_TRACE_INIT();
    ptx::mbar_init(ptx::smem_u32(&bars->drain), C::SERIAL ? 1 : 2);  // one commit per issuer
    for (int s = 0; s < kInfoDepth; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->info_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->info_empty[s]), info_readers<C::SERIAL, RAB, C::EPI_WARPS>());
    }
    bars->abort = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    if (RAB) ptx::prefetch_tmap(&tm_r);
    if (C::TWO) ptx::prefetch_tmap(&tm_m);
    if (C::STAGE) ptx::prefetch_tmap(&tm_o);
    if (KV && p.page_offsets) ptx::prefetch_tmap(&tm_c);
  }
  if (warp == C::MMA_WARP) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  if constexpr (C::RM) {
    // The diagonal B operand (16 keys x 16, K-major, rows of 64 bytes with the 64-byte
    // swizzle, the first 32 bytes used) holds c = 1/alpha on its diagonal, and the rab ring
    // starts zeroed: a rab box that is never loaded (all of its entries masked) then holds
    // finite values, so its products with the zeros of the diagonal stay finite (and 0 in
    // the entries that are not masked).
    uint4* z = reinterpret_cast<uint4*>(smem + C::OFF_R);
    const int n16 = (C::NR * C::RAB_BYTES + C::IDENT_BYTES) / 16;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) z[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (threadIdx.x < 16) {
      const uint32_t j = threadIdx.x;  // key row j, contraction column j
      const uint32_t off = swizzle<64>(j * 64 + (j >> 3) * 16) + (j & 7) * 2;
      *reinterpret_cast<uint16_t*>(smem + C::OFF_I + off) = (uint16_t)p.rab_ident;
    }
    ptx::fence_proxy_async_smem();  // the tensor core (async proxy) reads both
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  if (threadIdx.x == 0) {
    HSTU_TRACE_EV(p, trace::kRoleCta, trace::kStart, 0);
    HSTU_TRACE_RAW(p, trace::kRoleCta, ptx::globaltimer_ns());
  }

  // The work list is written by the launch before this one. Dependents (the next call's
  // work-list build) are released only after this wait: by then the call before this one,
  // which used the other work list, has completed.
  ptx::grid_dependency_wait();
  ptx::grid_dependents_launch();
  const long long total = (long long)(*p.work_count) * p.Nq * (C::WIDE ? 2 : 1);
  if (threadIdx.x == 0) HSTU_TRACE_EV(p, trace::kRoleCta, trace::kDepDone, 0);

  if (warp < C::EPI_WARPS) {
    epilogue<D, BF16, RAB, MASK, KV, F8>(p, bars, smem, tmem, &tm_o, total, warp, lane);
  } else if (warp == C::PRODUCER_WARP) {
    if (lane == 0) producer_k<D, RAB, KV, F8>(p, bars, smem, &tm_k, &tm_c, total);
  } else if (warp == C::Q_PRODUCER_WARP) {
    if (lane == 0) producer_q<D, RAB, KV, F8>(p, bars, smem, &tm_q, total);
  } else if (warp == C::V_PRODUCER_WARP) {
    if (lane == 0) producer_v<D, RAB, KV, F8>(p, bars, smem, &tm_v, &tm_c, total);
  } else if (warp == C::MMA_WARP) {
    if (lane == 0) {
      if constexpr (C::SERIAL)
        mma_serial_issuer<D, BF16, RAB, F8>(p, bars, smem, tmem, total);
      else
        mma_s_issuer<D, BF16, RAB, F8>(p, bars, smem, tmem, total);
    }
  } else if (warp == C::RAB_WARP) {
    if constexpr (RAB) {
      if (lane == 0) producer_r<D, RAB, MASK, KV, F8>(p, bars, smem, &tm_r, &tm_m, total);
    }
  } else if (warp == C::PV_WARP) {
    if (lane == 0 && !C::SERIAL) mma_pv_issuer<D, BF16, RAB, F8>(p, bars, smem, tmem, total);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    HSTU_TRACE_EV(p, trace::kRoleCta, trace::kEnd, 0);
    HSTU_TRACE_RAW(p, trace::kRoleCta, ptx::globaltimer_ns());
    HSTU_TRACE_FINISH(p);
  }
  if (bars->abort) {
    // Let TMA copies that were issued but never consumed land before the CTA exits.
    const uint64_t start = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - start < 200000ull) {
    }
  }
  ptx::tc_fence_after();
  if (warp == C::MMA_WARP) {
    __syncwarp();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tc
}  // namespace hstu
