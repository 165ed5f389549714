// Work-list builder for the persistent forward kernels.
//
// One work item is (sequence b, query tile of tile_m rows, query head h). The
// list holds (b, m-tile) pairs sorted by the number of key/value tiles the item
// visits, largest first (counting sort), so that the persistent kernel deals the
// longest items out first. Heads are expanded arithmetically by the kernel
// (item index = pair * Nq + h), which keeps the query heads of one GQA group
// adjacent in time and lets them share K/V tiles through L2.
//
// Launched with programmatic dependent launch after the previous forward kernel, the
// builder may start while that kernel's last CTAs still run (that kernel releases its
// dependents only after its own wait, so the forward call before it, which used the other
// of the plan's two work lists, has completed). It reads only the call's inputs and writes
// this call's work list, then waits for the previous kernel before it completes: the forward
// kernel behind it, which waits for the builder, therefore starts its work only after the
// previous call has finished. The index arrays are read before that wait, so the kernel
// before the builder must not write them after triggering its dependents early (the stream
// order note of hstu_fwd_run in the public header); a kernel that does not trigger early has
// completed before the builder starts.
//
// The builder also checks the caller's seq_offsets ("increasing from 0; the user
// must ensure validity", Inputs and Outputs table), and the key side (seq_offsets_k,
// the page table of the KV cache, at most as many queries as keys) and, if they are
// unusable, records HSTU_DEVERR_OFFSETS and publishes an empty list so that no kernel
// reads or writes outside the tensors.
#include "../../include/hstu_fwd.h"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace hstu {

namespace {

constexpr int kThreads = 256;  // small enough to share an SM with a forward CTA

__global__ void __launch_bounds__(kThreads) build_worklist_kernel(FwdParams p, uint32_t* work,
                                                                  int* work_count, int tile_m,
                                                                  int nbins) {
  // Let the dependent forward kernel start its prologue now; it waits for this
  // grid's completion (griddepcontrol.wait) before it reads the list.
  ptx::grid_dependents_launch();
  extern __shared__ int hist[];  // [nbins] counts, then [nbins] cursors
  int* cursor = hist + nbins;
  __shared__ int bad;
  for (int i = threadIdx.x; i < 2 * nbins; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();

  const long long T = p.total_tokens;
  for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
    long long a = seq_start(p, b);
    long long e = seq_start(p, b + 1);
    if (a < 0 || e < a || e > T || e - a > p.Sq) bad = 1;
    if (p.seq_offsets_k) {
      a = load_index(p.seq_offsets_k, b, p.index64);
      e = load_index(p.seq_offsets_k, b + 1, p.index64);
      if (a < 0 || e < a || e > p.total_tokens_k) bad = 1;
    }
    if (p.page_offsets) {
      a = load_index(p.page_offsets, b, p.index64);
      e = load_index(p.page_offsets, b + 1, p.index64);
      if (a < 0 || e < a || e > 0x7fffffffll) {
        bad = 1;
      } else if (e > a) {
        const long long last = load_index(p.last_page_len, b, p.index64);
        if (last < 1 || last > p.page_size || e - a > (long long)p.S) bad = 1;
        for (long long x = a; x < e; ++x) {
          const long long id = load_index(p.page_ids, x, p.index64);
          if (id < 0 || id >= p.num_pages) bad = 1;
        }
      }
    }
  }
  __syncthreads();
  if (p.seq_offsets_k || p.page_offsets) {  // key side: lengths, once every offset is in range
    const bool offsets_ok = !bad;
    __syncthreads();  // every thread has read the flag before it can be set again
    if (offsets_ok) {
      for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
        const SeqKV s = seq_kv(p, b);
        if (s.Lk > p.S || s.Lq > s.Lk) bad = 1;
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *p.next_item = 0;  // the forward kernel claims items from 0
  if (bad) {
    if (threadIdx.x == 0) {
      *work_count = 0;
      atomicCAS(p.err, HSTU_DEVERR_NONE, HSTU_DEVERR_OFFSETS);
    }
    ptx::grid_dependency_wait();
    return;
  }

  // key visits of a (sequence, m-tile): key tiles up to the last key its rows may see, plus
  // one when the cached history ends inside a visited tile that also holds new rows
  auto visits = [&](const SeqKV& kv, const SeqGeom& s, int mt) {
    const int off = (int)(kv.Lk - kv.Lq);  // position of query row 0
    const int kv_end = kv_end_for_rows(s, off + mt * tile_m, tile_m, p.mask_type);
    return key_visits(kv_end, split_tile((int)kv.hist, (int)kv.Lk));
  };
  // With a key side of its own (a few queries against long, often cached, key sequences)
  // the query tiles of one sequence read the same keys: they are kept next to each other
  // in the list, binned by the sequence's heaviest tile, so that they run at the same time
  // and the later reads of the keys hit L2. Without a mask every tile of a sequence visits
  // all of its keys, and its tiles are kept together the same way: interleaved with other
  // sequences' tiles, a sequence's keys are read again from HBM once the keys of all
  // sequences exceed L2. With a causal mask each tile is binned by its own count.
  const bool group = p.seq_offsets_k != nullptr || p.page_offsets != nullptr ||
                     p.mask_type == kMaskNone;
  // Per-tile bins: the tiles of a sequence are spread over `share` threads (tiles
  // mt = j, j + share, ...), so that a batch of few sequences keeps every warp busy.
  // Per-sequence bins: one thread per sequence.
  const int share = (!group && p.B < (int)blockDim.x) ? (int)blockDim.x / p.B : 1;
  // pass 1: histogram of key-visit counts; pass 2: scatter
  for (int pass = 0; pass < 2; ++pass) {
    for (int w = threadIdx.x; w < p.B * share; w += blockDim.x) {
      const int b = w % p.B, j = w / p.B;
      const SeqKV kv = seq_kv(p, b);
      const long long nc = p.num_context ? load_index(p.num_context, b, p.index64) : 0;
      const long long nt = p.num_targets ? load_index(p.num_targets, b, p.index64) : 0;
      const SeqGeom s = make_geom((int)kv.Lk, nc, nt, p.g, p.mask_type);
      const int mtiles = ceil_div((int)kv.Lq, tile_m);
      if (group) {
        int most = 0;
        for (int mt = 0; mt < mtiles; ++mt) most = max(most, visits(kv, s, mt));
        if (mtiles == 0) continue;
        if (pass == 0) {
          atomicAdd(&hist[most], mtiles);
        } else {
          const int pos = atomicAdd(&cursor[most], mtiles);
          for (int mt = 0; mt < mtiles; ++mt) work[pos + mt] = pack_item(b, mt);
        }
      } else {
        for (int mt = j; mt < mtiles; mt += share) {
          const int n = visits(kv, s, mt);
          if (pass == 0)
            atomicAdd(&hist[n], 1);
          else
            work[atomicAdd(&cursor[n], 1)] = pack_item(b, mt);
        }
      }
    }
    __syncthreads();
    if (pass == 0) {
      // exclusive scan, largest key-tile count first (cursor[n] = hist[n + 1] + ... +
      // hist[nbins - 1]): warp 0, 32 bins at a time with shuffles
      if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int base = 0; base < nbins; base += 32) {
          const int r = base + lane;  // the r-th bin from the top
          const int v = r < nbins ? hist[nbins - 1 - r] : 0;
          int x = v;
#pragma unroll
          for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x += y;
          }
          if (r < nbins) cursor[nbins - 1 - r] = carry + x - v;
          carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) *work_count = carry;
      }
      __syncthreads();
    }
  }
  // complete only after the kernel before this one in the stream
  ptx::grid_dependency_wait();
}

}  // namespace

cudaError_t launch_build_worklist(const FwdParams& p, uint32_t* work, int* work_count,
                                  int tile_m, cudaStream_t stream, bool pdl) {
  const int nbins = ceil_div(p.S, kTileN) + 2;  // visits: key tiles + one split tile
  const size_t smem = sizeof(int) * 2 * (size_t)nbins;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(build_worklist_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, build_worklist_kernel, p, work, work_count, tile_m, nbins);
}

}  // namespace hstu
