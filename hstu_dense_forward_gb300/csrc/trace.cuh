// Pipeline tracer of the tensor-core forward kernel (a build made with -DHSTU_TRACE=1).
//
// Selected threads of every CTA stamp events into a plan-owned device buffer. The buffer
// has kSlots launch slots (run r of a plan uses slot r % kSlots, so that the CTAs of
// back-to-back launches, which overlap, never share a region); a slot has one region of
// kEvents 64-bit words per (CTA, role). A word packs the event kind (8 bits), a 24-bit
// argument (tile or item counter) and the low 32 bits of the SM clock; the CTA role also
// stores the global timer at the CTA's start and end, which places the per-SM clocks on
// one time axis. Event counts live in shared memory while the CTA runs and are written to
// word 0 of each region at its end; a region that fills up stops recording (no write past
// it). In ordinary builds every hook compiles to nothing.
#pragma once
#include <stdint.h>

#ifndef HSTU_TRACE
#define HSTU_TRACE 0
#endif

namespace hstu {
namespace trace {

constexpr int kRoles = 8;
constexpr int kEvents = 1024;        // words per (CTA, role); word 0 holds the count
constexpr int kMaxCtas = 160;
constexpr int kSlots = 4;
constexpr size_t kSlotWords = (size_t)kMaxCtas * kRoles * kEvents;
constexpr size_t kBufferWords = kSlots * kSlotWords;

enum Role : int {
  kRoleCta = 0,   // thread 0: start / end (global timer)
  kRoleEpi = 1,   // epilogue warp 0, lane 0
  kRoleEpiB = 2,  // the last epilogue warp, lane 0 (the last warpgroup)
  kRoleS = 3,     // score-product issuer
  kRolePV = 4,    // O += P V issuer
  kRoleQ = 5,     // Q producer / item claimer
  kRoleK = 6,     // K producer
  kRoleV = 7,     // V producer
};

enum Event : int {
  kStart = 1,       // followed by a raw global-timer word
  kDepDone = 2,     // grid dependency wait returned
  kEnd = 3,         // followed by a raw global-timer word
  kItem = 4,        // a role starts work item k (arg k)
  kSReady = 5,      // epilogue: S(t) landed in TMEM (arg t)
  kSLoaded = 6,     // epilogue: S(t) read into registers
  kPDone = 7,       // epilogue: P(t) written and signalled
  kDrainBeg = 8,    // epilogue: O drain of the previous item begins
  kDrainEnd = 9,
  kIssue = 10,      // an issuer starts the products of tile t (its waits are over)
  kLoad = 11,       // a producer issues the loads of tile / item arg
};

#if HSTU_TRACE
__device__ __forceinline__ uint32_t clock32() {
  uint32_t c;
  asm volatile("mov.u32 %0, %%clock;" : "=r"(c));
  return c;
}

__device__ __forceinline__ uint32_t* counts() {
  __shared__ uint32_t n[kRoles];
  return n;
}

// Thread 0, before the CTA's first __syncthreads.
__device__ __forceinline__ void init() {
  for (int r = 0; r < kRoles; ++r) counts()[r] = 0;
}

__device__ __forceinline__ unsigned long long* region(unsigned long long* slot, int role) {
  return slot + ((size_t)blockIdx.x * kRoles + role) * kEvents;
}

__device__ __forceinline__ void put(unsigned long long* slot, int role, unsigned long long w) {
  if (slot == nullptr || blockIdx.x >= (unsigned)kMaxCtas) return;
  const uint32_t n = counts()[role];
  if (n + 1 >= (uint32_t)kEvents) return;
  region(slot, role)[1 + n] = w;
  counts()[role] = n + 1;
}

__device__ __forceinline__ void record(unsigned long long* slot, int role, int ev, uint32_t arg) {
  put(slot, role, ((unsigned long long)(ev & 0xff) << 56) |
                      ((unsigned long long)(arg & 0xffffffu) << 32) | clock32());
}

// Thread 0, after the CTA's last __syncthreads: the event counts into word 0.
__device__ __forceinline__ void finish(unsigned long long* slot) {
  if (slot == nullptr || blockIdx.x >= (unsigned)kMaxCtas) return;
  for (int r = 0; r < kRoles; ++r) region(slot, r)[0] = counts()[r];
}
#define HSTU_TRACE_INIT() ::hstu::trace::init()
#define HSTU_TRACE_EV(p, role, ev, arg) ::hstu::trace::record((p).trace, (role), (ev), (uint32_t)(arg))
#define HSTU_TRACE_RAW(p, role, value) ::hstu::trace::put((p).trace, (role), (value))
#define HSTU_TRACE_FINISH(p) ::hstu::trace::finish((p).trace)
#else
#define HSTU_TRACE_INIT() ((void)0)
#define HSTU_TRACE_EV(p, role, ev, arg) ((void)0)
#define HSTU_TRACE_RAW(p, role, value) ((void)0)
#define HSTU_TRACE_FINISH(p) ((void)0)
#endif

}  // namespace trace
}  // namespace hstu
