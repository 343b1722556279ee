// Device helpers shared by the verify-step kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tsd.h"

namespace tsd {

constexpr unsigned kFull = 0xffffffffu;

// Default budget of every bounded device wait (an mbarrier or a flag), in SM
// clock cycles: about one second at 2 GHz.  A wait that runs out records
// TSD_DEV_ERR_TIMEOUT and its kernel returns instead of hanging.
constexpr long long kWaitCycles = 2000000000ll;

// Order-preserving map of an fp32 value to uint32 (larger float -> larger
// key).  -0.0 is folded onto +0.0 so that the two compare equal, as they do
// for float comparison.
__device__ __forceinline__ uint32_t f32_order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float order_key_f32(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// A vocabulary candidate as one 64-bit integer: value in the high word,
// bit-inverted token id in the low word.  A larger candidate is a larger
// value, or an equal value with a smaller id -- the (value desc, id asc)
// order of top-k and of argmax with ties to the lowest id.  Distinct ids give
// distinct candidates.  0 is below every real candidate.
__device__ __forceinline__ uint64_t make_cand(float x, uint32_t id) {
  return ((uint64_t)f32_order_key(x) << 32) | (uint64_t)(~id);
}
__device__ __forceinline__ uint32_t cand_id(uint64_t c) { return ~(uint32_t)c; }
__device__ __forceinline__ float cand_val(uint64_t c) { return order_key_f32((uint32_t)(c >> 32)); }

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation (tsd::launch in tsd_host.h) may be scheduled while the kernel
// before it on the stream is still running.  Before its first global read or
// write each thread waits until that kernel has completed and its writes are
// visible (a no-op after an ordinary launch); then the CTA lets the next
// kernel be scheduled (its set-up overlaps this kernel's work).  Only set-up
// that touches no global memory may precede this call.
__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// L2 prefetch of [p, p + bytes) by the bulk-copy unit, narrowed to whole
// 16-byte units and to its first MiB.  A hint: nothing is returned and L2 stays coherent, so it
// may precede grid_dependency_sync (a kernel launched early warms L2 with its
// inputs while the previous kernel finishes).
__device__ __forceinline__ void prefetch_l2(const void* p, long bytes) {
  uintptr_t a = (uintptr_t)p, e = a + (uintptr_t)bytes;
  a = (a + 15) & ~(uintptr_t)15;
  e &= ~(uintptr_t)15;
  if (e > a + (1u << 20)) e = a + (1u << 20);   // at most 1 MiB per hint
  if (e > a)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(a), "r"((uint32_t)(e - a))
                 : "memory");
}

// First device error wins; request index in the low 24 bits.
__device__ __forceinline__ void report_error(int32_t* err, int code, int b) {
  if (err != nullptr) atomicCAS(err, 0, code | (b & 0xffffff));
}

// Insert candidate c into a warp-distributed list sorted in descending order
// (lane j holds the j-th largest; only lanes < k are meaningful).  The caller
// guarantees c is larger than the current k-th entry, so c lands in [0, k).
__device__ __forceinline__ void warp_list_insert(uint64_t& entry, uint64_t c, unsigned kmask, int lane) {
  const unsigned greater = __ballot_sync(kFull, entry > c) & kmask;
  const int pos = __popc(greater);
  const uint64_t up = __shfl_up_sync(kFull, entry, 1);
  if (lane > pos) entry = up;
  else if (lane == pos) entry = c;
}

// Offer one candidate per lane to the warp list; `thr` (warp-uniform) is the
// smallest key a new entry must beat and is raised as the list fills.
__device__ __forceinline__ void warp_list_offer(uint64_t& entry, uint64_t& thr, uint64_t c, int k,
                                                unsigned kmask, int lane) {
  unsigned pending = __ballot_sync(kFull, c > thr);
  while (pending) {
    const int src = __ffs(pending) - 1;
    pending &= pending - 1;
    const uint64_t cc = __shfl_sync(kFull, c, src);
    if (cc > thr) {
      warp_list_insert(entry, cc, kmask, lane);
      thr = __shfl_sync(kFull, entry, k - 1);
    }
  }
}

// Warp maximum of 64-bit keys: two 32-bit hardware reductions (the high word,
// then the low word among the lanes holding the highest high word) instead
// of five rounds of 64-bit shuffles.
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
  const uint32_t hi = (uint32_t)(v >> 32), lo = (uint32_t)v;
  const uint32_t hmax = __reduce_max_sync(kFull, hi);
  const uint32_t lmax = __reduce_max_sync(kFull, hi == hmax ? lo : 0u);
  return ((uint64_t)hmax << 32) | lmax;
}

// Top-k of the 32*NC candidates held by the warp (NC per lane), returned as
// a warp-distributed list (lane j holds the j-th largest, lanes >= k hold
// whatever).  Each lane first sorts its candidates in descending order (an
// odd-even transposition network, NC phases); then k rounds take the warp
// maximum of the lanes' first candidates, and the lane that held it (the
// candidates are distinct, so there is one) moves up its next one.  A round
// is two 32-bit reductions and one shift of the lane's list, instead of a
// search through all NC candidates.  Missing candidates are 0.  The lanes'
// arrays are consumed.
template <int NC>
__device__ __forceinline__ uint64_t warp_topk(uint64_t (&c)[NC], int k, int lane) {
#pragma unroll
  for (int ph = 0; ph < NC; ++ph) {
#pragma unroll
    for (int i = ph & 1; i + 1 < NC; i += 2) {
      const uint64_t a = c[i], b = c[i + 1];
      const bool sw = b > a;
      c[i] = sw ? b : a;
      c[i + 1] = sw ? a : b;
    }
  }
  uint64_t entry = 0ull;
  for (int r = 0; r < k; ++r) {
    const uint64_t w = warp_max_u64(c[0]);
    if (lane == r) entry = w;
    const bool mine = c[0] == w;
#pragma unroll
    for (int i = 0; i + 1 < NC; ++i) c[i] = mine ? c[i + 1] : c[i];
    c[NC - 1] = mine ? 0ull : c[NC - 1];
  }
  return entry;
}

}  // namespace tsd
