// Host-side helpers shared by the C entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tsd.h"

namespace tsd {

// Non-null and 16-byte aligned.
inline bool ok_ptr(const void* p) { return p != nullptr && (((uintptr_t)p) & 15u) == 0; }

// Null, or 16-byte aligned.
inline bool ok_opt_ptr(const void* p) { return (((uintptr_t)p) & 15u) == 0; }

// Number of nodes of the full k-ary draft tree of depth S (root excluded),
// saturated at 2^20.
inline long tree_node_count(int S, int k) {
  long total = 0, level = 1;
  for (int s = 1; s <= S; ++s) {
    level *= k;
    if (level > (1l << 20)) level = 1l << 20;
    total += level;
    if (total > (1l << 20)) return 1l << 20;
  }
  return total;
}

// Status of the launches just made.
inline tsd_status cuda_status() {
  return cudaGetLastError() == cudaSuccess ? TSD_OK : TSD_ERR_CUDA;
}

inline long ceil_div(long a, long b) { return (a + b - 1) / b; }

}  // namespace tsd
