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

// Kernel launches.  launch() sets programmatic stream serialisation: the
// kernel may be scheduled while the previous kernel on the stream is still
// finishing (each kernel calls grid_dependency_sync before touching global
// memory), which hides the launch gap between the step's small kernels, also
// inside a captured graph; after anything but a kernel (a copy, an event) the
// launch is ordered as usual.  launch_plain() keeps ordinary serialisation.
// Errors surface through cuda_status().
template <typename... KArgs, typename... Args>
inline void launch_with(bool programmatic, void (*kern)(KArgs...), dim3 grid, dim3 block,
                        size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  cudaLaunchKernelEx(&cfg, kern, args...);
}
template <typename... KArgs, typename... Args>
inline void launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                   Args... args) {
  launch_with(true, kern, grid, block, smem, st, args...);
}
template <typename... KArgs, typename... Args>
inline void launch_plain(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t st, Args... args) {
  launch_with(false, kern, grid, block, smem, st, args...);
}

}  // namespace tsd
