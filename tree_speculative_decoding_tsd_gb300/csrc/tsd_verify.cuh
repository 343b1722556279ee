// Shared declarations of the tree-verify attention paths.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "tsd.h"
#include "tsd_common.cuh"

namespace tsd {

// Kernel arguments of every verify path (passed by value).
struct VerifyArgs {
  const void* q;
  const void* kc;
  const void* vc;
  const int32_t* plen;
  const void* kt;
  const void* vt;
  const uint64_t* mask;
  void* out;
  float* lse;
  float* ws_o;    // [B][Hq][R][nsplit][dv] normalised partial outputs (fp32), or
  __nv_bfloat16* ws_ob;  // the same in bf16 (tcgen05 path of bf16 heads); one of the two is set
  float* ws_lse;  // [B][Hq][R][nsplit] log2-sum-exp of each partial
  int32_t* err;
  long long wait_cycles;   // budget of the tcgen05 kernels' pipeline waits (clock cycles)
  int B, R, Hq, Hkv, g, M, cap;
  int nsplit, split_len, nrg;
  int tree_split;  // 1: the tree tile is a split of its own (after the prefix splits)
  float qscale;   // softmax scale * log2(e): scores are kept in the log2 domain
  // paged cache (page_size > 0): kc/vc are page pools [num_pages][Hkv][page_size][d]
  // and key `pos` of request b lives in page page_table[b][pos / page_size]
  const int32_t* page_table;
  int max_pages, page_size, num_pages;
};

enum VerifyPathId { kPathGeneric = 0, kPathMma = 1, kPathTc = 2 };

struct VerifyPlan {
  int path;
  int rb;         // packed rows per CTA
  int nrg;        // row groups per KV head
  int nsplit;     // prefix splits (grid x); a request uses ceil(P / split_len)
  int split_len;
  int part_bf16;  // split partials stored in bf16 (1) or fp32 (0)
  int tree_split;  // the tree tile is a split of its own
  size_t ws_bytes;
};

// Fewer packed rows than this are not a dense contraction for the legacy
// mma.sync path: CUDA cores.
constexpr int kMmaMinRows = 64;
// The tcgen05 path puts the packed rows on the MMA N dimension (a multiple of
// 16), so it takes any count from 16 rows up.
constexpr int kTcMinRows = 16;

VerifyPlan plan_verify(const tsd_attn_desc& d);
bool launch_mma_path(const tsd_attn_desc& d, const VerifyArgs& a, const VerifyPlan& p,
                     cudaStream_t st);
bool launch_tc_path(const tsd_attn_desc& d, const VerifyArgs& a, const VerifyPlan& p,
                    cudaStream_t st);
bool launch_mla_tc_path(const tsd_attn_desc& d, const VerifyArgs& a, const VerifyPlan& p,
                        cudaStream_t st);
bool tc_path_available();

namespace {

// Row of key `pos` of (request b, KV head hk) in the cache, or in the page
// pool for a paged cache; -1 for a page index outside the pool (the caller
// reports TSD_DEV_ERR_BAD_PAGE and never dereferences it).
__device__ __forceinline__ long kv_row(const VerifyArgs& a, int b, int hk, int pos) {
  if (a.page_size == 0) return ((long)b * a.Hkv + hk) * a.cap + pos;
  const int pg = a.page_table[(long)b * a.max_pages + pos / a.page_size];
  if (pg < 0 || pg >= a.num_pages) return -1;
  return ((long)pg * a.Hkv + hk) * a.page_size + pos % a.page_size;
}

// First row of a 128-key prefix tile in a page pool (a tile never crosses a
// page: page sizes are multiples of 128); a page outside the pool is reported
// and row 0 is returned so the copy stays in bounds.  Kept out of line so the
// contiguous path's TMA issue loop is unchanged.
__device__ __noinline__ int paged_tile_row(const VerifyArgs& a, int b, int hk, int pos) {
  const long row = kv_row(a, b, hk, pos);
  if (row < 0) {
    report_error(a.err, TSD_DEV_ERR_BAD_PAGE, b);
    return 0;
  }
  return (int)row;
}

template <typename T> __device__ __forceinline__ T cvt_out(float x);
template <> __device__ __forceinline__ float cvt_out<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// NV consecutive elements (NV = 2, 4, 8 or 16) at p, 4 * NV-byte or
// 2 * NV-byte aligned: vector loads and stores.
template <int NV>
__device__ __forceinline__ void load_vec(const float* p, float (&x)[NV]) {
  if constexpr (NV == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x; x[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < NV; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + i);
      x[i] = v.x; x[i + 1] = v.y; x[i + 2] = v.z; x[i + 3] = v.w;
    }
  }
}
template <int NV>
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float (&x)[NV]) {
  constexpr int W = NV >= 8 ? 8 : NV;                 // bf16 per load
#pragma unroll
  for (int i = 0; i < NV; i += W) {
    uint32_t w[W / 2];
    if constexpr (W == 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(p + i);
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (W == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(p + i);
      w[0] = v.x; w[1] = v.y;
    } else {
      w[0] = *reinterpret_cast<const uint32_t*>(p + i);
    }
#pragma unroll
    for (int j = 0; j < W / 2; ++j) {
      x[i + 2 * j] = __uint_as_float(w[j] << 16);
      x[i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
}
template <int NV>
__device__ __forceinline__ void store_vec(float* p, const float (&x)[NV]) {
  if constexpr (NV == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
  } else {
#pragma unroll
    for (int i = 0; i < NV; i += 4)
      *reinterpret_cast<float4*>(p + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
  }
}
template <int NV>
__device__ __forceinline__ void store_vec(__nv_bfloat16* p, const float (&x)[NV]) {
  uint32_t w[NV / 2];
#pragma unroll
  for (int j = 0; j < NV / 2; ++j) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(x[2 * j], x[2 * j + 1]);
    w[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
  if constexpr (NV == 2) {
    *reinterpret_cast<uint32_t*>(p) = w[0];
  } else if constexpr (NV == 4) {
    *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int i = 0; i < NV / 2; i += 4)
      *reinterpret_cast<uint4*>(p + 2 * i) = make_uint4(w[i], w[i + 1], w[i + 2], w[i + 3]);
  }
}

// Splits that hold work for a request with prefix P: the prefix splits, and
// the tree tile either in the last of them or (tree_split) after them.
__device__ __forceinline__ int verify_splits(const VerifyArgs& a, int P) {
  const int npre = P > 0 ? (P + a.split_len - 1) / a.split_len : 0;
  return a.tree_split ? npre + 1 : max(npre, 1);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// acc += w_(j+u) * O_(j+u) for u < m (m <= U, in increasing u), lane-strided
// partials of DV = 32 * NV values at src[(j + u) * DV + 32 * t]; the weights
// sit on lanes j..j+m-1 of wl.  All loads are issued before the products.
__device__ __forceinline__ float part_f32(float x) { return x; }
__device__ __forceinline__ float part_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <int U, int NV, typename PT>
__device__ __forceinline__ void merge_batch(float (&acc)[NV], const PT* src, float wl, int j,
                                            int m) {
  float x[U][NV];
#pragma unroll
  for (int u = 0; u < U; ++u)
#pragma unroll
    for (int t = 0; t < NV; ++t)
      x[u][t] = u < m ? part_f32(src[(j + u) * NV * 32 + 32 * t]) : 0.f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const float w = __shfl_sync(kFull, wl, (j + u) & 31);
    if (u < m) {
#pragma unroll
      for (int t = 0; t < NV; ++t) acc[t] = fmaf(w, x[u][t], acc[t]);
    }
  }
}

// Merge the nsb split partials of one output row (b, r, h) with one warp.
// Each split s left a normalised output O_s and its log2-sum-exp L_s; the
// result is sum_s 2^(L_s - L) O_s with L = log2 sum_s 2^(L_s).
template <typename T, int DV, typename PT>
__device__ __forceinline__ void merge_splits(const VerifyArgs& a, const PT* parts, int b, int r,
                                             int h, int nsb, int lane) {
  const long row = ((long)b * a.R + r) * a.Hq + h;
  const long base = (((long)b * a.Hq + h) * a.R + r) * a.nsplit;
  constexpr int NV = DV / 32;
  constexpr int kB = NV > 4 ? 4 : 8;          // partials per batch of loads
  constexpr int kF = NV > 4 ? 4 : 16;         // splits of the one-round-trip path
  // A row of at most kF splits (the common case) has its partials' loads
  // issued together with the log-sum-exp loads, before the weights are known:
  // one memory round trip instead of two.  Lane j takes the NV consecutive
  // dims NV*j .. NV*j+NV-1 (vector loads and stores).
  if (nsb <= kF) {
    float x[kF][NV];
#pragma unroll
    for (int u = 0; u < kF; ++u) {
      if (u < nsb) {
        load_vec<NV>(parts + (base + u) * DV + NV * lane, x[u]);
      } else {
#pragma unroll
        for (int t = 0; t < NV; ++t) x[u][t] = 0.f;
      }
    }
    const float l = lane < nsb ? a.ws_lse[base + lane] : -INFINITY;
    float mx = l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    const float tot = mx + log2f(warp_sum(lane < nsb ? exp2f(l - mx) : 0.f));
    const float wl = lane < nsb ? exp2f(l - tot) : 0.f;
    float acc[NV];
#pragma unroll
    for (int t = 0; t < NV; ++t) acc[t] = 0.f;
#pragma unroll
    for (int u = 0; u < kF; ++u) {
      const float w = __shfl_sync(kFull, wl, u);
      if (u < nsb) {
#pragma unroll
        for (int t = 0; t < NV; ++t) acc[t] = fmaf(w, x[u][t], acc[t]);
      }
    }
    store_vec<NV>((T*)a.out + row * DV + NV * lane, acc);
    if (lane == 0) a.lse[row] = tot * 0.69314718055994531f;
    return;
  }
  // L = log2 sum_s 2^(L_s): maximum, then per-lane partial sums (split s on
  // lane s % 32, in increasing s) reduced across the warp
  const float l0 = lane < nsb ? a.ws_lse[base + lane] : -INFINITY;
  float mx = l0;
  for (int s = lane + 32; s < nsb; s += 32) mx = fmaxf(mx, a.ws_lse[base + s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  float sum = lane < nsb ? exp2f(l0 - mx) : 0.f;
  for (int s = lane + 32; s < nsb; s += 32) sum += exp2f(a.ws_lse[base + s] - mx);
  sum = warp_sum(sum);
  const float tot = mx + log2f(sum);
  float acc[NV];
#pragma unroll
  for (int t = 0; t < NV; ++t) acc[t] = 0.f;
  // acc = sum over s in increasing order of fma(w_s, O_s, acc); lane j of a
  // round of 32 splits holds w_(s0+j).  Batches of kB partials have their
  // loads in flight together; the rest is one predicated batch of kB or kB/2
  for (int s0 = 0; s0 < nsb; s0 += 32) {
    const int n = min(32, nsb - s0);
    const float wl = lane >= n ? 0.f : exp2f((s0 == 0 ? l0 : a.ws_lse[base + s0 + lane]) - tot);
    const PT* src = parts + (base + s0) * DV + lane;
    int j = 0;
    for (; j + kB <= n; j += kB) merge_batch<kB, NV>(acc, src, wl, j, kB);
    if (n - j > kB / 2) merge_batch<kB, NV>(acc, src, wl, j, n - j);
    else if (n - j > 0) merge_batch<kB / 2, NV>(acc, src, wl, j, n - j);
  }
#pragma unroll
  for (int t = 0; t < NV; ++t) ((T*)a.out)[row * DV + lane + 32 * t] = cvt_out<T>(acc[t]);
  if (lane == 0) a.lse[row] = tot * 0.69314718055994531f;
}

// Split merge: one warp per output row ((b*R + r)*Hq + h) of a request whose
// prefix spans several splits (a request held by one split is written
// directly by the attention kernel), spread over the
// whole GPU (merging in the last CTA of each request and head instead left
// one CTA with a serial tail of dependent loads: 10% slower attention on every
// workload).  It is launched with ordinary stream serialisation: launched
// early next to a multi-wave attention grid, its CTAs slowed the following
// kernels (5% on the batched step).
// PT: element type of the split partials (float, or bf16 on the tcgen05 path
// of bf16 heads).
template <typename T, int DV, typename PT = float>
__global__ void __launch_bounds__(128)
verify_combine_kernel(const __grid_constant__ VerifyArgs a) {
  grid_dependency_sync();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long row = (long)blockIdx.x * 4 + warp;
  if (row >= (long)a.B * a.R * a.Hq) return;
  const int b = (int)(row / ((long)a.R * a.Hq));
  const int r = (int)((row / a.Hq) % a.R);
  const int h = (int)(row % a.Hq);
  const int P = min(max(a.plen[b], 0), a.cap);
  const int nsb = verify_splits(a, P);
  if (nsb == 1) return;   // a request held by one split wrote its output directly
  const PT* parts;
  if constexpr (sizeof(PT) == 2) parts = a.ws_ob;
  else parts = a.ws_o;
  merge_splits<T, DV, PT>(a, parts, b, r, h, nsb, lane);
}

}  // namespace

}  // namespace tsd
