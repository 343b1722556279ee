// Vocabulary scan: per-chunk top-k (or argmax) of fp32 rows.
//
// Each row of length V is cut into `nchunk` chunks of `chunk_len` elements;
// one 256-thread CTA scans one chunk with 16-byte streaming loads and writes
// the chunk's k best candidates (64-bit keys, see make_cand) to
// out[row][chunk][0..k).  A second, per-request kernel merges the chunk lists:
// the row's top-k is the top-k of the union of its chunks' top-k lists, which
// is exact because candidates are distinct.
//
// Top-k mode keeps one sorted list per warp, one entry per lane.  An element
// is offered to the list only when it beats the list threshold, which is the
// larger of the warp's own k-th entry and a CTA-wide threshold published in
// shared memory: k entries at least that large already exist, and keys are
// distinct, so nothing at or below it can be in the chunk's top-k.  With
// random rows almost every element is rejected by one compare.
// Argmax mode (k = 1) keeps one running maximum per thread.
#pragma once

#include "tsd_common.cuh"

namespace tsd {

constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;
// Partitioning assumes the GB300's 152 SMs with 8 resident scan CTAs each.
constexpr int kScanTargetCtas = 152 * 8;
constexpr int kScanMinChunk = 2048;
// A row's chunk lists hold at most this many candidates, so the merge in the
// consumer kernel reads a short, fixed-size list per row.
constexpr int kScanMaxCand = 256;

struct ScanGeom {
  int nchunk;
  int chunk_len;  // multiple of 256 elements
};

inline ScanGeom scan_geometry(long rows, int V, int k) {
  long per_row = (kScanTargetCtas + rows - 1) / rows;
  long max_chunks = (V + kScanMinChunk - 1) / kScanMinChunk;
  if (per_row > max_chunks) per_row = max_chunks;
  if (per_row > kScanMaxCand / k) per_row = kScanMaxCand / k;
  if (per_row < 1) per_row = 1;
  long len = (V + per_row - 1) / per_row;
  len = (len + 255) / 256 * 256;
  ScanGeom g;
  g.chunk_len = (int)len;
  g.nchunk = (int)((V + len - 1) / len);
  return g;
}

__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }

template <bool kArgmax>
__global__ void __launch_bounds__(kScanThreads)
vocab_scan_kernel(const float* __restrict__ x, int V, int k, int nchunk, int chunk_len,
                  uint64_t* __restrict__ out) {
  __shared__ uint64_t s_list[kScanWarps][32];
  __shared__ unsigned long long s_thr;

  const long cta = blockIdx.x;
  const long row = cta / nchunk;
  const int chunk = (int)(cta - row * nchunk);
  const int c0 = chunk * chunk_len;
  const int c1 = min(V, c0 + chunk_len);
  const float* xr = x + row * (long)V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Elements [c0, a0) and [a1, c1) are read one by one; [a0, a1) as float4.
  // x itself is 16-byte aligned, so alignment depends on row * V + index.
  const int mis = (int)((row * (long)V + c0) & 3);
  int a0 = c0 + ((4 - mis) & 3);
  if (a0 > c1) a0 = c1;
  const int nvec = (c1 - a0) >> 2;
  const int a1 = a0 + nvec * 4;
  const float4* xv = reinterpret_cast<const float4*>(xr + a0);

  if (kArgmax) {
    // Each thread visits its elements in increasing index order and keeps the
    // first maximum (strict >); threads are then merged by (value, id) keys.
    float bx = -INFINITY;
    int bi = -1;
    auto take = [&](float x, int i) {
      if (x > bx || bi < 0) { bx = x; bi = i; }
    };
    for (int i = c0 + tid; i < a0; i += kScanThreads) take(xr[i], i);
    int v = tid;
    for (; v + 3 * kScanThreads < nvec; v += 4 * kScanThreads) {
      float4 f[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) f[u] = ld_stream(xv + v + u * kScanThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i0 = a0 + 4 * (v + u * kScanThreads);
        take(f[u].x, i0); take(f[u].y, i0 + 1); take(f[u].z, i0 + 2); take(f[u].w, i0 + 3);
      }
    }
    {
      float4 f[3];
      bool have[3];
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        have[u] = v + u * kScanThreads < nvec;
        if (have[u]) f[u] = ld_stream(xv + v + u * kScanThreads);
      }
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        if (!have[u]) continue;
        const int i0 = a0 + 4 * (v + u * kScanThreads);
        take(f[u].x, i0); take(f[u].y, i0 + 1); take(f[u].z, i0 + 2); take(f[u].w, i0 + 3);
      }
    }
    for (int i = a1 + tid; i < c1; i += kScanThreads) take(xr[i], i);
    uint64_t best = bi < 0 ? 0ull : make_cand(bx, (uint32_t)bi);
    best = warp_max_u64(best);
    if (lane == 0) s_list[warp][0] = best;
    __syncthreads();
    if (warp == 0) {
      uint64_t c = lane < kScanWarps ? s_list[lane][0] : 0;
      c = warp_max_u64(c);
      if (lane == 0) out[cta] = c;
    }
    return;
  }

  // ---- top-k mode: warp lists -------------------------------------------
  if (tid == 0) s_thr = 0ull;
  __syncthreads();
  const unsigned kmask = (k >= 32) ? kFull : ((1u << k) - 1u);
  uint64_t entry = 0, thr = 0;

  // scalar edges: the whole warp offers one element per lane at a time
  for (int base = c0 + warp * 32; base < a0; base += kScanThreads) {
    const int i = base + lane;
    const uint64_t c = i < a0 ? make_cand(xr[i], i) : 0ull;
    warp_list_offer(entry, thr, c, k, kmask, lane);
  }
  for (int base = a1 + warp * 32; base < c1; base += kScanThreads) {
    const int i = base + lane;
    const uint64_t c = i < c1 ? make_cand(xr[i], i) : 0ull;
    warp_list_offer(entry, thr, c, k, kmask, lane);
  }

  // main loop: every lane of the CTA takes 4 float4 per trip (warp-aligned so
  // that the whole warp runs the same number of trips)
  const int nvec_w = (nvec + 31) & ~31;
  for (int v0 = warp * 32; v0 < nvec_w; v0 += 4 * kScanThreads) {
    float4 f[4];
    bool have[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + u * kScanThreads + lane;
      have[u] = v < nvec;
      f[u] = have[u] ? ld_stream(xv + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // quick reject: nothing below the threshold's value can enter the list
    const float thr_v = thr == 0ull ? -INFINITY : cand_val(thr);
    float hi = -INFINITY;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (!have[u]) continue;
      hi = fmaxf(hi, fmaxf(fmaxf(f[u].x, f[u].y), fmaxf(f[u].z, f[u].w)));
    }
    if (v0 == warp * 32) {
      // first trip: the list is empty or nearly so and almost everything would
      // be offered -- take the top-k of this trip plus the current list in k
      // warp-wide rounds instead
      uint64_t cb[17];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t i0 = (uint32_t)(a0 + 4 * (v0 + u * kScanThreads + lane));
        cb[4 * u + 0] = have[u] ? make_cand(f[u].x, i0) : 0ull;
        cb[4 * u + 1] = have[u] ? make_cand(f[u].y, i0 + 1) : 0ull;
        cb[4 * u + 2] = have[u] ? make_cand(f[u].z, i0 + 2) : 0ull;
        cb[4 * u + 3] = have[u] ? make_cand(f[u].w, i0 + 3) : 0ull;
      }
      cb[16] = lane < k ? entry : 0ull;
      entry = warp_topk<17>(cb, k, lane);
      thr = __shfl_sync(kFull, entry, k - 1);
      if (lane == 0) atomicMax(&s_thr, (unsigned long long)thr);
    } else if (__any_sync(kFull, hi >= thr_v)) {
      // only elements at or above the threshold value are offered: one warp
      // round per pending element of the busiest lane, per float4
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
        unsigned pend = 0;
        if (have[u]) {
#pragma unroll
          for (int i = 0; i < 4; ++i) pend |= (e[i] >= thr_v) ? (1u << i) : 0u;
        }
        const uint32_t i0 = (uint32_t)(a0 + 4 * (v0 + u * kScanThreads + lane));
        while (__any_sync(kFull, pend != 0)) {
          uint64_t cnd = 0ull;
          if (pend) {
            const int i = __ffs(pend) - 1;
            pend &= pend - 1;
            const float x = i == 0 ? e[0] : i == 1 ? e[1] : i == 2 ? e[2] : e[3];
            cnd = make_cand(x, i0 + i);
          }
          warp_list_offer(entry, thr, cnd, k, kmask, lane);
        }
      }
      // publish the warp's k-th entry; adopt a larger CTA-wide threshold
      if (lane == 0) atomicMax(&s_thr, (unsigned long long)thr);
    }
    const uint64_t shared_thr = *(volatile unsigned long long*)&s_thr;
    thr = shared_thr > thr ? shared_thr : thr;
  }

  // merge the warps' lists in warp 0
  s_list[warp][lane] = entry;
  __syncthreads();
  if (warp == 0) {
    uint64_t cm[kScanWarps];
#pragma unroll
    for (int w = 0; w < kScanWarps; ++w) cm[w] = lane < k ? s_list[w][lane] : 0ull;
    entry = warp_topk<kScanWarps>(cm, k, lane);
    if (lane < k) out[cta * k + lane] = entry;
  }
}

}  // namespace tsd
