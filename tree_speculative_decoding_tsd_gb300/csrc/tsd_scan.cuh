// Vocabulary scan: per-chunk top-k (or argmax) of fp32 rows.
//
// Each row of length V is cut into `nchunk` chunks of `chunk_len` elements;
// one 256-thread CTA scans one chunk with 16-byte loads and writes the
// chunk's k best candidates (64-bit keys, see make_cand) to
// out[row][chunk][0..k).  A second, per-request kernel merges the chunk lists:
// the row's top-k is the top-k of the union of its chunks' top-k lists, which
// is exact because candidates are distinct.
//
// Top-k mode reads the chunk once from HBM; each thread keeps its best
// element (value and index) and its second largest value.  The k best of the
// 256 thread candidates are the chunk's top-k whenever no thread's second
// value reaches the k-th of them (every other element is then below its
// thread's best and below the k-th candidate) -- the common case, which needs
// no second look at the data.  Otherwise (two top-k elements in one thread,
// ties, or fewer than k elements) the k-th candidate's value T is a cut-off:
// k distinct elements are >= T, so the top-k is >= T and only threads whose
// best reaches T hold any of it; the warp re-reads just those threads'
// elements (from L2, where the first pass left them) and offers the ones >= T
// to a sorted warp list, and the CTA merges its eight warp lists.  NaN
// entries are never selected.
// Top-k mode also checks that the row is a probability vector as the tree
// rule needs it (no value above 1, no NaN) and reports a violation in the
// caller's error word.
// Argmax mode (k = 1) keeps one running maximum per thread.
#pragma once

#include "tsd_common.cuh"

namespace tsd {

constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;
// Partitioning assumes the GB300's 152 SMs with this many resident CTAs of
// each mode (the launch bounds below enforce the register budget for it).
constexpr int kScanSms = 152;
constexpr int kScanArgmaxPerSm = 8;
constexpr int kScanTopkPerSm = 4;
constexpr int kScanMinChunk = 2048;
// A row's chunk lists hold at most this many candidates, so the merge in the
// consumer kernel reads a short, fixed-size list per row.
constexpr int kScanMaxCand = 256;

struct ScanGeom {
  int nchunk;
  int chunk_len;  // multiple of 256 elements
  int one_wave;   // every CTA of the grid is resident at once
};

// Chunks per row: the count that minimises (waves of CTAs) x (chunk length +
// fixed per-chunk cost), so that the last wave is not a small tail.  Host
// code, no device query: workspace sizes follow from it and must not depend
// on the GPU.
inline ScanGeom scan_geometry(long rows, int V, int k, bool argmax) {
  const long slots = (long)kScanSms * (argmax ? kScanArgmaxPerSm : kScanTopkPerSm);
  const double overhead = argmax ? 512.0 : 4096.0;  // in element-times
  long pmax = (V + kScanMinChunk - 1) / kScanMinChunk;
  if (pmax > kScanMaxCand / k) pmax = kScanMaxCand / k;
  if (pmax < 1) pmax = 1;
  long best_p = 1;
  double best_t = 1e300;
  for (long p = 1; p <= pmax; ++p) {
    const long waves = (rows * p + slots - 1) / slots;
    const double t = (double)waves * ((double)V / (double)p + overhead);
    if (t < best_t * 0.999) { best_t = t; best_p = p; }
  }
  long len = (V + best_p - 1) / best_p;
  len = (len + 255) / 256 * 256;
  ScanGeom g;
  g.chunk_len = (int)len;
  g.nchunk = (int)((V + len - 1) / len);
  g.one_wave = rows * g.nchunk <= slots ? 1 : 0;
  return g;
}

__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }

// max(a, b, c) that returns NaN if any operand is NaN (three-operand
// max.NaN.f32, sm_100 and later)
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <bool kArgmax>
__global__ void __launch_bounds__(kScanThreads, kArgmax ? kScanArgmaxPerSm : kScanTopkPerSm)
vocab_scan_kernel(const float* __restrict__ x, int V, int k, int nchunk, int chunk_len,
                  uint64_t* __restrict__ out, int prefetch, int32_t* err, int rows_per_req) {
  __shared__ uint64_t s_list[kScanWarps][32];
  __shared__ uint64_t s_key[kScanThreads];
  __shared__ uint64_t s_wk;

  const long cta = blockIdx.x;
  const long row = cta / nchunk;
  const int chunk = (int)(cta - row * nchunk);
  const int c0 = chunk * chunk_len;
  const int c1 = min(V, c0 + chunk_len);
  const float* xr = x + row * (long)V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // a grid of one wave is resident while the previous kernel finishes: its
  // chunk is brought into L2 meanwhile (later waves would only add traffic)
  if (prefetch && tid == 0) prefetch_l2(xr + c0, (long)(c1 - c0) * 4);
  grid_dependency_sync();

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

  // ---- top-k mode -------------------------------------------------------
  // pass 1: stream the chunk once.  Each thread keeps its best element (the
  // largest value, its first index on ties: the candidate order), the second
  // largest value among its elements, and a maximum that keeps NaN (for the
  // range check); NaN is never taken.  (Eight 16-byte loads in flight per
  // thread: with about three CTAs per SM that keeps enough bytes in flight to
  // stream at HBM speed.)  A thread's elements are visited in increasing
  // index order: its front edge element, its float4s, its back edge element.
  float m = -INFINITY, m2 = -INFINITY, mn = -INFINITY;
  int mi = -1;
  auto take = [&](float x, int i) {
    const bool gt = x > m;
    m2 = gt ? m : fmaxf(m2, x);
    mi = gt ? i : mi;
    m = gt ? x : m;
  };
  if (c0 + tid < a0) {
    const float x = xr[c0 + tid];
    take(x, c0 + tid);
    mn = max3_nan(mn, x, -INFINITY);
  }
  {
    constexpr int U = 8;
    int v = tid;
    for (; v + (U - 1) * kScanThreads < nvec; v += U * kScanThreads) {
      float4 f[U];
#pragma unroll
      for (int u = 0; u < U; ++u) f[u] = __ldg(xv + v + u * kScanThreads);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i0 = a0 + 4 * (v + u * kScanThreads);
        take(f[u].x, i0); take(f[u].y, i0 + 1); take(f[u].z, i0 + 2); take(f[u].w, i0 + 3);
        mn = max3_nan(mn, max3_nan(f[u].x, f[u].y, f[u].z), f[u].w);
      }
    }
    float4 f[U - 1];
#pragma unroll
    for (int u = 0; u < U - 1; ++u)
      f[u] = v + u * kScanThreads < nvec ? __ldg(xv + v + u * kScanThreads)
                                         : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
    for (int u = 0; u < U - 1; ++u) {
      const int i0 = a0 + 4 * (v + u * kScanThreads);
      take(f[u].x, i0); take(f[u].y, i0 + 1); take(f[u].z, i0 + 2); take(f[u].w, i0 + 3);
      mn = max3_nan(mn, max3_nan(f[u].x, f[u].y, f[u].z), f[u].w);
    }
  }
  if (a1 + tid < c1) {
    const float x = xr[a1 + tid];
    take(x, a1 + tid);
    mn = max3_nan(mn, x, -INFINITY);
  }
  // a value above 1 (or NaN) breaks the score order the tree build relies on
  if (err != nullptr && __any_sync(kFull, !(mn <= 1.0f)) && lane == 0)
    report_error(err, TSD_DEV_ERR_BAD_PROBS, (int)(row / rows_per_req));

  // The k best of the 256 thread candidates, in order (warp 0, k rounds of a
  // warp maximum).  They are the chunk's top-k unless a thread holds a second
  // element that could rank among them (its second largest value reaches the
  // k-th candidate's value) or fewer than k threads hold an element: every
  // other element is below its thread's best and below the k-th candidate.
  s_key[tid] = mi >= 0 ? make_cand(m, (uint32_t)mi) : 0ull;
  __syncthreads();
  if (warp == 0) {
    uint64_t c[kScanThreads / 32];
#pragma unroll
    for (int j = 0; j < kScanThreads / 32; ++j) c[j] = s_key[j * 32 + lane];
    const uint64_t best = warp_topk<kScanThreads / 32>(c, k, lane);
    const uint64_t wk = __shfl_sync(kFull, best, k - 1);
    if (lane < k) s_key[lane] = best;           // (all reads of s_key above are done)
    if (lane == 0) s_wk = wk;
  }
  __syncthreads();
  const uint64_t wk = s_wk;
  const bool more = wk == 0ull || m2 >= cand_val(wk);
  if (!__syncthreads_or(more)) {
    if (warp == 0 && lane < k) out[cta * k + lane] = s_key[lane];
    return;
  }

  // Otherwise the rescans: cut-off T = the k-th candidate's value (k
  // distinct elements are >= T, so the chunk's top-k is >= T).
  const float cut = wk == 0ull ? -INFINITY : cand_val(wk);

  // the (at most 3 + 3) scalar edge elements are offered to the warp list directly
  const unsigned kmask = (k >= 32) ? kFull : ((1u << k) - 1u);
  uint64_t entry = 0, thr = 0;
  for (int base = c0 + warp * 32; base < a0; base += kScanThreads) {
    const int i = base + lane;
    const float x = i < a0 ? xr[i] : 0.f;
    const uint64_t c = (i < a0 && x == x) ? make_cand(x, i) : 0ull;
    warp_list_offer(entry, thr, c, k, kmask, lane);
  }
  for (int base = a1 + warp * 32; base < c1; base += kScanThreads) {
    const int i = base + lane;
    const float x = i < c1 ? xr[i] : 0.f;
    const uint64_t c = (i < c1 && x == x) ? make_cand(x, i) : 0ull;
    warp_list_offer(entry, thr, c, k, kmask, lane);
  }

  // pass 2: the warp re-reads the elements of its threads whose maximum
  // reaches T, all of them at once (one round trip per 32 float4s): item q
  // is float4 q % cmax of the (q / cmax)-th such thread
  const unsigned act = __ballot_sync(kFull, m >= cut);
  const int cmax = (nvec + kScanThreads - 1) / kScanThreads;   // float4s per thread, at most
  const int items = __popc(act) * cmax;
  for (int q0 = 0; q0 < items; q0 += 32) {
    const int q = q0 + lane;
    int vi = nvec;   // the float4 of item q, or nvec for none
    if (q < items) {
      const int a = q / cmax;
      vi = warp * 32 + (int)__fns(act, 0, a + 1) + (q - a * cmax) * kScanThreads;
    }
    const bool have = vi < nvec;
    const float4 f = have ? __ldg(xv + vi) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float e[4] = {f.x, f.y, f.z, f.w};
    unsigned pend = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) pend |= (have && e[i] >= cut) ? (1u << i) : 0u;
    const uint32_t i0 = (uint32_t)(a0 + 4 * vi);
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
