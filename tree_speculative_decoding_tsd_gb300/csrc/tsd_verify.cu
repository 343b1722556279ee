// tsd_tree_verify_attn: branch-aware tree attention over the shared prefix
// KV cache plus each node's own ancestors in the scratch pad.
//
// Source: "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4"
// (review), research gap item 1 (a candidate must see only its own
// ancestors, never another branch; batch order and logical dependency
// differ), "How it works" step 3 (A-B-B sees A and A-B, A-C sees only A) and
// step 5 (all chains are verified in one target pass).
//
// Work decomposition (flash-decoding): the query rows of one KV head -- all
// R tree rows x g query heads of the group ("packed rows") -- share every
// prefix key, so a CTA takes a group of packed rows, one KV head and one
// split of the prefix, and reads each prefix key once for all its rows.  The
// CTA that owns the last split of a request also takes the R scratch-pad rows,
// masked per packed row by the ancestor bitmask.  Partial results (normalised
// output and log2-sum-exp per split) are merged by verify_combine_kernel; with
// one split the attention kernel writes the final output directly.
//
// Paths:
//   generic (this file): CUDA-core fp32 arithmetic, one warp per key, lanes
//     split the head dim, warp-shuffle reductions for q.k; any dtype/dims.
//     Used for fp32 inputs (never TF32) and for bf16 heads with too few packed
//     rows for a tensor-core tile (fewer than 16 on the tcgen05 path).
//   tc (tsd_verify_tc.cu): bf16 GQA heads, head dim 128, >= 16 packed rows:
//     tcgen05 MMAs with TMEM accumulators, TMA-fed K/V ring (the default).
//     Latent heads (bf16, dk 576 / dv 512, V = K[:, :512]) with >= 64 packed
//     rows take the tcgen05 kernel of tsd_verify_mla.cu.
//   mma (tsd_verify_mma.cu): bf16 GQA heads (head dim 64 or 128) with >= 64
//     packed rows on the legacy warp-level mma.sync tensor-core path.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include <cuda_bf16.h>

#include "tsd_common.cuh"
#include "tsd_host.h"
#include "tsd_verify.cuh"

namespace tsd {
namespace {

constexpr int kGenThreads = 128;
constexpr int kGenWarps = kGenThreads / 32;

template <typename T> __device__ __forceinline__ float ldf(const T* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
// One CTA: packed rows [rg*RB, rg*RB+RB) of KV head hk of request b, prefix
// keys of split sp (and the tree rows if sp is the request's last split).
template <typename T, int DK, int DV, int RB, bool ALIAS>
__global__ void __launch_bounds__(kGenThreads)
verify_generic_kernel(const __grid_constant__ VerifyArgs a) {
  grid_dependency_sync();
  constexpr int NK = DK / 32, NV = DV / 32;
  __shared__ float sm_m[kGenWarps][RB], sm_l[kGenWarps][RB];
  __shared__ float sm_o[kGenWarps][RB][DV];

  const int sp = blockIdx.x;
  const int hk = blockIdx.y / a.nrg, rg = blockIdx.y % a.nrg;
  const int b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int P = min(max(a.plen[b], 0), a.cap);  // out-of-range lengths never read past the cache
  const int nsb = P > 0 ? (P + a.split_len - 1) / a.split_len : 1;
  if (sp >= nsb) return;
  const int k0 = sp * a.split_len, k1 = min(P, k0 + a.split_len);
  const bool with_tree = (sp == nsb - 1);

  float qv[RB][NK], o[RB][NV], m[RB], l[RB];
  uint64_t rmask[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    const int p = rg * RB + i;
    const bool valid = p < a.M;
    const int r = valid ? p / a.g : 0, h = hk * a.g + (valid ? p % a.g : 0);
    const T* qp = (const T*)a.q + (((long)b * a.R + r) * a.Hq + h) * DK;
#pragma unroll
    for (int t = 0; t < NK; ++t) qv[i][t] = valid ? ldf(qp + lane + 32 * t) * a.qscale : 0.f;
    rmask[i] = (valid && r > 0) ? a.mask[(long)b * a.R + r] : 0ull;
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int t = 0; t < NV; ++t) o[i][t] = 0.f;
  }
  const int nrows = min(RB, a.M - rg * RB);

  auto visit = [&](const T* kp, const T* vp, bool is_tree, int j) {
    float kv[NK], vv[NV];
#pragma unroll
    for (int t = 0; t < NK; ++t) kv[t] = ldf(kp + lane + 32 * t);
#pragma unroll
    for (int t = 0; t < NV; ++t) vv[t] = ldf(vp + lane + 32 * t);
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      if (i >= nrows) break;
      float d = 0.f;
#pragma unroll
      for (int t = 0; t < NK; ++t) d = fmaf(qv[i][t], kv[t], d);
      d = warp_sum(d);
      if (is_tree && j > 0 && !((rmask[i] >> (j - 1)) & 1ull)) continue;
      if (d > m[i]) {
        const float al = exp2f(m[i] - d);
        l[i] = fmaf(l[i], al, 1.f);
#pragma unroll
        for (int t = 0; t < NV; ++t) o[i][t] = fmaf(o[i][t], al, vv[t]);
        m[i] = d;
      } else {
        const float pr = exp2f(d - m[i]);
        l[i] += pr;
#pragma unroll
        for (int t = 0; t < NV; ++t) o[i][t] = fmaf(pr, vv[t], o[i][t]);
      }
    }
  };

  constexpr int vstride = ALIAS ? DK : DV;
  for (int j = k0 + warp; j < k1; j += kGenWarps) {
    const long row = kv_row(a, b, hk, j);
    if (row < 0) {   // page outside the pool: reported, never read
      if (lane == 0) report_error(a.err, TSD_DEV_ERR_BAD_PAGE, b);
      continue;
    }
    const T* kr = (const T*)a.kc + row * DK;
    visit(kr, ALIAS ? kr : (const T*)a.vc + row * DV, false, j);
  }
  if (with_tree) {
    const T* kt = (const T*)a.kt + ((long)b * a.R * a.Hkv + hk) * DK;
    const T* vt = ALIAS ? kt : (const T*)a.vt + ((long)b * a.R * a.Hkv + hk) * DV;
    for (int j = warp; j < a.R; j += kGenWarps)
      visit(kt + (long)j * a.Hkv * DK, vt + (long)j * a.Hkv * vstride, true, j);
  }

  // merge the four warps' running states
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    if (lane == 0) { sm_m[warp][i] = m[i]; sm_l[warp][i] = l[i]; }
#pragma unroll
    for (int t = 0; t < NV; ++t) sm_o[warp][i][lane + 32 * t] = o[i][t];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nrows * DV; idx += kGenThreads) {
    const int i = idx / DV, c = idx - i * DV;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kGenWarps; ++w) mx = fmaxf(mx, sm_m[w][i]);
    float lt = 0.f, ot = 0.f;
#pragma unroll
    for (int w = 0; w < kGenWarps; ++w) {
      const float wt = sm_m[w][i] == -INFINITY ? 0.f : exp2f(sm_m[w][i] - mx);
      lt = fmaf(sm_l[w][i], wt, lt);
      ot = fmaf(sm_o[w][i][c], wt, ot);
    }
    const float res = ot / lt;
    const float lse2 = mx + log2f(lt);
    const int p = rg * RB + i;
    const int r = p / a.g, h = hk * a.g + p % a.g;
    const long orow = ((long)b * a.R + r) * a.Hq + h;
    if (nsb == 1) {
      ((T*)a.out)[orow * DV + c] = cvt_out<T>(res);
      if (c == 0) a.lse[orow] = lse2 * 0.69314718055994531f;
    } else {
      const long prow = (((long)b * a.Hq + h) * a.R + r) * a.nsplit + sp;
      a.ws_o[prow * DV + c] = res;
      if (c == 0) a.ws_lse[prow] = lse2;
    }
  }
}

}  // namespace

// ---------------------------------------------------------------- planning --

// Path choice.  tsd_set_verify_path forces a path where it applies (the
// tests use it to check every path against the oracle); the default is the
// automatic choice below.
static std::atomic<int> g_forced_path{TSD_PATH_AUTO};
// Budget of the tcgen05 kernels' pipeline waits, in clock cycles (0 = default).
static std::atomic<long long> g_wait_budget{0};

static int choose_path(const tsd_attn_desc& d, int M) {
  const bool gqa_bf16 = d.dtype == TSD_BF16 && !d.v_aliases_k && d.dk == d.dv;
  const bool mma_ok = gqa_bf16 && (d.dk == 64 || d.dk == 128);
  const bool mla_bf16 = d.dtype == TSD_BF16 && d.v_aliases_k && d.dk == 576 && d.dv == 512;
  // tcgen05 with the packed rows on the MMA N dimension works from N = 16 up
  const bool tc_ok = ((gqa_bf16 && d.dk == 128 && M >= kTcMinRows) ||
                      (mla_bf16 && M >= kMmaMinRows)) && tc_path_available();
  switch (g_forced_path.load(std::memory_order_relaxed)) {
    case TSD_PATH_CUDA_CORE: return kPathGeneric;
    case TSD_PATH_MMA_SYNC: if (mma_ok) return kPathMma; break;
    case TSD_PATH_TCGEN05: if (tc_ok) return kPathTc; break;
    default: break;
  }
  if (tc_ok) return kPathTc;
  if (M < kMmaMinRows) return kPathGeneric;  // not a dense contraction
  if (mma_ok) return kPathMma;
  return kPathGeneric;
}

VerifyPlan plan_verify(const tsd_attn_desc& d) {
  VerifyPlan p{};
  const int M = d.R * (d.Hq / d.Hkv);
  p.path = choose_path(d, M);
  long ns;
  if (p.path == kPathTc && d.v_aliases_k) {
    // Splits only when the batch leaves the GPU short of CTAs (a split writes
    // fp32 partial outputs of 512 dims per packed row).
    // latent heads: 64 packed rows per CTA (the MMA N)
    p.nrg = (int)ceil_div(M, 64);
    p.rb = 64;
    const long units = (long)d.B * d.Hkv * p.nrg;
    ns = ceil_div(152L * 2, units);
    long len = ceil_div(ceil_div(d.cap, ns), 128) * 128;
    if (len < 512) len = 512;
    p.split_len = (int)len;
  } else if (p.path == kPathTc) {
    // packed rows on the MMA N dimension: at most 144 per CTA, multiple of 16
    p.nrg = (int)ceil_div(M, 144);
    // A grid that fills at most half the GPU with 256-key splits (a small
    // batch) takes twice the row groups: CTAs of fewer columns, a shorter
    // critical path (qwen-sized step 39.8 -> 38.8 us; the second CTA of a
    // tile finds it in L2).
    if ((long)d.B * d.Hkv * p.nrg * ceil_div(d.cap, 256) <= 76 && M >= 32) p.nrg *= 2;
    p.rb = (int)ceil_div(ceil_div(M, p.nrg), 16) * 16;
    // Splits.  A small batch takes about two waves of CTAs: splits of 256 to
    // 4096 keys, the shorter ones shortening the critical path (qwen-sized
    // step: 256-key splits 2.5 us faster than 512).  Once the batch has at
    // least 64 (request, KV head, row group) units, the split count ns
    // minimises the modelled time of full-length requests: waves of CTAs,
    // ceil(units * ns / 152), times the tiles of one CTA plus its set-up and
    // epilogue (about 4 tiles' worth).  For the batched workload (256 units of
    // <= 33 tiles) that is no split at all -- every CTA writes its output and
    // no merge runs -- and for long prefixes (128 units of 257 tiles) 7
    // splits, 6 full waves.  The split depends on B: results are
    // deterministic, but their rounding can differ between batch sizes.
    const long units = (long)d.B * d.Hkv * p.nrg;
    const long tiles = ceil_div(d.cap, 128);
    long len;
    if (units >= 64) {
      long best = -1, best_ns = 1;
      for (long n = 1; n <= 32 && n <= tiles; ++n) {
        const long per = ceil_div(tiles, n);
        const long cost = ceil_div(units * n, 152L) * (per + 4);
        if (best < 0 || cost < best) { best = cost; best_ns = n; }
      }
      len = ceil_div(tiles, best_ns) * 128;
    } else {
      ns = ceil_div(152L * 2, units);
      len = ceil_div(ceil_div(d.cap, ns), 128) * 128;  // whole 128-key tiles
      if (len < 256) len = 256;
      if (len > 4096) len = 4096;
    }
    p.split_len = (int)len;
  } else if (p.path == kPathMma) {
    // one warp per 16 packed rows, at most 8 warps per CTA, balanced groups
    const int nblk = (int)ceil_div(M, 16);
    p.nrg = (int)ceil_div(nblk, 8);
    p.rb = (int)ceil_div(nblk, p.nrg) * 16;
    ns = ceil_div(152L * 2, (long)d.Hkv * p.nrg);       // about two CTAs per SM for one request
    long len = ceil_div(d.cap, ns);
    len = ceil_div(len < 256 ? 256 : len, 64) * 64;       // whole 64-key tiles, >= 4 per split
    p.split_len = (int)len;
  } else {
    p.rb = d.dk > 128 ? 2 : 8;
    p.nrg = (int)ceil_div(M, p.rb);
    ns = ceil_div(152L * 4, (long)d.Hkv * p.nrg);
    const long max_ns = ceil_div(d.cap, 256);
    if (ns > max_ns) ns = max_ns;
    if (ns < 1) ns = 1;
    p.split_len = (int)ceil_div(d.cap, ns);
  }
  p.nsplit = (int)ceil_div(d.cap, p.split_len);
  // Short splits of the tcgen05 path of bf16 heads: the tree tile gets a split
  // (a CTA) of its own instead of lengthening the last prefix split, which is
  // the critical path when a split is a few tiles (qwen-sized step: 2 prefix
  // tiles per split).
  p.tree_split = (p.path == kPathTc && !d.v_aliases_k && p.nsplit > 1 && p.split_len <= 1024) ? 1 : 0;
  if (p.tree_split) ++p.nsplit;
  // The tcgen05 path of bf16 heads stores its split partials in bf16 (the
  // normalised partial output of a split is a convex combination of bf16
  // values; the merge weights stay fp32), halving the partials' traffic.
  p.part_bf16 = (p.path == kPathTc && !d.v_aliases_k) ? 1 : 0;
  const size_t pe = p.part_bf16 ? sizeof(__nv_bfloat16) : sizeof(float);
  p.ws_bytes = p.nsplit > 1
                   ? (size_t)d.B * d.Hq * d.R * p.nsplit * (d.dv * pe + sizeof(float))
                   : 0;
  return p;
}

template <typename T, int DK, int DV, int RB, bool ALIAS>
static void launch_generic(const VerifyArgs& a, const VerifyPlan& p, cudaStream_t st) {
  const dim3 grid(p.nsplit, a.Hkv * p.nrg, a.B);
  launch(verify_generic_kernel<T, DK, DV, RB, ALIAS>, dim3(grid), dim3(kGenThreads), 0, st, a);
  if (p.nsplit > 1) {
    const long rows = (long)a.B * a.R * a.Hq;
    launch_plain(verify_combine_kernel<T, DV>, dim3((unsigned)ceil_div(rows, 4)), dim3(128), 0,
                 st, a);
  }
}

bool launch_generic_path(const tsd_attn_desc& d, const VerifyArgs& a, const VerifyPlan& p,
                         cudaStream_t st) {
  const bool bf = d.dtype == TSD_BF16;
  if (d.v_aliases_k) {
    if (d.dk != 576 || d.dv != 512) return false;
    if (bf) launch_generic<__nv_bfloat16, 576, 512, 2, true>(a, p, st);
    else launch_generic<float, 576, 512, 2, true>(a, p, st);
    return true;
  }
  if (d.dk != d.dv) return false;
  if (d.dk == 128) {
    if (bf) launch_generic<__nv_bfloat16, 128, 128, 8, false>(a, p, st);
    else launch_generic<float, 128, 128, 8, false>(a, p, st);
    return true;
  }
  if (d.dk == 64) {
    if (bf) launch_generic<__nv_bfloat16, 64, 64, 8, false>(a, p, st);
    else launch_generic<float, 64, 64, 8, false>(a, p, st);
    return true;
  }
  return false;
}

}  // namespace tsd

using namespace tsd;

static bool desc_ok(const tsd_attn_desc* d) {
  if (d == nullptr) return false;
  if (d->B < 1 || d->B > 65535 || d->R < 1 || d->R > 65 || d->Hq < 1 || d->Hkv < 1 ||
      d->Hq % d->Hkv != 0 || d->cap < 1)
    return false;
  if (d->dtype != TSD_F32 && d->dtype != TSD_BF16) return false;
  if (!(d->scale > 0.f) || !(d->scale < 1e30f)) return false;
  const bool mla = d->v_aliases_k && d->dk == 576 && d->dv == 512;
  const bool gqa = !d->v_aliases_k && d->dk == d->dv && (d->dk == 64 || d->dk == 128);
  return mla || gqa;
}

extern "C" long long tsd_set_wait_budget(long long cycles) {
  return g_wait_budget.exchange(cycles > 0 ? cycles : 0);
}

extern "C" int tsd_set_verify_path(int path) {
  if (path < TSD_PATH_AUTO || path > TSD_PATH_TCGEN05) return -1;
  return g_forced_path.exchange(path);
}

extern "C" size_t tsd_verify_workspace_size(const tsd_attn_desc* d) {
  if (!desc_ok(d)) return 0;
  return plan_verify(*d).ws_bytes;
}

static tsd_status verify_impl(const tsd_attn_desc* d, const void* q, const void* kcache,
                              const void* vcache, const int32_t* page_table, int max_pages,
                              int page_size, int num_pages, const int32_t* prefix_len,
                              const void* ktree, const void* vtree, const uint64_t* mask,
                              void* out, float* lse, void* ws, size_t ws_bytes, int32_t* err,
                              tsd_stream_t stream) {
  if (!desc_ok(d)) return TSD_ERR_INVALID_ARG;
  if ((((uintptr_t)err) & 3u) != 0) return TSD_ERR_INVALID_ARG;
  if (!ok_ptr(q) || !ok_ptr(kcache) || !ok_ptr(prefix_len) || !ok_ptr(ktree) || !ok_ptr(mask) ||
      !ok_ptr(out) || !ok_ptr(lse))
    return TSD_ERR_INVALID_ARG;
  if (!d->v_aliases_k && (!ok_ptr(vcache) || !ok_ptr(vtree))) return TSD_ERR_INVALID_ARG;
  const bool paged = page_size > 0;
  if (paged && (page_size % 128 != 0 || max_pages < 1 || num_pages < 1 ||
                (long)max_pages * page_size != d->cap || !ok_ptr(page_table) ||
                (long)num_pages * d->Hkv * page_size > (1l << 31)))
    return TSD_ERR_INVALID_ARG;
  VerifyPlan p = plan_verify(*d);
  // the legacy mma.sync kernel addresses a contiguous cache only
  if (paged && p.path == kPathMma) p.path = kPathGeneric;
  if (ws_bytes < p.ws_bytes || (p.ws_bytes > 0 && !ok_ptr(ws))) return TSD_ERR_INVALID_ARG;

  VerifyArgs a{};
  a.q = q; a.kc = kcache; a.vc = vcache; a.plen = prefix_len;
  a.kt = ktree; a.vt = vtree; a.mask = mask;
  a.out = out; a.lse = lse;
  {
    const size_t nparts = (size_t)d->B * d->Hq * d->R * p.nsplit;
    a.ws_o = p.part_bf16 ? nullptr : (float*)ws;
    a.ws_ob = p.part_bf16 ? (__nv_bfloat16*)ws : nullptr;
    a.ws_lse = p.nsplit > 1 ? (float*)((char*)ws + nparts * d->dv *
                                                     (p.part_bf16 ? sizeof(__nv_bfloat16) : sizeof(float)))
                            : nullptr;
  }
  a.B = d->B; a.R = d->R; a.Hq = d->Hq; a.Hkv = d->Hkv; a.g = d->Hq / d->Hkv;
  a.M = d->R * a.g; a.cap = d->cap;
  a.nsplit = p.nsplit; a.split_len = p.split_len; a.nrg = p.nrg;
  a.tree_split = p.tree_split;
  a.qscale = d->scale * 1.4426950408889634f;
  a.err = err;
  {
    const long long wb = g_wait_budget.load(std::memory_order_relaxed);
    a.wait_cycles = wb > 0 && wb < kWaitCycles ? wb : kWaitCycles;
  }
  a.page_table = paged ? page_table : nullptr;
  a.max_pages = paged ? max_pages : 0;
  a.page_size = paged ? page_size : 0;
  a.num_pages = paged ? num_pages : 0;
  const cudaStream_t st = (cudaStream_t)stream;
  bool launched;
  if (p.path == kPathTc && d->v_aliases_k) launched = launch_mla_tc_path(*d, a, p, st);
  else if (p.path == kPathTc) launched = launch_tc_path(*d, a, p, st);
  else if (p.path == kPathMma) launched = launch_mma_path(*d, a, p, st);
  else launched = launch_generic_path(*d, a, p, st);
  if (!launched) return TSD_ERR_UNSUPPORTED;
  return cuda_status();
}

extern "C" tsd_status tsd_tree_verify_attn(const tsd_attn_desc* d, const void* q,
                                           const void* kcache, const void* vcache,
                                           const int32_t* prefix_len, const void* ktree,
                                           const void* vtree, const uint64_t* mask, void* out,
                                           float* lse, void* ws, size_t ws_bytes, int32_t* err,
                                           tsd_stream_t stream) {
  return verify_impl(d, q, kcache, vcache, nullptr, 0, 0, 0, prefix_len, ktree, vtree, mask, out,
                     lse, ws, ws_bytes, err, stream);
}

extern "C" tsd_status tsd_tree_verify_attn_paged(const tsd_attn_desc* d, const void* q,
                                                 const void* kpool, const void* vpool,
                                                 const int32_t* page_table, int max_pages,
                                                 int page_size, int num_pages,
                                                 const int32_t* prefix_len, const void* ktree,
                                                 const void* vtree, const uint64_t* mask,
                                                 void* out, float* lse, void* ws, size_t ws_bytes,
                                                 int32_t* err, tsd_stream_t stream) {
  if (page_size < 1) return TSD_ERR_INVALID_ARG;
  return verify_impl(d, q, kpool, vpool, page_table, max_pages, page_size, num_pages, prefix_len,
                     ktree, vtree, mask, out, lse, ws, ws_bytes, err, stream);
}
