// tsd_tree_build_conditioned: the best-first draft tree over an explicit
// candidate forest whose proposals are conditioned on their parent node
// (EAGLE-style drafting: each node's children come from the drafter's
// distribution at that node, not from a per-position marginal).
//
// Source: "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4"
// (review), "How it works" steps 1-2: after A the draft expands B and C; after
// B it proposes B and C, after C it proposes A and B (each node's children are
// its own proposals), the 7-node tree is then pruned to the D nodes of highest
// cumulative score.  "Cost-Aware Diffusion Draft Trees", Method item 2: for a
// fixed node count the best tree takes the nodes of highest prefix probability.
//
// One CTA per request:
//   1. cumulative scores level by level (round r fixes the candidates of depth
//      r as fp32(score(parent) * p), the same product order as a path walk);
//   2. one 64-bit key per candidate, (score desc, depth asc, index asc), and a
//      block-wide bitonic sort in shared memory;
//   3. the first D keys are rows 1..D (a child never precedes its parent: its
//      score is not larger and its depth is), then parents, masks and leaves.
#include "tsd_common.cuh"
#include "tsd_host.h"

namespace tsd {
namespace {

constexpr int kCondMaxCand = 2048;
constexpr int kCondMaxD = 64;
constexpr int kCondMaxDepth = kCondMaxD + 1;   // deeper candidates cannot be kept
constexpr int kCondThreads = 1024;

__global__ void __launch_bounds__(kCondThreads)
conditioned_tree_kernel(const float* __restrict__ cand_p, const int32_t* __restrict__ cand_tok,
                        const int32_t* __restrict__ cand_parent, int C, int D,
                        const int32_t* __restrict__ root_tok, int32_t* __restrict__ token,
                        int32_t* __restrict__ parent, int32_t* __restrict__ depth,
                        float* __restrict__ score, uint64_t* __restrict__ mask,
                        uint8_t* __restrict__ is_leaf, int32_t* __restrict__ err) {
  grid_dependency_sync();
  __shared__ uint64_t key[kCondMaxCand];
  __shared__ float sc[kCondMaxCand];
  __shared__ int32_t par[kCondMaxCand];
  __shared__ int32_t row_of[kCondMaxCand];
  __shared__ uint8_t dep[kCondMaxCand];
  __shared__ int32_t r_cand[kCondMaxD + 1], r_par[kCondMaxD + 1];
  __shared__ uint64_t r_mask[kCondMaxD + 1];
  __shared__ uint8_t has_child[kCondMaxD + 1];
  __shared__ int s_bad;

  const int b = blockIdx.x, tid = threadIdx.x;
  const long ci = (long)b * C;
  const long o = (long)b * (D + 1);
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int c = tid; c < C; c += kCondThreads) {
    const int pp = cand_parent[ci + c];
    const float p = cand_p[ci + c];
    if (pp < -1 || pp >= c || !(p >= 0.f && p <= 1.f)) s_bad = 1;
    par[c] = pp;
    sc[c] = -1.f;   // unresolved
    dep[c] = 0;
    row_of[c] = -1;
  }
  __syncthreads();

  // 1. scores, one depth per round: every thread first reads the state the
  // previous round left (its candidates' parents), then, after a barrier,
  // writes what it resolved, so no round sees a value written in the same round
  constexpr int kPer = kCondMaxCand / kCondThreads;
  for (int r = 1; r <= kCondMaxDepth; ++r) {
    float s_new[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int c = tid + j * kCondThreads;
      s_new[j] = -1.f;
      if (c >= C || sc[c] >= 0.f) continue;
      const int pp = par[c];
      if (pp < 0) {
        if (r == 1) s_new[j] = __fmul_rn(1.0f, cand_p[ci + c]);
      } else if (pp < c && dep[pp] == r - 1 && sc[pp] >= 0.f) {
        s_new[j] = __fmul_rn(sc[pp], cand_p[ci + c]);
      }
    }
    __syncthreads();
    int changed = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int c = tid + j * kCondThreads;
      if (s_new[j] >= 0.f) {
        sc[c] = s_new[j];
        dep[c] = (uint8_t)r;
        changed = 1;
      }
    }
    if (!__syncthreads_or(changed)) break;
  }

  // 2. keys and a bitonic sort (ascending key = descending priority)
  int n2 = 1;
  while (n2 < C) n2 <<= 1;
  for (int c = tid; c < n2; c += kCondThreads) {
    uint64_t k = ~0ull;
    if (c < C && sc[c] >= 0.f) {
      uint32_t bits = __float_as_uint(sc[c]);
      if (bits == 0x80000000u) bits = 0u;   // -0 scores as +0
      k = ((uint64_t)(~bits) << 32) | ((uint64_t)dep[c] << 16) | (uint64_t)c;
    }
    key[c] = k;
  }
  __syncthreads();
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < n2 / 2; i += kCondThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = ((lo & size) == 0);
        const uint64_t a = key[lo], e = key[hi];
        if ((a > e) == up) {
          key[lo] = e;
          key[hi] = a;
        }
      }
      __syncthreads();
    }
  }

  // 3. rows 1..D
  for (int i = tid; i < D; i += kCondThreads) {
    const uint64_t k = key[i];
    if (k == ~0ull) {
      s_bad = 1;   // fewer than D reachable candidates
      r_cand[i + 1] = -1;
    } else {
      const int c = (int)(k & 0xffffu);
      r_cand[i + 1] = c;
      row_of[c] = i + 1;
    }
  }
  __syncthreads();
  for (int i = 1 + tid; i <= D; i += kCondThreads) {
    const int c = r_cand[i];
    int pr = 0;
    if (c >= 0 && par[c] >= 0) {
      pr = row_of[par[c]];
      if (pr < 1 || pr >= i) s_bad = 1;   // the kept set is not ancestor-closed
    }
    r_par[i] = pr < 0 ? 0 : pr;
  }
  if (tid <= D) has_child[tid] = 0;
  __syncthreads();
  const bool bad = s_bad != 0;
  if (tid == 0) {
    r_mask[0] = 0ull;
    for (int i = 1; i <= D; ++i) {
      const int pr = r_par[i];
      r_mask[i] = (pr >= 0 && pr < i ? r_mask[pr] : 0ull) | (1ull << (i - 1));
    }
    if (bad) report_error(err, TSD_DEV_ERR_BAD_TREE, b);
  }
  if (tid >= 1 && tid <= D) has_child[r_par[tid]] = 1;
  __syncthreads();
  // outputs; a rejected forest gives the root and inert padding rows
  for (int i = tid; i <= D; i += kCondThreads) {
    if (i == 0) {
      token[o] = root_tok[b];
      parent[o] = -1;
      depth[o] = 0;
      score[o] = 1.0f;
      mask[o] = 0ull;
      is_leaf[o] = (bad || !has_child[0]) ? 1 : 0;
    } else if (bad) {
      token[o + i] = -1;
      parent[o + i] = 0;
      depth[o + i] = 0;
      score[o + i] = 0.f;
      mask[o + i] = 0ull;
      is_leaf[o + i] = 0;
    } else {
      const int c = r_cand[i];
      token[o + i] = cand_tok[ci + c];
      parent[o + i] = r_par[i];
      depth[o + i] = dep[c];
      score[o + i] = sc[c];
      mask[o + i] = r_mask[i];
      is_leaf[o + i] = has_child[i] ? 0 : 1;
    }
  }
}

}  // namespace
}  // namespace tsd

using namespace tsd;

extern "C" tsd_status tsd_tree_build_conditioned(const float* cand_p, const int32_t* cand_tok,
                                                 const int32_t* cand_parent, int B, int C, int D,
                                                 const int32_t* root_tok, int32_t* token,
                                                 int32_t* parent, int32_t* depth, float* score,
                                                 uint64_t* mask, uint8_t* is_leaf, int32_t* err,
                                                 tsd_stream_t stream) {
  if (B < 1 || B > 65535 || C < 1 || C > kCondMaxCand || D < 1 || D > kCondMaxD || D > C)
    return TSD_ERR_INVALID_ARG;
  if (!ok_ptr(cand_p) || !ok_ptr(cand_tok) || !ok_ptr(cand_parent) || !ok_ptr(root_tok) ||
      !ok_ptr(token) || !ok_ptr(parent) || !ok_ptr(depth) || !ok_ptr(score) || !ok_ptr(mask) ||
      !ok_ptr(is_leaf) || !ok_opt_ptr(err))
    return TSD_ERR_INVALID_ARG;
  launch(conditioned_tree_kernel, dim3(B), dim3(kCondThreads), 0, (cudaStream_t)stream, cand_p,
      cand_tok, cand_parent, C, D, root_tok, token, parent, depth, score, mask, is_leaf, err);
  return cuda_status();
}
