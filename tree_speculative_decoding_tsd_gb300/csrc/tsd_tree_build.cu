// tsd_tree_build: per-position top-k of the draft marginals, then the greedy
// best-first draft tree under a node budget.
//
// Sources: "Cost-Aware Diffusion Draft Trees for Speculative Decoding",
// Method items 1-2 (a one-pass drafter gives per-position marginals; for a
// fixed node count the best tree is the greedy best-first one, which always
// takes the node of highest prefix probability).  "Adapting Tree-Structured
// Speculative Decoding to DeepSeek-V4" (review), "How it works" steps 1-2
// (top-k expansion per step, then budget pruning to the D best nodes by
// cumulative score) and step 3 (attention gets layout and metadata only: here
// parent, depth and the ancestor bitmask).
//
// K1 vocab_scan_kernel<false>: per-chunk top-k of every (request, position)
//    row, HBM-bound (see tsd_scan.cuh).
// K2 best_first_tree_kernel: one CTA per request; warp p merges the chunk lists
//    of position p into its k best tokens, then warp 0 pops D nodes from a
//    frontier.  Popping a node pushes its first child and its next sibling
//    (children are the top-k of the next position in rank order, so a node's
//    first child and younger siblings never precede it); this visits nodes in
//    exactly the total order (score desc, depth asc, rank tuple asc).
#include "tsd_common.cuh"
#include "tsd_host.h"
#include "tsd_scan.cuh"

namespace tsd {
namespace {

constexpr int kMaxS = 16;
constexpr int kMaxK = 32;
constexpr int kMaxD = 64;
constexpr int kMaxFront = kMaxD + 2;

struct TreeSmem {
  float tp[kMaxS][kMaxK];     // top-k probabilities per position
  int32_t ti[kMaxS][kMaxK];   // top-k token ids per position
  // frontier
  float f_sc[kMaxFront];
  int32_t f_depth[kMaxFront], f_par[kMaxFront], f_rank[kMaxFront];
  uint64_t f_w0[kMaxFront], f_w1[kMaxFront];
  uint64_t f_key[kMaxFront];  // primary order key (smaller pops first)
  int32_t nf;
  // emitted rows
  float r_sc[kMaxD + 1];
  int32_t r_par[kMaxD + 1];
  uint64_t r_mask[kMaxD + 1], r_w0[kMaxD + 1], r_w1[kMaxD + 1];
};

// Rank tuple of a path, 5 bits per level, most significant first, so that
// equal-length tuples compare lexicographically as (w0, w1).
__device__ __forceinline__ void tuple_add(uint64_t& w0, uint64_t& w1, int level, uint64_t digit) {
  if (level < 12) w0 += digit << (59 - 5 * level);
  else w1 += digit << (59 - 5 * (level - 12));
}

// Primary key of a frontier entry: score descending (the bit pattern of a
// non-negative float grows with it), then depth, then the first 27 tuple bits.
// Entries with different keys are ordered by the key alone; equal keys (equal
// score and depth, same leading ranks) are resolved by the full comparison.
__device__ __forceinline__ uint64_t primary_key(float sc, int depth, uint64_t w0) {
  return ((uint64_t)(~__float_as_uint(sc)) << 32) | ((uint64_t)depth << 27) | (w0 >> 37);
}

// true if frontier entry a precedes entry b in the total order
__device__ __forceinline__ bool precedes(const TreeSmem& s, int a, int b) {
  if (s.f_sc[a] != s.f_sc[b]) return s.f_sc[a] > s.f_sc[b];
  if (s.f_depth[a] != s.f_depth[b]) return s.f_depth[a] < s.f_depth[b];
  if (s.f_w0[a] != s.f_w0[b]) return s.f_w0[a] < s.f_w0[b];
  return s.f_w1[a] < s.f_w1[b];
}

__global__ void __launch_bounds__(32 * kMaxS)
best_first_tree_kernel(const uint64_t* __restrict__ part, int S, int k, int D, int nchunk,
                       const int32_t* __restrict__ root_tok, int32_t* __restrict__ token,
                       int32_t* __restrict__ parent, int32_t* __restrict__ depth,
                       float* __restrict__ score, uint64_t* __restrict__ mask,
                       uint8_t* __restrict__ is_leaf) {
  __shared__ TreeSmem s;
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = D + 1;
  const long o = (long)b * R;
  const unsigned kmask = (k >= 32) ? kFull : ((1u << k) - 1u);

  // ---- warp p merges the chunk lists of position p into its top-k ----
  // (at most kScanMaxCand candidates: every lane loads its share up front)
  {
    const int p = warp;
    const int ncand = nchunk * k;
    const uint64_t* src = part + ((long)b * S + p) * ncand;
    constexpr int kPer = kScanMaxCand / 32;
    uint64_t c[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = lane + 32 * j;
      c[j] = i < ncand ? src[i] : 0ull;
    }
    uint64_t entry = 0, thr = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (32 * j >= ncand) break;
      warp_list_offer(entry, thr, c[j], k, kmask, lane);
    }
    if (lane < k) {
      s.tp[p][lane] = cand_val(entry);
      s.ti[p][lane] = (int32_t)cand_id(entry);
    }
  }
  __syncthreads();
  if (warp != 0) return;

  // ---- root row and the first frontier entry (rank 0 at depth 1) ----
  if (lane == 0) {
    s.r_sc[0] = 1.0f;
    s.r_par[0] = -1;
    s.r_mask[0] = 0ull;
    s.r_w0[0] = 0ull;
    s.r_w1[0] = 0ull;
    token[o] = root_tok[b];
    parent[o] = -1;
    depth[o] = 0;
    score[o] = 1.0f;
    mask[o] = 0ull;
  }
  __syncwarp();
  if (lane == 0) {
    s.f_sc[0] = __fmul_rn(1.0f, s.tp[0][0]);
    s.f_depth[0] = 1;
    s.f_par[0] = 0;
    s.f_rank[0] = 0;
    s.f_w0[0] = 0ull;
    s.f_w1[0] = 0ull;
    s.f_key[0] = primary_key(s.f_sc[0], 1, 0ull);
    s.nf = 1;
  }
  __syncwarp();

  // ---- D pops: warp-wide minimum of the primary keys ----
  for (int row = 1; row <= D; ++row) {
    const int nf = s.nf;
    uint64_t kmin = ~0ull;
    int best = -1;
    for (int e = lane; e < nf; e += 32) {
      const uint64_t ke = s.f_key[e];
      if (ke < kmin) { kmin = ke; best = e; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t ok = __shfl_xor_sync(kFull, kmin, off);
      const int oe = __shfl_xor_sync(kFull, best, off);
      if (ok < kmin || (ok == kmin && oe >= 0 && (best < 0 || oe < best))) { kmin = ok; best = oe; }
    }
    // several entries with the same primary key: full comparison among them
    int ties = 0;
    for (int e = lane; e < nf; e += 32) ties += (s.f_key[e] == kmin) ? 1 : 0;
    if (__popc(__ballot_sync(kFull, ties > 0)) > 1 || __any_sync(kFull, ties > 1)) {
      int b2 = -1;
      for (int e = lane; e < nf; e += 32)
        if (s.f_key[e] == kmin && (b2 < 0 || precedes(s, e, b2))) b2 = e;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const int other = __shfl_xor_sync(kFull, b2, off);
        if (other >= 0 && (b2 < 0 || precedes(s, other, b2))) b2 = other;
      }
      best = b2;
    }
    if (lane == 0 && best >= 0) {
      const float sc = s.f_sc[best];
      const int d = s.f_depth[best];
      const int par = s.f_par[best];
      const int rk = s.f_rank[best];
      const uint64_t w0 = s.f_w0[best], w1 = s.f_w1[best];
      const uint64_t m = s.r_mask[par] | (1ull << (row - 1));
      s.r_sc[row] = sc;
      s.r_par[row] = par;
      s.r_mask[row] = m;
      s.r_w0[row] = w0;
      s.r_w1[row] = w1;
      token[o + row] = s.ti[d - 1][rk];
      parent[o + row] = par;
      depth[o + row] = d;
      score[o + row] = sc;
      mask[o + row] = m;
      // the popped slot becomes the next sibling, or is removed
      if (rk + 1 < k) {
        const float nsc = __fmul_rn(s.r_sc[par], s.tp[d - 1][rk + 1]);
        uint64_t nw0 = w0, nw1 = w1;
        tuple_add(nw0, nw1, d - 1, 1ull);
        s.f_sc[best] = nsc;
        s.f_rank[best] = rk + 1;
        s.f_w0[best] = nw0;
        s.f_w1[best] = nw1;
        s.f_key[best] = primary_key(nsc, d, nw0);
      } else {
        const int last = s.nf - 1;
        s.f_sc[best] = s.f_sc[last];
        s.f_depth[best] = s.f_depth[last];
        s.f_par[best] = s.f_par[last];
        s.f_rank[best] = s.f_rank[last];
        s.f_w0[best] = s.f_w0[last];
        s.f_w1[best] = s.f_w1[last];
        s.f_key[best] = s.f_key[last];
        s.nf = last;
      }
      // first child (rank 0 at the next position)
      if (d < S) {
        const int e = s.nf;
        const float csc = __fmul_rn(sc, s.tp[d][0]);
        s.f_sc[e] = csc;
        s.f_depth[e] = d + 1;
        s.f_par[e] = row;
        s.f_rank[e] = 0;
        s.f_w0[e] = w0;
        s.f_w1[e] = w1;
        s.f_key[e] = primary_key(csc, d + 1, w0);
        s.nf = e + 1;
      }
    }
    __syncwarp();
  }

  // ---- leaves ----
  for (int r = lane; r < R; r += 32) {
    bool has_child = false;
    for (int c = 1; c < R; ++c) has_child |= (s.r_par[c] == r);
    is_leaf[o + r] = has_child ? 0 : 1;
  }
}

}  // namespace
}  // namespace tsd

using namespace tsd;

extern "C" size_t tsd_tree_build_workspace_size(int B, int S, int V, int k) {
  if (B < 1 || S < 1 || V < 1 || k < 1) return 0;
  const ScanGeom g = scan_geometry((long)B * S, V, k);
  return (size_t)B * S * g.nchunk * k * sizeof(uint64_t);
}

extern "C" tsd_status tsd_tree_build(const float* probs, int B, int S, int V, int k, int D,
                                     const int32_t* root_tok, int32_t* token, int32_t* parent,
                                     int32_t* depth, float* score, uint64_t* mask,
                                     uint8_t* is_leaf, void* ws, size_t ws_bytes, int32_t* err,
                                     tsd_stream_t stream) {
  (void)err;
  if (B < 1 || S < 1 || S > kMaxS || k < 1 || k > kMaxK || V < k || D < 1 || D > kMaxD)
    return TSD_ERR_INVALID_ARG;
  if (tree_node_count(S, k) < D) return TSD_ERR_INVALID_ARG;
  if ((long)B * S > (1l << 24) || (long)V > (1l << 30)) return TSD_ERR_INVALID_ARG;
  if (!ok_ptr(probs) || !ok_ptr(root_tok) || !ok_ptr(token) || !ok_ptr(parent) ||
      !ok_ptr(depth) || !ok_ptr(score) || !ok_ptr(mask) || !ok_ptr(is_leaf))
    return TSD_ERR_INVALID_ARG;
  const size_t need = tsd_tree_build_workspace_size(B, S, V, k);
  if (ws_bytes < need || !ok_ptr(ws)) return TSD_ERR_INVALID_ARG;

  const cudaStream_t st = (cudaStream_t)stream;
  const ScanGeom g = scan_geometry((long)B * S, V, k);
  const long ctas = (long)B * S * g.nchunk;
  uint64_t* part = (uint64_t*)ws;
  vocab_scan_kernel<false><<<(unsigned)ctas, kScanThreads, 0, st>>>(probs, V, k, g.nchunk,
                                                                    g.chunk_len, part);
  best_first_tree_kernel<<<B, 32 * S, 0, st>>>(part, S, k, D, g.nchunk, root_tok, token, parent,
                                           depth, score, mask, is_leaf);
  return cuda_status();
}
