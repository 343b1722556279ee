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
//    With a cost table (tsd_tree_build_adaptive) the pops stop early: the
//    greedy rule of "Cost-Aware Diffusion Draft Trees", Method items 1, 3-4,
//    adds the next node only while it raises the throughput objective
//    (1 + Phi) / (C_d + C_v(n)), Phi being the sum of the kept scores.
#include "tsd_common.cuh"
#include "tsd_host.h"
#include "tsd_scan.cuh"

namespace tsd {
namespace {

constexpr int kMaxS = 16;
constexpr int kMaxK = 32;
constexpr int kMaxD = 64;

struct TreeSmem {
  float tp[kMaxS][kMaxK];     // top-k probabilities per position
  int32_t ti[kMaxS][kMaxK];   // top-k token ids per position
  float cost[kMaxD + 1];      // adaptive mode: C_d + C_v(n), n = 0..D
  // the tree's rows, written by lane 0 as they are popped
  uint64_t r_mask[kMaxD + 1];
  float r_sc[kMaxD + 1];
  int32_t r_par[kMaxD + 1];
  int32_t r_tok[kMaxD + 1];
  int32_t r_dep[kMaxD + 1];
  uint8_t has_child[kMaxD + 1];
};

// Rank tuple of a path, 5 bits per level, most significant first, so that
// equal-length tuples compare lexicographically as (w0, w1).
__device__ __forceinline__ void tuple_add(uint64_t& w0, uint64_t& w1, int level, uint64_t digit) {
  if (level < 12) w0 += digit << (59 - 5 * level);
  else w1 += digit << (59 - 5 * (level - 12));
}

// Primary key of a frontier entry: the score's bit pattern inverted (the bit
// pattern of a non-negative float grows with it), so the smallest key is the
// highest score.  Entries with different keys are ordered by the key alone;
// equal keys (equal scores) are resolved by the full comparison.
__device__ __forceinline__ uint32_t score_key(float sc) { return ~__float_as_uint(sc); }

// Depth, parent row and rank of a frontier entry in one word (each < 256).
__device__ __forceinline__ int pack_dpr(int d, int par, int rk) { return d | (par << 8) | (rk << 16); }

// Full order between two frontier entries (score desc, depth asc, tuple asc).
__device__ __forceinline__ bool precedes(float sa, int da, uint64_t a0, uint64_t a1, float sb,
                                         int db, uint64_t b0, uint64_t b1) {
  if (sa != sb) return sa > sb;
  if (da != db) return da < db;
  if (a0 != b0) return a0 < b0;
  return a1 < b1;
}

// Per-lane register slots: frontier entry e lives in lane e % 32, slot e / 32.
// A pop removes one entry and adds at most two (net +1), and the last pop
// adds none, so pop r reads at most r entries and writes index <= r - 1 < D:
// ceil(D / 32) slots suffice; the kernel is instantiated for 1 and 2 slots
// (D <= 32, D <= 64) because every pick and put costs one select per slot.
template <int NS, typename T>
__device__ __forceinline__ T pick(const T (&v)[NS], int j) {
  T r = v[0];
#pragma unroll
  for (int i = 1; i < NS; ++i) r = (j == i) ? v[i] : r;
  return r;
}
template <int NS, typename T>
__device__ __forceinline__ void put(T (&v)[NS], int j, T x, bool pred) {
#pragma unroll
  for (int i = 0; i < NS; ++i) v[i] = (pred && j == i) ? x : v[i];
}
template <int NS, typename T>
__device__ __forceinline__ T bcast(const T (&v)[NS], int e) {
  return __shfl_sync(kFull, pick<NS>(v, e >> 5), e & 31);
}

template <int kSlots>
__global__ void __launch_bounds__(32 * kMaxS, 1)
best_first_tree_kernel(const uint64_t* __restrict__ part, int S, int k, int D, int nchunk,
                       const int32_t* __restrict__ root_tok, int32_t* __restrict__ token,
                       int32_t* __restrict__ parent, int32_t* __restrict__ depth,
                       float* __restrict__ score, uint64_t* __restrict__ mask,
                       uint8_t* __restrict__ is_leaf, const float* __restrict__ cost_d,
                       const float* __restrict__ cost_v, int32_t* __restrict__ n_nodes) {
  grid_dependency_sync();
  __shared__ TreeSmem s;
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = D + 1;
  const long o = (long)b * R;
  const bool adaptive = cost_v != nullptr;
  // the root token is loaded now, with the chunk lists, not after the merge
  // (where the popping warp would wait for it)
  const int32_t root = threadIdx.x == 0 ? root_tok[b] : 0;
  // adaptive mode: round cost of a tree with n nodes, fp32 C_d + C_v(n)
  if (adaptive)
    for (int n = threadIdx.x; n <= D; n += blockDim.x)
      s.cost[n] = __fadd_rn(cost_d[b], cost_v[(long)b * R + n]);

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
    const uint64_t entry = warp_topk<kPer>(c, k, lane);
    if (lane < k) {
      s.tp[p][lane] = cand_val(entry);
      s.ti[p][lane] = (int32_t)cand_id(entry);
    }
  }
  __syncthreads();
  if (warp != 0) return;

  // ---- frontier in registers, spread over the lanes; rows in shared memory ----
  // A frontier entry also carries its parent's score and ancestor mask, so a
  // pop needs no lookup of the parent row.  Lane 0 writes each popped row to
  // shared memory (no per-lane selects on the critical path).
  float f_sc[kSlots], f_psc[kSlots];
  uint32_t f_key[kSlots];
  int32_t f_dpr[kSlots];
  uint64_t f_w0[kSlots], f_w1[kSlots], f_pm[kSlots];
#pragma unroll
  for (int j = 0; j < kSlots; ++j) {
    f_sc[j] = 0.f; f_psc[j] = 0.f; f_key[j] = ~0u; f_dpr[j] = 0;
    f_w0[j] = 0ull; f_w1[j] = 0ull; f_pm[j] = 0ull;
  }
  // row 0 = root; frontier slot 0 = rank 0 at depth 1
  if (lane == 0) {
    s.r_sc[0] = 1.0f; s.r_par[0] = -1; s.r_tok[0] = root; s.r_dep[0] = 0;
    s.r_mask[0] = 0ull;
    f_sc[0] = __fmul_rn(1.0f, s.tp[0][0]); f_psc[0] = 1.0f; f_dpr[0] = pack_dpr(1, 0, 0);
    f_pm[0] = 0ull;
    f_key[0] = score_key(f_sc[0]);
  }
  int nf = 1;
  // Phi accumulation for the adaptive stop: A = 1 + Phi(first n nodes), fp32
  // in pop order.  Node n+1 is kept iff (A + s) * cost[n] > A * cost[n+1]
  // (fp32 products, i.e. the objective rises); the first failure ends the tree.
  float acc = 1.0f;
  int kept = D;

  for (int row = 1; row <= D; ++row) {
    // this lane's smallest key, then the warp's; one holder of one entry is
    // the common case, several entries with the key (equal scores) take the
    // full comparison
    uint32_t kmin = ~0u;
    int mine = -1;
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const int e = lane + 32 * j;
      // (a score of 0 has the key ~0u, so "no entry yet" is mine < 0)
      if (e < nf && (mine < 0 || f_key[j] < kmin)) { kmin = f_key[j]; mine = e; }
    }
    const uint32_t hmin = __reduce_min_sync(kFull, kmin);
    int ties = 0;
#pragma unroll
    for (int j = 0; j < kSlots; ++j) ties += (lane + 32 * j < nf && f_key[j] == hmin) ? 1 : 0;
    const unsigned hb = __ballot_sync(kFull, ties > 0);
    const unsigned hm = __ballot_sync(kFull, ties > 1);
    int best = __shfl_sync(kFull, mine, __ffs(hb) - 1);
    if (__popc(hb) > 1 || hm != 0u) {
      // equal scores: full order (depth, then rank tuple)
      int b2 = -1;
      float bs = 0.f; int bd = 0; uint64_t b0 = 0ull, b1 = 0ull;
#pragma unroll
      for (int j = 0; j < kSlots; ++j) {
        const int e = lane + 32 * j;
        const int dj = f_dpr[j] & 0xff;
        if (e < nf && f_key[j] == hmin &&
            (b2 < 0 || precedes(f_sc[j], dj, f_w0[j], f_w1[j], bs, bd, b0, b1))) {
          b2 = e; bs = f_sc[j]; bd = dj; b0 = f_w0[j]; b1 = f_w1[j];
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const int oe = __shfl_xor_sync(kFull, b2, off);
        const float os = __shfl_xor_sync(kFull, bs, off);
        const int od = __shfl_xor_sync(kFull, bd, off);
        const uint64_t o0 = __shfl_xor_sync(kFull, b0, off), o1 = __shfl_xor_sync(kFull, b1, off);
        if (oe >= 0 && (b2 < 0 || precedes(os, od, o0, o1, bs, bd, b0, b1))) {
          b2 = oe; bs = os; bd = od; b0 = o0; b1 = o1;
        }
      }
      best = b2;
    }
    // the popped entry and the new row
    const float sc = bcast<kSlots>(f_sc, best), psc = bcast<kSlots>(f_psc, best);
    if (adaptive) {
      const float acc1 = __fadd_rn(acc, sc);
      if (!(__fmul_rn(acc1, s.cost[row - 1]) > __fmul_rn(acc, s.cost[row]))) {
        kept = row - 1;
        break;
      }
      acc = acc1;
    }
    const int dpr = bcast<kSlots>(f_dpr, best);
    const int d = dpr & 0xff, par = (dpr >> 8) & 0xff, rk = dpr >> 16;
    const uint64_t w0 = bcast<kSlots>(f_w0, best), w1 = bcast<kSlots>(f_w1, best);
    const uint64_t pm = bcast<kSlots>(f_pm, best);
    const uint64_t m = pm | (1ull << (row - 1));
    if (lane == 0) {
      s.r_sc[row] = sc;
      s.r_par[row] = par;
      s.r_tok[row] = s.ti[d - 1][rk];
      s.r_dep[row] = d;
      s.r_mask[row] = m;
    }
    // nothing is popped after the last row: no new entries (so the frontier
    // never holds more than D entries when a pop reads it)
    if (row == D) break;
    // the popped slot becomes the next sibling, or takes the last entry
    const int bl = best & 31, bj = best >> 5;
    const int last = nf - 1;
    if (rk + 1 < k) {
      const float nsc = __fmul_rn(psc, s.tp[d - 1][rk + 1]);
      uint64_t nw0 = w0, nw1 = w1;
      tuple_add(nw0, nw1, d - 1, 1ull);
      const bool me = lane == bl;
      put<kSlots>(f_sc, bj, nsc, me); put<kSlots>(f_dpr, bj, pack_dpr(d, par, rk + 1), me);
      put<kSlots>(f_w0, bj, nw0, me); put<kSlots>(f_w1, bj, nw1, me);
      put<kSlots>(f_key, bj, score_key(nsc), me);
    } else {
      const float lsc = bcast<kSlots>(f_sc, last), lps = bcast<kSlots>(f_psc, last);
      const int ldpr = bcast<kSlots>(f_dpr, last);
      const uint64_t l0 = bcast<kSlots>(f_w0, last), l1 = bcast<kSlots>(f_w1, last);
      const uint32_t lk = bcast<kSlots>(f_key, last);
      const uint64_t lm = bcast<kSlots>(f_pm, last);
      const bool me = lane == bl;
      put<kSlots>(f_sc, bj, lsc, me); put<kSlots>(f_psc, bj, lps, me);
      put<kSlots>(f_dpr, bj, ldpr, me); put<kSlots>(f_w0, bj, l0, me);
      put<kSlots>(f_w1, bj, l1, me); put<kSlots>(f_key, bj, lk, me); put<kSlots>(f_pm, bj, lm, me);
      nf = last;
    }
    // first child (rank 0 at the next position)
    if (d < S) {
      const float csc = __fmul_rn(sc, s.tp[d][0]);
      const bool me = lane == (nf & 31);
      const int cj = nf >> 5;
      put<kSlots>(f_sc, cj, csc, me); put<kSlots>(f_psc, cj, sc, me);
      put<kSlots>(f_dpr, cj, pack_dpr(d + 1, row, 0), me);
      put<kSlots>(f_w0, cj, w0, me);
      put<kSlots>(f_w1, cj, w1, me); put<kSlots>(f_pm, cj, m, me);
      put<kSlots>(f_key, cj, score_key(csc), me);
      ++nf;
    }
  }
  __syncwarp();

  // ---- leaves and outputs (each lane writes its own rows) ----
  // Rows past the kept count (adaptive mode only) are inert padding: token -1
  // (no target token matches it), parent 0, depth 0, score 0, mask 0, not a
  // leaf, so verify, walk and commit treat them as never accepted.
  for (int r = lane; r <= D; r += 32) s.has_child[r] = 0;
  __syncwarp();
  for (int r = 1 + lane; r <= kept; r += 32) s.has_child[s.r_par[r]] = 1;
  __syncwarp();
  for (int r = lane; r <= D; r += 32) {
    if (r <= kept) {
      token[o + r] = s.r_tok[r];
      parent[o + r] = s.r_par[r];
      depth[o + r] = s.r_dep[r];
      score[o + r] = s.r_sc[r];
      mask[o + r] = s.r_mask[r];
      is_leaf[o + r] = s.has_child[r] ? 0 : 1;
    } else {
      token[o + r] = -1;
      parent[o + r] = 0;
      depth[o + r] = 0;
      score[o + r] = 0.f;
      mask[o + r] = 0ull;
      is_leaf[o + r] = 0;
    }
  }
  if (n_nodes != nullptr && lane == 0) n_nodes[b] = kept;
}

}  // namespace
}  // namespace tsd

using namespace tsd;

extern "C" size_t tsd_tree_build_workspace_size(int B, int S, int V, int k) {
  if (B < 1 || S < 1 || V < 1 || k < 1) return 0;
  const ScanGeom g = scan_geometry((long)B * S, V, k, false);
  return (size_t)B * S * g.nchunk * k * sizeof(uint64_t);
}

namespace {

tsd_status tree_build_impl(const float* probs, int B, int S, int V, int k, int D,
                           const int32_t* root_tok, const float* cost_d, const float* cost_v,
                           int32_t* token, int32_t* parent, int32_t* depth, float* score,
                           uint64_t* mask, uint8_t* is_leaf, int32_t* n_nodes, void* ws,
                           size_t ws_bytes, int32_t* err, tsd_stream_t stream) {
  if (B < 1 || S < 1 || S > kMaxS || k < 1 || k > kMaxK || V < k || D < 1 || D > kMaxD)
    return TSD_ERR_INVALID_ARG;
  if (tree_node_count(S, k) < D) return TSD_ERR_INVALID_ARG;
  if ((long)B * S > (1l << 24) || (long)V > (1l << 30)) return TSD_ERR_INVALID_ARG;
  if (!ok_ptr(probs) || !ok_ptr(root_tok) || !ok_ptr(token) || !ok_ptr(parent) ||
      !ok_ptr(depth) || !ok_ptr(score) || !ok_ptr(mask) || !ok_ptr(is_leaf) ||
      (((uintptr_t)err) & 3u) != 0)
    return TSD_ERR_INVALID_ARG;
  const size_t need = tsd_tree_build_workspace_size(B, S, V, k);
  if (ws_bytes < need || !ok_ptr(ws)) return TSD_ERR_INVALID_ARG;

  const cudaStream_t st = (cudaStream_t)stream;
  const ScanGeom g = scan_geometry((long)B * S, V, k, false);
  const long ctas = (long)B * S * g.nchunk;
  uint64_t* part = (uint64_t*)ws;
  launch(vocab_scan_kernel<false>, dim3((unsigned)ctas), dim3(kScanThreads), 0, st, probs, V, k,
      g.nchunk, g.chunk_len, part, g.one_wave, err, S);
  const auto tree_kernel = D <= 32 ? best_first_tree_kernel<1> : best_first_tree_kernel<2>;
  launch(tree_kernel, dim3(B), dim3(32 * S), 0, st, part, S, k, D, g.nchunk, root_tok, token,
      parent, depth, score, mask, is_leaf, cost_d, cost_v, n_nodes);
  return cuda_status();
}

}  // namespace

extern "C" tsd_status tsd_tree_build(const float* probs, int B, int S, int V, int k, int D,
                                     const int32_t* root_tok, int32_t* token, int32_t* parent,
                                     int32_t* depth, float* score, uint64_t* mask,
                                     uint8_t* is_leaf, void* ws, size_t ws_bytes, int32_t* err,
                                     tsd_stream_t stream) {
  return tree_build_impl(probs, B, S, V, k, D, root_tok, nullptr, nullptr, token, parent, depth,
                         score, mask, is_leaf, nullptr, ws, ws_bytes, err, stream);
}

extern "C" tsd_status tsd_tree_build_adaptive(const float* probs, int B, int S, int V, int k,
                                              int D_max, const int32_t* root_tok,
                                              const float* cost_d, const float* cost_v,
                                              int32_t* token, int32_t* parent, int32_t* depth,
                                              float* score, uint64_t* mask, uint8_t* is_leaf,
                                              int32_t* n_nodes, void* ws, size_t ws_bytes,
                                              int32_t* err, tsd_stream_t stream) {
  if (!ok_ptr(cost_d) || !ok_ptr(cost_v) || !ok_ptr(n_nodes)) return TSD_ERR_INVALID_ARG;
  return tree_build_impl(probs, B, S, V, k, D_max, root_tok, cost_d, cost_v, token, parent, depth,
                         score, mask, is_leaf, n_nodes, ws, ws_bytes, err, stream);
}
