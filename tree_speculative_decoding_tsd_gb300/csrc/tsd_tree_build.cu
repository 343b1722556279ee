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
  // the tree's rows, written as they are popped (by every lane of the
  // popping warp, so that each lane reads back only its own writes): score,
  // ancestor mask, and the popped entry (depth | parent row << 8 | rank << 16)
  uint64_t r_mask[kMaxD + 1];
  float r_sc[kMaxD + 1];
  int32_t r_dpr[kMaxD + 1];
  uint8_t has_child[kMaxD + 1];
};

// Rank tuple of a path, 5 bits per level, most significant first, so that
// equal-length tuples compare lexicographically as (w0, w1).
__device__ __forceinline__ void tuple_add(uint64_t& w0, uint64_t& w1, int level, uint64_t digit) {
  if (level < 12) w0 += digit << (59 - 5 * level);
  else w1 += digit << (59 - 5 * (level - 12));
}

// Depth, parent row and rank of a frontier entry in one word (each < 256).
__device__ __forceinline__ int pack_dpr(int d, int par, int rk) { return d | (par << 8) | (rk << 16); }

// Rank tuple of the entry dpr: its rank at its depth, then its ancestors'
// ranks, read from the popped rows (a parent row precedes its children, so
// the walk reaches the root in at most depth steps).
__device__ __forceinline__ void entry_tuple(const TreeSmem& s, int32_t dpr, uint64_t& w0,
                                            uint64_t& w1) {
  w0 = 0ull;
  w1 = 0ull;
  for (int it = 0; it < kMaxS; ++it) {
    const int d = dpr & 0xff, par = (dpr >> 8) & 0xff;
    tuple_add(w0, w1, d - 1, (uint64_t)(dpr >> 16));
    if (par == 0) break;
    dpr = s.r_dpr[par];
  }
}

// Full order between two frontier entries (score desc, depth asc, tuple asc).
__device__ __forceinline__ bool precedes(float sa, int da, uint64_t a0, uint64_t a1, float sb,
                                         int db, uint64_t b0, uint64_t b1) {
  if (sa != sb) return sa > sb;
  if (da != db) return da < db;
  if (a0 != b0) return a0 < b0;
  return a1 < b1;
}

// The frontier minus its best entry is a sorted list spread over the lanes,
// entry e in lane e % 32, slot e / 32.  A pop removes one entry and adds at
// most two (net +1), and the last pop adds none, so before pop r the frontier
// holds at most r entries and the list at most D - 1: ceil(D / 32) slots
// suffice (1 for D <= 32, 2 for D <= 64).
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
  // (zeros without a table: the pops read it in either mode)
  for (int n = threadIdx.x; n <= D; n += blockDim.x)
    s.cost[n] = adaptive ? __fadd_rn(cost_d[b], cost_v[(long)b * R + n]) : 0.f;

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

  // ---- the pops: one warp, rows in shared memory ----
  // An entry is (score, depth | parent row << 8 | rank << 16).  Its rank
  // tuple follows from its own and its ancestors' entries, so it is only
  // built where scores tie.  The best
  // entry not yet popped (t_*) is held by every lane; the rest of the
  // frontier is the sorted list L (l_*).  A pop's sibling and child go to
  // the places given by the count of L's entries before them (ballots: L is
  // sorted), and the new best entry and the new L are read off the merged
  // list, each lane gathering its new entry with one shuffle per slot.
  float l_sc[kSlots];
  int32_t l_dpr[kSlots];
#pragma unroll
  for (int j = 0; j < kSlots; ++j) { l_sc[j] = 0.f; l_dpr[j] = pack_dpr(1, 0, 0); }
  // row 0 = root
  s.r_sc[0] = 1.0f;
  s.r_mask[0] = 0ull;
  s.r_dpr[0] = 0;
  // the first entry: rank 0 at depth 1
  float t_sc = __fmul_rn(1.0f, s.tp[0][0]);
  int32_t t_dpr = pack_dpr(1, 0, 0);
  int nl = 0;
  // Phi accumulation for the adaptive stop: A = 1 + Phi(first n nodes), fp32
  // in pop order.  Node n+1 is kept iff (A + s) * cost[n] > A * cost[n+1]
  // (fp32 products, i.e. the objective rises); the first failure ends the tree.
  float acc = 1.0f;
  int kept = D;
  constexpr int kNone = 1 << 20;   // place of a candidate that is not inserted

  for (int row = 1; row <= D; ++row) {
    const int d = t_dpr & 0xff, par = (t_dpr >> 8) & 0xff, rk = t_dpr >> 16;
    const bool sib = rk + 1 < k, child = d < S;
    // this pop's reads, issued together
    const float psc = s.r_sc[par];
    const float q_sib = s.tp[d - 1][sib ? rk + 1 : rk];
    const float q_child = s.tp[child ? d : d - 1][0];
    const uint64_t pm = s.r_mask[par];
    const float h_sc = __shfl_sync(kFull, l_sc[0], 0);     // L[0]
    const int32_t h_dpr = __shfl_sync(kFull, l_dpr[0], 0);
    // (branch-free where it can be: a branch costs this serial loop more
    // than the selects it saves)
    // adaptive stop: the objective would fall with this node (the cost
    // table is read in either mode; without one the test is masked off)
    const float acc1 = __fadd_rn(acc, t_sc);
    const bool stop =
        adaptive && !(__fmul_rn(acc1, s.cost[row - 1]) > __fmul_rn(acc, s.cost[row]));
    acc = acc1;
    // (a stopped row is written too: rows past the kept count are never read)
    s.r_sc[row] = t_sc;
    s.r_dpr[row] = t_dpr;
    s.r_mask[row] = pm | (1ull << (row - 1));
    // nothing is popped after the last row: no new entries
    if (stop || row == D) {
      kept = stop ? row - 1 : D;
      break;
    }

    // the candidates: next sibling (depth d, rank rk + 1), first child
    // (depth d + 1, rank 0); on equal scores the sibling, less deep, first
    const float c1 = __fmul_rn(psc, q_sib), c2 = __fmul_rn(t_sc, q_child);
    const int32_t c1_dpr = pack_dpr(d, par, rk + 1), c2_dpr = pack_dpr(d + 1, row, 0);
    // their places in L: the entries of higher score, then of equal score
    // (those take the full order)
    int gt1 = 0, ge1 = 0, gt2 = 0, ge2 = 0;
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const bool v = lane + 32 * j < nl;
      gt1 += __popc(__ballot_sync(kFull, v && l_sc[j] > c1));
      ge1 += __popc(__ballot_sync(kFull, v && l_sc[j] >= c1));
      gt2 += __popc(__ballot_sync(kFull, v && l_sc[j] > c2));
      ge2 += __popc(__ballot_sync(kFull, v && l_sc[j] >= c2));
    }
    int p1 = gt1, p2 = gt2;
    if (ge1 != gt1 || ge2 != gt2) {
      // the child's tuple is the popped entry's; the sibling's is one more at depth d
      uint64_t t_w0, t_w1;
      entry_tuple(s, t_dpr, t_w0, t_w1);
      uint64_t s0 = t_w0, s1 = t_w1;
      tuple_add(s0, s1, d - 1, 1ull);
      p1 = 0;
      p2 = 0;
#pragma unroll
      for (int j = 0; j < kSlots; ++j) {
        const bool v = lane + 32 * j < nl;
        const int ed = l_dpr[j] & 0xff;
        uint64_t e0, e1;
        entry_tuple(s, l_dpr[j], e0, e1);
        p1 += __popc(__ballot_sync(kFull, v && precedes(l_sc[j], ed, e0, e1, c1, d, s0, s1)));
        p2 += __popc(__ballot_sync(kFull, v && precedes(l_sc[j], ed, e0, e1, c2, d + 1, t_w0, t_w1)));
      }
    }
    // places in L' = L with the candidates merged in
    const bool c1_first = c1 >= c2;
    const int P1 = sib ? p1 + (child && !c1_first ? 1 : 0) : kNone;
    const int P2 = child ? p2 + (sib && c1_first ? 1 : 0) : kNone;
    // the next best entry is L'[0]; the new L[j] is L'[j + 1], a candidate
    // or L[j + 1 - (candidates placed before it)]
    float g_sc[kSlots];
    int32_t g_dpr[kSlots];
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const int i = lane + 32 * j + 1;
      const int src = i - (P1 < i ? 1 : 0) - (P2 < i ? 1 : 0);
      const int sl = src & 31, sj = src >> 5;
      float vs = __shfl_sync(kFull, l_sc[0], sl);
      int32_t vd = __shfl_sync(kFull, l_dpr[0], sl);
#pragma unroll
      for (int jj = 1; jj < kSlots; ++jj) {
        const float a = __shfl_sync(kFull, l_sc[jj], sl);
        const int32_t ad = __shfl_sync(kFull, l_dpr[jj], sl);
        vs = sj == jj ? a : vs;
        vd = sj == jj ? ad : vd;
      }
      g_sc[j] = i == P1 ? c1 : (i == P2 ? c2 : vs);
      g_dpr[j] = i == P1 ? c1_dpr : (i == P2 ? c2_dpr : vd);
    }
#pragma unroll
    for (int j = 0; j < kSlots; ++j) { l_sc[j] = g_sc[j]; l_dpr[j] = g_dpr[j]; }
    t_sc = P1 == 0 ? c1 : (P2 == 0 ? c2 : h_sc);
    t_dpr = P1 == 0 ? c1_dpr : (P2 == 0 ? c2_dpr : h_dpr);
    nl += (sib ? 1 : 0) + (child ? 1 : 0) - 1;
  }
  __syncwarp();

  // ---- leaves and outputs (each lane writes its own rows) ----
  // Rows past the kept count (adaptive mode only) are inert padding: token -1
  // (no target token matches it), parent 0, depth 0, score 0, mask 0, not a
  // leaf, so verify, walk and commit treat them as never accepted.
  // (rows in fixed chunks r = lane + 32 j, j < 3, covering rows 0..64: a
  // loop whose trip count differs between lanes costs far more)
#pragma unroll
  for (int j = 0; j < 3; ++j)
    if (lane + 32 * j <= D) s.has_child[lane + 32 * j] = 0;
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int r = lane + 32 * j;
    if (r >= 1 && r <= kept) s.has_child[(s.r_dpr[r] >> 8) & 0xff] = 1;
  }
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int r = lane + 32 * j;
    if (r > D) continue;
    if (r <= kept) {
      const int32_t dpr = s.r_dpr[r];
      const int d = dpr & 0xff;
      if (r == 0) {
        token[o] = root;
        parent[o] = -1;
      } else {
        token[o + r] = s.ti[d - 1][dpr >> 16];
        parent[o + r] = (dpr >> 8) & 0xff;
      }
      depth[o + r] = d;
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
