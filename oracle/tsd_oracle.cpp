// Plain CPU oracle for the tree-speculative-decoding verify step.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
// restatement of what the verify step computes.  Only the test-suite, the
// smoke check and the CPU-baseline leg of the benchmark load it.  It shares no
// code, header, table or helper with the CUDA library and must never be linked
// into it.
//
// Sources (web pages; cited by title and section):
//   [V4TREE] "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for
//            Efficient Inference" (review page): Key idea; Background, research
//            gap item 1 (branch-aware causal verification); the toy example
//            "How it works" steps 1-6; "Secret weapon" (scratch pad, commit of
//            the accepted path only).
//   [CADD]   "Cost-Aware Diffusion Draft Trees for Speculative Decoding":
//            Method (per-position marginals from a one-pass drafter; greedy
//            best-first tree = highest prefix probability first).
//   [DSPARK] "DSpark: Speculative decoding ..." : Architecture, decoding cycle
//            (anchor D, drafts E F G H, E and F accepted, G rejected,
//            correction token G*).
//
// Readings taken where the pages are silent (each also listed in the design
// notes):
//   * Row 0 of every tree is the root (anchor) token; the budget D counts the
//     draft nodes only.  [V4TREE toy: 7 nodes incl. root A, budget 3 keeps 3
//     non-root nodes]
//   * A node's score is its prefix (cumulative) probability, computed as
//     fp32 round-to-nearest products in depth order.  Ties are broken by the
//     total order (score desc, depth asc, rank tuple lexicographic asc).
//   * The mask of row r has bit j-1 set iff row j (j >= 1) is an ancestor of r
//     or r itself; the root is visible to every row and is not in the mask.
//   * Softmax scale is passed in explicitly.
//   * Greedy acceptance: argmax with ties to the lowest id; if several children
//     carry the wanted token, the lowest row wins.
//
// Floating point: attention is computed in double from inputs converted
// exactly (fp32 or bf16 -> double).  Tree scores are fp32 on purpose (that is
// the quantity being ranked).  Build with -O2 -ffp-contract=off, no fast-math.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- helpers --

// Number of worker threads: 0 or negative means "all hardware threads".
int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  unsigned h = std::thread::hardware_concurrency();
  return h == 0 ? 1 : (int)h;
}

// Run fn(i) for i in [0, n) over nthreads std::threads (static striping).
template <class F>
void parallel_for(long n, int nthreads, F fn) {
  nthreads = resolve_threads(nthreads);
  if (nthreads <= 1 || n <= 1) {
    for (long i = 0; i < n; ++i) fn(i);
    return;
  }
  if (nthreads > n) nthreads = (int)n;
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t)
    pool.emplace_back([=, &fn]() {
      for (long i = t; i < n; i += nthreads) fn(i);
    });
  for (auto& th : pool) th.join();
}

// Exact widening of one stored element to double.  dtype 0 = fp32, 1 = bf16
// (a bf16 value is the upper half of an fp32 bit pattern).
inline double load_elem(const void* base, long idx, int dtype) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return (double)f;
}

// A draft path: the top-k rank chosen at each depth, and its fp32 score.
struct Path {
  float score;
  int len;
  int rank[16];
};

// The total order of the tree build: higher score first, then shorter path,
// then lexicographically smaller rank tuple.
bool path_before(const Path& a, const Path& b) {
  if (a.score != b.score) return a.score > b.score;
  if (a.len != b.len) return a.len < b.len;
  for (int i = 0; i < a.len; ++i)
    if (a.rank[i] != b.rank[i]) return a.rank[i] < b.rank[i];
  return false;
}

bool same_prefix(const Path& child, const Path& parent) {
  if (child.len != parent.len + 1) return false;
  for (int i = 0; i < parent.len; ++i)
    if (child.rank[i] != parent.rank[i]) return false;
  return true;
}

// Turn the D kept paths (already sorted in the total order) into the row
// arrays of one request.  Row 0 is the root.  Returns 0, or -1 if the kept set
// is not closed under taking parents (cannot happen for a valid build).
int emit_rows(const std::vector<Path>& kept, int k, const float* top_p,
              const int32_t* top_id, int32_t root_tok, int32_t* token,
              int32_t* parent, int32_t* depth, float* score, uint64_t* mask,
              uint8_t* is_leaf) {
  (void)top_p;
  const int D = (int)kept.size();
  token[0] = root_tok;
  parent[0] = -1;
  depth[0] = 0;
  score[0] = 1.0f;
  mask[0] = 0;
  for (int i = 0; i < D; ++i) {
    const Path& p = kept[i];
    const int row = i + 1;
    const int s = p.len - 1;  // position index of this node's token
    token[row] = top_id[s * k + p.rank[s]];
    depth[row] = p.len;
    score[row] = p.score;
    int par = -1;
    if (p.len == 1) {
      par = 0;
    } else {
      for (int j = 0; j < i; ++j)
        if (same_prefix(p, kept[j])) { par = j + 1; break; }
    }
    if (par < 0) return -1;
    parent[row] = par;
    mask[row] = (par == 0 ? 0ull : mask[par]) | (1ull << (row - 1));
  }
  for (int r = 0; r <= D; ++r) {
    bool has_child = false;
    for (int c = 1; c <= D; ++c)
      if (parent[c] == r) has_child = true;
    is_leaf[r] = has_child ? 0 : 1;
  }
  return 0;
}

}  // namespace

extern "C" {

int oracle_hardware_threads(void) { return resolve_threads(0); }

// ------------------------------------------------------------------ top-k --
// For every (request b, position s) row of probs[B][S][V], the k most probable
// tokens, ordered by (probability desc, token id asc).  [V4TREE toy step 1:
// "top-k is the number of branches kept per step"; CADD Method: per-position
// marginals from a one-pass block drafter.]  Plain definition: sort the whole
// row and keep the first k.
void oracle_topk(const float* probs, int B, int S, int V, int k,
                 float* top_p, int32_t* top_id, int nthreads) {
  if (k < 1 || k > V) return;
  parallel_for((long)B * S, nthreads, [&](long row) {
    const float* p = probs + row * (long)V;
    std::vector<int32_t> ids(V);
    for (int v = 0; v < V; ++v) ids[v] = v;
    std::sort(ids.begin(), ids.end(), [&](int32_t a, int32_t b) {
      if (p[a] != p[b]) return p[a] > p[b];
      return a < b;
    });
    for (int j = 0; j < k; ++j) {
      top_p[row * k + j] = p[ids[j]];
      top_id[row * k + j] = ids[j];
    }
  });
}

// ------------------------------------------------------------ tree build --
// Greedy best-first draft tree under budget D [CADD Method 2; V4TREE toy
// step 2 (budget pruning keeps the top-D nodes by cumulative score)].
// Children of a node at depth d are the top-k tokens of position d+1 (the
// per-position marginals of a one-pass drafter, [CADD Method]).
//
// oracle_tree_enum: the definition itself.  Enumerate every path of length
// 1..S over the rank indices, score it by fp32 products in depth order, sort
// by the total order and keep the first D.  Feasible while sum_l k^l is a few
// million.
//
// Inputs top_p/top_id are [B][S][k] (from oracle_topk).  Outputs are
// [B][1+D].  Returns 0, or -1 on an impossible budget.
int oracle_tree_enum(const float* top_p, const int32_t* top_id, int B, int S,
                     int k, int D, const int32_t* root_tok, int32_t* token,
                     int32_t* parent, int32_t* depth, float* score,
                     uint64_t* mask, uint8_t* is_leaf) {
  if (S < 1 || S > 16 || k < 1 || D < 1 || D > 64) return -1;
  for (int b = 0; b < B; ++b) {
    const float* tp = top_p + (long)b * S * k;
    const int32_t* ti = top_id + (long)b * S * k;
    std::vector<Path> all;
    // breadth-first enumeration: level l paths extend level l-1 paths
    std::vector<Path> level(1);
    level[0].score = 1.0f;
    level[0].len = 0;
    for (int l = 1; l <= S; ++l) {
      std::vector<Path> next;
      next.reserve(level.size() * (size_t)k);
      for (const Path& p : level)
        for (int r = 0; r < k; ++r) {
          Path c = p;
          c.len = l;
          c.rank[l - 1] = r;
          c.score = p.score * tp[(l - 1) * k + r];  // fp32 product
          next.push_back(c);
        }
      all.insert(all.end(), next.begin(), next.end());
      level.swap(next);
    }
    if ((long)all.size() < D) return -1;
    std::sort(all.begin(), all.end(), path_before);
    all.resize(D);
    const long o = (long)b * (D + 1);
    if (emit_rows(all, k, tp, ti, root_tok[b], token + o, parent + o,
                  depth + o, score + o, mask + o, is_leaf + o) != 0)
      return -1;
  }
  return 0;
}

// oracle_tree_beam: the same top-D, reached by a level-wise beam that keeps
// the D best paths of each level (under the same total order) and extends only
// those.  Exact: a path in the global top-D has all its ancestors in the global
// top-D (a child never precedes its parent: its score is a product with a
// factor <= 1 and it is longer), so at every level the global top-D members are
// among the top-D extensions of the previous level's beam.  Used where full
// enumeration is too large (k=10, S=8 gives 1.1e8 paths).
int oracle_tree_beam(const float* top_p, const int32_t* top_id, int B, int S,
                     int k, int D, const int32_t* root_tok, int32_t* token,
                     int32_t* parent, int32_t* depth, float* score,
                     uint64_t* mask, uint8_t* is_leaf) {
  if (S < 1 || S > 16 || k < 1 || D < 1 || D > 64) return -1;
  for (int b = 0; b < B; ++b) {
    const float* tp = top_p + (long)b * S * k;
    const int32_t* ti = top_id + (long)b * S * k;
    std::vector<Path> pool;
    std::vector<Path> beam(1);
    beam[0].score = 1.0f;
    beam[0].len = 0;
    for (int l = 1; l <= S; ++l) {
      std::vector<Path> next;
      for (const Path& p : beam)
        for (int r = 0; r < k; ++r) {
          Path c = p;
          c.len = l;
          c.rank[l - 1] = r;
          c.score = p.score * tp[(l - 1) * k + r];
          next.push_back(c);
        }
      std::sort(next.begin(), next.end(), path_before);
      if ((int)next.size() > D) next.resize(D);
      pool.insert(pool.end(), next.begin(), next.end());
      beam.swap(next);
    }
    if ((long)pool.size() < D) return -1;
    std::sort(pool.begin(), pool.end(), path_before);
    pool.resize(D);
    const long o = (long)b * (D + 1);
    if (emit_rows(pool, k, tp, ti, root_tok[b], token + o, parent + o,
                  depth + o, score + o, mask + o, is_leaf + o) != 0)
      return -1;
  }
  return 0;
}

// ----------------------------------------------------- verify attention --
// Branch-aware tree-verify attention [V4TREE research gap item 1: a candidate
// sees only its own ancestors, never another branch; toy step 3: A-B-B sees A
// and A-B, A-C sees only A].  For request b, tree row r, query head h (KV head
// h / (Hq/Hkv)) the visible keys are the prefix positions 0..P_b-1 of the
// persistent cache, the root row of the scratch pad, and every scratch row j
// >= 1 whose bit j-1 is set in mask[b][r].  Plain softmax attention in double:
//   s_j = scale * <q, k_j>,  m = max_j s_j,
//   o = sum_j e^{s_j - m} v_j / sum_j e^{s_j - m},  lse = m + ln sum_j e^{s_j-m}.
//
// Layouts: q[B][R][Hq][dk]; kcache[B][Hkv][cap][dk]; vcache[B][Hkv][cap][dv];
// ktree[B][R][Hkv][dk]; vtree[B][R][Hkv][dv]; mask[B][R].  If v_aliases_k, the
// value vector is the first dv entries of the key vector and vcache/vtree are
// ignored (latent-KV attention).  dtype 0 = fp32, 1 = bf16.
//
// sel: nsel triples (b, r, h) to compute, or NULL for all B*R*Hq rows in
// (b, r, h) order.  out[nrows][dv], lse[nrows] in double.
void oracle_verify_attn(int B, int R, int Hq, int Hkv, int dk, int dv,
                        int cap, int dtype, int v_aliases_k, double scale,
                        const void* q, const void* kcache, const void* vcache,
                        const int32_t* prefix_len, const void* ktree,
                        const void* vtree, const uint64_t* mask, int nsel,
                        const int32_t* sel, double* out, double* lse,
                        int nthreads) {
  const int g = Hq / Hkv;
  const long nrows = sel ? (long)nsel : (long)B * R * Hq;
  parallel_for(nrows, nthreads, [&](long i) {
    int b, r, h;
    if (sel) {
      b = sel[3 * i];
      r = sel[3 * i + 1];
      h = sel[3 * i + 2];
    } else {
      b = (int)(i / ((long)R * Hq));
      r = (int)((i / Hq) % R);
      h = (int)(i % Hq);
    }
    const int hk = h / g;
    std::vector<double> qv(dk);
    const long qoff = (((long)b * R + r) * Hq + h) * dk;
    for (int c = 0; c < dk; ++c) qv[c] = load_elem(q, qoff + c, dtype);

    // gather the visible keys as (key base, value base) element offsets
    struct KeyRef { const void* kb; long ko; const void* vb; long vo; };
    std::vector<KeyRef> keys;
    const int P = prefix_len[b];
    for (int t = 0; t < P; ++t) {
      const long ko = (((long)b * Hkv + hk) * cap + t) * dk;
      if (v_aliases_k)
        keys.push_back({kcache, ko, kcache, ko});
      else
        keys.push_back({kcache, ko, vcache, (((long)b * Hkv + hk) * cap + t) * dv});
    }
    const uint64_t m_r = (r == 0) ? 0ull : mask[(long)b * R + r];
    for (int j = 0; j < R; ++j) {
      const bool visible = (j == 0) || ((m_r >> (j - 1)) & 1ull);
      if (!visible) continue;
      const long ko = (((long)b * R + j) * Hkv + hk) * dk;
      if (v_aliases_k)
        keys.push_back({ktree, ko, ktree, ko});
      else
        keys.push_back({ktree, ko, vtree, (((long)b * R + j) * Hkv + hk) * dv});
    }

    std::vector<double> s(keys.size());
    double m = -INFINITY;
    for (size_t j = 0; j < keys.size(); ++j) {
      double dot = 0.0;
      for (int c = 0; c < dk; ++c) dot += qv[c] * load_elem(keys[j].kb, keys[j].ko + c, dtype);
      s[j] = scale * dot;
      if (s[j] > m) m = s[j];
    }
    double denom = 0.0;
    std::vector<double> acc(dv, 0.0);
    for (size_t j = 0; j < keys.size(); ++j) {
      const double w = std::exp(s[j] - m);
      denom += w;
      for (int c = 0; c < dv; ++c) acc[c] += w * load_elem(keys[j].vb, keys[j].vo + c, dtype);
    }
    for (int c = 0; c < dv; ++c) out[i * dv + c] = acc[c] / denom;
    lse[i] = m + std::log(denom);
  });
}

// ---------------------------------------------------------------- argmax --
// Greedy target choice per tree row: the id of the largest logit, ties to the
// lowest id.  [V4TREE toy step 5 / DSPARK decoding cycle: the target checks
// each draft token against its own prediction.]
void oracle_argmax(const float* logits, long rows, int V, int32_t* out,
                   int nthreads) {
  parallel_for(rows, nthreads, [&](long r) {
    const float* x = logits + r * (long)V;
    int best = 0;
    for (int v = 1; v < V; ++v)
      if (x[v] > x[best]) best = v;
    out[r] = best;
  });
}

// ----------------------------------------------------------- accept walk --
// Greedy accepted-path selection [V4TREE toy steps 5-6; DSPARK decoding cycle].
// Start at the root u = 0.  While some child c of u (parent[c] == u) carries
// token[c] == tgt[u], append the lowest such c and move to it.  The accepted
// length L is the number of appended draft rows; the bonus (correction) token
// is tgt at the last accepted row.  chain_id is the lowest leaf row whose
// ancestor-or-self set contains the last accepted row (the chain of the
// verify-preprocess decomposition [V4TREE toy step 4]); -1 when L = 0.
//
// tgt/token/parent/is_leaf are [B][R]; mask [B][R]; accept_rows [B][S+1] gets
// rows 0..L then -1.  Returns 0, or 1 if a tree is malformed (the request's
// outputs are then L=0 with the root only).
int oracle_accept_walk(const int32_t* tgt, int B, int R, int S,
                       const int32_t* token, const int32_t* parent,
                       const uint64_t* mask, const uint8_t* is_leaf,
                       int32_t* accept_len, int32_t* accept_rows,
                       int32_t* bonus, int32_t* chain_id) {
  int status = 0;
  for (int b = 0; b < B; ++b) {
    const long o = (long)b * R;
    int32_t* rows = accept_rows + (long)b * (S + 1);
    for (int i = 0; i <= S; ++i) rows[i] = -1;
    rows[0] = 0;
    int u = 0, L = 0;
    bool bad = false;
    for (;;) {
      int next = -1;
      for (int c = 1; c < R; ++c)
        if (parent[o + c] == u && token[o + c] == tgt[o + u]) { next = c; break; }
      if (next < 0) break;
      if (L == S) { bad = true; break; }
      ++L;
      rows[L] = next;
      u = next;
    }
    if (bad) {
      status = 1;
      for (int i = 1; i <= S; ++i) rows[i] = -1;
      u = 0;
      L = 0;
    }
    accept_len[b] = L;
    bonus[b] = tgt[o + u];
    int chain = -1;
    if (L > 0)
      for (int c = 1; c < R; ++c)
        if (is_leaf[o + c] && ((mask[o + c] >> (u - 1)) & 1ull)) { chain = c; break; }
    chain_id[b] = chain;
  }
  return status;
}

// ---------------------------------------------------------------- commit --
// Accepted-path commit [V4TREE "Secret weapon" and toy step 6: only the
// accepted chain's KV is written to the persistent cache; rejected branches in
// the scratch pad are dropped; the next round starts from the new prefix].
// For each request: scratch rows accept_rows[0..L] go, in order, to cache
// positions P_b .. P_b+L of every KV head; then prefix_len[b] = P_b + 1 + L.
// A request whose new length would exceed cap is skipped (nothing written) and
// reported: returns the number of skipped requests.  elem_bytes is 4 or 2.
int oracle_commit(int B, int R, int Hkv, int dk, int dv, int cap, int S,
                  int elem_bytes, int v_aliases_k, const void* ktree,
                  const void* vtree, const int32_t* accept_rows,
                  const int32_t* accept_len, void* kcache, void* vcache,
                  int32_t* prefix_len) {
  int skipped = 0;
  for (int b = 0; b < B; ++b) {
    const int L = accept_len[b];
    const int P = prefix_len[b];
    if (P + 1 + L > cap) { ++skipped; continue; }
    for (int i = 0; i <= L; ++i) {
      const int row = accept_rows[(long)b * (S + 1) + i];
      for (int h = 0; h < Hkv; ++h) {
        const long src_k = (((long)b * R + row) * Hkv + h) * dk;
        const long dst_k = (((long)b * Hkv + h) * cap + (P + i)) * dk;
        std::memcpy((char*)kcache + dst_k * elem_bytes,
                    (const char*)ktree + src_k * elem_bytes, (size_t)dk * elem_bytes);
        if (!v_aliases_k) {
          const long src_v = (((long)b * R + row) * Hkv + h) * dv;
          const long dst_v = (((long)b * Hkv + h) * cap + (P + i)) * dv;
          std::memcpy((char*)vcache + dst_v * elem_bytes,
                      (const char*)vtree + src_v * elem_bytes, (size_t)dv * elem_bytes);
        }
      }
    }
    prefix_len[b] = P + 1 + L;
  }
  return skipped;
}

}  // extern "C"
