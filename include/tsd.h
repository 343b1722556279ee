/*
 * tsd.h -- C ABI of the GB300 tree-speculative-decoding verify step.
 *
 * One verify step of tree-structured speculative decoding, as four calls on
 * one CUDA stream:
 *
 *   tsd_tree_build        per-position top-k of the draft marginals, then the
 *                         greedy best-first draft tree under a node budget D
 *   tsd_tree_verify_attn  branch-aware attention of every tree node over the
 *                         shared prefix KV cache plus its own ancestors
 *   tsd_accept_walk       target argmax per node, greedy walk to the accepted
 *                         path, bonus (correction) token, chain id
 *   tsd_commit_path       copy the accepted path's scratch KV into the cache
 *   tsd_accept_commit     the walk and the commit in one call (also in two
 *                         parts: tsd_target_argmax, tsd_walk_commit)
 *
 * Sources of the operations (web pages, by title and section):
 *   "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for
 *    Efficient Inference" (review): Key idea (tree under a verification
 *    budget D); Background, research gap item 1 (a candidate sees only its own
 *    ancestors); "How it works" toy example steps 1-6 (top-k expansion, budget
 *    pruning, tree attention fed with layout and metadata only, chains, greedy
 *    accepted path, commit of that path only); "Secret weapon" (scratch pad).
 *   "Cost-Aware Diffusion Draft Trees for Speculative Decoding": Method items
 *    1-2 (per-position marginals of a one-pass drafter; the greedy best-first
 *    tree picks the node of highest prefix probability).
 *   "DSpark: Speculative decoding ...": Architecture, decoding cycle (anchor
 *    token, accepted prefix, rejected draft, correction token).
 *
 * Conventions shared by every call
 *   - All array pointers are DEVICE pointers, allocated and owned by the
 *     caller, 16-byte aligned, dense row-major in the layouts given below.
 *     The library never allocates, frees or synchronises; scratch memory is a
 *     caller-provided workspace of the size the matching *_workspace_size call
 *     returns (for the current device).
 *   - Every call only enqueues kernels on `stream` and returns.  Outputs are
 *     valid once the stream has reached that point.  Kernels are launched
 *     with programmatic stream serialisation: one may be scheduled while the
 *     kernel before it on the stream is finishing, but it reads and writes
 *     no memory before that kernel has completed, so stream order is kept
 *     (its set-up and L2 prefetch hints overlap the predecessor).
 *   - The return value reports HOST-side validation and launch errors.  On any
 *     non-OK return nothing was enqueued, except TSD_ERR_CUDA from a failed
 *     launch (check cudaGetLastError semantics).
 *   - Problems found on the device (a request that would overflow the cache,
 *     a malformed caller-supplied tree) are written to the caller's `err`
 *     word: 0 means OK, otherwise (TSD_DEV_ERR_* code) | request index.  The
 *     first error wins; the library never clears `err` (the caller zeroes it).
 *     The offending request is skipped; the others are processed normally.
 *   - Row 0 of every tree is the root (the anchor token produced by the target
 *     in the previous round); rows 1..D are draft nodes; R = 1 + D.
 *   - Limits: 1 <= k <= 32, k <= V, 1 <= S <= 16, 1 <= D <= 64 and
 *     D <= sum_{s=1..S} k^s; Hq % Hkv == 0; head dims as listed per call.
 */
#ifndef TSD_H_
#define TSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream; ABI-identical to cudaStream_t (NULL = the legacy stream). */
typedef struct CUstream_st* tsd_stream_t;

typedef enum {
  TSD_OK = 0,
  TSD_ERR_INVALID_ARG = 1,    /* bad size, null or misaligned pointer, short workspace */
  TSD_ERR_UNSUPPORTED = 2,    /* a valid request the library does not implement */
  TSD_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
  TSD_ERR_DEVICE = 4,         /* reserved: device-side problems go to the err word */
  TSD_ERR_DEVICE_TIMEOUT = 5  /* a bounded device wait gave up */
} tsd_status;

/* Codes in the device error word (high byte); low 24 bits = request index. */
#define TSD_DEV_ERR_CAPACITY 0x01000000 /* commit would pass the cache capacity */
#define TSD_DEV_ERR_BAD_TREE 0x02000000 /* parent/row out of range, walk deeper than S */
#define TSD_DEV_ERR_TIMEOUT  0x03000000 /* a bounded wait inside a kernel gave up */
#define TSD_DEV_ERR_BAD_PAGE 0x04000000 /* page table entry outside the page pool */
#define TSD_DEV_ERR_BAD_PROBS 0x05000000 /* a draft probability above 1 or NaN */
#define TSD_DEV_ERR_MASK     0x7f000000

/* Element types of attention operands. */
#define TSD_F32 0
#define TSD_BF16 1

/* Static text for a status code. */
const char* tsd_status_string(tsd_status s);

/* Library version, major*10000 + minor*100 + patch. */
int tsd_version(void);

/* --------------------------------------------------------------------------
 * tsd_tree_build
 *
 * Per-position top-k then greedy best-first tree ("Cost-Aware Diffusion Draft
 * Trees", Method 2; V4 review, toy steps 1-2).
 *
 * probs     [B][S][V] fp32: the draft's per-position marginal distributions,
 *           values in [0, 1] (-0.0 counts as +0.0).  The best-first order
 *           relies on a child's score never exceeding its parent's, i.e. on
 *           p <= 1: a row holding a value above 1 or a NaN sets
 *           TSD_DEV_ERR_BAD_PROBS | b in err (the first error wins), and that
 *           request's tree is then unspecified (it is still a valid tree).
 * root_tok  [B] int32: the root (anchor) token of each request.
 * Outputs, all [B][1+D]:
 *   token   int32  row's token (row 0 = root_tok)
 *   parent  int32  parent row (-1 for the root)
 *   depth   int32  0 for the root, else 1..S
 *   score   fp32   prefix probability: fp32 product of the top-k
 *                  probabilities along the path, in depth order (1.0 for root)
 *   mask    uint64 bit j-1 set iff row j (j >= 1) is an ancestor of the row or
 *                  the row itself; the root is implicit (visible to all rows)
 *   is_leaf uint8  1 iff no row has this row as parent
 *
 * Children of a node at depth d are the k most probable tokens of position
 * d+1, ordered by (probability desc, token id asc).  Rows 1..D are the first D
 * paths in the total order (score desc, depth asc, tuple of top-k ranks
 * lexicographic asc), which lists parents before children.
 * ws: tsd_tree_build_workspace_size(B, S, V, k) bytes of device scratch.
 * -------------------------------------------------------------------------- */
size_t tsd_tree_build_workspace_size(int B, int S, int V, int k);

tsd_status tsd_tree_build(const float* probs, int B, int S, int V, int k, int D,
                          const int32_t* root_tok, int32_t* token,
                          int32_t* parent, int32_t* depth, float* score,
                          uint64_t* mask, uint8_t* is_leaf, void* ws,
                          size_t ws_bytes, int32_t* err, tsd_stream_t stream);

/* --------------------------------------------------------------------------
 * tsd_tree_build_adaptive
 *
 * The same tree with a per-request node count chosen by the cost-aware greedy
 * rule ("Cost-Aware Diffusion Draft Trees", Method items 1, 3 and 4): nodes
 * are taken in the best-first order of tsd_tree_build and node n+1 is kept
 * only while it raises the expected throughput (1 + Phi(T)) / (C_d + C_v(|T|)),
 * Phi being the sum of the kept nodes' scores (the expected number of
 * accepted draft tokens); the first node that does not raise it ends the
 * tree.  When C_v is convex and non-decreasing in the node count, the
 * objective is unimodal and this stop is its maximum over 0..D_max.
 * Arithmetic, fixed so that every implementation takes the same decision:
 *   A_0 = 1, A_n = fp32(A_{n-1} + score_n);  cost_n = fp32(C_d + C_v(n));
 *   keep node n+1  <=>  fp32(A_{n+1} * cost_n) > fp32(A_n * cost_{n+1}).
 *
 * cost_d   [B] fp32: drafting cost of the round (any time unit).
 * cost_v   [B][1+D_max] fp32: verify cost with n = 0..D_max draft nodes at the
 *          request's context length, in the same unit (for example from a
 *          convex fit to measured step latencies).
 * n_nodes  [B] int32 out: the kept count n* (0..D_max).
 * Other arguments and outputs as tsd_tree_build with D = D_max; rows
 * n*+1..D_max are inert padding (token -1, parent 0, depth 0, score 0,
 * mask 0, is_leaf 0), which tsd_tree_verify_attn, tsd_accept_walk and
 * tsd_commit_path accept and never take into the accepted path.  Leaves are
 * computed over the kept rows only.
 * ws: tsd_tree_build_workspace_size(B, S, V, k) bytes.
 * -------------------------------------------------------------------------- */
tsd_status tsd_tree_build_adaptive(const float* probs, int B, int S, int V, int k,
                                   int D_max, const int32_t* root_tok,
                                   const float* cost_d, const float* cost_v,
                                   int32_t* token, int32_t* parent, int32_t* depth,
                                   float* score, uint64_t* mask, uint8_t* is_leaf,
                                   int32_t* n_nodes, void* ws, size_t ws_bytes,
                                   int32_t* err, tsd_stream_t stream);

/* --------------------------------------------------------------------------
 * tsd_tree_build_conditioned
 *
 * The best-first tree over a caller-given candidate forest whose proposals are
 * conditioned on their parent node (EAGLE-style drafting: each node's children
 * are the drafter's proposals at that node), as in the V4 review's toy example
 * ("How it works" steps 1-2: B proposes B and C, C proposes A and B; the
 * expanded tree is pruned to the D nodes of highest cumulative score), with
 * the greedy best-first choice of "Cost-Aware Diffusion Draft Trees", Method
 * item 2.
 *
 * cand_p      [B][C] fp32 in [0, 1]: probability of candidate c given its parent
 * cand_tok    [B][C] int32: token of candidate c
 * cand_parent [B][C] int32: index of c's parent candidate (< c), or -1 for a
 *             child of the root (candidates are listed parents first)
 * Score of a candidate: fp32 product of cand_p along its path, in depth order
 * (1.0 for the root).  Rows 1..D are the first D candidates in the order
 * (score desc, depth asc, candidate index asc), which lists parents before
 * children; outputs as tsd_tree_build.  Limits: 1 <= C <= 2048, 1 <= D <=
 * min(64, C).  A forest with a parent index out of range, a probability outside
 * [0, 1] (or NaN), or fewer than D candidates within depth 65 sets
 * TSD_DEV_ERR_BAD_TREE | b in err and gives request b a root-only tree (rows
 * 1..D inert padding: token -1, parent 0, depth 0, score 0, mask 0, not leaf).
 * -------------------------------------------------------------------------- */
tsd_status tsd_tree_build_conditioned(const float* cand_p, const int32_t* cand_tok,
                                      const int32_t* cand_parent, int B, int C, int D,
                                      const int32_t* root_tok, int32_t* token,
                                      int32_t* parent, int32_t* depth, float* score,
                                      uint64_t* mask, uint8_t* is_leaf, int32_t* err,
                                      tsd_stream_t stream);

/* --------------------------------------------------------------------------
 * tsd_tree_verify_attn
 *
 * Branch-aware tree attention (V4 review, research gap item 1 and toy step 3).
 * For request b, tree row r and query head h (KV head h / (Hq/Hkv)), the
 * visible keys are the cached prefix positions 0..prefix_len[b]-1, the root
 * row of the scratch pad, and every scratch row j >= 1 with bit j-1 of
 * mask[b][r] set (for r = 0: the root only).  Output is
 *   out = softmax(scale * q . K^T) V,   lse = natural log of the softmax
 *   denominator including its max (logsumexp of the scaled scores),
 * accumulated in fp32; out has the element type of q.
 *
 * Layouts (element type `dtype`, TSD_F32 or TSD_BF16):
 *   q      [B][R][Hq][dk]
 *   kcache [B][Hkv][cap][dk]      vcache [B][Hkv][cap][dv]
 *   ktree  [B][R][Hkv][dk]        vtree  [B][R][Hkv][dv]   (scratch pad)
 *   prefix_len [B] int32 (0 <= P_b <= cap; values outside are clamped)
 *   mask   [B][R] uint64 (as produced by tsd_tree_build)
 *   out    [B][R][Hq][dv]         lse [B][R][Hq] fp32
 * With v_aliases_k (latent attention) the value is the first dv entries of
 * the key; vcache/vtree are ignored and may be NULL; dv <= dk.
 * Supported head dims: dk == dv in {64, 128}, or dk = 576, dv = 512 with
 * v_aliases_k.  fp32 inputs are computed on CUDA cores in fp32 (never TF32).
 * ws: tsd_verify_workspace_size(desc) bytes (0 is a valid size).
 * -------------------------------------------------------------------------- */
typedef struct {
  int B;            /* requests */
  int R;            /* tree rows per request, 1 + D, 1 <= R <= 65 */
  int Hq, Hkv;      /* query heads, KV heads (Hq % Hkv == 0) */
  int dk, dv;       /* key/query and value head dims */
  int cap;          /* cache capacity in tokens (positions per head) */
  int dtype;        /* TSD_F32 or TSD_BF16 */
  int v_aliases_k;  /* 1: value = key[:dv] (latent KV), 0: separate V */
  float scale;      /* softmax scale applied to q . k */
} tsd_attn_desc;

size_t tsd_verify_workspace_size(const tsd_attn_desc* desc);

tsd_status tsd_tree_verify_attn(const tsd_attn_desc* desc, const void* q,
                                const void* kcache, const void* vcache,
                                const int32_t* prefix_len, const void* ktree,
                                const void* vtree, const uint64_t* mask,
                                void* out, float* lse, void* ws,
                                size_t ws_bytes, int32_t* err,
                                tsd_stream_t stream);

/* Attention paths of tsd_tree_verify_attn / tsd_tree_verify_attn_paged.  The
 * automatic choice is tcgen05 for bf16 heads of 128 dims with at least 16
 * packed rows (tree rows x query heads per KV head) and for latent heads with
 * at least 64; the legacy mma.sync path for other bf16 heads of 64 or 128
 * dims with at least 64 packed rows; CUDA cores (fp32 arithmetic) otherwise. */
#define TSD_PATH_AUTO 0
#define TSD_PATH_CUDA_CORE 1
#define TSD_PATH_MMA_SYNC 2
#define TSD_PATH_TCGEN05 3

/* Diagnostic: force one attention path for the verify calls that follow, and
 * for tsd_verify_workspace_size (a forced path that cannot run a given call
 * falls back to the automatic choice).  No counterpart on the pages: it lets
 * tests check every path against an independent reference.  The setting is
 * process-wide; change it only while no other thread is enqueueing verify
 * calls, and size workspaces under the same setting as the calls.  Returns
 * the previous setting, or -1 (and changes nothing) for an unknown path. */
int tsd_set_verify_path(int path);

/* Diagnostic: the budget, in SM clock cycles, of the pipeline waits inside
 * the tcgen05 attention kernel of bf16 heads for the verify calls that follow
 * (the waits on its copy, product and softmax stages; the final waits that
 * let copies and products in flight land before the kernel exits keep the
 * default of about one second).  0 restores the default; a positive budget
 * below it makes those waits poll without sleeping and give up once it is
 * spent, after which the kernel writes no output for the CTA's rows and sets
 * TSD_DEV_ERR_TIMEOUT | b in err -- the path a stalled copy or product takes,
 * made reachable without a fault.  No counterpart on the pages.  Process-wide,
 * like tsd_set_verify_path.  Returns the previous setting (0 = default). */
long long tsd_set_wait_budget(long long cycles);

/* --------------------------------------------------------------------------
 * Paged KV cache: tsd_tree_verify_attn_paged, tsd_commit_path_paged
 *
 * The same calls over a cache held in fixed-size pages (V4 review, "Secret
 * weapon": the persistent cache and the scratch pad are separate, and only
 * the accepted path is written back).  The caller owns the pages and the
 * page table; these calls neither allocate nor move pages.
 *
 * kpool, vpool  [num_pages][Hkv][page_size][dk | dv]: page pools, element type
 *               as desc->dtype (vpool unused and may be NULL when V aliases K);
 *               one head's rows of a page are contiguous.
 * page_table    [B][max_pages] int32: page_table[b][j] is the pool page that
 *               holds positions j*page_size .. (j+1)*page_size - 1 of request b.
 * page_size     a multiple of 128; desc->cap must equal max_pages * page_size.
 * Position pos of request b, head h, is row
 *   (page_table[b][pos / page_size] * Hkv + h) * page_size + pos % page_size
 * of the pool.  Everything else (arguments, outputs, workspace sizes,
 * tolerances) is as for tsd_tree_verify_attn / tsd_commit_path; results are
 * identical to those calls on the gathered contiguous cache.  Only the pages
 * of positions the call reads (verify: 0..P-1) or writes (commit: P..P+L) are
 * looked up; such an entry outside [0, num_pages) is never dereferenced and
 * sets TSD_DEV_ERR_BAD_PAGE | b (verify: the request's output is not valid;
 * commit: the request is skipped).
 * -------------------------------------------------------------------------- */
tsd_status tsd_tree_verify_attn_paged(const tsd_attn_desc* desc, const void* q,
                                      const void* kpool, const void* vpool,
                                      const int32_t* page_table, int max_pages,
                                      int page_size, int num_pages,
                                      const int32_t* prefix_len, const void* ktree,
                                      const void* vtree, const uint64_t* mask,
                                      void* out, float* lse, void* ws, size_t ws_bytes,
                                      int32_t* err, tsd_stream_t stream);

tsd_status tsd_commit_path_paged(const tsd_attn_desc* desc, int S, const void* ktree,
                                 const void* vtree, const int32_t* accept_rows,
                                 const int32_t* accept_len, void* kpool, void* vpool,
                                 const int32_t* page_table, int max_pages, int page_size,
                                 int num_pages, int32_t* prefix_len, int32_t* err,
                                 tsd_stream_t stream);

/* --------------------------------------------------------------------------
 * tsd_accept_walk
 *
 * Greedy accepted-path selection (V4 review, toy steps 5-6; DSpark decoding
 * cycle).  tgt[r] = argmax_v logits[b][r][v] (ties to the lowest v).  Starting
 * at the root u = 0: while some child c of u (parent[c] == u) has token[c] ==
 * tgt[u], append the lowest such c and move to it.
 *
 * logits     [B][1+D][V] fp32 target logits of every tree row (no NaN).
 * token/parent [B][1+D] int32, mask [B][1+D] uint64, is_leaf [B][1+D] uint8:
 *            a tree as produced by tsd_tree_build (or any tree with parent[c]
 *            < c, depth <= S; a violation sets TSD_DEV_ERR_BAD_TREE).
 * Outputs:
 *   tgt          [B][1+D] int32, optional (NULL to skip): the argmax per row
 *   accept_len   [B] int32: L, the number of accepted draft rows
 *   accept_rows  [B][S+1] int32: 0, then the L accepted rows, then -1
 *   bonus        [B] int32: tgt at the last accepted row (next round's root)
 *   chain_id     [B] int32: lowest leaf row whose ancestor-or-self set holds
 *                the last accepted row (the chain of the tree's decomposition
 *                into root-to-leaf chains); -1 when L = 0
 * ws: tsd_accept_walk_workspace_size(B, D, V) bytes.
 * -------------------------------------------------------------------------- */
size_t tsd_accept_walk_workspace_size(int B, int D, int V);

tsd_status tsd_accept_walk(const float* logits, int B, int D, int S, int V,
                           const int32_t* token, const int32_t* parent,
                           const uint64_t* mask, const uint8_t* is_leaf,
                           int32_t* tgt, int32_t* accept_len,
                           int32_t* accept_rows, int32_t* bonus,
                           int32_t* chain_id, void* ws, size_t ws_bytes,
                           int32_t* err, tsd_stream_t stream);

/* --------------------------------------------------------------------------
 * tsd_accept_walk_static
 *
 * No counterpart on the pages: this is tsd_accept_walk for callers that cannot
 * allocate device memory -- code that is handed only its input and output
 * buffers, such as a custom operator inside another framework whose memory
 * planner owns the device heap, or a serving loop that allows no allocation
 * after start-up.  Arguments and results are those of tsd_accept_walk, minus
 * the workspace.  The scratch lives in a fixed 1 MiB array inside the library
 * (each GPU that loads the library holds it until the process exits); a call
 * whose tsd_accept_walk_workspace_size(B, D, V) exceeds 1 MiB returns
 * TSD_ERR_UNSUPPORTED.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress), so make that first call before any stream
 * capture.  The address is kept per device and looked up again when the
 * device's current context changes (a cudaDeviceReset gives the device a new
 * context and the array a new address): the first call after such a reset
 * must also come before any capture.  Calls that overlap on the GPU (on
 * different streams) share the array and race.  Nothing in the array needs
 * to start at zero.  The call allocates and frees nothing.
 * -------------------------------------------------------------------------- */
tsd_status tsd_accept_walk_static(const float* logits, int B, int D, int S, int V,
                                  const int32_t* token, const int32_t* parent,
                                  const uint64_t* mask, const uint8_t* is_leaf,
                                  int32_t* tgt, int32_t* accept_len,
                                  int32_t* accept_rows, int32_t* bonus,
                                  int32_t* chain_id, int32_t* err,
                                  tsd_stream_t stream);

/* --------------------------------------------------------------------------
 * tsd_accept_commit
 *
 * tsd_accept_walk followed by the commit of its accepted paths
 * (tsd_commit_path, or tsd_commit_path_paged when page_size > 0), in one call
 * and one kernel per request after the argmax scan: the walk's CTA copies the
 * path it found (V4 review, toy steps 5-6 and "Secret weapon").  Arguments are
 * those of the two calls: the walk's (logits .. chain_id, ws, err, stream),
 * then the commit's (desc, ktree, vtree, kcache / kpool, vcache / vpool,
 * page_table, max_pages, page_size, num_pages, prefix_len), with page_size = 0
 * (page_table NULL, max_pages and num_pages 0) for the contiguous cache.
 * desc->B must equal B and desc->R must equal D + 1.  accept_len and
 * accept_rows are written as by tsd_accept_walk (the commit does not read them
 * back).  Outputs, error codes and the cache contents are identical to the two
 * calls made in order.
 * ws: tsd_accept_walk_workspace_size(B, D, V) bytes.
 * -------------------------------------------------------------------------- */
tsd_status tsd_accept_commit(const float* logits, int B, int D, int S, int V,
                             const int32_t* token, const int32_t* parent,
                             const uint64_t* mask, const uint8_t* is_leaf,
                             int32_t* tgt, int32_t* accept_len,
                             int32_t* accept_rows, int32_t* bonus,
                             int32_t* chain_id, const tsd_attn_desc* desc,
                             const void* ktree, const void* vtree, void* kcache,
                             void* vcache, const int32_t* page_table, int max_pages,
                             int page_size, int num_pages, int32_t* prefix_len,
                             void* ws, size_t ws_bytes, int32_t* err,
                             tsd_stream_t stream);

/* --------------------------------------------------------------------------
 * tsd_target_argmax, tsd_walk_commit
 *
 * tsd_accept_commit in two parts.  The target argmax reads only the logits,
 * so a caller may run it on another stream, concurrently with the tree build
 * and the attention of the same step, and join the streams before the walk.
 *   tsd_target_argmax  writes the per-chunk argmax candidates of every row
 *                      of logits [B][1+D][V] to ws
 *                      (tsd_accept_walk_workspace_size(B, D, V) bytes).
 *   tsd_walk_commit    reads them from the same ws, merges them into tgt
 *                      and does the rest of tsd_accept_commit (walk, bonus,
 *                      chain id, commit); V is the logits' row length.
 * The caller orders the two (the argmax must have completed, with its writes
 * visible, before the walk starts: same stream, or an event between the
 * streams) and gives each its own ws while calls overlap.  In order on one
 * stream they are exactly tsd_accept_commit; arguments and device-side
 * errors as there.
 * -------------------------------------------------------------------------- */
tsd_status tsd_target_argmax(const float* logits, int B, int D, int V, void* ws,
                             size_t ws_bytes, tsd_stream_t stream);

tsd_status tsd_walk_commit(int B, int D, int S, int V, const int32_t* token,
                           const int32_t* parent, const uint64_t* mask,
                           const uint8_t* is_leaf, int32_t* tgt, int32_t* accept_len,
                           int32_t* accept_rows, int32_t* bonus, int32_t* chain_id,
                           const tsd_attn_desc* desc, const void* ktree,
                           const void* vtree, void* kcache, void* vcache,
                           const int32_t* page_table, int max_pages, int page_size,
                           int num_pages, int32_t* prefix_len, const void* ws,
                           size_t ws_bytes, int32_t* err, tsd_stream_t stream);

/* --------------------------------------------------------------------------
 * tsd_commit_path
 *
 * Accepted-path commit (V4 review, "Secret weapon" and toy step 6): only the
 * accepted chain's KV leaves the scratch pad.  For each request b with
 * P = prefix_len[b] and L = accept_len[b]: scratch rows accept_rows[b][0..L]
 * are copied, in order, to cache positions P..P+L of every KV head (K, and V
 * unless desc->v_aliases_k), then prefix_len[b] = P + 1 + L.  Rejected rows
 * and all other cache positions are left untouched.  A request with
 * P + 1 + L > cap is skipped and reported as TSD_DEV_ERR_CAPACITY; a row
 * index outside [0, R) as TSD_DEV_ERR_BAD_TREE.
 * desc gives B, R, Hkv, dk, dv, cap, dtype, v_aliases_k (Hq, scale unused).
 * S is the accept_rows row length minus one.  No workspace.
 * -------------------------------------------------------------------------- */
tsd_status tsd_commit_path(const tsd_attn_desc* desc, int S, const void* ktree,
                           const void* vtree, const int32_t* accept_rows,
                           const int32_t* accept_len, void* kcache,
                           void* vcache, int32_t* prefix_len, int32_t* err,
                           tsd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TSD_H_ */
