// tsd_accept_walk: target argmax per tree row, then the greedy walk from the
// root to the accepted path.
//
// Sources: "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4"
// (review), "How it works" steps 4-6 (the tree splits into root-to-leaf
// chains; the target checks all chains at once; the accepted prefix survives
// where a linear chain would die; only the accepted chain is kept) and
// "DSpark: Speculative decoding ...", Architecture, decoding cycle (drafts E
// and F accepted, G rejected, the target's own token G* becomes the
// correction / next anchor).
//
// K4 vocab_scan_kernel<true>: per-chunk argmax of every target-logit row
//    (HBM-bound scan; ties go to the lowest id).
// K5 accept_walk_kernel: one CTA per request.  Merges the chunk maxima into
//    tgt[r], checks the tree, walks (one warp): at row u, the child c
//    (parent[c] == u) with token[c] == tgt[u] is accepted (lowest row if
//    several), until no child matches.  Every row first checks, in parallel,
//    whether it matches the target at its parent, so a level of the walk is
//    one ballot.  In tsd_accept_commit the same CTA then
//    commits the accepted path (the commit of tsd_commit_path, with the path
//    taken from shared memory); its scratch-pad K/V rows were prefetched into
//    L2 at the kernel's start, so the copy reads L2.
#include "tsd_commit.cuh"
#include "tsd_common.cuh"
#include "tsd_host.h"
#include "tsd_scan.cuh"

#include <cuda.h>

#include <mutex>

namespace tsd {
namespace {

constexpr int kMaxR = 65;

constexpr int kWalkWarps = 32;   // one warp per tree row up to 32 rows: their chunk loads overlap

template <bool kCommit>
__global__ void __launch_bounds__(32 * kWalkWarps)
accept_walk_kernel(const uint64_t* __restrict__ part, int R, int S, int nchunk,
                   const int32_t* __restrict__ token, const int32_t* __restrict__ parent,
                   const uint64_t* __restrict__ mask, const uint8_t* __restrict__ is_leaf,
                   int32_t* __restrict__ tgt_out, int32_t* __restrict__ accept_len,
                   int32_t* __restrict__ accept_rows, int32_t* __restrict__ bonus,
                   int32_t* __restrict__ chain_id, int32_t* __restrict__ err, CommitArgs ca) {
  __shared__ int32_t s_tgt[kMaxR], s_tok[kMaxR], s_par[kMaxR];
  __shared__ uint64_t s_mask[kMaxR];
  __shared__ uint8_t s_leaf[kMaxR];
  __shared__ int32_t s_path[kCommitMaxRows];
  __shared__ int s_P, s_L;
  __shared__ CommitSmem s_commit;
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long o = (long)b * R;
  if (kCommit) {
    // the request's scratch-pad K/V rows into L2 (a hint, before the wait)
    const long kbytes = (long)R * ca.Hkv * ca.krow, vbytes = (long)R * ca.Hkv * ca.vrow;
    if (threadIdx.x == 0) prefetch_l2(ca.ktree + b * kbytes, kbytes);
    if (threadIdx.x == 32 && vbytes > 0) prefetch_l2(ca.vtree + b * vbytes, vbytes);
  }
  grid_dependency_sync();
  if (kCommit && threadIdx.x == 0) {
    s_P = ca.prefix_len[b];
    s_commit.code = kNoError;
  }

  // tree metadata, then tgt[r]: the largest of the row's chunk maxima.  Warp
  // w takes rows w, w+32, ...; its lanes split the (at most 256) chunks and
  // load them all at once.
  if (threadIdx.x < R) {   // (R <= 65: one row per thread)
    const int r = threadIdx.x;
    s_tok[r] = token[o + r];
    s_par[r] = parent[o + r];
    s_mask[r] = mask[o + r];
    s_leaf[r] = is_leaf[o + r];
  }
  for (int r = warp; r < R; r += kWalkWarps) {
    const uint64_t* src = part + (o + r) * nchunk;
    uint64_t c[kScanMaxCand / 32];
#pragma unroll
    for (int j = 0; j < kScanMaxCand / 32; ++j) {
      const int i = lane + 32 * j;
      c[j] = i < nchunk ? src[i] : 0ull;
    }
    uint64_t best = 0ull;
#pragma unroll
    for (int j = 0; j < kScanMaxCand / 32; ++j) best = c[j] > best ? c[j] : best;
    best = warp_max_u64(best);
    if (lane == 0) {
      const int32_t t = (int32_t)cand_id(best);
      s_tgt[r] = t;
      if (tgt_out != nullptr) tgt_out[o + r] = t;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // (Short serial code: loops whose trip count differs between lanes cost
    // far more than guarded straight-line chunks, so rows are taken in fixed
    // chunks c = 1 + lane + 32 j, j < 2, covering rows 1..64.)
    // Per row: its parent, whether the tree is valid there (0 <= parent < c),
    // whether it matches the target at its parent (token[c] == tgt[parent]),
    // and whether it is a leaf (for the chain id).
    int pc[2];
    bool mc[2], ok = true;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = 1 + lane + 32 * j;
      pc[j] = -1;
      mc[j] = false;
      if (c < R) {
        const int p = s_par[c];
        const bool valid = p >= 0 && p < c;
        ok = ok && valid;
        pc[j] = p;
        mc[j] = valid && s_tok[c] == s_tgt[valid ? p : 0];
      }
    }
    bool bad = !__all_sync(kFull, ok);

    // the walk: a level is one ballot per 32 rows (the lowest matching child of u)
    int32_t* rows = accept_rows + (long)b * (S + 1);
    int u = 0, L = 0;
    if (!bad) {
      for (;;) {
        int found = R;
        const unsigned b0 = __ballot_sync(kFull, mc[0] && pc[0] == u);
        if (b0) {
          found = __ffs(b0);
        } else {
          const unsigned b1 = __ballot_sync(kFull, mc[1] && pc[1] == u);
          if (b1) found = 32 + __ffs(b1);
        }
        if (found == R) break;
        if (L == S) { bad = true; break; }
        ++L;
        if (lane == 0) {
          rows[L] = found;
          s_path[L] = found;
        }
        u = found;
      }
    }
    if (bad) {
      if (lane == 0) report_error(err, TSD_DEV_ERR_BAD_TREE, b);
      u = 0;
      L = 0;
    }
    if (lane <= S) {   // (S <= 16)
      if (lane == 0) rows[0] = s_path[0] = 0;
      else if (lane > L) rows[lane] = s_path[lane] = -1;
    }

    // chain id: the lowest leaf whose ancestor-or-self set holds u
    int chain = -1;
    if (L > 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = 1 + lane + 32 * j;
        const bool hit = c < R && s_leaf[c] && ((s_mask[c] >> (u - 1)) & 1ull);
        const unsigned bal = __ballot_sync(kFull, hit);
        if (chain < 0 && bal) chain = 32 * j + __ffs(bal);
      }
    }
    if (lane == 0) {
      accept_len[b] = L;
      bonus[b] = s_tgt[u];
      chain_id[b] = chain;
      s_L = L;
    }
  }  // warp 0
  if (kCommit) {
    __syncthreads();
    const int r_tid = threadIdx.x <= S ? s_path[threadIdx.x] : 0;
    commit_request<32 * kWalkWarps>(ca, s_commit, b, s_P, s_L, r_tid);
  }
}

}  // namespace
}  // namespace tsd

using namespace tsd;

extern "C" size_t tsd_accept_walk_workspace_size(int B, int D, int V) {
  if (B < 1 || D < 0 || V < 1) return 0;
  const long rows = (long)B * (D + 1);
  const ScanGeom g = scan_geometry(rows, V, 1, true);
  return (size_t)rows * g.nchunk * sizeof(uint64_t);
}

extern "C" tsd_status tsd_accept_walk(const float* logits, int B, int D, int S, int V,
                                      const int32_t* token, const int32_t* parent,
                                      const uint64_t* mask, const uint8_t* is_leaf,
                                      int32_t* tgt, int32_t* accept_len, int32_t* accept_rows,
                                      int32_t* bonus, int32_t* chain_id, void* ws,
                                      size_t ws_bytes, int32_t* err, tsd_stream_t stream) {
  if (B < 1 || D < 1 || D > kMaxR - 1 || S < 1 || S > 16 || V < 1 || V > (1 << 30))
    return TSD_ERR_INVALID_ARG;
  if ((long)B * (D + 1) > (1l << 24)) return TSD_ERR_INVALID_ARG;
  if (!ok_ptr(logits) || !ok_ptr(token) || !ok_ptr(parent) || !ok_ptr(mask) ||
      !ok_ptr(is_leaf) || !ok_opt_ptr(tgt) || !ok_ptr(accept_len) || !ok_ptr(accept_rows) ||
      !ok_ptr(bonus) || !ok_ptr(chain_id) || !ok_opt_ptr(err))
    return TSD_ERR_INVALID_ARG;
  const size_t need = tsd_accept_walk_workspace_size(B, D, V);
  if (ws_bytes < need || !ok_ptr(ws)) return TSD_ERR_INVALID_ARG;

  const cudaStream_t st = (cudaStream_t)stream;
  const int R = D + 1;
  const long rows = (long)B * R;
  const ScanGeom g = scan_geometry(rows, V, 1, true);
  uint64_t* part = (uint64_t*)ws;
  launch(vocab_scan_kernel<true>, dim3((unsigned)(rows * g.nchunk)), dim3(kScanThreads), 0, st,
      logits, V, 1, g.nchunk, g.chunk_len, part, g.one_wave, nullptr, 1);
  launch(accept_walk_kernel<false>, dim3(B), dim3(32 * kWalkWarps), 0, st, part, R, S, g.nchunk,
      token, parent, mask, is_leaf, tgt, accept_len, accept_rows, bonus, chain_id, err,
      CommitArgs{});
  return cuda_status();
}

namespace {

tsd_status walk_tree_args(int B, int D, int S, int V, const int32_t* token, const int32_t* parent,
                          const uint64_t* mask, const uint8_t* is_leaf, const int32_t* tgt,
                          const int32_t* accept_len, const int32_t* accept_rows,
                          const int32_t* bonus, const int32_t* chain_id, const int32_t* err) {
  if (B < 1 || D < 1 || D > kMaxR - 1 || S < 1 || S > 16 || V < 1 || V > (1 << 30))
    return TSD_ERR_INVALID_ARG;
  if ((long)B * (D + 1) > (1l << 24)) return TSD_ERR_INVALID_ARG;
  if (!ok_ptr(token) || !ok_ptr(parent) || !ok_ptr(mask) || !ok_ptr(is_leaf) ||
      !ok_opt_ptr(tgt) || !ok_ptr(accept_len) || !ok_ptr(accept_rows) || !ok_ptr(bonus) ||
      !ok_ptr(chain_id) || !ok_opt_ptr(err))
    return TSD_ERR_INVALID_ARG;
  return TSD_OK;
}

// The argmax part of the walk: per-chunk argmax candidates of every tree
// row's target logits into ws.
void launch_target_argmax(const float* logits, int B, int D, int V, void* ws, cudaStream_t st) {
  const long rows = (long)B * (D + 1);
  const ScanGeom g = scan_geometry(rows, V, 1, true);
  launch(vocab_scan_kernel<true>, dim3((unsigned)(rows * g.nchunk)), dim3(kScanThreads), 0, st,
      logits, V, 1, g.nchunk, g.chunk_len, (uint64_t*)ws, g.one_wave, nullptr, 1);
}

}  // namespace

extern "C" tsd_status tsd_target_argmax(const float* logits, int B, int D, int V, void* ws,
                                        size_t ws_bytes, tsd_stream_t stream) {
  if (B < 1 || D < 1 || D > kMaxR - 1 || V < 1 || V > (1 << 30)) return TSD_ERR_INVALID_ARG;
  if ((long)B * (D + 1) > (1l << 24)) return TSD_ERR_INVALID_ARG;
  if (!ok_ptr(logits)) return TSD_ERR_INVALID_ARG;
  if (ws_bytes < tsd_accept_walk_workspace_size(B, D, V) || !ok_ptr(ws)) return TSD_ERR_INVALID_ARG;
  launch_target_argmax(logits, B, D, V, ws, (cudaStream_t)stream);
  return cuda_status();
}

extern "C" tsd_status tsd_walk_commit(int B, int D, int S, int V, const int32_t* token,
                                      const int32_t* parent, const uint64_t* mask,
                                      const uint8_t* is_leaf, int32_t* tgt, int32_t* accept_len,
                                      int32_t* accept_rows, int32_t* bonus, int32_t* chain_id,
                                      const tsd_attn_desc* desc, const void* ktree,
                                      const void* vtree, void* kcache, void* vcache,
                                      const int32_t* page_table, int max_pages, int page_size,
                                      int num_pages, int32_t* prefix_len, const void* ws,
                                      size_t ws_bytes, int32_t* err, tsd_stream_t stream) {
  const tsd_status wst = walk_tree_args(B, D, S, V, token, parent, mask, is_leaf, tgt,
                                        accept_len, accept_rows, bonus, chain_id, err);
  if (wst != TSD_OK) return wst;
  if (desc == nullptr || desc->B != B || desc->R != D + 1 || page_size < 0)
    return TSD_ERR_INVALID_ARG;
  CommitArgs ca;
  const tsd_status cst = commit_args(desc, S, ktree, vtree, accept_rows, accept_len, kcache,
                                     vcache, page_table, max_pages, page_size, num_pages,
                                     prefix_len, err, &ca);
  if (cst != TSD_OK) return cst;
  if (ws_bytes < tsd_accept_walk_workspace_size(B, D, V) || !ok_ptr(ws)) return TSD_ERR_INVALID_ARG;
  const int R = D + 1;
  const ScanGeom g = scan_geometry((long)B * R, V, 1, true);
  launch(accept_walk_kernel<true>, dim3(B), dim3(32 * kWalkWarps), 0, (cudaStream_t)stream,
      (const uint64_t*)ws, R, S, g.nchunk, token, parent, mask, is_leaf, tgt, accept_len,
      accept_rows, bonus, chain_id, err, ca);
  return cuda_status();
}

extern "C" tsd_status tsd_accept_commit(const float* logits, int B, int D, int S, int V,
                                        const int32_t* token, const int32_t* parent,
                                        const uint64_t* mask, const uint8_t* is_leaf,
                                        int32_t* tgt, int32_t* accept_len, int32_t* accept_rows,
                                        int32_t* bonus, int32_t* chain_id,
                                        const tsd_attn_desc* desc, const void* ktree,
                                        const void* vtree, void* kcache, void* vcache,
                                        const int32_t* page_table, int max_pages, int page_size,
                                        int num_pages, int32_t* prefix_len, void* ws,
                                        size_t ws_bytes, int32_t* err, tsd_stream_t stream) {
  // both parts' checks before anything is enqueued
  const tsd_status wst = walk_tree_args(B, D, S, V, token, parent, mask, is_leaf, tgt,
                                        accept_len, accept_rows, bonus, chain_id, err);
  if (wst != TSD_OK) return wst;
  if (!ok_ptr(logits)) return TSD_ERR_INVALID_ARG;
  if (desc == nullptr || desc->B != B || desc->R != D + 1 || page_size < 0)
    return TSD_ERR_INVALID_ARG;
  CommitArgs ca;
  const tsd_status cst = commit_args(desc, S, ktree, vtree, accept_rows, accept_len, kcache,
                                     vcache, page_table, max_pages, page_size, num_pages,
                                     prefix_len, err, &ca);
  if (cst != TSD_OK) return cst;
  if (ws_bytes < tsd_accept_walk_workspace_size(B, D, V) || !ok_ptr(ws)) return TSD_ERR_INVALID_ARG;
  launch_target_argmax(logits, B, D, V, ws, (cudaStream_t)stream);
  return tsd_walk_commit(B, D, S, V, token, parent, mask, is_leaf, tgt, accept_len, accept_rows,
                         bonus, chain_id, desc, ktree, vtree, kcache, vcache, page_table,
                         max_pages, page_size, num_pages, prefix_len, ws, ws_bytes, err, stream);
}

// ---------------------------------------------------------------------------
// tsd_accept_walk_static: the same walk for callers that cannot allocate.
//
// Some callers are only ever handed their input and output buffers: a custom
// operator running inside another framework whose memory planner owns the
// device heap, or a serving loop that forbids any allocation after start-up.
// They cannot call cudaMalloc and have no workspace to pass.  This entry point
// keeps the per-chunk argmax candidates in a fixed array that is part of the
// library image instead (every GPU that loads the library holds it until the
// process exits), and allocates nothing itself.
// ---------------------------------------------------------------------------

namespace {

constexpr size_t kWalkStaticScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) uint64_t g_walk_static_scratch[kWalkStaticScratchBytes / 8];

// Device address of the array in the current context.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress; the first call on a device does it, and it is looked
// up again whenever the device's current context is a different one (after a
// cudaDeviceReset the array lives in the new context).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (CtxGetCurrentFn)p;
  });
  return fn;
}

uint64_t* walk_static_scratch() {
  constexpr int kMaxDevices = 64;
  static uint64_t* addr[kMaxDevices] = {};
  static CUcontext owner[kMaxDevices] = {};
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CUcontext ctx = nullptr;
  const CtxGetCurrentFn get = ctx_get_current();
  if (get != nullptr && get(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || ctx == nullptr || owner[dev] != ctx) {
    // (the lookup makes the device's primary context current if none is)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_walk_static_scratch) != cudaSuccess) return nullptr;
    addr[dev] = (uint64_t*)p;
    ctx = nullptr;
    if (get != nullptr) get(&ctx);
    owner[dev] = ctx;
  }
  return addr[dev];
}

}  // namespace

extern "C" tsd_status tsd_accept_walk_static(const float* logits, int B, int D, int S, int V,
                                             const int32_t* token, const int32_t* parent,
                                             const uint64_t* mask, const uint8_t* is_leaf,
                                             int32_t* tgt, int32_t* accept_len,
                                             int32_t* accept_rows, int32_t* bonus,
                                             int32_t* chain_id, int32_t* err,
                                             tsd_stream_t stream) {
  if (B < 1 || D < 1 || D > kMaxR - 1 || S < 1 || S > 16 || V < 1 || V > (1 << 30))
    return TSD_ERR_INVALID_ARG;
  if ((long)B * (D + 1) > (1l << 24)) return TSD_ERR_INVALID_ARG;
  if (!ok_ptr(logits) || !ok_ptr(token) || !ok_ptr(parent) || !ok_ptr(mask) ||
      !ok_ptr(is_leaf) || !ok_opt_ptr(tgt) || !ok_ptr(accept_len) || !ok_ptr(accept_rows) ||
      !ok_ptr(bonus) || !ok_ptr(chain_id) || !ok_opt_ptr(err))
    return TSD_ERR_INVALID_ARG;
  // the fixed scratch bounds the problem size
  if (tsd_accept_walk_workspace_size(B, D, V) > kWalkStaticScratchBytes) return TSD_ERR_UNSUPPORTED;
  uint64_t* part = walk_static_scratch();
  if (part == nullptr) return TSD_ERR_CUDA;

  // Every scratch slot the walk reads is written by the scan of the same call,
  // so nothing needs clearing.  Calls that overlap on the GPU share the array
  // and race.
  const cudaStream_t st = (cudaStream_t)stream;
  const int R = D + 1;
  const long rows = (long)B * R;
  const ScanGeom g = scan_geometry(rows, V, 1, true);
  launch(vocab_scan_kernel<true>, dim3((unsigned)(rows * g.nchunk)), dim3(kScanThreads), 0, st,
      logits, V, 1, g.nchunk, g.chunk_len, part, g.one_wave, nullptr, 1);
  launch(accept_walk_kernel<false>, dim3(B), dim3(32 * kWalkWarps), 0, st, part, R, S, g.nchunk,
      token, parent, mask, is_leaf, tgt, accept_len, accept_rows, bonus, chain_id, err,
      CommitArgs{});
  return cuda_status();
}
