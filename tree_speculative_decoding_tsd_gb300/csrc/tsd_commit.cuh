// The accepted-path commit of one request, shared by commit_path_kernel
// (tsd_commit_path) and the walk kernel's fused form (tsd_accept_commit).
//
// Source: "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4"
// (review), "Secret weapon" and "How it works" step 6: only the accepted
// path's KV leaves the scratch pad; the next round starts from the extended
// prefix.
#pragma once

#include "tsd_common.cuh"

namespace tsd {

constexpr int kCommitMaxRows = 17;   // 1 + S, S <= 16

struct CommitArgs {
  const char* ktree;
  const char* vtree;
  const int32_t* accept_rows;
  const int32_t* accept_len;
  char* kcache;
  char* vcache;
  int32_t* prefix_len;
  int32_t* err;
  int R, Hkv, cap, S;
  int kvec, vvec;   // 16-byte vectors per K row / V row (vvec = 0 if V aliases K)
  long krow, vrow;  // bytes per K row / V row
  // paged cache (page_size > 0): position pos of request b lives in page
  // page_table[b][pos / page_size] of the pools [num_pages][Hkv][page_size][row]
  const int32_t* page_table;
  int max_pages, page_size, num_pages;
};

// Shared-memory state of a commit: path entry i's scratch-pad row and cache
// row (head 0), and the smallest error code any thread found.
struct CommitSmem {
  int32_t src[kCommitMaxRows];
  long dst[kCommitMaxRows];
  int code;
};

constexpr int kCommitUnroll = 4;          // 16-byte loads in flight per thread
constexpr int kNoError = 0x7fffffff;      // above every TSD_DEV_ERR_* code

// Cache row of position pos of (request b, head 0), and the row stride between
// heads; -1 for a page outside the pool.
__device__ __forceinline__ long cache_row0(const CommitArgs& a, int b, int pos) {
  if (a.page_size == 0) return (long)b * a.Hkv * a.cap + pos;
  const int pg = a.page_table[(long)b * a.max_pages + pos / a.page_size];
  if (pg < 0 || pg >= a.num_pages) return -1;
  return (long)pg * a.Hkv * a.page_size + pos % a.page_size;
}

// Commit request b with prefix length P and path length L; r_tid is path
// entry tid (read for tid <= S).  Called by every thread of a CTA of
// kThreads threads, after s.code was set to kNoError and a barrier.  Thread
// i validates entry i (row index, page of P + i); the threads then split the
// (row, head, K|V, 16-byte vector) copies, kCommitUnroll loads in flight
// each; thread 0 writes the new prefix length or reports the error.
template <int kThreads>
__device__ __forceinline__ void commit_request(const CommitArgs& a, CommitSmem& s, int b, int P,
                                               int L, int r_tid) {
  const int tid = threadIdx.x;
  int code = 0;
  if (L < 0 || L > a.S) code = TSD_DEV_ERR_BAD_TREE;
  else if (P < 0 || (long)P + 1 + L > a.cap) code = TSD_DEV_ERR_CAPACITY;
  else if (tid <= L) {
    const long d0 = cache_row0(a, b, P + tid);
    if (r_tid < 0 || r_tid >= a.R) code = TSD_DEV_ERR_BAD_TREE;
    else if (d0 < 0) code = TSD_DEV_ERR_BAD_PAGE;
    s.src[tid] = r_tid;
    s.dst[tid] = d0;
  }
  // one code for the request: the smallest one any thread found
  if (code != 0) atomicMin(&s.code, code);
  __syncthreads();
  code = s.code == kNoError ? 0 : s.code;

  if (code == 0) {
    const int per_head = a.kvec + a.vvec;
    const int per_row = a.Hkv * per_head;
    const int work = (L + 1) * per_row;
    const long hstride = a.page_size ? a.page_size : a.cap;
    // (the same trip count for every thread: a loop whose count differs
    // between the lanes of a warp costs far more than a guarded body)
    for (int w0 = 0; w0 < work; w0 += kThreads * kCommitUnroll) {
      // all loads of the batch first, then the stores (the stores could alias
      // the sources as far as the compiler knows)
      int4 v[kCommitUnroll];
      int4* dst[kCommitUnroll];
#pragma unroll
      for (int u = 0; u < kCommitUnroll; ++u) {
        const int w = w0 + tid + u * kThreads;
        dst[u] = nullptr;
        if (w < work) {
          const int i = w / per_row;
          const int rem = w - i * per_row;
          const int h = rem / per_head;
          const int e = rem - h * per_head;
          const long src_row = ((long)b * a.R + s.src[i]) * a.Hkv + h;
          const long dst_row = s.dst[i] + h * hstride;
          const int4* src;
          if (e < a.kvec) {
            src = reinterpret_cast<const int4*>(a.ktree + src_row * a.krow) + e;
            dst[u] = reinterpret_cast<int4*>(a.kcache + dst_row * a.krow) + e;
          } else {
            src = reinterpret_cast<const int4*>(a.vtree + src_row * a.vrow) + (e - a.kvec);
            dst[u] = reinterpret_cast<int4*>(a.vcache + dst_row * a.vrow) + (e - a.kvec);
          }
          v[u] = __ldg(src);
        }
      }
#pragma unroll
      for (int u = 0; u < kCommitUnroll; ++u)
        if (dst[u] != nullptr) *dst[u] = v[u];
    }
  }
  if (tid == 0) {
    if (code == 0) a.prefix_len[b] = P + 1 + L;
    else report_error(a.err, code, b);
  }
}

}  // namespace tsd

namespace tsd {

// Host: the argument checks of tsd_commit_path(_paged) (page_size 0 for the
// contiguous cache), and the kernel arguments they give; defined in
// tsd_commit.cu.
tsd_status commit_args(const tsd_attn_desc* d, int S, const void* ktree, const void* vtree,
                       const int32_t* accept_rows, const int32_t* accept_len, void* kcache,
                       void* vcache, const int32_t* page_table, int max_pages, int page_size,
                       int num_pages, int32_t* prefix_len, int32_t* err, CommitArgs* out);

}  // namespace tsd
