// tsd_commit_path: copy the accepted path's scratch-pad KV into the
// persistent cache and advance the prefix length.
//
// Source: "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4"
// (review), "Secret weapon" and "How it works" step 6: verification results
// stay in a scratch pad; after the accepted path is chosen only that path's
// KV is written to the persistent cache, the other branches are dropped, and
// the next round starts from the extended prefix.  (Token-level KV refresh is
// all a sliding-window / dense cache needs.)
//
// K6 commit_path_kernel: one CTA per request.  Thread 0 reads the prefix and
// path lengths once for the CTA (and writes the new prefix length at the end);
// thread i checks path entry i and resolves its cache row; then the threads
// split the (row, head, K|V, 16-byte vector) copies, kCommitUnroll loads in
// flight each.  (At most (S+1) x Hkv rows of a few KB move per
// request: one CTA is enough, and a cluster's launch and barrier cost more
// than they save.)
#include "tsd_common.cuh"
#include "tsd_host.h"

namespace tsd {
namespace {

constexpr int kCommitThreads = 512;
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

// Cache row of position pos of (request b, head 0), and the row stride between
// heads; -1 for a page outside the pool.
__device__ __forceinline__ long cache_row0(const CommitArgs& a, int b, int pos) {
  if (a.page_size == 0) return (long)b * a.Hkv * a.cap + pos;
  const int pg = a.page_table[(long)b * a.max_pages + pos / a.page_size];
  if (pg < 0 || pg >= a.num_pages) return -1;
  return (long)pg * a.Hkv * a.page_size + pos % a.page_size;
}

constexpr int kCommitUnroll = 4;   // 16-byte loads in flight per thread
constexpr int kNoError = 0x7fffffff;   // above every TSD_DEV_ERR_* code

__global__ void __launch_bounds__(kCommitThreads) commit_path_kernel(CommitArgs a) {
  __shared__ int32_t s_src[kCommitMaxRows];   // scratch-pad row of path entry i
  __shared__ long s_dst[kCommitMaxRows];      // cache row of position P + i, head 0
  __shared__ int s_P, s_L, s_code;
  grid_dependency_sync();
  const int b = blockIdx.x, tid = threadIdx.x;
  // path entry tid, read together with the lengths (one memory round trip)
  const int r_tid = tid <= a.S ? a.accept_rows[(long)b * (a.S + 1) + tid] : 0;
  // one read of the prefix and path lengths, shared by the whole CTA
  if (tid == 0) {
    s_P = a.prefix_len[b];
    s_L = a.accept_len[b];
    s_code = kNoError;
  }
  __syncthreads();
  const int P = s_P, L = s_L;

  // validation: thread i checks path entry i (row index, page of P + i)
  int code = 0;
  if (L < 0 || L > a.S) code = TSD_DEV_ERR_BAD_TREE;
  else if (P < 0 || (long)P + 1 + L > a.cap) code = TSD_DEV_ERR_CAPACITY;
  else if (tid <= L) {
    const int r = r_tid;
    const long d0 = cache_row0(a, b, P + tid);
    if (r < 0 || r >= a.R) code = TSD_DEV_ERR_BAD_TREE;
    else if (d0 < 0) code = TSD_DEV_ERR_BAD_PAGE;
    s_src[tid] = r;
    s_dst[tid] = d0;
  }
  // one code for the request: the smallest one any thread found
  if (code != 0) atomicMin(&s_code, code);
  __syncthreads();
  code = s_code == kNoError ? 0 : s_code;

  if (code == 0) {
    const int per_head = a.kvec + a.vvec;
    const int per_row = a.Hkv * per_head;
    const int work = (L + 1) * per_row;
    const long hstride = a.page_size ? a.page_size : a.cap;
    for (int w0 = tid; w0 < work; w0 += kCommitThreads * kCommitUnroll) {
      // all loads of the batch first, then the stores (the stores could alias
      // the sources as far as the compiler knows)
      int4 v[kCommitUnroll];
      int4* dst[kCommitUnroll];
#pragma unroll
      for (int u = 0; u < kCommitUnroll; ++u) {
        const int w = w0 + u * kCommitThreads;
        dst[u] = nullptr;
        if (w < work) {
          const int i = w / per_row;
          const int rem = w - i * per_row;
          const int h = rem / per_head;
          const int e = rem - h * per_head;
          const long src_row = ((long)b * a.R + s_src[i]) * a.Hkv + h;
          const long dst_row = s_dst[i] + h * hstride;
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

}  // namespace
}  // namespace tsd

using namespace tsd;

static tsd_status commit_impl(const tsd_attn_desc* d, int S, const void* ktree, const void* vtree,
                              const int32_t* accept_rows, const int32_t* accept_len, void* kcache,
                              void* vcache, const int32_t* page_table, int max_pages,
                              int page_size, int num_pages, int32_t* prefix_len, int32_t* err,
                              tsd_stream_t stream) {
  if (d == nullptr) return TSD_ERR_INVALID_ARG;
  if (d->B < 1 || d->B > 65535 || d->R < 1 || d->R > 65 || d->Hkv < 1 || d->dk < 1 ||
      d->cap < 1 || S < 1 || S > 16)
    return TSD_ERR_INVALID_ARG;
  if (d->dtype != TSD_F32 && d->dtype != TSD_BF16) return TSD_ERR_INVALID_ARG;
  const int es = d->dtype == TSD_F32 ? 4 : 2;
  const bool alias = d->v_aliases_k != 0;
  if (!alias && d->dv < 1) return TSD_ERR_INVALID_ARG;
  if (((long)d->dk * es) % 16 != 0 || (!alias && ((long)d->dv * es) % 16 != 0))
    return TSD_ERR_INVALID_ARG;
  if (!ok_ptr(ktree) || !ok_ptr(accept_rows) || !ok_ptr(accept_len) || !ok_ptr(kcache) ||
      !ok_ptr(prefix_len) || (((uintptr_t)err) & 3u) != 0)
    return TSD_ERR_INVALID_ARG;
  if (!alias && (!ok_ptr(vtree) || !ok_ptr(vcache))) return TSD_ERR_INVALID_ARG;
  const bool paged = page_size > 0;
  if (paged && (max_pages < 1 || num_pages < 1 || (long)max_pages * page_size != d->cap ||
                !ok_ptr(page_table)))
    return TSD_ERR_INVALID_ARG;

  CommitArgs a;
  a.ktree = (const char*)ktree;
  a.vtree = (const char*)vtree;
  a.accept_rows = accept_rows;
  a.accept_len = accept_len;
  a.kcache = (char*)kcache;
  a.vcache = (char*)vcache;
  a.prefix_len = prefix_len;
  a.err = err;
  a.R = d->R;
  a.Hkv = d->Hkv;
  a.cap = d->cap;
  a.S = S;
  a.krow = (long)d->dk * es;
  a.vrow = alias ? 0 : (long)d->dv * es;
  a.kvec = (int)(a.krow / 16);
  a.vvec = (int)(a.vrow / 16);
  a.page_table = paged ? page_table : nullptr;
  a.max_pages = paged ? max_pages : 0;
  a.page_size = paged ? page_size : 0;
  a.num_pages = paged ? num_pages : 0;
  launch(commit_path_kernel, dim3(d->B), dim3(kCommitThreads), 0, (cudaStream_t)stream, a);
  return cuda_status();
}

extern "C" tsd_status tsd_commit_path(const tsd_attn_desc* d, int S, const void* ktree,
                                      const void* vtree, const int32_t* accept_rows,
                                      const int32_t* accept_len, void* kcache, void* vcache,
                                      int32_t* prefix_len, int32_t* err, tsd_stream_t stream) {
  return commit_impl(d, S, ktree, vtree, accept_rows, accept_len, kcache, vcache, nullptr, 0, 0,
                     0, prefix_len, err, stream);
}

extern "C" tsd_status tsd_commit_path_paged(const tsd_attn_desc* d, int S, const void* ktree,
                                            const void* vtree, const int32_t* accept_rows,
                                            const int32_t* accept_len, void* kpool, void* vpool,
                                            const int32_t* page_table, int max_pages,
                                            int page_size, int num_pages, int32_t* prefix_len,
                                            int32_t* err, tsd_stream_t stream) {
  if (page_size < 1) return TSD_ERR_INVALID_ARG;
  return commit_impl(d, S, ktree, vtree, accept_rows, accept_len, kpool, vpool, page_table,
                     max_pages, page_size, num_pages, prefix_len, err, stream);
}
