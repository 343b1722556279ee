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
#include "tsd_commit.cuh"
#include "tsd_host.h"

namespace tsd {
namespace {

constexpr int kCommitThreads = 512;

__global__ void __launch_bounds__(kCommitThreads) commit_path_kernel(CommitArgs a) {
  __shared__ CommitSmem s;
  __shared__ int s_P, s_L;
  grid_dependency_sync();
  const int b = blockIdx.x, tid = threadIdx.x;
  // path entry tid, read together with the lengths (one memory round trip)
  const int r_tid = tid <= a.S ? a.accept_rows[(long)b * (a.S + 1) + tid] : 0;
  // one read of the prefix and path lengths, shared by the whole CTA
  if (tid == 0) {
    s_P = a.prefix_len[b];
    s_L = a.accept_len[b];
    s.code = kNoError;
  }
  __syncthreads();
  commit_request<kCommitThreads>(a, s, b, s_P, s_L, r_tid);
}

}  // namespace
}  // namespace tsd

using namespace tsd;

namespace tsd {

tsd_status commit_args(const tsd_attn_desc* d, int S, const void* ktree, const void* vtree,
                       const int32_t* accept_rows, const int32_t* accept_len, void* kcache,
                       void* vcache, const int32_t* page_table, int max_pages, int page_size,
                       int num_pages, int32_t* prefix_len, int32_t* err, CommitArgs* out) {
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

  CommitArgs& a = *out;
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
  return TSD_OK;
}

}  // namespace tsd

static tsd_status commit_impl(const tsd_attn_desc* d, int S, const void* ktree, const void* vtree,
                              const int32_t* accept_rows, const int32_t* accept_len, void* kcache,
                              void* vcache, const int32_t* page_table, int max_pages,
                              int page_size, int num_pages, int32_t* prefix_len, int32_t* err,
                              tsd_stream_t stream) {
  CommitArgs a;
  const tsd_status st = commit_args(d, S, ktree, vtree, accept_rows, accept_len, kcache, vcache,
                                    page_table, max_pages, page_size, num_pages, prefix_len, err,
                                    &a);
  if (st != TSD_OK) return st;
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
