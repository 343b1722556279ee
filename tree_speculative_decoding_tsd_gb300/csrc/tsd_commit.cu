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
// K6 commit_path_kernel: one CTA per request.  Its threads split the (row,
// head, K|V, 16-byte vector) copies; every thread reads the old prefix length
// before the block barrier and thread 0 writes the new one after it.  (At most
// (S+1) x Hkv rows of a few KB move per request: one CTA is enough, and a
// cluster's launch and barrier cost more than they save.)
#include "tsd_common.cuh"
#include "tsd_host.h"

namespace tsd {
namespace {

constexpr int kCommitThreads = 256;

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

// Cache row of position pos of (request b, head h); -1 for a page outside the pool.
__device__ __forceinline__ long cache_row(const CommitArgs& a, int b, int h, int pos) {
  if (a.page_size == 0) return ((long)b * a.Hkv + h) * a.cap + pos;
  const int pg = a.page_table[(long)b * a.max_pages + pos / a.page_size];
  if (pg < 0 || pg >= a.num_pages) return -1;
  return ((long)pg * a.Hkv + h) * a.page_size + pos % a.page_size;
}

__global__ void __launch_bounds__(kCommitThreads) commit_path_kernel(CommitArgs a) {
  const int b = blockIdx.x;
  const int P = a.prefix_len[b];
  const int L = a.accept_len[b];
  const int32_t* rows = a.accept_rows + (long)b * (a.S + 1);

  int code = 0;
  if (L < 0 || L > a.S) code = TSD_DEV_ERR_BAD_TREE;
  else if (P < 0 || (long)P + 1 + L > a.cap) code = TSD_DEV_ERR_CAPACITY;
  else
    for (int i = 0; i <= L; ++i) {
      if (rows[i] < 0 || rows[i] >= a.R) code = TSD_DEV_ERR_BAD_TREE;
      else if (cache_row(a, b, 0, P + i) < 0) code = TSD_DEV_ERR_BAD_PAGE;
    }

  if (code == 0) {
    const int per_head = a.kvec + a.vvec;
    const long work = (long)(L + 1) * a.Hkv * per_head;
    for (long w = threadIdx.x; w < work; w += kCommitThreads) {
      const int i = (int)(w / ((long)a.Hkv * per_head));
      const int rem = (int)(w - (long)i * a.Hkv * per_head);
      const int h = rem / per_head;
      const int e = rem - h * per_head;
      const long src_row = ((long)b * a.R + rows[i]) * a.Hkv + h;
      const long dst_row = cache_row(a, b, h, P + i);
      const int4* src;
      int4* dst;
      if (e < a.kvec) {
        src = reinterpret_cast<const int4*>(a.ktree + src_row * a.krow) + e;
        dst = reinterpret_cast<int4*>(a.kcache + dst_row * a.krow) + e;
      } else {
        src = reinterpret_cast<const int4*>(a.vtree + src_row * a.vrow) + (e - a.kvec);
        dst = reinterpret_cast<int4*>(a.vcache + dst_row * a.vrow) + (e - a.kvec);
      }
      *dst = __ldg(src);
    }
  }
  // every thread has read prefix_len[b] before anyone passes this barrier
  __syncthreads();
  if (threadIdx.x == 0) {
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
  commit_path_kernel<<<d->B, kCommitThreads, 0, (cudaStream_t)stream>>>(a);
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
