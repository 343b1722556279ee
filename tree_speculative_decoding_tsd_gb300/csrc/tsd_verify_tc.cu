// tcgen05 (5th-generation tensor core) path of tsd_tree_verify_attn for bf16
// GQA heads with dk == dv == 128 and at least 16 packed query rows.
//
// Layout choice.  The packed query rows of one KV head (R tree rows x g query
// heads: 68, 132 or 260 for the workloads here) rarely fill 128-row MMA tiles,
// so the products are computed transposed, with the packed rows on the MMA N
// dimension (a multiple of 16, padded by at most 15 rows):
//   S^T[key][n]  = K_tile . Q^T     M = 128 keys,  N = packed rows, K = dk
//   O^T[d][n]   += V_tile^T . P^T   M = 128 (dv),  N = packed rows, K = 128 keys
// Both accumulators live in tensor memory (fp32); S^T is double-buffered.
//
// Roles (576 threads): warps 0-15 softmax/epilogue (warpgroup w/4 owns a
// quarter of the columns, warp w%4 owns TMEM lanes 32(w%4)..+31, i.e. 32 keys
// of a tile or 32 dims of O^T); warp 16 allocates TMEM and issues the MMAs
// (one thread); warp 17 issues the TMA loads (one thread per ring).  K and V
// tiles of 128 keys (32 KB each) arrive by cp.async.bulk.tensor with 128-byte
// swizzle into two separate two-stage rings: a K stage is refilled as soon as its S^T product is done, a V
// stage as soon as its O^T product is done, so each load is issued about two
// tiles ahead of its use.  mbarriers order TMA -> MMA -> softmax -> MMA.
//
// Softmax with keys on lanes: a thread holds one key's scores for all of its
// columns, so a row's max and sum are cross-lane reductions.  The running max
// m[n] is therefore lazy.  Each tile is first processed optimistically with
// the current m (p = 2^min(x, 64), x = s*scale*log2e - m), adding p to the
// per-lane partial sums and writing P^T.  If any x exceeded 8 (or on the first
// tile) the warpgroup recomputes the tile exactly: column maxima by a warp
// reduce-scatter plus a shared-memory pass, alpha = 2^(m_old - m_new), O^T
// columns rescaled, and every partial sum replaced by (l - p_opt)*alpha + p_new
// (the subtraction's rounding error is scaled by alpha, below 2^-24 of the new
// sum).  Probabilities therefore stay <= 2^8, safe in bf16/fp32.  Row sums are
// reduced across lanes once, at the end.
//
// Every mbarrier wait is bounded (about a second); a timeout sets
// TSD_DEV_ERR_TIMEOUT in the error word, all roles stop, in-flight copies and
// MMAs are waited for (again bounded) and the tensor memory is released.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "tsd_common.cuh"
#include "tsd_host.h"
#include "tsd_tcgen05.cuh"
#include "tsd_verify.cuh"

namespace tsd {
namespace {

constexpr int kKeys = 128;          // keys per tile (MMA M of S^T)
constexpr int kD = 128;             // head dim
constexpr int kSoftWarps = 16;                  // 4 warpgroups, one quarter of the columns each
constexpr int kThreadsTC = (kSoftWarps + 2) * 32;
constexpr int kMmaWarp = 16, kTmaWarp = 17;
constexpr uint32_t kBox = kKeys * 128;          // one [128 rows][64 bf16] swizzled box: 16 KB
constexpr uint32_t kTileBytes = 2 * kBox;       // one K or V tile: 32 KB
constexpr uint32_t kOffK = 0;                   // K ring: 2 x 32 KB
constexpr uint32_t kOffV = 2 * kTileBytes;      // V ring: 2 x 32 KB
constexpr uint32_t kOffQ = 4 * kTileBytes;      // 128 KB
constexpr int kPagedTiles = 64;  // paged cache: tile rows resolved at set-up
constexpr float kOverflow = 8.0f;               // log2 headroom of the lazy max
constexpr int kPrefetch = 3;                    // prefix tiles prefetched into L2 ahead

template <int N>
struct TcLayout {
  static constexpr uint32_t q_bytes = 2u * N * 128u;
  static constexpr uint32_t off_pt = kOffQ + ((q_bytes + 1023u) / 1024u) * 1024u;
  static constexpr uint32_t pt_blocks = (N + 63) / 64;
  static constexpr uint32_t off_misc = off_pt + pt_blocks * kBox;
  static constexpr int NH = N / 4;                // columns per warpgroup
  // misc area
  static constexpr uint32_t off_m = off_misc;                       // float[N]   running max
  static constexpr uint32_t off_alpha = off_m + 4 * N;              // float[N]   rescale factors
  static constexpr uint32_t off_negm = off_alpha + 4 * N;             // float[N]   -m (0 if m = -inf)
  static constexpr uint32_t off_red = off_negm + 4 * N;             // float[16][NH] per-warp partials
  static constexpr uint32_t off_lsum = off_red + 4 * kSoftWarps * NH;  // float[N] row sums
  static constexpr uint32_t off_rmask = (off_lsum + 4 * N + 7) / 8 * 8;  // u64[N] tree masks
  static constexpr uint32_t off_ooff = off_rmask + 8 * N;           // i64[N] output offsets
  static constexpr uint32_t off_bar = off_ooff + 8 * N;             // mbarriers
  static constexpr int nbar = 13;
  static constexpr uint32_t off_flags = off_bar + 8 * nbar;          // tmem addr, abort flag
  static constexpr uint32_t off_tiles = off_flags + 16;  // int[kPagedTiles] tile rows (paged)
  static constexpr uint32_t total = off_tiles + 4 * kPagedTiles;
  static_assert(total + 1024 <= 232448, "shared memory budget");
};

// barrier indices
enum { BAR_K_FULL = 0, BAR_K_EMPTY = 2, BAR_V_FULL = 4, BAR_V_EMPTY = 6, BAR_S_FULL = 8,
       BAR_P_FULL = 10, BAR_PV_DONE = 11, BAR_FINAL = 12 };

struct TcMaps {
  CUtensorMap k, v, kt, vt;
};

template <int N, bool kPaged>
__global__ void __launch_bounds__(kThreadsTC, 1)
verify_tc_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ VerifyArgs a,
                 int rows_per_cta) {
  using L = TcLayout<N>;
  if (threadIdx.x == kTmaWarp * 32) {
    tma_desc_prefetch(&maps.k);
    tma_desc_prefetch(&maps.v);
    tma_desc_prefetch(&maps.kt);
    tma_desc_prefetch(&maps.vt);
  }
  // While the previous kernel finishes: L2 prefetch of this CTA's first two
  // prefix tiles (K and V, one warp each; contiguous cache only, the page
  // table may still be being written) and of its Q rows.  Hints only.
  {
    const int w = threadIdx.x >> 5, ln = threadIdx.x & 31;
    const int hk0 = blockIdx.y / a.nrg, b0 = blockIdx.z;
    const int kp0 = blockIdx.x * a.split_len;
    if (!kPaged && w < 4 && ln == 0) {
      const int t = w >> 1;
      const CUtensorMap* m = (w & 1) ? &maps.v : &maps.k;
      if (kp0 + t * kKeys < a.cap) {
        const int y = (b0 * a.Hkv + hk0) * a.cap + kp0 + t * kKeys;
        tma_prefetch_2d(m, 0, y);
        tma_prefetch_2d(m, 64, y);
      }
    } else if (w == 4) {
      // packed rows [p0, p1) of this row group: for each tree row, the heads
      // of this KV head are one contiguous run of q
      const int p0 = (blockIdx.y % a.nrg) * rows_per_cta;
      const int p1 = min(p0 + rows_per_cta, a.M);
      for (int tr = p0 / a.g + ln; tr <= (p1 - 1) / a.g; tr += 32) {
        const int h0 = max(p0, tr * a.g) - tr * a.g, h1 = min(p1, (tr + 1) * a.g) - tr * a.g;
        const __nv_bfloat16* qr =
            (const __nv_bfloat16*)a.q + (((long)b0 * a.R + tr) * a.Hq + hk0 * a.g + h0) * kD;
        prefetch_l2(qr, (long)(h1 - h0) * kD * 2);
      }
    }
  }
  grid_dependency_sync();
  constexpr int NH = L::NH;
  // 128-byte-swizzled TMA boxes and MMA operands need 1024-byte-aligned atoms:
  // align the dynamic shared-memory base by hand (1 KB of slack is requested)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = su32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  float* m_run = (float*)(smem + L::off_m);
  float* alpha = (float*)(smem + L::off_alpha);
  float* red = (float*)(smem + L::off_red);
  float* lsum = (float*)(smem + L::off_lsum);
  uint64_t* rmask = (uint64_t*)(smem + L::off_rmask);
  volatile uint32_t* flags = (volatile uint32_t*)(smem + L::off_flags);  // [0] tmem, [1] abort
  const uint32_t bar0 = sbase + L::off_bar;
  auto bar = [&](int i) { return bar0 + 8u * i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sp = blockIdx.x;
  const int hk = blockIdx.y / a.nrg, rg = blockIdx.y % a.nrg;
  const int b = blockIdx.z;
  const int P = min(max(a.plen[b], 0), a.cap);
  const int nsb = P > 0 ? (P + a.split_len - 1) / a.split_len : 1;
  if (sp >= nsb) return;  // uniform for the whole CTA, before any barrier or allocation
  const int k0 = sp * a.split_len, k1 = min(P, k0 + a.split_len);
  const int n_pre = k1 > k0 ? (k1 - k0 + kKeys - 1) / kKeys : 0;
  const int n_tree = (sp == nsb - 1) ? 1 : 0;   // R <= 65 < 128: one tile
  const int ntiles = n_pre + n_tree;
  const int row_base = rg * rows_per_cta;
  const int rows_here = min(rows_per_cta, a.M - row_base);

  // ---------------------------------------------------------------- set-up
  // The TMA thread initialises the barriers and starts the first loads at
  // once, so they overlap the Q staging and the TMEM allocation.
  // first row of prefix tile t in the cache, or in the page pool
  // paged cache: the set-up resolves the first kPagedTiles tile rows into
  // shared memory (tiles_ready of them, 0 until the set-up barrier)
  int* tile_rows = (int*)(smem + L::off_tiles);
  int tiles_ready = 0;
  auto ycoord = [&](int t) {
    if constexpr (kPaged) {
      if (t < tiles_ready) return tile_rows[t];
      return paged_tile_row(a, b, hk, k0 + t * kKeys);
    } else {
      return (b * a.Hkv + hk) * a.cap + k0 + t * kKeys;
    }
  };
  auto tma_k = [&](int t, int stage) {
    const uint32_t dst = sbase + kOffK + stage * kTileBytes;
    const uint32_t fb = bar(BAR_K_FULL + stage);
    mbar_expect_tx(fb, kTileBytes);
    if (t < n_pre) {
      tma_2d(dst, &maps.k, 0, ycoord(t), fb);
      tma_2d(dst + kBox, &maps.k, 64, ycoord(t), fb);
    } else {
      tma_3d(dst, &maps.kt, 0, hk, b * a.R, fb);
      tma_3d(dst + kBox, &maps.kt, 64, hk, b * a.R, fb);
    }
  };
  auto tma_v = [&](int t, int stage) {
    const uint32_t dst = sbase + kOffV + stage * kTileBytes;
    const uint32_t fb = bar(BAR_V_FULL + stage);
    mbar_expect_tx(fb, kTileBytes);
    if (t < n_pre) {
      tma_2d(dst, &maps.v, 0, ycoord(t), fb);
      tma_2d(dst + kBox, &maps.v, 64, ycoord(t), fb);
    } else {
      tma_3d(dst, &maps.vt, 0, hk, b * a.R, fb);
      tma_3d(dst + kBox, &maps.vt, 64, hk, b * a.R, fb);
    }
  };
  // L2 prefetch of a prefix tile a few tiles ahead of its smem load
  auto prefetch = [&](int t) {
    if (t < n_pre) {
      tma_prefetch_2d(&maps.k, 0, ycoord(t));
      tma_prefetch_2d(&maps.k, 64, ycoord(t));
      tma_prefetch_2d(&maps.v, 0, ycoord(t));
      tma_prefetch_2d(&maps.v, 64, ycoord(t));
    }
  };
  if (warp == kTmaWarp && lane == 0) {
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(bar(BAR_K_FULL + s2), 1);
      mbar_init(bar(BAR_K_EMPTY + s2), 1);
      mbar_init(bar(BAR_V_FULL + s2), 1);
      mbar_init(bar(BAR_V_EMPTY + s2), 1);
      mbar_init(bar(BAR_S_FULL + s2), 1);
    }
    mbar_init(bar(BAR_P_FULL), kSoftWarps);
    mbar_init(bar(BAR_PV_DONE), 1);
    mbar_init(bar(BAR_FINAL), 1);
    flags[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kTmaWarp) {
    // the first K and V tiles from two threads at once (a thread issues about
    // one box per ~570 cycles, and the set-up barrier waits for both); the
    // second K tile and the L2 prefetches follow after the barrier
    __syncwarp();
    if (lane == 0) tma_k(0, 0);
    else if (lane == 1) tma_v(0, 0);
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
        sbase + L::off_flags));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  float* negm = (float*)(smem + L::off_negm);
  long long* ooff = (long long*)(smem + L::off_ooff);
  if (warp < kSoftWarps) {
    // Q tile (K-major, 128-byte swizzle: two boxes of [N][64]) by cp.async
    for (int idx = tid; idx < N * 16; idx += kSoftWarps * 32) {
      const int n = idx >> 4, c = idx & 15;
      const bool valid = n < rows_here;
      const __nv_bfloat16* src = (const __nv_bfloat16*)a.q;
      if (valid) {
        const int p = row_base + n;
        const int tr = p / a.g, qh = hk * a.g + p % a.g;
        src += (((long)b * a.R + tr) * a.Hq + qh) * kD + c * 8;
      }
      cp_async16(sbase + kOffQ + (c >> 3) * (N * 128u) + n * 128u + (((c & 7) ^ (n & 7)) << 4),
                 src, valid);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    for (int n = tid; n < N; n += kSoftWarps * 32) {
      uint64_t mk = 0ull;
      if (n < rows_here) {
        const int tr = (row_base + n) / a.g;
        mk = tr > 0 ? a.mask[(long)b * a.R + tr] : 0ull;
      }
      rmask[n] = mk;
      m_run[n] = -INFINITY;
      negm[n] = 0.f;
    }
    if constexpr (kPaged)
      for (int t = tid; t < min(n_pre, kPagedTiles); t += kSoftWarps * 32)
        tile_rows[t] = paged_tile_row(a, b, hk, k0 + t * kKeys);
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = flags[0];
  if constexpr (kPaged) tiles_ready = min(n_pre, kPagedTiles);
  const uint32_t tm_s[2] = {tmem, tmem + (uint32_t)N};
  const uint32_t tm_o = tmem + 2u * N;

  // ------------------------------------------------------------------ TMA
  // One thread per ring (a thread completes about one TMA box per ~570
  // cycles, so the K and V streams are issued side by side): K_t after
  // S^T_{t-2} freed its stage, V_t after O^T_{t-2} freed its stage.
  if (warp == kTmaWarp) {
    if (lane == 0) {
      int nk = 1;
      if (ntiles > 1) {
        tma_k(1, 1);
        nk = 2;
      }
      for (int t = 2; t < 2 + kPrefetch; ++t) prefetch(t);
      for (int t = 2; t < ntiles && !flags[1]; ++t) {
        if (!mbar_wait(bar(BAR_K_EMPTY + (t & 1)), ((t - 2) >> 1) & 1)) { flags[1] = 1; break; }
        tma_k(t, t & 1);
        prefetch(t + kPrefetch);
        ++nk;
      }
      // no copy may still be in flight when the CTA leaves
      for (int st = 0; st < 2; ++st) {
        const int ck = (nk - st + 1) / 2;  // loads into stage st
        if (ck > 0) mbar_wait(bar(BAR_K_FULL + st), (ck - 1) & 1);
      }
    } else if (lane == 1) {
      int nv = 1;
      for (int tv = 1; tv < ntiles && !flags[1]; ++tv) {
        if (tv >= 2 && !mbar_wait(bar(BAR_V_EMPTY + (tv & 1)), ((tv - 2) >> 1) & 1)) {
          flags[1] = 1;
          break;
        }
        tma_v(tv, tv & 1);
        ++nv;
      }
      for (int st = 0; st < 2; ++st) {
        const int cv = (nv - st + 1) / 2;
        if (cv > 0) mbar_wait(bar(BAR_V_FULL + st), (cv - 1) & 1);
      }
    }
  }

  // ------------------------------------------------------------------ MMA
  else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t idesc_qk = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
                                ((uint32_t)(kKeys >> 4) << 24);
      const uint32_t idesc_pv = idesc_qk | (1u << 15) | (1u << 16);
      // descriptor bases (built once): K stage 0, V stage 0, Q^T, P^T
      const uint64_t kd0 = smem_desc(sbase + kOffK, 16, 1024);
      const uint64_t vd0 = smem_desc(sbase + kOffV, kBox, 1024);
      const uint64_t qd0 = smem_desc(sbase + kOffQ, 16, 1024);
      const uint64_t ptd0 = smem_desc(sbase + L::off_pt, kBox, 1024);
      auto issue_qk = [&](int t) -> bool {
        const int st = t & 1;
        if (!mbar_wait(bar(BAR_K_FULL + st), (t >> 1) & 1)) return false;
        fence_after();
        const uint64_t kd = kd0 + (uint64_t)(st * (kTileBytes >> 4));
        mma_f16(tm_s[st], kd, qd0, idesc_qk, 0u);
#pragma unroll
        for (int kk = 1; kk < kD / 16; ++kk)
          mma_f16_acc(tm_s[st], kd + (((kk >> 2) * kBox + (kk & 3) * 32) >> 4),
                      qd0 + (((kk >> 2) * (N * 128u) + (kk & 3) * 32) >> 4), idesc_qk);
        mma_commit(bar(BAR_S_FULL + st));
        mma_commit(bar(BAR_K_EMPTY + st));
        return true;
      };
      bool ok = issue_qk(0);
      for (int t = 0; ok && t < ntiles; ++t) {
        if (t + 1 < ntiles && !issue_qk(t + 1)) { ok = false; break; }
        if (!mbar_wait(bar(BAR_P_FULL), t & 1) || flags[1]) { ok = false; break; }
        if (!mbar_wait(bar(BAR_V_FULL + (t & 1)), (t >> 1) & 1)) { ok = false; break; }
        fence_after();
        const uint64_t vd = vd0 + (uint64_t)((t & 1) * (kTileBytes >> 4));
        if (t == 0) mma_f16(tm_o, vd, ptd0, idesc_pv, 0u);
        else mma_f16_acc(tm_o, vd, ptd0, idesc_pv);
#pragma unroll
        for (int kk = 1; kk < kKeys / 16; ++kk)
          mma_f16_acc(tm_o, vd + 128 * kk, ptd0 + 128 * kk, idesc_pv);
        mma_commit(bar(BAR_PV_DONE));
        mma_commit(bar(BAR_V_EMPTY + (t & 1)));
      }
      if (!ok) flags[1] = 1;
      // every MMA issued so far has completed once this commit lands: wait for
      // it before the TMEM is released
      mma_commit(bar(BAR_FINAL));
      mbar_wait(bar(BAR_FINAL), 0);
    }
  }

  // -------------------------------------------------------------- softmax
  else {
    const int wg = warp >> 2, q = warp & 3;
    const int c0 = wg * NH;                  // first column of this warpgroup
    const int key = q * 32 + lane;           // TMEM lane = key of the tile / dim of O^T
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float c = a.qscale;
    constexpr int NCH = NH / 4;              // chunks of 4 columns (one tcgen05.ld.x4 each)
    constexpr int GRP = 6;                   // chunks loaded per tcgen05.wait::ld
    float l[NH];                             // this key lane's partial row sums
    uint32_t pp[NH / 2];                     // this tile's probabilities, packed bf16x2
#pragma unroll
    for (int n = 0; n < NH; ++n) l[n] = 0.f;
    bool failed = false;

    for (int t = 0; t < ntiles; ++t) {
      const int st = t & 1;
      // tcgen05.ld is warp-collective: the whole warp agrees on the wait
      const bool ok = __all_sync(kFull, mbar_wait(bar(BAR_S_FULL + st), (t >> 1) & 1));
      fence_after();
      const bool is_tree = t >= n_pre;
      const int nvalid = is_tree ? a.R : min(kKeys, k1 - (k0 + t * kKeys));
      const uint32_t srow = tm_s[st] + lane_off + (uint32_t)c0;
      // masked scores of chunk j (columns c0 + 4j .. +3) of this key
      auto masked = [&](float (&v)[4], int j) {
        if (key >= nvalid) {
#pragma unroll
          for (int i = 0; i < 4; ++i) v[i] = -INFINITY;
        } else if (is_tree && key > 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (!((rmask[c0 + 4 * j + i] >> (key - 1)) & 1ull)) v[i] = -INFINITY;
        }
      };
      // x = s*c - m (log2 domain), p = 2^min(x, 64); returns max x
      auto probs = [&](float (&v)[4], int j) {
        const float4 nm = *(const float4*)(negm + c0 + 4 * j);
        const float x0 = fmaf(v[0], c, nm.x), x1 = fmaf(v[1], c, nm.y);
        const float x2 = fmaf(v[2], c, nm.z), x3 = fmaf(v[3], c, nm.w);
        v[0] = ex2(fminf(x0, 64.f));
        v[1] = ex2(fminf(x1, 64.f));
        v[2] = ex2(fminf(x2, 64.f));
        v[3] = ex2(fminf(x3, 64.f));
        return fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
      };
      auto load1 = [&](float (&v)[4], int j) {
        tmem_ld4(srow + 4u * j, v);
        tmem_wait_ld();
        masked(v, j);
      };

      // optimistic pass with the current running max (not on the first tile,
      // which always takes the exact path below: nothing to take back out)
      float xmax = -INFINITY;
      if (ok && t > 0) {
#pragma unroll
        for (int j0 = 0; j0 < NCH; j0 += GRP) {
          float v[GRP][4];
#pragma unroll
          for (int u = 0; u < GRP; ++u)
            if (j0 + u < NCH) tmem_ld4(srow + 4u * (j0 + u), v[u]);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < GRP; ++u) {
            const int j = j0 + u;
            if (j >= NCH) break;
            masked(v[u], j);
            xmax = fmaxf(xmax, probs(v[u], j));
#pragma unroll
            for (int i = 0; i < 4; ++i) l[4 * j + i] += v[u][i];
            pp[2 * j] = pack_bf16x2(v[u][0], v[u][1]);
            pp[2 * j + 1] = pack_bf16x2(v[u][2], v[u][3]);
          }
        }
      }
      // one barrier in the common case; the rare path takes a second one
      const bool local_stop = !ok || failed || flags[1] != 0;
      bool slow = false;
      if (wg_bar_or(wg, local_stop || t == 0 || xmax > kOverflow)) {
        if (wg_bar_or(wg, local_stop)) { failed = true; break; }
        slow = true;
        // exact column maxima of this tile, then the new running max
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float v[4];
          load1(v, j);
          const float r = warp_reduce_scatter<4, true>(v, lane);
          if (lane < 4) red[warp * NH + 4 * j + lane] = r;
        }
        wg_bar(wg);
        for (int n = tid & 127; n < NH; n += 128) {
          float mx = -INFINITY;
#pragma unroll
          for (int w = 0; w < 4; ++w) mx = fmaxf(mx, red[(wg * 4 + w) * NH + n]);
          const float m_old = m_run[c0 + n];
          const float m_new = fmaxf(m_old, mx * c);
          alpha[c0 + n] = (m_old == -INFINITY) ? 0.f : ex2(m_old - m_new);
          m_run[c0 + n] = m_new;
        }
        wg_bar(wg);
        // take the optimistic probabilities back out (recomputed bit-identically)
        if (t > 0) {
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            float v[4];
            load1(v, j);
            probs(v, j);
#pragma unroll
            for (int i = 0; i < 4; ++i) l[4 * j + i] -= v[i];
          }
        }
        wg_bar(wg);
        for (int n = tid & 127; n < NH; n += 128) {
          const float mu = m_run[c0 + n];
          negm[c0 + n] = mu == -INFINITY ? 0.f : -mu;
        }
        wg_bar(wg);
        // exact probabilities with the new max; old sums rescaled by alpha
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float v[4];
          load1(v, j);
          probs(v, j);
#pragma unroll
          for (int i = 0; i < 4; ++i) l[4 * j + i] = fmaf(l[4 * j + i], alpha[c0 + 4 * j + i], v[i]);
          pp[2 * j] = pack_bf16x2(v[0], v[1]);
          pp[2 * j + 1] = pack_bf16x2(v[2], v[3]);
        }
      }
      // P^T is single-buffered: the previous tile's O^T product must be done
      if (t > 0 && !__all_sync(kFull, mbar_wait(bar(BAR_PV_DONE), (t - 1) & 1))) failed = true;
      fence_after();
      if (slow && t > 0 && !failed) {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float v[4];
          tmem_ld4(tm_o + lane_off + (uint32_t)(c0 + 4 * j), v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 4; ++i) v[i] *= alpha[c0 + 4 * j + i];
          tmem_st4(tm_o + lane_off + (uint32_t)(c0 + 4 * j), v);
        }
        tmem_wait_st();
      }
      // P^T row of this key (MN-major, 128-byte swizzle, blocks of 64 columns)
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int n0 = c0 + 4 * j;
        const uint32_t off = L::off_pt + (n0 >> 6) * kBox + key * 128u +
                             ((((n0 & 63) >> 3) ^ (key & 7)) << 4) + ((n0 & 4) << 1);
        *(uint2*)(smem + off) = make_uint2(pp[2 * j], pp[2 * j + 1]);
      }
      // V rows of keys past the range may hold anything: zero them (the
      // warpgroup of the first columns does it)
      if (wg == 0 && key >= nvalid) {
        if (!mbar_wait(bar(BAR_V_FULL + st), (t >> 1) & 1)) failed = true;
        uint8_t* vrow = smem + kOffV + st * kTileBytes + key * 128u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          *(uint4*)(vrow + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
          *(uint4*)(vrow + kBox + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P_FULL));
    }

    // ---------------------------------------------------------- epilogue
    bool ok = !failed && (ntiles == 0 ||
                          __all_sync(kFull, mbar_wait(bar(BAR_PV_DONE), (ntiles - 1) & 1)));
    fence_after();
    const bool stop = wg_bar_or(wg, !ok || flags[1] != 0);
    if (!stop) {
      // row sums across the 128 key lanes
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = l[4 * j + i];
        const float r = warp_reduce_scatter<4, false>(v, lane);
        if (lane < 4) red[warp * NH + 4 * j + lane] = r;
      }
      wg_bar(wg);
      // per column: 1/l into alpha[], destination offset, log-sum-exp
      for (int n = tid & 127; n < NH; n += 128) {
        const int col = c0 + n;
        float ls = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) ls += red[(wg * 4 + w) * NH + n];
        alpha[col] = 1.f / ls;
        if (col < rows_here) {
          const int p = row_base + col;
          const int tr = p / a.g, qh = hk * a.g + p % a.g;
          const float lse2 = m_run[col] + log2f(ls);
          if (a.nsplit == 1) {
            const long orow = ((long)b * a.R + tr) * a.Hq + qh;
            ooff[col] = orow * kD;
            a.lse[orow] = lse2 * 0.69314718055994531f;
          } else {
            const long prow = (((long)b * a.Hq + qh) * a.R + tr) * a.nsplit + sp;
            ooff[col] = prow * kD;
            a.ws_lse[prow] = lse2;
          }
        }
      }
      wg_bar(wg);
      const int d = key;  // O^T lane = output dim
      // GRP chunks of O^T per TMEM wait, then their stores
#pragma unroll
      for (int j0 = 0; j0 < NCH; j0 += GRP) {
        float v[GRP][4];
#pragma unroll
        for (int u = 0; u < GRP; ++u)
          if (j0 + u < NCH) tmem_ld4(tm_o + lane_off + (uint32_t)(c0 + 4 * (j0 + u)), v[u]);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < GRP; ++u) {
          if (j0 + u >= NCH) break;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = c0 + 4 * (j0 + u) + i;
            if (col >= rows_here) break;
            const float res = v[u][i] * alpha[col];
            if (a.nsplit == 1) ((__nv_bfloat16*)a.out)[ooff[col] + d] = __float2bfloat16_rn(res);
            else a.ws_o[ooff[col] + d] = res;
          }
        }
      }
    }
    if (failed && lane == 0) flags[1] = 1;
  }

  // --------------------------------------------------------------- teardown
  fence_before();
  __syncthreads();
  if (flags[1] && tid == 0) report_error(a.err, TSD_DEV_ERR_TIMEOUT, b);
  fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem));
  }
}

// --------------------------------------------------------------- host side

// rows x 128 bf16 (row pitch 256 B), boxes of [128 rows][64 cols], 128B swizzle
bool encode_2d(CUtensorMap* m, const void* base, long rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kKeys};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B*R][Hkv][128] bf16, boxes of [128 rows][1 head][64 cols]
bool encode_3d(CUtensorMap* m, const void* base, int Hkv, long rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)Hkv, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)Hkv * kD * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kKeys};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
void launch_tc(const TcMaps& maps, const VerifyArgs& a, const VerifyPlan& p, cudaStream_t st) {
  const uint32_t smem = TcLayout<N>::total + 1024;
  const auto kern = a.page_size > 0 ? verify_tc_kernel<N, true> : verify_tc_kernel<N, false>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const dim3 grid(p.nsplit, a.Hkv * p.nrg, a.B);
  launch(kern, dim3(grid), dim3(kThreadsTC), smem, st, maps, a, p.rb);
}

}  // namespace

bool tc_path_available() { return encode_fn() != nullptr; }

bool launch_tc_path(const tsd_attn_desc& d, const VerifyArgs& a, const VerifyPlan& p,
                    cudaStream_t st) {
  if (d.dk != kD || d.dv != kD || d.v_aliases_k || d.dtype != TSD_BF16) return false;
  if (encode_fn() == nullptr) return false;
  TcMaps maps;
  const long cache_rows = a.page_size > 0 ? (long)a.num_pages * d.Hkv * a.page_size
                                          : (long)d.B * d.Hkv * d.cap;
  if (!encode_2d(&maps.k, a.kc, cache_rows) || !encode_2d(&maps.v, a.vc, cache_rows) ||
      !encode_3d(&maps.kt, a.kt, d.Hkv, (long)d.B * d.R) ||
      !encode_3d(&maps.vt, a.vt, d.Hkv, (long)d.B * d.R))
    return false;
  switch (p.rb) {
    case 16: launch_tc<16>(maps, a, p, st); break;
    case 32: launch_tc<32>(maps, a, p, st); break;
    case 48: launch_tc<48>(maps, a, p, st); break;
    case 64: launch_tc<64>(maps, a, p, st); break;
    case 80: launch_tc<80>(maps, a, p, st); break;
    case 96: launch_tc<96>(maps, a, p, st); break;
    case 112: launch_tc<112>(maps, a, p, st); break;
    case 128: launch_tc<128>(maps, a, p, st); break;
    case 144: launch_tc<144>(maps, a, p, st); break;
    default: return false;
  }
  if (p.nsplit > 1) {
    const long rows = (long)a.B * a.R * a.Hq;
    launch_plain(verify_combine_kernel<__nv_bfloat16, 128>, dim3((unsigned)ceil_div(rows, 4)),
                 dim3(128), 0, st, a);
  }
  return true;
}

}  // namespace tsd
