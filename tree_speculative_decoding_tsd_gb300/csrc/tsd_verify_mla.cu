// tcgen05 path of tsd_tree_verify_attn for latent heads (bf16): one KV head
// of 576 dims whose rows serve as keys and whose first 512 dims serve as
// values (V = K[:, :512]), shared by all g = Hq query heads.
//
// Source: "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4"
// (review): the tree verify must run on the target's own attention; for the
// latent-attention layout every query head of every tree row reads the same
// compressed KV row, so the packed rows of a request (R tree rows x 128 heads)
// form a dense contraction against each prefix tile.
//
// Products, transposed as in the GQA tcgen05 path (packed query rows on the
// MMA N dimension, N = 64 per CTA):
//   S^T[key][n]  = K_tile . Q^T     M = 128 keys, N = 64, K = 576 in 9 pieces of 64
//   O^T[d][n]   += V_tile^T . P^T   4 M-tiles of 128 dims, N = 64, K = 128 keys
// Tensor memory: S^T double-buffered (2 x 64 columns) and O^T (4 x 64), 384
// of 512 columns.  Shared memory: Q^T resident (9 boxes of [64 rows][64 dims],
// 72 KB), a 4-slot ring of 32 KB boxes and P^T (16 KB).  A box is two 64-dim
// pieces of 128 keys ([2][128 keys][64 dims], 128-byte swizzle), loaded by
// one 3-D TMA copy; a tile takes five K boxes (pieces 0-1, ..., 6-7, 8 and an
// out-of-range piece that the copy fills with zeros) and four V boxes (pieces
// 2u, 2u+1: exactly the 128 dims of O^T M-tile u).  A 128-key tile of latent
// rows is 144 KB, too large to stay resident beside Q, so the value dims are
// loaded a second time; every row-group CTA of a request reads the same
// tiles, so those loads are served by L2.
//
// Issue rates set the design: the tensor core needs 48 cycles for an
// M128 x N64 x K16 MMA, a thread issuing TMA copies manages about one per
// ~300-600 cycles, and every wait/commit around an MMA batch costs a few
// hundred cycles.  So boxes are large (8 MMAs per wait and commit), the S^T
// and O^T MMAs are issued by two threads, and two warps issue the copies.
//
// Roles (640 threads): warps 0-15 softmax/epilogue (warpgroup w/4 owns 16 of
// the 64 columns, warp w%4 owns TMEM lanes 32(w%4)..+31: 32 keys of a tile or
// 32 dims of an O^T M-tile); warp 16 allocates TMEM and issues the S^T MMAs;
// warp 17 issues the O^T MMAs (one thread) and zeroes the value rows of keys
// past the valid range of a partial tile (whole warp) so that 0 x garbage
// never reaches O; warps 18-19 issue the TMA copies (one thread each, boxes
// alternating).  Softmax: the lazy-maximum scheme of the GQA tcgen05 path (an
// optimistic pass with the running maximum, an exact recomputation when a
// score exceeds it by more than 2^8 or on the first tile).  Every mbarrier
// wait is bounded; a timeout sets TSD_DEV_ERR_TIMEOUT, all roles stop,
// in-flight copies and MMAs are waited for and the tensor memory is released.
#include "tsd_common.cuh"
#include "tsd_host.h"
#include "tsd_tcgen05.cuh"
#include "tsd_verify.cuh"

namespace tsd {
namespace {

constexpr int kKeys = 128;                      // keys per tile (MMA M of S^T)
constexpr int kDK = 576, kDV = 512;
constexpr int kKP = kDK / 64;                   // 64-dim pieces per key row
constexpr int kKB = (kKP + 1) / 2;              // K boxes per tile
constexpr int kVU = kDV / 128;                  // V boxes (O^T M-tiles) per tile
constexpr int kSoftWarps = 16;
constexpr int kSWarp = 16, kOWarp = 17, kTmaWarp0 = 18, kTmaWarps = 2;
constexpr int kThreads = (kSoftWarps + 2 + kTmaWarps) * 32;
constexpr uint32_t kPiece = kKeys * 128;        // [128 rows][64 bf16] swizzled: 16 KB
constexpr uint32_t kBox = 2 * kPiece;           // one ring slot
constexpr int kSlots = 4;
constexpr uint32_t kOffRing = 0;
constexpr uint32_t kOffQ = kOffRing + kSlots * kBox;
constexpr int kPagedTiles = 64;  // paged cache: tile rows resolved at set-up
constexpr float kOverflow = 8.0f;               // log2 headroom of the lazy max
constexpr int kPrefetch = 2;                    // prefix tiles prefetched into L2 ahead

template <int N>
struct MlaLayout {
  static constexpr uint32_t q_box = (uint32_t)N * 128u;   // one [N][64] box of Q^T
  static constexpr uint32_t off_pt = kOffQ + kKP * q_box;
  static constexpr uint32_t pt_blocks = (N + 63) / 64;
  static constexpr uint32_t off_misc = off_pt + pt_blocks * kPiece;
  static constexpr int NH = N / 4;
  static constexpr uint32_t off_m = off_misc;
  static constexpr uint32_t off_alpha = off_m + 4 * N;
  static constexpr uint32_t off_negm = off_alpha + 4 * N;
  static constexpr uint32_t off_red = off_negm + 4 * N;
  static constexpr uint32_t off_rmask = (off_red + 4 * kSoftWarps * NH + 7) / 8 * 8;
  static constexpr uint32_t off_ooff = off_rmask + 8 * N;
  static constexpr uint32_t off_bar = off_ooff + 8 * N;
  static constexpr int nbar = 16;
  static constexpr uint32_t off_flags = off_bar + 8 * nbar;
  static constexpr uint32_t off_tiles = off_flags + 16;  // int[kPagedTiles] tile rows (paged)
  static constexpr uint32_t total = off_tiles + 4 * kPagedTiles;  // flags: [0] tmem [1] abort [2] K seen [3] V seen
  static_assert(q_box % 1024 == 0, "Q boxes must keep 1 KB swizzle alignment");
  static_assert(off_pt % 1024 == 0, "P^T must keep 1 KB swizzle alignment");
  static_assert(total + 1024 <= 232448, "shared memory budget");
  static_assert(6 * N <= 512, "tensor memory budget");
};

enum { BAR_FULL = 0, BAR_EMPTY = kSlots, BAR_S_FULL = 2 * kSlots, BAR_S_FREE = 2 * kSlots + 2,
       BAR_P_FULL = 2 * kSlots + 4, BAR_PV_DONE = 2 * kSlots + 5, BAR_FIN_S = 2 * kSlots + 6,
       BAR_FIN_O = 2 * kSlots + 7 };

struct MlaMaps {
  CUtensorMap k, kt;
};

template <int N, bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
verify_mla_kernel(const __grid_constant__ MlaMaps maps, const __grid_constant__ VerifyArgs a,
                  int rows_per_cta) {
  using L = MlaLayout<N>;
  if (threadIdx.x == kTmaWarp0 * 32) {
    tma_desc_prefetch(&maps.k);
    tma_desc_prefetch(&maps.kt);
  }
  grid_dependency_sync();
  constexpr int NH = L::NH;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = su32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  float* m_run = (float*)(smem + L::off_m);
  float* alpha = (float*)(smem + L::off_alpha);
  float* negm = (float*)(smem + L::off_negm);
  float* red = (float*)(smem + L::off_red);
  uint64_t* rmask = (uint64_t*)(smem + L::off_rmask);
  long long* ooff = (long long*)(smem + L::off_ooff);
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
  // keys of tile t that exist (the rest are masked and their values zeroed)
  auto nvalid_of = [&](int t) { return t >= n_pre ? a.R : min(kKeys, k1 - (k0 + t * kKeys)); };

  // The ring carries one sequence of boxes, in the order the MMAs use them:
  //   K_0 (5 boxes), K_1, V_0 (4 boxes), K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
  // Box i goes to slot i % 4 as that slot's (i / 4)-th load, so the phase of
  // every FULL / EMPTY wait follows from the position alone.
  auto step_start = [&](int s) { return kKB * s + kVU * (s > 0 ? s - 1 : 0); };
  auto pos_k = [&](int t, int j) { return step_start(t) + j; };
  auto pos_v = [&](int t, int u) { return step_start(t + 1) + (t + 1 < ntiles ? kKB : 0) + u; };
  const int nbox = (kKB + kVU) * ntiles;
  // The K boxes are consumed by one thread and the V boxes by another, each in
  // its own order.  A parity wait is only sound while the barrier is at most
  // one phase behind its target, so before waiting for position p a consumer
  // makes sure the box at p - 4 (same slot, previous load) has been seen to
  // land: its own kind by program order, the other kind through the other
  // consumer's count of boxes seen (flags[2] for K, flags[3] for V).
  // Returns -1 for "none needed", else 2 * index + (1 if a V box).
  auto prev_box = [&](int p) {
    const int q = p - kSlots;
    if (q < 0) return -1;
    if (q < kKB) return 2 * q;                      // K_0 box q
    const int s2 = 1 + (q - kKB) / (kKB + kVU), r = (q - kKB) % (kKB + kVU);
    if (s2 < ntiles && r < kKB) return 2 * (s2 * kKB + r);
    return 2 * ((s2 - 1) * kVU + r - (s2 < ntiles ? kKB : 0)) + 1;
  };
  // wait until the other consumer has seen box `idx` of its kind land (bounded)
  auto seen_by_other = [&](int counter, int idx) {
    const long long t0 = clock64();
    while ((int)flags[counter] <= idx) {
      if (flags[1] || clock64() - t0 > kWaitCycles) return false;
    }
    return true;
  };

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
  // box of pieces z, z+1 of tile t
  auto load_box = [&](uint32_t dst, int t, int z, uint32_t fb) {
    if (t < n_pre) tma_3d(dst, &maps.k, 0, ycoord(t), z, fb);
    else tma_4d(dst, &maps.kt, 0, hk, b * a.R, z, fb);
  };
  auto prefetch = [&](int t) {
    if (t < n_pre) {
#pragma unroll 1
      for (int j = 0; j < kKB; ++j) tma_prefetch_3d(&maps.k, 0, ycoord(t), 2 * j);
    }
  };

  // ---------------------------------------------------------------- set-up
  if (tid == kTmaWarp0 * 32) {
    for (int sl = 0; sl < kSlots; ++sl) {
      mbar_init(bar(BAR_FULL + sl), 1);
      mbar_init(bar(BAR_EMPTY + sl), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BAR_S_FULL + i), 1);
      mbar_init(bar(BAR_S_FREE + i), kSoftWarps);
    }
    mbar_init(bar(BAR_P_FULL), kSoftWarps);
    mbar_init(bar(BAR_PV_DONE), 1);
    mbar_init(bar(BAR_FIN_S), 1);
    mbar_init(bar(BAR_FIN_O), 1);
    flags[1] = 0;
    flags[2] = 0;
    flags[3] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    for (int t = 0; t < 1 + kPrefetch; ++t) prefetch(t);
  }
  if (warp == kSWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
        sbase + L::off_flags));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  if (warp < kSoftWarps) {
    // Q^T (K-major, 128-byte swizzle: 9 boxes of [N][64]) by cp.async
    for (int idx = tid; idx < N * (kDK / 8); idx += kSoftWarps * 32) {
      const int n = idx / (kDK / 8), c = idx % (kDK / 8);
      const bool valid = n < rows_here;
      const __nv_bfloat16* src = (const __nv_bfloat16*)a.q;
      if (valid) {
        const int p = row_base + n;
        const int tr = p / a.g, qh = hk * a.g + p % a.g;
        src += (((long)b * a.R + tr) * a.Hq + qh) * kDK + c * 8;
      }
      cp_async16(sbase + kOffQ + (c >> 3) * L::q_box + n * 128u + (((c & 7) ^ (n & 7)) << 4),
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
  const uint32_t tm_o = tmem + 2u * N;            // M-tile u at tm_o + u * N
  const uint32_t idesc_qk = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
                            ((uint32_t)(kKeys >> 4) << 24);
  const uint32_t idesc_pv = idesc_qk | (1u << 15) | (1u << 16);

  // ------------------------------------------------------------------ TMA
  if (warp >= kTmaWarp0) {
    const int w = warp - kTmaWarp0;
    if (lane == 0) {
      bool ok = true;
      int p = 0;
      auto put = [&](int t, int z) {
        if (ok && p % kTmaWarps == w) {
          const int sl = p % kSlots;
          if (p >= kSlots && (flags[1] || !mbar_wait(bar(BAR_EMPTY + sl), ((p / kSlots) - 1) & 1))) {
            ok = false;
          } else {
            mbar_expect_tx(bar(BAR_FULL + sl), kBox);
            load_box(sbase + kOffRing + sl * kBox, t, z, bar(BAR_FULL + sl));
          }
        }
        ++p;
      };
      for (int s = 0; ok && s <= ntiles; ++s) {
        if (s < ntiles) {
          if (w == 0 && s > 0) prefetch(s + kPrefetch);
          for (int j = 0; j < kKB; ++j) put(s, 2 * j);
        }
        if (s > 0)
          for (int u = 0; u < kVU; ++u) put(s - 1, 2 * u);
      }
      if (!ok) flags[1] = 1;
      // no copy may still be in flight when the CTA leaves
      if (w == 0)
        for (int sl = 0; sl < kSlots && sl < nbox; ++sl) {
          const int last = sl + ((nbox - 1 - sl) / kSlots) * kSlots;
          mbar_wait(bar(BAR_FULL + sl), (last / kSlots) & 1);
        }
    }
  }

  // -------------------------------------------------------------- S^T MMAs
  else if (warp == kSWarp) {
    if (lane == 0) {
      const uint64_t kd0 = smem_desc(sbase + kOffRing, 16, 1024);
      const uint64_t qd0 = smem_desc(sbase + kOffQ, 16, 1024);
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int st = t & 1;
        // S^T buffer st was last read by the softmax of tile t - 2
        if (t >= 2 && !mbar_wait(bar(BAR_S_FREE + st), ((t >> 1) - 1) & 1)) { ok = false; break; }
        for (int j = 0; j < kKB; ++j) {
          const int p = pos_k(t, j), sl = p % kSlots, pv = prev_box(p);
          if ((pv >= 0 && (pv & 1) && !seen_by_other(3, pv >> 1)) || flags[1] ||
              !mbar_wait(bar(BAR_FULL + sl), (p / kSlots) & 1)) {
            ok = false;
            break;
          }
          __threadfence_block();
          flags[2] = (uint32_t)(t * kKB + j + 1);
          fence_after();
          const uint64_t ad = kd0 + (uint64_t)(sl * (kBox >> 4));
          const uint64_t bd = qd0 + (uint64_t)(2 * j * (L::q_box >> 4));
          if (j == 0) mma_f16(tm_s[st], ad, bd, idesc_qk, 0u);
          else mma_f16_acc(tm_s[st], ad, bd, idesc_qk);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk) mma_f16_acc(tm_s[st], ad + 2 * kk, bd + 2 * kk, idesc_qk);
          if (2 * j + 1 < kKP) {
            const uint64_t ad1 = ad + (kPiece >> 4), bd1 = bd + (L::q_box >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_f16_acc(tm_s[st], ad1 + 2 * kk, bd1 + 2 * kk, idesc_qk);
          }
          mma_commit(bar(BAR_EMPTY + sl));
        }
        if (ok) mma_commit(bar(BAR_S_FULL + st));
      }
      if (!ok) flags[1] = 1;
      // every MMA issued by this thread has completed once this commit lands
      mma_commit(bar(BAR_FIN_S));
      mbar_wait(bar(BAR_FIN_S), 0);
    }
  }

  // -------------------------------------------------------------- O^T MMAs
  else if (warp == kOWarp) {
    const uint64_t vd0 = smem_desc(sbase + kOffRing, kPiece, 1024);
    const uint64_t ptd0 = smem_desc(sbase + L::off_pt, kPiece, 1024);
    bool ok = true;
    for (int t = 0; ok && t < ntiles; ++t) {
      if (!__all_sync(kFull, mbar_wait(bar(BAR_P_FULL), t & 1)) ||
          __any_sync(kFull, flags[1] != 0)) {
        ok = false;
        break;
      }
      const int nvalid = nvalid_of(t);
      for (int u = 0; u < kVU; ++u) {
        const int p = pos_v(t, u), sl = p % kSlots, pv = prev_box(p);
        const bool prev_ok = pv < 0 || (pv & 1) || seen_by_other(2, pv >> 1);
        if (!__all_sync(kFull, prev_ok && mbar_wait(bar(BAR_FULL + sl), (p / kSlots) & 1))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          __threadfence_block();
          flags[3] = (uint32_t)(t * kVU + u + 1);
        }
        if (nvalid < kKeys) {
          // value rows of keys past the range may hold anything: zero them
          for (int key = nvalid + lane; key < kKeys; key += 32) {
            uint8_t* r0 = smem + kOffRing + sl * kBox + key * 128u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              *(uint4*)(r0 + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
              *(uint4*)(r0 + kPiece + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
          __syncwarp();
        }
        fence_after();
        if (lane == 0) {
          const uint64_t ad = vd0 + (uint64_t)(sl * (kBox >> 4));
          if (t == 0) mma_f16(tm_o + u * N, ad, ptd0, idesc_pv, 0u);
          else mma_f16_acc(tm_o + u * N, ad, ptd0, idesc_pv);
#pragma unroll
          for (int kk = 1; kk < kKeys / 16; ++kk)
            mma_f16_acc(tm_o + u * N, ad + 128 * kk, ptd0 + 128 * kk, idesc_pv);
          mma_commit(bar(BAR_EMPTY + sl));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit(bar(BAR_PV_DONE));
      __syncwarp();
    }
    if (!ok && lane == 0) flags[1] = 1;
    if (lane == 0) {
      mma_commit(bar(BAR_FIN_O));
      mbar_wait(bar(BAR_FIN_O), 0);
    }
    __syncwarp();
  }

  // -------------------------------------------------------------- softmax
  else {
    const int wg = warp >> 2, q = warp & 3;
    const int c0 = wg * NH;
    const int key = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float c = a.qscale;
    constexpr int NCH = NH / 4;
    float l[NH];
    uint32_t pp[NH / 2];
#pragma unroll
    for (int n = 0; n < NH; ++n) l[n] = 0.f;
    bool failed = false;

    for (int t = 0; t < ntiles; ++t) {
      const int st = t & 1;
      const bool ok = __all_sync(kFull, mbar_wait(bar(BAR_S_FULL + st), (t >> 1) & 1));
      fence_after();
      const bool is_tree = t >= n_pre;
      const int nvalid = nvalid_of(t);
      const uint32_t srow = tm_s[st] + lane_off + (uint32_t)c0;
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

      float xmax = -INFINITY;
      if (ok) {
        float v[NCH][4];
#pragma unroll
        for (int j = 0; j < NCH; ++j) tmem_ld4(srow + 4u * j, v[j]);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          masked(v[j], j);
          xmax = fmaxf(xmax, probs(v[j], j));
#pragma unroll
          for (int i = 0; i < 4; ++i) l[4 * j + i] += v[j][i];
          pp[2 * j] = pack_bf16x2(v[j][0], v[j][1]);
          pp[2 * j + 1] = pack_bf16x2(v[j][2], v[j][3]);
        }
      }
      const bool local_stop = !ok || failed || flags[1] != 0;
      bool slow = false;
      if (wg_bar_or(wg, local_stop || t == 0 || xmax > kOverflow)) {
        if (wg_bar_or(wg, local_stop)) { failed = true; break; }
        slow = true;
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
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float v[4];
          load1(v, j);
          probs(v, j);
#pragma unroll
          for (int i = 0; i < 4; ++i) l[4 * j + i] -= v[i];
        }
        wg_bar(wg);
        for (int n = tid & 127; n < NH; n += 128) {
          const float mu = m_run[c0 + n];
          negm[c0 + n] = mu == -INFINITY ? 0.f : -mu;
        }
        wg_bar(wg);
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
      // every read of S^T is done: its buffer may take tile t + 2
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_S_FREE + st));
      // P^T is single-buffered: the previous tile's O^T products must be done
      if (t > 0 && !__all_sync(kFull, mbar_wait(bar(BAR_PV_DONE), (t - 1) & 1))) failed = true;
      fence_after();
      if (slow && t > 0 && !failed) {
#pragma unroll 1
        for (int u = 0; u < kVU; ++u) {
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            float v[4];
            const uint32_t ta = tm_o + u * N + lane_off + (uint32_t)(c0 + 4 * j);
            tmem_ld4(ta, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] *= alpha[c0 + 4 * j + i];
            tmem_st4(ta, v);
          }
        }
        tmem_wait_st();
      }
      // P^T row of this key (MN-major, 128-byte swizzle, blocks of 64 columns)
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int n0 = c0 + 4 * j;
        const uint32_t off = L::off_pt + (n0 >> 6) * kPiece + key * 128u +
                             ((((n0 & 63) >> 3) ^ (key & 7)) << 4) + ((n0 & 4) << 1);
        *(uint2*)(smem + off) = make_uint2(pp[2 * j], pp[2 * j + 1]);
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
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = l[4 * j + i];
        const float r = warp_reduce_scatter<4, false>(v, lane);
        if (lane < 4) red[warp * NH + 4 * j + lane] = r;
      }
      wg_bar(wg);
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
          if (nsb == 1) {
            const long orow = ((long)b * a.R + tr) * a.Hq + qh;
            ooff[col] = orow * kDV;
            a.lse[orow] = lse2 * 0.69314718055994531f;
          } else {
            const long prow = (((long)b * a.Hq + qh) * a.R + tr) * a.nsplit + sp;
            ooff[col] = prow * kDV;
            a.ws_lse[prow] = lse2;
          }
        }
      }
      wg_bar(wg);
#pragma unroll 1
      for (int u = 0; u < kVU; ++u) {
        const int d = u * 128 + key;  // O^T lane = output dim
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float v[4];
          tmem_ld4(tm_o + u * N + lane_off + (uint32_t)(c0 + 4 * j), v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = c0 + 4 * j + i;
            if (col >= rows_here) break;
            const float res = v[i] * alpha[col];
            if (nsb == 1) ((__nv_bfloat16*)a.out)[ooff[col] + d] = __float2bfloat16_rn(res);
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
  if (warp == kSWarp) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem));
  }
}

// Latent rows [rows][576] bf16 viewed as (64 dims, rows, 9 pieces) with
// strides (1152 B, 128 B): a box of (64, 128 rows, 2 pieces) lands as
// [2][128][64] with 128-byte swizzle; pieces past the 9th read as zeros.
bool encode_latent(CUtensorMap* m, const void* base, long rows) {
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)kKP};
  const cuuint64_t strides[2] = {(cuuint64_t)kDK * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)kKeys, 2};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tree rows [B*R][Hkv][576] bf16 as (64 dims, Hkv, B*R, 9 pieces), boxes of
// (64, 1 head, 128 rows, 2 pieces); rows past B*R read as zeros.
bool encode_latent_tree(CUtensorMap* m, const void* base, int Hkv, long rows) {
  const cuuint64_t dims[4] = {64, (cuuint64_t)Hkv, (cuuint64_t)rows, (cuuint64_t)kKP};
  const cuuint64_t strides[3] = {(cuuint64_t)kDK * 2, (cuuint64_t)Hkv * kDK * 2, 128};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kKeys, 2};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
void launch_mla(const MlaMaps& maps, const VerifyArgs& a, const VerifyPlan& p, cudaStream_t st) {
  const uint32_t smem = MlaLayout<N>::total + 1024;
  const auto kern = a.page_size > 0 ? verify_mla_kernel<N, true> : verify_mla_kernel<N, false>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  const dim3 grid(p.nsplit, a.Hkv * p.nrg, a.B);
  launch(kern, dim3(grid), dim3(kThreads), smem, st, maps, a, p.rb);
}

}  // namespace

bool launch_mla_tc_path(const tsd_attn_desc& d, const VerifyArgs& a, const VerifyPlan& p,
                        cudaStream_t st) {
  if (d.dk != kDK || d.dv != kDV || !d.v_aliases_k || d.dtype != TSD_BF16) return false;
  if (encode_fn() == nullptr || p.rb != 64) return false;
  MlaMaps maps;
  const long cache_rows = a.page_size > 0 ? (long)a.num_pages * d.Hkv * a.page_size
                                          : (long)d.B * d.Hkv * d.cap;
  if (!encode_latent(&maps.k, a.kc, cache_rows) ||
      !encode_latent_tree(&maps.kt, a.kt, d.Hkv, (long)d.B * d.R))
    return false;
  launch_mla<64>(maps, a, p, st);
  if (p.nsplit > 1) {
    const long rows = (long)a.B * a.R * a.Hq;
    launch_plain(verify_combine_kernel<__nv_bfloat16, kDV>, dim3((unsigned)ceil_div(rows, 4)),
                 dim3(128), 0, st, a);
  }
  return true;
}

}  // namespace tsd
