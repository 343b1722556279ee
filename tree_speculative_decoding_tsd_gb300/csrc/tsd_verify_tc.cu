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
// What bounds it.  Both products read their operands from shared memory,
// which delivers 128 bytes per clock to the tensor core, the TMA writes and
// the softmax's P^T stores together: per 128-key tile that is 64 KB of K/V
// arriving, K and Q^T read by S^T, V and P^T read by O^T, and P^T written --
// about 236 KB at 144 packed rows, ~0.9 us at 2 GHz.  P^T_t is written into
// the ring stage that held K_t (dead once S^T_t is done), so a 3-stage K ring
// gives P^T three buffers without more shared memory, the softmax of tile t
// never waits for O^T_(t-1), and the tensor core always has the next product
// queued.  Measured (per-CTA clock stamps at every hand-off), the tile period
// is set by the cycle of one K stage -- copy landed (~1.5 us under load),
// S^T product, softmax (~1.3 us), O^T product, release, next copy issued --
// divided by the three stages; the shared-memory capacity (Q^T, three K/P^T
// stages, two V stages) leaves no room for a fourth.
//
// Roles (608 threads): warps 0-15 softmax/epilogue (warpgroup w/4 owns a
// quarter of the columns, warp w%4 owns TMEM lanes 32(w%4)..+31, i.e. 32 keys
// of a tile or 32 dims of O^T); warp 16 allocates TMEM and issues the MMAs
// (one thread); warps 17 and 18 issue the K and V loads (a thread completes
// about one TMA operation per ~300-600 cycles, so each stream has its own
// warp).  A K or V tile (128 keys, 32 KB) is one TMA box of a 3-D tensor map
// with 128-byte swizzle.  K_t is loaded once O^T_(t-3) has consumed the
// P^T that shared its stage, V_t once O^T_(t-2) is done.  mbarriers order
// TMA -> MMA -> softmax -> MMA.
//
// Columns.  Warpgroup w takes the octets of columns 32u + 8w .. +7 (and, when
// N/16 is odd, the quad 32(N/32) + 4w .. +3), so its P^T rows are 16-byte
// (or 8-byte) stores at per-thread offsets fixed for the whole kernel.  P^T is
// kept MN-major without swizzle: 8x8 core matrices of 128 contiguous bytes,
// the 16 groups of 8 keys of one 8-column core column adjacent (128 B apart),
// core columns 2 KB apart, so the 32 keys of a warp store 512 contiguous
// bytes and the 16 keys of one K step of the O^T product are 256 contiguous
// bytes per core column.  (With the groups of 8 keys N/8 cores apart the
// long workload's verify took 2% longer; ncu counts the same shared-memory
// store wavefronts for both layouts.)
//
// Softmax with keys on lanes: a thread holds one key's scores for its
// columns, so a column's max and sum are cross-lane reductions, and the
// running max m[n] is lazy.  Each half of a thread's columns is turned into
// x = s*scale*log2(e) - m with packed fp32 pairs and the largest x is taken
// (phase 1); one warpgroup barrier decides.  If no x passed 8 the tile keeps
// the old max: p = 2^x <= 256 (phase 2).  Otherwise (and always on a CTA's
// first tile) the warpgroup computes the tile's column maxima, re-centres x
// on the new max, and scales the partial sums and the O^T columns by
// 2^(m_old - m_new) before phase 2.  Row sums are reduced across lanes once,
// at the end.
//
// Every mbarrier wait is bounded; a timeout sets TSD_DEV_ERR_TIMEOUT in the
// error word, all roles stop, in-flight copies and MMAs are waited for and the
// tensor memory is released.  The pipeline waits take their budget from the
// call (about a second by default, see tsd_set_wait_budget); the teardown
// waits for copies and products in flight always keep the full budget.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "tsd_common.cuh"
#include "tsd_host.h"
#include "tsd_tcgen05.cuh"
#include "tsd_verify.cuh"

namespace tsd {
namespace {

constexpr int kKeys = 128;                      // keys per tile (MMA M of S^T)
constexpr int kD = 128;                         // head dim
constexpr int kSoftWarps = 16;                  // 4 warpgroups, one quarter of the columns each
constexpr int kThreadsTC = (kSoftWarps + 3) * 32;
constexpr int kMmaWarp = 16, kTmaWarp = 17, kTmaVWarp = 18;
constexpr uint32_t kBox = kKeys * 128;          // one [128 rows][64 bf16] swizzled half: 16 KB
constexpr uint32_t kTileBytes = 2 * kBox;       // one K or V tile: 32 KB
constexpr int kKStages = 3;                     // K ring (each stage then holds that tile's P^T)
constexpr int kPagedTiles = 64;  // paged cache: tile rows resolved at set-up
constexpr float kOverflow = 8.0f;               // log2 headroom of the lazy max
// Prefix tiles prefetched into L2 ahead of their shared-memory load.  One is
// best measured (batched workload: 1 tile 125 us, 3 tiles 128, 5 tiles 136):
// deeper prefetches only compete with the loads for L2 and DRAM.
constexpr int kPrefetch = 1;
constexpr int kLptMaxBatch = 64;                // longest-first request order up to this batch

template <int N>
struct TcLayout {
  static constexpr uint32_t pt_bytes = 256u * N;                 // P^T: 128 keys x N bf16
  static constexpr uint32_t stage =
      ((pt_bytes > kTileBytes ? pt_bytes : kTileBytes) + 1023u) / 1024u * 1024u;
  static constexpr uint32_t off_k = 0;                           // K ring
  static constexpr uint32_t off_v = kKStages * stage;            // V ring: 2 x 32 KB
  static constexpr uint32_t off_q = off_v + 2 * kTileBytes;      // Q: N rows x 256 B
  static constexpr uint32_t q_bytes = 2u * N * 128u;
  static constexpr uint32_t off_misc = off_q + (q_bytes + 1023u) / 1024u * 1024u;
  static constexpr int NH = N / 4;                // columns per warpgroup
  static constexpr int NO = N / 32;               // column octets per warpgroup
  static constexpr bool HQ = (N / 16) & 1;        // plus one quad
  static constexpr int NU = NO + (HQ ? 1 : 0);    // column units (octets, then the quad)
  static constexpr int U0 = NO / 2;               // units of the first half: [0, U0)
  // misc area
  static constexpr uint32_t off_m = off_misc;                       // float[N]   running max
  static constexpr uint32_t off_alpha = off_m + 4 * N;              // float[N]   rescale factors
  static constexpr uint32_t off_negm = off_alpha + 4 * N;           // float[N]   -m (0 if m = -inf)
  static constexpr uint32_t off_red = off_negm + 4 * N;             // float[16][NH] per-warp partials
  static constexpr uint32_t off_shift = off_red + 4 * kSoftWarps * NH;  // float[N] max shifts
  static constexpr uint32_t off_rmask = (off_shift + 4 * N + 7) / 8 * 8;  // u64[N] tree masks
  static constexpr uint32_t off_ooff = off_rmask + 8 * N;           // i64[N] output offsets
  static constexpr uint32_t off_bar = off_ooff + 8 * N;             // mbarriers
  static constexpr int nbar = 17;
  static constexpr uint32_t off_flags = off_bar + 8 * nbar;  // tmem addr, abort flag, request
  static constexpr uint32_t off_tiles = off_flags + 16;  // int[kPagedTiles] tile rows (paged)
  static constexpr uint32_t total = off_tiles + 4 * kPagedTiles;
  static_assert(total + 1024 <= 232448, "shared memory budget");
  // warpgroup-local column lc (0..NH-1) -> column of S^T / P^T / O^T
  __device__ static int col(int lc, int wg) {
    return lc < 8 * NO ? 32 * (lc >> 3) + 8 * wg + (lc & 7) : 32 * NO + 4 * wg + (lc - 8 * NO);
  }
};

// Barrier indices.  K_FULL/K_EMPTY per K stage, V_FULL/V_EMPTY per V stage,
// S_FULL per S^T buffer, P_FULL per tile parity, PV_DONE per O^T product,
// O_DONE once after the last O^T product.
// A warpgroup may run one tile ahead of another (S^T_(t+1) is issued before
// O^T_t), never two (S^T_(t+2) waits for P_FULL_t): the 16 softmax warps'
// arrivals for tile t go to the P_FULL barrier of t's parity, so an early
// arrival for t+1 never counts toward t.  A softmax warp waits on PV_DONE only
// from tile t, when products 0..t-2 are known complete, so its parity is
// unambiguous; the epilogue waits on O_DONE.
enum { BAR_K_FULL = 0, BAR_K_EMPTY = 3, BAR_V_FULL = 6, BAR_V_EMPTY = 8, BAR_S_FULL = 10,
       BAR_P_FULL = 12, BAR_PV_DONE = 14, BAR_FINAL = 15, BAR_O_DONE = 16 };

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
  // Requests are taken longest first when the batch has 2 to 64 of them
  // (grid z is the rank of the request in (prefix length desc, index asc)
  // order), so that the last wave holds the shortest CTAs.
  const bool lpt = a.B > 1 && a.B <= kLptMaxBatch;
  // While the previous kernel finishes: L2 prefetch of this CTA's first two
  // prefix tiles (K and V, one warp each; contiguous cache only, the page
  // table may still be being written) and of its Q rows.  Hints only, and
  // only where the request is known before the prefix lengths are read.
  if (!lpt) {
    const int w = threadIdx.x >> 5, ln = threadIdx.x & 31;
    const int hk0 = blockIdx.x / a.nrg, b0 = blockIdx.z;
    const int kp0 = blockIdx.y * a.split_len;
    if (!kPaged && w < 4 && ln == 0) {
      const int t = w >> 1;
      const CUtensorMap* m = (w & 1) ? &maps.v : &maps.k;
      if (kp0 + t * kKeys < a.cap)
        tma_prefetch_3d(m, 0, (b0 * a.Hkv + hk0) * a.cap + kp0 + t * kKeys, 0);
    } else if (w == 4) {
      // packed rows [p0, p1) of this row group: for each tree row, the heads
      // of this KV head are one contiguous run of q
      const int p0 = (blockIdx.x % a.nrg) * rows_per_cta;
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
  constexpr int NH = L::NH, NO = L::NO, NU = L::NU, U0 = L::U0;
  // 128-byte-swizzled TMA boxes and MMA operands need 1024-byte-aligned atoms:
  // align the dynamic shared-memory base by hand (1 KB of slack is requested)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = su32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  float* m_run = (float*)(smem + L::off_m);
  float* alpha = (float*)(smem + L::off_alpha);
  float* negm = (float*)(smem + L::off_negm);
  float* red = (float*)(smem + L::off_red);
  float* shiftv = (float*)(smem + L::off_shift);
  uint64_t* rmask = (uint64_t*)(smem + L::off_rmask);
  long long* ooff = (long long*)(smem + L::off_ooff);
  volatile uint32_t* flags = (volatile uint32_t*)(smem + L::off_flags);  // [0] tmem, [1] abort, [2] b
  const uint32_t bar0 = sbase + L::off_bar;
  auto bar = [&](int i) { return bar0 + 8u * i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sp = blockIdx.y;
  const int hk = blockIdx.x / a.nrg, rg = blockIdx.x % a.nrg;
  int b = blockIdx.z;
  if (lpt) {
    // warp 0 ranks the requests (lane l holds requests l and l + 32); the one
    // of rank blockIdx.z is this CTA's
    if (warp == 0) {
      const int i0 = lane, i1 = lane + 32;
      const int p0 = i0 < a.B ? min(max(a.plen[i0], 0), a.cap) : -1;
      const int p1 = i1 < a.B ? min(max(a.plen[i1], 0), a.cap) : -1;
      int r0 = 0, r1 = 0;
      for (int j = 0; j < a.B; ++j) {
        const int pj = __shfl_sync(kFull, j < 32 ? p0 : p1, j & 31);
        r0 += (pj > p0 || (pj == p0 && j < i0)) ? 1 : 0;
        r1 += (pj > p1 || (pj == p1 && j < i1)) ? 1 : 0;
      }
      if (i0 < a.B && r0 == (int)blockIdx.z) flags[2] = (uint32_t)i0;
      if (i1 < a.B && r1 == (int)blockIdx.z) flags[2] = (uint32_t)i1;
    }
    __syncthreads();
    b = (int)flags[2];
  }
  const int P = min(max(a.plen[b], 0), a.cap);
  const int nsb = verify_splits(a, P);
  if (sp >= nsb) return;  // uniform for the whole CTA, before any barrier or allocation
  // (a tree-only split starts at P: no prefix tiles)
  const int k0 = min(sp * a.split_len, P), k1 = min(P, k0 + a.split_len);
  const int n_pre = k1 > k0 ? (k1 - k0 + kKeys - 1) / kKeys : 0;
  const int n_tree = (sp == nsb - 1) ? 1 : 0;   // R <= 65 < 128: one tile
  const int ntiles = n_pre + n_tree;
  const int row_base = rg * rows_per_cta;
  const int rows_here = min(rows_per_cta, a.M - row_base);

  // ---------------------------------------------------------------- set-up
  // The K thread initialises the barriers and starts the first K loads at
  // once, so they overlap the Q staging and the TMEM allocation.
  // Paged cache: the set-up resolves the first kPagedTiles tile rows into
  // shared memory (tiles_ready of them, 0 until the set-up barrier).
  int* tile_rows = (int*)(smem + L::off_tiles);
  int tiles_ready = 0;
  // first row of prefix tile t in the cache, or in the page pool
  auto ycoord = [&](int t) {
    if constexpr (kPaged) {
      if (t < tiles_ready) return tile_rows[t];
      return paged_tile_row(a, b, hk, k0 + t * kKeys);
    } else {
      return (b * a.Hkv + hk) * a.cap + k0 + t * kKeys;
    }
  };
  auto tma_k = [&](int t) {
    const int stg = t % kKStages;
    const uint32_t dst = sbase + L::off_k + stg * L::stage;
    const uint32_t fb = bar(BAR_K_FULL + stg);
    mbar_expect_tx(fb, kTileBytes);
    if (t < n_pre) tma_3d(dst, &maps.k, 0, ycoord(t), 0, fb);
    else tma_4d(dst, &maps.kt, 0, hk, b * a.R, 0, fb);
  };
  auto tma_v = [&](int t) {
    const uint32_t dst = sbase + L::off_v + (t & 1) * kTileBytes;
    const uint32_t fb = bar(BAR_V_FULL + (t & 1));
    mbar_expect_tx(fb, kTileBytes);
    if (t < n_pre) tma_3d(dst, &maps.v, 0, ycoord(t), 0, fb);
    else tma_4d(dst, &maps.vt, 0, hk, b * a.R, 0, fb);
  };
  // L2 prefetch of a prefix tile's K or V a few tiles ahead of its smem load
  auto prefetch = [&](const CUtensorMap* m, int t) {
    if (t < n_pre) tma_prefetch_3d(m, 0, ycoord(t), 0);
  };
  if (warp == kTmaWarp && lane == 0) {
    for (int s3 = 0; s3 < kKStages; ++s3) {
      mbar_init(bar(BAR_K_FULL + s3), 1);
      mbar_init(bar(BAR_K_EMPTY + s3), 1);
    }
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(bar(BAR_V_FULL + s2), 1);
      mbar_init(bar(BAR_V_EMPTY + s2), 1);
      mbar_init(bar(BAR_S_FULL + s2), 1);
    }
    mbar_init(bar(BAR_P_FULL), kSoftWarps);
    mbar_init(bar(BAR_P_FULL + 1), kSoftWarps);
    mbar_init(bar(BAR_PV_DONE), 1);
    mbar_init(bar(BAR_FINAL), 1);
    mbar_init(bar(BAR_O_DONE), 1);
    flags[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    // the first K tiles at once; V_0 (needed only after the first softmax)
    // follows the set-up barrier from its own warp
    tma_k(0);
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
        sbase + L::off_flags));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
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
      cp_async16(sbase + L::off_q + (c >> 3) * (N * 128u) + n * 128u + (((c & 7) ^ (n & 7)) << 4),
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
  // S^T buffer i at column i*N (arithmetic, not an array indexed at run time,
  // which would live in local memory)
  auto tm_s = [&](int i) { return tmem + (uint32_t)(i * N); };
  const uint32_t tm_o = tmem + 2u * N;

  // ------------------------------------------------------------------ TMA
  // One warp per ring, one load and one L2 prefetch per tile each.
  if (warp == kTmaWarp) {
    if (lane == 0) {
      int nk = 1;
      for (int t = 1; t < kKStages && t < ntiles; ++t, ++nk) tma_k(t);
      for (int t = kKStages; t < kKStages + kPrefetch; ++t) prefetch(&maps.k, t);
      // K_t reuses the stage of tile t-3 once O^T_(t-3) has read its P^T
      for (int t = kKStages; t < ntiles && !flags[1]; ++t) {
        if (!mbar_wait(bar(BAR_K_EMPTY + t % kKStages), (t / kKStages - 1) & 1, a.wait_cycles)) {
          flags[1] = 1;
          break;
        }
        tma_k(t);
        prefetch(&maps.k, t + kPrefetch);
        ++nk;
      }
      // no copy may still be in flight when the CTA leaves
      for (int st = 0; st < kKStages; ++st) {
        const int ck = (nk - st + kKStages - 1) / kKStages;  // loads into stage st
        if (ck > 0) mbar_wait(bar(BAR_K_FULL + st), (ck - 1) & 1);
      }
    }
  } else if (warp == kTmaVWarp) {
    if (lane == 0) {
      int nv = 0;
      for (int t = 1; t < 1 + kPrefetch; ++t) prefetch(&maps.v, t);
      for (int tv = 0; tv < ntiles && !flags[1]; ++tv) {
        if (tv >= 2 && !mbar_wait(bar(BAR_V_EMPTY + (tv & 1)), ((tv - 2) >> 1) & 1, a.wait_cycles)) {
          flags[1] = 1;
          break;
        }
        tma_v(tv);
        prefetch(&maps.v, tv + kPrefetch);
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
      // descriptor bases (built once): K stage 0, V stage 0, Q^T, and P^T in
      // K stage 0 (MN-major without swizzle, where the leading offset is the
      // stride between groups of 8 keys, 128 B, and the stride offset the one
      // between cores along N, 2 KB: the 16 key groups of 8 columns are one
      // contiguous 2 KB block, so a warp's 32 keys store 512 contiguous bytes)
      const uint64_t kd0 = smem_desc(sbase + L::off_k, 16, 1024);
      const uint64_t vd0 = smem_desc(sbase + L::off_v, kBox, 1024);
      const uint64_t qd0 = smem_desc(sbase + L::off_q, 16, 1024);
      const uint64_t ptd0 = smem_desc_interleave(sbase + L::off_k, 128, 2048);
      auto issue_qk = [&](int t) -> bool {
        const int stg = t % kKStages;
        if (!mbar_wait(bar(BAR_K_FULL + stg), (t / kKStages) & 1, a.wait_cycles)) return false;
        fence_after();
        const uint64_t kd = kd0 + (uint64_t)(stg * (L::stage >> 4));
        const uint32_t ts = tm_s(t & 1);
        mma_f16(ts, kd, qd0, idesc_qk, 0u);
#pragma unroll
        for (int kk = 1; kk < kD / 16; ++kk)
          mma_f16_acc(ts, kd + (((kk >> 2) * kBox + (kk & 3) * 32) >> 4),
                      qd0 + (((kk >> 2) * (N * 128u) + (kk & 3) * 32) >> 4), idesc_qk);
        mma_commit(bar(BAR_S_FULL + (t & 1)));
        return true;
      };
      bool ok = issue_qk(0);
      for (int t = 0; ok && t < ntiles; ++t) {
        if (t + 1 < ntiles && !issue_qk(t + 1)) { ok = false; break; }
        if (!mbar_wait(bar(BAR_P_FULL + (t & 1)), (t >> 1) & 1, a.wait_cycles) || flags[1]) { ok = false; break; }
        if (!mbar_wait(bar(BAR_V_FULL + (t & 1)), (t >> 1) & 1, a.wait_cycles)) { ok = false; break; }
        fence_after();
        const int stg = t % kKStages;
        const uint64_t vd = vd0 + (uint64_t)((t & 1) * (kTileBytes >> 4));
        const uint64_t pd = ptd0 + (uint64_t)(stg * (L::stage >> 4));
        if (t == 0) mma_f16(tm_o, vd, pd, idesc_pv, 0u);
        else mma_f16_acc(tm_o, vd, pd, idesc_pv);
#pragma unroll
        for (int kk = 1; kk < kKeys / 16; ++kk)
          mma_f16_acc(tm_o, vd + 128 * kk, pd + (uint64_t)(16 * kk), idesc_pv);
        mma_commit(bar(BAR_PV_DONE));
        mma_commit(bar(BAR_V_EMPTY + (t & 1)));
        mma_commit(bar(BAR_K_EMPTY + stg));
        if (t == ntiles - 1) mma_commit(bar(BAR_O_DONE));
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
    const int key = q * 32 + lane;           // TMEM lane = key of the tile / dim of O^T
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    // P^T row of this key: octet u at pt_oct + 8192u (columns 32u + 8wg..+7,
    // core column 4u + wg), the quad at pt_quad (offsets within a K stage)
    const uint32_t pt_key = (uint32_t)key * 16u;
    const uint32_t pt_oct = pt_key + (uint32_t)wg * 2048u;
    const uint32_t pt_quad = pt_key + (4u * NO + (uint32_t)(wg >> 1)) * 2048u + (uint32_t)(wg & 1) * 8u;
    // first S^T / O^T column (and per-column smem slot) of octet 0 and of the quad
    const int c_oct = 8 * wg, c_quad = 32 * NO + 4 * wg;
    const float2 c2 = make_float2(a.qscale, a.qscale);
    float2 l2[NH / 2];                       // this key lane's partial row sums, by pairs
#pragma unroll
    for (int i = 0; i < NH / 2; ++i) l2[i] = make_float2(0.f, 0.f);
    bool failed = false;

    for (int t = 0; t < ntiles; ++t) {
      const int st = t & 1;
      // tcgen05.ld is warp-collective: the whole warp agrees on the wait
      const bool ok = __all_sync(kFull, mbar_wait(bar(BAR_S_FULL + st), (t >> 1) & 1, a.wait_cycles));
      fence_after();
      const bool is_tree = t >= n_pre;
      const int nvalid = is_tree ? a.R : min(kKeys, k1 - (k0 + t * kKeys));
      const uint32_t srow = tm_s(st) + lane_off;
      uint8_t* pt_stage = smem + L::off_k + (t % kKStages) * L::stage;
      bool pv_waited = false;                // O^T_(t-1) known complete

      // The warpgroup's column units are taken in two halves (a quarter of
      // the registers each way: 19 warps leave 96 registers per thread).
      bool stop_now = false;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ua = h == 0 ? 0 : U0, ub = h == 0 ? U0 : NU;
        if (ua >= ub) continue;
        constexpr int VMAX = 8 * (NO - NO / 2) + 4;
        const int lc0 = 8 * ua;              // first warpgroup-local column of the half
        const int ncol = (ub == NU && L::HQ) ? 8 * (ub - 1 - ua) + 4 : 8 * (ub - ua);
        // Phase 1: this key's scores for the half's columns, turned into
        // x = s*scale*log2(e) - m (m the column's running max, 0 while it is
        // -inf), and the largest x.  Masked keys are -inf before the product.
        float v[VMAX];
        if (ok) {
#pragma unroll
          for (int u = ua; u < ub; ++u) {
            float* x = v + 8 * (u - ua);
            if (u < NO) tmem_ld8(srow + (uint32_t)(32 * u + c_oct), x);
            else tmem_ld4(srow + (uint32_t)c_quad, x[0], x[1], x[2], x[3]);
          }
          tmem_wait_ld();
        }
        if (is_tree || nvalid < kKeys) {     // the tree tile and a ragged last tile only
          if (key >= nvalid) {
#pragma unroll
            for (int e = 0; e < VMAX; ++e) v[e] = -INFINITY;
          } else if (is_tree && key > 0) {
            // visibility of this key (tree row) to each of the half's columns
            uint32_t vis = 0u;
#pragma unroll 1
            for (int e = 0; e < ncol; ++e)
              vis |= (uint32_t)((rmask[L::col(lc0 + e, wg)] >> (key - 1)) & 1ull) << e;
#pragma unroll
            for (int e = 0; e < VMAX; ++e)
              if (!((vis >> e) & 1u)) v[e] = -INFINITY;
          }
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int u = ua; u < ub; ++u) {
          float* x = v + 8 * (u - ua);
          const int nq = u < NO ? 2 : 1;     // quads in this unit
          const int c = u < NO ? 32 * u + c_oct : c_quad;
#pragma unroll
          for (int j = 0; j < nq; ++j) {
            const float4 nm = *(const float4*)(negm + c + 4 * j);
            const float2 x01 = __ffma2_rn(make_float2(x[4 * j], x[4 * j + 1]), c2,
                                          make_float2(nm.x, nm.y));
            const float2 x23 = __ffma2_rn(make_float2(x[4 * j + 2], x[4 * j + 3]), c2,
                                          make_float2(nm.z, nm.w));
            x[4 * j] = x01.x;
            x[4 * j + 1] = x01.y;
            x[4 * j + 2] = x23.x;
            x[4 * j + 3] = x23.y;
            tmax = max3f(tmax, x01.x, x01.y);
            tmax = max3f(tmax, x23.x, x23.y);
          }
        }

        // One barrier in the common case.  If some x passed the headroom (and
        // always on a CTA's first tile) the warpgroup takes the exact path for
        // the half: the tile's column maxima, the new running max, x
        // re-centred on it, the partial sums and the O^T columns scaled by
        // 2^(m_old - m_new).  The stop decision is taken on the first
        // non-empty half (ua == 0).
        const bool local_stop = ua == 0 && (!ok || failed || flags[1] != 0);
        if (wg_bar_or(wg, local_stop || t == 0 || tmax > kOverflow)) {
          if (ua == 0 && wg_bar_or(wg, local_stop)) {
            stop_now = true;
            break;
          }
#pragma unroll
          for (int e4 = 0; e4 < VMAX / 4; ++e4) {
            if (4 * e4 >= ncol) break;
            float r4[4] = {v[4 * e4], v[4 * e4 + 1], v[4 * e4 + 2], v[4 * e4 + 3]};
            const float r = warp_reduce_scatter<4, true>(r4, lane);
            if (lane < 4) red[warp * NH + lc0 + 4 * e4 + lane] = r;
          }
          wg_bar(wg);
          for (int n = lc0 + (tid & 127); n < lc0 + ncol; n += 128) {
            const int col = L::col(n, wg);
            float X = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) X = fmaxf(X, red[(wg * 4 + w) * NH + n]);
            const float m_old = m_run[col];
            float m_new, sh, al;
            if (m_old == -INFINITY) {        // x was s*c itself; nothing accumulated yet
              m_new = X;
              sh = X == -INFINITY ? 0.f : X;
              al = 0.f;
            } else {                         // x = s*c - m_old
              sh = fmaxf(X, 0.f);
              m_new = m_old + sh;
              al = ex2(-sh);
            }
            m_run[col] = m_new;
            alpha[col] = al;
            shiftv[col] = sh;
            negm[col] = m_new == -INFINITY ? 0.f : -m_new;
          }
          wg_bar(wg);
          // the previous tile's O^T product must be complete before its
          // columns are rescaled in TMEM
          if (t > 0 && !pv_waited) {
            if (!__all_sync(kFull, mbar_wait(bar(BAR_PV_DONE), (t - 1) & 1, a.wait_cycles))) failed = true;
            fence_after();
            pv_waited = true;
          }
#pragma unroll
          for (int u = ua; u < ub; ++u) {
            float* x = v + 8 * (u - ua);
            const int nq = u < NO ? 2 : 1;
            const int c = u < NO ? 32 * u + c_oct : c_quad;
            const int li = u < NO ? 4 * u : 4 * NO;   // first l2 pair of the unit
#pragma unroll
            for (int j = 0; j < nq; ++j) {
              const float4 sh = *(const float4*)(shiftv + c + 4 * j);
              const float4 al = *(const float4*)(alpha + c + 4 * j);
              x[4 * j] -= sh.x;
              x[4 * j + 1] -= sh.y;
              x[4 * j + 2] -= sh.z;
              x[4 * j + 3] -= sh.w;
              l2[li + 2 * j] = __fmul2_rn(l2[li + 2 * j], make_float2(al.x, al.y));
              l2[li + 2 * j + 1] = __fmul2_rn(l2[li + 2 * j + 1], make_float2(al.z, al.w));
            }
            if (t > 0 && !failed) {
              float o[8];
              const uint32_t ta = tm_o + lane_off + (uint32_t)c;
              if (u < NO) tmem_ld8(ta, o);
              else tmem_ld4(ta, o[0], o[1], o[2], o[3]);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < nq; ++j) {
                const float4 al = *(const float4*)(alpha + c + 4 * j);
                o[4 * j] *= al.x;
                o[4 * j + 1] *= al.y;
                o[4 * j + 2] *= al.z;
                o[4 * j + 3] *= al.w;
              }
              if (u < NO) tmem_st8(ta, o);
              else tmem_st4(ta, o[0], o[1], o[2], o[3]);
            }
          }
          tmem_wait_st();
        }
        // Phase 2: p = 2^x (x <= 8 here), partial row sums, P^T row of this key
#pragma unroll
        for (int u = ua; u < ub; ++u) {
          const float* x = v + 8 * (u - ua);
          const int li = u < NO ? 4 * u : 4 * NO;
          float p[8];
#pragma unroll
          for (int e = 0; e < (u < NO ? 8 : 4); ++e) p[e] = ex2(x[e]);
          l2[li] = __fadd2_rn(l2[li], make_float2(p[0], p[1]));
          l2[li + 1] = __fadd2_rn(l2[li + 1], make_float2(p[2], p[3]));
          if (u < NO) {
            l2[li + 2] = __fadd2_rn(l2[li + 2], make_float2(p[4], p[5]));
            l2[li + 3] = __fadd2_rn(l2[li + 3], make_float2(p[6], p[7]));
            *(uint4*)(pt_stage + pt_oct + 8192u * u) =
                make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                           pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7]));
          } else {
            *(uint2*)(pt_stage + pt_quad) = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
          }
        }
      }
      if (stop_now) {
        failed = true;
        break;
      }
      // V rows of keys past the range may hold anything: zero them (the
      // warpgroup of the first columns does it)
      if (wg == 0 && key >= nvalid) {
        if (!mbar_wait(bar(BAR_V_FULL + st), (t >> 1) & 1, a.wait_cycles)) {
          failed = true;                     // the copy may still be landing: no writes
        } else {
          uint8_t* vrow = smem + L::off_v + st * kTileBytes + key * 128u;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            *(uint4*)(vrow + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
            *(uint4*)(vrow + kBox + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P_FULL + (t & 1)));
    }

    // ---------------------------------------------------------- epilogue
    // (a failed V wait above is per lane: agree on it across the warp)
    failed = __any_sync(kFull, failed);
    const bool ok = !failed && __all_sync(kFull, mbar_wait(bar(BAR_O_DONE), 0, a.wait_cycles));
    fence_after();
    const bool stop = wg_bar_or(wg, !ok || flags[1] != 0);
    if (!stop) {
      // row sums across the 128 key lanes
#pragma unroll
      for (int i = 0; i < NH / 4; ++i) {
        float r4[4] = {l2[2 * i].x, l2[2 * i].y, l2[2 * i + 1].x, l2[2 * i + 1].y};
        const float r = warp_reduce_scatter<4, false>(r4, lane);
        if (lane < 4) red[warp * NH + 4 * i + lane] = r;
      }
      wg_bar(wg);
      // per column: 1/l into alpha[], destination offset, log-sum-exp
      for (int n = tid & 127; n < NH; n += 128) {
        const int col = L::col(n, wg);
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
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        float o[8];
        const int c = u < NO ? 32 * u + c_oct : c_quad;
        if (u < NO) tmem_ld8(tm_o + lane_off + (uint32_t)c, o);
        else tmem_ld4(tm_o + lane_off + (uint32_t)c, o[0], o[1], o[2], o[3]);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < (u < NO ? 8 : 4); ++e) {
          const int col = c + e;
          if (col >= rows_here) continue;
          const float res = o[e] * alpha[col];
          if (nsb == 1) ((__nv_bfloat16*)a.out)[ooff[col] + d] = __float2bfloat16_rn(res);
          else a.ws_ob[ooff[col] + d] = __float2bfloat16_rn(res);
        }
      }
    }
    if (!ok && lane == 0) flags[1] = 1;      // a failed wait of this warp's, or O_DONE's
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

// Prefix cache viewed as (64 dims, rows, 2 halves) with strides (256 B, 128 B):
// one box of [2 halves][128 rows][64 dims] (32 KB, 128-byte swizzle) is a whole
// K or V tile in the layout the MMA descriptors expect.
bool encode_pair(CUtensorMap* m, const void* base, long rows) {
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, 2};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)kKeys, 2};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scratch pad [B*R][Hkv][128] as (64 dims, Hkv, rows, 2 halves): one box of
// [2][128 rows][1 head][64] holds a head's tree rows (rows past B*R read as 0).
bool encode_tree_pair(CUtensorMap* m, const void* base, int Hkv, long rows) {
  const cuuint64_t dims[4] = {64, (cuuint64_t)Hkv, (cuuint64_t)rows, 2};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)Hkv * kD * 2, 128};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kKeys, 2};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
void launch_tc(const TcMaps& maps, const VerifyArgs& a, const VerifyPlan& p, cudaStream_t st) {
  const uint32_t smem = TcLayout<N>::total + 1024;
  const auto kern = a.page_size > 0 ? verify_tc_kernel<N, true> : verify_tc_kernel<N, false>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  // (KV head and row group fastest, then the split: the last CTAs of the
  // grid are the last split, which only requests with the longest prefixes
  // use, so a grid just past one wave ends with CTAs that return at once;
  // the row groups of a head run side by side and share its tiles in L2)
  const dim3 grid(a.Hkv * p.nrg, p.nsplit, a.B);
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
  if (!encode_pair(&maps.k, a.kc, cache_rows) || !encode_pair(&maps.v, a.vc, cache_rows) ||
      !encode_tree_pair(&maps.kt, a.kt, d.Hkv, (long)d.B * d.R) ||
      !encode_tree_pair(&maps.vt, a.vt, d.Hkv, (long)d.B * d.R))
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
    launch_plain(verify_combine_kernel<__nv_bfloat16, 128, __nv_bfloat16>,
                 dim3((unsigned)ceil_div(rows, 4)), dim3(128), 0, st, a);
  }
  return true;
}

}  // namespace tsd
