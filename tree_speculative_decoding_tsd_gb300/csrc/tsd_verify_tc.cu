// tcgen05 (5th-generation tensor core) path of tsd_tree_verify_attn for bf16
// GQA heads with dk == dv == 128 and at least 64 packed query rows.
//
// Layout choice.  The packed query rows of one KV head (R tree rows x g query
// heads: 68, 132 or 260 for the workloads here) rarely fill 128-row MMA tiles,
// so the products are computed transposed, with the packed rows on the MMA N
// dimension (a multiple of 16, padded by at most 15 rows):
//   S^T[key][n]  = K_tile . Q^T     M = 128 keys,  N = packed rows, K = dk
//   O^T[d][n]   += V_tile^T . P^T   M = 128 (dv),  N = packed rows, K = 128 keys
// Both accumulators live in tensor memory (fp32); S^T is double-buffered.
//
// Roles (320 threads): warps 0-7 softmax/epilogue (warpgroup w/4 owns half of
// the columns, warp w%4 owns TMEM lanes 32(w%4)..+31, i.e. 32 keys of a tile
// or 32 dims of O^T); warp 8 allocates TMEM and issues the MMAs (one thread);
// warp 9 issues the TMA loads (one thread).  K/V tiles of 128 keys (64 KB per
// stage, two stages) arrive by cp.async.bulk.tensor with 128-byte swizzle;
// mbarriers order TMA -> MMA -> softmax -> MMA.
//
// Softmax with keys on lanes: a thread holds one key's scores for all of its
// columns, so a row's max and sum are cross-lane reductions.  The running max
// m[n] is therefore lazy: it is recomputed exactly (warp reduce-scatter plus a
// shared-memory pass) on the first tile and whenever a score exceeds it by more
// than 8 in the log2 domain (probabilities stay <= 2^8, safe in bf16/fp32);
// O^T columns and the partial sums are then rescaled by 2^(m_old - m_new).
// Row sums accumulate per key lane and are reduced once, at the end.
//
// Every mbarrier wait is bounded (about a second); a timeout sets
// TSD_DEV_ERR_TIMEOUT in the error word, all roles stop, in-flight copies and
// MMAs are waited for (again bounded) and the tensor memory is released.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "tsd_common.cuh"
#include "tsd_host.h"
#include "tsd_verify.cuh"

namespace tsd {
namespace {

constexpr int kKeys = 128;          // keys per tile (MMA M of S^T)
constexpr int kD = 128;             // head dim
constexpr int kSoftWarps = 8;
constexpr int kThreadsTC = (kSoftWarps + 2) * 32;
constexpr int kMmaWarp = 8, kTmaWarp = 9;
constexpr uint32_t kBox = kKeys * 128;          // one [128 rows][64 bf16] swizzled box: 16 KB
constexpr uint32_t kStageBytes = 4 * kBox;      // K (2 boxes) + V (2 boxes)
constexpr uint32_t kOffQ = 2 * kStageBytes;     // 128 KB
constexpr float kOverflow = 8.0f;               // log2 headroom of the lazy max
constexpr long long kWaitCycles = 2000000000ll; // ~1 s at 2 GHz

template <int N>
struct TcLayout {
  static constexpr uint32_t q_bytes = 2u * N * 128u;
  static constexpr uint32_t off_pt = kOffQ + ((q_bytes + 1023u) / 1024u) * 1024u;
  static constexpr uint32_t pt_blocks = (N + 63) / 64;
  static constexpr uint32_t off_misc = off_pt + pt_blocks * kBox;
  static constexpr int NH = N / 2;                // columns per warpgroup
  // misc area
  static constexpr uint32_t off_m = off_misc;                       // float[N]   running max
  static constexpr uint32_t off_alpha = off_m + 4 * N;              // float[N]   rescale factors
  static constexpr uint32_t off_red = off_alpha + 4 * N;            // float[8][NH] per-warp partials
  static constexpr uint32_t off_lsum = off_red + 4 * 8 * NH;        // float[N]   row sums
  static constexpr uint32_t off_rmask = (off_lsum + 4 * N + 7) / 8 * 8;  // u64[N] tree masks
  static constexpr uint32_t off_bar = off_rmask + 8 * N;            // mbarriers
  static constexpr int nbar = 10;
  static constexpr uint32_t off_flags = off_bar + 8 * nbar;          // tmem addr, abort flag
  static constexpr uint32_t total = off_flags + 16;
  static_assert(total + 1024 <= 232448, "shared memory budget");
};

// barrier indices
enum { BAR_KV_FULL = 0, BAR_KV_EMPTY = 2, BAR_S_FULL = 4, BAR_P_FULL = 6, BAR_PV_DONE = 7,
       BAR_FINAL = 8 };

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > kWaitCycles) return false;
  }
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 format).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// Named barrier over one warpgroup (128 threads) returning the OR of pred.
__device__ __forceinline__ bool wg_bar_or(int wg, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
      " bar.red.or.pred po, %2, 128, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(1 + wg)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ void wg_bar(int wg) {
  asm volatile("bar.sync %0, 128;\n" ::"r"(1 + wg) : "memory");
}

// Reduce-scatter over the 32 lanes of a warp for a group of G columns held in
// v[0..G): afterwards lane l holds, in v[0], the reduction over all 32 lanes of
// column (l % G).  G is 8, 16 or 32; MAX selects max, else sum.
template <int G, bool MAX>
__device__ __forceinline__ float warp_reduce_scatter(float* v, int lane) {
#pragma unroll
  for (int s = G / 2; s >= 1; s >>= 1) {
    const bool upper = lane & s;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = upper ? v[i] : v[i + s];
      const float keep = upper ? v[i + s] : v[i];
      const float recv = __shfl_xor_sync(kFull, send, s);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float r = v[0];
#pragma unroll
  for (int s = G; s < 32; s <<= 1) {
    const float o = __shfl_xor_sync(kFull, r, s);
    r = MAX ? fmaxf(r, o) : r + o;
  }
  return r;
}

// Column reduction over the 32 lanes for the NH columns in x[]: the results
// land in red[col] (one writer per column).
template <int NH, bool MAX>
__device__ __forceinline__ void warp_columns(const float* x, float* red, int lane) {
  constexpr int n32 = NH / 32;
  constexpr int rem = NH - 32 * n32;          // 0, 8, 16 or 24
#pragma unroll
  for (int gi = 0; gi < n32; ++gi) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = x[32 * gi + i];
    const float r = warp_reduce_scatter<32, MAX>(v, lane);
    red[32 * gi + lane] = r;
  }
  if (rem >= 16) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = x[32 * n32 + i];
    const float r = warp_reduce_scatter<16, MAX>(v, lane);
    if (lane < 16) red[32 * n32 + lane] = r;
  }
  if (rem % 16 == 8) {
    constexpr int base = NH - 8;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = x[base + i];
    const float r = warp_reduce_scatter<8, MAX>(v, lane);
    if (lane < 8) red[base + lane] = r;
  }
}

struct TcMaps {
  CUtensorMap k, v, kt, vt;
};

template <int N>
__global__ void __launch_bounds__(kThreadsTC, 1)
verify_tc_kernel(const __grid_constant__ TcMaps maps, VerifyArgs a, int rows_per_cta) {
  using L = TcLayout<N>;
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
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
        sbase + L::off_flags));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  if (tid == kTmaWarp * 32) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(BAR_KV_FULL + s), 1);
      mbar_init(bar(BAR_KV_EMPTY + s), 1);
      mbar_init(bar(BAR_S_FULL + s), 1);
    }
    mbar_init(bar(BAR_P_FULL), kSoftWarps);
    mbar_init(bar(BAR_PV_DONE), 1);
    mbar_init(bar(BAR_FINAL), 1);
    flags[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp < kSoftWarps) {
    // Q tile (K-major, 128-byte swizzle: two boxes of [N][64]) and tree masks
    for (int idx = tid; idx < N * 16; idx += kSoftWarps * 32) {
      const int n = idx >> 4, c = idx & 15;
      const int p = row_base + n;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (n < rows_here) {
        const int tr = p / a.g, qh = hk * a.g + p % a.g;
        val = *(const uint4*)((const __nv_bfloat16*)a.q + (((long)b * a.R + tr) * a.Hq + qh) * kD + c * 8);
      }
      const uint32_t off = kOffQ + (c >> 3) * (N * 128u) + n * 128u + (((c & 7) ^ (n & 7)) << 4);
      *(uint4*)(smem + off) = val;
    }
    for (int n = tid; n < N; n += kSoftWarps * 32) {
      uint64_t mk = 0ull;
      if (n < rows_here) {
        const int tr = (row_base + n) / a.g;
        mk = tr > 0 ? a.mask[(long)b * a.R + tr] : 0ull;
      }
      rmask[n] = mk;
      m_run[n] = -INFINITY;
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = flags[0];
  const uint32_t tm_s[2] = {tmem, tmem + (uint32_t)N};
  const uint32_t tm_o = tmem + 2u * N;

  // ------------------------------------------------------------------ TMA
  if (warp == kTmaWarp) {
    if (lane == 0) {
      int issued[2] = {0, 0};
      for (int t = 0; t < ntiles; ++t) {
        const int st = t & 1;
        if (t >= 2 && !mbar_wait(bar(BAR_KV_EMPTY + st), ((t >> 1) - 1) & 1)) {
          flags[1] = 1;
          break;
        }
        if (flags[1]) break;
        const uint32_t dst = sbase + st * kStageBytes;
        const uint32_t fb = bar(BAR_KV_FULL + st);
        mbar_expect_tx(fb, kStageBytes);
        if (t < n_pre) {
          const int y = (b * a.Hkv + hk) * a.cap + k0 + t * kKeys;
          tma_2d(dst, &maps.k, 0, y, fb);
          tma_2d(dst + kBox, &maps.k, 64, y, fb);
          tma_2d(dst + 2 * kBox, &maps.v, 0, y, fb);
          tma_2d(dst + 3 * kBox, &maps.v, 64, y, fb);
        } else {
          const int z = b * a.R;
          tma_3d(dst, &maps.kt, 0, hk, z, fb);
          tma_3d(dst + kBox, &maps.kt, 64, hk, z, fb);
          tma_3d(dst + 2 * kBox, &maps.vt, 0, hk, z, fb);
          tma_3d(dst + 3 * kBox, &maps.vt, 64, hk, z, fb);
        }
        ++issued[st];
      }
      // no copy may still be in flight when the CTA leaves
      for (int st = 0; st < 2; ++st)
        if (issued[st] > 0) mbar_wait(bar(BAR_KV_FULL + st), (issued[st] - 1) & 1);
    }
  }

  // ------------------------------------------------------------------ MMA
  else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t idesc_qk = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
                                ((uint32_t)(kKeys >> 4) << 24);
      const uint32_t idesc_pv = idesc_qk | (1u << 15) | (1u << 16);
      const uint32_t qa = sbase + kOffQ, pta = sbase + L::off_pt;
      auto issue_qk = [&](int t) -> bool {
        const int st = t & 1;
        if (!mbar_wait(bar(BAR_KV_FULL + st), (t >> 1) & 1)) return false;
        fence_after();
        const uint32_t kb = sbase + st * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t ad = smem_desc(kb + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(qa + (kk >> 2) * (N * 128u) + (kk & 3) * 32, 16, 1024);
          mma_f16(tm_s[st], ad, bd, idesc_qk, kk > 0);
        }
        mma_commit(bar(BAR_S_FULL + st));
        return true;
      };
      bool ok = ntiles == 0 || issue_qk(0);
      for (int t = 0; ok && t < ntiles; ++t) {
        if (t + 1 < ntiles && !issue_qk(t + 1)) { ok = false; break; }
        if (!mbar_wait(bar(BAR_P_FULL), t & 1) || flags[1]) { ok = false; break; }
        fence_after();
        const uint32_t vb = sbase + (t & 1) * kStageBytes + 2 * kBox;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t ad = smem_desc(vb + kk * 2048, kBox, 1024);
          const uint64_t bd = smem_desc(pta + kk * 2048, kBox, 1024);
          mma_f16(tm_o, ad, bd, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(BAR_PV_DONE));
        mma_commit(bar(BAR_KV_EMPTY + (t & 1)));
      }
      if (!ok) flags[1] = 1;
      // every MMA issued so far has completed once this barrier flips
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
    // the warpgroup's columns are handled in two halves of H0 and H1 columns
    constexpr int H0 = ((NH / 2 + 7) / 8) * 8, H1 = NH - H0;
    float l[NH];
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
      // scores of this key for columns [h0, h0 + H) with the masks applied
      auto load = [&](float* x, int h0, int H) {
        for (int j = 0; j < H / 8; ++j) {
          float v[8];
          tmem_ld8(tm_s[st] + lane_off + (uint32_t)(c0 + h0 + 8 * j), v);
#pragma unroll
          for (int i = 0; i < 8; ++i) x[8 * j + i] = v[i];
        }
        tmem_wait_ld();
        if (key >= nvalid) {
          for (int n = 0; n < H; ++n) x[n] = -INFINITY;
        } else if (is_tree && key > 0) {
          for (int n = 0; n < H; ++n)
            if (!((rmask[c0 + h0 + n] >> (key - 1)) & 1ull)) x[n] = -INFINITY;
        }
      };
      // pass A: does any score pass the lazy max by more than the headroom?
      bool over = (t == 0);
      if (ok) {
        float x[H0];
        load(x, 0, H0);
#pragma unroll
        for (int n = 0; n < H0; ++n) {
          const float mu = m_run[c0 + n];
          over |= fmaf(x[n], c, -(mu == -INFINITY ? 0.f : mu)) > kOverflow;
        }
        load(x, H0, H1);
#pragma unroll
        for (int n = 0; n < H1; ++n) {
          const float mu = m_run[c0 + H0 + n];
          over |= fmaf(x[n], c, -(mu == -INFINITY ? 0.f : mu)) > kOverflow;
        }
      }
      const bool stop = wg_bar_or(wg, !ok || failed || flags[1] != 0);
      if (stop) { failed = true; break; }
      const bool any_over = wg_bar_or(wg, over);
      if (any_over) {
        // exact column maxima of this tile, then the new running max
        float x[H0];
        load(x, 0, H0);
        warp_columns<H0, true>(x, red + warp * NH, lane);
        load(x, H0, H1);
        warp_columns<H1, true>(x, red + warp * NH + H0, lane);
        wg_bar(wg);
        for (int n = tid & 127; n < NH; n += 128) {
          float mx = -INFINITY;
#pragma unroll
          for (int w = 0; w < 4; ++w) mx = fmaxf(mx, red[(wg * 4 + w) * NH + n]);
          const float m_old = m_run[c0 + n];
          const float m_new = fmaxf(m_old, mx * c);
          alpha[c0 + n] = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
          m_run[c0 + n] = m_new;
        }
        wg_bar(wg);
      }
      // PV of the previous tile must be done before O^T or P^T are touched
      if (t > 0 && !__all_sync(kFull, mbar_wait(bar(BAR_PV_DONE), (t - 1) & 1))) failed = true;
      fence_after();
      if (any_over && t > 0 && !failed) {
#pragma unroll
        for (int n = 0; n < NH; ++n) l[n] *= alpha[c0 + n];
        for (int j = 0; j < NH / 8; ++j) {
          float v[8];
          tmem_ld8(tm_o + lane_off + (uint32_t)(c0 + 8 * j), v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] *= alpha[c0 + 8 * j + i];
          tmem_st8(tm_o + lane_off + (uint32_t)(c0 + 8 * j), v);
        }
        tmem_wait_st();
      }
      // pass B: probabilities, partial row sums, P^T row of this key
      // (MN-major, 128-byte swizzle, blocks of 64 columns)
      auto emit = [&](float* x, int h0, int H) {
        for (int n = 0; n < H; ++n) {
          const float mu = m_run[c0 + h0 + n];
          x[n] = exp2f(fmaf(x[n], c, -(mu == -INFINITY ? 0.f : mu)));
        }
        for (int j = 0; j < H / 8; ++j) {
          const int n0 = c0 + h0 + 8 * j;
          uint4 pk;
          pk.x = pack_bf16x2(x[8 * j], x[8 * j + 1]);
          pk.y = pack_bf16x2(x[8 * j + 2], x[8 * j + 3]);
          pk.z = pack_bf16x2(x[8 * j + 4], x[8 * j + 5]);
          pk.w = pack_bf16x2(x[8 * j + 6], x[8 * j + 7]);
          const uint32_t off = L::off_pt + (n0 >> 6) * kBox + key * 128u +
                               ((((n0 & 63) >> 3) ^ (key & 7)) << 4);
          *(uint4*)(smem + off) = pk;
        }
      };
      {
        float x[H0];
        load(x, 0, H0);
        emit(x, 0, H0);
#pragma unroll
        for (int n = 0; n < H0; ++n) l[n] += x[n];
        load(x, H0, H1);
        emit(x, H0, H1);
#pragma unroll
        for (int n = 0; n < H1; ++n) l[H0 + n] += x[n];
      }
      // V rows of keys past the range may hold anything: zero them
      if (key >= nvalid) {
        if (!mbar_wait(bar(BAR_KV_FULL + st), (t >> 1) & 1)) failed = true;
        uint8_t* vrow = smem + st * kStageBytes + 2 * kBox + key * 128u;
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
      warp_columns<H0, false>(l, red + warp * NH, lane);
      warp_columns<H1, false>(l + H0, red + warp * NH + H0, lane);
      wg_bar(wg);
      for (int n = tid & 127; n < NH; n += 128) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) sum += red[(wg * 4 + w) * NH + n];
        lsum[c0 + n] = sum;
      }
      wg_bar(wg);
      const int d = key;  // O^T lane = output dim
      for (int j = 0; j < NH / 8; ++j) {
        float v[8];
        tmem_ld8(tm_o + lane_off + (uint32_t)(c0 + 8 * j), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = c0 + 8 * j + i;
          if (n >= rows_here) continue;
          const int p = row_base + n;
          const int tr = p / a.g, qh = hk * a.g + p % a.g;
          const float ls = lsum[n];
          const float res = v[i] / ls;
          if (a.nsplit == 1) {
            const long orow = ((long)b * a.R + tr) * a.Hq + qh;
            ((__nv_bfloat16*)a.out)[orow * kD + d] = __float2bfloat16_rn(res);
            if (d == 0) a.lse[orow] = (m_run[n] + log2f(ls)) * 0.69314718055994531f;
          } else {
            const long prow = (((long)b * a.Hq + qh) * a.R + tr) * a.nsplit + sp;
            a.ws_o[prow * kD + d] = res;
            if (d == 0) a.ws_lse[prow] = m_run[n] + log2f(ls);
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

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
  cudaFuncSetAttribute(verify_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const dim3 grid(p.nsplit, a.Hkv * p.nrg, a.B);
  verify_tc_kernel<N><<<grid, kThreadsTC, smem, st>>>(maps, a, p.rb);
}

}  // namespace

bool tc_path_available() { return encode_fn() != nullptr; }

bool launch_tc_path(const tsd_attn_desc& d, const VerifyArgs& a, const VerifyPlan& p,
                    cudaStream_t st) {
  if (d.dk != kD || d.dv != kD || d.v_aliases_k || d.dtype != TSD_BF16) return false;
  if (encode_fn() == nullptr) return false;
  TcMaps maps;
  if (!encode_2d(&maps.k, a.kc, (long)d.B * d.Hkv * d.cap) ||
      !encode_2d(&maps.v, a.vc, (long)d.B * d.Hkv * d.cap) ||
      !encode_3d(&maps.kt, a.kt, d.Hkv, (long)d.B * d.R) ||
      !encode_3d(&maps.vt, a.vt, d.Hkv, (long)d.B * d.R))
    return false;
  switch (p.rb) {
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
    verify_combine_kernel<__nv_bfloat16, 128><<<(unsigned)ceil_div(rows, 4), 128, 0, st>>>(a);
  }
  return true;
}

}  // namespace tsd
