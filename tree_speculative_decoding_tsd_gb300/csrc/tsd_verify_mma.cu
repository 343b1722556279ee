// Tensor-core path of tsd_tree_verify_attn for bf16 GQA heads (dk == dv in
// {64, 128}) with at least 64 packed query rows per KV head.
//
// Same decomposition as the generic path (a CTA takes a group of packed rows
// of one KV head and one prefix split; the request's last split also takes
// the scratch-pad tree rows under the ancestor mask), but the two products
// run on the tensor cores with mma.sync m16n8k16 (bf16 in, fp32 accumulate):
//   S = Q K^T   one warp per 16 packed rows, Q kept in registers
//   O += P V    P re-packed from the S accumulators in registers
// K/V tiles of 64 keys stream through a 3-stage cp.async ring in shared
// memory (16-byte chunks XOR-swizzled by row so ldmatrix is conflict-free);
// keys past the end of the range are zero-filled by the copy itself and
// masked to -inf.  Online softmax in the log2 domain (scale folded into one
// FFMA before exp2).
#include <cuda_bf16.h>

#include "tsd_common.cuh"
#include "tsd_host.h"
#include "tsd_verify.cuh"

namespace tsd {
namespace {

constexpr int kTK = 64;        // keys per tile
constexpr int kStages = 3;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0: write 16 zero bytes, read nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int DK>
__global__ void __launch_bounds__(256)
verify_mma_kernel(const __grid_constant__ VerifyArgs a, int rows_per_cta) {
  grid_dependency_sync();
  constexpr int CH = DK / 8;                 // 16-byte chunks per K/V row
  constexpr int TILE_CHUNKS = kTK * CH;      // uint4 per K (or V) tile
  extern __shared__ __align__(128) uint4 smem[];
  uint4* ks = smem;                           // [stage][kTK][CH] (swizzled)
  uint4* vs = smem + kStages * TILE_CHUNKS;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int sp = blockIdx.x;
  const int hk = blockIdx.y / a.nrg, rg = blockIdx.y % a.nrg;
  const int b = blockIdx.z;
  const int P = min(max(a.plen[b], 0), a.cap);
  const int nsb = P > 0 ? (P + a.split_len - 1) / a.split_len : 1;
  if (sp >= nsb) return;
  const int k0 = sp * a.split_len, k1 = min(P, k0 + a.split_len);
  const int n_pre = k1 > k0 ? (k1 - k0 + kTK - 1) / kTK : 0;
  const int n_tree = (sp == nsb - 1) ? (a.R + kTK - 1) / kTK : 0;
  const int ntiles = n_pre + n_tree;

  const __nv_bfloat16* kc = (const __nv_bfloat16*)a.kc + ((long)b * a.Hkv + hk) * a.cap * DK;
  const __nv_bfloat16* vc = (const __nv_bfloat16*)a.vc + ((long)b * a.Hkv + hk) * a.cap * DK;
  const __nv_bfloat16* kt = (const __nv_bfloat16*)a.kt + ((long)b * a.R * a.Hkv + hk) * DK;
  const __nv_bfloat16* vt = (const __nv_bfloat16*)a.vt + ((long)b * a.R * a.Hkv + hk) * DK;

  auto load_tile = [&](int stage, int t) {
    const __nv_bfloat16 *kb, *vb;
    long stride;
    int nvalid;
    if (t < n_pre) {
      const int key0 = k0 + t * kTK;
      nvalid = min(kTK, k1 - key0);
      kb = kc + (long)key0 * DK;
      vb = vc + (long)key0 * DK;
      stride = DK;
    } else {
      const int j0 = (t - n_pre) * kTK;
      nvalid = min(kTK, a.R - j0);
      kb = kt + (long)j0 * a.Hkv * DK;
      vb = vt + (long)j0 * a.Hkv * DK;
      stride = (long)a.Hkv * DK;
    }
    const uint32_t kdst = smem_u32(ks + stage * TILE_CHUNKS);
    const uint32_t vdst = smem_u32(vs + stage * TILE_CHUNKS);
    for (int idx = tid; idx < TILE_CHUNKS; idx += nthr) {
      const int row = idx / CH, ch = idx - row * CH;
      const bool ok = row < nvalid;
      const long off = (ok ? row * stride : 0) + ch * 8;
      const uint32_t so = (uint32_t)((row * CH + (ch ^ (row & 7))) * 16);
      cp_async16(kdst + so, kb + off, ok);
      cp_async16(vdst + so, vb + off, ok);
    }
  };

  // ---- this warp's 16 packed rows: Q fragments and tree masks ----
  const int g = lane >> 2, tq = lane & 3;
  const int pr0 = rg * rows_per_cta + warp * 16 + g, pr1 = pr0 + 8;
  const bool v0 = pr0 < a.M, v1 = pr1 < a.M;
  const int tr0 = v0 ? pr0 / a.g : 0, tr1 = v1 ? pr1 / a.g : 0;
  const int qh0 = hk * a.g + (v0 ? pr0 % a.g : 0), qh1 = hk * a.g + (v1 ? pr1 % a.g : 0);
  const uint32_t* q0 = (const uint32_t*)((const __nv_bfloat16*)a.q +
                                         (((long)b * a.R + tr0) * a.Hq + qh0) * DK);
  const uint32_t* q1 = (const uint32_t*)((const __nv_bfloat16*)a.q +
                                         (((long)b * a.R + tr1) * a.Hq + qh1) * DK);
  uint32_t qf[DK / 16][4];
#pragma unroll
  for (int kk = 0; kk < DK / 16; ++kk) {
    qf[kk][0] = v0 ? q0[kk * 8 + tq] : 0u;
    qf[kk][1] = v1 ? q1[kk * 8 + tq] : 0u;
    qf[kk][2] = v0 ? q0[kk * 8 + 4 + tq] : 0u;
    qf[kk][3] = v1 ? q1[kk * 8 + 4 + tq] : 0u;
  }
  const uint64_t msk0 = tr0 > 0 ? a.mask[(long)b * a.R + tr0] : 0ull;
  const uint64_t msk1 = tr1 > 0 ? a.mask[(long)b * a.R + tr1] : 0ull;

  float o[DK / 8][4];
#pragma unroll
  for (int j = 0; j < DK / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float c = a.qscale;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) load_tile(s, s);
    cp_async_commit();
  }

  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      const int tn = t + kStages - 1;
      if (tn < ntiles) load_tile(tn % kStages, tn);
      cp_async_commit();
    }
    const int stage = t % kStages;
    const uint32_t kbase = smem_u32(ks + stage * TILE_CHUNKS);
    const uint32_t vbase = smem_u32(vs + stage * TILE_CHUNKS);

    // ---- S = Q K^T (16 x 64) ----
    float s[8][4];
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
    const int mat = lane >> 3, r8 = lane & 7;
#pragma unroll
    for (int kk = 0; kk < DK / 16; ++kk) {
#pragma unroll
      for (int nb = 0; nb < 8; nb += 2) {
        const int key = (nb + (mat >> 1)) * 8 + r8;
        const int ch = 2 * kk + (mat & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + (uint32_t)((key * CH + (ch ^ (key & 7))) * 16), b0, b1, b2, b3);
        mma_bf16(s[nb], qf[kk], b0, b1);
        mma_bf16(s[nb + 1], qf[kk], b2, b3);
      }
    }

    // ---- masks ----
    if (t < n_pre) {
      const int nvalid = min(kTK, k1 - (k0 + t * kTK));
      if (nvalid < kTK) {
#pragma unroll
        for (int nb = 0; nb < 8; ++nb)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (nb * 8 + 2 * tq + (e & 1) >= nvalid) s[nb][e] = -INFINITY;
      }
    } else {
      const int j0 = (t - n_pre) * kTK;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = j0 + nb * 8 + 2 * tq + (e & 1);
          const uint64_t m = (e < 2) ? msk0 : msk1;
          const bool vis = j < a.R && (j == 0 || ((m >> (j - 1)) & 1ull));
          if (!vis) s[nb][e] = -INFINITY;
        }
    }

    // ---- online softmax (log2 domain) ----
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float mx = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) mx = fmaxf(mx, fmaxf(s[nb][2 * i], s[nb][2 * i + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      const float m_new = fmaxf(mrow[i], mx * c);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(mrow[i] - m_use);
      mrow[i] = m_new;
      float sum = 0.f;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) {
        s[nb][2 * i] = exp2f(fmaf(s[nb][2 * i], c, -m_use));
        s[nb][2 * i + 1] = exp2f(fmaf(s[nb][2 * i + 1], c, -m_use));
        sum += s[nb][2 * i] + s[nb][2 * i + 1];
      }
      lrow[i] = fmaf(lrow[i], alpha, sum);
#pragma unroll
      for (int j = 0; j < DK / 8; ++j) {
        o[j][2 * i] *= alpha;
        o[j][2 * i + 1] *= alpha;
      }
    }

    // ---- O += P V ----
#pragma unroll
    for (int kk = 0; kk < kTK / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int jn = 0; jn < DK / 8; jn += 2) {
        const int key = kk * 16 + 8 * (mat & 1) + r8;
        const int ch = jn + (mat >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + (uint32_t)((key * CH + (ch ^ (key & 7))) * 16), b0, b1, b2, b3);
        mma_bf16(o[jn], pa, b0, b1);
        mma_bf16(o[jn + 1], pa, b2, b3);
      }
    }
  }
  cp_async_wait<0>();

  // ---- finalize ----
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    lrow[i] += __shfl_xor_sync(kFull, lrow[i], 1);
    lrow[i] += __shfl_xor_sync(kFull, lrow[i], 2);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool valid = i == 0 ? v0 : v1;
    if (!valid) continue;
    const int tr = i == 0 ? tr0 : tr1, qh = i == 0 ? qh0 : qh1;
    const float inv = 1.f / lrow[i];
    const float lse2 = mrow[i] + log2f(lrow[i]);
    if (nsb == 1) {
      const long orow = ((long)b * a.R + tr) * a.Hq + qh;
      uint32_t* dst = (uint32_t*)((__nv_bfloat16*)a.out + orow * DK);
#pragma unroll
      for (int j = 0; j < DK / 8; ++j)
        dst[j * 4 + tq] = pack_bf16(o[j][2 * i] * inv, o[j][2 * i + 1] * inv);
      if (tq == 0) a.lse[orow] = lse2 * 0.69314718055994531f;
    } else {
      const long prow = (((long)b * a.Hq + qh) * a.R + tr) * a.nsplit + sp;
      float2* dst = (float2*)(a.ws_o + prow * DK);
#pragma unroll
      for (int j = 0; j < DK / 8; ++j)
        dst[j * 4 + tq] = make_float2(o[j][2 * i] * inv, o[j][2 * i + 1] * inv);
      if (tq == 0) a.ws_lse[prow] = lse2;
    }
  }
}

}  // namespace

bool launch_mma_path(const tsd_attn_desc& d, const VerifyArgs& a, const VerifyPlan& p,
                     cudaStream_t st) {
  const dim3 grid(p.nsplit, a.Hkv * p.nrg, a.B);
  const int threads = p.rb / 16 * 32;
  const size_t smem = (size_t)kStages * 2 * kTK * d.dk * 2;
  if (d.dk == 128) {
    cudaFuncSetAttribute(verify_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    launch(verify_mma_kernel<128>, dim3(grid), dim3(threads), smem, st, a, p.rb);
  } else if (d.dk == 64) {
    cudaFuncSetAttribute(verify_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    launch(verify_mma_kernel<64>, dim3(grid), dim3(threads), smem, st, a, p.rb);
  } else {
    return false;
  }
  if (p.nsplit > 1) {
    const long rows = (long)a.B * a.R * a.Hq;
    if (d.dk == 128)
      launch_plain(verify_combine_kernel<__nv_bfloat16, 128>, dim3((unsigned)ceil_div(rows, 4)),
                   dim3(128), 0, st, a);
    else
      launch_plain(verify_combine_kernel<__nv_bfloat16, 64>, dim3((unsigned)ceil_div(rows, 4)),
                   dim3(128), 0, st, a);
  }
  return true;
}

}  // namespace tsd
