// Tensor-core attention of the DiT head ("GR00T N1.7", action): blocks
// alternate cross-attention of the state + action tokens into the bound VL
// context K/V ([B, S, heads, Dh], boolean visibility mask) and self-attention
// among those tokens (K/V from this step's projection).  Per head, vla.cpp
// Eq. (2): softmax(q K^T / sqrt(d) + M) V, with M = -inf on masked keys; a
// row whose keys are all masked yields 0.
//
// One CTA per (head, sample); its query rows (tokens, <= 32) split over two
// warps of 16.  64-key tiles staged by cp.async in padded shared memory
// (row stride Dh + 8 elements: 8 consecutive rows hit distinct bank groups for
// ldmatrix); mma.sync m16n8k16 bf16 with fp32 online softmax.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace g3 {

namespace {

constexpr int KT = 64;      // keys per tile
constexpr int QROWS = 32;   // query rows per CTA (two warps)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const uint32_t s = ptx::smem_u32(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(pred ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(ptx::smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(ptx::smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int DH>
__global__ void __launch_bounds__(64) attn_dit_kernel(AttnArgs a) {
  constexpr int LD = DH + 8;   // padded row (elements)
  constexpr int CH = DH / 8;   // 16-byte chunks per row
  __shared__ __align__(128) bf16 sQ[QROWS * LD];
  __shared__ __align__(128) bf16 sK[KT * LD];
  __shared__ __align__(128) bf16 sV[KT * LD];
  __shared__ float sMaskNeg[KT];

  ptx::pdl_launch_dependents();
  const int head = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = head / (a.Hq / a.Hkv);
  const bf16* Kp = a.k_slot >= 0 ? (const bf16*)a.table[a.k_slot] : nullptr;
  const bf16* Vp = a.v_slot >= 0 ? (const bf16*)a.table[a.v_slot] : nullptr;
  const uint8_t* mask = a.mask_slot >= 0 ? (const uint8_t*)a.table[a.mask_slot] : nullptr;
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(a.ts);

  // queries: rows t < Tq of (b, head)
  for (int i = tid; i < QROWS * CH; i += 64) {
    const int r = i / CH, c = i % CH;
    const bool ok = r < a.Tq;
    const bf16* src = (const bf16*)a.q + ((long long)b * a.Tq + (ok ? r : 0)) * a.ldq + (long long)head * DH + c * 8;
    cp_async16(sQ + r * LD + c * 8, src, ok);
  }
  cp_async_commit();

  const float sl2 = rsqrtf((float)DH) * 1.4426950408889634f;
  float o[DH / 8][4];
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int g = lane >> 2, tq = lane & 3;
  const int nkeys = a.P + a.S;

  for (int kt = 0; kt < nkeys; kt += KT) {
    __syncthreads();
    for (int i = tid; i < KT * CH; i += 64) {
      const int r = i / CH, c = i % CH;
      const int s = kt + r;
      const bool ok = s < nkeys;
      const bf16 *ks, *vs;
      if (ok && s < a.P) {
        const long long off = (((long long)b * a.P + s) * a.Hkv + kvh) * DH;
        ks = Kp + off;
        vs = Vp + off;
      } else {
        const long long off = ((long long)b * a.Tq + (ok ? s - a.P : 0)) * a.lds + (long long)kvh * DH;
        ks = (const bf16*)a.ks + off;
        vs = (const bf16*)a.vs + off;
      }
      cp_async16(sK + r * LD + c * 8, ok ? (const void*)(ks + c * 8) : a.q, ok);
      cp_async16(sV + r * LD + c * 8, ok ? (const void*)(vs + c * 8) : a.q, ok);
    }
    for (int r = tid; r < KT; r += 64) {
      const int s = kt + r;
      bool vis = s < nkeys;
      if (vis && s < a.P && mask) vis = mask[(long long)b * a.P + s] != 0;
      sMaskNeg[r] = vis ? 0.f : -INFINITY;
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();

    float sacc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
      uint32_t qa[4];
      ldsm_x4(qa, sQ + (warp * 16 + (lane & 15)) * LD + (ks * 2 + (lane >> 4)) * 8);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t kb[4];
        const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = ks * 2 + ((lane >> 3) & 1);
        ldsm_x4(kb, sK + r * LD + c * 8);
        mma16816(sacc[2 * np], qa, kb[0], kb[1]);
        mma16816(sacc[2 * np + 1], qa, kb[2], kb[3]);
      }
    }
    float mnew[2] = {mrow[0], mrow[1]};
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v = sacc[j][e] * sl2 + sMaskNeg[j * 8 + tq * 2 + (e & 1)];
        sacc[j][e] = v;
        mnew[e >> 1] = fmaxf(mnew[e >> 1], v);
      }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mnew[hh] = fmaxf(mnew[hh], __shfl_xor_sync(0xffffffffu, mnew[hh], 1));
      mnew[hh] = fmaxf(mnew[hh], __shfl_xor_sync(0xffffffffu, mnew[hh], 2));
    }
    float corr[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      // a tile whose keys are all masked leaves the running state unchanged
      corr[hh] = mnew[hh] == -INFINITY ? 1.f : exp2f(mrow[hh] - mnew[hh]);
      mrow[hh] = mnew[hh];
      lrow[hh] *= corr[hh];
    }
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) {
      o[i][0] *= corr[0];
      o[i][1] *= corr[0];
      o[i][2] *= corr[1];
      o[i][3] *= corr[1];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float m = mrow[e >> 1];
        const float p = m == -INFINITY ? 0.f : exp2f(sacc[j][e] - m);
        sacc[j][e] = p;
        lrow[e >> 1] += p;
      }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
      pa[1] = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
      pa[2] = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
      pa[3] = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
      for (int dn = 0; dn < DH / 16; ++dn) {
        uint32_t vb[4];
        const int r = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int c = dn * 2 + (lane >> 4);
        ldsm_x4_t(vb, sV + r * LD + c * 8);
        mma16816(o[2 * dn], pa, vb[0], vb[1]);
        mma16816(o[2 * dn + 1], pa, vb[2], vb[3]);
      }
    }
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    lrow[hh] += __shfl_xor_sync(0xffffffffu, lrow[hh], 1);
    lrow[hh] += __shfl_xor_sync(0xffffffffu, lrow[hh], 2);
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int t = warp * 16 + g + 8 * hh;
    if (t >= a.Tq) continue;
    const float inv = lrow[hh] > 0.f ? 1.f / lrow[hh] : 0.f;
    bf16* orow = (bf16*)a.out + ((long long)b * a.Tq + t) * a.ldo + (long long)head * DH;
#pragma unroll
    for (int i = 0; i < DH / 8; ++i)
      *reinterpret_cast<__nv_bfloat162*>(orow + i * 8 + tq * 2) =
          __floats2bfloat162_rn(o[i][2 * hh] * inv, o[i][2 * hh + 1] * inv);
  }
}

}  // namespace

bool attn_dit_supported(const AttnArgs& a) {
  return (a.Dh == 48 || a.Dh == 64) && a.Tq <= QROWS && a.Hkv > 0 && a.Hq % a.Hkv == 0;
}

cudaError_t attention_dit(const AttnArgs& a, cudaStream_t s, bool pdl) {
  if (a.B <= 0 || a.Hq <= 0) return cudaSuccess;
  if (!attn_dit_supported(a)) return cudaErrorInvalidValue;
  const dim3 grid(a.Hq, a.B);
  if (a.Dh == 48) return launch_k(attn_dit_kernel<48>, grid, 64, 0, s, pdl, a);
  return launch_k(attn_dit_kernel<64>, grid, 64, 0, s, pdl, a);
}

}  // namespace g3
