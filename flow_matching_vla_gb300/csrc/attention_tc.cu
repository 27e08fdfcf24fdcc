// Tensor-core attention of the action expert over prefix ++ own K/V.
//
// "pi0.5 Design", Attention and the K/V pool: the expert has one K/V head,
// so its Hq query heads fold into the row axis -- for sample b, query row
// r = t * Hq + h (token t, head h) -- and every row attends the same keys:
// the bound prefix K/V (P rows) followed by the H action tokens' own K/V
// computed this step.  The fold is exact because the mask is all ones.
// Attention per row is vla.cpp Eq. (2): softmax(q K^T / sqrt(d)) V.
//
// Flash-decoding over keys: grid (row tiles of 64, S key splits, B); the S
// CTAs of one row tile form a thread-block cluster.  Each CTA runs an online
// softmax over its key range with mma.sync m16n8k16 (bf16 in, fp32
// accumulate): 4 warps x 16 rows, 64-key sub-tiles staged in XOR-swizzled
// shared memory by cp.async.  The S partial (max, sum, O) triples are then
// combined through distributed shared memory, in split order (deterministic),
// each CTA finishing 64/S rows.
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace g3 {

namespace cg = cooperative_groups;

namespace {

constexpr int ROWS = 64;   // query rows per CTA (4 warps x 16)
constexpr int KT = 64;     // keys per sub-tile

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const uint32_t s = ptx::smem_u32(smem);
  const int n = pred ? 16 : 0;  // src-size 0: zero-fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
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

// Row r of a [rows][DH] bf16 tile, 16-byte chunk c, XOR-swizzled by r % 8.
template <int DH>
__device__ __forceinline__ int swz(int r, int c) {
  return r * DH + ((c ^ (r & 7)) << 3);
}

template <int DH>
struct AttnSmem {
  static constexpr int TILE = ROWS * DH * 2;   // Q, K or V tile (64 rows)
  static constexpr int OPART = ROWS * DH * 4;  // fp32 partial O
  // tiles | sM, sL (read by peers) | local combine scratch (weights, sums, 1/sum)
  static constexpr int TOTAL = 3 * TILE + 2 * ROWS * 4 + 3 * ROWS * 4 + 16;
  static_assert(OPART + 2 * ROWS * 4 <= 3 * TILE + 2 * ROWS * 4, "partial fits");
};

template <int DH>
__global__ void __launch_bounds__(128) attn_fold_kernel(AttnFoldArgs a) {
  using L = AttnSmem<DH>;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = reinterpret_cast<bf16*>(smem + L::TILE);
  bf16* sV = reinterpret_cast<bf16*>(smem + 2 * L::TILE);
  float* sO = reinterpret_cast<float*>(smem);                       // after the key loop
  float* sM = reinterpret_cast<float*>(smem + 3 * L::TILE);
  float* sL = sM + ROWS;

  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int split = (int)cluster.block_rank();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z;
  const int r0 = blockIdx.x * ROWS;
  const int nrows = a.Hq * a.H;
  const int nkeys = a.P + a.H;
  const int chunk = ((nkeys + S - 1) / S + KT - 1) / KT * KT;
  const int k_begin = split * chunk;
  const int k_end = min(nkeys, k_begin + chunk);
  constexpr int CH = DH / 8;  // 16-byte chunks per row

  ptx::pdl_launch_dependents();
  ptx::pdl_wait();

  const bf16* Kp = reinterpret_cast<const bf16*>(a.table[a.k_slot]);
  const bf16* Vp = reinterpret_cast<const bf16*>(a.table[a.v_slot]);
  const bf16* qkv = reinterpret_cast<const bf16*>(a.qkv);

  // Q tile: folded row r = t * Hq + h -> qkv[(b*H + t) * ldq + h * DH]
  for (int i = tid; i < ROWS * CH; i += 128) {
    const int r = i / CH, c = i % CH;
    const int gr = r0 + r;
    const bool ok = gr < nrows;
    const int t = ok ? gr / a.Hq : 0, h = ok ? gr % a.Hq : 0;
    const bf16* src = qkv + ((long long)b * a.H + t) * a.ldq + h * DH + c * 8;
    cp_async16(sQ + swz<DH>(r, c), src, ok);
  }
  cp_async_commit();

  const float sl2 = rsqrtf((float)DH) * 1.4426950408889634f;  // 1/sqrt(d) * log2(e)
  float o[DH / 8][4];
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int g = lane >> 2, tq = lane & 3;

  for (int kt = k_begin; kt < k_end; kt += KT) {
    __syncthreads();  // previous sub-tile fully consumed
    for (int i = tid; i < KT * CH; i += 128) {
      const int r = i / CH, c = i % CH;
      const int s = kt + r;
      const bool ok = s < k_end;
      const bf16 *ks, *vs;
      if (s < a.P) {
        ks = Kp + ((long long)b * a.P + s) * DH;
        vs = Vp + ((long long)b * a.P + s) * DH;
      } else {
        const long long row = (long long)b * a.H + (ok ? s - a.P : 0);
        ks = qkv + row * a.ldq + a.k_off;
        vs = qkv + row * a.ldq + a.v_off;
      }
      cp_async16(sK + swz<DH>(r, c), ok ? (const void*)(ks + c * 8) : (const void*)qkv, ok);
      cp_async16(sV + swz<DH>(r, c), ok ? (const void*)(vs + c * 8) : (const void*)qkv, ok);
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();

    // S = Q K^T for this warp's 16 rows x 64 keys
    float sacc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
      uint32_t qa[4];
      {
        const int r = warp * 16 + (lane & 15);
        const int c = ks * 2 + (lane >> 4);
        ldsm_x4(qa, sQ + swz<DH>(r, c));
      }
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t kb[4];
        const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = ks * 2 + ((lane >> 3) & 1);
        ldsm_x4(kb, sK + swz<DH>(r, c));
        mma16816(sacc[2 * np], qa, kb[0], kb[1]);
        mma16816(sacc[2 * np + 1], qa, kb[2], kb[3]);
      }
    }
    // online softmax (rows g and g + 8 of the warp tile); keys past k_end are masked
    float mnew[2] = {mrow[0], mrow[1]};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kt + j * 8 + tq * 2 + (e & 1);
        const float v = key < k_end ? sacc[j][e] * sl2 : -INFINITY;
        sacc[j][e] = v;
        mnew[e >> 1] = fmaxf(mnew[e >> 1], v);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mnew[h] = fmaxf(mnew[h], __shfl_xor_sync(0xffffffffu, mnew[h], 1));
      mnew[h] = fmaxf(mnew[h], __shfl_xor_sync(0xffffffffu, mnew[h], 2));
    }
    float corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      corr[h] = exp2f(mrow[h] - mnew[h]);  // mrow = -inf on the first tile: 0
      mrow[h] = mnew[h];
      lrow[h] *= corr[h];
    }
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) {
      o[i][0] *= corr[0];
      o[i][1] *= corr[0];
      o[i][2] *= corr[1];
      o[i][3] *= corr[1];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = exp2f(sacc[j][e] - mrow[e >> 1]);
        sacc[j][e] = p;
        lrow[e >> 1] += p;
      }
    }
    // O += P V  (P from the S accumulators, 16 keys per k-step)
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
        ldsm_x4_t(vb, sV + swz<DH>(r, c));
        mma16816(o[2 * dn], pa, vb[0], vb[1]);
        mma16816(o[2 * dn + 1], pa, vb[2], vb[3]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
  }
  __syncthreads();  // tiles no longer read: reuse them for the partial
  {
    const int ra = warp * 16 + g, rb = ra + 8;
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) {
      const int col = i * 8 + tq * 2;
      *reinterpret_cast<float2*>(sO + ra * DH + col) = make_float2(o[i][0], o[i][1]);
      *reinterpret_cast<float2*>(sO + rb * DH + col) = make_float2(o[i][2], o[i][3]);
    }
    if (tq == 0) {
      sM[ra] = mrow[0];
      sM[rb] = mrow[1];
      sL[ra] = lrow[0];
      sL[rb] = lrow[1];
    }
  }
  cluster.sync();

  // combine: this CTA finishes rows [split*RP, split*RP + RP) of the tile.
  // (1) per row and split, the split's running max and sum -> weights
  const int RP = ROWS / S;
  float* sW = sL + ROWS;       // [S][RP]: split maxima, then weights exp2(m_s - max)  (local)
  float* sLs = sW + ROWS;      // [S][RP]: split sums                                 (local)
  float* sInv = sLs + ROWS;    // [RP]: 1 / sum_s w_s l_s                             (local)
  if (tid < S * RP) {
    const int s = tid / RP, rr = split * RP + tid % RP;
    sW[tid] = cluster.map_shared_rank(sM, s)[rr];
    sLs[tid] = cluster.map_shared_rank(sL, s)[rr];
  }
  __syncthreads();
  if (tid < RP) {
    float mx = -INFINITY;
    for (int s = 0; s < S; ++s) mx = fmaxf(mx, sW[s * RP + tid]);
    float lsum = 0.f;
    for (int s = 0; s < S; ++s) {
      const float ms = sW[s * RP + tid];
      const float w = ms == -INFINITY ? 0.f : exp2f(ms - mx);
      lsum += w * sLs[s * RP + tid];
      sW[s * RP + tid] = w;
    }
    sInv[tid] = lsum > 0.f ? 1.f / lsum : 0.f;
  }
  __syncthreads();
  // (2) weighted sum of the S partial O rows, loads issued together, summed in split order
  bf16* out = reinterpret_cast<bf16*>(a.out);
  for (int i = tid; i < RP * (DH / 2); i += 128) {
    const int lr = i / (DH / 2);
    const int rr = split * RP + lr;
    const int col = (i % (DH / 2)) * 2;
    const int gr = r0 + rr;
    if (gr >= nrows) continue;
    float2 v[16];
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < S) v[s] = *reinterpret_cast<const float2*>(cluster.map_shared_rank(sO, s) + rr * DH + col);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < S) {
        const float w = sW[s * RP + lr];
        acc0 += w * v[s].x;
        acc1 += w * v[s].y;
      }
    const float inv = sInv[lr];
    const int t = gr / a.Hq, h = gr % a.Hq;
    *reinterpret_cast<__nv_bfloat162*>(out + ((long long)b * a.H + t) * a.ldo + h * DH + col) =
        __floats2bfloat162_rn(acc0 * inv, acc1 * inv);
  }
  cluster.sync();
}

template <int DH>
cudaError_t launch_fold(const AttnFoldArgs& a, int S, cudaStream_t s, bool pdl) {
  using L = AttnSmem<DH>;
  auto kern = attn_fold_kernel<DH>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.Hq * a.H + ROWS - 1) / ROWS, S, a.B);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = L::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = S;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

int attn_fold_splits(const AttnFoldArgs& a, int sm_count) {
  const int tiles = (a.Hq * a.H + ROWS - 1) / ROWS * a.B;
  const int nkeys = a.P + a.H;
  int S = 1;
  while (S < 16 && tiles * S * 2 <= 2 * sm_count && (nkeys + 2 * S - 1) / (2 * S) >= KT) S *= 2;
  return S;
}

bool attn_fold_supported(int Dh) { return Dh == 64 || Dh == 128 || Dh == 256; }

cudaError_t attention_fold(const AttnFoldArgs& a, int S, cudaStream_t s, bool pdl) {
  if (a.B <= 0 || a.Hq * a.H <= 0) return cudaSuccess;
  if (S < 1 || S > 16 || (S & (S - 1))) return cudaErrorInvalidValue;
  switch (a.Dh) {
    case 64: return launch_fold<64>(a, S, s, pdl);
    case 128: return launch_fold<128>(a, S, s, pdl);
    case 256: return launch_fold<256>(a, S, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace g3
