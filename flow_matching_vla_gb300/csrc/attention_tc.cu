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
// shared memory by cp.async (the bound prefix rows before the dependency
// wait).  The S partial (max, sum, O) triples go to an L2-resident workspace;
// after one cluster barrier each CTA combines 64/S rows in split order
// (deterministic).  With S = 1 the CTA normalises and stores directly.
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

constexpr int RING = 3;    // resident K/V sub-tile buffers

template <int DH>
struct AttnSmem {
  static constexpr int TILE = ROWS * DH * 2;   // Q, K or V tile (64 rows)
  // Q | RING x (K, V) | combine scratch (weights, sums, 1/sum)
  static constexpr int TOTAL = (1 + 2 * RING) * TILE + 3 * ROWS * 4 + 16;
};

__device__ __forceinline__ void cp_async_wait_upto(int n) {  // at most n newer groups pending
  if (n <= 0)
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  else if (n == 1)
    asm volatile("cp.async.wait_group 1;" ::: "memory");
  else
    asm volatile("cp.async.wait_group 2;" ::: "memory");
}

template <int DH>
__global__ void __launch_bounds__(128) attn_fold_kernel(AttnFoldArgs a) {
  using L = AttnSmem<DH>;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  // K/V sub-tile buffer i: K at smem + (1 + 2i) TILE, V right after it
  auto sK = [&](int i) { return reinterpret_cast<bf16*>(smem + (1 + 2 * i) * L::TILE); };
  auto sV = [&](int i) { return reinterpret_cast<bf16*>(smem + (2 + 2 * i) * L::TILE); };
  float* sW = reinterpret_cast<float*>(smem + (1 + 2 * RING) * L::TILE);   // combine scratch [S][RP]
  float* sLs = sW + ROWS;
  float* sInv = sLs + ROWS;

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
  // The bound prefix K/V and the pointer table are never written inside the
  // loop: stage the prefix rows of the first RING sub-tiles before waiting on
  // the kernel that produces this step's Q and suffix K/V.
  const bf16* Kp = reinterpret_cast<const bf16*>(a.table[a.k_slot]);
  const bf16* Vp = reinterpret_cast<const bf16*>(a.table[a.v_slot]);
  const bf16* qkv = reinterpret_cast<const bf16*>(a.qkv);
  // phase 0: prefix rows only, 1: suffix and out-of-range rows only, 2: all rows
  auto issue_kv = [&](int kt, int phase, int buf) {
    for (int i = tid; i < KT * CH; i += 128) {
      const int r = i / CH, c = i % CH;
      const int s = kt + r;
      const bool pre = s < a.P && s < k_end;
      if ((phase == 0 && !pre) || (phase == 1 && pre)) continue;
      const bool ok = s < k_end;
      const bf16 *ks, *vs;
      if (pre) {
        ks = Kp + ((long long)b * a.P + s) * DH;
        vs = Vp + ((long long)b * a.P + s) * DH;
      } else {
        const long long row = (long long)b * a.H + (ok ? s - a.P : 0);
        ks = qkv + row * a.ldq + a.k_off;
        vs = qkv + row * a.ldq + a.v_off;
      }
      cp_async16(sK(buf) + swz<DH>(r, c), ok ? (const void*)(ks + c * 8) : (const void*)qkv, ok);
      cp_async16(sV(buf) + swz<DH>(r, c), ok ? (const void*)(vs + c * 8) : (const void*)qkv, ok);
    }
  };
  const int nsub = (k_end - k_begin + KT - 1) / KT;   // 0 when the split is empty
  const int first = nsub < RING ? nsub : RING;
  for (int i = 0; i < first; ++i) issue_kv(k_begin + i * KT, 0, i);
  ptx::pdl_wait();
  if (tid == 0) kstamp(a.ts);

  // Q tile: folded row r = t * Hq + h -> qkv[(b*H + t) * ldq + h * DH]
  for (int i = tid; i < ROWS * CH; i += 128) {
    const int r = i / CH, c = i % CH;
    const int gr = r0 + r;
    const bool ok = gr < nrows;
    const int t = ok ? gr / a.Hq : 0, h = ok ? gr % a.Hq : 0;
    const bf16* src = qkv + ((long long)b * a.H + t) * a.ldq + h * DH + c * 8;
    cp_async16(sQ + swz<DH>(r, c), src, ok);
  }
  for (int i = 0; i < first; ++i) issue_kv(k_begin + i * KT, 1, i);
  cp_async_commit();

  const float sl2 = rsqrtf((float)DH) * 1.4426950408889634f;  // 1/sqrt(d) * log2(e)
  float o[DH / 8][4];
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int g = lane >> 2, tq = lane & 3;

  for (int it = 0; it < nsub; ++it) {
    const int kt = k_begin + it * KT;
    const int buf = it % RING;
    // sub-tile `it` landed: the first RING arrived with Q; a later one was the
    // refill group issued RING iterations ago, newer refills may stay pending
    if (it == 0)
      cp_async_wait_all();
    else if (it >= RING)
      cp_async_wait_upto(min(RING - 1, nsub - 1 - it));
    __syncthreads();
    const bf16* cK = sK(buf);
    const bf16* cV = sV(buf);
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
        ldsm_x4(kb, cK + swz<DH>(r, c));
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
        ldsm_x4_t(vb, cV + swz<DH>(r, c));
        mma16816(o[2 * dn], pa, vb[0], vb[1]);
        mma16816(o[2 * dn + 1], pa, vb[2], vb[3]);
      }
    }
    if (it + RING < nsub) {  // buffer `buf` fully consumed by every warp: refill it
      __syncthreads();
      issue_kv(k_begin + (it + RING) * KT, 2, buf);
      cp_async_commit();
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
  }
  const int ra = warp * 16 + g, rb = ra + 8;
  bf16* out = reinterpret_cast<bf16*>(a.out);

  if (S == 1) {  // whole key range in this CTA: normalise and store
    const float inva = lrow[0] > 0.f ? 1.f / lrow[0] : 0.f;
    const float invb = lrow[1] > 0.f ? 1.f / lrow[1] : 0.f;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int gr = r0 + (hr ? rb : ra);
      if (gr >= nrows) continue;
      const int t = gr / a.Hq, h = gr % a.Hq;
      bf16* orow = out + ((long long)b * a.H + t) * a.ldo + h * DH;
      const float inv = hr ? invb : inva;
#pragma unroll
      for (int i = 0; i < DH / 8; ++i)
        *reinterpret_cast<__nv_bfloat162*>(orow + i * 8 + tq * 2) =
            __floats2bfloat162_rn(o[i][2 * hr] * inv, o[i][2 * hr + 1] * inv);
    }
    return;
  }

  // split keys: park (O, max, sum) in the L2-resident workspace, one cluster
  // barrier, then this CTA combines rows [split*RP, split*RP + RP) in split order
  const long long tile = (long long)b * gridDim.x + blockIdx.x;
  constexpr int PART = ROWS * DH + 2 * ROWS;   // floats per split partial
  float* my = a.ws + (tile * S + split) * PART;
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) {
    const int col = i * 8 + tq * 2;
    *reinterpret_cast<float2*>(my + ra * DH + col) = make_float2(o[i][0], o[i][1]);
    *reinterpret_cast<float2*>(my + rb * DH + col) = make_float2(o[i][2], o[i][3]);
  }
  if (tq == 0) {
    my[ROWS * DH + ra] = mrow[0];
    my[ROWS * DH + rb] = mrow[1];
    my[ROWS * DH + ROWS + ra] = lrow[0];
    my[ROWS * DH + ROWS + rb] = lrow[1];
  }
  cluster.sync();

  const float* base = a.ws + tile * S * PART;
  const int RP = ROWS / S;
  if (tid < S * RP) {  // (1) per row and split: max and sum -> weights
    const int sp = tid / RP, rr = split * RP + tid % RP;
    sW[tid] = base[sp * PART + ROWS * DH + rr];
    sLs[tid] = base[sp * PART + ROWS * DH + ROWS + rr];
  }
  __syncthreads();
  if (tid < RP) {
    float mx = -INFINITY;
    for (int sp = 0; sp < S; ++sp) mx = fmaxf(mx, sW[sp * RP + tid]);
    float lsum = 0.f;
    for (int sp = 0; sp < S; ++sp) {
      const float ms = sW[sp * RP + tid];
      const float w = ms == -INFINITY ? 0.f : exp2f(ms - mx);
      lsum += w * sLs[sp * RP + tid];
      sW[sp * RP + tid] = w;
    }
    sInv[tid] = lsum > 0.f ? 1.f / lsum : 0.f;
  }
  __syncthreads();
  // (2) weighted sum of the S partial rows; U items per thread with their loads in flight together
  constexpr int U = 4;
  const int items = RP * (DH / 2);
#pragma unroll 1
  for (int it0 = tid; it0 < items; it0 += 128 * U) {
    float2 acc[U];
    int lr[U], col[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int it = it0 + u * 128;
      lr[u] = it / (DH / 2);
      col[u] = (it % (DH / 2)) * 2;
      ok[u] = it < items && r0 + split * RP + lr[u] < nrows;
      acc[u] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int sp = 0; sp < 16; ++sp) {
      if (sp < S) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (ok[u]) {
            const float w = sW[sp * RP + lr[u]];
            const float2 v = *reinterpret_cast<const float2*>(base + sp * PART + (split * RP + lr[u]) * DH + col[u]);
            acc[u].x += w * v.x;
            acc[u].y += w * v.y;
          }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (ok[u]) {
        const int gr = r0 + split * RP + lr[u];
        const int t = gr / a.Hq, h = gr % a.Hq;
        const float inv = sInv[lr[u]];
        *reinterpret_cast<__nv_bfloat162*>(out + ((long long)b * a.H + t) * a.ldo + h * DH + col[u]) =
            __floats2bfloat162_rn(acc[u].x * inv, acc[u].y * inv);
      }
  }
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

long long attn_fold_workspace_floats(const AttnFoldArgs& a, int S) {
  if (S == 1) return 0;
  const long long tiles = (long long)(a.Hq * a.H + ROWS - 1) / ROWS * a.B;
  return tiles * S * (ROWS * (long long)a.Dh + 2 * ROWS);
}

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
  if (attn_fold_workspace_floats(a, S) > a.ws_floats) return cudaErrorInvalidValue;
  switch (a.Dh) {
    case 64: return launch_fold<64>(a, S, s, pdl);
    case 128: return launch_fold<128>(a, S, s, pdl);
    case 256: return launch_fold<256>(a, S, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace g3
