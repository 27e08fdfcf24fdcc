// Attention of the DiT head ("GR00T N1.7", action): blocks alternate
// cross-attention of the state + action tokens into the bound VL context K/V
// ([B, S, heads, Dh], boolean visibility mask; text mask when block % 4 == 0,
// image mask otherwise) and self-attention among those tokens (K/V from this
// step's projection).  Per head, vla.cpp Eq. (2): softmax(q K^T / sqrt(d) + M) V
// with M = -inf on masked keys; a row whose keys are all masked yields 0.
//
// One CTA per (head, sample), 9 warps:
//  * warp 8 streams 64-key K and V tiles of the head by TMA (a 3-D tensor map
//    over [B, rows, heads * Dh], box Dh x 64 rows; rows past the keys read as
//    zeros) into a ring of NST slots.  Cross-attention K/V are bound inputs no
//    kernel of the step writes, so the first NST tiles are requested before the
//    programmatic-launch wait; the queries (and self-attention K/V) after it.
//  * warps 0..7 = 2 row groups (16 query rows each) x 4 key groups: key group g
//    takes tiles g, g + 4, ... with mma.sync m16n8k16 and an fp32 online
//    softmax, and frees each slot for the producer.  (17 query rows per head
//    against a head's own K/V fill 1/8 of a 128-row tcgen05 tile, so the
//    warp-level MMA is the right size here.)
//  * the four key groups' partial (max, sum, O) are merged on chip and the
//    normalised rows written out.
// Every mbarrier wait is bounded: a wait that gives up records the error word,
// the CTA drains the copies it issued and returns.
#include <math.h>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace g3 {

namespace {

constexpr int KT = 64;        // keys per tile
constexpr int QROWS = 32;     // query rows per CTA (two row groups of 16)
constexpr int KGROUPS = 4;    // key groups
constexpr int kConsumers = 2 * KGROUPS * 32;
constexpr int kThreads = kConsumers + 32;   // + the TMA producer warp
constexpr long long kDrainPolls = 1LL << 22;

template <int DH>
struct DitSmem {
  static constexpr int NST = DH == 48 ? 6 : 5;        // ring slots (K + V tile each)
  static constexpr int TILE = KT * DH * 2;            // one K or V tile, bf16 rows of DH
  static constexpr int Q_BYTES = QROWS * DH * 2;
  static constexpr int OFF_KV = ((Q_BYTES + 1023) / 1024) * 1024;
  static constexpr int OFF_PART = OFF_KV + NST * 2 * TILE;        // [KGROUPS][QROWS][DH] fp32
  static constexpr int OFF_ML = OFF_PART + KGROUPS * QROWS * DH * 4;   // m, l: [KGROUPS][QROWS] each
  static constexpr int OFF_BAR = OFF_ML + 2 * KGROUPS * QROWS * 4;
  static constexpr int NBAR = 1 + 2 * NST;                         // q_full, full[NST], empty[NST]
  static constexpr int TOTAL = OFF_BAR + NBAR * 8 + 16 + 1024;     // + abort word, alignment slack
};

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(ptx::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(ptx::smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
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

// tmQ: the query columns (cols of the qkv rows, Tq tokens, B samples), box DH x 32 x 1.
// tmK / tmV: cross -- (Hkv * DH, P rows, B) of the bound context; self -- this step's
// K / V columns of the qkv rows.  Box DH x 64 x 1; head kvh at x = kvh * DH.
template <int DH>
__global__ void __launch_bounds__(kThreads, 1)
    attn_dit_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, AttnArgs a, int* err, long long lim) {
  using L = DitSmem<DH>;
  constexpr int NST = L::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  uint8_t* sKV = smem + L::OFF_KV;
  float* part = reinterpret_cast<float*>(smem + L::OFF_PART);
  float* pm = reinterpret_cast<float*>(smem + L::OFF_ML);
  float* pl = pm + KGROUPS * QROWS;
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* full = q_full + 1;
  uint64_t* empty = full + NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NST);

  const int head = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = head / (a.Hq / a.Hkv);
  const bool cross = a.P > 0;
  const int nkeys = cross ? a.P : a.S;
  const int nt = (nkeys + KT - 1) / KT;
  const uint8_t* mask = (cross && a.mask_slot >= 0) ? (const uint8_t*)a.table[a.mask_slot] : nullptr;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int s = 0; s < NST; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 2);   // the two row-group warps of the tile's key group
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::pdl_launch_dependents();
  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(err, 1);
  };

  if (warp == 2 * KGROUPS) {
    // ---------------- producer ----------------
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      auto issue = [&](int t) {
        const int s = t % NST;
        ptx::mbar_arrive_expect_tx(&full[s], 2 * L::TILE);
        tma_load_3d(sKV + s * 2 * L::TILE, &tmK, &full[s], kvh * DH, t * KT, b);
        tma_load_3d(sKV + s * 2 * L::TILE + L::TILE, &tmV, &full[s], kvh * DH, t * KT, b);
      };
      const int first = nt < NST ? nt : NST;
      int issued = 0;
      if (cross)   // bound context K/V: nothing in this step writes them
        for (; issued < first; ++issued) issue(issued);
      ptx::pdl_wait();
      kstamp(a.ts);
      ptx::mbar_arrive_expect_tx(q_full, L::Q_BYTES);
      tma_load_3d(sQ, &tmQ, q_full, head * DH, 0, b);
      for (; issued < first; ++issued) issue(issued);
      for (int t = NST; t < nt; ++t) {
        if (!ptx::mbar_wait(&empty[t % NST], ((t / NST) - 1) & 1, lim)) {
          fail();
          break;
        }
        issue(t);
        issued = t + 1;
      }
      // the CTA may leave early only once every copy it started has landed
      const long long drain = lim > kDrainPolls ? lim : kDrainPolls;
      ptx::mbar_wait(q_full, 0, drain);
      for (int t = issued - 1; t >= 0 && t >= issued - NST; --t) ptx::mbar_wait(&full[t % NST], (t / NST) & 1, drain);
    }
  } else {
    // ---------------- consumers: row group rg, key group kg ----------------
    const int rg = warp & 1, kg = warp >> 1;
    const int g = lane >> 2, tq = lane & 3;
    const float sl2 = rsqrtf((float)DH) * 1.4426950408889634f;
    float o[DH / 8][4];
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    const bool ok = ptx::mbar_wait(q_full, 0, lim);
    if (!ok) fail();
    uint32_t qa[DH / 16][4];
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
      qa[ks][0] = qa[ks][1] = qa[ks][2] = qa[ks][3] = 0u;
      if (ok) ldsm_x4(qa[ks], sQ + (rg * 16 + (lane & 15)) * DH + (ks * 2 + (lane >> 4)) * 8);
    }
    for (int t = kg; ok && t < nt; t += KGROUPS) {
      const int s = t % NST;
      if (!ptx::mbar_wait(&full[s], (t / NST) & 1, lim) || *abort_flag) {
        fail();
        break;
      }
      const bf16* sK = reinterpret_cast<const bf16*>(sKV + s * 2 * L::TILE);
      const bf16* sV = sK + KT * DH;
      // additive mask of this lane's 16 key columns: j * 8 + tq * 2 + {0, 1}
      float neg[8][2];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = t * KT + j * 8 + tq * 2 + e;
          bool vis = key < nkeys;
          if (vis && mask) vis = mask[(long long)b * a.P + key] != 0;
          neg[j][e] = vis ? 0.f : -INFINITY;
        }
      float sacc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t kb[4];
          const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int c = ks * 2 + ((lane >> 3) & 1);
          ldsm_x4(kb, sK + r * DH + c * 8);
          mma16816(sacc[2 * np], qa[ks], kb[0], kb[1]);
          mma16816(sacc[2 * np + 1], qa[ks], kb[2], kb[3]);
        }
      }
      float mnew[2] = {mrow[0], mrow[1]};
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v = sacc[j][e] * sl2 + neg[j][e & 1];
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
          ldsm_x4_t(vb, sV + r * DH + c * 8);
          mma16816(o[2 * dn], pa, vb[0], vb[1]);
          mma16816(o[2 * dn + 1], pa, vb[2], vb[3]);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[s]);
    }
    // this key group's partial rows: unnormalised O, running max and sum
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      lrow[hh] += __shfl_xor_sync(0xffffffffu, lrow[hh], 1);
      lrow[hh] += __shfl_xor_sync(0xffffffffu, lrow[hh], 2);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = rg * 16 + g + 8 * hh;
      float* prow = part + (kg * QROWS + r) * DH;
#pragma unroll
      for (int i = 0; i < DH / 8; ++i)
        *reinterpret_cast<float2*>(prow + i * 8 + tq * 2) = make_float2(o[i][2 * hh], o[i][2 * hh + 1]);
      if (tq == 0) {
        pm[kg * QROWS + r] = mrow[hh];
        pl[kg * QROWS + r] = lrow[hh];
      }
    }
  }
  __syncthreads();
  if (*abort_flag || threadIdx.x >= kConsumers) return;
  // merge the key groups: row r = tid / 8, DH / 8 columns per thread
  constexpr int CPT = DH / 8;
  const int r = threadIdx.x >> 3, c0 = (threadIdx.x & 7) * CPT;
  if (r >= a.Tq) return;
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < KGROUPS; ++k) M = fmaxf(M, pm[k * QROWS + r]);
  float w[KGROUPS], Lsum = 0.f;
#pragma unroll
  for (int k = 0; k < KGROUPS; ++k) {
    const float mk = pm[k * QROWS + r];
    w[k] = mk == -INFINITY ? 0.f : exp2f(mk - M);
    Lsum += w[k] * pl[k * QROWS + r];
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;   // every key masked: the row is 0
  bf16* orow = (bf16*)a.out + ((long long)b * a.Tq + r) * a.ldo + (long long)head * DH + c0;
#pragma unroll
  for (int c = 0; c < CPT; c += 2) {
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int k = 0; k < KGROUPS; ++k) {
      const float2 pv = *reinterpret_cast<const float2*>(part + (k * QROWS + r) * DH + c0 + c);
      v0 = fmaf(w[k], pv.x, v0);
      v1 = fmaf(w[k], pv.y, v1);
    }
    *reinterpret_cast<__nv_bfloat162*>(orow + c) = __floats2bfloat162_rn(v0 * inv, v1 * inv);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode_dit = nullptr;

// 3-D bf16 map (cols, rows, samples) with the given strides (bytes), box (dh, box_rows, 1), no swizzle.
cudaError_t map3(CUtensorMap* m, const void* base, long long cols, long long rows, long long samples,
                 long long row_stride, long long sample_stride, int dh, int box_rows) {
  if (!g_encode_dit) {
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&g_encode_dit, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !g_encode_dit) return cudaErrorNotSupported;
  }
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)samples};
  const cuuint64_t strides[2] = {(cuuint64_t)row_stride, (cuuint64_t)sample_stride};
  const cuuint32_t box[3] = {(cuuint32_t)dh, (cuuint32_t)box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode_dit(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int DH>
cudaError_t launch_dit(const CUtensorMap* maps, const AttnArgs& a, int* err, long long lim, cudaStream_t s,
                       bool pdl) {
  using L = DitSmem<DH>;
  static_assert(L::TOTAL <= 232448, "shared memory of the DiT attention");
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_dit_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_k(attn_dit_kernel<DH>, dim3(a.Hq, a.B), dim3(kThreads), L::TOTAL, s, pdl, maps[0], maps[1], maps[2],
                  a, err, lim);
}

}  // namespace

bool attn_dit_supported(const AttnArgs& a, const void* kp, const void* vp) {
  if (!((a.Dh == 48 || a.Dh == 64) && a.Tq >= 1 && a.Tq <= QROWS && a.Hkv > 0 && a.Hq % a.Hkv == 0)) return false;
  // one key source: the bound context (cross) or this step's tokens (self, at most one tile)
  const bool cross = a.P > 0 && a.S == 0 && kp && vp;
  const bool self = a.P == 0 && a.S >= 1 && a.S <= KT && a.ks && a.vs && a.S == a.Tq;
  if (!cross && !self) return false;
  // TMA: 16-byte aligned bases and strides
  auto al = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  if (!al(a.q) || (a.ldq * 2) % 16 || (a.Dh * 2) % 16) return false;
  if (cross && (!al(kp) || !al(vp) || (a.Hkv * a.Dh * 2) % 16)) return false;
  if (self && (!al(a.ks) || !al(a.vs) || (a.lds * 2) % 16)) return false;
  return true;
}

cudaError_t attention_dit(const AttnArgs& a, const void* kp, const void* vp, int* err, long long wait_limit,
                          cudaStream_t s, bool pdl) {
  if (a.B <= 0 || a.Hq <= 0) return cudaSuccess;
  if (!attn_dit_supported(a, kp, vp)) return cudaErrorInvalidValue;
  const int D = a.Dh;
  const long long hd = (long long)a.Hkv * D;   // the K (or V) columns of all heads
  CUtensorMap maps[3];
  cudaError_t e = map3(&maps[0], a.q, a.ldq, a.Tq, a.B, (long long)a.ldq * 2, (long long)a.Tq * a.ldq * 2, D, QROWS);
  if (e != cudaSuccess) return e;
  if (a.P > 0) {   // the bound context [B, P, Hkv, Dh]
    e = map3(&maps[1], kp, hd, a.P, a.B, hd * 2, (long long)a.P * hd * 2, D, KT);
    if (e == cudaSuccess) e = map3(&maps[2], vp, hd, a.P, a.B, hd * 2, (long long)a.P * hd * 2, D, KT);
  } else {         // this step's keys / values: hd columns of the projection rows (row stride lds)
    e = map3(&maps[1], a.ks, hd, a.S, a.B, (long long)a.lds * 2, (long long)a.Tq * a.lds * 2, D, KT);
    if (e == cudaSuccess)
      e = map3(&maps[2], a.vs, hd, a.S, a.B, (long long)a.lds * 2, (long long)a.Tq * a.lds * 2, D, KT);
  }
  if (e != cudaSuccess) return e;
  if (D == 48) return launch_dit<48>(maps, a, err, wait_limit, s, pdl);
  return launch_dit<64>(maps, a, err, wait_limit, s, pdl);
}

}  // namespace g3
