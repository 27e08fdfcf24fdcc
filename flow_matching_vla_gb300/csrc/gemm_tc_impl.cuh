// Tensor-core GEMM for the denoise step: Y[M, N] = X[M, K] W[N, K]^T, bf16 in,
// fp32 accumulate in tensor memory (tcgen05.mma, kind::f16), fused epilogues.
//
// Shapes are weight-streaming: N (weight rows) is large, M (token rows) is
// 17..1600.  The weight therefore plays the MMA's M role ("swap-AB"): each
// CTA owns 128 weight rows and BN tokens, D[128, BN] lives in TMEM.
//
//  * TMA (cp.async.bulk.tensor, 128-byte swizzle) streams 128x64 weight tiles
//    (L2 evict-first) and BNx64 activation tiles (L2 evict-last) through a
//    STAGES-deep mbarrier ring; one thread issues loads, one issues MMAs.
//  * Split-K across a thread-block cluster (1 x 1 x S): for 64/128-token tiles
//    each CTA parks its fp32 partial in its idle pipeline memory and hands every
//    peer the 128/S rows that peer reduces with one shared-to-peer bulk copy;
//    256-token tiles go through an L2-resident workspace; either way the S
//    partials are summed in rank order (deterministic).  Residual GEMMs may
//    instead leave their partials for the next norm kernel (EPI_PARTIAL).
//    Without a split the epilogue runs straight from the TMEM registers
//    (adjacent lanes swap one value to form output pairs).
//  * E4M3 weights (WF_E4M3): code tiles are widened into bf16 A tiles held in
//    tensor memory; the row scales finish the accumulator in the epilogue.
//  * Programmatic dependent launch: weight tiles (which no earlier kernel
//    writes) are prefetched before griddepcontrol.wait; activations after.
//  * Every mbarrier wait is bounded; on timeout the CTA records an error
//    flag for the host, drains its own in-flight copies and exits normally.
#pragma once
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "epilogue.cuh"
#include "gemm_tc.h"
#include "tc_ptx.cuh"

namespace g3 {

namespace cg = cooperative_groups;

namespace {

constexpr int BM = 128;  // weight rows per CTA (MMA M)
constexpr int BK = 64;   // K elements per stage: one 128-byte swizzle row of bf16
constexpr int A_BYTES = BM * BK * 2;

// Weight paths (WF): WF_SMEM -- bf16 weight tiles stay in shared memory and the
// MMA reads A from there.  WF_E4M3 -- E4M3 weights with A in TENSOR memory: the
// producer streams 128 x 128-byte code tiles (128 K elements) into a 2-slot ring,
// four warps widen them exactly to bf16 into the stage's A tile in tensor memory
// (lane = weight row, 32-bit column j = K elements 2j, 2j+1), and the MMA reads A
// from there, so after the dependency wait shared memory only feeds the
// activations to the tensor core (an MMA with N = 64 reading both operands from
// shared memory is bound by that: ~48 cycles measured).  The same tensor-memory A
// for bf16 weights (a plain copy instead of the widening) measured slower at
// batch 1 than WF_SMEM: it doubles the bytes moved through the ring.
constexpr int WF_SMEM = 0, WF_E4M3 = 1;

template <int BN, int STAGES, int WF = WF_SMEM>
struct TcSmem {
  static constexpr bool F8 = WF == WF_E4M3, TA = WF != WF_SMEM;
  static constexpr int BKX = F8 ? 2 * BK : BK;    // K elements per stage
  static constexpr int A_STAGE = TA ? 0 : BM * BKX * 2;   // bf16 A tile of a stage in shared memory
  static constexpr int A_COLS = BKX / 2;          // TA: tensor-memory columns of one stage's A tile
  static constexpr int TMEM_NEED = BN + (TA ? STAGES * A_COLS : 0);
  static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128
                                 : TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int B_BYTES = BN * BKX * 2;
  static constexpr int STAGE_BYTES = A_STAGE + B_BYTES;
  static constexpr int PIPE = STAGES * STAGE_BYTES;
  static constexpr int RAW = TA ? 2 : 0;          // E4M3 code tiles in flight to tensor memory
  static constexpr int RAW_BYTES = BM * 128;
  static constexpr int BAR_OFF = PIPE + RAW * RAW_BYTES;
  static constexpr int NBAR = 2 * STAGES + 2 + (TA ? STAGES + 2 * RAW : 0);
  static constexpr int BAR = NBAR * 8 + 16;
  static constexpr int TOTAL = BAR_OFF + BAR + 1024;  // + alignment slack
  // split-K reduced on chip: the idle pipeline holds this CTA's fp32 partial
  // tile and the row slices its peers send it (one tile's worth)
  static constexpr int PART_BYTES = BN * BM * 4;
  static constexpr bool ONCHIP = 2 * PART_BYTES <= PIPE;
};

// Bulk copy of ``bytes`` (multiple of 16, 16-byte aligned) from this CTA's shared
// memory into a peer's (cluster addresses), completing on the peer's mbarrier.
__device__ __forceinline__ uint32_t mapa_u32(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ void bulk_to_peer(uint32_t rdst, uint32_t src, uint32_t bytes, uint32_t rbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(rdst),
      "r"(src), "r"(bytes), "r"(rbar)
      : "memory");
}

// 3-D tensor store of one staged box (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(ptx::smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Element (r, c) of an fp32 [BM rows][BN] tile in shared memory: 16-byte chunk
// c / 4 of row r stored at chunk (c / 4) ^ ((r / 2) % 8), so both the
// row-per-lane writes from TMEM and the row-pair-per-lane reads of the
// reduction spread over the banks.
template <int BN>
__device__ __forceinline__ int part_idx(int r, int c) {
  return r * BN + ((((c >> 2) ^ ((r >> 1) & 7)) << 2) | (c & 3));
}

// On-chip split-K reduction, rank ``rank`` of S: rows [rank*R, rank*R + R) of
// the tile summed over the S partials in rank order -- this CTA's from
// ``part``, peer p's slice of those rows from ``recv`` slot p ([R][BN] each,
// chunks swizzled by tile row) -- then the KIND epilogue.  One item is a row
// pair and 4 consecutive tokens; the loops are kept rolled because this code
// runs once per CTA on a cold instruction cache.
template <int BN, int KIND, int ACT = ACT_NONE>
__device__ __forceinline__ void reduce_onchip(const Epi& e, const float* part, const float* recv, int S, int rank,
                                           int m0, int n0, int M, int N) {
  const int R = BM / S, pairs = R / 2, items = pairs * (BN / 4);
  const int tok = KIND == EPI_ROPE ? e.tok_rope : 1;
#pragma unroll 1
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int p = it % pairs, q = it / pairs;
    const int rr = rank * R + 2 * p, j0 = 4 * q;
    const int n = n0 + rr;
    if (n >= N || m0 + j0 >= M) continue;
    const EpiRun<KIND, ACT> run(e, n);
    float2 cs[4];
    if (KIND == EPI_ROPE) {
      int j = (m0 + j0) % tok;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        cs[t] = run.rope_ ? run.rope_cs(j) : make_float2(1.f, 0.f);
        j = j + 1 == tok ? 0 : j + 1;
      }
    }
    const int ch = (q ^ ((rr >> 1) & 7)) << 2;   // rows rr and rr + 1 share the swizzle phase
    const int lr = rr - rank * R;
    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
#pragma unroll 1
    for (int sp = 0; sp < S; ++sp) {
      const float* b = sp == rank ? part + rr * BN : recv + (sp * R + lr) * BN;
      const float4 u0 = *reinterpret_cast<const float4*>(b + ch);
      const float4 u1 = *reinterpret_cast<const float4*>(b + BN + ch);
      s0.x += u0.x; s0.y += u0.y; s0.z += u0.z; s0.w += u0.w;
      s1.x += u1.x; s1.y += u1.y; s1.z += u1.z; s1.w += u1.w;
    }
    const float a0[4] = {s0.x, s0.y, s0.z, s0.w}, a1[4] = {s1.x, s1.y, s1.z, s1.w};
    float o0[4], o1[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) run.compute(a0[t], a1[t], KIND == EPI_ROPE ? cs[t] : make_float2(1.f, 0.f), o0[t], o1[t]);
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (m0 + j0 + t < M) run.store(m0 + j0 + t, o0[t], o1[t]);
  }
}

// Rank ``rank`` of an S-way split sums rows [rank*128/S, (rank+1)*128/S) of the
// tile over the S partials (layout [split][token][row]) in split order and
// applies the epilogue.  U items per thread keep U*S loads in flight.
template <int U>
__device__ __forceinline__ void reduce_rows(const Epi& e, const float* __restrict__ base, int S, int rank,
                                            int m0, int n0, int M, int N, int BN) {
  const int R = BM / S, pairs = R / 2, items = pairs * BN;
  const int nt = blockDim.x;
#pragma unroll 1
  for (int it0 = threadIdx.x; it0 < items; it0 += nt * U) {
    int mm[U], nn[U], jj[U], rr[U];
    bool ok[U];
    EpiPre pre[U];
    float2 acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int it = it0 + u * nt;
      const int p = it % pairs, j = it / pairs;
      rr[u] = rank * R + 2 * p;
      jj[u] = j;
      mm[u] = m0 + j;
      nn[u] = n0 + rr[u];
      ok[u] = it < items && mm[u] < M && nn[u] < N;
      if (ok[u]) pre[u] = epi_prefetch<bf16>(e, mm[u], nn[u]);
      acc[u] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int s = 0; s < 16 / U; ++s) {
      if (s < S) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (ok[u]) {
            const float2 v = *reinterpret_cast<const float2*>(base + ((long long)s * BN + jj[u]) * BM + rr[u]);
            acc[u].x += v.x;
            acc[u].y += v.y;
          }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (ok[u]) epi_pair<bf16>(e, mm[u], nn[u], acc[u].x, acc[u].y, pre[u]);
  }
}

// Epilogue of accumulator columns [c_begin, c_end) of this warp's TMEM lanes
// (SCALED: each lane's accumulator row times ``sc``, the FP8 row scale).
template <int KIND, int ACT = ACT_NONE, bool SCALED = false>
__device__ __forceinline__ void tile_epilogue(const Epi& e, uint32_t taddr, int c_begin, int c_end, int m0,
                                              int n_even, int M, int N, bool odd, float sc = 1.f) {
  const EpiRun<KIND, ACT> run(e, n_even < N ? n_even : 0);
  const bool live = n_even < N;
  const int tok = KIND == EPI_ROPE ? e.tok_rope : 1;
#pragma unroll 1
  for (int c0 = c_begin; c0 < c_end; c0 += 32) {
    float v[32];
    ptx::tmem_ld32(taddr + (uint32_t)c0, v);
    if constexpr (SCALED) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= sc;
    }
    epi_columns<KIND, ACT>(run, v, odd, m0 + c0 + (odd ? 1 : 0), live ? M : 0, tok);
  }
}

constexpr int kThreads = 256;  // 8 warps: warps 0 and 3 TMA, warp 1 MMA, all 8 share the epilogue
constexpr long long kDrainPolls = 1LL << 22;   // bounded wait for a CTA's own copies after an abort

// Memory later kernels read, to be pulled into L2 while this kernel runs.
struct L2Ahead {
  const void* p[3];
  long long bytes[3];
};
// This CTA's share of each range, 128-byte lines spread over ``nthreads`` threads (t < nthreads).
__device__ __forceinline__ void prefetch_lines_l2(const L2Ahead& ah, int t, int nthreads) {
  const long long ctas = (long long)gridDim.x * gridDim.y * gridDim.z;
  const long long cta = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
#pragma unroll 1
  for (int i = 0; i < 3; ++i) {
    if (!ah.p[i] || ah.bytes[i] < 128) continue;
    const long long lines = ah.bytes[i] / 128;
    const long long per = (lines + ctas - 1) / ctas;
    const long long l0 = cta * per, l1 = l0 + per < lines ? l0 + per : lines;
    const char* base = static_cast<const char*>(ah.p[i]);
    for (long long l = l0 + t; l < l1; l += nthreads)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(base + l * 128) : "memory");
  }
}
inline L2Ahead l2_ahead(const GemmArgs& a) {
  L2Ahead r;
  for (int i = 0; i < 3; ++i) {
    r.p[i] = a.l2[i].p;
    r.bytes[i] = a.l2[i].bytes;
  }
  return r;
}

// ---------------------------------------------------------------------------
// E4M3 weights (GR00T_WFMT_FP8).  Roles: warp 0 streams the 128 x 128-byte code
// tiles (no dependency wait: no kernel writes weights); warp 2 waits for the
// previous kernel and streams the activation stages; warps 3..7 widen each code
// tile into the stage's bf16 A tile; warp 1 issues the MMAs once both halves of
// a stage are in place.  E4M3 -> f16 -> f32 -> bf16 is exact (3 mantissa bits,
// exponents 2^-9 .. 2^8), so the MMA sums e4m3(code) * x exactly as the bf16
// path sums w * x; the row scale is applied in the epilogue.
// ---------------------------------------------------------------------------
constexpr int kTaMovers = 4;   // warps 4..7: one per tensor-memory lane quadrant

// 16 E4M3 codes -> 8 bf16 pairs (element 2j in the low half of word j).
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4& in, uint32_t (&o)[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t f16x2;
      const unsigned short pair = (unsigned short)(w[i] >> (16 * h));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f16x2) : "h"(pair));
      __half2 hv = *reinterpret_cast<__half2*>(&f16x2);
      const float2 f = __half22float2(hv);
      __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
      o[2 * i + h] = *reinterpret_cast<uint32_t*>(&b);
    }
  }
}

template <int BN, int STAGES, int WF>
__device__ __forceinline__ void ta_main_loop(const CUtensorMap& tmW, const CUtensorMap& tmX, uint8_t* sA,
                                             uint8_t* sB, uint8_t* sRaw, uint64_t* full, uint64_t* empty,
                                             uint64_t* done, uint64_t* cvt_full, uint64_t* raw_full,
                                             uint64_t* raw_empty, uint32_t tmem, int* abort_flag, int* err,
                                             long long wait_limit, int n0, int m0, int kb0, int nkb, int warp,
                                             int lane) {
  using L = TcSmem<BN, STAGES, WF>;
  constexpr int RAW = L::RAW, BKX = L::BKX;
  (void)sA;
  auto fail = [&]() {
    atomicExch(abort_flag, 1);
    atomicExch(err, 1);
  };
  if (warp == 0) {
    if (lane == 0) {   // code tiles: [128 rows][128 bytes], 128-byte swizzle
      const uint64_t pw = ptx::policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int r = i % RAW;
        if (i >= RAW && !ptx::mbar_wait(&raw_empty[r], ((i / RAW) & 1) ^ 1, wait_limit)) {
          fail();
          break;
        }
        ptx::mbar_arrive_expect_tx(&raw_full[r], L::RAW_BYTES);
        ptx::tma_load_2d(sRaw + r * L::RAW_BYTES, &tmW, &raw_full[r], (kb0 + i) * BKX, n0, pw);
        issued = i + 1;
      }
      if (*abort_flag)   // drain this thread's copies in flight (bounded)
        for (int i = issued - 1; i >= 0 && i >= issued - RAW; --i)
          ptx::mbar_wait(&raw_full[i % RAW], (i / RAW) & 1, wait_limit);
    }
  } else if (warp == 2) {
    if (lane == 0) {   // activations: BKX / 64 boxes of 64 columns per stage, after the dependency wait
      const uint64_t px = ptx::policy_evict_last();
      ptx::pdl_wait();
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES && !ptx::mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, wait_limit)) {
          fail();
          break;
        }
        ptx::mbar_arrive_expect_tx(&full[s], L::B_BYTES);
#pragma unroll
        for (int h = 0; h < BKX / 64; ++h)
          ptx::tma_load_2d(sB + s * L::B_BYTES + h * (BN * 128), &tmX, &full[s], (kb0 + i) * BKX + h * 64, m0, px);
        issued = i + 1;
      }
      if (*abort_flag)
        for (int i = issued - 1; i >= 0 && i >= issued - STAGES; --i)
          ptx::mbar_wait(&full[i % STAGES], (i / STAGES) & 1, wait_limit);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16(BM, BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        if (!ptx::mbar_wait(&cvt_full[s], (i / STAGES) & 1, wait_limit) ||
            !ptx::mbar_wait(&full[s], (i / STAGES) & 1, wait_limit)) {
          fail();
          break;
        }
        ptx::tc_fence_after();
        const uint32_t ta = tmem + (uint32_t)(BN + s * L::A_COLS);
#pragma unroll
        for (int k = 0; k < BKX / 16; ++k) {   // 8 columns (16 K elements) of A per step; B: 64-column boxes
          const uint64_t bd = ptx::sdesc_sw128(ptx::smem_u32(sB + s * L::B_BYTES + (k >> 2) * (BN * 128)));
          ptx::mma_bf16_tmem_a(tmem, ta + 8 * k, bd + 2 * (k & 3), idesc, (i | k) != 0);
        }
        ptx::mma_commit(&empty[s]);
      }
      ptx::mma_commit(done);
    }
  } else if (warp >= 4) {
    // movers: warp w owns weight rows 32 (w % 4) .. +31 (its tensor-memory lane
    // quadrant); a lane widens its row's 128 codes (16-byte chunk c stored at chunk
    // c ^ (row % 8)) into 64 columns of the stage's A tile
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    for (int i = 0; i < nkb; ++i) {
      const int r = i % RAW, s = i % STAGES;
      if (!ptx::mbar_wait(&raw_full[r], (i / RAW) & 1, wait_limit) ||
          (i >= STAGES && !ptx::mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, wait_limit))) {
        fail();
        break;
      }
      ptx::tc_fence_after();
      const uint8_t* src = sRaw + r * L::RAW_BYTES + row * 128;
      const uint32_t ta = lane_base + (uint32_t)(BN + s * L::A_COLS);
      uint32_t a[64];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 in = *reinterpret_cast<const uint4*>(src + ((c ^ (row & 7)) << 4));
        uint32_t o[8];
        e4m3x16_to_bf16(in, o);
#pragma unroll
        for (int j = 0; j < 8; ++j) a[8 * c + j] = o[j];
      }
      ptx::tmem_st32u(ta, a);
      ptx::tmem_st32u(ta + 32, a + 32);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&raw_empty[r]);
        ptx::mbar_arrive(&cvt_full[s]);
      }
    }
  }
}

// EK >= 0: only epilogue kind EK is compiled in (EPI_PARTIAL; or EPI_ROPE /
// EPI_GEGLU / EPI_STORE without split or with the on-chip reduction), a smaller kernel for
// once-per-CTA code on a cold instruction cache; EK = -1: every kind and path.
template <int BN, int STAGES, int WF = WF_SMEM, int EK = -1>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmO, int M, int N, int kb_per_split, Epi e,
                   float* __restrict__ ws, int* err, long long wait_limit, L2Ahead ahead) {
  using L = TcSmem<BN, STAGES, WF>;
  constexpr bool F8 = L::F8, TA = L::TA;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::A_STAGE;
  uint8_t* sRaw = smem + L::PIPE;               // TA: weight tiles on their way to tensor memory
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* done = empty + STAGES;
  uint64_t* recv_bar = done + 1;                // split-K: the peers' row slices landed
  uint64_t* cvt_full = recv_bar + 1;            // TA: [STAGES] the stage's A tile is in tensor memory
  uint64_t* raw_full = cvt_full + (TA ? STAGES : 0);   // TA: [RAW] a weight tile landed
  uint64_t* raw_empty = raw_full + L::RAW;             // TA: [RAW] the movers read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(raw_empty + L::RAW);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)gridDim.z;                 // split-K factor (the cluster size when reducing here)
  constexpr bool kSpec = EK >= 0;
  const int kind = kSpec ? EK : e.kind;
  const bool onchip = L::ONCHIP && S > 1 && kind != EPI_PARTIAL;
  const int rank = (int)blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BM, m0 = blockIdx.y * BN;
  const int kb0 = blockIdx.z * kb_per_split;
  const int nkb = kb_per_split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], TA ? 1 : 2);   // bf16 weights: the weight and the activation producer arrive
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(done, 1);
    ptx::mbar_init(recv_bar, 1);
    if constexpr (TA) {
      for (int s = 0; s < STAGES; ++s) ptx::mbar_init(&cvt_full[s], kTaMovers);
      for (int r = 0; r < L::RAW; ++r) {
        ptx::mbar_init(&raw_full[r], 1);
        ptx::mbar_init(&raw_empty[r], kTaMovers);
      }
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
    if (onchip) ptx::mbar_arrive_expect_tx(recv_bar, (uint32_t)((S - 1) * (BM / S) * BN * 4));
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
  }
  if (warp == 2) ptx::tmem_alloc(tmem_slot, L::TMEM_COLS);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ptx::pdl_launch_dependents();
  // warps with no main-loop role pull the memory the next kernels read into L2 by plain
  // line prefetches, which leave this CTA's TMA stream alone: warps 4..7 on the bf16
  // path, warp 3 on the E4M3 path
  if (!TA && warp >= 4) prefetch_lines_l2(ahead, threadIdx.x - 128, 128);
  if (TA && warp == 3) prefetch_lines_l2(ahead, lane, 32);

  if constexpr (TA) {
    ta_main_loop<BN, STAGES, WF>(tmW, tmX, sA, sB, sRaw, full, empty, done, cvt_full, raw_full, raw_empty, tmem,
                             abort_flag, err, wait_limit, n0, m0, kb0, nkb, warp, lane);
  } else if ((warp == 0 || warp == 3) && lane == 0) {
    // two producers, each with its own stream of TMA requests (a thread's requests are
    // served one after another): warp 0 the weight tiles -- no kernel writes weights, so
    // they need no dependency wait and run ahead of it -- and warp 3 the activation tiles
    // after the wait.  Each arrives on the stage's full barrier with its own bytes.
    const bool wprod = warp == 0;
    if (!wprod) {
      ptx::pdl_wait();
      kstamp(e.ts);
    }
    const uint64_t pol = wprod ? ptx::policy_evict_first() : ptx::policy_evict_last();
    const uint32_t bytes = wprod ? (uint32_t)L::A_STAGE : (uint32_t)L::B_BYTES;
    int issued = 0;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      if (i >= STAGES && !ptx::mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, wait_limit)) {
        atomicExch(abort_flag, 1);
        atomicExch(err, 1);
        break;
      }
      if (*(volatile int*)abort_flag) break;
      ptx::mbar_arrive_expect_tx(&full[s], bytes);
      if (wprod)
        ptx::tma_load_2d(sA + s * L::A_STAGE, &tmW, &full[s], (kb0 + i) * BK, n0, pol);
      else
        ptx::tma_load_2d(sB + s * L::B_BYTES, &tmX, &full[s], (kb0 + i) * BK, m0, pol);
      issued = i + 1;
    }
    if (*(volatile int*)abort_flag) {
      // drain: wait (bounded) for the stages this thread armed last, whose copies may be in flight
      const long long drain = wait_limit > kDrainPolls ? wait_limit : kDrainPolls;
      for (int i = issued - 1; i >= 0 && i >= issued - STAGES; --i)
        ptx::mbar_wait(&full[i % STAGES], (i / STAGES) & 1, drain);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16(BM, BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        if (!ptx::mbar_wait(&full[s], (i / STAGES) & 1, wait_limit)) {
          atomicExch(abort_flag, 1);
          atomicExch(err, 1);
          break;
        }
        ptx::tc_fence_after();
        const uint64_t ad = ptx::sdesc_sw128(ptx::smem_u32(sA + s * L::A_STAGE));
        const uint64_t bd = ptx::sdesc_sw128(ptx::smem_u32(sB + s * L::B_BYTES));
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)  // 16 bf16 = 32 bytes = 2 descriptor units per MMA
          ptx::mma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (i | k) != 0);
        ptx::mma_commit(&empty[s]);
      }
      ptx::mma_commit(done);
    }
  }
  __syncwarp();
  // every thread waits for the previous kernel before touching activation memory
  ptx::pdl_wait();
  if (TA && threadIdx.x == 96) kstamp(e.ts);   // warp 3 has no main-loop role on the E4M3 path

  if (!ptx::mbar_wait(done, 0, wait_limit)) {
    atomicExch(abort_flag, 1);
    atomicExch(err, 1);
  }
  __syncthreads();
  ptx::tc_fence_after();
  const bool aborted = *abort_flag != 0;
  // TMEM lane quadrant q = warp % 4 holds weight rows 32q..32q+31; the two warps
  // of a quadrant split the BN token columns
  const int quad = warp & 3;
  const int row = quad * 32 + lane;          // TMEM lane = weight row n0 + row
  const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16);
  const int c_begin = (warp >> 2) * (BN / 2), c_end = c_begin + BN / 2;
  // F8: the accumulator holds sum_k e4m3(code) x; the row's scale finishes it
  const float wsc = F8 ? (n0 + row < N ? e.wscale[n0 + row] : 0.f) : 1.f;

  if (EK == EPI_PARTIAL && e.tstore) {
    // split partial to the consumer's buffer [split][M][ldo] by tensor stores: each warp
    // stages its [BN/2 tokens][32 rows] fp32 block, [token][row] (128-byte rows), in the
    // idle pipeline memory (every MMA has completed), and its lane 0 writes one
    // [32 tokens][32 rows] box per 32 tokens through a [split][M][N] map, which clips
    // tokens past M within the split
    float* stg = reinterpret_cast<float*>(smem) + warp * (BN / 2) * 32;
    const int nb = n0 + quad * 32;   // this warp's first row (N % 32 == 0: all its rows or none are < N)
    if (!aborted && nb < N) {
#pragma unroll 1
      for (int c0 = c_begin; c0 < c_end; c0 += 32) {
        if (m0 + c0 >= M) break;
        float v[32];
        ptx::tmem_ld32(taddr + (uint32_t)c0, v);
        float* sp = stg + (c0 - c_begin) * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j) sp[j * 32 + lane] = F8 ? v[j] * wsc : v[j];
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the tensor stores read these writes
      __syncwarp();
      if (lane == 0) {
        for (int c0 = c_begin; c0 < c_end && m0 + c0 < M; c0 += 32)
          tma_store_3d(&tmO, stg + (c0 - c_begin) * 32, nb, m0 + c0, (int)blockIdx.z);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
      }
      __syncwarp();
    }
  } else if (kind == EPI_PARTIAL) {
    // split partial straight to the consumer's buffer: out[(split * M + m) * ldo + n]
    float* part = reinterpret_cast<float*>(e.out) + (long long)blockIdx.z * M * e.ldo;
    const int n = n0 + row;
    if (!aborted) {  // CTA-uniform: every lane takes part in tcgen05.ld
#pragma unroll 1
      for (int c0 = c_begin; c0 < c_end; c0 += 32) {
        float v[32];
        ptx::tmem_ld32(taddr + (uint32_t)c0, v);
        if (n < N) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (m0 + c0 + j < M) part[(long long)(m0 + c0 + j) * e.ldo + n] = F8 ? v[j] * wsc : v[j];
        }
      }
    }
  } else if (S == 1) {
    // direct epilogue from registers: lanes (2i, 2i+1) hold rows (n, n+1); swap
    // one value per column pair so each lane finishes one (n, n+1) output pair
    const int n_even = n0 + (row & ~1);
    const bool odd = lane & 1;
    if constexpr (EK == EPI_ROPE || EK == EPI_GEGLU) {
      if (!aborted) tile_epilogue<EK, ACT_NONE, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc);
    } else if constexpr (EK == EPI_STORE) {
      if (!aborted) {
        if (e.act == ACT_SWISH)
          tile_epilogue<EPI_STORE, ACT_SWISH, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc);
        else if (e.act == ACT_GELU)
          tile_epilogue<EPI_STORE, ACT_GELU, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc);
        else
          tile_epilogue<EPI_STORE, ACT_NONE, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc);
      }
    } else if constexpr (!kSpec) {
      if (!aborted) {
        switch (e.kind) {
          case EPI_STORE:
            if (e.act == ACT_SWISH)
              tile_epilogue<EPI_STORE, ACT_SWISH, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc);
            else if (e.act == ACT_GELU)
              tile_epilogue<EPI_STORE, ACT_GELU, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc);
            else
              tile_epilogue<EPI_STORE, ACT_NONE, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc);
            break;
          case EPI_ROPE: tile_epilogue<EPI_ROPE, ACT_NONE, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc); break;
          case EPI_GEGLU: tile_epilogue<EPI_GEGLU, ACT_NONE, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc); break;
          default: tile_epilogue<EPI_RESID, ACT_NONE, F8>(e, taddr, c_begin, c_end, m0, n_even, M, N, odd, wsc); break;
        }
      }
    }
  } else if (onchip) {
    // split-K on chip: park this CTA's fp32 partial in its idle pipeline memory,
    // one cluster barrier, then one bulk copy per peer hands it the R = 128/S
    // rows it reduces; the epilogue operands are fetched meanwhile
    float* part = reinterpret_cast<float*>(smem);
    float* recv = part + BN * BM;   // [S][R][BN]: slot p = rows of peer p (own slot unused)
    const int R = BM / S;
    if (!aborted) {
#pragma unroll 1
      for (int c0 = c_begin; c0 < c_end; c0 += 32) {
        float v[32];
        ptx::tmem_ld32(taddr + (uint32_t)c0, v);
        if constexpr (F8) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= wsc;
        }
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(part + part_idx<BN>(row, c0 + j)) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the bulk copies read these writes
    cluster.sync();
    if (threadIdx.x == 0) {
      for (int q = 0; q < S; ++q) {
        if (q == rank) continue;
        bulk_to_peer(mapa_u32(ptx::smem_u32(recv + (long long)rank * R * BN), (uint32_t)q),
                     ptx::smem_u32(part + (long long)q * R * BN), (uint32_t)(R * BN * 4),
                     mapa_u32(ptx::smem_u32(recv_bar), (uint32_t)q));
      }
    }
    if (!ptx::mbar_wait(recv_bar, 0, wait_limit)) {
      atomicExch(abort_flag, 1);
      atomicExch(err, 1);
    }
    // every copy into this CTA has landed: arrive now, wait at the end, so the
    // barrier that keeps each source alive overlaps the reduction
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    if (!aborted && !*abort_flag) {
      if constexpr (EK == EPI_ROPE || EK == EPI_GEGLU) {
        reduce_onchip<BN, EK>(e, part, recv, S, rank, m0, n0, M, N);
      } else if constexpr (EK == EPI_STORE) {
        if (e.act == ACT_SWISH)
          reduce_onchip<BN, EPI_STORE, ACT_SWISH>(e, part, recv, S, rank, m0, n0, M, N);
        else if (e.act == ACT_GELU)
          reduce_onchip<BN, EPI_STORE, ACT_GELU>(e, part, recv, S, rank, m0, n0, M, N);
        else
          reduce_onchip<BN, EPI_STORE, ACT_NONE>(e, part, recv, S, rank, m0, n0, M, N);
      } else if constexpr (!kSpec) {
        switch (e.kind) {
          case EPI_STORE:
            if (e.act == ACT_SWISH)
              reduce_onchip<BN, EPI_STORE, ACT_SWISH>(e, part, recv, S, rank, m0, n0, M, N);
            else if (e.act == ACT_GELU)
              reduce_onchip<BN, EPI_STORE, ACT_GELU>(e, part, recv, S, rank, m0, n0, M, N);
            else
              reduce_onchip<BN, EPI_STORE, ACT_NONE>(e, part, recv, S, rank, m0, n0, M, N);
            break;
          case EPI_ROPE: reduce_onchip<BN, EPI_ROPE>(e, part, recv, S, rank, m0, n0, M, N); break;
          case EPI_GEGLU: reduce_onchip<BN, EPI_GEGLU>(e, part, recv, S, rank, m0, n0, M, N); break;
          default: reduce_onchip<BN, EPI_RESID>(e, part, recv, S, rank, m0, n0, M, N); break;
        }
      }
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // every copy out of this CTA landed
  } else {
    // split-K: park the fp32 partial in the L2-resident workspace, one cluster
    // barrier (release/acquire orders the global writes), then each rank sums
    // its 128/S rows over the S partials in rank order.
    const long long tile = (long long)blockIdx.y * gridDim.x + blockIdx.x;
    float* my = ws + ((tile * S + (long long)blockIdx.z) * BN) * BM;
    if (!aborted) {
#pragma unroll 1
      for (int c0 = c_begin; c0 < c_end; c0 += 32) {
        float v[32];
        ptx::tmem_ld32(taddr + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) my[(c0 + j) * BM + row] = F8 ? v[j] * wsc : v[j];
      }
    }
    cluster.sync();
    const float* base = ws + (tile * S) * BN * BM;
    if (!kSpec && !aborted) {   // (the specialised kernels are not launched on this path)
      if (S <= 2)
        reduce_rows<8>(e, base, S, rank, m0, n0, M, N, BN);
      else if (S <= 4)
        reduce_rows<4>(e, base, S, rank, m0, n0, M, N, BN);
      else if (S <= 8)
        reduce_rows<2>(e, base, S, rank, m0, n0, M, N, BN);
      else
        reduce_rows<1>(e, base, S, rank, m0, n0, M, N, BN);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Persistent variant for many tiles (large token counts): one CTA per SM walks
// the tiles; warp 0 streams the weight tiles and warp 10 the activation tiles
// continuously across tiles (two TMA request streams), warp 1 issues the MMAs
// into one of two TMEM accumulators (2 x BN columns), and warps 2..9 drain the
// other accumulator through the epilogue, so the epilogue of tile i overlaps
// the main loop of tile i + 1.  Tiles are ordered token-tile fastest:
// concurrently running CTAs share weight tiles in L2.
//
// CL = 2: the CTAs run as clusters of two over adjacent weight tiles of the
// same token tile.  Each loads its own weight tile and one half of the shared
// activation tile, multicast into both CTAs' shared memory, so the L2 serves
// each activation tile once per pair (a third less L2 traffic per MMA).  A
// stage's slot is refilled only once both CTAs' MMAs released it (each MMA
// warp arrives on both CTAs' empty barriers).
// ---------------------------------------------------------------------------
constexpr int kPersThreads = 352;   // warp 0 weight TMA, 1 MMA, 2..9 epilogue, 10 activation TMA
constexpr int kPersEpiWarps = 8;
constexpr int kStgBox = 32 * 16 * 2;   // one staged output box: [32 tokens][16 outputs] bf16
constexpr int kStgChunk = 2 * kStgBox;   // a chunk of 32 token columns: up to two boxes

template <int BN, int STAGES>
struct PersSmem {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int PIPE = STAGES * STAGE_BYTES;
  static constexpr int STG = PIPE;   // per epilogue warp: two chunk buffers (double-buffered tensor stores)
  static constexpr int BAR_OFF = STG + kPersEpiWarps * 2 * kStgChunk;
  static constexpr int BAR = (2 * STAGES + 4) * 8 + 16;
  static constexpr int TOTAL = BAR_OFF + BAR + 1024;
  static_assert(TOTAL <= 232448, "shared memory of the persistent GEMM");
};

// 2-D tensor store of one staged box, completion tracked by bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(ptx::smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}

// Epilogue of accumulator columns [c_begin, c_end) of this warp's 32 TMEM lanes
// (output rows n_base .. n_base + 31, all < N) with the outputs staged in shared
// memory and written by tensor stores.  Per 32-token chunk the warp's outputs
// leave as one or two [32 tokens][16 outputs] boxes issued by lane 0, instead of
// 16 to 32 scattered 2- or 4-byte stores per lane (measured ~90 cycles each when
// all epilogue warps store at once).  Box x origins: plain pairs (EPI_STORE, and
// the non-rotated rows of EPI_ROPE) n_base and n_base + 16; RoPE rows the two
// halves of the head, head * hd + i and head * hd + i + hd / 2 for the warp's 16
// frequencies i; GeGLU n_base / 2.  Two chunk buffers per warp: before one is
// rewritten, the group that read it two chunks earlier has finished reading
// (``ck`` counts this warp's chunks).  M = 0: compute and staging only (the
// instruction-cache warm-up), nothing is stored and ``ck`` is unchanged.
template <int KIND, int ACT>
__device__ __forceinline__ void tile_epilogue_ts(const Epi& e, const CUtensorMap* tmO, uint32_t taddr, int c_begin,
                                                 int c_end, int m0, int n_base, int M, int lane, uint8_t* stg,
                                                 int& ck) {
  const bool odd = lane & 1;
  const int p = lane >> 1;   // this lane's pair: rows n_base + 2p, n_base + 2p + 1
  const EpiRun<KIND, ACT> run(e, n_base + 2 * p);
  const bool rot = KIND == EPI_ROPE && run.rope_;
  int x0 = n_base, x1 = n_base + 16;
  if (rot) {
    x0 = (n_base / e.hd) * e.hd + (n_base % e.hd) / 2;
    x1 = x0 + e.hd / 2;
  } else if (KIND == EPI_GEGLU) {
    x0 = n_base / 2;
  }
  constexpr bool kTwo = KIND != EPI_GEGLU;
#pragma unroll 1
  for (int c0 = c_begin; c0 < c_end; c0 += 32) {
    if (M > 0 && m0 + c0 >= M) break;   // every later chunk is past the last token too
    float v[32];
    ptx::tmem_ld32(taddr + (uint32_t)c0, v);
    float2 cs[16];
    if (KIND == EPI_ROPE) {
      int j = (m0 + c0 + (odd ? 1 : 0)) % e.tok_rope;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        cs[q] = run.rope_ ? run.rope_cs(j) : make_float2(1.f, 0.f);
        j += 2;
        if (j >= e.tok_rope) j -= e.tok_rope;
        if (j >= e.tok_rope) j -= e.tok_rope;
      }
    }
    float o0[16], o1[16];
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const float send = odd ? v[c] : v[c + 1];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
      run.compute(odd ? recv : v[c], odd ? v[c + 1] : recv, KIND == EPI_ROPE ? cs[c >> 1] : make_float2(1.f, 0.f),
                  o0[c >> 1], o1[c >> 1]);
    }
    uint8_t* buf = stg + (ck & 1) * kStgChunk;
    if (M > 0 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
    __syncwarp();
    // token row 2q + odd of the chunk; [token][16 outputs] bf16 rows of 32 bytes
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int row = (2 * q + (odd ? 1 : 0)) * 32;
      if (rot) {
        *reinterpret_cast<bf16*>(buf + row + 2 * p) = __float2bfloat16_rn(o0[q]);
        *reinterpret_cast<bf16*>(buf + kStgBox + row + 2 * p) = __float2bfloat16_rn(o1[q]);
      } else if (KIND == EPI_GEGLU) {
        *reinterpret_cast<bf16*>(buf + row + 2 * p) = __float2bfloat16_rn(o0[q]);
      } else {
        *reinterpret_cast<__nv_bfloat162*>(buf + (p >> 3) * kStgBox + row + 4 * (p & 7)) =
            __floats2bfloat162_rn(o0[q], o1[q]);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the tensor store reads these writes
    __syncwarp();
    if (M > 0) {
      if (lane == 0) {
        tma_store_2d(tmO, buf, x0, m0 + c0);
        if (kTwo) tma_store_2d(tmO, buf + kStgBox, x1, m0 + c0);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
      ++ck;
    }
  }
}

// EK >= 0: the tensor-store epilogue of that kind is the only one compiled in
// (a smaller kernel: its epilogue runs once per tile on a cold instruction cache);
// EK = -1: every epilogue kind, chosen at run time.
template <int BN, int STAGES, int CL, int EK>
__global__ void __launch_bounds__(kPersThreads, 1)
    gemm_tc_persistent(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmO, int M, int N, int KB, Epi e, int* err,
                       long long wait_limit) {
  using L = PersSmem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // accumulator b ready for the epilogue
  uint64_t* tempty = tfull + 2;       // accumulator b drained by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (M + BN - 1) / BN;
  const int nt_pairs = ((N + BM - 1) / BM + CL - 1) / CL;   // groups of CL adjacent weight tiles
  const int ptiles = nt_pairs * mt;
  const int rank = CL > 1 ? (int)(blockIdx.x % CL) : 0;   // rank in the cluster (clusters of consecutive CTAs)
  const int cid = (int)blockIdx.x / CL, ncl = (int)gridDim.x / CL;
  constexpr int kEpiWarps = kPersEpiWarps;
  constexpr uint16_t kAll = (uint16_t)((1u << CL) - 1);
  // tile p of this cluster: weight rows n0 (this CTA's of the group), tokens m0
  auto tile_n0 = [&](int p) { return ((p / mt) * CL + rank) * BM; };
  auto tile_m0 = [&](int p) { return (p % mt) * BN; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 2);    // the weight and the activation producer arrive
      ptx::mbar_init(&empty[s], CL);  // every CTA's MMA warp of the cluster releases the slot
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&tfull[b], 1);
      ptx::mbar_init(&tempty[b], kEpiWarps);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
  }
  if (warp == 2) ptx::tmem_alloc(tmem_slot, 2 * BN);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (CL > 1) ptx::cluster_sync_all();   // the peer's barriers exist before anything targets them
  const uint32_t tmem = *tmem_slot;
  ptx::pdl_launch_dependents();

  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(err, 1);
  };
  long long stages_used = 0;   // weight producer: stage uses issued (for the final release wait)

  if ((warp == 0 || warp == 10) && lane == 0) {
    // two producers with their own TMA request streams (a thread's requests are served
    // one after another): warp 0 the weight tiles, which no kernel writes, so they run
    // ahead of the dependency wait; warp 10 the activation tiles (this CTA's 1/CL of
    // each, multicast to the cluster) after it
    const bool wprod = warp == 0;
    if (!wprod) {
      ptx::pdl_wait();
      kstamp(e.ts);
    }
    const uint64_t pol = wprod ? ptx::policy_evict_first() : ptx::policy_evict_last();
    const uint32_t bytes = wprod ? (uint32_t)A_BYTES : (uint32_t)L::B_BYTES;   // B: all CL parts land here
    long long it = 0, issued = 0;
    for (int p = cid; p < ptiles && !*abort_flag; p += ncl) {
      const int n0 = tile_n0(p), m0 = tile_m0(p);
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = (int)(it % STAGES);
        if (it >= STAGES && !ptx::mbar_wait(&empty[s], (uint32_t)(((it / STAGES) & 1) ^ 1), wait_limit)) {
          fail();
          break;
        }
        ptx::mbar_arrive_expect_tx(&full[s], bytes);
        if (wprod) {
          ptx::tma_load_2d(sA + s * A_BYTES, &tmW, &full[s], kb * BK, n0, pol);
        } else if (CL == 1) {
          ptx::tma_load_2d(sB + s * L::B_BYTES, &tmX, &full[s], kb * BK, m0, pol);
        } else {
          constexpr int HB = BN / CL;   // rows of this CTA's part (the map's box)
          ptx::tma_load_2d_mc(sB + s * L::B_BYTES + rank * HB * 128, &tmX, &full[s], kb * BK, m0 + rank * HB, kAll,
                              pol);
        }
        issued = it + 1;
      }
    }
    if (*abort_flag) {  // drain the copies into this CTA (bounded)
      const long long drain = wait_limit > kDrainPolls ? wait_limit : kDrainPolls;
      for (long long i = issued - 1; i >= 0 && i >= issued - STAGES; --i)
        ptx::mbar_wait(&full[i % STAGES], (uint32_t)((i / STAGES) & 1), drain);
    }
    stages_used = it;
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16(BM, BN);
      long long it = 0;
      int lt = 0;
      for (int p = cid; p < ptiles && !*abort_flag; p += ncl, ++lt) {
        const int b = lt & 1;
        if (lt >= 2 && !ptx::mbar_wait(&tempty[b], (uint32_t)(((lt >> 1) & 1) ^ 1), wait_limit)) {
          fail();
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * BN);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          if (!ptx::mbar_wait(&full[s], (uint32_t)((it / STAGES) & 1), wait_limit)) {
            fail();
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t ad = ptx::sdesc_sw128(ptx::smem_u32(sA + s * A_BYTES));
          const uint64_t bd = ptx::sdesc_sw128(ptx::smem_u32(sB + s * L::B_BYTES));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) ptx::mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
          if (CL == 1)
            ptx::mma_commit(&empty[s]);
          else
            ptx::mma_commit_mc(&empty[s], kAll);
        }
        ptx::mma_commit(&tfull[b]);
        if (!ok) break;
      }
    }
  } else if (warp >= 2 && warp < 2 + kEpiWarps) {
    ptx::pdl_wait();
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int c_begin = (ew >> 2) * (BN / 2), c_end = c_begin + BN / 2;
    const bool odd = lane & 1;
    constexpr bool kSpec = EK >= 0;
    const bool ts = kSpec || e.tstore != 0;   // outputs leave through shared memory and tensor stores
    uint8_t* stg = smem + L::STG + ew * 2 * kStgChunk;
    int ck = 0;   // this warp's staged chunks (tensor-store path)
    // tensor-store epilogue over columns [cb, ce) of rows n_base .. n_base + 31 (< N)
    auto ts_pass = [&](uint32_t taddr, int cb, int ce, int m0, int n_base, int Mx, int& k) {
      if constexpr (EK == EPI_ROPE) {
        tile_epilogue_ts<EPI_ROPE, ACT_NONE>(e, &tmO, taddr, cb, ce, m0, n_base, Mx, lane, stg, k);
      } else if constexpr (EK == EPI_GEGLU) {
        tile_epilogue_ts<EPI_GEGLU, ACT_NONE>(e, &tmO, taddr, cb, ce, m0, n_base, Mx, lane, stg, k);
      } else {
        switch (e.kind) {
          case EPI_STORE:
            if (e.act == ACT_SWISH)
              tile_epilogue_ts<EPI_STORE, ACT_SWISH>(e, &tmO, taddr, cb, ce, m0, n_base, Mx, lane, stg, k);
            else if (e.act == ACT_GELU)
              tile_epilogue_ts<EPI_STORE, ACT_GELU>(e, &tmO, taddr, cb, ce, m0, n_base, Mx, lane, stg, k);
            else
              tile_epilogue_ts<EPI_STORE, ACT_NONE>(e, &tmO, taddr, cb, ce, m0, n_base, Mx, lane, stg, k);
            break;
          case EPI_ROPE:
            tile_epilogue_ts<EPI_ROPE, ACT_NONE>(e, &tmO, taddr, cb, ce, m0, n_base, Mx, lane, stg, k);
            break;
          case EPI_GEGLU:
            tile_epilogue_ts<EPI_GEGLU, ACT_NONE>(e, &tmO, taddr, cb, ce, m0, n_base, Mx, lane, stg, k);
            break;
          default: break;
        }
      }
    };
    // per-lane stores (and the residual kinds) over columns [cb, ce)
    auto lane_pass = [&](uint32_t taddr, int cb, int ce, int m0, int n_even, int Mx) {
      if constexpr (!kSpec) {
        switch (e.kind) {
          case EPI_STORE:
            if (e.act == ACT_SWISH)
              tile_epilogue<EPI_STORE, ACT_SWISH>(e, taddr, cb, ce, m0, n_even, Mx, N, odd);
            else if (e.act == ACT_GELU)
              tile_epilogue<EPI_STORE, ACT_GELU>(e, taddr, cb, ce, m0, n_even, Mx, N, odd);
            else
              tile_epilogue<EPI_STORE, ACT_NONE>(e, taddr, cb, ce, m0, n_even, Mx, N, odd);
            break;
          case EPI_ROPE: tile_epilogue<EPI_ROPE>(e, taddr, cb, ce, m0, n_even, Mx, N, odd); break;
          case EPI_GEGLU: tile_epilogue<EPI_GEGLU>(e, taddr, cb, ce, m0, n_even, Mx, N, odd); break;
          default: tile_epilogue<EPI_RESID>(e, taddr, cb, ce, m0, n_even, Mx, N, odd); break;
        }
      }
    };
    {
      // Warm-up while the first tile's main loop runs: one pass of this
      // kernel's epilogue over 32 columns of the idle second accumulator with
      // no token in range (M = 0: nothing is stored).  The epilogue code runs
      // once per tile on a cold instruction cache otherwise (measured: the
      // first 32 columns of a tile took ~2.5 us longer than the next ones).
      const int n_base = (cid < ptiles ? tile_n0(cid) : 0) + quad * 32;
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)BN;
      int ck_warm = 0;
      if (ts) {
        if (n_base < N) ts_pass(taddr, c_begin, c_begin + 32, 0, n_base, 0, ck_warm);
      } else {
        lane_pass(taddr, c_begin, c_begin + 32, 0, n_base + (lane & ~1), 0);
      }
    }
    int lt = 0;
    for (int p = cid; p < ptiles; p += ncl, ++lt) {
      const int b = lt & 1;
      if (!ptx::mbar_wait(&tfull[b], (uint32_t)((lt >> 1) & 1), wait_limit)) {
        fail();
        break;
      }
      ptx::tc_fence_after();
      if (*abort_flag) break;
      const int n0 = tile_n0(p), m0 = tile_m0(p);
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * BN);
      if (ts) {
        if (n0 + quad * 32 < N) ts_pass(taddr, c_begin, c_end, m0, n0 + quad * 32, M, ck);
      } else {
        lane_pass(taddr, c_begin, c_end, m0, n0 + quad * 32 + (lane & ~1), M);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[b]);
    }
    // the tensor stores have read their staging buffers and written their outputs
    if (ts && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }
  if (CL > 1 && warp == 0 && lane == 0) {
    // every release of this CTA's slots (its own MMA warp's and the peer's) has arrived:
    // after this no MMA warp of the cluster signals this CTA's barriers any more
    const long long drain = wait_limit > kDrainPolls ? wait_limit : kDrainPolls;
    for (long long i = stages_used - 1; i >= 0 && i >= stages_used - STAGES; --i)
      ptx::mbar_wait(&empty[i % STAGES], (uint32_t)((i / STAGES) & 1), drain);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (CL > 1) ptx::cluster_sync_all();   // no copy or release targets a CTA that has left
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 2 * BN);
  }
}

template <int BN, int STAGES, int CL, int EK>
cudaError_t launch_persistent(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& to, const GemmArgs& a,
                              int sm_count, int* err, long long lim, cudaStream_t s, bool pdl) {
  using L = PersSmem<BN, STAGES>;
  auto kern = gemm_tc_persistent<BN, STAGES, CL, EK>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e1 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e1 != cudaSuccess) return e1;
    configured = true;
  }
  const int ptiles = (((a.N + BM - 1) / BM + CL - 1) / CL) * ((a.M + BN - 1) / BN);
  const int clusters = ptiles < sm_count / CL ? ptiles : sm_count / CL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * CL);
  cfg.blockDim = dim3(kPersThreads);
  cfg.dynamicSmemBytes = L::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, tw, tx, to, a.M, a.N, a.K / BK, a.epi, err, lim);
}

template <int BN, int STAGES, int WF>
cudaError_t launch_ta(const CUtensorMap& tw, const CUtensorMap& tx, const GemmArgs& a, int S, float* ws,
                      int* err, long long lim, cudaStream_t s, bool pdl) {
  using L = TcSmem<BN, STAGES, WF>;
  static_assert(L::TOTAL <= 232448, "shared memory of the tensor-memory-A GEMM");
  static_assert(L::TMEM_NEED <= 512, "tensor memory of the tensor-memory-A GEMM");
  auto kern = gemm_tc_kernel<BN, STAGES, WF>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e1 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e1 != cudaSuccess) return e1;
    e1 = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e1 != cudaSuccess) return e1;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.N + BM - 1) / BM, (a.M + BN - 1) / BN, S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = a.epi.kind == EPI_PARTIAL ? 1 : S;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const int KB = a.K / L::BKX;
  return cudaLaunchKernelEx(&cfg, kern, tw, tx, tw, a.M, a.N, KB / S, a.epi, ws, err, lim, l2_ahead(a));
}

template <int BN, int STAGES, int EK = -1>
cudaError_t launch(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& to, const GemmArgs& a, int S,
                   float* ws, int* err, long long lim, cudaStream_t s, bool pdl) {
  using L = TcSmem<BN, STAGES>;
  auto kern = gemm_tc_kernel<BN, STAGES, WF_SMEM, EK>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e1 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e1 != cudaSuccess) return e1;
    e1 = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e1 != cudaSuccess) return e1;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.N + BM - 1) / BM, (a.M + BN - 1) / BN, S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = a.epi.kind == EPI_PARTIAL ? 1 : S;   // partials need no cluster
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const int KB = a.K / BK;
  return cudaLaunchKernelEx(&cfg, kern, tw, tx, to, a.M, a.N, KB / S, a.epi, ws, err, lim, l2_ahead(a));
}

}  // namespace

}  // namespace g3
