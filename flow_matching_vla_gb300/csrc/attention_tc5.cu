// tcgen05 / TMEM attention of the action expert over prefix ++ own K/V.
//
// Same computation as the head-folded attention ("pi0.5 Design", Attention
// and the K/V pool: one KV head, the Hq query heads folded into rows, all-ones
// mask; vla.cpp Eq. (2) per row), on the 5th-generation tensor cores:
//
//  * a CTA owns 128 folded rows (r = t * Hq + h) and a range of 64-key tiles;
//    the prefix tiles come from the bound per-layer K/V (a flat [B, P] region or
//    a paged pool's slots, through a per-sample map: rows past P read as zeros),
//    the suffix tiles from this step's QKV projection;
//  * warps 0 and 10 issue TMA: Q once through a 4-D map over [tokens][heads][Dh]
//    whose box lands exactly in folded-row order; K and V tiles through
//    separate rings (128-byte swizzle, 64-element boxes; for Dh = 256 three K
//    slots and two V slots), a K slot freed as soon as S = QK^T read it, a V
//    slot when P V did.  The row tiles of one sample (and split) read the same
//    key tiles, so they run as a cluster: each CTA loads 1/CT of every K and V
//    tile (CT = row tiles, 2 or 4) and multicasts it into all CT CTAs, and a
//    slot is refilled once every CTA's MMA released it -- a tile is fetched
//    once per sample, and each SM issues a quarter of the requests;
//  * warp 1 issues tcgen05.mma: S = Q K^T into one of two TMEM buffers
//    (kind::f16, K-major operands), and O += P V into a TMEM accumulator with
//    V read MN-major straight from its [key][dim] tile; with a paged pool bound,
//    the first row tile's CTAs also store the suffix K/V tiles into the pool's
//    slots [P, P + H);
//  * warps 2..5 (one per TMEM lane quadrant, one thread per row, all keys of a
//    tile) run the softmax in registers: exp2 of scaled scores against a
//    running maximum that is only raised -- and O rescaled in TMEM -- when a
//    tile's maximum exceeds it by more than 8 (2^8 headroom, exact arithmetic
//    otherwise), and write P (bf16 pairs) into one of two TMEM buffers, from
//    which the P V MMA reads its A operand (no shared-memory round trip, no
//    exchange between threads of a row); warps 6..9 join for the output tile;
//  * the output tile (O / sum, bf16) is staged in the idle Q buffer and written
//    with one tensor store: to the attention output, or with S key splits as a
//    partial (with (max, sum)) to the workspace, where a warp-per-row kernel
//    merges the S splits.
// All mbarrier waits are bounded (error flag, drained copies, freed TMEM).
#include <cudaTypedefs.h>
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace g3 {


namespace {

constexpr int ROWS = 128;   // folded query rows per CTA (MMA M)
constexpr int KT = 64;      // keys per tile (MMA N of S, K of PV)
// warp 0: K loads, 1: MMA, 2..5: softmax (one warp per TMEM lane quadrant, a thread
// per row), 6..9 with 2..5: the output tile (half of O's columns each), 10: V loads
constexpr int kThreads = 352;
constexpr int kSlack = 256;   // alignment slack of the dynamic shared memory (checked)
constexpr int kMaxSplits = 32;   // key splits (a lane of the merge kernel's warp per split)
constexpr long long kDrainPolls = 1LL << 22;   // bounded wait for this CTA's own copies after an abort

template <int DH>
struct T5Smem {
  static constexpr int BOXES = DH / 64;          // 64-element column boxes per row block
  static constexpr int Q_BYTES = ROWS * DH * 2;
  static constexpr int KV_BYTES = KT * DH * 2;   // one K (or V) tile
  static constexpr int NK = DH == 256 ? 3 : 4;   // K ring slots
  static constexpr int NV = DH == 256 ? 2 : 4;   // V ring slots
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_X = OFF_V + NV * KV_BYTES;   // per row: (sum, max) handed to the staging warps
  static constexpr int OFF_BAR = OFF_X + 2 * ROWS * 4;
  static constexpr int NBAR = 1 + 2 * NK + 3 + 3 + 2 + 2 + 2 * NV;
  static constexpr int TOTAL = OFF_BAR + NBAR * 8 + 16 + kSlack;
  static_assert(TOTAL <= 232448, "shared memory of the tcgen05 attention");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && KV_BYTES % 1024 == 0, "128-byte-swizzled tiles");
};

// MN-major (V) descriptor: 64-element rows of 128 bytes along N in groups of 8 K-rows
// (1024 bytes); consecutive 64-element N blocks ``lbo`` bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
      "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
      "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One TMA request per tile: a tensor copy keeps its issuing thread busy for a
// fixed time (~0.25 us measured) whatever its size, so whole tiles move in one
// request rather than one per 64-column box.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(ptx::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(ptx::smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_hint(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z,
                                                 int w, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(ptx::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(ptx::smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z,
                                            int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];" ::"r"(ptx::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(ptx::smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
// Multicast variants: the box lands at the same offset in every CTA of ``mask``,
// completing on the mbarrier at the same offset in each.
__device__ __forceinline__ void tma_load_3d_mc(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z,
                                               uint16_t mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6, %7;" ::"r"(ptx::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(ptx::smem_u32(bar)), "r"(x), "r"(y), "r"(z), "h"(mask), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_mc(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z,
                                               int w, uint16_t mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7, %8;" ::"r"(ptx::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(ptx::smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w), "h"(mask),
      "l"(policy)
      : "memory");
}
// Tensor stores of a shared-memory tile (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(ptx::smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* m, const void* src, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(ptx::smem_u32(src)), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ void tma_store_5d(const CUtensorMap* m, const void* src, int x, int y, int z, int w,
                                             int v) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(ptx::smem_u32(src)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v)
      : "memory");
}
__device__ __forceinline__ void tma_store_drain() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(ptx::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(ptx::smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Key tile i of sample b: prefix tiles first (64-key steps over [0, P)), then suffix tiles over [P, P + H).
struct KeyTile {
  bool prefix;
  int row;    // first row: within sample b's prefix (the prefix map is per sample) or in the suffix map ([B*H])
  int valid;  // keys of the tile in range
  int srow;   // suffix tiles: first suffix row of the tile within the sample
};
__device__ __forceinline__ KeyTile key_tile(int i, int b, int P, int H) {
  const int np = (P + KT - 1) / KT;
  KeyTile t;
  if (i < np) {
    t.prefix = true;
    t.row = i * KT;
    t.valid = min(KT, P - i * KT);
    t.srow = 0;
  } else {
    const int j = (i - np) * KT;
    t.prefix = false;
    t.row = b * H + j;
    t.valid = min(KT, H - j);
    t.srow = j;
  }
  return t;
}

template <int DH>
__global__ void __launch_bounds__(kThreads, 1)
    attn_t5_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKp,
                   const __grid_constant__ CUtensorMap tmVp, const __grid_constant__ CUtensorMap tmKs,
                   const __grid_constant__ CUtensorMap tmVs, const __grid_constant__ CUtensorMap tmO,
                   const __grid_constant__ CUtensorMap tmPk, const __grid_constant__ CUtensorMap tmPv,
                   AttnT5Args a) {
  using L = T5Smem<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (smem - smem_raw > kSlack) {   // the layout assumes (almost) 1024-byte aligned dynamic memory
    if (threadIdx.x == 0) atomicExch(a.err, 1);
    return;
  }
  constexpr int NK = L::NK, NV = L::NV;
  uint8_t* sQ = smem + L::OFF_Q;
  uint8_t* sK = smem + L::OFF_K;
  uint8_t* sV = smem + L::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;           // [NK] K tile of ring slot landed
  uint64_t* k_empty = k_full + NK;       // [NK] S = QK^T read it
  uint64_t* s_full = k_empty + NK;       // [3] S buffer b computed
  uint64_t* s_empty = s_full + 3;        // [3] the softmax read it
  uint64_t* p_full = s_empty + 3;        // [2] P buffer b written
  uint64_t* pv_done = p_full + 2;        // [2] the PV reading P buffer b completed
  uint64_t* v_full = pv_done + 2;        // [NV] V tile of ring slot landed
  uint64_t* v_empty = v_full + NV;       // [NV] PV read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBAR);
  float* xm = reinterpret_cast<float*>(smem + L::OFF_X);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int S = (int)gridDim.y;
  const int split = (int)blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int r0 = blockIdx.x * ROWS;
  const int nrows = a.Hq * a.H;
  const int ntiles = (a.P + KT - 1) / KT + (a.H + KT - 1) / KT;
  const int tps = (ntiles + S - 1) / S;
  const int t_begin = split * tps;
  const int t_end = min(ntiles, t_begin + tps);
  const int nt = t_end > t_begin ? t_end - t_begin : 0;
  const long long lim = a.wait_limit;
  // a bound K/V pool takes this step's suffix K/V into its slots [P, P + H): the CTAs of
  // the first row tile own the suffix tiles of their key range and store them from shared memory
  const bool pool_writer = a.pool_k != nullptr && blockIdx.x == 0;
  const int CT = a.ct > 1 ? a.ct : 1;                 // CTAs of the cluster (row tiles of the sample)
  const int crank = CT > 1 ? (int)(blockIdx.x % CT) : 0;
  const uint16_t cmask = (uint16_t)((1u << CT) - 1);

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int i = 0; i < NK; ++i) {
      ptx::mbar_init(&k_full[i], 1);
      ptx::mbar_init(&k_empty[i], CT);   // every CTA of the cluster releases a multicast slot
    }
    for (int i = 0; i < NV; ++i) {
      ptx::mbar_init(&v_full[i], 1);
      ptx::mbar_init(&v_empty[i], CT);
    }
    for (int i = 0; i < 3; ++i) {
      ptx::mbar_init(&s_full[i], 1);
      ptx::mbar_init(&s_empty[i], 4);   // the four softmax warps read S
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&p_full[i], 4);    // the four softmax warps wrote P
      ptx::mbar_init(&pv_done[i], 1);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmKp);
    ptx::prefetch_tmap(&tmVp);
    ptx::prefetch_tmap(&tmKs);
    ptx::prefetch_tmap(&tmVs);
    ptx::prefetch_tmap(&tmO);
  }
  if (warp == 2) ptx::tmem_alloc(tmem_slot, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (CT > 1) ptx::cluster_sync_all();   // the peers' barriers exist before any copy or release targets them
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem;              // O: DH columns
  const uint32_t tS = tmem + 256;        // S buffers: 3 x 64 columns (S runs two tiles ahead of P V)
  const uint32_t tP = tmem + 448;        // P buffers: 2 x 32 columns of bf16 pairs (lane = row)
  ptx::pdl_launch_dependents();
  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(a.err, 1);
  };

  constexpr uint32_t idS = ptx::idesc_bf16(ROWS, KT);
  constexpr uint32_t idO = ptx::idesc_bf16(ROWS, DH) | (1u << 16);   // B (V) MN-major
  // S(j) = Q K(j)^T into S buffer j % 3
  auto issue_s = [&](int j) -> bool {
    const int st = j % NK, sb = j % 3;
    if (!ptx::mbar_wait(&k_full[st], (j / NK) & 1, lim)) return false;
    if (j >= 3 && !ptx::mbar_wait(&s_empty[sb], ((j / 3) - 1) & 1, lim)) return false;
    ptx::tc_fence_after();
    const KeyTile kt = key_tile(t_begin + j, b, a.P, a.H);
    if (pool_writer && !kt.prefix)   // rows past H fall outside the pool map
      tma_store_4d(&tmPk, sK + st * L::KV_BYTES, 0, kt.srow, b, 0);
    const uint32_t q0 = ptx::smem_u32(sQ), k0 = ptx::smem_u32(sK + st * L::KV_BYTES);
#pragma unroll
    for (int x = 0; x < L::BOXES; ++x)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        ptx::mma_bf16(tS + sb * KT, ptx::sdesc_sw128(q0 + x * ROWS * 128) + 2 * k,
                      ptx::sdesc_sw128(k0 + x * KT * 128) + 2 * k, idS, (x | k) != 0);
    ptx::mma_commit(&s_full[sb]);
    if (pool_writer && !kt.prefix) {   // the slot is refilled only after the store read it
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
    if (CT == 1)
      ptx::mma_commit(&k_empty[st]);
    else
      ptx::mma_commit_mc(&k_empty[st], cmask);
    return true;
  };
  // O += P(j) V(j), P from TMEM buffer j & 1
  auto issue_pv = [&](int j) -> bool {
    const int st = j % NV, pb = j & 1;
    if (!ptx::mbar_wait(&p_full[pb], (j >> 1) & 1, lim)) return false;
    if (!ptx::mbar_wait(&v_full[st], (j / NV) & 1, lim)) return false;
    ptx::tc_fence_after();
    const KeyTile vt = key_tile(t_begin + j, b, a.P, a.H);
    if (pool_writer && !vt.prefix) tma_store_4d(&tmPv, sV + st * L::KV_BYTES, 0, vt.srow, b, 0);
    const uint32_t v0 = ptx::smem_u32(sV + st * L::KV_BYTES);
#pragma unroll
    for (int k = 0; k < KT / 16; ++k)   // 16 keys per MMA: 8 P columns; 2 K-row groups of 1024 bytes of V
      ptx::mma_bf16_tmem_a(tO, tP + pb * (KT / 2) + 8 * k, sdesc_sw128_mn(v0 + k * 2048, KT * 128), idO,
                           j > 0 || k > 0);
    ptx::mma_commit(&pv_done[pb]);
    if (pool_writer && !vt.prefix) {
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
    if (CT == 1)
      ptx::mma_commit(&v_empty[st]);
    else
      ptx::mma_commit_mc(&v_empty[st], cmask);
    return true;
  };
  if (warp == 0 || warp == 10) {
    // ---------------- TMA producers: warp 0 streams K tiles, warp 10 V tiles ----------------
    if (lane == 0) {
      const bool is_k = warp == 0;
      const int NS = is_k ? NK : NV;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = is_k ? sK : sV;
      const CUtensorMap* pmap = is_k ? &tmKp : &tmVp;
      auto load = [&](int i) {
        const int st = i % NS;
        const KeyTile kt = key_tile(t_begin + i, b, a.P, a.H);
        uint8_t* dst = ring + st * L::KV_BYTES;
        ptx::mbar_arrive_expect_tx(&full[st], L::KV_BYTES);   // the whole tile lands here (all CT parts)
        // [Dh/64 boxes][KT rows][64 columns] in one request; prefix: 4-D map (columns, rows
        // [0, P) of the sample, samples, boxes) so rows past P read as zeros, never as a
        // neighbour's rows or a pool's other slots.  In a cluster this CTA loads boxes
        // [crank * part, (crank + 1) * part) and multicasts them
        const int part = L::BOXES / CT;
        if (CT == 1) {
          if (kt.prefix)
            tma_load_4d_hint(dst, pmap, &full[st], 0, kt.row, b, 0, ptx::policy_evict_first());
          else
            tma_load_3d_hint(dst, is_k ? &tmKs : &tmVs, &full[st], 0, kt.row, 0, ptx::policy_evict_last());
        } else {
          uint8_t* dpart = dst + crank * part * KT * 128;
          if (kt.prefix)
            tma_load_4d_mc(dpart, pmap, &full[st], 0, kt.row, b, crank * part, cmask, ptx::policy_evict_first());
          else
            tma_load_3d_mc(dpart, is_k ? &tmKs : &tmVs, &full[st], 0, kt.row, crank * part, cmask,
                           ptx::policy_evict_last());
        }
      };
      // bound prefix tiles do not depend on the previous kernel: stage them first
      int pre = 0;
      for (; pre < NS && pre < nt; ++pre)
        if (!key_tile(t_begin + pre, b, a.P, a.H).prefix) break;
      for (int i = 0; i < pre; ++i) load(i);
      ptx::pdl_wait();
      if (is_k) kstamp(a.ts);
      if (is_k) {
        ptx::mbar_arrive_expect_tx(q_full, L::Q_BYTES);
        const int tokens_per_tile = ROWS / a.Hq;
        // [Dh/64 boxes][tokens][heads][64 columns]: folded row r = t * Hq + h, one request
        tma_load_4d(sQ, &tmQ, q_full, 0, 0, b * a.H + blockIdx.x * tokens_per_tile, 0);
      }
      int loaded = pre;
      for (int i = pre; i < nt && !*abort_flag; ++i) {
        const int st = i % NS;
        if (i >= NS && !ptx::mbar_wait(&empty[st], ((i / NS) & 1) ^ 1, lim)) {
          fail();
          break;
        }
        load(i);
        loaded = i + 1;
      }
      const long long drain = lim > kDrainPolls ? lim : kDrainPolls;
      if (*abort_flag) {  // drain this thread's in-flight copies before the CTA can exit
        if (is_k) ptx::mbar_wait(q_full, 0, drain);
        for (int i = loaded - 1; i >= 0 && i >= loaded - NS; --i)
          ptx::mbar_wait(&full[i % NS], (i / NS) & 1, drain);
      }
      if (CT > 1)   // every CTA's release of this ring has arrived: no MMA warp signals it any more
        for (int i = loaded - 1; i >= 0 && i >= loaded - NS; --i)
          ptx::mbar_wait(&empty[i % NS], (i / NS) & 1, drain);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (lane 0; the other lanes idle until the end) ----------------
    // order on the tensor pipe: S(0), S(1), then S(j + 2) ahead of P(j) V(j), so the
    // softmax of tile j has two S batches of time before its P V is due
    if (lane == 0) {
      bool ok = ptx::mbar_wait(q_full, 0, lim);
      for (int j = 0; ok && j < 2 && j < nt; ++j) ok = issue_s(j);
      for (int j = 0; ok && j < nt; ++j) {
        if (j + 2 < nt) ok = issue_s(j + 2);
        if (ok) ok = issue_pv(j);
      }
      if (!ok) fail();
      if (pool_writer) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // pool writes done
    }
  } else {
    // ---------------- softmax (warps 2..5, a thread per row) and the output tile (2..9) ----------------
    const int quad = warp & 3, g = (warp - 2) >> 2;   // g: which half of O's columns the warp stages
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    constexpr int OH = DH / 2;                          // O columns per half
    const float sl2 = rsqrtf((float)DH) * 1.4426950408889634f;
    ptx::pdl_wait();
    float m_used = -INFINITY, l = 0.f;
    if (g == 0) {
      for (int j = 0; j < nt; ++j) {
        const int sb = j % 3;
        if (!ptx::mbar_wait(&s_full[sb], (j / 3) & 1, lim)) { fail(); break; }
        ptx::tc_fence_after();
        float sv[KT];
        ptx::tmem_ld32(tS + sb * KT + lane_off, *reinterpret_cast<float(*)[32]>(sv));
        ptx::tmem_ld32(tS + sb * KT + 32 + lane_off, *reinterpret_cast<float(*)[32]>(sv + 32));
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&s_empty[sb]);
        const int valid = key_tile(t_begin + j, b, a.P, a.H).valid;   // keys of the tile in range
        // tile maximum of the raw scores (4 independent chains); keys past the tile end masked
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < KT; ++c) {
          if (c >= valid) sv[c] = -INFINITY;
          mq[c & 3] = fmaxf(mq[c & 3], sv[c]);
        }
        const float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * sl2;
        // raise the running maximum only when this tile exceeds it by more than 2^8
        const bool raise = mt > m_used + 8.f;
        const float m_new = raise ? mt : m_used;
        const float corr = raise ? ex2_approx(m_used - m_new) : 1.f;   // 0 on the first tile
        float pq[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[KT / 2];
#pragma unroll
        for (int c = 0; c < KT; c += 2) {
          // p = 2^(s * log2e / sqrt(d) - m): the scale folded into one fma
          const float p0 = ex2_approx(fmaf(sv[c], sl2, -m_new));
          const float p1 = ex2_approx(fmaf(sv[c + 1], sl2, -m_new));
          pq[(c >> 1) & 3] += p0 + p1;
          __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);   // key c in the low half
          pk[c >> 1] = *reinterpret_cast<uint32_t*>(&h2);
        }
        l = l * corr + ((pq[0] + pq[1]) + (pq[2] + pq[3]));
        const int pb = j & 1;
        // P buffer pb is free once PV(j-2) has completed
        if (j >= 2 && !ptx::mbar_wait(&pv_done[pb], ((j - 2) >> 1) & 1, lim)) { fail(); break; }
        const bool rescale = j >= 1 && __any_sync(0xffffffffu, raise);
        // O is stable once PV(j-1) has completed: needed only to rescale it
        if (rescale && !ptx::mbar_wait(&pv_done[pb ^ 1], ((j - 1) >> 1) & 1, lim)) { fail(); break; }
        ptx::tc_fence_after();
        if (rescale) {  // rescale this thread's O row in TMEM (corr = 1 on rows that did not raise)
#pragma unroll 1
          for (int c0 = 0; c0 < DH; c0 += 32) {
            float o[32];
            ptx::tmem_ld32(tO + c0 + lane_off, o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] *= corr;
            tmem_st32(tO + c0 + lane_off, o);
          }
        }
        m_used = m_new;
        ptx::tmem_st32u(tP + pb * (KT / 2) + lane_off, pk);   // P row: column c = keys 2c, 2c + 1
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&p_full[pb]);
      }
      // the last PV (it follows every earlier one on the tensor pipe)
      if (nt > 0 && !*abort_flag && !ptx::mbar_wait(&pv_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, lim)) fail();
      xm[row] = l;
      xm[ROWS + row] = m_used;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");   // the rows' (sum, max) are in shared memory
    ptx::tc_fence_after();
    l = xm[row];
    m_used = xm[ROWS + row];
    const bool aborted = *abort_flag != 0;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    long long slot = 0;
    if (S > 1) {
      // this split's partial -> workspace: O / l as bf16 and (max, sum);
      // attn_t5_combine merges the S splits of every row
      const long long tiles = (long long)gridDim.x * gridDim.z;
      slot = ((long long)b * gridDim.x + blockIdx.x) * S + split;
      float2* wml = reinterpret_cast<float2*>(reinterpret_cast<bf16*>(a.ws) + tiles * S * ROWS * DH);
      if (g == 0) wml[slot * ROWS + row] = make_float2(nt > 0 ? m_used : -INFINITY, l);
    }
    // O / l as bf16 into the idle Q buffer in the store map's layout: box j holds
    // columns [64j, 64j + 64) as 128-byte rows (row = folded row), 16-byte chunk c
    // of row r at chunk c ^ (r % 8); then one tensor store moves the whole tile
    // (whole 128-byte lines instead of one scattered row segment per lane)
#pragma unroll 1
    for (int c0 = g * OH; c0 < g * OH + OH; c0 += 32) {
      float o[32];
      if (nt > 0 && !aborted) {
        ptx::tmem_ld32(tO + c0 + lane_off, o);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = 0.f;
      }
      uint8_t* dst = sQ + (c0 >> 6) * (ROWS * 128) + row * 128;
      const int p0 = (c0 & 63) >> 3;   // first 16-byte chunk of these 32 columns in the box row
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w;
        uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(o[8 * q + 2 * i] * inv, o[8 * q + 2 * i + 1] * inv);
          wp[i] = *reinterpret_cast<uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(dst + (((p0 + q) ^ (row & 7)) << 4)) = w;
      }
    }
    fence_proxy_async_smem();
    asm volatile("bar.sync 1, 256;" ::: "memory");   // the 8 softmax warps staged the tile
    if (warp == 2 && lane == 0) {
      if (S > 1)
        tma_store_3d(&tmO, sQ, 0, (int)(slot * ROWS), 0);
      else   // rows past this sample's H tokens fall outside the map and are dropped
        tma_store_5d(&tmO, sQ, 0, 0, r0 / a.Hq, b, 0);
      tma_store_drain();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (CT > 1) ptx::cluster_sync_all();   // no copy or release targets a CTA that has left
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Merge of the S key splits: a warp per folded query row.  Lane s < S reads
// split s's (max, sum); the weights l_s 2^(m_s - M) / sum_s l_s 2^(m_s - M) are
// shared by shuffles; each lane then sums its DH / 32 columns of the S
// normalised partials (all S loads issued together) and stores the row.
template <int DH>
__global__ void __launch_bounds__(256) attn_t5_combine_kernel(AttnT5Args a, int S) {
  ptx::pdl_launch_dependents();
  constexpr int PER = DH / 32;   // columns per lane: 8, 4 or 2
  const int lane = threadIdx.x & 31;
  const int nrows = a.Hq * a.H;
  const int tiles_x = (nrows + ROWS - 1) / ROWS;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);   // b * nrows + gr
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(a.ts2);
  if (gw >= (long long)a.B * nrows) return;
  const int b = (int)(gw / nrows), gr = (int)(gw % nrows);
  const long long tiles = (long long)tiles_x * a.B;
  const long long slot0 = ((long long)b * tiles_x + gr / ROWS) * S;
  const int row = gr % ROWS;
  const bf16* part = reinterpret_cast<const bf16*>(a.ws);
  const float2* wml = reinterpret_cast<const float2*>(part + tiles * S * ROWS * DH);
  typedef typename std::conditional<PER == 8, uint4, typename std::conditional<PER == 4, uint2, uint32_t>::type>::type V;
  V v[kMaxSplits];   // the partial rows, loaded together with the (max, sum) pairs
#pragma unroll
  for (int sp = 0; sp < kMaxSplits; ++sp)
    if (sp < S) v[sp] = *reinterpret_cast<const V*>(part + ((slot0 + sp) * ROWS + row) * DH + lane * PER);
  const float2 ml = lane < S ? wml[(slot0 + lane) * ROWS + row] : make_float2(-INFINITY, 0.f);
  float mx = ml.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float e = ml.x == -INFINITY ? 0.f : ml.y * exp2f(ml.x - mx);
  const float tot = warp_sum(e);
  const float w = tot > 0.f ? e / tot : 0.f;
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
#pragma unroll
  for (int sp = 0; sp < kMaxSplits; ++sp) {
    if (sp >= S) break;
    const float ws = __shfl_sync(0xffffffffu, w, sp);
    const uint32_t* u = reinterpret_cast<const uint32_t*>(&v[sp]);
#pragma unroll
    for (int q = 0; q < PER / 2; ++q) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[q]));
      acc[2 * q] += ws * f.x;
      acc[2 * q + 1] += ws * f.y;
    }
  }
  V outv;
  uint32_t* op = reinterpret_cast<uint32_t*>(&outv);
#pragma unroll
  for (int q = 0; q < PER / 2; ++q) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
    op[q] = *reinterpret_cast<uint32_t*>(&h2);
  }
  const int t = gr / a.Hq, h = gr % a.Hq;
  *reinterpret_cast<V*>((bf16*)a.out + ((long long)b * a.H + t) * a.ldo + h * DH + lane * PER) = outv;
}

template <int DH>
cudaError_t launch_t5(const AttnT5Args& a, const CUtensorMap* maps, int S, cudaStream_t s, bool pdl) {
  using L = T5Smem<DH>;
  auto kern = attn_t5_kernel<DH>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.Hq * a.H + ROWS - 1) / ROWS, S, a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.ct > 1 ? a.ct : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.ct > 1 ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6],
                                     maps[7], a);
  if (e != cudaSuccess || S == 1) return e;
  const long long warps = (long long)a.B * a.Hq * a.H;
  return launch_k(attn_t5_combine_kernel<DH>, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, pdl, a, S);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode5 = nullptr;

cudaError_t encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box) {
  if (!g_encode5) {
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&g_encode5, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !g_encode5) return cudaErrorNotSupported;
  }
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode5(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool attn_t5_supported(int Dh, int Hq) { return (Dh == 64 || Dh == 128 || Dh == 256) && Hq > 0 && ROWS % Hq == 0; }

int attn_t5_cluster(const AttnT5Args& a) {
  // the row tiles of a sample as one cluster when there are 2 or 4 of them and the
  // Dh/64 column boxes of a key tile split evenly between them
  const int tiles_x = (a.Hq * a.H + ROWS - 1) / ROWS;
  const int boxes = a.Dh / 64;
  return (tiles_x == 2 || tiles_x == 4) && boxes % tiles_x == 0 ? tiles_x : 1;
}

int attn_t5_splits(const AttnT5Args& a, int sm_count, int cap) {
  // at most one CTA per SM and kMaxSplits (or cap) splits; then as few splits as keep
  // that many key tiles per split, so no split is left empty
  const int tiles = (a.Hq * a.H + ROWS - 1) / ROWS * a.B;
  const int ntiles = (a.P + KT - 1) / KT + (a.H + KT - 1) / KT;
  int S = sm_count / (tiles > 0 ? tiles : 1);
  S = S < 1 ? 1 : (S > kMaxSplits ? kMaxSplits : S);
  if (cap > 0 && S > cap) S = cap;
  if (S > ntiles) S = ntiles > 0 ? ntiles : 1;
  const int tps = (ntiles + S - 1) / S;
  return tps > 0 ? (ntiles + tps - 1) / tps : 1;
}

long long attn_t5_workspace_floats(const AttnT5Args& a, int S) {
  if (S == 1) return 0;
  const long long tiles = (long long)(a.Hq * a.H + ROWS - 1) / ROWS * a.B;
  const long long bytes = tiles * S * ROWS * ((long long)a.Dh * 2 + 8);
  return (bytes + 3) / 4;
}

// maps: [0] Q (4-D: 64 columns, Hq heads, B*H tokens, Dh/64 boxes inside qkv), [1] prefix K, [2] prefix V
//       (4-D per sample, rows [0, P) at the sample stride),
//       [3] suffix K, [4] suffix V (3-D: 64 columns, B*H rows of qkv, Dh/64 boxes; based at k_off / v_off),
//       [5] the output tile: S > 1 the workspace partials [slot * 128 + row][Dh], S = 1 the
//           attention output [B][H][Hq][Dh] inside out (row stride ldo),
//       [6], [7] a bound pool's suffix slots of K and V: (64 columns, H rows, B samples of
//           pool_cap rows, Dh/64 boxes) from row P (copies of [1] when no pool is bound)
cudaError_t attn_t5_maps(const AttnT5Args& a, const void* kp, const void* vp, int S, CUtensorMap* maps) {
  const int D = a.Dh;
  const cuuint32_t nbox = (cuuint32_t)(D / 64);
  // Q: (64 columns, heads, tokens, Dh/64 boxes) over the q columns of qkv
  const cuuint64_t qd[4] = {64, (cuuint64_t)a.Hq, (cuuint64_t)a.B * a.H, nbox};
  const cuuint64_t qs[3] = {(cuuint64_t)D * 2, (cuuint64_t)a.ldq * 2, 128};
  const cuuint32_t qb[4] = {64, (cuuint32_t)a.Hq, (cuuint32_t)(ROWS / a.Hq), nbox};
  cudaError_t e = encode(&maps[0], a.qkv, 4, qd, qs, qb);
  if (e != cudaSuccess) return e;
  // K / V tiles: box = one 64-key tile of all Dh/64 column boxes (in a cluster of ct row
  // tiles: 1/ct of them, each CTA's part).  Prefix: (64 columns, P rows, B samples ps rows
  // apart -- ps = P, or a pool's capacity -- Dh/64 boxes)
  const cuuint32_t part = nbox / (cuuint32_t)(a.ct > 1 ? a.ct : 1);
  const cuuint32_t kb[3] = {64, KT, part};
  const cuuint32_t kb4[4] = {64, KT, 1, part};
  const long long prows = a.P > 0 ? a.P : 1, pstride = a.ps > 0 ? a.ps : prows;
  const cuuint64_t pd[4] = {64, (cuuint64_t)prows, (cuuint64_t)a.B, nbox};
  const cuuint64_t ps[3] = {(cuuint64_t)D * 2, (cuuint64_t)pstride * D * 2, 128};
  // with no prefix the prefix maps are never used: point them at the suffix rows
  e = encode(&maps[1], a.P > 0 ? kp : a.qkv, 4, pd, ps, kb4);
  if (e != cudaSuccess) return e;
  e = encode(&maps[2], a.P > 0 ? vp : a.qkv, 4, pd, ps, kb4);
  if (e != cudaSuccess) return e;
  const cuuint64_t sd[3] = {64, (cuuint64_t)a.B * a.H, nbox};
  const cuuint64_t ss[2] = {(cuuint64_t)a.ldq * 2, 128};
  e = encode(&maps[3], static_cast<const bf16*>(a.qkv) + a.k_off, 3, sd, ss, kb);
  if (e != cudaSuccess) return e;
  e = encode(&maps[4], static_cast<const bf16*>(a.qkv) + a.v_off, 3, sd, ss, kb);
  if (e != cudaSuccess) return e;
  if (a.pool_k) {
    const cuuint64_t pd4[4] = {64, (cuuint64_t)a.H, (cuuint64_t)a.B, nbox};
    const cuuint64_t ps4[3] = {(cuuint64_t)D * 2, (cuuint64_t)a.pool_cap * D * 2, 128};
    const cuuint32_t pb4[4] = {64, KT, 1, nbox};
    e = encode(&maps[6], static_cast<const bf16*>(a.pool_k) + (long long)a.P * D, 4, pd4, ps4, pb4);
    if (e != cudaSuccess) return e;
    e = encode(&maps[7], static_cast<const bf16*>(a.pool_v) + (long long)a.P * D, 4, pd4, ps4, pb4);
    if (e != cudaSuccess) return e;
  } else {
    maps[6] = maps[1];
    maps[7] = maps[1];
  }
  if (S > 1) {
    // (64 columns, partial rows, Dh/64 boxes): one 128-row tile per request
    const long long rows = (long long)((a.Hq * a.H + ROWS - 1) / ROWS) * a.B * S * ROWS;
    const cuuint64_t od[3] = {64, (cuuint64_t)rows, nbox};
    const cuuint64_t os[2] = {(cuuint64_t)D * 2, 128};
    const cuuint32_t ob[3] = {64, ROWS, nbox};
    return encode(&maps[5], a.ws, 3, od, os, ob);
  }
  // (64 columns, heads, tokens, samples, Dh/64 boxes): a tile's folded rows in box order,
  // tokens past H outside the map
  const cuuint64_t od[5] = {64, (cuuint64_t)a.Hq, (cuuint64_t)a.H, (cuuint64_t)a.B, nbox};
  const cuuint64_t os[4] = {(cuuint64_t)D * 2, (cuuint64_t)a.ldo * 2, (cuuint64_t)a.H * a.ldo * 2, 128};
  const cuuint32_t ob[5] = {64, (cuuint32_t)a.Hq, (cuuint32_t)(ROWS / a.Hq), 1, nbox};
  return encode(&maps[5], a.out, 5, od, os, ob);
}

cudaError_t attention_t5(const AttnT5Args& a, const CUtensorMap* maps, int S, cudaStream_t s, bool pdl) {
  if (a.B <= 0 || a.Hq * a.H <= 0) return cudaSuccess;
  if (!attn_t5_supported(a.Dh, a.Hq) || S < 1 || S > kMaxSplits) return cudaErrorInvalidValue;
  if (attn_t5_workspace_floats(a, S) > a.ws_floats) return cudaErrorInvalidValue;
  switch (a.Dh) {
    case 64: return launch_t5<64>(a, maps, S, s, pdl);
    case 128: return launch_t5<128>(a, maps, S, s, pdl);
    case 256: return launch_t5<256>(a, maps, S, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace g3
