// Adaptive norms and the small projections at the ends of a denoise step.
//
//  * AdaRMS ("pi0.5 Design", Component contract): y = rms_norm(h) (1 + scale) + shift,
//    scale/shift read from the step's modulation row of the sample.
//  * AdaLayerNorm ("GR00T N1.7", Build-time constants): y = LN(h) (1 + scale) + shift,
//    (scale, shift) for the blocks and (shift, scale) for the final norm.
//  * Step head / tail: action_in_proj fused with the first AdaRMS; final norm +
//    action_out_proj + the device Euler update x += dt * v (vla.cpp Eq. (1)).
//
// One CTA per token row; the row is staged in shared memory in fp32 and the
// reduction is fp32 (the fp32-reduction RMSNorm of "Optimizing GR00T-N1.7
// Training", 3.3).  These kernels move a few hundred KB per step; they are
// latency-bound, not bandwidth-bound.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace g3 {

namespace {

// Normalise the fp32 row in shared memory (in place) and apply the modulation.
template <typename T>
__device__ void norm_row(float* row, int D, int m, const NormArgs& na, float* red) {
  float mean = 0.f;
  if (na.kind == NORM_LN) {
    float s = 0.f;
    for (int i = threadIdx.x; i < D; i += blockDim.x) s += row[i];
    mean = block_sum(s, red) / (float)D;
  }
  float q = 0.f;
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    const float d = row[i] - mean;
    q += d * d;
  }
  const float r = rsqrtf(block_sum(q, red) / (float)D + na.eps);
  const T* mod = na.mod ? (const T*)na.mod + (long long)(m / na.tok) * na.mod_bstride : nullptr;
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    float y = (row[i] - mean) * r;
    if (mod) y = y * (1.f + to_f(mod[na.scale_off + i])) + to_f(mod[na.shift_off + i]);
    row[i] = y;
  }
  __syncthreads();
}

// Residual row m (optionally updated from split-K partials) into shared memory.
// h[m] += gate * sum_s part[s][m]: the sum runs in split order, then one fma
// per element -- the same arithmetic a single-pass epilogue would do.
template <typename T>
__device__ __forceinline__ void load_residual(float* __restrict__ h, int D, int m, const NormArgs& na,
                                              float* row) {
  float* hr = h + (long long)m * D;
  if (!na.part) {
    for (int i = threadIdx.x; i < D; i += blockDim.x) row[i] = hr[i];
    __syncthreads();
    return;
  }
  const T* g = na.gate ? (const T*)na.gate + (long long)(m / na.tok) * na.mod_bstride : nullptr;
  // 4 elements per thread, the (<= 16) partial loads issued together, summed in split order
  for (int i = threadIdx.x * 4; i < D; i += blockDim.x * 4) {
    float4 v[16];
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < na.part_S) v[s] = *reinterpret_cast<const float4*>(na.part + ((long long)s * na.part_M + m) * D + i);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < na.part_S) {
        acc.x += v[s].x;
        acc.y += v[s].y;
        acc.z += v[s].z;
        acc.w += v[s].w;
      }
    float4 hv = *reinterpret_cast<const float4*>(hr + i);
    float gg[4] = {1.f, 1.f, 1.f, 1.f};
    if (g) {
#pragma unroll
      for (int q = 0; q < 4; ++q) gg[q] = to_f(g[i + q]);
    }
    hv.x += gg[0] * acc.x;
    hv.y += gg[1] * acc.y;
    hv.z += gg[2] * acc.z;
    hv.w += gg[3] * acc.w;
    *reinterpret_cast<float4*>(hr + i) = hv;
    row[i] = hv.x;
    row[i + 1] = hv.y;
    row[i + 2] = hv.z;
    row[i + 3] = hv.w;
  }
  __syncthreads();
}

template <typename T>
__global__ void adanorm_kernel(float* __restrict__ h, int D, T* __restrict__ out, NormArgs na) {
  ptx::pdl_launch_dependents();
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(na.ts);
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + D;
  const int m = blockIdx.x;
  load_residual<T>(h, D, m, na, row);
  norm_row<T>(row, D, m, na, red);
  T* o = out + (long long)m * D;
  for (int i = threadIdx.x; i < D; i += blockDim.x) o[i] = from_f<T>(row[i]);
}

template <typename T>
__global__ void expert_in_kernel(const float* __restrict__ x, int A, const T* __restrict__ w_in,
                                 const float* __restrict__ b_in, float* __restrict__ h, int D,
                                 T* __restrict__ out, NormArgs na) {
  ptx::pdl_launch_dependents();
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(na.ts);
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + D;
  float* xs = sm + D + 33;
  const int m = blockIdx.x;
  for (int a = threadIdx.x; a < A; a += blockDim.x) xs[a] = x[(long long)m * A + a];
  __syncthreads();
  float* hr = h + (long long)m * D;
  for (int f = threadIdx.x; f < D; f += blockDim.x) {
    const T* w = w_in + (long long)f * A;
    float acc = b_in[f];
    for (int a = 0; a < A; ++a) acc = fmaf(xs[a], to_f(w[a]), acc);
    row[f] = acc;
    hr[f] = acc;
  }
  __syncthreads();
  norm_row<T>(row, D, m, na, red);
  T* o = out + (long long)m * D;
  for (int i = threadIdx.x; i < D; i += blockDim.x) o[i] = from_f<T>(row[i]);
}

template <typename T>
__global__ void out_euler_kernel(float* __restrict__ h, int D, int H, int ro, int tok,
                                 const T* __restrict__ w_out, const float* __restrict__ b_out,
                                 int A, NormArgs na, float* __restrict__ x,
                                 const float* __restrict__ dts, int k, int do_euler,
                                 float* __restrict__ v_out) {
  ptx::pdl_launch_dependents();
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(na.ts);
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + D;
  const int m = blockIdx.x;                       // action row b * H + j
  const long long hrow = (long long)(m / H) * tok + ro + m % H;
  // the modulation row is indexed per sample: pass the residual row so m / tok = b
  load_residual<T>(h, D, (int)hrow, na, row);
  norm_row<T>(row, D, (int)hrow, na, red);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int a = warp; a < A; a += nw) {
    const T* w = w_out + (long long)a * D;
    float acc = 0.f;
    for (int i = lane; i < D; i += 32) acc = fmaf(row[i], to_f(w[i]), acc);
    acc = warp_sum(acc);
    if (lane == 0) {
      const float v = acc + b_out[a];
      if (v_out) v_out[(long long)m * A + a] = v;
      if (do_euler) x[(long long)m * A + a] += dts[k] * v;
    }
  }
}

template <typename T>
__global__ void dit_in_kernel(const float* __restrict__ x, int A, const T* __restrict__ w1,
                              const float* __restrict__ b1, T* __restrict__ a_out, int D, int M,
                              const float* __restrict__ state, int ns, int tok,
                              float* __restrict__ h, unsigned long long* ts) {
  ptx::pdl_launch_dependents();
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(ts);
  extern __shared__ float xs[];
  const int blk = blockIdx.x;
  if (blk >= M) {  // state-token rows: copy the bound embedding into the residual stream
    const int idx = blk - M, b = idx / ns, j = idx % ns;
    const float* src = state + ((long long)b * ns + j) * D;
    float* dst = h + ((long long)b * tok + j) * D;
    for (int i = threadIdx.x; i < D; i += blockDim.x) dst[i] = src[i];
    return;
  }
  for (int a = threadIdx.x; a < A; a += blockDim.x) xs[a] = x[(long long)blk * A + a];
  __syncthreads();
  for (int f = threadIdx.x; f < D; f += blockDim.x) {
    const T* w = w1 + (long long)f * A;
    float acc = b1[f];
    for (int a = 0; a < A; ++a) acc = fmaf(xs[a], to_f(w[a]), acc);
    a_out[(long long)blk * D + f] = from_f<T>(acc);
  }
}

// ---------------- many rows: a warp per row, the row in registers ----------------
// Lane l of the warp that owns a row holds the elements (k * 32 + l) * 4 .. + 3
// for k < D / 128 (D a multiple of 128, at most 128 * kMaxQuads), so every
// load and store of the warp covers 512 contiguous bytes and the reductions
// are warp shuffles with no block barrier.  The modulation rows (written when
// the schedule was set, before any kernel of the step) are fetched before
// the programmatic-launch wait; the residual and split-K partials after it.
constexpr int kMaxQuads = 12;   // D <= 1536
constexpr int kNormRowsPerCta = 4;

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}
// Raw (undecoded) quad of activations: 8 bytes of bf16 or 16 of fp32.
template <typename T> struct RawQuad;
template <> struct RawQuad<bf16> {
  typedef uint2 type;
  static __device__ __forceinline__ uint2 load(const bf16* p) { return *reinterpret_cast<const uint2*>(p); }
  static __device__ __forceinline__ float4 f(uint2 u) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
};
template <> struct RawQuad<float> {
  typedef float4 type;
  static __device__ __forceinline__ float4 load(const float* p) { return *reinterpret_cast<const float4*>(p); }
  static __device__ __forceinline__ float4 f(float4 u) { return u; }
};

__device__ __forceinline__ void add4(float4& a, const float4 b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

// Residual row into registers: x = h[row] (+ gate * sum of the split-K partials,
// in split order).  NS >= 0: that many partials, all loads issued together;
// NS < 0: na.part_S of them, one split at a time.  ``write_back`` stores the
// updated residual row.
template <typename T, int NS, int NQ>
__device__ __forceinline__ void warp_load_residual(float* __restrict__ h, long long row, int nq, int lane,
                                                   const NormArgs& na, float4 (&x)[NQ], int D,
                                                   bool write_back) {
  typedef RawQuad<T> RQ;
  float* hr = h + row * D;
#pragma unroll
  for (int k = 0; k < NQ; ++k)
    if (k < nq) x[k] = ld4(hr + (k * 32 + lane) * 4);
  if (NS == 0 || !na.part) return;
  const T* g = na.gate ? (const T*)na.gate + (row / na.tok) * na.mod_bstride : nullptr;
  typename RQ::type gq[NQ];
  float4 acc[NQ];
  if (NS > 0) {
    float4 v[NS > 0 ? NS : 1][NQ];
#pragma unroll
    for (int sp = 0; sp < (NS > 0 ? NS : 1); ++sp)
#pragma unroll
      for (int k = 0; k < NQ; ++k)
        if (k < nq) v[sp][k] = ld4(na.part + ((long long)sp * na.part_M + row) * D + (k * 32 + lane) * 4);
#pragma unroll
    for (int k = 0; k < NQ; ++k)
      if (k < nq && g) gq[k] = RQ::load(g + (k * 32 + lane) * 4);
#pragma unroll
    for (int k = 0; k < NQ; ++k)
      if (k < nq) {
        acc[k] = v[0][k];
#pragma unroll
        for (int sp = 1; sp < (NS > 0 ? NS : 1); ++sp) add4(acc[k], v[sp][k]);
      }
  } else {
#pragma unroll
    for (int k = 0; k < NQ; ++k)
      if (k < nq && g) gq[k] = RQ::load(g + (k * 32 + lane) * 4);
#pragma unroll
    for (int k = 0; k < NQ; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < na.part_S; ++sp)
#pragma unroll
      for (int k = 0; k < NQ; ++k)
        if (k < nq) add4(acc[k], ld4(na.part + ((long long)sp * na.part_M + row) * D + (k * 32 + lane) * 4));
  }
#pragma unroll
  for (int k = 0; k < NQ; ++k)
    if (k < nq) {
      const float4 gg = g ? RQ::f(gq[k]) : make_float4(1.f, 1.f, 1.f, 1.f);
      x[k].x = fmaf(gg.x, acc[k].x, x[k].x);
      x[k].y = fmaf(gg.y, acc[k].y, x[k].y);
      x[k].z = fmaf(gg.z, acc[k].z, x[k].z);
      x[k].w = fmaf(gg.w, acc[k].w, x[k].w);
      if (write_back) st4(hr + (k * 32 + lane) * 4, x[k]);
    }
}

// x <- norm(x) * (1 + scale) + shift over the row held by the warp (mod quads
// already loaded; has_mod false: plain norm).
template <typename T, int NQ>
__device__ __forceinline__ void warp_norm_mod(float4 (&x)[NQ], int nq, int D, const NormArgs& na,
                                              const typename RawQuad<T>::type (&sc)[NQ],
                                              const typename RawQuad<T>::type (&sh)[NQ], bool has_mod) {
  typedef RawQuad<T> RQ;
  float mean = 0.f;
  if (na.kind == NORM_LN) {
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NQ; ++k)
      if (k < nq) s += (x[k].x + x[k].y) + (x[k].z + x[k].w);
    mean = warp_sum(s) / (float)D;
  }
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < NQ; ++k)
    if (k < nq) {
      const float a = x[k].x - mean, b = x[k].y - mean, c = x[k].z - mean, d = x[k].w - mean;
      q += (a * a + b * b) + (c * c + d * d);
    }
  const float r = rsqrtf(warp_sum(q) / (float)D + na.eps);
#pragma unroll
  for (int k = 0; k < NQ; ++k)
    if (k < nq) {
      float4 y = make_float4((x[k].x - mean) * r, (x[k].y - mean) * r, (x[k].z - mean) * r, (x[k].w - mean) * r);
      if (has_mod) {
        const float4 a = RQ::f(sc[k]), b = RQ::f(sh[k]);
        y.x = y.x * (1.f + a.x) + b.x;
        y.y = y.y * (1.f + a.y) + b.y;
        y.z = y.z * (1.f + a.z) + b.z;
        y.w = y.w * (1.f + a.w) + b.w;
      }
      x[k] = y;
    }
}

template <typename T, int NQ>
__device__ __forceinline__ void warp_load_mod(const NormArgs& na, long long row, int nq, int lane,
                                              typename RawQuad<T>::type (&sc)[NQ],
                                              typename RawQuad<T>::type (&sh)[NQ]) {
  if (!na.mod) return;
  const T* mod = (const T*)na.mod + (row / na.tok) * na.mod_bstride;
#pragma unroll
  for (int k = 0; k < NQ; ++k)
    if (k < nq) {
      sc[k] = RawQuad<T>::load(mod + na.scale_off + (k * 32 + lane) * 4);
      sh[k] = RawQuad<T>::load(mod + na.shift_off + (k * 32 + lane) * 4);
    }
}

template <typename T, int NS, int NQ>
__global__ void __launch_bounds__(32 * kNormRowsPerCta) adanorm_rows_kernel(float* __restrict__ h, int D, int M,
                                                                          T* __restrict__ out, NormArgs na) {
  ptx::pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * kNormRowsPerCta + (threadIdx.x >> 5);
  const int nq = D >> 7;
  typename RawQuad<T>::type sc[NQ], sh[NQ];
  if (m < M) warp_load_mod<T, NQ>(na, m, nq, lane, sc, sh);
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(na.ts);
  if (m >= M) return;
  float4 x[NQ];
  warp_load_residual<T, NS, NQ>(h, m, nq, lane, na, x, D, true);
  warp_norm_mod<T, NQ>(x, nq, D, na, sc, sh, na.mod != nullptr);
  T* o = out + (long long)m * D;
#pragma unroll
  for (int k = 0; k < NQ; ++k)
    if (k < nq) st4(o + (k * 32 + lane) * 4, x[k]);
}

// Few rows: a CTA per row, D / 4 threads, one quad of the row per thread kept
// in registers.  The modulation (and gate) quads are fetched before the
// programmatic-launch wait; the residual quad and all S split-K partial quads
// after it, in one round trip.
template <typename T>
__global__ void __launch_bounds__(512) adanorm_cta_kernel(float* __restrict__ h, int D, T* __restrict__ out,
                                                          NormArgs na) {
  ptx::pdl_launch_dependents();
  __shared__ float red[33];
  typedef RawQuad<T> RQ;
  const int m = blockIdx.x;
  const int i = threadIdx.x * 4;
  typename RQ::type sc, sh, gq;
  const long long mrow = (long long)(m / na.tok) * na.mod_bstride;
  if (na.mod) {
    sc = RQ::load((const T*)na.mod + mrow + na.scale_off + i);
    sh = RQ::load((const T*)na.mod + mrow + na.shift_off + i);
  }
  if (na.part && na.gate) gq = RQ::load((const T*)na.gate + mrow + i);
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(na.ts);
  float* hr = h + (long long)m * D + i;
  float4 x = ld4(hr);
  if (na.part) {
    float4 v[16];
#pragma unroll
    for (int sp = 0; sp < 16; ++sp)
      if (sp < na.part_S) v[sp] = ld4(na.part + ((long long)sp * na.part_M + m) * D + i);
    float4 acc = v[0];
#pragma unroll
    for (int sp = 1; sp < 16; ++sp)
      if (sp < na.part_S) add4(acc, v[sp]);
    const float4 g = na.gate ? RQ::f(gq) : make_float4(1.f, 1.f, 1.f, 1.f);
    x.x = fmaf(g.x, acc.x, x.x);
    x.y = fmaf(g.y, acc.y, x.y);
    x.z = fmaf(g.z, acc.z, x.z);
    x.w = fmaf(g.w, acc.w, x.w);
    st4(hr, x);
  }
  float mean = 0.f;
  if (na.kind == NORM_LN) mean = block_sum((x.x + x.y) + (x.z + x.w), red) / (float)D;
  const float a = x.x - mean, b = x.y - mean, c = x.z - mean, d = x.w - mean;
  const float r = rsqrtf(block_sum((a * a + b * b) + (c * c + d * d), red) / (float)D + na.eps);
  float4 y = make_float4(a * r, b * r, c * r, d * r);
  if (na.mod) {
    const float4 s4 = RQ::f(sc), t4 = RQ::f(sh);
    y.x = y.x * (1.f + s4.x) + t4.x;
    y.y = y.y * (1.f + s4.y) + t4.y;
    y.z = y.z * (1.f + s4.z) + t4.z;
    y.w = y.w * (1.f + s4.w) + t4.w;
  }
  st4(out + (long long)m * D + i, y);
}

// Eight values per call: w[0..7] = p[0..7] (p 16-byte aligned).
__device__ __forceinline__ void ld8(const bf16* p, float (&w)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t r[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r[i]));
    w[2 * i] = f.x;
    w[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void ld8(const float* p, float (&w)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// Step head for many rows: kInRows token rows per CTA, D / 4 threads, thread t
// owns features 4t .. 4t + 3 of every row, so each CTA reads W_in once for
// kInRows rows.  h = x W_in^T + b_in (fp32, written), out = AdaRMS(h).
constexpr int kInRows = 8;

template <typename T>
__global__ void __launch_bounds__(256) expert_in_rows_kernel(const float* __restrict__ x, int A,
                                                             const T* __restrict__ w_in,
                                                             const float* __restrict__ b_in,
                                                             float* __restrict__ h, int D, int M,
                                                             T* __restrict__ out, NormArgs na) {
  ptx::pdl_launch_dependents();
  __shared__ float xs[kInRows][64];
  __shared__ float red[kInRows][9];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nw = blockDim.x >> 5;
  const int f0 = 4 * t;
  const int m0 = blockIdx.x * kInRows;
  typedef RawQuad<T> RQ;
  typename RQ::type sc[kInRows], sh[kInRows];
  const float4 bias = *reinterpret_cast<const float4*>(b_in + f0);
#pragma unroll
  for (int r = 0; r < kInRows; ++r)
    if (m0 + r < M && na.mod) {
      const T* mod = (const T*)na.mod + (long long)((m0 + r) / na.tok) * na.mod_bstride;
      sc[r] = RQ::load(mod + na.scale_off + f0);
      sh[r] = RQ::load(mod + na.shift_off + f0);
    }
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(na.ts);
  for (int i = t; i < kInRows * A; i += blockDim.x) {
    const int r = i / A, a = i % A;
    xs[r][a] = m0 + r < M ? x[(long long)(m0 + r) * A + a] : 0.f;
  }
  __syncthreads();
  float acc[kInRows][4];
#pragma unroll
  for (int r = 0; r < kInRows; ++r) {
    acc[r][0] = bias.x;
    acc[r][1] = bias.y;
    acc[r][2] = bias.z;
    acc[r][3] = bias.w;
  }
  for (int a0 = 0; a0 < A; a0 += 8) {
    float w[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j) ld8(w_in + (long long)(f0 + j) * A + a0, w[j]);
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int r = 0; r < kInRows; ++r) {
        const float xv = xs[r][a0 + a];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[r][j] = fmaf(xv, w[j][a], acc[r][j]);
      }
  }
  // sum of squares of each row over the CTA
#pragma unroll
  for (int r = 0; r < kInRows; ++r) {
    const float q = warp_sum((acc[r][0] * acc[r][0] + acc[r][1] * acc[r][1]) +
                             (acc[r][2] * acc[r][2] + acc[r][3] * acc[r][3]));
    if (lane == 0) red[r][warp] = q;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kInRows; ++r) {
    const int m = m0 + r;
    if (m >= M) break;
    float q = 0.f;
    for (int w = 0; w < nw; ++w) q += red[r][w];
    const float rs = rsqrtf(q / (float)D + na.eps);
    st4(h + (long long)m * D + f0, make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]));
    float4 y = make_float4(acc[r][0] * rs, acc[r][1] * rs, acc[r][2] * rs, acc[r][3] * rs);
    if (na.mod) {
      const float4 a = RQ::f(sc[r]), b = RQ::f(sh[r]);
      y.x = y.x * (1.f + a.x) + b.x;
      y.y = y.y * (1.f + a.y) + b.y;
      y.z = y.z * (1.f + a.z) + b.z;
      y.w = y.w * (1.f + a.w) + b.w;
    }
    st4(out + (long long)m * D + f0, y);
  }
}

// v[a] for a = lane after a butterfly reduce-scatter: lane l enters with 32
// partial dot products p[0..31]; 31 shuffles leave lane a holding sum_l p_l[a].
__device__ __forceinline__ float reduce_scatter32(float (&p)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < o; ++j) {
      const float send = hi ? p[j] : p[j + o];
      const float keep = hi ? p[j + o] : p[j];
      p[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return p[0];
}

// Step tail for many rows: a warp per action row -- residual (+ pending
// partials), final norm, v = y W_out^T + b_out (A <= 32, reduce-scatter so
// lane a owns v[a]) and the Euler update.  The residual row is not written
// back: nothing reads it before the next step's head overwrites it.
template <typename T, int NS, int NQ>
__global__ void __launch_bounds__(32 * kNormRowsPerCta) out_euler_rows_kernel(
    float* __restrict__ h, int D, int M, int H, int ro, const T* __restrict__ w_out,
    const float* __restrict__ b_out, int A, NormArgs na, float* __restrict__ x, const float* __restrict__ dts,
    int k, int do_euler, float* __restrict__ v_out) {
  ptx::pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * kNormRowsPerCta + (threadIdx.x >> 5);
  const int nq = D >> 7;
  const long long row = (long long)(m / H) * na.tok + ro + m % H;
  typename RawQuad<T>::type sc[NQ], sh[NQ];
  if (m < M) warp_load_mod<T, NQ>(na, row, nq, lane, sc, sh);
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(na.ts);
  if (m >= M) return;
  float4 y[NQ];
  warp_load_residual<T, NS, NQ>(h, row, nq, lane, na, y, D, false);
  warp_norm_mod<T, NQ>(y, nq, D, na, sc, sh, na.mod != nullptr);
  float p[32];
#pragma unroll
  for (int a = 0; a < 32; ++a) {
    float s = 0.f;
    if (a < A) {
      const T* w = w_out + (long long)a * D;
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        if (q < nq) {
          const float4 wv = ld4(w + (q * 32 + lane) * 4);
          s = fmaf(y[q].x, wv.x, s);
          s = fmaf(y[q].y, wv.y, s);
          s = fmaf(y[q].z, wv.z, s);
          s = fmaf(y[q].w, wv.w, s);
        }
    }
    p[a] = s;
  }
  const float dot = reduce_scatter32(p, lane);
  if (lane < A) {
    const float v = dot + b_out[lane];
    if (v_out) v_out[(long long)m * A + lane] = v;
    if (do_euler) x[(long long)m * A + lane] += dts[k] * v;
  }
}

inline int threads_for(int D) { return D <= 512 ? 128 : 256; }

// Token rows from which the multi-row kernels replace the CTA-per-row ones.
constexpr int kRowsMin = 256;

}  // namespace

// The warp-per-row kernels want D a multiple of 128 (at most 128 * kMaxQuads)
// and 16-byte aligned rows of h, the partials and the output.
static bool rows_ok(int D, const void* p0, const void* p1 = nullptr, const void* p2 = nullptr) {
  auto al = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  return D % 128 == 0 && D <= 128 * kMaxQuads && al(p0) && al(p1) && al(p2);
}
// The modulation and gate quads: 16-byte aligned rows and offsets in whole quads of 16 bytes.
static bool mod_ok(const NormArgs& na, size_t es) {
  auto al = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  const long long q = 16 / (long long)es;
  return al(na.mod) && al(na.gate) && na.mod_bstride % q == 0 && na.scale_off % q == 0 && na.shift_off % q == 0;
}

template <typename T, int NQ, template <typename, int, int> class K, typename... Args>
static cudaError_t launch_rows_nq(int blocks, int S, bool has_part, cudaStream_t s, bool pdl, Args... args) {
  const int threads = 32 * kNormRowsPerCta;
  if (!has_part) return launch_k(K<T, 0, NQ>::fn, blocks, threads, 0, s, pdl, args...);
  switch (S) {
    case 1: return launch_k(K<T, 1, NQ>::fn, blocks, threads, 0, s, pdl, args...);
    case 2: return launch_k(K<T, 2, NQ>::fn, blocks, threads, 0, s, pdl, args...);
    default: return launch_k(K<T, -1, NQ>::fn, blocks, threads, 0, s, pdl, args...);
  }
}
// NQ (quads per lane) 8 up to D = 1024, else 12; S partials unrolled for 1 and 2.
template <typename T, template <typename, int, int> class K, typename... Args>
static cudaError_t launch_rows(int D, int blocks, int S, bool has_part, cudaStream_t s, bool pdl, Args... args) {
  if (D <= 1024) return launch_rows_nq<T, 8, K>(blocks, S, has_part, s, pdl, args...);
  return launch_rows_nq<T, 12, K>(blocks, S, has_part, s, pdl, args...);
}
template <typename T, int NS, int NQ> struct AdanormRows {
  static constexpr auto fn = adanorm_rows_kernel<T, NS, NQ>;
};
template <typename T, int NS, int NQ> struct OutEulerRows {
  static constexpr auto fn = out_euler_rows_kernel<T, NS, NQ>;
};

cudaError_t adanorm(DType dt, float* h, int D, int M, void* out, NormArgs na, cudaStream_t s, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (M >= kRowsMin && rows_ok(D, h, out, na.part) && mod_ok(na, dt == DT_F32 ? 4 : 2)) {  // warp per row
    const int blocks = (M + kNormRowsPerCta - 1) / kNormRowsPerCta;
    if (dt == DT_F32)
      return launch_rows<float, AdanormRows>(D, blocks, na.part_S, na.part != nullptr, s, pdl, h, D, M, (float*)out,
                                             na);
    return launch_rows<bf16, AdanormRows>(D, blocks, na.part_S, na.part != nullptr, s, pdl, h, D, M, (bf16*)out, na);
  }
  if (D % 128 == 0 && D <= 2048 && (!na.part || na.part_S <= 16) && rows_ok(D, h, out, na.part) &&
      mod_ok(na, dt == DT_F32 ? 4 : 2)) {  // few rows: a CTA per row, the row in registers
    if (dt == DT_F32) return launch_k(adanorm_cta_kernel<float>, M, D / 4, 0, s, pdl, h, D, (float*)out, na);
    return launch_k(adanorm_cta_kernel<bf16>, M, D / 4, 0, s, pdl, h, D, (bf16*)out, na);
  }
  const size_t smem = (D + 33) * sizeof(float);
  if (dt == DT_F32)
    return launch_k(adanorm_kernel<float>, M, threads_for(D), smem, s, pdl, h, D, (float*)out, na);
  return launch_k(adanorm_kernel<bf16>, M, threads_for(D), smem, s, pdl, h, D, (bf16*)out, na);
}

cudaError_t expert_in(DType dt, const float* x, int A, const void* w_in, const float* b_in,
                      float* h, int D, int M, void* out, NormArgs na, cudaStream_t s, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (M >= kRowsMin && D % 128 == 0 && D <= 1024 && A % 8 == 0 && A <= 64 && rows_ok(D, h, out, w_in) &&
      rows_ok(D, b_in) && mod_ok(na, dt == DT_F32 ? 4 : 2)) {
    const int blocks = (M + kInRows - 1) / kInRows;
    if (dt == DT_F32)
      return launch_k(expert_in_rows_kernel<float>, blocks, D / 4, 0, s, pdl, x, A, (const float*)w_in, b_in, h,
                      D, M, (float*)out, na);
    return launch_k(expert_in_rows_kernel<bf16>, blocks, D / 4, 0, s, pdl, x, A, (const bf16*)w_in, b_in, h, D,
                    M, (bf16*)out, na);
  }
  const size_t smem = (D + 33 + A) * sizeof(float);
  if (dt == DT_F32)
    return launch_k(expert_in_kernel<float>, M, threads_for(D), smem, s, pdl, x, A, (const float*)w_in,
                    b_in, h, D, (float*)out, na);
  return launch_k(expert_in_kernel<bf16>, M, threads_for(D), smem, s, pdl, x, A, (const bf16*)w_in, b_in,
                  h, D, (bf16*)out, na);
}

cudaError_t out_euler(DType dt, float* h, int D, int M, int H, int ro, const void* w_out,
                      const float* b_out, int A, NormArgs na, float* x, const float* dts, int k,
                      int do_euler, float* v_out, cudaStream_t s, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (M >= kRowsMin && A <= 32 && rows_ok(D, h, w_out, na.part) && mod_ok(na, dt == DT_F32 ? 4 : 2)) {
    const int blocks = (M + kNormRowsPerCta - 1) / kNormRowsPerCta;
    if (dt == DT_F32)
      return launch_rows<float, OutEulerRows>(D, blocks, na.part_S, na.part != nullptr, s, pdl, h, D, M, H, ro,
                                              (const float*)w_out, b_out, A, na, x, dts, k, do_euler, v_out);
    return launch_rows<bf16, OutEulerRows>(D, blocks, na.part_S, na.part != nullptr, s, pdl, h, D, M, H, ro,
                                           (const bf16*)w_out, b_out, A, na, x, dts, k, do_euler, v_out);
  }
  const size_t smem = (D + 33) * sizeof(float);
  const int tok = na.tok;
  if (dt == DT_F32)
    return launch_k(out_euler_kernel<float>, M, 256, smem, s, pdl, h, D, H, ro, tok, (const float*)w_out,
                    b_out, A, na, x, dts, k, do_euler, v_out);
  return launch_k(out_euler_kernel<bf16>, M, 256, smem, s, pdl, h, D, H, ro, tok, (const bf16*)w_out, b_out,
                  A, na, x, dts, k, do_euler, v_out);
}

cudaError_t dit_in(DType dt, const float* x, int A, const void* w1, const float* b1, void* a_out,
                   int D, int M, const float* state, int ns, int tok, int B, float* h,
                   cudaStream_t s, bool pdl, unsigned long long* ts) {
  const int blocks = M + (state ? B * ns : 0);
  if (blocks <= 0) return cudaSuccess;
  const size_t smem = A * sizeof(float);
  if (dt == DT_F32)
    return launch_k(dit_in_kernel<float>, blocks, threads_for(D), smem, s, pdl, x, A, (const float*)w1, b1,
                    (float*)a_out, D, M, state, ns, tok, h, ts);
  return launch_k(dit_in_kernel<bf16>, blocks, threads_for(D), smem, s, pdl, x, A, (const bf16*)w1, b1,
                  (bf16*)a_out, D, M, state, ns, tok, h, ts);
}

}  // namespace g3
