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
                              float* __restrict__ h) {
  ptx::pdl_launch_dependents();
  ptx::pdl_wait();
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

// Warp per row, for many rows: the row lives in registers (D/64 float2 per
// lane), reductions are warp shuffles, no block barriers; 8 rows per CTA.
constexpr int kRowsPerCta = 8;
constexpr int kMaxPairsPerLane = 16;  // D <= 1024

template <typename T>
__global__ void __launch_bounds__(256, 2) adanorm_rows_kernel(float* __restrict__ h, int D, int M,
                                                           T* __restrict__ out, NormArgs na) {
  ptx::pdl_launch_dependents();
  ptx::pdl_wait();
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (m >= M) return;
  const int np = D / 64;  // float2 per lane
  float* hr = h + (long long)m * D;
  float2 x[kMaxPairsPerLane];
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k)
    if (k < np) x[k] = *reinterpret_cast<const float2*>(hr + (k * 32 + lane) * 2);
  if (na.part) {  // h += gate * sum_s part[s] (split order), written back
    const T* g = na.gate ? (const T*)na.gate + (long long)(m / na.tok) * na.mod_bstride : nullptr;
    float2 acc[kMaxPairsPerLane];
#pragma unroll
    for (int k = 0; k < kMaxPairsPerLane; ++k) acc[k] = make_float2(0.f, 0.f);
    for (int sp = 0; sp < na.part_S; ++sp) {
      const float* pr = na.part + ((long long)sp * na.part_M + m) * D;
#pragma unroll
      for (int k = 0; k < kMaxPairsPerLane; ++k)
        if (k < np) {
          const float2 v = *reinterpret_cast<const float2*>(pr + (k * 32 + lane) * 2);
          acc[k].x += v.x;
          acc[k].y += v.y;
        }
    }
#pragma unroll
    for (int k = 0; k < kMaxPairsPerLane; ++k)
      if (k < np) {
        const int i = (k * 32 + lane) * 2;
        const float g0 = g ? to_f(g[i]) : 1.f, g1 = g ? to_f(g[i + 1]) : 1.f;
        x[k].x += g0 * acc[k].x;
        x[k].y += g1 * acc[k].y;
        *reinterpret_cast<float2*>(hr + i) = x[k];
      }
  }
  float mean = 0.f;
  if (na.kind == NORM_LN) {
    float sacc = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxPairsPerLane; ++k)
      if (k < np) sacc += x[k].x + x[k].y;
    mean = warp_sum(sacc) / (float)D;
  }
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k)
    if (k < np) {
      const float a = x[k].x - mean, b = x[k].y - mean;
      q += a * a + b * b;
    }
  const float r = rsqrtf(warp_sum(q) / (float)D + na.eps);
  const T* mod = na.mod ? (const T*)na.mod + (long long)(m / na.tok) * na.mod_bstride : nullptr;
  T* o = out + (long long)m * D;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k)
    if (k < np) {
      const int i = (k * 32 + lane) * 2;
      float y0 = (x[k].x - mean) * r, y1 = (x[k].y - mean) * r;
      if (mod) {
        y0 = y0 * (1.f + to_f(mod[na.scale_off + i])) + to_f(mod[na.shift_off + i]);
        y1 = y1 * (1.f + to_f(mod[na.scale_off + i + 1])) + to_f(mod[na.shift_off + i + 1]);
      }
      o[i] = from_f<T>(y0);
      o[i + 1] = from_f<T>(y1);
    }
}

inline int threads_for(int D) { return D <= 512 ? 128 : 256; }

}  // namespace

cudaError_t adanorm(DType dt, float* h, int D, int M, void* out, NormArgs na, cudaStream_t s, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (M > 1024 && D <= 64 * kMaxPairsPerLane) {  // many rows: warp per row
    const int blocks = (M + kRowsPerCta - 1) / kRowsPerCta;
    if (dt == DT_F32)
      return launch_k(adanorm_rows_kernel<float>, blocks, 32 * kRowsPerCta, 0, s, pdl, h, D, M, (float*)out, na);
    return launch_k(adanorm_rows_kernel<bf16>, blocks, 32 * kRowsPerCta, 0, s, pdl, h, D, M, (bf16*)out, na);
  }
  const size_t smem = (D + 33) * sizeof(float);
  if (dt == DT_F32)
    return launch_k(adanorm_kernel<float>, M, threads_for(D), smem, s, pdl, h, D, (float*)out, na);
  return launch_k(adanorm_kernel<bf16>, M, threads_for(D), smem, s, pdl, h, D, (bf16*)out, na);
}

cudaError_t expert_in(DType dt, const float* x, int A, const void* w_in, const float* b_in,
                      float* h, int D, int M, void* out, NormArgs na, cudaStream_t s, bool pdl) {
  if (M <= 0) return cudaSuccess;
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
                   cudaStream_t s, bool pdl) {
  const int blocks = M + (state ? B * ns : 0);
  if (blocks <= 0) return cudaSuccess;
  const size_t smem = A * sizeof(float);
  if (dt == DT_F32)
    return launch_k(dit_in_kernel<float>, blocks, threads_for(D), smem, s, pdl, x, A, (const float*)w1, b1,
                    (float*)a_out, D, M, state, ns, tok, h);
  return launch_k(dit_in_kernel<bf16>, blocks, threads_for(D), smem, s, pdl, x, A, (const bf16*)w1, b1,
                  (bf16*)a_out, D, M, state, ns, tok, h);
}

}  // namespace g3
