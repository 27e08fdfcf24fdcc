// Device-side helpers shared by the kernels of the denoise loop (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace g3 {

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024); every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* scratch /* >= 33 floats */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float t = lane < nw ? scratch[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) scratch[32] = t;
  }
  __syncthreads();
  return scratch[32];
}

// swish(x) = x * sigmoid(x)
__device__ __forceinline__ float swishf(float x) { return x / (1.f + expf(-x)); }

// GeLU, tanh approximation: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
__device__ __forceinline__ float gelu_tanhf(float x) {
  const float c = 0.7978845608028654f;
  return 0.5f * x * (1.f + tanhf(c * (x + 0.044715f * x * x * x)));
}

// The same GeLU with the hardware tanh.approx.f32 instruction (relative error
// about 2^-11, below the bf16 rounding of its output); used on the bf16 path.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float gelu_tanh_fast(float x) {
  const float c = 0.7978845608028654f;
  return 0.5f * x * (1.f + tanh_approx(c * (x + 0.044715f * x * x * x)));
}

// 2^x with the hardware ex2.approx instruction (relative error about 2^-22).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// GeLU used by the epilogues: accurate tanh for fp32 activations, hardware tanh for bf16.
template <typename T> __device__ __forceinline__ float gelu_act(float x);
template <> __device__ __forceinline__ float gelu_act<float>(float x) { return gelu_tanhf(x); }
template <> __device__ __forceinline__ float gelu_act<bf16>(float x) { return gelu_tanh_fast(x); }

// Dependency-release stamp for timing a launch inside the step's chain: the
// global timer (ns) at the moment this grid's programmatic dependency wait
// returned, i.e. when the previous kernel of the stream had completed.  One
// store by the calling thread of the first CTA; ``ts`` null (the default):
// nothing.  Call it from one thread, right after griddepcontrol.wait.
__device__ __forceinline__ void kstamp(unsigned long long* ts) {
  if (ts != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    *ts = t;
  }
}

}  // namespace g3
