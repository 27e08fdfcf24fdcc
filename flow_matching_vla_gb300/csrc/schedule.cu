// Set-up kernels: the time embedding of the hoisted schedule, the RoPE table
// of the bound prefix length, and the weight re-layout done at create.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace g3 {

namespace {

// Sinusoidal embedding of tau_k on the uniform grid of vla.cpp Eq. (1):
// tau_k = 1 - k/T (direction -1) or k/T (direction +1); entries i < E/2 are
// sin(tau w_i), the rest cos(tau w_{i - E/2}), w_i = 2 pi / period_i with
// period_i = 4e-3 * (4 / 4e-3)^(i / (E/2 - 1)).  Computed in double.
template <typename T>
__global__ void time_embed_kernel(int T_, int B, int E, int direction, T* __restrict__ temb,
                                  float* __restrict__ dts) {
  const int r = blockIdx.x;  // row k * B + b
  const int k = r / B;
  const double tau = direction < 0 ? 1.0 - (double)k / T_ : (double)k / T_;
  const int half = E / 2;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double frac = (double)i / (double)(half - 1);
    const double period = 4e-3 * pow(4.0 / 4e-3, frac);
    const double ang = tau * (2.0 * M_PI / period);
    temb[(long long)r * E + i] = from_f<T>((float)sin(ang));
    temb[(long long)r * E + half + i] = from_f<T>((float)cos(ang));
  }
  if (threadIdx.x == 0 && r % B == 0) {
    const double tn = direction < 0 ? 1.0 - (double)(k + 1) / T_ : (double)(k + 1) / T_;
    dts[k] = (float)(tn - tau);
  }
}

__global__ void rope_table_kernel(int P, int H, int hd, double theta, float2* __restrict__ tab) {
  const int half = hd / 2;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= H * half) return;
  const int j = idx / half, i = idx % half;
  const double ang = (double)(P + j) * pow(theta, -2.0 * i / hd);
  tab[idx] = make_float2((float)cos(ang), (float)sin(ang));
}

__device__ __forceinline__ int perm_src(int r, int mode, int p0, int p1) {
  if (mode == PERM_ROPE) {  // p0 = rows holding rotate-half heads, p1 = head_dim
    if (r >= p0) return r;
    const int head = r / p1, j = r % p1;
    return head * p1 + ((j & 1) ? (j >> 1) + p1 / 2 : (j >> 1));
  }
  if (mode == PERM_GEGLU)  // p0 = F: row 2f <- gate f, row 2f+1 <- up f
    return (r & 1) ? p0 + (r >> 1) : (r >> 1);
  return r;
}

__global__ void permute_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                    int row_vec, int mode, int p0, int p1) {
  const int r = blockIdx.x;
  const int sr = perm_src(r, mode, p0, p1);
  const uint4* s = src + (long long)sr * row_vec;
  uint4* d = dst + (long long)r * row_vec;
  for (int i = threadIdx.x; i < row_vec; i += blockDim.x) d[i] = s[i];
}

__global__ void permute_floats_kernel(const float* __restrict__ src, float* __restrict__ dst, int rows, int mode,
                                      int p0, int p1) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < rows) dst[r] = src[perm_src(r, mode, p0, p1)];
}

template <typename T>
__global__ void to_f32_kernel(const T* __restrict__ src, float* __restrict__ dst, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = to_f(src[i]);
}

}  // namespace

cudaError_t time_embed(DType dt, int T, int B, int E, int direction, void* temb, float* dts,
                       cudaStream_t s) {
  if (dt == DT_F32)
    time_embed_kernel<float><<<T * B, 128, 0, s>>>(T, B, E, direction, (float*)temb, dts);
  else
    time_embed_kernel<bf16><<<T * B, 128, 0, s>>>(T, B, E, direction, (bf16*)temb, dts);
  return cudaGetLastError();
}

cudaError_t rope_table(int P, int H, int hd, float theta, float2* tab, cudaStream_t s) {
  const int n = H * (hd / 2);
  if (n <= 0) return cudaSuccess;
  rope_table_kernel<<<(n + 127) / 128, 128, 0, s>>>(P, H, hd, (double)theta, tab);
  return cudaGetLastError();
}

cudaError_t permute_rows(const void* src, void* dst, int rows, int row_bytes, int mode, int p0,
                         int p1, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (row_bytes % 16 || ((uintptr_t)src & 15) || ((uintptr_t)dst & 15)) return cudaErrorInvalidValue;
  permute_rows_kernel<<<rows, 128, 0, s>>>((const uint4*)src, (uint4*)dst, row_bytes / 16, mode, p0,
                                           p1);
  return cudaGetLastError();
}

cudaError_t permute_floats(const float* src, float* dst, int rows, int mode, int p0, int p1, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  permute_floats_kernel<<<(rows + 255) / 256, 256, 0, s>>>(src, dst, rows, mode, p0, p1);
  return cudaGetLastError();
}

cudaError_t to_f32(DType dt, const void* src, float* dst, long long n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  if (dt == DT_F32)
    to_f32_kernel<float><<<blocks, 256, 0, s>>>((const float*)src, dst, n);
  else
    to_f32_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)src, dst, n);
  return cudaGetLastError();
}


namespace {

template <typename T>
__global__ void state_rows_kernel(const float* __restrict__ src, int M, int K, T* __restrict__ dst, int Kp) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)M * Kp) return;
  const int m = (int)(i / Kp), k = (int)(i % Kp);
  dst[i] = from_f<T>(k < K ? src[(long long)m * K + k] : 0.f);
}

}  // namespace

cudaError_t state_rows(DType dt, const float* src, int M, int K, void* dst, int Kp, cudaStream_t s) {
  const long long n = (long long)M * Kp;
  if (n <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((n + 255) / 256);
  if (dt == DT_F32)
    state_rows_kernel<float><<<blocks, 256, 0, s>>>(src, M, K, (float*)dst, Kp);
  else
    state_rows_kernel<bf16><<<blocks, 256, 0, s>>>(src, M, K, (bf16*)dst, Kp);
  return cudaGetLastError();
}

namespace {

__global__ void bounded_wait_probe_kernel(const volatile int* never, int* err, long long limit) {
  if (threadIdx.x != 0) return;
  for (long long i = 0; i < limit; ++i)
    if (*never != 0) return;
  atomicExch(err, 1);
}

__global__ void stamp_tail_kernel(unsigned long long* ts) {
  ptx::pdl_launch_dependents();
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(ts);
}

}  // namespace

cudaError_t bounded_wait_probe(const int* never, int* err, long long limit, cudaStream_t s) {
  bounded_wait_probe_kernel<<<1, 32, 0, s>>>(never, err, limit);
  return cudaGetLastError();
}

cudaError_t stamp_tail(unsigned long long* ts, cudaStream_t s, bool pdl) {
  return launch_k(stamp_tail_kernel, dim3(1), dim3(32), 0, s, pdl, ts);
}

}  // namespace g3
