// CUDA-core attention, vla.cpp Eq. (2): o = softmax(q K^T / sqrt(d) + M) V.
//
// One warp per (sample, query token, query head) with an online (running
// max / running sum) softmax over the keys, fp32 throughout.  Keys are the
// bound prefix / VL context (through the device pointer table, optional
// visibility mask) followed by the suffix keys computed this step (the
// action tokens' own K/V, "pi0.5 Design", Attention and the K/V pool; or the
// state+action tokens for DiT self-attention).  A row with no visible key
// writes zeros.  This is the fp32 path and the cross-check of the tensor-core
// kernel; head_dim <= 256.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace g3 {

namespace {

constexpr int kMaxPerLane = 8;  // head_dim <= 256

template <typename T>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnArgs a) {
  ptx::pdl_launch_dependents();
  ptx::pdl_wait();
  if (threadIdx.x == 0) kstamp(a.ts);
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  const long long total = (long long)a.B * a.Tq * a.Hq;
  if (w >= total) return;
  const int head = (int)(w % a.Hq);
  const int t = (int)((w / a.Hq) % a.Tq);
  const int b = (int)(w / ((long long)a.Hq * a.Tq));
  const int kvh = head / (a.Hq / a.Hkv);
  const int Dh = a.Dh;
  const float scale = rsqrtf((float)Dh);

  const T* q = (const T*)a.q + ((long long)b * a.Tq + t) * a.ldq + (long long)head * Dh;
  float qv[kMaxPerLane], o[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int d = lane + 32 * i;
    qv[i] = d < Dh ? to_f(q[d]) : 0.f;
    o[i] = 0.f;
  }
  const T* Kp = a.k_slot >= 0 ? (const T*)a.table[a.k_slot] : nullptr;
  const T* Vp = a.v_slot >= 0 ? (const T*)a.table[a.v_slot] : nullptr;
  const uint8_t* mask = a.mask_slot >= 0 ? (const uint8_t*)a.table[a.mask_slot] : nullptr;

  float mx = -INFINITY, l = 0.f;
  const int nkeys = a.P + a.S;
  for (int s = 0; s < nkeys; ++s) {
    const T *kr, *vr;
    if (s < a.P) {
      if (mask && !mask[(long long)b * a.P + s]) continue;
      const long long off = (((long long)b * a.P + s) * a.Hkv + kvh) * Dh;
      kr = Kp + off;
      vr = Vp + off;
    } else {
      const long long off = ((long long)b * a.Tq + (s - a.P)) * a.lds + (long long)kvh * Dh;
      kr = (const T*)a.ks + off;
      vr = (const T*)a.vs + off;
    }
    float d = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int dd = lane + 32 * i;
      if (dd < Dh) d = fmaf(qv[i], to_f(kr[dd]), d);
    }
    d = warp_sum(d) * scale;
    const float mn = fmaxf(mx, d);
    const float c = expf(mx - mn);
    const float p = expf(d - mn);
    l = l * c + p;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int dd = lane + 32 * i;
      if (dd < Dh) o[i] = o[i] * c + p * to_f(vr[dd]);
    }
    mx = mn;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  T* out = (T*)a.out + ((long long)b * a.Tq + t) * a.ldo + (long long)head * Dh;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int d = lane + 32 * i;
    if (d < Dh) out[d] = from_f<T>(o[i] * inv);
  }
}

}  // namespace

cudaError_t attention_simt(DType dt, const AttnArgs& a, cudaStream_t s, bool pdl) {
  const long long total = (long long)a.B * a.Tq * a.Hq;
  if (total <= 0) return cudaSuccess;
  if (a.Dh > 32 * kMaxPerLane || a.Hkv <= 0 || a.Hq % a.Hkv) return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)((total + 3) / 4);
  if (dt == DT_F32) return launch_k(attn_simt_kernel<float>, blocks, 128, 0, s, pdl, a);
  return launch_k(attn_simt_kernel<bf16>, blocks, 128, 0, s, pdl, a);
}

}  // namespace g3
