// GEMM epilogues of the denoise step, applied to adjacent output pairs (n, n+1).
//
// Pairs make every fused epilogue local to one thread or two adjacent lanes:
//  * RoPE (rotate-half, "Optimizing GR00T-N1.7 Training" 3.3): the Q/K weight
//    rows are stored interleaved, row 2i = original row i, row 2i+1 = original
//    row i + hd/2, so a pair is exactly one rotation (x_i, x_{i+hd/2}).
//  * GeGLU: gate/up rows interleaved, row 2f = gate f, row 2f+1 = up f.
//  * gated residual h += gate * acc ("pi0.5 Design": AdaRMS gate).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace g3 {

template <typename T>
__device__ __forceinline__ void store_pair(T* p, float a0, float a1);
template <>
__device__ __forceinline__ void store_pair<float>(float* p, float a0, float a1) {
  *reinterpret_cast<float2*>(p) = make_float2(a0, a1);
}
template <>
__device__ __forceinline__ void store_pair<bf16>(bf16* p, float a0, float a1) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a0, a1);
}

template <typename T>
__device__ __forceinline__ void epi_pair(const Epi& e, int m, int n, float a0, float a1) {
  switch (e.kind) {
    case EPI_STORE: {
      if (e.bias) {
        a0 += e.bias[n];
        a1 += e.bias[n + 1];
      }
      if (e.act == ACT_SWISH) {
        a0 = swishf(a0);
        a1 = swishf(a1);
      } else if (e.act == ACT_GELU) {
        a0 = gelu_act<T>(a0);
        a1 = gelu_act<T>(a1);
      }
      const long long r = e.rg ? (long long)(m / e.rg) * e.rs + e.ro + m % e.rg : (long long)m;
      if (e.out_f32)
        store_pair<float>((float*)e.out + r * e.ldo + n, a0, a1);
      else
        store_pair<T>((T*)e.out + r * e.ldo + n, a0, a1);
      break;
    }
    case EPI_ROPE: {
      T* o = (T*)e.out + (long long)m * e.ldo;
      if (n < e.rope_cols) {
        const int head = n / e.hd, i = (n % e.hd) >> 1, half = e.hd >> 1;
        const float2 cs = e.rope_tab[(m % e.tok_rope) * half + i];
        o[head * e.hd + i] = from_f<T>(a0 * cs.x - a1 * cs.y);
        o[head * e.hd + i + half] = from_f<T>(a1 * cs.x + a0 * cs.y);
      } else {
        store_pair<T>(o + n, a0, a1);
      }
      break;
    }
    case EPI_RESID_GATED: {
      const T* g = (const T*)e.gate + (long long)(m / e.tok) * e.gate_bstride + n;
      float2* h = reinterpret_cast<float2*>(e.resid + (long long)m * e.ldr + n);
      float2 v = *h;
      v.x += to_f(g[0]) * a0;
      v.y += to_f(g[1]) * a1;
      *h = v;
      break;
    }
    case EPI_RESID: {
      float2* h = reinterpret_cast<float2*>(e.resid + (long long)m * e.ldr + n);
      float2 v = *h;
      v.x += a0;
      v.y += a1;
      *h = v;
      break;
    }
    case EPI_GEGLU: {
      T* o = (T*)e.out + (long long)m * e.ldo + (n >> 1);
      *o = from_f<T>(gelu_act<T>(a0) * a1);
      break;
    }
    default:
      break;
  }
}

// Operands of an epilogue that do not depend on the accumulator (residual row
// and gate), loaded ahead so their latency overlaps the partial-sum loads.
struct EpiPre {
  float2 h;
  float2 g;
  float2 cs;   // RoPE (cos, sin) of the pair
};

template <typename T>
__device__ __forceinline__ EpiPre epi_prefetch(const Epi& e, int m, int n) {
  EpiPre p;
  p.h = make_float2(0.f, 0.f);
  p.g = make_float2(1.f, 1.f);
  p.cs = make_float2(1.f, 0.f);
  if (e.kind == EPI_ROPE && n < e.rope_cols) {
    const int i = (n % e.hd) >> 1, half = e.hd >> 1;
    p.cs = e.rope_tab[(m % e.tok_rope) * half + i];
  } else if (e.kind == EPI_RESID_GATED || e.kind == EPI_RESID) {
    p.h = *reinterpret_cast<const float2*>(e.resid + (long long)m * e.ldr + n);
    if (e.kind == EPI_RESID_GATED) {
      const T* g = (const T*)e.gate + (long long)(m / e.tok) * e.gate_bstride + n;
      p.g = make_float2(to_f(g[0]), to_f(g[1]));
    }
  }
  return p;
}

template <typename T>
__device__ __forceinline__ void epi_pair(const Epi& e, int m, int n, float a0, float a1, const EpiPre& p) {
  if (e.kind == EPI_RESID_GATED || e.kind == EPI_RESID) {
    *reinterpret_cast<float2*>(e.resid + (long long)m * e.ldr + n) =
        make_float2(p.h.x + p.g.x * a0, p.h.y + p.g.y * a1);
    return;
  }
  if (e.kind == EPI_ROPE && n < e.rope_cols) {   // rotation with the prefetched (cos, sin)
    T* o = (T*)e.out + (long long)m * e.ldo;
    const int head = n / e.hd, i = (n % e.hd) >> 1, half = e.hd >> 1;
    o[head * e.hd + i] = from_f<T>(a0 * p.cs.x - a1 * p.cs.y);
    o[head * e.hd + i + half] = from_f<T>(a1 * p.cs.x + a0 * p.cs.y);
    return;
  }
  epi_pair<T>(e, m, n, a0, a1);
}



// ---------------------------------------------------------------------------
// Epilogue of one thread's output pairs for a run of token columns, with the
// per-thread invariants hoisted (the thread's weight rows n, n+1 are fixed).
// Split into a branch-free compute() and a store(), so that a lane's 16 column
// pairs form 16 independent dependency chains the compiler can interleave (a
// guard around each pair serialises them: measured ~60 ns per pair).  ACT is
// the activation of EPI_STORE.  Used by the tensor-core kernels.
// ---------------------------------------------------------------------------
template <int KIND, int ACT = ACT_NONE>
struct EpiRun {
  __device__ __forceinline__ EpiRun(const Epi& e, int n) : e_(e), n_(n) {
    if (KIND == EPI_STORE) {
      b0_ = e.bias ? e.bias[n] : 0.f;
      b1_ = e.bias ? e.bias[n + 1] : 0.f;
    } else if (KIND == EPI_ROPE) {
      rope_ = n < e.rope_cols;
      if (rope_) {
        const int head = n / e.hd, i = (n % e.hd) >> 1;
        half_ = e.hd >> 1;
        i_ = i;
        col0_ = head * e.hd + i;
      }
    }
  }
  // RoPE (cos, sin) of token index j (j < tok_rope) for this thread's frequency.
  __device__ __forceinline__ float2 rope_cs(int j) const { return e_.rope_tab[j * half_ + i_]; }
  // Outputs of the pair (a0, a1) = rows (n, n+1) of one token column.
  __device__ __forceinline__ void compute(float a0, float a1, float2 cs, float& o0, float& o1) const {
    if (KIND == EPI_STORE) {
      a0 += b0_;
      a1 += b1_;
      if (ACT == ACT_SWISH) {
        a0 = swishf(a0);
        a1 = swishf(a1);
      } else if (ACT == ACT_GELU) {
        a0 = gelu_tanh_fast(a0);
        a1 = gelu_tanh_fast(a1);
      }
      o0 = a0;
      o1 = a1;
    } else if (KIND == EPI_ROPE) {
      o0 = rope_ ? a0 * cs.x - a1 * cs.y : a0;
      o1 = rope_ ? a1 * cs.x + a0 * cs.y : a1;
    } else if (KIND == EPI_GEGLU) {
      o0 = gelu_tanh_fast(a0) * a1;
      o1 = 0.f;
    } else {
      o0 = a0;
      o1 = a1;
    }
  }
  // Store the outputs of token column m.
  __device__ __forceinline__ void store(int m, float o0, float o1) const {
    if (KIND == EPI_STORE) {
      const long long r = e_.rg ? (long long)(m / e_.rg) * e_.rs + e_.ro + m % e_.rg : (long long)m;
      if (e_.out_f32)
        store_pair<float>((float*)e_.out + r * e_.ldo + n_, o0, o1);
      else
        store_pair<bf16>((bf16*)e_.out + r * e_.ldo + n_, o0, o1);
    } else if (KIND == EPI_ROPE) {
      bf16* o = (bf16*)e_.out + (long long)m * e_.ldo;
      if (rope_) {
        o[col0_] = __float2bfloat16_rn(o0);
        o[col0_ + half_] = __float2bfloat16_rn(o1);
      } else {
        store_pair<bf16>(o + n_, o0, o1);
      }
    } else if (KIND == EPI_GEGLU) {
      ((bf16*)e_.out)[(long long)m * e_.ldo + (n_ >> 1)] = __float2bfloat16_rn(o0);
    } else {  // residual kinds: operands loaded here
      const EpiPre p = epi_prefetch<bf16>(e_, m, n_);
      epi_pair<bf16>(e_, m, n_, o0, o1, p);
    }
  }
  // compute + store of one pair (callers with one pair at a time)
  __device__ __forceinline__ void operator()(int m, float2 cs, float a0, float a1) const {
    float o0, o1;
    compute(a0, a1, cs, o0, o1);
    store(m, o0, o1);
  }
  const Epi& e_;
  int n_;
  float b0_ = 0.f, b1_ = 0.f;
  bool rope_ = false;
  int half_ = 0, i_ = 0, col0_ = 0;
};

// 32 accumulator columns c0..c0+31 of rows (n, n+1) held by a lane pair; this
// lane finishes columns of parity ``odd``.  For RoPE the 16 (cos, sin) pairs
// are loaded together up front (token index kept in [0, tok_rope), so every
// load is in bounds even past M).  All 16 pairs are computed before any store,
// unconditionally; only the stores are guarded.
template <int KIND, int ACT>
__device__ __forceinline__ void epi_columns(const EpiRun<KIND, ACT>& run, const float (&v)[32], bool odd,
                                            int m_first, int M, int tok_rope) {
  float2 cs[16];
  if (KIND == EPI_ROPE) {
    int j = m_first % tok_rope;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      cs[q] = run.rope_ ? run.rope_cs(j) : make_float2(1.f, 0.f);
      j += 2;  // next column of this parity; tok_rope may be 1
      if (j >= tok_rope) j -= tok_rope;
      if (j >= tok_rope) j -= tok_rope;
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
  if constexpr (KIND == EPI_RESID || KIND == EPI_RESID_GATED) {
    // read-modify-write of the residual rows: the residual (and gate) loads of 8
    // columns are issued before their stores, so they are in flight together (a
    // store between them would order each load after the previous store)
#pragma unroll
    for (int q0 = 0; q0 < 16; q0 += 8) {
      EpiPre pre[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (m_first + 2 * (q0 + q) < M) pre[q] = epi_prefetch<bf16>(run.e_, m_first + 2 * (q0 + q), run.n_);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (m_first + 2 * (q0 + q) < M)
          epi_pair<bf16>(run.e_, m_first + 2 * (q0 + q), run.n_, o0[q0 + q], o1[q0 + q], pre[q]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q)
      if (m_first + 2 * q < M) run.store(m_first + 2 * q, o0[q], o1[q]);
  }
}
}  // namespace g3
