// Host-side launch interface of the denoise-loop kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace g3 {

enum DType : int { DT_F32 = 0, DT_BF16 = 1 };

// ---- GEMM epilogues ---------------------------------------------------------
// Every GEMM computes acc[m][n] = sum_k A[m][k] * W[n][k] (fp32 accumulation)
// and hands adjacent output pairs (n, n+1), n even, to one epilogue.
enum EpiKind : int {
  EPI_STORE = 0,        // out[r(m)][n] = act(acc + bias[n])            (act dtype, or fp32 if out_f32)
  EPI_ROPE = 1,         // fused Q/K RoPE: rows < rope_cols hold rotate-half pairs (see runtime)
  EPI_RESID_GATED = 2,  // h[m][n] += gate[m / tok][n] * acc            (fp32 residual)
  EPI_RESID = 3,        // h[m][n] += acc
  EPI_GEGLU = 4,        // out[m][n/2] = gelu(acc[n]) * acc[n+1]          (interleaved gate/up rows)
  EPI_PARTIAL = 5,      // split-K partial: out[(split * M + m) * ldo + n] = acc (fp32); the
                        // consumer (norm / out_proj kernel) sums the splits into the residual
};
enum Act : int { ACT_NONE = 0, ACT_SWISH = 1, ACT_GELU = 2 };

struct Epi {
  int kind = EPI_STORE;
  int act = ACT_NONE;
  int out_f32 = 0;          // EPI_STORE: write fp32 instead of the activation dtype
  void* out = nullptr;      // output matrix
  int ldo = 0;              // its leading dimension (elements)
  const float* bias = nullptr;  // [N] fp32, nullable
  // row remap for EPI_STORE: r(m) = (m / rg) * rs + ro + m % rg   (rg = 0: r(m) = m)
  int rg = 0, rs = 0, ro = 0;
  // residual epilogues
  float* resid = nullptr;   // fp32 [M][ldr]
  int ldr = 0;
  const void* gate = nullptr;  // activation dtype; gate for row m: gate + (m / tok) * gate_bstride
  long long gate_bstride = 0;
  int tok = 1;
  // RoPE: columns [0, rope_cols) are (Hq + Hkv) heads of rotate-half pairs, head_dim hd
  int rope_cols = 0, hd = 0;
  const float2* rope_tab = nullptr;  // [tok_rope][hd/2] (cos, sin) for positions P + j
  int tok_rope = 1;                  // token rows per sample
  // E4M3 weights: fp32 scale of weight row n (output column n); the tensor-core
  // E4M3 GEMM multiplies each accumulator row by it before the epilogue
  const float* wscale = nullptr;
  // dependency-release stamp of this launch (nullable; see kstamp in common.cuh)
  unsigned long long* ts = nullptr;
  // persistent tensor-core GEMM: outputs staged in shared memory and written by
  // tensor stores through the output map passed beside (set by the launcher)
  int tstore = 0;
};

struct GemmArgs {
  const void* A = nullptr;  // activations [M][lda]
  int lda = 0;
  const void* W = nullptr;  // weights [N][ldw]
  int ldw = 0;
  int M = 0, N = 0, K = 0;
  Epi epi;
  // optional L2 prefetch of memory later kernels read (e.g. the next layer's
  // weights), spread over the CTAs and issued before the dependency wait
  struct Prefetch {
    const void* p = nullptr;
    long long bytes = 0;
  } l2[3];
};

// CUDA-core GEMM (any shape with N even).
cudaError_t gemm_simt(DType dt, const GemmArgs& a, cudaStream_t s, bool pdl);

// ---- normalisation / projection kernels ------------------------------------
enum NormKind : int { NORM_RMS = 0, NORM_LN = 1 };
struct NormArgs {
  // optional residual update first: h[m] += gate_b * sum_{s < S} part[s][m]   (rank order)
  const float* part = nullptr;   // fp32 [S][M][D]
  int part_S = 0, part_M = 0;
  const void* gate = nullptr;    // activation dtype, per sample: gate + b * mod_bstride (nullable: 1)
  int kind = NORM_RMS;
  float eps = 1e-6f;
  const void* mod = nullptr;     // activation dtype; row for sample b: mod + b * mod_bstride
  long long mod_bstride = 0;
  int scale_off = 0, shift_off = 0;   // offsets of scale and shift inside the row
  int tok = 1;                   // token rows per sample
  unsigned long long* ts = nullptr;   // dependency-release stamp (nullable)
};

// out[m] = norm(h[m]) * (1 + scale) + shift for m < M (mod == nullptr: plain norm)
// (with na.part: h[m] += gate * sum of the split-K partials first, written back)
cudaError_t adanorm(DType dt, float* h, int D, int M, void* out, NormArgs na, cudaStream_t s, bool pdl);

// EXPERT step head: h[m] = x[m] W_in^T + b_in (fp32), then out[m] = AdaRMS(h[m]).
cudaError_t expert_in(DType dt, const float* x, int A, const void* w_in, const float* b_in, float* h,
                      int D, int M, void* out, NormArgs na, cudaStream_t s, bool pdl);

// Final norm + action_out_proj + Euler: rows m < M of the action tokens.
// h row of action token m: (m / H) * tok + ro + m % H.  v = norm(h) W_out^T + b_out;
// v_out[m] = v (nullable); if do_euler: x[m] += dt[k] * v.
cudaError_t out_euler(DType dt, float* h, int D, int M, int H, int ro, const void* w_out,
                      const float* b_out, int A, NormArgs na, float* x, const float* dts, int k,
                      int do_euler, float* v_out, cudaStream_t s, bool pdl);

// DIT step head: a[m] = x[m] W1^T + b1 (activation dtype) for the M action rows, and the
// state tokens copied into the residual rows (b * tok + j, j < ns) from state [B][ns][D].
cudaError_t dit_in(DType dt, const float* x, int A, const void* w1, const float* b1, void* a_out,
                   int D, int M, const float* state, int ns, int tok, int B, float* h,
                   cudaStream_t s, bool pdl, unsigned long long* ts = nullptr);

// ---- attention ----------------------------------------------------------------
struct AttnArgs {
  const void* q = nullptr;  // query of (b, t, head): q + (b*Tq + t)*ldq + head*Dh
  int ldq = 0;
  int B = 0, Tq = 0, Hq = 0, Hkv = 1, Dh = 0;
  const void* const* table = nullptr;  // device pointer table (prefix K/V, masks)
  int k_slot = -1, v_slot = -1, mask_slot = -1;  // slots in the table (-1: none)
  int P = 0;                // prefix keys per sample: table[k_slot] is [B][P][Hkv][Dh]
  const void* ks = nullptr; // suffix keys of (b, j, kvh): ks + (b*Tq + j)*lds + kvh*Dh
  const void* vs = nullptr;
  int lds = 0;
  int S = 0;                // suffix keys per sample
  void* out = nullptr;      // output of (b, t, head): out + (b*Tq + t)*ldo + head*Dh
  int ldo = 0;
  unsigned long long* ts = nullptr;   // dependency-release stamp (nullable)
};
cudaError_t attention_simt(DType dt, const AttnArgs& a, cudaStream_t s, bool pdl);

// Attention of the DiT head (bf16, Dh 48 or 64, <= 32 query tokens, masks): K/V tiles
// staged by TMA, mma.sync per head, key groups merged on chip.  Either cross-attention
// (a.P > 0, a.S == 0; kp / vp = the bound context's K / V, the host's copies of the
// table entries) or self-attention (a.P == 0, a.S == a.Tq <= 64; kp / vp unused).
bool attn_dit_supported(const AttnArgs& a, const void* kp, const void* vp);
cudaError_t attention_dit(const AttnArgs& a, const void* kp, const void* vp, int* err, long long wait_limit,
                          cudaStream_t s, bool pdl);

// Tensor-core attention of the expert family (one KV head, heads folded into rows).
struct AttnFoldArgs {
  const void* qkv = nullptr;   // bf16 [B*H][ldq]: q heads at 0, suffix k at k_off, v at v_off
  int ldq = 0, k_off = 0, v_off = 0;
  int B = 0, H = 0, Hq = 0, Dh = 0, P = 0;
  const void* const* table = nullptr;  // prefix K/V [B][P][Dh] at table[k_slot], table[v_slot]
  int k_slot = 0, v_slot = 0;
  void* out = nullptr;         // bf16 [B*H][ldo], head h at column h*Dh
  int ldo = 0;
  float* ws = nullptr;         // split partials (L2-resident scratch)
  long long ws_floats = 0;
  unsigned long long* ts = nullptr;   // dependency-release stamp (nullable)
};
bool attn_fold_supported(int Dh);
long long attn_fold_workspace_floats(const AttnFoldArgs& a, int S);
int attn_fold_splits(const AttnFoldArgs& a, int sm_count);
cudaError_t attention_fold(const AttnFoldArgs& a, int S, cudaStream_t s, bool pdl);

// tcgen05 / TMEM attention of the expert family (same computation as attention_fold).
struct AttnT5Args {
  const void* qkv = nullptr;  // bf16 [B*H][ldq]
  int ldq = 0, k_off = 0, v_off = 0;
  int B = 0, H = 0, Hq = 0, Dh = 0, P = 0;
  void* out = nullptr;        // bf16 [B*H][ldo]
  int ldo = 0;
  float* ws = nullptr;        // split partials (L2-resident scratch)
  long long ws_floats = 0;
  int* err = nullptr;         // device error word (bounded waits)
  long long wait_limit = 0;
  int ps = 0;                 // rows per sample of the bound prefix K/V (0: P; a pool: its capacity)
  void* pool_k = nullptr;     // a bound pool's K and V planes: this step's suffix K/V go to
  void* pool_v = nullptr;     // rows [P, P + H) of each sample's slot (nullptr: no pool)
  int pool_cap = 0;
  int ct = 1;                 // CTAs per cluster sharing every key tile by multicast (attn_t5_cluster)
  unsigned long long* ts = nullptr;    // dependency-release stamp of the main kernel (nullable)
  unsigned long long* ts2 = nullptr;   // ... and of the split merge (nullable)
};
}  // namespace g3
#include <cuda.h>
namespace g3 {
bool attn_t5_supported(int Dh, int Hq);
int attn_t5_splits(const AttnT5Args& a, int sm_count, int cap = 0);   // cap > 0: at most cap splits
int attn_t5_cluster(const AttnT5Args& a);   // the cluster size for a.ct (1: no multicast)
long long attn_t5_workspace_floats(const AttnT5Args& a, int S);
// maps[8]: Q, prefix K, prefix V, suffix K, suffix V, the output tile (S: the key splits), pool K, pool V
cudaError_t attn_t5_maps(const AttnT5Args& a, const void* kp, const void* vp, int S, CUtensorMap* maps);
cudaError_t attention_t5(const AttnT5Args& a, const CUtensorMap* maps, int S, cudaStream_t s, bool pdl);

// ---- schedule / bind / create helpers --------------------------------------------
// temb[k*B + b][E] (activation dtype) of tau_k; dts[k] = tau_{k+1} - tau_k.
cudaError_t time_embed(DType dt, int T, int B, int E, int direction, void* temb, float* dts,
                       cudaStream_t s);
// tab[j][i] = (cos, sin)((P + j) * theta^(-2i/hd)), j < H, i < hd/2
cudaError_t rope_table(int P, int H, int hd, float theta, float2* tab, cudaStream_t s);

enum PermMode : int { PERM_NONE = 0, PERM_ROPE = 1, PERM_GEGLU = 2 };
// dst row r <- src row perm(r); rows of row_bytes bytes (multiple of 16, 16B-aligned pointers)
cudaError_t permute_rows(const void* src, void* dst, int rows, int row_bytes, int mode, int p0,
                         int p1, cudaStream_t s);
// dst[r] <- src[perm(r)] for one float per row (the row scales of an FP8 matrix)
cudaError_t permute_floats(const float* src, float* dst, int rows, int mode, int p0, int p1, cudaStream_t s);
// dst[i] = float(src[i]) for a DType source
cudaError_t to_f32(DType dt, const void* src, float* dst, long long n, cudaStream_t s);
// dst[m][k] = (DType) src[m][k] for k < K, 0 for K <= k < Kp: fp32 rows [M][K] into
// activation rows [M][Kp] (the state encoder's input, K padded for the tensor cores)
cudaError_t state_rows(DType dt, const float* src, int M, int K, void* dst, int Kp, cudaStream_t s);

// One thread waits up to ``limit`` polls for *never to become nonzero; when the
// limit passes it sets *err = 1 and returns (the bounded-wait error path).
cudaError_t bounded_wait_probe(const int* never, int* err, long long limit, cudaStream_t s);
// A one-thread kernel that writes its dependency-release stamp into *ts: placed
// after the loop's last launch, it closes that launch's interval.
cudaError_t stamp_tail(unsigned long long* ts, cudaStream_t s, bool pdl);

}  // namespace g3
