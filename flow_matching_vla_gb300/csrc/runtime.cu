// C ABI of the denoise loop: context, weight re-layout, bind, schedule, denoise.
//
// The step structure follows "pi0.5 Design" (expert) and "GR00T N1.7" (DiT):
// the prefix K/V is bound once, the time conditioning is hoisted into a
// modulation table that re-runs only when (steps, batch) change, and the T
// Euler steps (vla.cpp Eq. (1)) replay as one CUDA graph.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "gemm_tc.h"
#include "gr00t.h"
#include "kernels.h"

// Size (fp32 elements) of the fixed scratch array of the allocation-free step.
#define G3_NOALLOC_SCRATCH_FLOATS (3 << 20)
// Descriptor slots the allocation-free step uses instead of the descriptor cache
// (a launch takes at most this many descriptors from tmap(); they are copied into
// the kernel parameters at launch).
constexpr int kSpillMaps = 4;

using namespace g3;

struct gr00t_ctx {
  gr00t_geometry g{};
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  std::string err;

  // derived sizes
  DType dt = DT_BF16;
  size_t esz = 2;            // bytes per weight / activation element
  int D = 0, L = 0, Hq = 0, Hkv = 1, Dh = 0, F = 0, H = 0, A = 0, Ns = 0, E = 0;
  int tok = 0;               // token rows per sample: H + Ns
  int S = 0, R = 0;          // modulation sites and row width
  int qd = 0;                // Hq * Dh
  int Mmax = 0;
  std::vector<int> nqkv;     // rows of each layer's qkv projection

  // one device arena
  char* arena = nullptr;
  size_t arena_bytes = 0;

  // weights (activation dtype; the per-layer projections E4M3 codes when fp8w), biases (fp32)
  bool fp8w = false;          // GR00T_WFMT_FP8: per-layer projections as codes + row scales
  std::vector<void*> w_qkv, w_o, w_up, w_down;
  std::vector<float*> s_qkv, s_o, s_up, s_down;   // fp8w: fp32 scale of each output row
  // DiT with context_dim: cross K/V projections of the even blocks, their outputs, the features
  std::vector<void*> w_ck, w_cv, ctx_k, ctx_v;
  void* ctx_feat = nullptr;
  void *w_tin = nullptr, *w_tout = nullptr, *w_cond = nullptr, *w_in = nullptr, *w_out = nullptr;
  void *w_enc1 = nullptr, *w_enc2 = nullptr, *w_enc3 = nullptr;
  // DiT state encoder (state_dim > 0): W_s1 with its K padded to Ks (a multiple of 64),
  // its input rows, hidden rows and the encoded state tokens
  int Ks = 0;
  void *w_s1 = nullptr, *w_s2 = nullptr, *state_in = nullptr, *state_hid = nullptr;
  float *b_s1 = nullptr, *b_s2 = nullptr, *state_tok = nullptr;
  float *b_tin = nullptr, *b_tout = nullptr, *b_cond = nullptr, *b_in = nullptr, *b_out = nullptr;
  float *b_enc1 = nullptr, *b_enc2 = nullptr, *b_enc3 = nullptr;

  // activations
  float* h = nullptr;
  void *n = nullptr, *qkv = nullptr, *att = nullptr, *u = nullptr, *a_enc = nullptr, *e_enc = nullptr;
  float *x = nullptr, *xtmp = nullptr;
  // schedule
  void *temb = nullptr, *t1 = nullptr, *cvec = nullptr, *mod = nullptr;
  float *dts = nullptr, *atb = nullptr;
  float2* rope_tab = nullptr;
  const void** table = nullptr;   // device pointer table: K_l, V_l (2L), text, image, state
  int* err_flag = nullptr;

  // state
  bool bound = false, scheduled = false;
  int bB = 0, bP = 0, sT = 0, sB = 0;
  // a bound paged K/V pool (EXPERT): per-layer base of [2][B][cap][1][Dh]; rows per sample
  std::vector<void*> pool;
  int pool_cap = 0;
  std::vector<const void*> host_table;

  // graph cache (one entry)
  cudaGraphExec_t gexec = nullptr;
  int gT = -1, gB = -1, gP = -1;

  // options
  int opt_graph = 1, opt_gemm = 0, opt_attn = 0;
  long long wait_limit = 1 << 20;
  int launches = 0;  // kernel launches of the last enqueued step

  // tensor-core GEMM: SM count and a cache of TMA descriptors
  int device = 0;
  int sm_count = 148;
  float* gemm_ws = nullptr;   // split-K partials (L2-resident scratch)
  long long gemm_ws_floats = 0;
  std::map<std::tuple<const void*, long long, long long, long long, int>, CUtensorMap> tmaps;
  int opt_pdl = 1;
  int opt_attn_splits = 0;  // expert attention key-split cap (0: automatic)
  int opt_persistent = 1;   // persistent tensor-core GEMM for unsplit large-M shapes
  // TMA multicast (measured ~1 % slower each at batch 32 with the current kernels)
  int opt_mcast = 0;        // persistent GEMM: pairs of CTAs share activation tiles by TMA multicast
  int opt_attn_mcast = 2;   // expert attention: the row tiles of a sample share key tiles by TMA
                            // multicast (2: where each CTA streams at most 4 key tiles)
  int opt_tstore = 1;       // persistent GEMM epilogues through shared memory and tensor stores
  int opt_l2_ahead = 0;     // each GEMM's idle warps prefetch the next GEMM's weights into L2 (measured: no gain)
  long long noalloc_limit = -1;   // scratch bound of the allocation-free step (-1: the whole fixed array)
  int split_cap = 4;        // GEMMs that reduce their split-K partials in-kernel
  int resid_split_cap = 8;  // residual GEMMs whose partials the next kernel folds in

  // split-K partials a residual GEMM left for the next norm / out_proj kernel
  struct Pending {
    const float* part = nullptr;
    int S = 0, M = 0;
    const void* gate = nullptr;
  } pending;

  // launch stamps (GR00T_OPT_TIME_KERNELS): one device slot per launch of the loop
  int stamp_on = 0;
  unsigned long long* stamps = nullptr;
  int stamp_cap = 0, stamp_used = 0;
  bool in_loop = false;         // stamps are taken by the launches of the whole loop only
  std::vector<int> stamp_cls;   // kernel class of each stamped launch

  // the allocation-free step: its fixed scratch array (device address looked up at
  // create) and descriptor slots that stand in for the descriptor cache
  float* noalloc_addr = nullptr;
  bool no_host_alloc = false;
  CUtensorMap tmap_spill[kSpillMaps];
  unsigned tmap_spill_next = 0;

  // test hooks: a bounded wait on a word nothing writes (GR00T_OPT_TEST_STALL);
  // the residual stream of one block copied out (gr00t_debug_dump)
  int opt_stall = 0;           // polls of the probe's bounded wait (0: no probe)
  int* never_set = nullptr;
  int* err_host = nullptr;   // page-locked copy of the device error word (synchronous calls)
  float* dump_out = nullptr;
  int dump_layer = -2;
};

namespace {

thread_local std::string g_create_err;

cudaError_t noalloc_scratch(int dev, float** out);

int set_err(gr00t_ctx* c, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c)
    c->err = buf;
  else
    g_create_err = buf;
  return code;
}

#define CK(ctx, call)                                                                      \
  do {                                                                                     \
    cudaError_t e_ = (call);                                                               \
    if (e_ != cudaSuccess)                                                                 \
      return set_err((ctx), GR00T_ECUDA, "%s failed: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

int validate(const gr00t_geometry* g, char* msg, size_t len) {
  auto bad = [&](int code, const char* why) {
    if (msg && len) snprintf(msg, len, "%s", why);
    return code;
  };
  if (!g) return bad(GR00T_EINVAL, "geometry is NULL");
  if (g->abi_version != GR00T_ABI_VERSION) return bad(GR00T_EINVAL, "abi_version mismatch");
  if (g->family != GR00T_FAMILY_EXPERT && g->family != GR00T_FAMILY_DIT)
    return bad(GR00T_EINVAL, "unknown family");
  if (g->dtype != GR00T_DTYPE_FP32 && g->dtype != GR00T_DTYPE_BF16)
    return bad(GR00T_EINVAL, "unknown dtype");
  if (g->mlp_kind != GR00T_MLP_GELU && g->mlp_kind != GR00T_MLP_GEGLU)
    return bad(GR00T_EINVAL, "unknown mlp_kind");
  if (g->layers < 1 || g->layers > 512) return bad(GR00T_EINVAL, "layers out of range [1, 512]");
  if (g->hidden < 64 || g->hidden > 8192 || g->hidden % 64)
    return bad(GR00T_EINVAL, "hidden must be a multiple of 64 in [64, 8192]");
  if (g->mlp_dim < 64 || g->mlp_dim % 64 || g->mlp_dim > 65536)
    return bad(GR00T_EINVAL, "mlp_dim must be a multiple of 64 in [64, 65536]");
  if (g->q_heads < 1 || g->head_dim < 2 || g->head_dim % 2 || g->head_dim > 256)
    return bad(GR00T_EINVAL, "head_dim must be even and <= 256, q_heads >= 1");
  if ((g->q_heads * g->head_dim) % 64) return bad(GR00T_EINVAL, "q_heads*head_dim must be a multiple of 64");
  if (g->horizon < 1 || g->horizon > 4096) return bad(GR00T_EINVAL, "horizon out of range");
  if (g->action_dim < 1 || g->action_dim > 1024) return bad(GR00T_EINVAL, "action_dim out of range");
  if (g->time_dim < 4 || g->time_dim % 2 || g->time_dim > 65536) return bad(GR00T_EINVAL, "time_dim must be even, >= 4");
  if (g->time_mlp != 0 && g->time_mlp != 1) return bad(GR00T_EINVAL, "time_mlp must be 0 or 1");
  if (g->direction != -1 && g->direction != 1) return bad(GR00T_EINVAL, "direction must be -1 or +1");
  if (g->max_batch < 1 || g->max_batch > 65536) return bad(GR00T_EINVAL, "max_batch out of range");
  if (g->max_steps < 1 || g->max_steps > 4096) return bad(GR00T_EINVAL, "max_steps out of range");
  if (g->max_prefix < 0 || g->max_prefix > (1 << 20)) return bad(GR00T_EINVAL, "max_prefix out of range");
  if (!(g->norm_eps > 0.f)) return bad(GR00T_EINVAL, "norm_eps must be > 0");
  if (g->weight_format != GR00T_WFMT_NATIVE && g->weight_format != GR00T_WFMT_FP8)
    return bad(GR00T_EINVAL, "unknown weight_format");
  if (g->weight_format == GR00T_WFMT_FP8) {
    if (g->dtype != GR00T_DTYPE_BF16) return bad(GR00T_EINVAL, "FP8 weights need dtype BF16");
    if (g->hidden % 128 || g->mlp_dim % 128 || (g->q_heads * g->head_dim) % 128)
      return bad(GR00T_EINVAL, "FP8 weights need hidden, mlp_dim and q_heads*head_dim multiples of 128");
  }
  if (g->context_dim < 0 || g->context_dim > 16384 || g->context_dim % 64)
    return bad(GR00T_EINVAL, "context_dim must be 0 or a multiple of 64 up to 16384");
  if (g->context_dim > 0 && g->family != GR00T_FAMILY_DIT)
    return bad(GR00T_EINVAL, "context_dim (bind-time cross K/V projection) is a DiT-family field");
  if (g->state_dim < 0 || g->state_dim > 4096) return bad(GR00T_EINVAL, "state_dim must be in [0, 4096]");
  if (g->state_dim > 0 && (g->family != GR00T_FAMILY_DIT || g->state_tokens < 1))
    return bad(GR00T_EINVAL, "state_dim (bind-time state encoder) needs the DiT family with state_tokens >= 1");
  if (g->family == GR00T_FAMILY_EXPERT) {
    if (g->kv_heads != 1)
      return bad(GR00T_EINVAL, "expert family needs kv_heads == 1 (the head fold is exact only with one KV head)");
    if (g->state_tokens != 0) return bad(GR00T_EINVAL, "expert family has no state tokens");
    if (!(g->rope_theta > 0.f)) return bad(GR00T_EINVAL, "rope_theta must be > 0");
  } else {
    if (g->kv_heads != g->q_heads) return bad(GR00T_EINVAL, "DiT family needs kv_heads == q_heads");
    if (g->state_tokens < 0 || g->state_tokens > 16) return bad(GR00T_EINVAL, "state_tokens out of range");
    if (g->max_prefix < 1) return bad(GR00T_EINVAL, "DiT family needs max_prefix >= 1");
    if (g->q_heads * g->head_dim != g->hidden)
      return bad(GR00T_EINVAL, "DiT family needs q_heads*head_dim == hidden");
  }
  const long long mmax = (long long)g->max_batch * (g->horizon + g->state_tokens);
  if (mmax > (1 << 24)) return bad(GR00T_EINVAL, "max_batch * tokens too large");
  if (msg && len) msg[0] = 0;
  return GR00T_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Plan {
  std::vector<std::pair<void**, size_t>> req;
  void add(void** p, size_t bytes) { req.emplace_back(p, bytes); }
  size_t total() const {
    size_t t = 0;
    for (auto& r : req) t += align256(r.second);
    return t;
  }
};

void plan_buffers(gr00t_ctx* c, Plan& pl) {
  const size_t es = c->esz;
  const int L = c->L, D = c->D, E = c->E;
  const bool dit = c->g.family == GR00T_FAMILY_DIT;
  c->w_qkv.assign(L, nullptr);
  c->w_o.assign(L, nullptr);
  c->w_up.assign(L, nullptr);
  c->w_down.assign(L, nullptr);
  c->s_qkv.assign(L, nullptr);
  c->s_o.assign(L, nullptr);
  c->s_up.assign(L, nullptr);
  c->s_down.assign(L, nullptr);
  const int up_rows = (c->g.mlp_kind == GR00T_MLP_GEGLU ? 2 : 1) * c->F;
  const size_t wes = c->fp8w ? 1 : es;   // bytes per element of the per-layer projections
  for (int l = 0; l < L; ++l) {
    pl.add(&c->w_qkv[l], (size_t)c->nqkv[l] * D * wes);
    pl.add(&c->w_o[l], (size_t)D * c->qd * wes);
    pl.add(&c->w_up[l], (size_t)up_rows * D * wes);
    pl.add(&c->w_down[l], (size_t)D * c->F * wes);
    if (c->fp8w) {
      pl.add((void**)&c->s_qkv[l], (size_t)c->nqkv[l] * 4);
      pl.add((void**)&c->s_o[l], (size_t)D * 4);
      pl.add((void**)&c->s_up[l], (size_t)up_rows * 4);
      pl.add((void**)&c->s_down[l], (size_t)D * 4);
    }
  }
  if (c->g.time_mlp) {
    pl.add(&c->w_tin, (size_t)E * E * es);
    pl.add(&c->w_tout, (size_t)E * E * es);
    pl.add((void**)&c->b_tin, (size_t)E * 4);
    pl.add((void**)&c->b_tout, (size_t)E * 4);
  }
  pl.add(&c->w_cond, (size_t)c->S * c->R * E * es);
  pl.add((void**)&c->b_cond, (size_t)c->S * c->R * 4);
  if (!dit) {
    pl.add(&c->w_in, (size_t)D * c->A * es);
    pl.add((void**)&c->b_in, (size_t)D * 4);
  } else {
    pl.add(&c->w_enc1, (size_t)D * c->A * es);
    pl.add((void**)&c->b_enc1, (size_t)D * 4);
    pl.add(&c->w_enc2, (size_t)D * (D + E) * es);
    pl.add((void**)&c->b_enc2, (size_t)D * 4);
    pl.add(&c->w_enc3, (size_t)D * D * es);
    pl.add((void**)&c->b_enc3, (size_t)D * 4);
  }
  pl.add(&c->w_out, (size_t)c->A * D * es);
  pl.add((void**)&c->b_out, (size_t)c->A * 4);
  if (dit && c->g.state_dim > 0) {
    const size_t rows = (size_t)c->g.max_batch * c->Ns;
    pl.add(&c->w_s1, (size_t)D * c->Ks * es);
    pl.add((void**)&c->b_s1, (size_t)D * 4);
    pl.add(&c->w_s2, (size_t)D * D * es);
    pl.add((void**)&c->b_s2, (size_t)D * 4);
    pl.add(&c->state_in, rows * c->Ks * es);
    pl.add(&c->state_hid, rows * D * es);
    pl.add((void**)&c->state_tok, rows * D * 4);
  }
  c->w_ck.assign(L, nullptr);
  c->w_cv.assign(L, nullptr);
  c->ctx_k.assign(L, nullptr);
  c->ctx_v.assign(L, nullptr);
  if (dit && c->g.context_dim > 0) {
    const size_t kd = (size_t)c->Hkv * c->Dh, Dc = (size_t)c->g.context_dim;
    const size_t rows = (size_t)c->g.max_batch * c->g.max_prefix;
    for (int l = 0; l < L; l += 2) {
      pl.add(&c->w_ck[l], kd * Dc * es);
      pl.add(&c->w_cv[l], kd * Dc * es);
      pl.add(&c->ctx_k[l], rows * kd * es);
      pl.add(&c->ctx_v[l], rows * kd * es);
    }
    pl.add(&c->ctx_feat, rows * Dc * es);
  }

  int nq = 0;
  for (int v : c->nqkv) nq = v > nq ? v : nq;
  const size_t M = c->Mmax;
  const size_t MA = (size_t)c->g.max_batch * c->H;
  pl.add((void**)&c->h, M * D * 4);
  pl.add(&c->n, M * D * es);
  pl.add(&c->qkv, M * nq * es);
  pl.add(&c->att, M * c->qd * es);
  pl.add(&c->u, M * c->F * es);
  pl.add((void**)&c->x, MA * c->A * 4);
  pl.add((void**)&c->xtmp, MA * c->A * 4);
  if (dit) {
    pl.add(&c->a_enc, MA * D * es);
    pl.add(&c->e_enc, MA * D * es);
  }
  const size_t TB = (size_t)c->g.max_steps * c->g.max_batch;
  pl.add(&c->temb, TB * E * es);
  if (c->g.time_mlp) {
    pl.add(&c->t1, TB * E * es);
    pl.add(&c->cvec, TB * E * es);
  }
  pl.add(&c->mod, TB * c->S * c->R * es);
  pl.add((void**)&c->dts, (size_t)c->g.max_steps * 4);
  if (dit) pl.add((void**)&c->atb, (size_t)c->g.max_steps * D * 4);
  if (!dit) pl.add((void**)&c->rope_tab, (size_t)c->H * (c->Dh / 2) * sizeof(float2));
  pl.add((void**)&c->table, (size_t)(2 * L + 3) * sizeof(void*));
  // split-K plans keep tiles * S <= 17/16 of the SM count; BN <= 256, 128 rows each
  c->gemm_ws_floats = (long long)(c->sm_count + c->sm_count / 16 + 1) * 256 * 128;
  pl.add((void**)&c->gemm_ws, (size_t)c->gemm_ws_floats * 4);
  pl.add((void**)&c->err_flag, 64);
  pl.add((void**)&c->never_set, 64);
}

// Copy one weight matrix [rows][cols] into library memory, re-laid-out by ``mode``.
int upload_matrix(gr00t_ctx* c, const void* src, bool on_dev, void* dst, int rows, int cols,
                  int mode, int p0, int p1, void* staging, size_t esz = 0) {
  const size_t row_bytes = (size_t)cols * (esz ? esz : c->esz);
  const size_t bytes = row_bytes * rows;
  if (mode == PERM_NONE) {
    CK(c, cudaMemcpyAsync(dst, src, bytes, on_dev ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                          c->stream));
    return GR00T_OK;
  }
  const void* s = src;
  if (!on_dev || ((uintptr_t)src & 15)) {
    CK(c, cudaMemcpyAsync(staging, src, bytes, on_dev ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                          c->stream));
    s = staging;
  }
  CK(c, permute_rows(s, dst, rows, (int)row_bytes, mode, p0, p1, c->stream));
  // the staging buffer is reused by the next matrix: order host copies after this permute
  CK(c, cudaStreamSynchronize(c->stream));
  return GR00T_OK;
}

// One fp32 scale per row of an FP8 matrix, re-ordered like its rows.
int upload_scales(gr00t_ctx* c, const void* src, bool on_dev, float* dst, int rows, int mode, int p0, int p1,
                  void* staging) {
  const void* s = src;
  if (!on_dev || ((uintptr_t)src & 3)) {
    CK(c, cudaMemcpyAsync(staging, src, (size_t)rows * 4, on_dev ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                          c->stream));
    s = staging;
  }
  CK(c, permute_floats((const float*)s, dst, rows, mode, p0, p1, c->stream));
  CK(c, cudaStreamSynchronize(c->stream));
  return GR00T_OK;
}

int upload_bias(gr00t_ctx* c, const void* src, bool on_dev, float* dst, long long n, void* staging) {
  const void* s = src;
  if (!on_dev) {
    CK(c, cudaMemcpyAsync(staging, src, n * c->esz, cudaMemcpyHostToDevice, c->stream));
    s = staging;
  }
  CK(c, to_f32(c->dt, s, dst, n, c->stream));
  CK(c, cudaStreamSynchronize(c->stream));
  return GR00T_OK;
}

int check_weights(gr00t_ctx* c, const gr00t_weights* w) {
  if (!w) return set_err(c, GR00T_EINVAL, "weights is NULL");
  if (w->location != GR00T_MEM_HOST && w->location != GR00T_MEM_DEVICE)
    return set_err(c, GR00T_EINVAL, "weights.location must be GR00T_MEM_HOST or GR00T_MEM_DEVICE");
  const bool dit = c->g.family == GR00T_FAMILY_DIT;
  if (!w->cond_w || !w->cond_b || !w->action_out_w || !w->action_out_b)
    return set_err(c, GR00T_EINVAL, "cond_w/cond_b/action_out_w/action_out_b are required");
  if (c->g.time_mlp && (!w->time_mlp_in_w || !w->time_mlp_in_b || !w->time_mlp_out_w || !w->time_mlp_out_b))
    return set_err(c, GR00T_EINVAL, "time_mlp set but time MLP weights missing");
  if (!dit && (!w->action_in_w || !w->action_in_b))
    return set_err(c, GR00T_EINVAL, "expert family needs action_in_w/action_in_b");
  if (dit && (!w->enc_w1 || !w->enc_b1 || !w->enc_w2 || !w->enc_b2 || !w->enc_w3 || !w->enc_b3))
    return set_err(c, GR00T_EINVAL, "DiT family needs enc_w1..enc_b3");
  if (!w->qkv_w || !w->o_w || !w->up_w || !w->down_w)
    return set_err(c, GR00T_EINVAL, "per-layer weight arrays are required");
  for (int l = 0; l < c->L; ++l)
    if (!w->qkv_w[l] || !w->o_w[l] || !w->up_w[l] || !w->down_w[l])
      return set_err(c, GR00T_EINVAL, "layer %d has a NULL weight", l);
  if (c->g.context_dim > 0) {
    if (!w->cross_k_w || !w->cross_v_w)
      return set_err(c, GR00T_EINVAL, "context_dim set: the cross_k_w / cross_v_w arrays are required");
    for (int l = 0; l < c->L; l += 2)
      if (!w->cross_k_w[l] || !w->cross_v_w[l]) return set_err(c, GR00T_EINVAL, "block %d has a NULL cross weight", l);
  }
  if (c->g.state_dim > 0 && (!w->state_w1 || !w->state_b1 || !w->state_w2 || !w->state_b2))
    return set_err(c, GR00T_EINVAL, "state_dim set: the state encoder weights state_w1..state_b2 are required");
  if (c->fp8w) {
    if (!w->qkv_s || !w->o_s || !w->up_s || !w->down_s)
      return set_err(c, GR00T_EINVAL, "FP8 weights need the per-layer scale arrays qkv_s/o_s/up_s/down_s");
    for (int l = 0; l < c->L; ++l)
      if (!w->qkv_s[l] || !w->o_s[l] || !w->up_s[l] || !w->down_s[l])
        return set_err(c, GR00T_EINVAL, "layer %d has a NULL scale", l);
  }
  return GR00T_OK;
}

int upload_weights(gr00t_ctx* c, const gr00t_weights* w) {
  const bool on_dev = w->location == GR00T_MEM_DEVICE;
  const int D = c->D, E = c->E;
  const bool dit = c->g.family == GR00T_FAMILY_DIT;
  const bool geglu = c->g.mlp_kind == GR00T_MLP_GEGLU;
  // staging: the largest matrix
  size_t big = (size_t)c->S * c->R * E;
  big = std::max(big, (size_t)c->Hkv * c->Dh * (size_t)c->g.context_dim);
  for (int l = 0; l < c->L; ++l) {
    big = std::max(big, (size_t)c->nqkv[l] * D);
    big = std::max(big, (size_t)(geglu ? 2 : 1) * c->F * D);
  }
  void* staging = nullptr;
  CK(c, cudaMalloc(&staging, big * c->esz + 256));
  int rc = GR00T_OK;
  auto M = [&](const void* s, void* d, int rows, int cols, int mode, int p0, int p1) {
    if (rc == GR00T_OK) rc = upload_matrix(c, s, on_dev, d, rows, cols, mode, p0, p1, staging);
  };
  // per-layer projections: E4M3 codes (1 byte) and their row scales when fp8w
  auto P = [&](const void* s, const void* sc, void* d, float* dsc, int rows, int cols, int mode, int p0, int p1) {
    if (rc == GR00T_OK)
      rc = upload_matrix(c, s, on_dev, d, rows, cols, mode, p0, p1, staging, c->fp8w ? 1 : c->esz);
    if (rc == GR00T_OK && c->fp8w) rc = upload_scales(c, sc, on_dev, dsc, rows, mode, p0, p1, staging);
  };
  auto Bv = [&](const void* s, float* d, long long n) {
    if (rc == GR00T_OK) rc = upload_bias(c, s, on_dev, d, n, staging);
  };
  for (int l = 0; l < c->L; ++l) {
    const bool rope = !dit;  // expert: q heads and the k head carry rotate-half RoPE
    auto sc = [&](const void* const* a) { return c->fp8w ? a[l] : nullptr; };
    P(w->qkv_w[l], sc(w->qkv_s), c->w_qkv[l], c->s_qkv[l], c->nqkv[l], D, rope ? PERM_ROPE : PERM_NONE,
      (c->Hq + c->Hkv) * c->Dh, c->Dh);
    P(w->o_w[l], sc(w->o_s), c->w_o[l], c->s_o[l], D, c->qd, PERM_NONE, 0, 0);
    P(w->up_w[l], sc(w->up_s), c->w_up[l], c->s_up[l], (geglu ? 2 : 1) * c->F, D, geglu ? PERM_GEGLU : PERM_NONE,
      c->F, 0);
    P(w->down_w[l], sc(w->down_s), c->w_down[l], c->s_down[l], D, c->F, PERM_NONE, 0, 0);
  }
  if (c->g.time_mlp) {
    M(w->time_mlp_in_w, c->w_tin, E, E, PERM_NONE, 0, 0);
    M(w->time_mlp_out_w, c->w_tout, E, E, PERM_NONE, 0, 0);
    Bv(w->time_mlp_in_b, c->b_tin, E);
    Bv(w->time_mlp_out_b, c->b_tout, E);
  }
  M(w->cond_w, c->w_cond, c->S * c->R, E, PERM_NONE, 0, 0);
  Bv(w->cond_b, c->b_cond, (long long)c->S * c->R);
  if (!dit) {
    M(w->action_in_w, c->w_in, D, c->A, PERM_NONE, 0, 0);
    Bv(w->action_in_b, c->b_in, D);
  } else {
    M(w->enc_w1, c->w_enc1, D, c->A, PERM_NONE, 0, 0);
    Bv(w->enc_b1, c->b_enc1, D);
    M(w->enc_w2, c->w_enc2, D, D + E, PERM_NONE, 0, 0);
    Bv(w->enc_b2, c->b_enc2, D);
    M(w->enc_w3, c->w_enc3, D, D, PERM_NONE, 0, 0);
    Bv(w->enc_b3, c->b_enc3, D);
  }
  M(w->action_out_w, c->w_out, c->A, D, PERM_NONE, 0, 0);
  Bv(w->action_out_b, c->b_out, c->A);
  if (dit && c->g.state_dim > 0 && rc == GR00T_OK) {
    // W_s1 [D][state_dim] into [D][Ks], zero columns past state_dim (the tensor-core GEMM's K)
    cudaError_t e = cudaMemsetAsync(c->w_s1, 0, (size_t)D * c->Ks * c->esz, c->stream);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(c->w_s1, (size_t)c->Ks * c->esz, w->state_w1, (size_t)c->g.state_dim * c->esz,
                            (size_t)c->g.state_dim * c->esz, D, on_dev ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                            c->stream);
    if (e != cudaSuccess) rc = set_err(c, GR00T_ECUDA, "state encoder upload failed: %s", cudaGetErrorString(e));
    M(w->state_w2, c->w_s2, D, D, PERM_NONE, 0, 0);
    Bv(w->state_b1, c->b_s1, D);
    Bv(w->state_b2, c->b_s2, D);
  }
  if (dit && c->g.context_dim > 0)
    for (int l = 0; l < c->L; l += 2) {
      M(w->cross_k_w[l], c->w_ck[l], c->Hkv * c->Dh, c->g.context_dim, PERM_NONE, 0, 0);
      M(w->cross_v_w[l], c->w_cv[l], c->Hkv * c->Dh, c->g.context_dim, PERM_NONE, 0, 0);
    }
  cudaError_t e1 = cudaStreamSynchronize(c->stream);
  cudaError_t e2 = cudaFree(staging);
  if (rc != GR00T_OK) return rc;
  if (e1 != cudaSuccess || e2 != cudaSuccess)
    return set_err(c, GR00T_ECUDA, "weight upload failed: %s",
                   cudaGetErrorString(e1 != cudaSuccess ? e1 : e2));
  return GR00T_OK;
}

// ---- the step ------------------------------------------------------------------

// Launch stamps: with GR00T_OPT_TIME_KERNELS set, every kernel launch of the
// loop gets its own slot of a device array into which it writes the global
// timer when its dependency wait returns (kstamp); consecutive stamps bound
// each launch's share of the chain without changing the launches themselves.
unsigned long long* next_ts(gr00t_ctx* c, int cls) {
  if (!c->stamp_on || !c->in_loop || !c->stamps || c->stamp_used >= c->stamp_cap) return nullptr;
  c->stamp_cls.push_back(cls);
  return c->stamps + c->stamp_used++;
}

const CUtensorMap* tmap(gr00t_ctx* c, const void* ptr, long long rows, long long cols, long long ld,
                        int box_rows) {
  auto key = std::make_tuple(ptr, rows, cols, ld, box_rows);
  auto it = c->tmaps.find(key);
  if (it != c->tmaps.end()) return &it->second;
  CUtensorMap m;
  // box_rows -1: E4M3 codes (uint8, 128 x 128-byte boxes); -2: a bf16 GEMM output for
  // tensor stores (16 columns x 32 rows); <= -100: fp32 split partials [S = -100 - box_rows]
  // [rows][cols] for tensor stores (32 x 32 boxes); else bf16, 64 columns x box_rows
  const cudaError_t e = box_rows <= -100 ? tc_make_part_map(&m, ptr, rows, cols, ld, -100 - box_rows)
                        : box_rows == -2 ? tc_make_out_map(&m, ptr, rows, cols, ld)
                        : box_rows < 0 ? tc_make_map_e4m3(&m, ptr, rows, cols, ld)
                                       : tc_make_map(&m, ptr, rows, cols, ld, box_rows);
  if (e != cudaSuccess) return nullptr;
  if (c->no_host_alloc) {
    // the allocation-free step adds nothing to the cache: the descriptor goes to
    // a fixed slot of the context (kernels take descriptors by value at launch)
    CUtensorMap* slot = &c->tmap_spill[c->tmap_spill_next++ % kSpillMaps];
    *slot = m;
    return slot;
  }
  return &c->tmaps.emplace(key, m).first->second;
}

// The split-K plan of a tensor-core GEMM (E4M3 weights: stages of 128 K elements).
TcPlan plan_of(gr00t_ctx* c, int M, int N, int K, bool e4m3, bool partial) {
  const int cap = partial ? c->resid_split_cap : c->split_cap;
  return e4m3 ? tc_plan_e4m3(M, N, K, c->sm_count, cap, partial) : tc_plan(M, N, K, c->sm_count, cap, partial);
}
TcPlan plan_of(gr00t_ctx* c, const GemmArgs& a, bool partial) {
  return plan_of(c, a.M, a.N, a.K, a.epi.wscale != nullptr, partial);
}

bool tc_ok(gr00t_ctx* c, int M, int N, int K, bool e4m3) {
  if (c->dt != DT_BF16 || c->opt_gemm != 0) return false;
  return e4m3 ? tc_supported_e4m3(M, N, K) : tc_supported(M, N, K);
}
bool tc_ok(gr00t_ctx* c, const GemmArgs& a) { return tc_ok(c, a.M, a.N, a.K, a.epi.wscale != nullptr); }

int gemm(gr00t_ctx* c, GemmArgs a, int cls = GR00T_KCLASS_OTHER) {
  ++c->launches;
  a.epi.ts = next_ts(c, cls);
  if (a.epi.wscale) {   // E4M3 weights: the tensor-core path is the only one
    if (!tc_ok(c, a))
      return set_err(c, GR00T_EUNSUPPORTED, "FP8 weights need the tensor-core GEMM (GEMM path 0, K %% 128 == 0)");
    const TcPlan p = plan_of(c, a, a.epi.kind == EPI_PARTIAL);
    const CUtensorMap* tw = tmap(c, a.W, a.N, a.K, a.ldw, -1);
    const CUtensorMap* tx = tmap(c, a.A, a.M, a.K, a.lda, p.BN);
    if (!tw || !tx) return set_err(c, GR00T_ECUDA, "TMA descriptor encode failed (alignment?)");
    CK(c, gemm_tc_e4m3(*tw, *tx, a, p, c->gemm_ws, c->gemm_ws_floats, c->err_flag, c->wait_limit, c->stream,
                       c->opt_pdl != 0));
    return GR00T_OK;
  }
  if (c->dt == DT_BF16 && c->opt_gemm == 0 && tc_supported(a.M, a.N, a.K)) {
    const bool partial = a.epi.kind == EPI_PARTIAL;
    TcPlan p = tc_plan(a.M, a.N, a.K, c->sm_count, partial ? c->resid_split_cap : c->split_cap, partial);
    const bool pers = c->opt_persistent && tc_use_persistent(p, a.M);
    // persistent tiles over two or more weight tiles: pairs of CTAs share each activation tile
    if (pers && c->opt_mcast && (a.N + 127) / 128 >= 2) p.CL = 2;
    const CUtensorMap* tw = tmap(c, a.W, a.N, a.K, a.ldw, 128);
    const CUtensorMap* tx = tmap(c, a.A, a.M, a.K, a.lda, p.BN / p.CL);
    if (!tw || !tx) return set_err(c, GR00T_ECUDA, "TMA descriptor encode failed (alignment?)");
    const CUtensorMap* to = nullptr;
    if (pers && c->opt_tstore && tc_tstore_ok(a.epi, a.N)) {
      // the persistent GEMM's outputs leave by tensor stores
      to = tmap(c, a.epi.out, a.M, a.epi.kind == EPI_GEGLU ? a.N / 2 : a.N, a.epi.ldo, -2);
      a.epi.tstore = to ? 1 : 0;
    }
    if (pers)
      CK(c, gemm_tc_persistent_launch(*tw, *tx, to, a, p, c->sm_count, c->err_flag, c->wait_limit, c->stream,
                                      c->opt_pdl != 0));
    else {
      if (a.epi.kind == EPI_PARTIAL && p.BN <= 128 && c->opt_tstore && tc_partial_tstore_ok(a.epi, a.N)) {
        // the split partials of tiles of up to 128 tokens leave by tensor stores (measured:
        // faster for 64-token tiles; 256-token tiles keep the per-lane stores, which already
        // write whole 128-byte lines, where staging only adds shared-memory traffic)
        to = tmap(c, a.epi.out, a.M, a.N, a.epi.ldo, -100 - p.S);
        a.epi.tstore = to ? 1 : 0;
      }
      CK(c, gemm_tc(*tw, *tx, to, a, p, c->gemm_ws, c->gemm_ws_floats, c->err_flag, c->wait_limit, c->stream,
                    c->opt_pdl != 0));
    }
  } else {
    CK(c, gemm_simt(c->dt, a, c->stream, c->opt_pdl != 0));
  }
  return GR00T_OK;
}

// Residual GEMM h += gate * (A W^T).  When the tensor-core plan splits K, the
// S fp32 partials go to the scratch workspace and the next norm / out_proj
// kernel folds them into h (pending), saving a reduction phase here.
int gemm_resid(gr00t_ctx* c, GemmArgs a, int cls) {
  if (tc_ok(c, a)) {
    const TcPlan p = plan_of(c, a, true);
    if (p.S > 1 && (long long)p.S * a.M * a.N <= c->gemm_ws_floats) {
      c->pending.part = c->gemm_ws;
      c->pending.S = p.S;
      c->pending.M = a.M;
      c->pending.gate = a.epi.kind == EPI_RESID_GATED ? a.epi.gate : nullptr;
      a.epi.kind = EPI_PARTIAL;
      a.epi.out = c->gemm_ws;
      a.epi.ldo = a.N;
    }
  }
  const int rc = gemm(c, a, cls);
  if (rc != GR00T_OK) c->pending = gr00t_ctx::Pending();   // nothing was enqueued to fold
  return rc;
}

// Attach (and clear) pending partials to the next norm's arguments.
NormArgs take_pending(gr00t_ctx* c, NormArgs na) {
  na.part = c->pending.part;
  na.part_S = c->pending.S;
  na.part_M = c->pending.M;
  na.gate = c->pending.gate;
  c->pending = gr00t_ctx::Pending();
  return na;
}

#define RC(x)                          \
  do {                                 \
    int rc_ = (x);                     \
    if (rc_ != GR00T_OK) return rc_;   \
  } while (0)

inline const char* ptr_at(const void* p, long long elems, size_t esz) {
  return (const char*)p + elems * (long long)esz;
}

// Test hook (GR00T_OPT_TEST_STALL): a bounded wait on a word nothing writes,
// enqueued ahead of a step, so the bounded-wait error path can be exercised
// without any copy or tensor-core operation in flight.
int stall_probe(gr00t_ctx* c) {
  if (!c->opt_stall) return GR00T_OK;
  ++c->launches;
  CK(c, bounded_wait_probe(c->never_set, c->err_flag, c->opt_stall, c->stream));
  return GR00T_OK;
}

// Residual stream after block ``layer`` into the dump target (gr00t_debug_dump).
int dump_h(gr00t_ctx* c, int layer) {
  if (!c->dump_out || layer != c->dump_layer) return GR00T_OK;
  CK(c, cudaMemcpyAsync(c->dump_out, c->h, (size_t)c->bB * c->tok * c->D * sizeof(float),
                        cudaMemcpyDeviceToDevice, c->stream));
  return GR00T_OK;
}

// Enqueue one denoise step k on the stream: x (fp32 [B][H][A]) in; v_out
// (nullable) receives the velocity; with do_euler x += dt_k * v.
int enqueue_step(gr00t_ctx* c, int k, float* x, float* v_out, int do_euler) {
  c->launches = 0;
  c->pending = gr00t_ctx::Pending();   // partials of an earlier, failed enqueue are not this step's
  const int B = c->bB, P = c->bP, D = c->D, L = c->L, H = c->H, tok = c->tok;
  const int M = B * tok, MA = B * H, R = c->R;
  const long long bstride = (long long)c->S * R;
  const size_t es = c->esz;
  const char* mod_k = ptr_at(c->mod, (long long)k * B * bstride, es);
  const bool dit = c->g.family == GR00T_FAMILY_DIT;
  cudaStream_t s = c->stream;
  RC(stall_probe(c));

  auto site = [&](int si) { return (const void*)(mod_k + (long long)si * R * es); };
  // GR00T_OPT_L2_PREFETCH: each GEMM's idle warps pull the next GEMM's weights (and the
  // attention's bound K/V) into L2 while its own weights stream
  const size_t wes = c->fp8w ? 1 : es;
  const int up_rows = (c->g.mlp_kind == GR00T_MLP_GEGLU ? 2 : 1) * c->F;
  (void)up_rows;
  auto wbytes = [&](long long rows, long long cols) { return rows * cols * (long long)wes; };
  auto ahead = [&](GemmArgs& g, const void* p, long long bytes) {
    if (!c->opt_l2_ahead || !p || bytes <= 0) return;
    for (auto& slot : g.l2)
      if (!slot.p) {
        slot.p = p;
        slot.bytes = bytes;
        return;
      }
  };
  // Kernels read the modulation table before their programmatic-launch wait.
  // The table is written when the schedule is set, so the head of step 0 is
  // launched without the early-launch attribute: it (and so every later
  // kernel) starts only once that write has completed.
  const bool pdl_head = c->opt_pdl != 0 && k > 0 && !c->opt_stall;
  NormArgs base;
  base.eps = c->g.norm_eps;
  base.mod_bstride = bstride;
  base.tok = tok;
  auto norm = [&](NormArgs na) -> int {
    ++c->launches;
    na.ts = next_ts(c, GR00T_KCLASS_NORM);
    CK(c, adanorm(c->dt, c->h, D, M, c->n, take_pending(c, na), s, c->opt_pdl != 0));
    return GR00T_OK;
  };

  if (!dit) {
    NormArgs na = base;
    na.kind = NORM_RMS;
    na.mod = site(0);
    na.scale_off = 0;
    na.shift_off = D;
    ++c->launches;
    {
      NormArgs nh = na;
      nh.ts = next_ts(c, GR00T_KCLASS_NORM);
      CK(c, expert_in(c->dt, x, c->A, c->w_in, c->b_in, c->h, D, M, c->n, nh, s, pdl_head));
    }
    RC(dump_h(c, -1));
    const int nq = c->nqkv[0];
    for (int l = 0; l < L; ++l) {
      GemmArgs g;
      g.A = c->n; g.lda = D; g.W = c->w_qkv[l]; g.ldw = D; g.M = M; g.N = nq; g.K = D;
      g.epi.wscale = c->fp8w ? c->s_qkv[l] : nullptr;
      g.epi.kind = EPI_ROPE; g.epi.out = c->qkv; g.epi.ldo = nq;
      g.epi.rope_cols = (c->Hq + 1) * c->Dh; g.epi.hd = c->Dh; g.epi.rope_tab = c->rope_tab;
      g.epi.tok_rope = tok;
      // while this GEMM streams its weights: the O projection's weights and this layer's
      // prefix K/V into L2 (a bound pool keeps samples ``capacity`` rows apart, so only a
      // flat binding's K/V is one contiguous range)
      ahead(g, c->w_o[l], wbytes(D, c->qd));
      if (P > 0 && c->pool.empty()) {
        ahead(g, c->host_table[2 * l], (long long)B * P * c->Dh * es);
        ahead(g, c->host_table[2 * l + 1], (long long)B * P * c->Dh * es);
      }
      RC(gemm(c, g, GR00T_KCLASS_QKV_GEMM));

      ++c->launches;
      // bf16: the tcgen05 kernel (key splits merged by a second kernel when the
      // row tiles alone do not fill the GPU); the mma.sync and CUDA-core
      // kernels remain selectable
      if (c->dt == DT_BF16 && (c->opt_attn == 0 || c->opt_attn == 3) && attn_t5_supported(c->Dh, c->Hq)) {
        AttnT5Args a5;
        a5.qkv = c->qkv; a5.ldq = nq; a5.k_off = c->qd; a5.v_off = c->qd + c->Dh;
        a5.B = B; a5.H = H; a5.Hq = c->Hq; a5.Dh = c->Dh; a5.P = P;
        a5.out = c->att; a5.ldo = c->qd;
        a5.ws = c->gemm_ws; a5.ws_floats = c->gemm_ws_floats;
        a5.err = c->err_flag; a5.wait_limit = c->wait_limit;
        const int splits = attn_t5_splits(a5, c->sm_count, c->opt_attn_splits);
        if (!c->pool.empty()) {   // prefix rows at stride cap; this step's suffix K/V into slots [P, P + H)
          a5.ps = c->pool_cap;
          a5.pool_cap = c->pool_cap;
          a5.pool_k = c->pool[l];
          a5.pool_v = (char*)c->pool[l] + (size_t)B * c->pool_cap * c->Dh * es;
        }
        // the key-tile cluster pays where each CTA streams only a few key tiles, so the
        // latency of its first tiles dominates (batch 1: pi05 4.97 vs 5.46 us per launch);
        // over long key ranges it costs ~1 % (batch 8 with a 4096-token prefix, batch 32)
        const int key_tiles = (P + 63) / 64 + (H + 63) / 64;
        const bool few = (key_tiles + splits - 1) / splits <= 4;
        a5.ct = c->opt_attn_mcast == 1 || (c->opt_attn_mcast == 2 && few) ? attn_t5_cluster(a5) : 1;
        CUtensorMap maps[8];
        CK(c, attn_t5_maps(a5, c->host_table[2 * l], c->host_table[2 * l + 1], splits, maps));
        a5.ts = next_ts(c, GR00T_KCLASS_ATTENTION);
        if (splits > 1) {   // the split merge is a second kernel
          ++c->launches;
          a5.ts2 = next_ts(c, GR00T_KCLASS_ATTENTION);
        }
        CK(c, attention_t5(a5, maps, splits, s, c->opt_pdl != 0));
      } else if (!c->pool.empty()) {
        return set_err(c, GR00T_EUNSUPPORTED, "a bound K/V pool needs the tcgen05 attention (bf16, attention path 0 or 3)");
      } else if (c->dt == DT_BF16 && (c->opt_attn == 0 || c->opt_attn == 2) && attn_fold_supported(c->Dh)) {
        AttnFoldArgs af;
        af.qkv = c->qkv; af.ldq = nq; af.k_off = c->qd; af.v_off = c->qd + c->Dh;
        af.B = B; af.H = H; af.Hq = c->Hq; af.Dh = c->Dh; af.P = P;
        af.table = c->table; af.k_slot = 2 * l; af.v_slot = 2 * l + 1;
        af.out = c->att; af.ldo = c->qd;
        af.ws = c->gemm_ws; af.ws_floats = c->gemm_ws_floats;   // kernels run in order: one scratch
        af.ts = next_ts(c, GR00T_KCLASS_ATTENTION);
        CK(c, attention_fold(af, attn_fold_splits(af, c->sm_count), s, c->opt_pdl != 0));
      } else {
        AttnArgs at;
        at.q = c->qkv; at.ldq = nq; at.B = B; at.Tq = tok; at.Hq = c->Hq; at.Hkv = 1; at.Dh = c->Dh;
        at.table = c->table; at.k_slot = 2 * l; at.v_slot = 2 * l + 1; at.P = P;
        at.ks = ptr_at(c->qkv, (long long)c->qd, es); at.vs = ptr_at(c->qkv, (long long)c->qd + c->Dh, es);
        at.lds = nq; at.S = tok; at.out = c->att; at.ldo = c->qd;
        at.ts = next_ts(c, GR00T_KCLASS_ATTENTION);
        CK(c, attention_simt(c->dt, at, s, c->opt_pdl != 0));
      }

      GemmArgs go;
      go.A = c->att; go.lda = c->qd; go.W = c->w_o[l]; go.ldw = c->qd; go.M = M; go.N = D; go.K = c->qd;
      go.epi.wscale = c->fp8w ? c->s_o[l] : nullptr;
      go.epi.kind = EPI_RESID_GATED; go.epi.resid = c->h; go.epi.ldr = D;
      go.epi.gate = ptr_at(site(2 * l), 2LL * D, es); go.epi.gate_bstride = bstride; go.epi.tok = tok;
      ahead(go, c->w_up[l], wbytes(up_rows, D));
      RC(gemm_resid(c, go, GR00T_KCLASS_O_GEMM));

      NormArgs n2 = na;
      n2.mod = site(2 * l + 1);
      RC(norm(n2));

      GemmArgs gu;
      gu.A = c->n; gu.lda = D; gu.W = c->w_up[l]; gu.ldw = D; gu.M = M; gu.K = D;
      gu.epi.wscale = c->fp8w ? c->s_up[l] : nullptr;
      if (c->g.mlp_kind == GR00T_MLP_GEGLU) {
        gu.N = 2 * c->F; gu.epi.kind = EPI_GEGLU;
      } else {
        gu.N = c->F; gu.epi.kind = EPI_STORE; gu.epi.act = ACT_GELU;
      }
      gu.epi.out = c->u; gu.epi.ldo = c->F;
      ahead(gu, c->w_down[l], wbytes(D, c->F));
      RC(gemm(c, gu, GR00T_KCLASS_UP_GEMM));

      GemmArgs gd;
      gd.A = c->u; gd.lda = c->F; gd.W = c->w_down[l]; gd.ldw = c->F; gd.M = M; gd.N = D; gd.K = c->F;
      gd.epi.wscale = c->fp8w ? c->s_down[l] : nullptr;
      gd.epi.kind = EPI_RESID_GATED; gd.epi.resid = c->h; gd.epi.ldr = D;
      gd.epi.gate = ptr_at(site(2 * l + 1), 2LL * D, es); gd.epi.gate_bstride = bstride; gd.epi.tok = tok;
      ahead(gd, c->w_qkv[(l + 1) % L], wbytes(c->nqkv[(l + 1) % L], D));
      RC(gemm_resid(c, gd, GR00T_KCLASS_DOWN_GEMM));

      if (l + 1 < L) {
        NormArgs n3 = na;
        n3.mod = site(2 * l + 2);
        RC(norm(n3));   // folds this layer's down partials into h
        RC(dump_h(c, l));
      }
    }
    NormArgs nf = na;
    nf.mod = site(2 * L);
    if (c->dump_out && c->dump_layer == L - 1) {
      // dump of the last layer: fold its partials into h first (the step tail folds
      // them without writing h back)
      NormArgs nd = na;
      nd.mod = nullptr;
      RC(norm(nd));
      RC(dump_h(c, L - 1));
    }
    ++c->launches;
    nf.ts = next_ts(c, GR00T_KCLASS_NORM);
    CK(c, out_euler(c->dt, c->h, D, MA, H, 0, c->w_out, c->b_out, c->A, take_pending(c, nf), x, c->dts, k,
                    do_euler, v_out, s, c->opt_pdl != 0));
    return GR00T_OK;
  }

  // ---- DiT family ----
  const int E = c->E, Ns = c->Ns;
  ++c->launches;
  CK(c, dit_in(c->dt, x, c->A, c->w_enc1, c->b_enc1, c->a_enc, D, MA, (const float*)c->host_table[2 * L + 2],
               Ns, tok, B, c->h, s, pdl_head, next_ts(c, GR00T_KCLASS_NORM)));
  {
    GemmArgs g;  // e = swish(a W2[:, :D]^T + atb_k), atb_k holds W2's time half and b2
    g.A = c->a_enc; g.lda = D; g.W = c->w_enc2; g.ldw = D + E; g.M = MA; g.N = D; g.K = D;
    g.epi.kind = EPI_STORE; g.epi.act = ACT_SWISH; g.epi.bias = c->atb + (long long)k * D;
    g.epi.out = c->e_enc; g.epi.ldo = D;
    RC(gemm(c, g));
    GemmArgs g3a;  // action tokens into the residual rows after the state tokens
    g3a.A = c->e_enc; g3a.lda = D; g3a.W = c->w_enc3; g3a.ldw = D; g3a.M = MA; g3a.N = D; g3a.K = D;
    g3a.epi.kind = EPI_STORE; g3a.epi.out_f32 = 1; g3a.epi.bias = c->b_enc3; g3a.epi.out = c->h;
    g3a.epi.ldo = D; g3a.epi.rg = H; g3a.epi.rs = tok; g3a.epi.ro = Ns;
    RC(gemm(c, g3a));
  }
  RC(dump_h(c, -1));
  NormArgs na = base;
  na.kind = NORM_LN;
  na.scale_off = 0;
  na.shift_off = D;
  for (int i = 0; i < L; ++i) {
    NormArgs n1 = na;
    n1.mod = site(i);
    RC(norm(n1));   // folds block i-1's down partials into h
    RC(dump_h(c, i - 1));
    const int nq = c->nqkv[i];
    GemmArgs g;
    g.A = c->n; g.lda = D; g.W = c->w_qkv[i]; g.ldw = D; g.M = M; g.N = nq; g.K = D;
    g.epi.wscale = c->fp8w ? c->s_qkv[i] : nullptr;
    g.epi.kind = EPI_STORE; g.epi.out = c->qkv; g.epi.ldo = nq;
    ahead(g, c->w_o[i], wbytes(D, c->qd));
    if (i % 2 == 0) {   // the cross block's context K/V
      const long long kvb = (long long)B * P * c->Hkv * c->Dh * es;
      ahead(g, c->host_table[2 * i], kvb);
      ahead(g, c->host_table[2 * i + 1], kvb);
    }
    RC(gemm(c, g, GR00T_KCLASS_QKV_GEMM));
    AttnArgs at;
    at.q = c->qkv; at.ldq = nq; at.B = B; at.Tq = tok; at.Hq = c->Hq; at.Hkv = c->Hkv; at.Dh = c->Dh;
    at.table = c->table; at.out = c->att; at.ldo = c->qd;
    if (i % 2 == 0) {  // cross-attention into the bound VL context
      at.k_slot = 2 * i; at.v_slot = 2 * i + 1; at.P = P;
      at.mask_slot = (i % 4 == 0) ? 2 * L : 2 * L + 1;
      if (!c->host_table[at.mask_slot]) at.mask_slot = -1;
      at.S = 0;
    } else {  // self-attention over the state + action tokens
      at.P = 0; at.ks = ptr_at(c->qkv, (long long)c->qd, es); at.vs = ptr_at(c->qkv, 2LL * c->qd, es);
      at.lds = nq; at.S = tok;
    }
    ++c->launches;
    at.ts = next_ts(c, GR00T_KCLASS_ATTENTION);
    const void* kp = i % 2 == 0 ? c->host_table[2 * i] : nullptr;
    const void* vp = i % 2 == 0 ? c->host_table[2 * i + 1] : nullptr;
    if (c->dt == DT_BF16 && c->opt_attn == 0 && attn_dit_supported(at, kp, vp))
      CK(c, attention_dit(at, kp, vp, c->err_flag, c->wait_limit, s, c->opt_pdl != 0));
    else
      CK(c, attention_simt(c->dt, at, s, c->opt_pdl != 0));
    GemmArgs go;
    go.A = c->att; go.lda = c->qd; go.W = c->w_o[i]; go.ldw = c->qd; go.M = M; go.N = D; go.K = c->qd;
    go.epi.wscale = c->fp8w ? c->s_o[i] : nullptr;
    go.epi.kind = EPI_RESID; go.epi.resid = c->h; go.epi.ldr = D;
    ahead(go, c->w_up[i], wbytes(c->F, D));
    RC(gemm_resid(c, go, GR00T_KCLASS_O_GEMM));
    NormArgs n3 = na;
    n3.mod = nullptr;
    RC(norm(n3));
    GemmArgs gu;
    gu.A = c->n; gu.lda = D; gu.W = c->w_up[i]; gu.ldw = D; gu.M = M; gu.N = c->F; gu.K = D;
    gu.epi.wscale = c->fp8w ? c->s_up[i] : nullptr;
    gu.epi.kind = EPI_STORE; gu.epi.act = ACT_GELU; gu.epi.out = c->u; gu.epi.ldo = c->F;
    ahead(gu, c->w_down[i], wbytes(D, c->F));
    RC(gemm(c, gu, GR00T_KCLASS_UP_GEMM));
    GemmArgs gd;
    gd.A = c->u; gd.lda = c->F; gd.W = c->w_down[i]; gd.ldw = c->F; gd.M = M; gd.N = D; gd.K = c->F;
    gd.epi.wscale = c->fp8w ? c->s_down[i] : nullptr;
    gd.epi.kind = EPI_RESID; gd.epi.resid = c->h; gd.epi.ldr = D;
    ahead(gd, c->w_qkv[(i + 1) % L], wbytes(c->nqkv[(i + 1) % L], D));
    RC(gemm_resid(c, gd, GR00T_KCLASS_DOWN_GEMM));
  }
  NormArgs nf = na;
  nf.mod = site(L);
  nf.scale_off = D;  // final row splits (shift, scale)
  nf.shift_off = 0;
  if (c->dump_out && c->dump_layer == L - 1) {
    NormArgs nd = na;
    nd.mod = nullptr;
    RC(norm(nd));
    RC(dump_h(c, L - 1));
  }
  ++c->launches;
  nf.ts = next_ts(c, GR00T_KCLASS_NORM);
  CK(c, out_euler(c->dt, c->h, D, MA, H, Ns, c->w_out, c->b_out, c->A, take_pending(c, nf), x, c->dts, k,
                  do_euler, v_out, s, c->opt_pdl != 0));
  return GR00T_OK;
}

// Enqueue the T steps of the loop (the tail stamp closes the last launch's interval).
int enqueue_loop(gr00t_ctx* c) {
  c->stamp_used = 0;
  c->stamp_cls.clear();
  c->in_loop = true;
  int rc = GR00T_OK;
  for (int k = 0; k < c->sT && rc == GR00T_OK; ++k) rc = enqueue_step(c, k, c->x, nullptr, 1);
  unsigned long long* ts = rc == GR00T_OK ? next_ts(c, 0) : nullptr;
  c->in_loop = false;
  if (ts) CK(c, stamp_tail(ts, c->stream, c->opt_pdl != 0));
  return rc;
}

int ensure_graph(gr00t_ctx* c) {
  if (c->gexec && c->gT == c->sT && c->gB == c->bB && c->gP == c->bP) return GR00T_OK;
  if (c->gexec) {
    cudaGraphExecDestroy(c->gexec);
    c->gexec = nullptr;
  }
  cudaGraph_t graph = nullptr;
  CK(c, cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
  const int rc = enqueue_loop(c);
  cudaError_t e = cudaStreamEndCapture(c->stream, &graph);
  if (rc != GR00T_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (e != cudaSuccess) return set_err(c, GR00T_ECUDA, "graph capture failed: %s", cudaGetErrorString(e));
  e = cudaGraphInstantiate(&c->gexec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) {
    c->gexec = nullptr;
    return set_err(c, GR00T_ECUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
  }
  c->gT = c->sT;
  c->gB = c->bB;
  c->gP = c->bP;
  return GR00T_OK;
}

int check_ready(gr00t_ctx* c) {
  if (!c->bound) return set_err(c, GR00T_ESTATE, "no prefix K/V bound (call gr00t_bind_prefix_kv)");
  if (!c->scheduled) return set_err(c, GR00T_ESTATE, "no schedule (call gr00t_set_schedule)");
  if (c->bB != c->sB)
    return set_err(c, GR00T_ESTATE, "batch of the bind (%d) differs from the schedule's (%d)", c->bB, c->sB);
  return GR00T_OK;
}

int run_loop(gr00t_ctx* c) {
  if (c->opt_graph) {
    RC(ensure_graph(c));
    CK(c, cudaGraphLaunch(c->gexec, c->stream));
  } else {
    RC(enqueue_loop(c));
  }
  return GR00T_OK;
}

// Synchronise the stream and turn a set device error word into GR00T_ETIMEOUT
// (the word is cleared, so the context stays usable).
int sync_and_check(gr00t_ctx* c) {
  CK(c, cudaMemcpyAsync(c->err_host, c->err_flag, sizeof(int), cudaMemcpyDeviceToHost, c->stream));
  CK(c, cudaStreamSynchronize(c->stream));
  const int f = *(volatile int*)c->err_host;
  if (f != 0) {
    CK(c, cudaMemsetAsync(c->err_flag, 0, sizeof(int), c->stream));
    CK(c, cudaStreamSynchronize(c->stream));
    return set_err(c, GR00T_ETIMEOUT,
                   "a bounded device wait gave up (error word %d): the results of the work enqueued since the "
                   "last check are not valid", f);
  }
  return GR00T_OK;
}

void free_ctx(gr00t_ctx* c) {
  if (!c) return;
  if (c->stream) cudaStreamSynchronize(c->stream);
  if (c->gexec) cudaGraphExecDestroy(c->gexec);
  if (c->stamps) cudaFree(c->stamps);
  if (c->err_host) cudaFreeHost(c->err_host);
  if (c->arena) cudaFree(c->arena);
  if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
  delete c;
}
}  // namespace

// ---- exported ------------------------------------------------------------------

extern "C" int gr00t_validate_geometry(const gr00t_geometry* g, char* msg, size_t msg_len) {
  return validate(g, msg, msg_len);
}

extern "C" int gr00t_create(const gr00t_geometry* g, const gr00t_weights* w, void* stream,
                            gr00t_ctx** out) {
  if (!out) return set_err(nullptr, GR00T_EINVAL, "out is NULL");
  *out = nullptr;
  char msg[256];
  int rc = validate(g, msg, sizeof msg);
  if (rc != GR00T_OK) return set_err(nullptr, rc, "invalid geometry: %s", msg);

  // host-side checks of the geometry and the weight pointers first: nothing touches the GPU
  // before they pass
  gr00t_ctx* c = new gr00t_ctx();
  c->g = *g;
  c->dt = g->dtype == GR00T_DTYPE_BF16 ? DT_BF16 : DT_F32;
  c->esz = c->dt == DT_BF16 ? 2 : 4;
  c->fp8w = g->weight_format == GR00T_WFMT_FP8;
  c->D = g->hidden; c->L = g->layers; c->Hq = g->q_heads; c->Hkv = g->kv_heads; c->Dh = g->head_dim;
  c->F = g->mlp_dim; c->H = g->horizon; c->A = g->action_dim; c->Ns = g->state_tokens; c->E = g->time_dim;
  c->tok = c->H + c->Ns;
  c->qd = c->Hq * c->Dh;
  c->Ks = (g->state_dim + 63) / 64 * 64;
  const bool dit = g->family == GR00T_FAMILY_DIT;
  c->S = dit ? c->L + 1 : 2 * c->L + 1;
  c->R = (dit ? 2 : 3) * c->D;
  c->Mmax = g->max_batch * c->tok;
  c->nqkv.resize(c->L);
  for (int l = 0; l < c->L; ++l)
    c->nqkv[l] = (dit && l % 2 == 0) ? c->qd : c->qd + 2 * c->Hkv * c->Dh;
  rc = check_weights(c, w);
  if (rc != GR00T_OK) {
    g_create_err = c->err;
    delete c;
    return rc;
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  cudaDeviceProp prop;
  if (e == cudaSuccess) e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) {
    delete c;
    return set_err(nullptr, GR00T_ECUDA, "no CUDA device: %s", cudaGetErrorString(e));
  }
  if (!(prop.major == 10 && prop.minor == 3)) {
    delete c;
    return set_err(nullptr, GR00T_EUNSUPPORTED, "device %s is sm_%d%d; this library is built for sm_103a",
                   prop.name, prop.major, prop.minor);
  }
  c->sm_count = prop.multiProcessorCount;
  c->device = dev;
  if (stream) {
    c->stream = (cudaStream_t)stream;
  } else {
    e = cudaStreamCreate(&c->stream);
    if (e != cudaSuccess) {
      delete c;
      return set_err(nullptr, GR00T_ECUDA, "cudaStreamCreate failed: %s", cudaGetErrorString(e));
    }
    c->own_stream = true;
  }
  // the allocation-free step's fixed scratch array: the module holding it is loaded
  // (and the array placed on the device) here, so that step itself never is the first
  // to touch it
  e = noalloc_scratch(dev, &c->noalloc_addr);
  if (e == cudaSuccess) e = cudaMallocHost((void**)&c->err_host, 64);
  if (e != cudaSuccess) {
    set_err(nullptr, GR00T_ECUDA, "set-up failed: %s", cudaGetErrorString(e));
    free_ctx(c);
    return GR00T_ECUDA;
  }
  *c->err_host = 0;
  Plan pl;
  plan_buffers(c, pl);
  c->arena_bytes = pl.total();
  e = cudaMalloc((void**)&c->arena, c->arena_bytes);
  if (e != cudaSuccess) {
    c->arena = nullptr;
    set_err(nullptr, GR00T_ENOMEM, "cudaMalloc of %zu bytes failed: %s", c->arena_bytes, cudaGetErrorString(e));
    free_ctx(c);
    return GR00T_ENOMEM;
  }
  size_t off = 0;
  for (auto& r : pl.req) {
    *r.first = c->arena + off;
    off += align256(r.second);
  }
  rc = upload_weights(c, w);
  if (rc == GR00T_OK) {
    e = cudaMemsetAsync(c->err_flag, 0, 64, c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->never_set, 0, 64, c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->table, 0, (2 * c->L + 3) * sizeof(void*), c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) rc = set_err(c, GR00T_ECUDA, "init failed: %s", cudaGetErrorString(e));
  }
  if (rc != GR00T_OK) {
    g_create_err = c->err;
    free_ctx(c);
    return rc;
  }
  c->host_table.assign(2 * c->L + 3, nullptr);
  *out = c;
  return GR00T_OK;
}

extern "C" int gr00t_bind_prefix_kv(gr00t_ctx* c, int batch, int prefix, const void* const* k,
                                    const void* const* v, const uint8_t* text_mask,
                                    const uint8_t* image_mask, const float* state_tokens) {
  if (!c) return GR00T_EINVAL;
  const bool dit = c->g.family == GR00T_FAMILY_DIT;
  if (batch < 1 || batch > c->g.max_batch)
    return set_err(c, GR00T_EINVAL, "batch %d outside [1, %d]", batch, c->g.max_batch);
  if (prefix < (dit ? 1 : 0) || prefix > c->g.max_prefix)
    return set_err(c, GR00T_EINVAL, "prefix %d outside [%d, %d]", prefix, dit ? 1 : 0, c->g.max_prefix);
  if (!dit && (text_mask || image_mask))
    return set_err(c, GR00T_EINVAL, "the expert family takes no mask (its head fold needs the all-ones mask)");
  if (!dit && state_tokens) return set_err(c, GR00T_EINVAL, "the expert family has no state tokens");
  if (dit && c->Ns > 0 && !state_tokens) return set_err(c, GR00T_EINVAL, "state_tokens required");
  if (prefix > 0 && (!k || !v)) return set_err(c, GR00T_EINVAL, "k/v pointer arrays are NULL");
  if (dit && c->g.state_dim > 0 && state_tokens) {
    // the raw robot state [batch, Ns, state_dim] -> the library's state tokens [batch, Ns, D]
    const int M = batch * c->Ns, D = c->D;
    CK(c, state_rows(c->dt, state_tokens, M, c->g.state_dim, c->state_in, c->Ks, c->stream));
    c->launches = 0;
    GemmArgs g1;
    g1.A = c->state_in; g1.lda = c->Ks; g1.W = c->w_s1; g1.ldw = c->Ks; g1.M = M; g1.N = D; g1.K = c->Ks;
    g1.epi.kind = EPI_STORE; g1.epi.act = ACT_SWISH; g1.epi.bias = c->b_s1; g1.epi.out = c->state_hid;
    g1.epi.ldo = D;
    RC(gemm(c, g1));
    GemmArgs g2;
    g2.A = c->state_hid; g2.lda = D; g2.W = c->w_s2; g2.ldw = D; g2.M = M; g2.N = D; g2.K = D;
    g2.epi.kind = EPI_STORE; g2.epi.out_f32 = 1; g2.epi.bias = c->b_s2; g2.epi.out = c->state_tok; g2.epi.ldo = D;
    RC(gemm(c, g2));
    state_tokens = c->state_tok;
  }
  std::vector<const void*> t(2 * c->L + 3, nullptr);
  for (int l = 0; l < c->L; ++l) {
    if (dit && l % 2 == 1) continue;
    if (prefix == 0) continue;
    if (!k[l] || !v[l]) return set_err(c, GR00T_EINVAL, "layer %d K/V pointer is NULL", l);
    t[2 * l] = k[l];
    t[2 * l + 1] = v[l];
  }
  t[2 * c->L] = text_mask;
  t[2 * c->L + 1] = image_mask;
  t[2 * c->L + 2] = state_tokens;
  CK(c, cudaMemcpyAsync(c->table, t.data(), t.size() * sizeof(void*), cudaMemcpyHostToDevice, c->stream));
  if (!dit) CK(c, rope_table(prefix, c->H, c->Dh, c->g.rope_theta, c->rope_tab, c->stream));
  // masks / state are read through host_table at capture (slot presence, state pointer)
  const bool layout_change = c->bB != batch || c->bP != prefix || t != c->host_table ||
                             (c->host_table[2 * c->L] == nullptr) != (text_mask == nullptr) ||
                             (c->host_table[2 * c->L + 1] == nullptr) != (image_mask == nullptr) ||
                             c->host_table[2 * c->L + 2] != state_tokens;
  if (layout_change && c->gexec) {
    cudaGraphExecDestroy(c->gexec);
    c->gexec = nullptr;
  }
  c->host_table = t;
  c->bB = batch;
  c->bP = prefix;
  c->bound = true;
  if (!c->pool.empty()) {   // a plain bind replaces a bound pool
    c->pool.clear();
    c->pool_cap = 0;
    if (c->gexec) {
      cudaGraphExecDestroy(c->gexec);
      c->gexec = nullptr;
    }
  }
  return GR00T_OK;
}

extern "C" int gr00t_bind_kv_pool(gr00t_ctx* c, int batch, int prefix, int capacity, void* const* pools) {
  if (!c) return GR00T_EINVAL;
  if (c->g.family != GR00T_FAMILY_EXPERT)
    return set_err(c, GR00T_EINVAL, "the paged K/V pool is an expert-family binding (one KV head)");
  if (!pools) return set_err(c, GR00T_EINVAL, "pools is NULL");
  if (capacity < prefix + c->H || capacity % 128)
    return set_err(c, GR00T_EINVAL, "capacity %d must be a multiple of 128 holding prefix + horizon = %d", capacity,
                   prefix + c->H);
  for (int l = 0; l < c->L; ++l)
    if (!pools[l]) return set_err(c, GR00T_EINVAL, "layer %d pool is NULL", l);
  // plane-major: every sample's K slot, then every sample's V slot
  std::vector<const void*> k(c->L), v(c->L);
  for (int l = 0; l < c->L; ++l) {
    k[l] = pools[l];
    v[l] = (const char*)pools[l] + (size_t)batch * capacity * c->Dh * c->esz;
  }
  RC(gr00t_bind_prefix_kv(c, batch, prefix, k.data(), v.data(), nullptr, nullptr, nullptr));
  c->pool.assign(pools, pools + c->L);
  c->pool_cap = capacity;
  if (c->gexec) {   // the attention's tensor maps embed the pool layout
    cudaGraphExecDestroy(c->gexec);
    c->gexec = nullptr;
  }
  return GR00T_OK;
}

extern "C" int gr00t_bind_context(gr00t_ctx* c, int batch, int prefix, const void* features,
                                  const uint8_t* text_mask, const uint8_t* image_mask,
                                  const float* state_tokens) {
  if (!c) return GR00T_EINVAL;
  if (c->g.family != GR00T_FAMILY_DIT || c->g.context_dim <= 0)
    return set_err(c, GR00T_ESTATE, "gr00t_bind_context needs a DiT geometry with context_dim > 0");
  if (!features) return set_err(c, GR00T_EINVAL, "features is NULL");
  if (batch < 1 || batch > c->g.max_batch)
    return set_err(c, GR00T_EINVAL, "batch %d outside [1, %d]", batch, c->g.max_batch);
  if (prefix < 1 || prefix > c->g.max_prefix)
    return set_err(c, GR00T_EINVAL, "prefix %d outside [1, %d]", prefix, c->g.max_prefix);
  const int Dc = c->g.context_dim, kd = c->Hkv * c->Dh, M = batch * prefix;
  // a library copy of the features: one fixed operand address for the cached tensor maps
  CK(c, cudaMemcpyAsync(c->ctx_feat, features, (size_t)M * Dc * c->esz, cudaMemcpyDeviceToDevice, c->stream));
  c->launches = 0;
  for (int l = 0; l < c->L; l += 2) {
    for (int which = 0; which < 2; ++which) {
      GemmArgs a;
      a.A = c->ctx_feat; a.lda = Dc; a.W = which ? c->w_cv[l] : c->w_ck[l]; a.ldw = Dc;
      a.M = M; a.N = kd; a.K = Dc;
      a.epi.kind = EPI_STORE; a.epi.out = which ? c->ctx_v[l] : c->ctx_k[l]; a.epi.ldo = kd;
      RC(gemm(c, a));
    }
  }
  return gr00t_bind_prefix_kv(c, batch, prefix, (const void* const*)c->ctx_k.data(),
                              (const void* const*)c->ctx_v.data(), text_mask, image_mask, state_tokens);
}

extern "C" int gr00t_set_schedule(gr00t_ctx* c, int steps, int batch) {
  if (!c) return GR00T_EINVAL;
  if (steps < 1 || steps > c->g.max_steps)
    return set_err(c, GR00T_EINVAL, "steps %d outside [1, %d]", steps, c->g.max_steps);
  if (batch < 1 || batch > c->g.max_batch)
    return set_err(c, GR00T_EINVAL, "batch %d outside [1, %d]", batch, c->g.max_batch);
  if (c->scheduled && c->sT == steps && c->sB == batch) return GR00T_OK;
  const int TB = steps * batch, E = c->E, D = c->D;
  c->launches = 0;
  CK(c, time_embed(c->dt, steps, batch, E, c->g.direction, c->temb, c->dts, c->stream));
  const void* cin = c->temb;
  if (c->g.time_mlp) {
    GemmArgs a;
    a.A = c->temb; a.lda = E; a.W = c->w_tin; a.ldw = E; a.M = TB; a.N = E; a.K = E;
    a.epi.kind = EPI_STORE; a.epi.act = ACT_SWISH; a.epi.bias = c->b_tin; a.epi.out = c->t1; a.epi.ldo = E;
    RC(gemm(c, a));
    GemmArgs b2 = a;
    b2.A = c->t1; b2.W = c->w_tout; b2.epi.bias = c->b_tout; b2.epi.out = c->cvec;
    RC(gemm(c, b2));
    cin = c->cvec;
  }
  GemmArgs m;
  m.A = cin; m.lda = E; m.W = c->w_cond; m.ldw = E; m.M = TB; m.N = c->S * c->R; m.K = E;
  m.epi.kind = EPI_STORE; m.epi.bias = c->b_cond; m.epi.out = c->mod; m.epi.ldo = c->S * c->R;
  RC(gemm(c, m));
  if (c->g.family == GR00T_FAMILY_DIT) {
    // action_time_bias [steps][D] = W2[:, D:] temb(tau_k) + b2, from the b = 0 rows
    GemmArgs t;
    t.A = c->temb; t.lda = batch * E; t.W = (const char*)c->w_enc2 + (size_t)D * c->esz; t.ldw = D + E;
    t.M = steps; t.N = D; t.K = E;
    t.epi.kind = EPI_STORE; t.epi.out_f32 = 1; t.epi.bias = c->b_enc2; t.epi.out = c->atb; t.epi.ldo = D;
    RC(gemm(c, t));
  }
  if (c->gexec && (c->gT != steps || c->gB != batch)) {
    cudaGraphExecDestroy(c->gexec);
    c->gexec = nullptr;
  }
  c->sT = steps;
  c->sB = batch;
  c->scheduled = true;
  return GR00T_OK;
}

extern "C" int gr00t_debug_cond_step(gr00t_ctx* c, int k, void* hoisted, void* per_step) {
  if (!c) return GR00T_EINVAL;
  if (!hoisted || !per_step) return set_err(c, GR00T_EINVAL, "hoisted/per_step is NULL");
  if (!c->scheduled) return set_err(c, GR00T_ESTATE, "no schedule (call gr00t_set_schedule)");
  if (k < 0 || k >= c->sT) return set_err(c, GR00T_EINVAL, "step %d outside [0, %d)", k, c->sT);
  const int B = c->sB, E = c->E, SR = c->S * c->R;
  const size_t rows_bytes = (size_t)B * SR * c->esz;
  CK(c, cudaMemcpyAsync(hoisted, (const char*)c->mod + (size_t)k * rows_bytes, rows_bytes,
                        cudaMemcpyDeviceToDevice, c->stream));
  // the same chain as gr00t_set_schedule on the B time-embedding rows of step k alone
  // (the hoist's intermediates t1 / cvec serve as scratch: no kernel of a step reads them)
  const void* temb_k = (const char*)c->temb + (size_t)k * B * E * c->esz;
  const void* cin = temb_k;
  if (c->g.time_mlp) {
    GemmArgs a;
    a.A = temb_k; a.lda = E; a.W = c->w_tin; a.ldw = E; a.M = B; a.N = E; a.K = E;
    a.epi.kind = EPI_STORE; a.epi.act = ACT_SWISH; a.epi.bias = c->b_tin; a.epi.out = c->t1; a.epi.ldo = E;
    RC(gemm(c, a));
    GemmArgs b2 = a;
    b2.A = c->t1; b2.W = c->w_tout; b2.epi.bias = c->b_tout; b2.epi.out = c->cvec;
    RC(gemm(c, b2));
    cin = c->cvec;
  }
  GemmArgs m;
  m.A = cin; m.lda = E; m.W = c->w_cond; m.ldw = E; m.M = B; m.N = SR; m.K = E;
  m.epi.kind = EPI_STORE; m.epi.bias = c->b_cond; m.epi.out = per_step; m.epi.ldo = SR;
  RC(gemm(c, m));
  return GR00T_OK;
}

extern "C" int gr00t_denoise(gr00t_ctx* c, const float* x_noise, float* actions) {
  if (!c) return GR00T_EINVAL;
  if (!x_noise || !actions) return set_err(c, GR00T_EINVAL, "x_noise/actions is NULL");
  RC(check_ready(c));
  const size_t bytes = (size_t)c->bB * c->H * c->A * sizeof(float);
  CK(c, cudaMemcpyAsync(c->x, x_noise, bytes, cudaMemcpyDeviceToDevice, c->stream));
  RC(run_loop(c));
  CK(c, cudaMemcpyAsync(actions, c->x, bytes, cudaMemcpyDeviceToDevice, c->stream));
  return GR00T_OK;
}

extern "C" int gr00t_denoise_host(gr00t_ctx* c, const float* x_noise_host, float* actions_host) {
  if (!c) return GR00T_EINVAL;
  if (!x_noise_host || !actions_host) return set_err(c, GR00T_EINVAL, "x_noise/actions is NULL");
  RC(check_ready(c));
  const size_t bytes = (size_t)c->bB * c->H * c->A * sizeof(float);
  CK(c, cudaMemcpyAsync(c->x, x_noise_host, bytes, cudaMemcpyHostToDevice, c->stream));
  RC(run_loop(c));
  CK(c, cudaMemcpyAsync(actions_host, c->x, bytes, cudaMemcpyDeviceToHost, c->stream));
  return sync_and_check(c);
}

extern "C" int gr00t_denoise_step(gr00t_ctx* c, int k, const float* x_in, float* v_out) {
  if (!c) return GR00T_EINVAL;
  if (!x_in || !v_out) return set_err(c, GR00T_EINVAL, "x_in/v_out is NULL");
  RC(check_ready(c));
  if (k < 0 || k >= c->sT) return set_err(c, GR00T_EINVAL, "step %d outside [0, %d)", k, c->sT);
  const size_t bytes = (size_t)c->bB * c->H * c->A * sizeof(float);
  CK(c, cudaMemcpyAsync(c->xtmp, x_in, bytes, cudaMemcpyDeviceToDevice, c->stream));
  RC(enqueue_step(c, k, c->xtmp, v_out, 0));
  return GR00T_OK;
}

extern "C" int gr00t_destroy(gr00t_ctx* c) {
  if (!c) return GR00T_EINVAL;
  free_ctx(c);
  return GR00T_OK;
}

extern "C" const char* gr00t_last_error(const gr00t_ctx* c) {
  return c ? c->err.c_str() : g_create_err.c_str();
}

extern "C" int gr00t_set_option(gr00t_ctx* c, int option, int64_t value) {
  if (!c) return GR00T_EINVAL;
  switch (option) {
    case GR00T_OPT_USE_GRAPH:
      c->opt_graph = value ? 1 : 0;
      return GR00T_OK;
    case GR00T_OPT_GEMM_PATH:
      if (value != 0 && value != 1) return set_err(c, GR00T_EINVAL, "GEMM path must be 0 or 1");
      c->opt_gemm = (int)value;
      break;
    case GR00T_OPT_ATTN_PATH:
      if (value < 0 || value > 3) return set_err(c, GR00T_EINVAL, "attention path must be 0, 1, 2 or 3");
      c->opt_attn = (int)value;
      break;
    case GR00T_OPT_WAIT_LIMIT:
      if (value < 0) return set_err(c, GR00T_EINVAL, "wait limit must be >= 0");
      c->wait_limit = value;
      break;
    case GR00T_OPT_PERSISTENT_GEMM:
      c->opt_persistent = value ? 1 : 0;
      break;
    case GR00T_OPT_GEMM_MULTICAST:
      c->opt_mcast = value ? 1 : 0;
      break;
    case GR00T_OPT_ATTN_MULTICAST:
      if (value < 0 || value > 2) return set_err(c, GR00T_EINVAL, "attention multicast: 0, 1 or 2 (automatic)");
      c->opt_attn_mcast = (int)value;
      break;
    case GR00T_OPT_GEMM_TSTORE:
      c->opt_tstore = value ? 1 : 0;
      break;
    case GR00T_OPT_L2_PREFETCH:
      c->opt_l2_ahead = value ? 1 : 0;
      break;
    case GR00T_OPT_ATTN_SPLIT_CAP:
      if (value < 0 || value > 32) return set_err(c, GR00T_EINVAL, "attention split cap: 0 (automatic) .. 32");
      c->opt_attn_splits = (int)value;
      break;
    case GR00T_OPT_NOALLOC_LIMIT:
      if (value < 0 || value > G3_NOALLOC_SCRATCH_FLOATS)
        return set_err(c, GR00T_EINVAL, "no-alloc limit: 0 .. %lld floats", (long long)G3_NOALLOC_SCRATCH_FLOATS);
      c->noalloc_limit = value;
      break;
    case GR00T_OPT_SPLIT_CAP:
    case GR00T_OPT_RESID_SPLIT_CAP:
      if (value < 1 || value > 16 || (value & (value - 1))) return set_err(c, GR00T_EINVAL, "split cap: 1, 2, 4, 8 or 16");
      (option == GR00T_OPT_SPLIT_CAP ? c->split_cap : c->resid_split_cap) = (int)value;
      break;
    case GR00T_OPT_TIME_KERNELS: {
      if (value != 0 && value != 1) return set_err(c, GR00T_EINVAL, "launch stamps: 0 or 1");
      c->stamp_on = (int)value;
      // one slot per launch of a whole loop at max_steps, plus the tail stamp
      const int need = value ? c->g.max_steps * (8 * c->L + 16) + 1 : 0;
      if (need > c->stamp_cap) {
        if (c->stamps) CK(c, cudaFree(c->stamps));
        c->stamps = nullptr;
        c->stamp_cap = 0;
        CK(c, cudaMalloc((void**)&c->stamps, (size_t)need * sizeof(unsigned long long)));
        c->stamp_cap = need;
      }
      break;
    }
    case GR00T_OPT_TEST_STALL:
      if (value < 0 || value > (1 << 24)) return set_err(c, GR00T_EINVAL, "test stall: 0 .. 2^24 polls");
      c->opt_stall = (int)value;
      break;
    default:
      return set_err(c, GR00T_EINVAL, "unknown option %d", option);
  }
  if (c->gexec) {  // kernels baked into the graph change
    cudaGraphExecDestroy(c->gexec);
    c->gexec = nullptr;
  }
  return GR00T_OK;
}

extern "C" int gr00t_get_info(gr00t_ctx* c, int what, int64_t* value) {
  if (!c || !value) return GR00T_EINVAL;
  switch (what) {
    case GR00T_INFO_KERNELS_PER_STEP:
      *value = c->launches;
      return GR00T_OK;
    case GR00T_INFO_WEIGHT_BYTES: {
      long long b = 0;
      const int up_rows = (c->g.mlp_kind == GR00T_MLP_GEGLU ? 2 : 1) * c->F;
      for (int l = 0; l < c->L; ++l) {
        const long long rows = (long long)c->nqkv[l] + c->D + up_rows + c->D;   // output rows (FP8: one scale each)
        b += ((long long)c->nqkv[l] * c->D + (long long)c->D * c->qd + (long long)up_rows * c->D +
              (long long)c->D * c->F) * (c->fp8w ? 1 : (long long)c->esz) + (c->fp8w ? rows * 4 : 0);
      }
      b += (long long)c->A * c->D * c->esz;
      if (c->g.family == GR00T_FAMILY_EXPERT)
        b += (long long)c->D * c->A * c->esz;
      else
        b += ((long long)c->D * c->A + (long long)c->D * c->D * 2) * c->esz;
      *value = b;
      return GR00T_OK;
    }
    case GR00T_INFO_DEVICE_BYTES:
      *value = (int64_t)c->arena_bytes;
      return GR00T_OK;
    case GR00T_INFO_MOD_ROW:
      *value = (int64_t)c->S * c->R;
      return GR00T_OK;
    case GR00T_INFO_ERROR_FLAG: {
      int f = 0;
      CK(c, cudaMemcpyAsync(&f, c->err_flag, sizeof f, cudaMemcpyDeviceToHost, c->stream));
      CK(c, cudaStreamSynchronize(c->stream));
      *value = f;
      return GR00T_OK;
    }
    default:
      return set_err(c, GR00T_EINVAL, "unknown info %d", what);
  }
}

extern "C" int gr00t_kernel_times(gr00t_ctx* c, float* us, int* kclass, int max, int* count) {
  if (!c || !count || (max > 0 && !us)) return GR00T_EINVAL;
  *count = 0;
  CK(c, cudaStreamSynchronize(c->stream));
  const int n = c->stamp_used;
  if (!c->stamp_on || n < 2) return GR00T_OK;
  std::vector<unsigned long long> t(n);
  CK(c, cudaMemcpy(t.data(), c->stamps, (size_t)n * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
  int m = 0;
  for (int i = 0; i + 1 < n && m < max; ++i, ++m) {
    us[m] = (float)((double)(long long)(t[i + 1] - t[i]) * 1e-3);
    if (kclass) kclass[m] = c->stamp_cls[i];
  }
  *count = m;
  return GR00T_OK;
}

extern "C" int gr00t_sync(gr00t_ctx* c) {
  if (!c) return GR00T_EINVAL;
  return sync_and_check(c);
}

extern "C" int gr00t_debug_dump(gr00t_ctx* c, int k, const float* x_in, int layer, float* h_out) {
  if (!c) return GR00T_EINVAL;
  if (!x_in || !h_out) return set_err(c, GR00T_EINVAL, "x_in/h_out is NULL");
  RC(check_ready(c));
  if (k < 0 || k >= c->sT) return set_err(c, GR00T_EINVAL, "step %d outside [0, %d)", k, c->sT);
  if (layer < -1 || layer >= c->L) return set_err(c, GR00T_EINVAL, "layer %d outside [-1, %d)", layer, c->L);
  const size_t bytes = (size_t)c->bB * c->H * c->A * sizeof(float);
  CK(c, cudaMemcpyAsync(c->xtmp, x_in, bytes, cudaMemcpyDeviceToDevice, c->stream));
  c->dump_out = h_out;
  c->dump_layer = layer;
  const int rc = enqueue_step(c, k, c->xtmp, nullptr, 0);
  c->dump_out = nullptr;
  c->dump_layer = -2;
  return rc;
}

// ---- allocation-free step ------------------------------------------------------
//
// Scratch of gr00t_denoise_step_noalloc: a fixed array in the library's device
// image, 12 MiB of fp32 on every GPU that loads the library, held until the
// process exits.  Host code cannot use the symbol itself as a device address;
// its device address is looked up once per device with that device current.
static __device__ __align__(256) float g_noalloc_scratch[G3_NOALLOC_SCRATCH_FLOATS];

namespace {

std::mutex g_noalloc_mu;
constexpr int kMaxDevices = 256;
float* g_noalloc_addr[kMaxDevices] = {};

// Device address of the fixed scratch array on device ``dev`` (current).
cudaError_t noalloc_scratch(int dev, float** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_addr[dev];
  return cudaSuccess;
}

// Scratch (fp32 elements) one GEMM of the step uses when the scratch holds ``cap``
// elements; mirrors gemm() / gemm_resid().
long long gemm_scratch(gr00t_ctx* c, int M, int N, int K, bool resid, long long cap, bool e4m3 = false) {
  if (!tc_ok(c, M, N, K, e4m3)) return 0;
  if (resid) {
    const TcPlan p = plan_of(c, M, N, K, e4m3, true);
    if (p.S > 1 && (long long)p.S * M * N <= cap) return (long long)p.S * M * N;
  }
  return tc_workspace_floats(plan_of(c, M, N, K, e4m3, false), M, N);
}

// Largest scratch any kernel of one denoise step needs at the bound (batch, prefix).
long long step_scratch(gr00t_ctx* c, long long cap) {
  const int B = c->bB, D = c->D, M = B * c->tok, MA = B * c->H;
  long long need = 0;
  auto take = [&](long long v) { need = v > need ? v : need; };
  const int up_rows = (c->g.mlp_kind == GR00T_MLP_GEGLU ? 2 : 1) * c->F;
  if (c->g.family == GR00T_FAMILY_DIT) {
    take(gemm_scratch(c, MA, D, D, false, cap));
    for (int l = 0; l < c->L; ++l) {
      take(gemm_scratch(c, M, c->nqkv[l], D, false, cap, c->fp8w));
      take(gemm_scratch(c, M, D, c->qd, true, cap, c->fp8w));
      take(gemm_scratch(c, M, up_rows, D, false, cap, c->fp8w));
      take(gemm_scratch(c, M, D, c->F, true, cap, c->fp8w));
    }
    return need;
  }
  take(gemm_scratch(c, M, c->nqkv[0], D, false, cap, c->fp8w));
  take(gemm_scratch(c, M, D, c->qd, true, cap, c->fp8w));
  take(gemm_scratch(c, M, up_rows, D, false, cap, c->fp8w));
  take(gemm_scratch(c, M, D, c->F, true, cap, c->fp8w));
  if (c->dt == DT_BF16 && (c->opt_attn == 0 || c->opt_attn == 3) && attn_t5_supported(c->Dh, c->Hq)) {
    AttnT5Args a5;
    a5.B = B; a5.H = c->H; a5.Hq = c->Hq; a5.Dh = c->Dh; a5.P = c->bP;
    take(attn_t5_workspace_floats(a5, attn_t5_splits(a5, c->sm_count, c->opt_attn_splits)));
  } else if (c->dt == DT_BF16 && (c->opt_attn == 0 || c->opt_attn == 2) && attn_fold_supported(c->Dh)) {
    AttnFoldArgs af;
    af.B = B; af.H = c->H; af.Hq = c->Hq; af.Dh = c->Dh; af.P = c->bP;
    take(attn_fold_workspace_floats(af, attn_fold_splits(af, c->sm_count)));
  }
  return need;
}

}  // namespace

extern "C" int gr00t_denoise_step_noalloc(gr00t_ctx* c, int k, const float* x_in, float* v_out) {
  if (!c) return GR00T_EINVAL;
  if (!x_in || !v_out) return set_err(c, GR00T_EINVAL, "x_in/v_out is NULL");
  RC(check_ready(c));
  if (k < 0 || k >= c->sT) return set_err(c, GR00T_EINVAL, "step %d outside [0, %d)", k, c->sT);
  int dev = -1;
  CK(c, cudaGetDevice(&dev));
  if (dev != c->device)
    return set_err(c, GR00T_EINVAL, "device %d is current; the context lives on device %d", dev, c->device);
  // the step's launch sequence is the regular entry point's (planned against the
  // context's own scratch); it runs here only if its scratch fits the fixed array
  const long long cap = c->noalloc_limit >= 0 ? c->noalloc_limit : G3_NOALLOC_SCRATCH_FLOATS;
  const long long need = step_scratch(c, c->gemm_ws_floats);
  if (need > cap)
    return set_err(c, GR00T_EINVAL,
                   "this step needs %lld floats of scratch at batch %d, prefix %d; the no-alloc bound is %lld of "
                   "the fixed array's %lld (use gr00t_denoise_step)", need, c->bB, c->bP, cap,
                   (long long)G3_NOALLOC_SCRATCH_FLOATS);
  // the array's device address was looked up by gr00t_create on this device
  float* const scratch = c->noalloc_addr;
  if (!scratch) return set_err(c, GR00T_ESTATE, "the fixed scratch array was not set up on this device");
  const size_t bytes = (size_t)c->bB * c->H * c->A * sizeof(float);
  CK(c, cudaMemcpyAsync(c->xtmp, x_in, bytes, cudaMemcpyDeviceToDevice, c->stream));
  // same launch sequence as gr00t_denoise_step, scratch taken from the fixed array and
  // tensor-map descriptors from fixed slots of the context instead of its cache
  float* const own = c->gemm_ws;
  const long long own_floats = c->gemm_ws_floats;
  c->gemm_ws = scratch;
  c->gemm_ws_floats = cap;
  c->no_host_alloc = true;
  const int rc = enqueue_step(c, k, c->xtmp, v_out, 0);
  c->no_host_alloc = false;
  c->gemm_ws = own;
  c->gemm_ws_floats = own_floats;
  return rc;
}
