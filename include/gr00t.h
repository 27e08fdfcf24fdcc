/*
 * gr00t.h -- C ABI of the GB300 (sm_103a) flow-matching action-expert denoise loop.
 *
 * The library runs the hot path of a flow-matching Vision-Language-Action
 * policy: the action expert's denoise loop.  The prefix (vision-language)
 * K/V is computed elsewhere and bound once; the library hoists the time
 * conditioning, then integrates an action chunk from noise with T Euler
 * steps, each step one evaluation of the expert stack.
 *
 * Two model families share the interface:
 *   GR00T_FAMILY_EXPERT -- pi0.5-style action expert ("pi0.5 Design",
 *       TensorRT Edge-LLM developer guide): AdaRMS norms, a single shared KV
 *       head, attention over prefix K/V ++ the action tokens' own K/V.
 *   GR00T_FAMILY_DIT    -- GR00T-N1.7-style DiT head ("GR00T N1.7",
 *       TensorRT Edge-LLM developer guide): AdaLayerNorm, blocks alternating
 *       cross-attention into the VL context and self-attention over the
 *       state + action tokens.
 *
 * Inputs of a request are bound once before the loop: per-layer prefix K/V
 * (gr00t_bind_prefix_kv), the pages' paged K/V pool (gr00t_bind_kv_pool,
 * EXPERT), or VL features whose cross K/V the library projects itself
 * (gr00t_bind_context, DIT).  The per-layer projections may be streamed as
 * E4M3 codes with row scales (GR00T_WFMT_FP8).
 *
 * Conventions shared by every call:
 *   - Every function returns GR00T_OK (0) or a negative GR00T_E* status.
 *     gr00t_last_error() gives a one-line text for the context's last error.
 *   - Work is enqueued on the CUDA stream given to gr00t_create and is
 *     asynchronous unless stated otherwise.  A context is not thread-safe
 *     (one stream, one caller), as the pages' runtimes are not.
 *   - Matrices are row-major.  Weights use the nn.Linear layout [out, in].
 *   - "bf16" tensors are raw IEEE bfloat16 bit patterns (uint16_t).
 *   - Nothing here allocates on a call except gr00t_create (and graph
 *     instantiation on the first denoise of a new (steps, batch, prefix) or
 *     binding layout).
 *   - No call ever falls back to the CPU.  Without a usable sm_103a device
 *     gr00t_create returns GR00T_ECUDA.
 */
#ifndef GR00T_H_
#define GR00T_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GR00T_ABI_VERSION 3

/* ---- status codes ------------------------------------------------------ */
#define GR00T_OK 0
#define GR00T_EINVAL (-1)      /* bad argument or geometry; nothing was done   */
#define GR00T_ENOMEM (-2)      /* a device allocation failed                   */
#define GR00T_ECUDA (-3)       /* a CUDA runtime/driver call failed            */
#define GR00T_ESTATE (-4)      /* call out of order (e.g. denoise before bind) */
#define GR00T_EUNSUPPORTED (-5)/* valid request the library does not implement */
#define GR00T_ETIMEOUT (-6)    /* a bounded device wait gave up                */

/* ---- enumerations ------------------------------------------------------ */
#define GR00T_FAMILY_EXPERT 0
#define GR00T_FAMILY_DIT 1
#define GR00T_DTYPE_FP32 0
#define GR00T_DTYPE_BF16 1
#define GR00T_MLP_GELU 0       /* u = gelu_tanh(n W_up^T)                        */
#define GR00T_MLP_GEGLU 1      /* u = gelu_tanh(n W_gate^T) * (n W_up^T)         */
#define GR00T_MEM_HOST 0
#define GR00T_MEM_DEVICE 1

/*
 * Geometry of one expert.  Validated by gr00t_create before anything is
 * allocated ("GR00T N1.7", Checkpoint: a wrong architecture is rejected
 * before anything is built; "pi0.5 Design", Runtime boundary: unsupported
 * configurations are rejected when loading).
 *
 * EXPERT family: kv_heads must be 1 (the head fold is exact only with a
 * single KV head and an all-ones mask, "pi0.5 Design", Attention and the K/V
 * pool); the modulation table has 2*layers+1 sites of width 3*hidden, packed
 * (scale, shift, gate), site 2i = layer i input norm, 2i+1 = its post-
 * attention norm, 2*layers = final norm ("pi0.5 Design", Component contract).
 * DIT family: kv_heads == q_heads; layers even; blocks alternate cross-
 * attention (even index) and self-attention (odd index) ("GR00T N1.7",
 * action); layers+1 sites of width 2*hidden, (scale, shift) for blocks and
 * (shift, scale) for the final norm ("GR00T N1.7", Build-time constants).
 */
typedef struct gr00t_geometry {
  int32_t abi_version;   /* GR00T_ABI_VERSION                                */
  int32_t family;        /* GR00T_FAMILY_*                                    */
  int32_t dtype;         /* GR00T_DTYPE_*: weight, K/V and activation type    */
  int32_t layers;        /* transformer layers / DiT blocks                   */
  int32_t hidden;        /* D, residual width (multiple of 64)               */
  int32_t q_heads;       /* query heads                                      */
  int32_t kv_heads;      /* K/V heads (EXPERT: 1; DIT: q_heads)              */
  int32_t head_dim;      /* Dh (EXPERT: 64 or 256; DIT: 48)                   */
  int32_t mlp_dim;       /* F, MLP width (multiple of 64)                     */
  int32_t mlp_kind;      /* GR00T_MLP_*                                       */
  int32_t horizon;       /* H, action tokens per chunk                        */
  int32_t action_dim;    /* A, command dimensions per action                  */
  int32_t state_tokens;  /* DIT: state tokens ahead of the actions (0 or 1)   */
  int32_t time_dim;      /* E, sinusoidal time-embedding width (even, >= 4)   */
  int32_t time_mlp;      /* 1: c = swish(W_out swish(W_in temb + b) + b)      */
  int32_t direction;     /* -1: integrate tau 1 -> 0; +1: tau 0 -> 1          */
  int32_t max_batch;     /* largest batch a schedule/bind may use             */
  int32_t max_prefix;    /* largest prefix / VL-context length                */
  int32_t max_steps;     /* largest denoise step count                        */
  float rope_theta;      /* RoPE base (EXPERT family)                         */
  float norm_eps;        /* epsilon of RMSNorm / LayerNorm                    */
  int32_t weight_format; /* GR00T_WFMT_*: storage of the per-layer projections */
  int32_t context_dim;   /* DIT: width of the VL features gr00t_bind_context projects
                            into the cross K/V (multiple of 64); 0: K/V bound directly */
  int32_t state_dim;     /* DIT: width of the raw robot state the binds embed with the
                            state encoder (<= 4096); 0: state tokens bound already embedded */
} gr00t_geometry;

/* Storage of the per-layer projections (qkv_w, o_w, up_w, down_w).  FP8: each
 * matrix is uint8 E4M3 codes [out, in] (sign bit 7, exponent bits 6..3 with
 * bias 7, mantissa bits 2..0, no infinities) with one fp32 scale per output row
 * (qkv_s .. down_s): the real weight is e4m3(code) * scale.  Streaming half the
 * bytes is the lever of the bandwidth-bound small-batch loop ("pi0.5 Design",
 * precision notes; vla.cpp Table V).  Requires dtype BF16: activations stay
 * bf16 and the codes are widened to bf16 on chip, exactly. */
#define GR00T_WFMT_NATIVE 0   /* the geometry's dtype                           */
#define GR00T_WFMT_FP8 1      /* E4M3 codes + per-row fp32 scales (dtype BF16)  */

/*
 * Weights, all in the geometry's dtype (fp32 or bf16), nn.Linear [out, in].
 * ``location`` says whether every pointer is host or device memory.  The
 * library COPIES them into its own re-laid-out device buffers during
 * gr00t_create; the caller may free them as soon as it returns.
 * Pointers a family does not use must be NULL.
 *
 *   time_mlp_{in,out}_w [E, E], _b [E]       if time_mlp
 *   cond_w [S, R, E], cond_b [S, R]          the S adaptive-norm Denses
 *                                            ("pi0.5 Design": 37 [3072,1024])
 *   EXPERT: action_in_w [D, A], action_in_b [D]
 *   DIT:    enc_w1 [D, A], enc_b1 [D], enc_w2 [D, D+E] acting on
 *           concat(W1 x + b1, temb(tau)), enc_b2 [D], enc_w3 [D, D], enc_b3 [D]
 *   action_out_w [A, D], action_out_b [A]
 *   DIT with state_dim > 0: the state encoder state_w1 [D, state_dim],
 *           state_b1 [D], state_w2 [D, D], state_b2 [D]:
 *           s_tok = state_w2 swish(state_w1 s + state_b1) + state_b2
 *   per layer l (arrays of ``layers`` pointers; with GR00T_WFMT_FP8 these four
 *   are uint8 E4M3 codes and qkv_s .. down_s their fp32 row scales):
 *     qkv_w[l]  EXPERT: [Hq*Dh + 2*Dh, D] rows (q heads, k, v)
 *               DIT even l: [Hq*Dh, D] (q only); odd l: [3*Hq*Dh, D] (q, k, v)
 *     o_w[l]    [D, Hq*Dh]
 *     up_w[l]   GEGLU: [2F, D], rows [0,F) gate, [F,2F) up;  GELU: [F, D]
 *     down_w[l] [D, F]
 */
typedef struct gr00t_weights {
  int32_t location; /* GR00T_MEM_HOST or GR00T_MEM_DEVICE */
  const void* time_mlp_in_w;
  const void* time_mlp_in_b;
  const void* time_mlp_out_w;
  const void* time_mlp_out_b;
  const void* cond_w;
  const void* cond_b;
  const void* action_in_w;
  const void* action_in_b;
  const void* enc_w1;
  const void* enc_b1;
  const void* enc_w2;
  const void* enc_b2;
  const void* enc_w3;
  const void* enc_b3;
  const void* action_out_w;
  const void* action_out_b;
  const void* const* qkv_w;
  const void* const* o_w;
  const void* const* up_w;
  const void* const* down_w;
  /* GR00T_WFMT_FP8 only (else NULL): per layer, fp32 scale of each output row
   * of qkv_w / o_w / up_w / down_w, in the same location as the codes */
  const void* const* qkv_s;
  const void* const* o_s;
  const void* const* up_s;
  const void* const* down_s;
  /* DIT with context_dim > 0 (else NULL): per block, the cross-attention K and V
   * projections [kv_heads*head_dim, context_dim] of the even blocks (odd entries
   * NULL), in the geometry's dtype, no bias */
  const void* const* cross_k_w;
  const void* const* cross_v_w;
  /* DIT with state_dim > 0 (else NULL): the state encoder, in the geometry's dtype */
  const void* state_w1;
  const void* state_b1;
  const void* state_w2;
  const void* state_b2;
} gr00t_weights;

typedef struct gr00t_ctx gr00t_ctx;

/*
 * Check a geometry without touching the GPU.  Returns GR00T_OK or
 * GR00T_EINVAL / GR00T_EUNSUPPORTED; ``msg`` (may be NULL) receives a
 * NUL-terminated reason of at most ``msg_len`` bytes.
 */
int gr00t_validate_geometry(const gr00t_geometry* g, char* msg, size_t msg_len);

/*
 * Create a context on the current CUDA device: validate the geometry, copy
 * and re-lay-out the weights, allocate every buffer the loop needs for
 * (max_batch, max_prefix, max_steps).  ``stream`` is a cudaStream_t (may be
 * NULL for the legacy default stream); every later call enqueues on it.
 * The device must be sm_103 (GB300).  On failure *out is NULL and nothing
 * stays allocated.  Synchronous.
 */
int gr00t_create(const gr00t_geometry* g, const gr00t_weights* w, void* stream, gr00t_ctx** out);

/*
 * Bind the per-request prefix / VL-context K/V for the whole denoise loop
 * ("GR00T N1.7", Who runs what: the backbone's K/V is produced once per
 * request and reused by every denoise step; "pi0.5 Design", sequence diagram).
 *
 * ``k``, ``v``: arrays of ``layers`` DEVICE pointers, each to a contiguous
 * [batch, prefix, kv_heads, head_dim] tensor in the geometry's dtype.  EXPERT:
 * every layer, keys already rotated by RoPE at positions 0..prefix-1.  DIT:
 * even layers only (odd entries ignored, may be NULL).  The memory is
 * BORROWED: the caller keeps it alive and unchanged until the next bind or
 * gr00t_destroy.  Rebinding new pointers re-captures the loop's CUDA graph on
 * the next gr00t_denoise (its TMA descriptors embed the K/V addresses).
 *
 * ``text_mask``/``image_mask``: DIT only, DEVICE uint8 [batch, prefix],
 * 1 = visible; block i reads the text mask when i % 4 == 0 and the image
 * mask otherwise ("GR00T N1.7", action).  NULL = all visible.  Must be NULL
 * for EXPERT (its head fold needs the all-ones mask).
 * ``state_tokens``: DIT only, DEVICE fp32 [batch, state_tokens, hidden], the
 * embedded robot state placed ahead of the action tokens; borrowed.  With
 * state_dim > 0 it is instead the RAW robot state [batch, state_tokens,
 * state_dim] (fp32), which this call embeds with the state encoder into
 * library-owned tokens on the tensor cores ("GR00T N1.7", action: the robot
 * state enters beside the noisy actions and its encoder is one of the
 * per-embodiment modules; it does not change across a request's denoise
 * steps, so it is embedded once, here); read on the stream, not borrowed.
 * 1 <= batch <= max_batch; 0 <= prefix <= max_prefix (EXPERT), 1 <= prefix
 * (DIT).  Enqueues a small copy on the stream.
 */
int gr00t_bind_prefix_kv(gr00t_ctx* ctx, int batch, int prefix, const void* const* k,
                         const void* const* v, const uint8_t* text_mask,
                         const uint8_t* image_mask, const float* state_tokens);

/*
 * DIT with context_dim > 0: project the per-request VL features into the cross
 * K/V of every even block and bind them ("GR00T N1.7", vl_backbone: the VL
 * engine ends with the DiT's cross-attention K/V projections, producing
 * cross_k / cross_v [B, S, 32, 48] for the even blocks; the step runs once per
 * request, before the denoise loop).  K_i = features W_k,i^T, V_i = features
 * W_v,i^T on the tensor cores into library-owned [batch, prefix, kv_heads,
 * head_dim] buffers, then bound as by gr00t_bind_prefix_kv.
 *
 * ``features``: DEVICE [batch, prefix, context_dim] in the geometry's dtype,
 * read asynchronously on the stream (keep it unchanged until the stream has
 * run this call's work).  Masks and state tokens as for gr00t_bind_prefix_kv.
 * GR00T_ESTATE for a geometry without context_dim; GR00T_EINVAL for a batch or
 * prefix out of range or a NULL features pointer.  Enqueues 2 GEMMs per cross
 * block and a small copy on the stream.
 */
int gr00t_bind_context(gr00t_ctx* ctx, int batch, int prefix, const void* features, const uint8_t* text_mask,
                       const uint8_t* image_mask, const float* state_tokens);

/*
 * EXPERT: bind the pages' paged K/V pool directly ("pi0.5 Design", Attention
 * and the K/V pool): per layer one DEVICE buffer [2][batch][capacity][1][head_dim]
 * in the geometry's dtype, plane-major -- every sample's K slot, then every
 * sample's V slot (the V plane begins past every slot's K) -- with pages of 128
 * rows under an identity page table, so a slot is a flat [capacity, head_dim]
 * region.  Slot rows [0, prefix) hold the prefix K/V (keys rotated by RoPE at
 * positions 0..prefix-1); every denoise step writes its action tokens' K/V into
 * rows [prefix, prefix + horizon), as the pages' attention plugin appends them
 * (after a denoise they hold the last step's).  ``capacity``: a multiple of 128
 * with capacity >= prefix + horizon (the pages round prefix + horizon up to 256).
 * The pools are BORROWED and WRITTEN: keep them alive until the next bind or
 * gr00t_destroy.  Needs the tensor-core attention (bf16, GR00T_OPT_ATTN_PATH 0
 * or 3); a later gr00t_bind_prefix_kv replaces the pool binding.
 */
int gr00t_bind_kv_pool(gr00t_ctx* ctx, int batch, int prefix, int capacity, void* const* pools);

/*
 * Hoist the time conditioning for a step count and batch ("pi0.5 Design",
 * cond component: the time embedder and the AdaRMS Denses leave the
 * per-step graph and are evaluated again only for a new step count or batch;
 * "GR00T N1.7", Build-time constants).  Builds the modulation table
 * [steps * batch, sites, row] (rows [step][request]), the Euler step sizes
 * on the uniform grid of vla.cpp Eq. (1), and for DIT the action_time_bias
 * [steps, hidden].  A call with the same (steps, batch) as the last one is a
 * no-op.  1 <= steps <= max_steps; 1 <= batch <= max_batch.
 */
int gr00t_set_schedule(gr00t_ctx* ctx, int steps, int batch);

/*
 * Run the whole denoise loop: T = steps Euler steps x_{k+1} = x_k +
 * (tau_{k+1} - tau_k) v(x_k, tau_k) (vla.cpp Eq. (1)), starting from the
 * caller's noise.  ``x_noise`` and ``actions`` are DEVICE fp32 [batch,
 * horizon, action_dim] (batch of the last bind, which must equal the last
 * schedule's); they may alias.  Returns the model-space chunk (before any
 * policy unnormalisation).  Requires a bind and a schedule (GR00T_ESTATE
 * otherwise).  The T steps replay as one CUDA graph captured on the first
 * call for a (steps, batch, prefix).  Asynchronous on the stream.
 */
int gr00t_denoise(gr00t_ctx* ctx, const float* x_noise, float* actions);

/*
 * gr00t_denoise with HOST buffers: copies ``x_noise`` in, runs the loop,
 * copies the chunk out and synchronises the stream before returning.
 * Page-locked host memory gives asynchronous copies; pageable works.
 */
int gr00t_denoise_host(gr00t_ctx* ctx, const float* x_noise_host, float* actions_host);

/*
 * One velocity evaluation at step k of the current schedule (teacher
 * forcing, for tests): ``v_out`` = v(x_in, tau_k); x_in is not modified.
 * DEVICE fp32 [batch, horizon, action_dim].  0 <= k < steps.  Runs eagerly.
 */
int gr00t_denoise_step(gr00t_ctx* ctx, int k, const float* x_in, float* v_out);

/*
 * gr00t_denoise_step with no allocation and no use of the context's scratch
 * workspace.  (No counterpart in the source pages: this is an interface
 * addition of this library.)
 *
 * Who it is for: callers that are not allowed to allocate device memory at
 * the point where they run a step -- e.g. a controller that fixed its device
 * memory budget at start-up and treats any later allocation as an error, or a
 * host program that lends this library a context and forbids it from taking
 * memory of its own.  This call never calls cudaMalloc, cudaFree or any other
 * allocating routine (device or host): the scratch that the tensor-core GEMMs
 * (split-K partials) and the attention (per-split partials) need comes from a
 * fixed array compiled into the library -- 12 MiB of fp32 (3 * 2^20 floats) in
 * the device image of every GPU that loads the library, held until the process
 * exits -- and its TMA descriptors are encoded into fixed slots of the context
 * rather than added to the context's descriptor cache.
 *
 * Same arguments, inputs, outputs and results as gr00t_denoise_step.
 * Set-up: gr00t_create looks up the array's device address on the context's
 * device (which loads the library's device code there and places the array),
 * so this call only reads the cached address; it must run with the context's
 * device current.  The call runs gr00t_denoise_step's
 * own launch sequence; a step whose scratch need in that sequence, at the
 * bound (batch, prefix), exceeds the array returns GR00T_EINVAL with the need
 * in gr00t_last_error, before anything is enqueued.  All calls in the process
 * share the one array: calls that overlap on the GPU (other streams, other
 * contexts) race on it.  The array keeps the last call's contents; every
 * kernel writes the scratch it reads within the same step, so nothing in it
 * has to start at zero.
 */
int gr00t_denoise_step_noalloc(gr00t_ctx* ctx, int k, const float* x_in, float* v_out);

/* Free everything the context owns (synchronises its stream first). */
int gr00t_destroy(gr00t_ctx* ctx);

/* Text of the context's last error ("" if none).  ctx may be NULL: the
 * last error of a failed gr00t_create on this thread. */
const char* gr00t_last_error(const gr00t_ctx* ctx);

/* ---- options and introspection ----------------------------------------- */
#define GR00T_OPT_USE_GRAPH 1     /* 1 (default): replay the loop as a CUDA graph */
#define GR00T_OPT_GEMM_PATH 2     /* 0: tensor-core path where supported (default), 1: CUDA-core path */
#define GR00T_OPT_WAIT_LIMIT 3    /* spin-wait iteration limit of bounded device waits (>= 0) */
#define GR00T_OPT_ATTN_PATH 4     /* expert family: 0 (default): tcgen05/TMEM kernel for bf16 (its key splits
                                     merged by a second kernel), else CUDA cores; 1: CUDA-core kernel;
                                     2: mma.sync head-folded kernel; 3: tcgen05/TMEM kernel */
#define GR00T_OPT_TIME_KERNELS 5  /* 1: every kernel launch of the loop records the global timer (ns)
                                     when its dependency wait returns -- one store by one thread, the
                                     launches and their programmatic-launch chain unchanged; read with
                                     gr00t_kernel_times.  0 (default): off */
#define GR00T_OPT_SPLIT_CAP 6     /* largest split-K factor of GEMMs that reduce in-kernel (1..16, power of 2; default 4) */
#define GR00T_OPT_RESID_SPLIT_CAP 7 /* same for residual GEMMs whose partials the next kernel folds in (default 8) */
#define GR00T_OPT_PERSISTENT_GEMM 8 /* 1 (default): persistent tensor-core GEMM for unsplit shapes with > 64 tokens */
#define GR00T_OPT_L2_PREFETCH 9   /* 1: the idle warps of every split tensor-core GEMM prefetch, with plain line
                                     prefetches, the next GEMM's weights (and the attention's bound K/V) into
                                     L2 while the GEMM streams its own (default 0: measured no gain) */
#define GR00T_OPT_NOALLOC_LIMIT 10 /* scratch (fp32 elements) gr00t_denoise_step_noalloc may take from its fixed
                                      array: 0 .. 3 * 2^20 (default: the whole array).  With the split planner's
                                      one-wave rule no step on a 152-SM GPU needs the whole array, so a lower
                                      limit is how the refusal is exercised */
#define GR00T_OPT_ATTN_SPLIT_CAP 11 /* expert family, tcgen05 attention: at most this many key splits
                                       (1 .. 32; 0 = automatic: as many as fill the SMs, up to 32) */
#define GR00T_OPT_GEMM_MULTICAST 13 /* 1: the persistent tensor-core GEMM runs as clusters of two CTAs over
                                       adjacent weight tiles that share each activation tile by TMA
                                       multicast; 0 (default, measured faster): one CTA per tile stream */
#define GR00T_OPT_ATTN_MULTICAST 14 /* 1: the expert attention runs the 2 or 4 row tiles of a sample as one
                                       cluster that fetches every key tile once and multicasts it; 0: each
                                       row tile fetches its own copies; 2 (default): the cluster where
                                       each CTA streams at most 4 key tiles (many key splits, e.g. batch 1),
                                       else not (both measured faster there) */
#define GR00T_OPT_GEMM_TSTORE 15   /* 1 (default): the persistent tensor-core GEMM stages its bf16 outputs (plain,
                                      RoPE, GeGLU epilogues), and the split GEMM with tiles of up to 128 tokens
                                      its fp32 residual partials, in shared memory and writes them with tensor
                                      stores; 0: every lane stores its own outputs */
#define GR00T_OPT_TEST_STALL 12   /* test hook: > 0 enqueues ahead of every step a one-thread kernel
                                     that waits this many polls for a device word nothing writes, then
                                     sets the device error word -- the bounded-wait error path with no
                                     copy or tensor-core operation in flight (0 = off, the default) */
int gr00t_set_option(gr00t_ctx* ctx, int option, int64_t value);

#define GR00T_INFO_KERNELS_PER_STEP 1   /* kernel launches of one denoise step            */
#define GR00T_INFO_WEIGHT_BYTES 2       /* bytes of weights one step reads                */
#define GR00T_INFO_DEVICE_BYTES 3       /* device memory the context owns                 */
#define GR00T_INFO_ERROR_FLAG 4         /* device error word (bounded waits), 0 if clean  */
#define GR00T_INFO_MOD_ROW 5            /* elements of one modulation-table row (all sites of a step and request) */
int gr00t_get_info(gr00t_ctx* ctx, int what, int64_t* value);

/* Kernel classes of one denoise step (gr00t_kernel_times). */
#define GR00T_KCLASS_QKV_GEMM 1    /* fused Q/K/V projection (+ RoPE epilogue)          */
#define GR00T_KCLASS_ATTENTION 2   /* attention over prefix ++ suffix K/V                */
#define GR00T_KCLASS_O_GEMM 3      /* output projection + (gated) residual               */
#define GR00T_KCLASS_UP_GEMM 4     /* MLP gate/up projection + GeGLU / GeLU              */
#define GR00T_KCLASS_DOWN_GEMM 5   /* MLP down projection + (gated) residual             */
#define GR00T_KCLASS_NORM 6        /* adaptive norms, step head and tail                 */
#define GR00T_KCLASS_OTHER 7       /* DiT action-encoder GEMMs                           */

/*
 * Per-launch durations of the most recent gr00t_denoise run with
 * GR00T_OPT_TIME_KERNELS = 1, in launch order: us[i] = stamp[i + 1] - stamp[i]
 * in microseconds, where stamp[i] is the global timer when launch i's
 * dependency wait returned (the previous kernel had completed) and a
 * one-thread tail kernel closes the last interval.  Each launch is thus
 * charged its share of the programmatic-launch chain, including its release
 * gap, and the durations of one loop add up to the loop's device time (less
 * the first launch's start-up).  ``kclass`` (nullable) receives each launch's
 * GR00T_KCLASS_*.  Writes at most ``max`` entries and their number to
 * ``*count`` (0 when stamps are off).  Synchronises the stream.
 */
int gr00t_kernel_times(gr00t_ctx* ctx, float* us, int* kclass, int max, int* count);

/*
 * Synchronise the context's stream and report the outcome of the bounded
 * device waits of everything enqueued since the last check: GR00T_ETIMEOUT
 * when one gave up (the device error word was set; the outputs of that work
 * are not valid), GR00T_OK otherwise.  The word is cleared, so the context
 * stays usable.  gr00t_denoise_host performs the same check before it returns;
 * the asynchronous calls cannot, so call this after them where the outcome
 * matters.
 */
int gr00t_sync(gr00t_ctx* ctx);

/*
 * Test-only: one velocity evaluation at step k from ``x_in`` (as
 * gr00t_denoise_step, the velocity discarded) with the fp32 residual stream
 * after block ``layer`` copied into ``h_out`` -- DEVICE fp32 [batch, tokens,
 * hidden], tokens = state_tokens + horizon; layer -1 gives the stream after
 * the step's input projection.  Intermediate tensors localise where two
 * implementations diverge (vla.cpp, Section III-E).  0 <= k < steps,
 * -1 <= layer < layers.  Asynchronous on the stream.
 */
int gr00t_debug_dump(gr00t_ctx* ctx, int k, const float* x_in, int layer, float* h_out);

/*
 * Test-only: the hoist check ("pi0.5 Design", cond component: the hoisted cond
 * work must equal its per-step evaluation).  Copies the modulation rows of step
 * k that gr00t_set_schedule hoisted into ``hoisted`` and evaluates the same
 * step's cond work on its own -- time MLP (where the geometry has one) and the
 * cond Dense over that step's ``batch`` time-embedding rows only, a GEMM of
 * batch rows instead of steps x batch -- into ``per_step``.  Both DEVICE
 * [batch][GR00T_INFO_MOD_ROW] in the geometry's dtype, batch = the scheduled
 * batch.  The two differ only in the GEMMs' accumulation order.  GR00T_ESTATE
 * without a schedule; 0 <= k < steps.  Asynchronous on the stream.
 */
int gr00t_debug_cond_step(gr00t_ctx* ctx, int k, void* hoisted, void* per_step);

#ifdef __cplusplus
}
#endif
#endif /* GR00T_H_ */
