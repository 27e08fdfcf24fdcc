"""Seeded synthetic inputs for the flow-matching action-expert denoise loop.

This module is shared by the CPU oracle (``oracle/``) and the CUDA path's
tests and benchmark.  It holds NO arithmetic of the method: it only draws
random tensors, rounds them to the storage type, and describes the shapes of
the five workloads.  Every tensor comes from ``(seed, tensor name)`` so both
sides see identical bytes on any machine.

Workloads (shapes from the pi0.5 expert geometry of "pi0.5 Design" and the
GR00T N1.7 DiT head of "GR00T N1.7", TensorRT Edge-LLM developer guide):

* ``tiny``   -- 2-layer expert, fp32, hidden 256, 4x64 query heads, 1 KV head,
  GeLU MLP 1024, prefix 64, horizon 16, action_dim 8, batch 1, 4 steps.
* ``pi05``   -- 18-layer pi0.5 expert, bf16, hidden 1024, 8x256 query heads,
  1 KV head, GeGLU 4096, 37 AdaRMS sites from a hoisted [3072,1024] Dense each,
  prefix 968 (3 views x 256 + 200 text), horizon 50, action_dim 32, batch 1,
  10 steps.
* ``gr00t``  -- 32-block DiT, bf16, hidden 1536, 32x48 heads, cross-attention
  over 300 VL tokens on even blocks, self-attention over 1 state + 16 action
  tokens on odd blocks, batch 1, 4 steps.
* ``pi05_b32`` -- ``pi05`` at batch 32, per-sample prefix.
* ``pi05_long`` -- ``pi05`` at batch 8 with a 4096-token prefix per sample.

Plus small cases (``small_bf16``, ``small_dit``, ...) that the oracle runs in
seconds while still spanning several GEMM/attention tiles with ragged tails.
"""
from __future__ import annotations

import copy
import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

FAMILY_EXPERT = 0  # pi0.5-style action expert (AdaRMS, single KV head)
FAMILY_DIT = 1     # GR00T-style DiT (AdaLayerNorm, cross/self attention)
DTYPE_FP32 = 0
DTYPE_BF16 = 1
MLP_GELU = 0
MLP_GEGLU = 1
WFMT_NATIVE = 0   # weights in the workload dtype
WFMT_FP8 = 1      # per-layer projections as E4M3 codes + one fp32 scale per output row

_BASE = dict(
    family=FAMILY_EXPERT, dtype=DTYPE_BF16, layers=2, hidden=256, q_heads=4,
    kv_heads=1, head_dim=64, mlp_dim=1024, mlp_kind=MLP_GELU, horizon=16,
    action_dim=8, state_tokens=0, batch=1, prefix=64, steps=4,
    time_dim=256, time_mlp=0, rope_theta=10000.0, norm_eps=1e-6,
    direction=-1, weight_format=WFMT_NATIVE, context_dim=0, state_dim=0,
)


def _g(**kw):
    g = dict(_BASE)
    g.update(kw)
    return g


_PI05 = dict(family=FAMILY_EXPERT, dtype=DTYPE_BF16, layers=18, hidden=1024,
             q_heads=8, kv_heads=1, head_dim=256, mlp_dim=4096,
             mlp_kind=MLP_GEGLU, horizon=50, action_dim=32, batch=1,
             prefix=968, steps=10, time_dim=1024, time_mlp=1, direction=-1)
_GR00T = dict(family=FAMILY_DIT, dtype=DTYPE_BF16, layers=32, hidden=1536,
              q_heads=32, kv_heads=32, head_dim=48, mlp_dim=6144,
              mlp_kind=MLP_GELU, horizon=16, action_dim=32, state_tokens=1,
              batch=1, prefix=300, steps=4, time_dim=1536, time_mlp=1,
              direction=+1)

CONFIGS = {
    # the five workloads
    "tiny": _g(dtype=DTYPE_FP32),
    "pi05": _g(**_PI05),
    "gr00t": _g(**_GR00T),
    "pi05_b32": _g(**dict(_PI05, batch=32)),
    "pi05_long": _g(**dict(_PI05, batch=8, prefix=4096)),
    # small cases: several tiles, ragged tails, seconds on the oracle
    "small_bf16": _g(layers=2, hidden=256, q_heads=2, head_dim=256,
                     mlp_dim=512, mlp_kind=MLP_GEGLU, horizon=50,
                     action_dim=32, batch=3, prefix=200, steps=3,
                     time_dim=256, time_mlp=1),
    "small_fp32": _g(dtype=DTYPE_FP32, layers=2, hidden=256, q_heads=2,
                     head_dim=256, mlp_dim=512, mlp_kind=MLP_GEGLU,
                     horizon=50, action_dim=32, batch=2, prefix=200,
                     steps=3, time_dim=256, time_mlp=1),
    "small_dit": _g(family=FAMILY_DIT, layers=4, hidden=384, q_heads=8,
                    kv_heads=8, head_dim=48, mlp_dim=1536, horizon=16,
                    action_dim=32, state_tokens=1, batch=2, prefix=300,
                    steps=4, time_dim=384, time_mlp=1, direction=+1),
    # FP8 weight streaming (E4M3 per-layer projections): full-size and small
    "pi05_fp8": _g(**dict(_PI05, weight_format=WFMT_FP8)),
    "gr00t_fp8": _g(**dict(_GR00T, weight_format=WFMT_FP8)),
    "small_fp8": _g(layers=2, hidden=256, q_heads=2, head_dim=256,
                    mlp_dim=512, mlp_kind=MLP_GEGLU, horizon=50,
                    action_dim=32, batch=3, prefix=200, steps=3,
                    time_dim=256, time_mlp=1, weight_format=WFMT_FP8),
    "small_dit_fp8": _g(family=FAMILY_DIT, layers=4, hidden=384, q_heads=8,
                        kv_heads=8, head_dim=48, mlp_dim=1536, horizon=16,
                        action_dim=32, state_tokens=1, batch=2, prefix=300,
                        steps=4, time_dim=384, time_mlp=1, direction=+1,
                        weight_format=WFMT_FP8),
    # DiT with the cross K/V projected at bind time from VL features [B, P, context_dim]
    "gr00t_ctx": _g(**dict(_GR00T, context_dim=2048)),
    "small_dit_ctx": _g(family=FAMILY_DIT, layers=4, hidden=384, q_heads=8,
                        kv_heads=8, head_dim=48, mlp_dim=1536, horizon=16,
                        action_dim=32, state_tokens=1, batch=2, prefix=300,
                        steps=4, time_dim=384, time_mlp=1, direction=+1,
                        context_dim=256),
    # DiT with the robot state encoded at bind time: raw state [B, Ns, state_dim]
    "gr00t_state": _g(**dict(_GR00T, state_dim=132)),
    "small_dit_state": _g(family=FAMILY_DIT, layers=4, hidden=384, q_heads=8,
                          kv_heads=8, head_dim=48, mlp_dim=1536, horizon=16,
                          action_dim=32, state_tokens=1, batch=2, prefix=300,
                          steps=4, time_dim=384, time_mlp=1, direction=+1,
                          state_dim=40),
    "small_dit_fp32": _g(family=FAMILY_DIT, dtype=DTYPE_FP32, layers=2,
                         hidden=192, q_heads=4, kv_heads=4, head_dim=48,
                         mlp_dim=768, horizon=16, action_dim=32,
                         state_tokens=1, batch=2, prefix=77, steps=4,
                         time_dim=192, time_mlp=1, direction=+1),
}


def config(name: str, **overrides) -> dict:
    """Return a copy of a named geometry, optionally with fields overridden."""
    g = copy.deepcopy(CONFIGS[name])
    g.update(overrides)
    g["name"] = name
    return g


# ----------------------------------------------------------------------------
# Derived sizes (shape bookkeeping only)
# ----------------------------------------------------------------------------

def norm_sites(g: dict) -> int:
    """Number of adaptive-norm sites (rows of one modulation-table entry)."""
    if g["family"] == FAMILY_EXPERT:
        return 2 * g["layers"] + 1
    return g["layers"] + 1


def row_width(g: dict) -> int:
    """Width of one modulation row: (scale, shift, gate) or (scale, shift)."""
    return (3 if g["family"] == FAMILY_EXPERT else 2) * g["hidden"]


def qkv_rows(g: dict, layer: int) -> int:
    """Output rows of the layer's fused Q/K/V projection."""
    qd = g["q_heads"] * g["head_dim"]
    kd = g["kv_heads"] * g["head_dim"]
    if g["family"] == FAMILY_DIT and layer % 2 == 0:
        return qd  # cross-attention block: K/V come projected from the context
    return qd + 2 * kd


def up_rows(g: dict) -> int:
    return (2 if g["mlp_kind"] == MLP_GEGLU else 1) * g["mlp_dim"]


def tokens(g: dict) -> int:
    """Token rows per sample inside the stack."""
    return g["horizon"] + g["state_tokens"]


def weight_shapes(g: dict) -> dict:
    """Name -> shape of every weight tensor, nn.Linear [out, in] layout."""
    D, A, E, L = g["hidden"], g["action_dim"], g["time_dim"], g["layers"]
    S, R = norm_sites(g), row_width(g)
    qd = g["q_heads"] * g["head_dim"]
    sh = {}
    if g["time_mlp"]:
        sh["time_mlp_in_w"] = (E, E)
        sh["time_mlp_in_b"] = (E,)
        sh["time_mlp_out_w"] = (E, E)
        sh["time_mlp_out_b"] = (E,)
    sh["cond_w"] = (S, R, E)
    sh["cond_b"] = (S, R)
    if g["family"] == FAMILY_EXPERT:
        sh["action_in_w"] = (D, A)
        sh["action_in_b"] = (D,)
    else:
        sh["enc_w1"] = (D, A)
        sh["enc_b1"] = (D,)
        sh["enc_w2"] = (D, D + E)   # input = concat(action features, time embedding)
        sh["enc_b2"] = (D,)
        sh["enc_w3"] = (D, D)
        sh["enc_b3"] = (D,)
    sh["action_out_w"] = (A, D)
    sh["action_out_b"] = (A,)
    for l in range(L):
        sh[f"qkv_w.{l}"] = (qkv_rows(g, l), D)
        sh[f"o_w.{l}"] = (D, qd)
        sh[f"up_w.{l}"] = (up_rows(g), D)
        sh[f"down_w.{l}"] = (D, g["mlp_dim"])
    Ds = g.get("state_dim", 0)
    if g["family"] == FAMILY_DIT and Ds > 0:   # the state encoder: state_dim -> D -> D
        sh["state_w1"] = (D, Ds)
        sh["state_b1"] = (D,)
        sh["state_w2"] = (D, D)
        sh["state_b2"] = (D,)
    Dc = g.get("context_dim", 0)
    if g["family"] == FAMILY_DIT and Dc > 0:   # cross K/V projections of the even blocks
        kd = g["kv_heads"] * g["head_dim"]
        for l in range(0, L, 2):
            sh[f"cross_k_w.{l}"] = (kd, Dc)
            sh[f"cross_v_w.{l}"] = (kd, Dc)
    return sh


# ----------------------------------------------------------------------------
# Random draws
# ----------------------------------------------------------------------------

_CHUNK = 1 << 22  # elements per independently seeded block (fixed: bytes do not depend on threads)
_POOL = None


def _rng(seed: int, name: str, block: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), zlib.crc32(name.encode()), int(block)]))


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1))
    return _POOL


def _round_bf16_inplace(a: np.ndarray) -> None:
    bits = a.view(np.uint32)
    lsb = bits >> np.uint32(16)
    lsb &= np.uint32(1)
    lsb += np.uint32(0x7FFF)
    bits += lsb
    bits &= np.uint32(0xFFFF0000)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bfloat16 (ties to even); returns float32."""
    a = np.array(a, dtype=np.float32, copy=True, order="C")
    _round_bf16_inplace(a.reshape(-1))
    return a


def _normal_many(jobs):
    """Draw several tensors at once; ``jobs`` = [(seed, name, shape, std, bf16)].

    Each tensor is ~N(0, std^2), float32, drawn in fixed-size blocks seeded by
    (seed, name, block index), so its bytes never depend on the thread count.
    """
    outs, work = [], []
    for seed, name, shape, std, bf16 in jobs:
        out = np.empty(shape, dtype=np.float32)
        outs.append(out)
        flat = out.reshape(-1)
        for i in range((flat.size + _CHUNK - 1) // _CHUNK):
            work.append((seed, name, i, flat[i * _CHUNK:(i + 1) * _CHUNK], std, bf16))

    def fill(job):
        seed, name, i, blk, std, bf16 = job
        _rng(seed, name, i).standard_normal(out=blk, dtype=np.float32)
        if std != 1.0:
            blk *= np.float32(std)
        if bf16:
            _round_bf16_inplace(blk)

    list(_pool().map(fill, work))
    return outs


def _normal(seed, name, shape, std, bf16):
    return _normal_many([(seed, name, shape, std, bf16)])[0]


FP8_LAYERED = ("qkv_w", "o_w", "up_w", "down_w")   # the projections stored as E4M3 in FP8 workloads


def _e4m3_codes(y: np.ndarray) -> np.ndarray:
    """Storage codes of values |y| <= 448 in the E4M3 8-bit format (sign bit 7,
    exponent field bits 6..3 with bias 7, mantissa bits 2..0; subnormals below
    2^-6), magnitudes truncated toward zero.  Any code is a valid input: both
    sides of the parity tests read the same codes."""
    a = np.abs(y).astype(np.float64)
    f, x = np.frexp(a)                       # a = f * 2^x, f in [0.5, 1)
    normal = a >= 2.0 ** -6
    e = np.clip(x + 6, 1, 15)                # biased exponent of a = 2f * 2^(x - 1)
    m = np.clip(np.floor((2.0 * f - 1.0) * 8.0), 0, 7)
    m = np.where(e == 15, np.minimum(m, 6), m)   # (15, 7) is NaN
    sub = np.clip(np.floor(a * 2.0 ** 9), 0, 7)
    mag = np.where(normal, e * 8 + m, sub).astype(np.uint8)
    return np.where(y < 0, mag | np.uint8(0x80), mag).astype(np.uint8)


def _to_fp8_rows(w: np.ndarray):
    """(codes, scales) of a [out, in] matrix: scale = max |row| / 448 per row."""
    amax = np.max(np.abs(w), axis=1).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    y = np.clip(w / scale[:, None], -448.0, 448.0)
    return _e4m3_codes(y), scale


def make_weights(g: dict, seed: int = 0, std: float = 0.02) -> dict:
    """Weights ~N(0, std), rounded to bf16 for bf16 workloads (float32 arrays).

    FP8 workloads (``weight_format`` WFMT_FP8) store the per-layer projections
    as uint8 E4M3 codes ``name`` plus float32 row scales ``name + '.scale'``.
    """
    bf16 = g["dtype"] == DTYPE_BF16
    shapes = weight_shapes(g)
    arrs = _normal_many([(seed, "w." + k, s, std, bf16) for k, s in shapes.items()])
    w = dict(zip(shapes.keys(), arrs))
    if g.get("weight_format", WFMT_NATIVE) == WFMT_FP8:
        for k in list(w):
            if k.split(".")[0] in FP8_LAYERED:
                w[k], w[k + ".scale"] = _to_fp8_rows(w[k])
    return w


def make_prefix_kv(g: dict, seed: int = 0, batch: int | None = None, prefix: int | None = None):
    """Per-layer prefix / VL-context K and V, ~N(0,1), [B, P, Hkv, Dh].

    Expert family: every layer has prefix K/V (single KV head).  DiT family:
    only cross-attention (even) blocks have them; odd entries are None.
    """
    B = g["batch"] if batch is None else batch
    P = g["prefix"] if prefix is None else prefix
    bf16 = g["dtype"] == DTYPE_BF16
    shp = (B, P, g["kv_heads"], g["head_dim"])
    layers = [l for l in range(g["layers"]) if not (g["family"] == FAMILY_DIT and l % 2 == 1)]
    jobs = []
    for l in layers:
        jobs += [(seed, f"k.{l}", shp, 1.0, bf16), (seed, f"v.{l}", shp, 1.0, bf16)]
    arrs = _normal_many(jobs)
    K = [None] * g["layers"]
    V = [None] * g["layers"]
    for j, l in enumerate(layers):
        K[l], V[l] = arrs[2 * j], arrs[2 * j + 1]
    return K, V


def make_noise(g: dict, seed: int = 0, batch: int | None = None) -> np.ndarray:
    """Initial action chunk x ~N(0,1), float32 [B, H, A]."""
    B = g["batch"] if batch is None else batch
    return _rng(seed, "x_noise").standard_normal(size=(B, g["horizon"], g["action_dim"]), dtype=np.float32)


def make_state_tokens(g: dict, seed: int = 0, batch: int | None = None):
    """DiT family: embedded state token(s) ~N(0,1), float32 [B, n_state, D]."""
    if g["state_tokens"] == 0:
        return None
    B = g["batch"] if batch is None else batch
    return _rng(seed, "state").standard_normal(size=(B, g["state_tokens"], g["hidden"]), dtype=np.float32)


def make_raw_state(g: dict, seed: int = 0, batch: int | None = None):
    """DiT family with state_dim > 0: the raw robot state ~N(0,1), float32
    [B, n_state, state_dim] (bf16-rounded for bf16 workloads), the input of the
    bind-time state encoder."""
    if g["state_tokens"] == 0 or g.get("state_dim", 0) == 0:
        return None
    B = g["batch"] if batch is None else batch
    return _normal(seed, "state_raw", (B, g["state_tokens"], g["state_dim"]), 1.0, g["dtype"] == DTYPE_BF16)


def make_masks(g: dict, seed: int = 0, batch: int | None = None, kind: str = "ones"):
    """DiT family: (text_mask, image_mask), uint8 [B, P], 1 = visible.

    ``kind='ones'`` gives all-visible masks; ``kind='random'`` marks each
    context token visible with probability 1/2 (at least one per row).
    """
    if g["family"] != FAMILY_DIT:
        return None, None
    B = g["batch"] if batch is None else batch
    P = g["prefix"]
    if kind == "ones":
        m = np.ones((B, P), np.uint8)
        return m, m.copy()
    out = []
    for name in ("text_mask", "image_mask"):
        m = (_rng(seed, name).random((B, P)) < 0.5).astype(np.uint8)
        m[:, 0] = 1
        out.append(m)
    return tuple(out)


def make_context_features(g: dict, seed: int = 0, batch: int | None = None) -> np.ndarray:
    """DiT family with context_dim > 0: VL features ~N(0,1), [B, P, context_dim]
    (bf16-rounded for bf16 workloads), the input of the bind-time K/V projections."""
    B = g["batch"] if batch is None else batch
    return _normal(seed, "features", (B, g["prefix"], g["context_dim"]), 1.0, g["dtype"] == DTYPE_BF16)


def make_case(name_or_geom, seed: int = 0, **overrides) -> dict:
    """Everything one denoise call needs: geometry, weights, prefix, noise.

    DiT workloads with ``context_dim`` > 0 carry VL ``features`` instead of
    bound K/V (K and V are lists of None): the cross K/V are projected from them.
    DiT workloads with ``state_dim`` > 0 carry the raw robot state ``state_raw``
    instead of the embedded ``state`` tokens (None): the state encoder embeds it.
    """
    g = config(name_or_geom, **overrides) if isinstance(name_or_geom, str) else dict(name_or_geom)
    tm, im = make_masks(g, seed)
    feats = None
    if g["family"] == FAMILY_DIT and g.get("context_dim", 0) > 0:
        feats = make_context_features(g, seed)
        K, V = [None] * g["layers"], [None] * g["layers"]
    else:
        K, V = make_prefix_kv(g, seed)
    raw = make_raw_state(g, seed) if g["family"] == FAMILY_DIT else None
    state = None if raw is not None else make_state_tokens(g, seed)
    return dict(geom=g, weights=make_weights(g, seed), K=K, V=V, x_noise=make_noise(g, seed),
                state=state, state_raw=raw, text_mask=tm, image_mask=im, features=feats, seed=seed)
