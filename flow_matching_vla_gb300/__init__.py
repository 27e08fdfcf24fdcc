"""GB300 (sm_103a) flow-matching action-expert denoise loop.

Python binding of the C-ABI library ``libgr00t.so`` (``include/gr00t.h``).
It marshals arguments only: geometry and weights into the C structs, torch
tensors into device pointers, the torch stream into the library's stream.
Every step of the loop runs in the library's CUDA kernels; without the
compiled library (or without a GB300) the calls raise, there is no fallback.

    loop = DenoiseLoop(geom, weights)           # gr00t_create
    loop.bind_prefix_kv(K, V)                   # gr00t_bind_prefix_kv
    loop.set_schedule(steps=10, batch=1)        # gr00t_set_schedule (hoisted cond)
    actions = loop.denoise(x_noise)             # gr00t_denoise

``geom`` is a dict with the fields of ``gr00t_geometry`` (family, dtype,
layers, hidden, q_heads, kv_heads, head_dim, mlp_dim, mlp_kind, horizon,
action_dim, state_tokens, time_dim, time_mlp, direction, rope_theta,
norm_eps) plus optional max_batch / max_prefix / max_steps (defaults: the
dict's batch / prefix / steps).  ``weights`` maps the names of
``gr00t_weights`` to arrays ([out, in] layout; per-layer tensors named
``qkv_w.<l>``, ``o_w.<l>``, ``up_w.<l>``, ``down_w.<l>``).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _abi
from ._abi import (DTYPE_BF16, DTYPE_FP32, FAMILY_DIT, FAMILY_EXPERT, MLP_GEGLU, MLP_GELU,
                   OPT_ATTN_PATH, OPT_GEMM_PATH, OPT_TIME_KERNELS, OPT_USE_GRAPH, OPT_WAIT_LIMIT,
                   OPT_SPLIT_CAP, OPT_RESID_SPLIT_CAP, OPT_PERSISTENT_GEMM, OPT_L2_PREFETCH, OPT_NOALLOC_LIMIT,
                   OPT_ATTN_SPLIT_CAP, OPT_TEST_STALL, OPT_GEMM_MULTICAST, OPT_ATTN_MULTICAST, OPT_GEMM_TSTORE, ETIMEOUT,
                   INFO_DEVICE_BYTES, INFO_ERROR_FLAG, INFO_KERNELS_PER_STEP, INFO_WEIGHT_BYTES, INFO_MOD_ROW,
                   KCLASS_ATTENTION, KCLASS_DOWN_GEMM, KCLASS_NORM, KCLASS_O_GEMM, KCLASS_QKV_GEMM,
                   KCLASS_UP_GEMM, KCLASS_OTHER, KCLASS_NAMES, WFMT_NATIVE, WFMT_FP8)

__all__ = ["DenoiseLoop", "Gr00tError", "validate_geometry", "load_library", "FAMILY_EXPERT",
           "FAMILY_DIT", "DTYPE_FP32", "DTYPE_BF16", "MLP_GELU", "MLP_GEGLU"]

_SINGLE = ("time_mlp_in_w", "time_mlp_in_b", "time_mlp_out_w", "time_mlp_out_b", "cond_w", "cond_b",
           "action_in_w", "action_in_b", "enc_w1", "enc_b1", "enc_w2", "enc_b2", "enc_w3", "enc_b3",
           "action_out_w", "action_out_b", "state_w1", "state_b1", "state_w2", "state_b2")
_LAYERED = ("qkv_w", "o_w", "up_w", "down_w")


class Gr00tError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{_abi.STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def load_library(path=None):
    return _abi.load(path)


def _geometry(g: dict) -> _abi.Geometry:
    s = _abi.Geometry()
    s.abi_version = _abi.ABI_VERSION
    for f in ("family", "dtype", "layers", "hidden", "q_heads", "kv_heads", "head_dim", "mlp_dim",
              "mlp_kind", "horizon", "action_dim", "state_tokens", "time_dim", "time_mlp",
              "direction"):
        setattr(s, f, int(g[f]))
    s.max_batch = int(g.get("max_batch", g.get("batch", 1)))
    s.max_prefix = int(g.get("max_prefix", g.get("prefix", 0)))
    s.max_steps = int(g.get("max_steps", g.get("steps", 1)))
    s.rope_theta = float(g.get("rope_theta", 10000.0))
    s.norm_eps = float(g.get("norm_eps", 1e-6))
    s.weight_format = int(g.get("weight_format", WFMT_NATIVE))
    s.context_dim = int(g.get("context_dim", 0))
    s.state_dim = int(g.get("state_dim", 0))
    return s


def validate_geometry(g: dict):
    """(status, message) of gr00t_validate_geometry; needs no GPU."""
    lib = _abi.load()
    buf = ctypes.create_string_buffer(256)
    rc = lib.gr00t_validate_geometry(ctypes.byref(_geometry(g)), buf, len(buf))
    return rc, buf.value.decode()


def _torch():
    import torch
    return torch


def _storage_tensor(a, dtype_code):
    """A contiguous CPU/GPU torch tensor of the storage dtype holding ``a``."""
    torch = _torch()
    t = a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a))
    want = torch.bfloat16 if dtype_code == DTYPE_BF16 else torch.float32
    if t.dtype != want:
        t = t.to(want)
    return t.contiguous()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


class DenoiseLoop:
    """One gr00t context: weights resident on the GPU, prefix bound, schedule hoisted."""

    def __init__(self, geom: dict, weights: dict, stream=None, device_weights: bool = False):
        torch = _torch()
        self._lib = _abi.load()
        self.geom = dict(geom)
        self._g = _geometry(self.geom)
        self.dtype_code = int(geom["dtype"])
        self.torch_dtype = torch.bfloat16 if self.dtype_code == DTYPE_BF16 else torch.float32
        # The library enqueues on ``stream`` (default: torch's current stream).  On the
        # legacy default stream it creates its own blocking stream, which the driver
        # orders implicitly with the default stream torch uses.
        if stream is None:
            stream = torch.cuda.current_stream()
        self.stream = stream
        L = int(geom["layers"])
        keep = []
        w = _abi.Weights()
        w.location = _abi.MEM_DEVICE if device_weights else _abi.MEM_HOST
        for name in _SINGLE:
            if name in weights:
                t = _storage_tensor(weights[name], self.dtype_code)
                if device_weights:
                    t = t.cuda()
                keep.append(t)
                setattr(w, name, _ptr(t))
        arrays = {}
        fp8 = int(geom.get("weight_format", WFMT_NATIVE)) == WFMT_FP8
        for name in _LAYERED:
            for suffix, field in (("", name), (".scale", name[:-1] + "s")):
                if suffix and not fp8:
                    continue
                ts = []
                for l in range(L):
                    a = weights[f"{name}.{l}{suffix}"]
                    if fp8 and not suffix:     # E4M3 codes, passed as stored
                        t = a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a))
                        t = t.view(torch.uint8).contiguous()
                    elif suffix:               # fp32 row scales
                        t = _storage_tensor(a, DTYPE_FP32)
                    else:
                        t = _storage_tensor(a, self.dtype_code)
                    if device_weights:
                        t = t.cuda()
                    ts.append(t)
                keep += ts
                arr = (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])
                arrays[field] = arr
                setattr(w, field, ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)))
        if int(geom.get("context_dim", 0)) > 0:   # DiT cross K/V projections, even blocks
            for field in ("cross_k_w", "cross_v_w"):
                ts = [None if l % 2 else _storage_tensor(weights[f"{field}.{l}"], self.dtype_code) for l in range(L)]
                if device_weights:
                    ts = [None if t is None else t.cuda() for t in ts]
                keep += [t for t in ts if t is not None]
                arr = (ctypes.c_void_p * L)(*[0 if t is None else t.data_ptr() for t in ts])
                arrays[field] = arr
                setattr(w, field, ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)))
        ctx = ctypes.c_void_p()
        with torch.cuda.device(self.stream.device):
            rc = self._lib.gr00t_create(ctypes.byref(self._g), ctypes.byref(w),
                                        ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(ctx))
        if rc != 0:
            raise Gr00tError(rc, self._lib.gr00t_last_error(None).decode())
        self._ctx = ctx
        self._bound = ()
        self.batch = None

    # -- helpers --------------------------------------------------------------
    def _check(self, rc):
        if rc != 0:
            raise Gr00tError(rc, self._lib.gr00t_last_error(self._ctx).decode())

    def close(self):
        if getattr(self, "_ctx", None):
            self._lib.gr00t_destroy(self._ctx)
            self._ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- API --------------------------------------------------------------------
    def bind_prefix_kv(self, K, V, text_mask=None, image_mask=None, state=None):
        """Bind per-layer K/V (device tensors [B, P, Hkv, Dh]; None for DiT odd blocks)."""
        torch = _torch()
        L = int(self.geom["layers"])
        ks, vs = [], []
        B = P = None
        for l in range(L):
            k, v = K[l], V[l]
            if k is None:
                ks.append(None)
                vs.append(None)
                continue
            for t in (k, v):
                if not (t.is_cuda and t.is_contiguous() and t.dtype == self.torch_dtype):
                    raise ValueError("K/V must be contiguous CUDA tensors of the geometry dtype")
            B, P = int(k.shape[0]), int(k.shape[1])
            ks.append(k)
            vs.append(v)
        if B is None:
            raise ValueError("no K/V given")
        karr = (ctypes.c_void_p * L)(*[0 if t is None else t.data_ptr() for t in ks])
        varr = (ctypes.c_void_p * L)(*[0 if t is None else t.data_ptr() for t in vs])
        masks = []
        for m in (text_mask, image_mask):
            if m is not None:
                if not (m.is_cuda and m.dtype == torch.uint8 and m.is_contiguous()):
                    raise ValueError("masks must be contiguous CUDA uint8 tensors")
            masks.append(m)
        if state is not None and not (state.is_cuda and state.dtype == torch.float32 and state.is_contiguous()):
            raise ValueError("state tokens must be a contiguous CUDA float32 tensor")
        self._check(self._lib.gr00t_bind_prefix_kv(
            self._ctx, B, P, ctypes.cast(karr, ctypes.POINTER(ctypes.c_void_p)),
            ctypes.cast(varr, ctypes.POINTER(ctypes.c_void_p)),
            None if masks[0] is None else _ptr(masks[0]), None if masks[1] is None else _ptr(masks[1]),
            None if state is None else _ptr(state)))
        self._bound = (ks, vs, masks, state)   # the library borrows these
        self.batch = B
        return self

    def bind_kv_pool(self, pools, prefix: int):
        """EXPERT: bind per-layer paged K/V pools (device tensors [2, B, capacity, 1, Dh]
        of the geometry dtype, prefix K/V in slot rows [0, prefix)); each step writes its
        suffix K/V into rows [prefix, prefix + H).  The pools are borrowed and written."""
        L = int(self.geom["layers"])
        for t in pools:
            if not (t.is_cuda and t.is_contiguous() and t.dtype == self.torch_dtype and t.dim() == 5):
                raise ValueError("pools must be contiguous 5-D CUDA tensors [2, B, capacity, 1, Dh]")
        B, cap = int(pools[0].shape[1]), int(pools[0].shape[2])
        arr = (ctypes.c_void_p * L)(*[t.data_ptr() for t in pools])
        self._check(self._lib.gr00t_bind_kv_pool(self._ctx, B, int(prefix), cap,
                                                 ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))))
        self._bound = (list(pools),)
        self.batch = B
        return self

    def bind_context(self, features, text_mask=None, image_mask=None, state=None):
        """DiT with context_dim: project VL features (device tensor [B, P, context_dim]
        of the geometry dtype) into the cross K/V on the GPU and bind them."""
        torch = _torch()
        if not (features.is_cuda and features.is_contiguous() and features.dtype == self.torch_dtype):
            raise ValueError("features must be a contiguous CUDA tensor of the geometry dtype")
        for m in (text_mask, image_mask):
            if m is not None and not (m.is_cuda and m.dtype == torch.uint8 and m.is_contiguous()):
                raise ValueError("masks must be contiguous CUDA uint8 tensors")
        if state is not None and not (state.is_cuda and state.dtype == torch.float32 and state.is_contiguous()):
            raise ValueError("state tokens must be a contiguous CUDA float32 tensor")
        B, P = int(features.shape[0]), int(features.shape[1])
        self._check(self._lib.gr00t_bind_context(
            self._ctx, B, P, _ptr(features), None if text_mask is None else _ptr(text_mask),
            None if image_mask is None else _ptr(image_mask), None if state is None else _ptr(state)))
        self._bound = (features, [text_mask, image_mask], state)
        self.batch = B
        return self

    def set_schedule(self, steps: int, batch: int):
        self._check(self._lib.gr00t_set_schedule(self._ctx, int(steps), int(batch)))
        self.steps = int(steps)
        return self

    def _chunk(self, x):
        torch = _torch()
        if not (x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()):
            raise ValueError("action chunks are contiguous CUDA float32 tensors [B, H, A]")
        return x

    def denoise(self, x_noise, out=None):
        x_noise = self._chunk(x_noise)
        if out is None:
            out = _torch().empty_like(x_noise)
        self._check(self._lib.gr00t_denoise(self._ctx, _ptr(x_noise), _ptr(self._chunk(out))))
        return out

    def denoise_host(self, x_noise, out):
        """Host-buffer variant: CPU float32 tensors (pinned for async copies); synchronous."""
        self._check(self._lib.gr00t_denoise_host(self._ctx, _ptr(x_noise), _ptr(out)))
        return out

    def denoise_step(self, k: int, x_in, v_out=None):
        x_in = self._chunk(x_in)
        if v_out is None:
            v_out = _torch().empty_like(x_in)
        self._check(self._lib.gr00t_denoise_step(self._ctx, int(k), _ptr(x_in), _ptr(self._chunk(v_out))))
        return v_out

    def denoise_step_noalloc(self, k: int, x_in, v_out):
        """gr00t_denoise_step_noalloc: the same step with scratch from the library's fixed array."""
        self._check(self._lib.gr00t_denoise_step_noalloc(self._ctx, int(k), _ptr(self._chunk(x_in)),
                                                         _ptr(self._chunk(v_out))))
        return v_out

    def set_option(self, option: int, value: int):
        self._check(self._lib.gr00t_set_option(self._ctx, int(option), int(value)))

    def kernel_times(self, max_count: int = 1 << 16):
        """(durations in us, kernel classes) of every launch of the last denoise run with
        OPT_TIME_KERNELS = 1, each launch charged its share of the launch chain."""
        buf = (ctypes.c_float * max_count)()
        cls = (ctypes.c_int * max_count)()
        n = ctypes.c_int()
        self._check(self._lib.gr00t_kernel_times(self._ctx, buf, cls, max_count, ctypes.byref(n)))
        return list(buf[:n.value]), list(cls[:n.value])

    def sync(self):
        """gr00t_sync: wait for the stream; raise Gr00tError(ETIMEOUT) if a bounded device wait gave up."""
        self._check(self._lib.gr00t_sync(self._ctx))

    def debug_dump(self, k: int, x_in, layer: int, h_out=None):
        """gr00t_debug_dump: residual stream [B, tokens, hidden] (fp32) after block ``layer``
        (-1: after the input projection) of velocity evaluation k from ``x_in``."""
        torch = _torch()
        x_in = self._chunk(x_in)
        if h_out is None:
            tok = int(self.geom["horizon"]) + int(self.geom.get("state_tokens", 0))
            h_out = torch.empty((x_in.shape[0], tok, int(self.geom["hidden"])), dtype=torch.float32,
                                device=x_in.device)
        if not (h_out.is_cuda and h_out.dtype == torch.float32 and h_out.is_contiguous()):
            raise ValueError("h_out must be a contiguous CUDA float32 tensor")
        self._check(self._lib.gr00t_debug_dump(self._ctx, int(k), _ptr(x_in), int(layer), _ptr(h_out)))
        return h_out

    def debug_cond_step(self, k: int, batch: int):
        """gr00t_debug_cond_step: (hoisted, per_step) modulation rows of step k, each
        [batch, row] in the geometry's dtype (batch = the scheduled batch)."""
        torch = _torch()
        row = self.info(INFO_MOD_ROW)
        dt = torch.bfloat16 if int(self.geom["dtype"]) == DTYPE_BF16 else torch.float32
        hoisted = torch.empty((int(batch), row), dtype=dt, device="cuda")
        per_step = torch.empty_like(hoisted)
        self._check(self._lib.gr00t_debug_cond_step(self._ctx, int(k), _ptr(hoisted), _ptr(per_step)))
        return hoisted, per_step

    def info(self, what: int) -> int:
        v = ctypes.c_int64()
        self._check(self._lib.gr00t_get_info(self._ctx, int(what), ctypes.byref(v)))
        return int(v.value)


def from_case(case: dict, stream=None, steps=None, device_weights=False, **geom_overrides):
    """Create, bind and schedule a loop from a dict holding ``geom``, ``weights``,
    ``K``, ``V`` and optionally ``text_mask``, ``image_mask``, ``state``
    (numpy arrays or tensors).  Inputs are copied to the GPU once; returns
    (loop, dict of the device tensors the loop borrows)."""
    torch = _torch()
    g = dict(case["geom"])
    g.update(geom_overrides)
    loop = DenoiseLoop(g, case["weights"], stream=stream, device_weights=device_weights)
    dt = loop.torch_dtype

    def dev(a, dtype):
        if a is None:
            return None
        t = a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a))
        return t.to(device="cuda", dtype=dtype).contiguous()

    tm = dev(case.get("text_mask"), torch.uint8)
    im = dev(case.get("image_mask"), torch.uint8)
    # the embedded state tokens, or (state_dim > 0) the raw robot state the bind encodes
    st = dev(case.get("state") if case.get("state_raw") is None else case["state_raw"], torch.float32)
    if case.get("features") is not None:   # cross K/V projected on the GPU at bind time
        feats = dev(case["features"], dt)
        torch.cuda.synchronize()
        loop.bind_context(feats, tm, im, st)
        loop.set_schedule(steps or g["steps"], int(feats.shape[0]))
        return loop, dict(features=feats, text_mask=tm, image_mask=im, state=st)
    K = [dev(k, dt) for k in case["K"]]
    V = [dev(v, dt) for v in case["V"]]
    torch.cuda.synchronize()
    loop.bind_prefix_kv(K, V, tm, im, st)
    B = next(k.shape[0] for k in K if k is not None)
    loop.set_schedule(steps or g["steps"], B)
    return loop, dict(K=K, V=V, text_mask=tm, image_mask=im, state=st)
