"""ctypes mirror of ``include/gr00t.h`` and the library loader.

Argument marshalling only: no step of the denoise loop runs here.  Loading
fails loudly when the compiled library is missing; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
HEADER = os.path.join(ROOT, "include", "gr00t.h")
LIB_PATH = os.path.join(PKG, "libgr00t.so")

ABI_VERSION = 3
WFMT_NATIVE, WFMT_FP8 = 0, 1
OK, EINVAL, ENOMEM, ECUDA, ESTATE, EUNSUPPORTED, ETIMEOUT = 0, -1, -2, -3, -4, -5, -6
FAMILY_EXPERT, FAMILY_DIT = 0, 1
DTYPE_FP32, DTYPE_BF16 = 0, 1
MLP_GELU, MLP_GEGLU = 0, 1
MEM_HOST, MEM_DEVICE = 0, 1
OPT_USE_GRAPH, OPT_GEMM_PATH, OPT_WAIT_LIMIT, OPT_ATTN_PATH, OPT_TIME_KERNELS = 1, 2, 3, 4, 5
OPT_SPLIT_CAP, OPT_RESID_SPLIT_CAP, OPT_PERSISTENT_GEMM, OPT_L2_PREFETCH = 6, 7, 8, 9
OPT_ATTN_SPLIT_CAP = 11
OPT_TEST_STALL = 12
OPT_GEMM_MULTICAST = 13
OPT_ATTN_MULTICAST = 14
OPT_GEMM_TSTORE = 15
OPT_NOALLOC_LIMIT = 10
KCLASS_QKV_GEMM, KCLASS_ATTENTION, KCLASS_O_GEMM, KCLASS_UP_GEMM, KCLASS_DOWN_GEMM, KCLASS_NORM = 1, 2, 3, 4, 5, 6
KCLASS_OTHER = 7
KCLASS_NAMES = {1: "qkv_gemm", 2: "attention", 3: "o_gemm", 4: "up_gemm", 5: "down_gemm", 6: "norm",
                7: "other"}
INFO_KERNELS_PER_STEP, INFO_WEIGHT_BYTES, INFO_DEVICE_BYTES, INFO_ERROR_FLAG = 1, 2, 3, 4
INFO_MOD_ROW = 5

STATUS_NAMES = {OK: "OK", EINVAL: "EINVAL", ENOMEM: "ENOMEM", ECUDA: "ECUDA", ESTATE: "ESTATE",
                EUNSUPPORTED: "EUNSUPPORTED", ETIMEOUT: "ETIMEOUT"}


class Geometry(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "abi_version", "family", "dtype", "layers", "hidden", "q_heads", "kv_heads", "head_dim",
        "mlp_dim", "mlp_kind", "horizon", "action_dim", "state_tokens", "time_dim", "time_mlp",
        "direction", "max_batch", "max_prefix", "max_steps")] + [
        ("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float), ("weight_format", ctypes.c_int32),
        ("context_dim", ctypes.c_int32), ("state_dim", ctypes.c_int32)]


_VP = ctypes.c_void_p
_VPP = ctypes.POINTER(ctypes.c_void_p)


class Weights(ctypes.Structure):
    _fields_ = [("location", ctypes.c_int32)] + [(n, _VP) for n in (
        "time_mlp_in_w", "time_mlp_in_b", "time_mlp_out_w", "time_mlp_out_b", "cond_w", "cond_b",
        "action_in_w", "action_in_b", "enc_w1", "enc_b1", "enc_w2", "enc_b2", "enc_w3", "enc_b3",
        "action_out_w", "action_out_b")] + [(n, _VPP) for n in (
        "qkv_w", "o_w", "up_w", "down_w", "qkv_s", "o_s", "up_s", "down_s", "cross_k_w", "cross_v_w")] + [
        (n, _VP) for n in ("state_w1", "state_b1", "state_w2", "state_b2")]


# exported symbol -> (restype, argtypes)
SIGNATURES = {
    "gr00t_validate_geometry": (ctypes.c_int, [ctypes.POINTER(Geometry), ctypes.c_char_p, ctypes.c_size_t]),
    "gr00t_create": (ctypes.c_int, [ctypes.POINTER(Geometry), ctypes.POINTER(Weights), _VP,
                                    ctypes.POINTER(_VP)]),
    "gr00t_bind_prefix_kv": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, _VPP, _VPP, _VP, _VP, _VP]),
    "gr00t_bind_context": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, _VP, _VP, _VP, _VP]),
    "gr00t_bind_kv_pool": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, ctypes.c_int, _VPP]),
    "gr00t_set_schedule": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int]),
    "gr00t_denoise": (ctypes.c_int, [_VP, _VP, _VP]),
    "gr00t_denoise_host": (ctypes.c_int, [_VP, _VP, _VP]),
    "gr00t_denoise_step": (ctypes.c_int, [_VP, ctypes.c_int, _VP, _VP]),
    "gr00t_denoise_step_noalloc": (ctypes.c_int, [_VP, ctypes.c_int, _VP, _VP]),
    "gr00t_destroy": (ctypes.c_int, [_VP]),
    "gr00t_last_error": (ctypes.c_char_p, [_VP]),
    "gr00t_set_option": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int64]),
    "gr00t_get_info": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]),
    "gr00t_kernel_times": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int),
                                          ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
    "gr00t_sync": (ctypes.c_int, [_VP]),
    "gr00t_debug_dump": (ctypes.c_int, [_VP, ctypes.c_int, _VP, ctypes.c_int, _VP]),
    "gr00t_debug_cond_step": (ctypes.c_int, [_VP, ctypes.c_int, _VP, _VP]),
}

_lib = None


def header_functions(path: str = HEADER) -> list[str]:
    """Names of the functions ``include/gr00t.h`` declares."""
    text = open(path).read()
    return sorted(set(re.findall(r"\b(gr00t_[a-z_]+)\s*\(", text)))


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libgr00t.so (built by ``flow_matching_vla_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build it with `python -m flow_matching_vla_gb300.build` "
            "(the denoise loop has no CPU fallback)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib
