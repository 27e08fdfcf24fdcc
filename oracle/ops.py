"""Elementary operations of the denoise step, written out from their definitions.

Test infrastructure (see ``oracle/__init__.py``).  Plain numpy, no blocking or
fusion: each function is the textbook formula.
"""
from __future__ import annotations

import numpy as np


def swish(x):
    """swish(x) = x * sigmoid(x) (a.k.a. SiLU)."""
    return x / (1.0 + np.exp(-x))


def gelu_tanh(x):
    """GeLU, tanh approximation (reading S6: the pages do not name the variant).

    gelu(x) = 0.5 x (1 + tanh( sqrt(2/pi) (x + 0.044715 x^3) )).
    """
    c = float(np.sqrt(2.0 / np.pi))
    return 0.5 * x * (1.0 + np.tanh(c * (x + 0.044715 * x * x * x)))


def rms_norm(h, eps):
    """RMSNorm without a learned weight: h / sqrt(mean(h^2) + eps) over the last axis.

    The fp32-reduction RMSNorm of "Optimizing GR00T-N1.7 Training" section 3.3;
    AdaRMS (reading S1) scales and shifts this result.
    """
    ms = np.mean(h * h, axis=-1, keepdims=True)
    return h / np.sqrt(ms + eps)


def layer_norm(h, eps):
    """Non-affine LayerNorm over the last axis: (h - mean) / sqrt(var + eps)."""
    mu = np.mean(h, axis=-1, keepdims=True)
    d = h - mu
    var = np.mean(d * d, axis=-1, keepdims=True)
    return d / np.sqrt(var + eps)


def rope_rotate_half(x, positions, theta):
    """Rotary position embedding, rotate-half convention.

    "Optimizing GR00T-N1.7 Training", section 3.3: x * cos + rotate_half(x) * sin
    with rotate_half(x) = concat(-x[d/2:], x[:d/2]).  Frequency of pair i is
    theta^(-2i/d) (reading S7).  ``x``: [..., T, d]; ``positions``: [T].
    """
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]   # [T, d/2]
    cos = np.concatenate([np.cos(ang), np.cos(ang)], axis=-1).astype(x.dtype)
    sin = np.concatenate([np.sin(ang), np.sin(ang)], axis=-1).astype(x.dtype)
    rot = np.concatenate([-x[..., half:], x[..., :half]], axis=-1)
    return x * cos + rot * sin


def attention(q, k, v, visible=None):
    """One attention head, vla.cpp Eq. (2): softmax(Q K^T / sqrt(d_k) + M) V.

    ``q``: [Tq, d], ``k``/``v``: [Tk, d], ``visible``: optional bool [Tk]
    (M = 0 where visible, -inf elsewhere).  Softmax is over keys, computed with
    the row maximum subtracted.  A row whose keys are all masked returns zeros
    (reading S8: Eq. (2) is undefined there).
    """
    d = q.shape[-1]
    s = (q @ k.T) * q.dtype.type(1.0 / np.sqrt(d))
    if visible is not None:
        if not np.any(visible):
            return np.zeros((q.shape[0], v.shape[-1]), dtype=q.dtype)
        s = np.where(np.asarray(visible, bool)[None, :], s, -np.inf)
    s = s - np.max(s, axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / np.sum(p, axis=-1, keepdims=True)
    return p @ v


def error_metrics(a, a_ref):
    """vla.cpp Eq. (5): e_inf = max|A - A_ref|, e_rel = ||A - A_ref||_2 / ||A_ref||_2.

    When ||A_ref|| = 0 the relative error is undefined and the absolute
    2-norm of the difference is returned in its place, as the page prescribes.
    """
    a = np.asarray(a, np.float64).ravel()
    r = np.asarray(a_ref, np.float64).ravel()
    diff = a - r
    e_inf = float(np.max(np.abs(diff))) if diff.size else 0.0
    nr = float(np.linalg.norm(r))
    e_rel = float(np.linalg.norm(diff)) / nr if nr > 0 else float(np.linalg.norm(diff))
    return e_inf, e_rel


def e4m3_decode(codes):
    """Values of 8-bit E4M3 floating-point codes (the OCP 8-bit floating point
    format that FP8 weight streaming uses, "pi0.5 Design", precision notes).

    Bit 7 is the sign, bits 6..3 the exponent field e (bias 7), bits 2..0 the
    mantissa field m.  e = 0: subnormal, (m / 8) * 2^-6.  e >= 1: (1 + m / 8) *
    2^(e - 7).  The format has no infinities: e = 15 with m = 7 is NaN, so the
    largest finite magnitude is (1 + 6/8) * 2^8 = 448.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((c & 0x7) == 7), np.nan, mag)
    return sign * mag


def dequantize_rows(codes, scales):
    """W[n, k] = e4m3(codes[n, k]) * scales[n]: row-scaled FP8 weights ([out, in]
    codes, one scale per output row) as the real matrix they stand for."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, None]
