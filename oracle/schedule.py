"""Integration schedule, time embedding and the hoisted modulation table.

Test infrastructure (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import numpy as np

from .ops import swish

FAMILY_EXPERT = 0


def schedule(direction, steps):
    """Uniform integration grid tau_0..tau_T and the step sizes of Eq. (1).

    vla.cpp section III-A: pi0 / SmolVLA integrate 1 -> 0, GR00T-N1.7 0 -> 1.
    Reading S5: the grid is uniform, tau_k = 1 - k/T (direction -1) or
    tau_k = k/T (direction +1); dt_k = tau_{k+1} - tau_k.
    """
    k = np.arange(steps + 1, dtype=np.float64)
    taus = (1.0 - k / steps) if direction < 0 else (k / steps)
    return taus, taus[1:] - taus[:-1]


def euler(x0, velocity_fn, direction, steps, record=False):
    """Flow-matching Euler integration, vla.cpp Eq. (1).

    X^{k+1} = X^k + (tau_{k+1} - tau_k) v(X^k, tau_k), k = 0..T-1, on the
    uniform grid of ``schedule``; ``velocity_fn(x, k, tau_k)`` returns v.
    Returns X^T and, with ``record``, the list of velocities.
    """
    taus, dts = schedule(direction, steps)
    x = np.asarray(x0)
    vs = []
    for k in range(steps):
        v = velocity_fn(x, k, taus[k])
        if record:
            vs.append(v)
        x = x + x.dtype.type(dts[k]) * v
    return x, vs


def time_embedding(tau, dim, min_period=4e-3, max_period=4.0):
    """Sinusoidal embedding of the flow time tau (reading S3).

    For i < dim/2: sin(tau * w_i); for i >= dim/2: cos(tau * w_{i-dim/2}),
    with w_i = 2 pi / period_i and period_i geometric from min_period
    (i = 0) to max_period (i = dim/2 - 1).
    """
    half = dim // 2
    frac = np.arange(half, dtype=np.float64) / (half - 1)
    period = min_period * (max_period / min_period) ** frac
    ang = float(tau) * (2.0 * np.pi / period)
    return np.concatenate([np.sin(ang), np.cos(ang)])


def time_condition(g, w, tau, dtype=np.float64):
    """Conditioning vector c(tau) fed to the adaptive-norm Denses.

    "pi0.5 Design", Checkpoint: pi0.5 carries time_mlp_in / time_mlp_out.
    Reading S4: c = swish(W_out swish(W_in temb + b_in) + b_out) when the
    geometry has a time MLP, else c = temb (the tiny workload: a Dense of the
    sinusoid directly).
    """
    t = time_embedding(tau, g["time_dim"]).astype(dtype)
    if not g["time_mlp"]:
        return t
    a = swish(w["time_mlp_in_w"].astype(dtype) @ t + w["time_mlp_in_b"].astype(dtype))
    return swish(w["time_mlp_out_w"].astype(dtype) @ a + w["time_mlp_out_b"].astype(dtype))


def modulation_row(g, w, tau, site, dtype=np.float64):
    """One adaptive-norm Dense evaluated at tau: W_site c(tau) + b_site."""
    c = time_condition(g, w, tau, dtype)
    return w["cond_w"][site].astype(dtype) @ c + w["cond_b"][site].astype(dtype)


def modulation_table(g, w, steps, batch, dtype=np.float64):
    """The hoisted table [steps * batch, sites, row], rows ordered [step][request].

    "pi0.5 Design", Component contract (adarms_modulation): rows are
    [step][request]; within an entry, row 2i is layer i's input_layernorm,
    2i+1 its post_attention_layernorm, the last the final norm; the last axis
    packs (scale, shift, gate).  "GR00T N1.7", Build-time constants: [steps,
    33, 3072], row i = block i's norm1, last row proj_out_1; the raw
    projection is stored and the consumer owns the split.  The GR00T table
    has no batch axis; here both families carry one so the layout is uniform
    (reading S14).  Every (step, request) entry is the same Dense evaluated at
    tau_k, exactly what per-step evaluation would give.
    """
    taus, _ = schedule(g["direction"], steps)
    S = w["cond_w"].shape[0]
    R = w["cond_w"].shape[1]
    out = np.empty((steps * batch, S, R), dtype=dtype)
    for k in range(steps):
        c = time_condition(g, w, taus[k], dtype)
        for s in range(S):
            row = w["cond_w"][s].astype(dtype) @ c + w["cond_b"][s].astype(dtype)
            for b in range(batch):
                out[k * batch + b, s] = row
    return out
