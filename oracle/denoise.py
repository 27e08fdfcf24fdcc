"""Family-independent entry points: Euler integration and one velocity step.

Test infrastructure (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import numpy as np

from .dit import action_time_bias, dit_denoise, dit_velocity, encode_state, project_context
from .expert import expert_denoise, expert_velocity
from .schedule import euler, modulation_table

FAMILY_EXPERT = 0


def _kv(case, dtype):
    """The case's bound K/V, or (DiT with VL features) their cross projections."""
    if case.get("features") is not None:
        return project_context(case["geom"], case["weights"], case["features"], dtype)
    return case["K"], case["V"]


def _state(case, dtype):
    """The case's state tokens, or (DiT with a raw robot state) their encoding."""
    if case.get("state_raw") is not None:
        return encode_state(case["geom"], case["weights"], case["state_raw"], dtype)
    return case["state"]


def denoise(case, steps=None, dtype=np.float64, record=False):
    """Full denoise loop for a ``synth.make_case`` dictionary."""
    g, w = case["geom"], case["weights"]
    T = g["steps"] if steps is None else steps
    if g["family"] == FAMILY_EXPERT:
        return expert_denoise(g, w, case["x_noise"], case["K"], case["V"], T, dtype, record)
    K, V = _kv(case, dtype)
    return dit_denoise(g, w, case["x_noise"], K, V, T, case["text_mask"],
                       case["image_mask"], _state(case, dtype), dtype, record)


def velocity(case, x, k, steps=None, dtype=np.float64, mod=None, atb=None):
    """Velocity at step k of a T-step schedule from the state ``x`` (teacher forcing)."""
    g, w = case["geom"], case["weights"]
    T = g["steps"] if steps is None else steps
    B = x.shape[0]
    if mod is None:
        mod = modulation_table(g, w, T, B, dtype)
    rows = mod[k * B:(k + 1) * B]
    if g["family"] == FAMILY_EXPERT:
        return expert_velocity(g, w, x, rows, case["K"], case["V"], dtype)
    if atb is None:
        atb = action_time_bias(g, w, T, dtype)
    K, V = _kv(case, dtype)
    return dit_velocity(g, w, x, rows, atb[k], K, V, case["text_mask"],
                        case["image_mask"], _state(case, dtype), dtype)
