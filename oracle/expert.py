"""pi0.5-style action expert: one velocity evaluation and the denoise loop.

Test infrastructure (see ``oracle/__init__.py``).  Per sample, per layer,
per head, in the order the pages give; no head fold, no blocking.
"""
from __future__ import annotations

import numpy as np

from .ops import dequantize_rows, attention, gelu_tanh, rms_norm, rope_rotate_half
from .schedule import euler, modulation_table


def _w(w, name, dtype):
    """Weight ``name`` as a real matrix: FP8 weights (codes with a ``.scale``
    entry per output row) are dequantized, the rest are taken as stored."""
    if name + ".scale" in w:
        return dequantize_rows(w[name], w[name + ".scale"]).astype(dtype, copy=False)
    return w[name].astype(dtype, copy=False)


def ada_rms(h, row, eps):
    """AdaRMS (reading S1 of "pi0.5 Design", Component contract, adarms_modulation).

    The row packs (scale, shift, gate) along its last axis;
    y = rms_norm(h) * (1 + scale) + shift.  Returns (y, gate).
    """
    D = h.shape[-1]
    scale, shift, gate = row[:D], row[D:2 * D], row[2 * D:3 * D]
    return rms_norm(h, eps) * (1.0 + scale) + shift, gate


def expert_velocity(g, w, x, mod_k, K, V, dtype=np.float64, trace=None):
    """Velocity v_theta(x_t, tau_k, C) of the action expert ("pi0.5 Design").

    ``x``: [B, H, A]; ``mod_k``: [B, 2L+1, 3D] (this step's modulation rows,
    one per request); ``K``/``V``: per layer [B, P, 1, Dh] prefix K/V, bound
    once per request and reused by every step ("pi0.5 Design", sequence diagram).

    Per layer l (rows of the hoisted table per the Component contract):
      n  = AdaRMS(h, row 2l)                         input_layernorm
      q, k_s, v_s = n W_qkv^T                        single KV head
      q, k_s rotated at positions P + j               (reading S7)
      o  = softmax(q [K_pre; k_s]^T / sqrt(Dh)) [V_pre; v_s]   per head,
           attending over prefix ++ own K/V ("Attention and the K/V pool";
           vla.cpp Eq. (2))
      h += gate_a * (o W_o^T)                        gated residual (S1)
      n2 = AdaRMS(h, row 2l+1)                       post_attention_layernorm
      u  = gelu(n2 W_gate^T) * (n2 W_up^T)  (GeGLU) or gelu(n2 W_up^T) (GeLU)
      h += gate_m * (u W_down^T)
    then v = AdaRMS(h, row 2L) W_out^T + b_out (the last row is the final
    norm; its gate is unused), with h = x W_in^T + b_in at the start
    ("pi0.5 Design": velocity through action_out_proj).
    """
    B, H, A = x.shape
    D, L, Hq, Dh = g["hidden"], g["layers"], g["q_heads"], g["head_dim"]
    eps, theta = g["norm_eps"], g["rope_theta"]
    F = g["mlp_dim"]
    assert g["kv_heads"] == 1, "the expert attends over a single shared KV head"
    P = K[0].shape[1] if L > 0 else 0
    pos = P + np.arange(H)
    x = x.astype(dtype, copy=False)
    v_out = np.empty((B, H, A), dtype=dtype)
    for b in range(B):
        h = x[b] @ _w(w, "action_in_w", dtype).T + _w(w, "action_in_b", dtype)
        if trace is not None:
            trace.setdefault("h_in", []).append(h.copy())
        for l in range(L):
            n, gate_a = ada_rms(h, mod_k[b, 2 * l].astype(dtype), eps)
            qkv = n @ _w(w, f"qkv_w.{l}", dtype).T
            q = qkv[:, :Hq * Dh].reshape(H, Hq, Dh)
            k_s = rope_rotate_half(qkv[:, Hq * Dh:Hq * Dh + Dh], pos, theta)
            v_s = qkv[:, Hq * Dh + Dh:Hq * Dh + 2 * Dh]
            keys = np.concatenate([K[l][b, :, 0, :].astype(dtype), k_s], axis=0)
            vals = np.concatenate([V[l][b, :, 0, :].astype(dtype), v_s], axis=0)
            o = np.empty((H, Hq * Dh), dtype=dtype)
            for hd in range(Hq):
                q_h = rope_rotate_half(q[:, hd, :], pos, theta)
                o[:, hd * Dh:(hd + 1) * Dh] = attention(q_h, keys, vals)
            h = h + gate_a * (o @ _w(w, f"o_w.{l}", dtype).T)
            n2, gate_m = ada_rms(h, mod_k[b, 2 * l + 1].astype(dtype), eps)
            up = n2 @ _w(w, f"up_w.{l}", dtype).T
            if up.shape[-1] == 2 * F:   # GeGLU: rows [0, F) gate, [F, 2F) up (reading S6)
                u = gelu_tanh(up[:, :F]) * up[:, F:]
            else:
                u = gelu_tanh(up)
            h = h + gate_m * (u @ _w(w, f"down_w.{l}", dtype).T)
            if trace is not None:
                trace.setdefault(f"h.{l}", []).append(h.copy())
        n, _ = ada_rms(h, mod_k[b, 2 * L].astype(dtype), eps)
        v_out[b] = n @ _w(w, "action_out_w", dtype).T + _w(w, "action_out_b", dtype)
    return v_out


def expert_denoise(g, w, x_noise, K, V, steps, dtype=np.float64, record=False):
    """Flow-matching Euler loop, vla.cpp Eq. (1), over the expert velocity.

    X^{k+1} = X^k + (tau_{k+1} - tau_k) v(X^k, tau_k), k = 0..T-1, with the
    modulation table hoisted once for (steps, batch) ("pi0.5 Design": cond
    re-runs only when the step count or batch changes).
    """
    B = x_noise.shape[0]
    mod = modulation_table(g, w, steps, B, dtype)
    x, vs = euler(x_noise.astype(dtype),
                  lambda x, k, tau: expert_velocity(g, w, x, mod[k * B:(k + 1) * B], K, V, dtype),
                  g["direction"], steps, record)
    return (x, vs) if record else x
