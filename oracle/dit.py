"""GR00T-style DiT action head: one velocity evaluation and the denoise loop.

Test infrastructure (see ``oracle/__init__.py``).  Per sample, per block,
per head; no blocking.
"""
from __future__ import annotations

import numpy as np

from .ops import dequantize_rows, attention, gelu_tanh, layer_norm, swish
from .schedule import euler, modulation_table, schedule, time_embedding


def _w(w, name, dtype):
    """Weight ``name`` as a real matrix: FP8 weights (codes with a ``.scale``
    entry per output row) are dequantized, the rest are taken as stored."""
    if name + ".scale" in w:
        return dequantize_rows(w[name], w[name + ".scale"]).astype(dtype, copy=False)
    return w[name].astype(dtype, copy=False)


def project_context(g, w, features, dtype=np.float64):
    """Cross-attention K/V of every even (cross) block from the VL features
    ("GR00T N1.7", vl_backbone: the VL engine ends with the DiT's cross-attention
    K/V projections, cross_k / cross_v [B, S, 32, 48] for even blocks only).

    ``features``: [B, S, context_dim].  K_i = features W_k,i^T and V_i = features
    W_v,i^T, no bias (reading S11), reshaped to [B, S, kv_heads, head_dim];
    odd blocks get None.  Returns (K, V) lists indexed by block.
    """
    B, S, _ = features.shape
    Hkv, Dh = g["kv_heads"], g["head_dim"]
    f = features.astype(dtype, copy=False)
    K, V = [None] * g["layers"], [None] * g["layers"]
    for l in range(0, g["layers"], 2):
        K[l] = (f @ _w(w, f"cross_k_w.{l}", dtype).T).reshape(B, S, Hkv, Dh)
        V[l] = (f @ _w(w, f"cross_v_w.{l}", dtype).T).reshape(B, S, Hkv, Dh)
    return K, V


def encode_state(g, w, state_raw, dtype=np.float64):
    """Robot-state token(s) from the raw state ("GR00T N1.7", action: the action
    component takes the robot state [B, 1, state_dim] beside the noisy actions,
    and the checkpoint's state encoder is one of the per-embodiment modules
    resolved at build time).  The page names the module, not its layers; the
    reading taken here (S18) is a two-layer MLP in the style of the action
    encoder: s_tok = W_s2 swish(W_s1 s + b_s1) + b_s2, hidden width D.  The state
    does not change across the denoise steps of a request, so it is embedded
    once, when the request's inputs are bound.

    ``state_raw``: [B, Ns, state_dim]; returns [B, Ns, D].
    """
    s = state_raw.astype(dtype, copy=False)
    hid = swish(s @ _w(w, "state_w1", dtype).T + _w(w, "state_b1", dtype))
    return hid @ _w(w, "state_w2", dtype).T + _w(w, "state_b2", dtype)


def action_time_bias(g, w, steps, dtype=np.float64):
    """Hoisted action_time_bias [steps, D] ("GR00T N1.7", Build-time constants).

    The page moves the part of the encoder's second projection that only
    sees the time embedding out of the step.  W2 acts on concat(W1 x + b1,
    temb(tau)); its time columns applied to the sinusoid of tau_k, plus W2's
    bias, form the bias row of step k: atb_k = W2[:, D:] temb(tau_k) + b2
    (reading S3 for temb).
    """
    D = g["hidden"]
    taus, _ = schedule(g["direction"], steps)
    w2t = _w(w, "enc_w2", dtype)[:, D:]
    out = np.empty((steps, D), dtype=dtype)
    for k in range(steps):
        out[k] = w2t @ time_embedding(taus[k], g["time_dim"]).astype(dtype) + _w(w, "enc_b2", dtype)
    return out


def dit_velocity(g, w, x, mod_k, atb_k, K, V, text_mask, image_mask, state, dtype=np.float64, trace=None):
    """Velocity of the DiT head ("GR00T N1.7", action component).

    ``x``: [B, H, A]; ``mod_k``: [B, L+1, 2D]; ``atb_k``: [D]; ``K``/``V``:
    per even block [B, S, Hkv, Dh] projected VL-context K/V, bound once;
    masks: uint8 [B, S] (1 = visible) or None; ``state``: [B, Ns, D].

      action encoder: e = swish((x W1^T + b1) W2[:, :D]^T + atb_k);
                      tok = e W3^T + b3
      h = [state ; tok]
      block i:  n = LN(h) (1 + scale_i) + shift_i, row i split (scale, shift)
                even i: cross-attention of n W_q^T over (K_i, V_i), mask =
                        text if i % 4 == 0 else image
                odd i:  self-attention, q/k/v = n W_qkv^T over the Ns+H tokens
                h += o W_o^T
                h += gelu(LN(h) W_1^T) W_2^T     (reading S9: plain FF)
      final:    n = LN(h) (1 + scale) + shift, row L split (shift, scale)
                v = n[Ns:] W_out^T + b_out

    ``trace`` (a dict, optional) receives per sample the residual stream after
    the encoder ("h_in") and after every block i ("h.<i>"), [Ns + H, D] each.
    """
    B, H, A = x.shape
    D, L, Hq, Dh = g["hidden"], g["layers"], g["q_heads"], g["head_dim"]
    eps = g["norm_eps"]
    Ns = g["state_tokens"]
    x = x.astype(dtype, copy=False)
    v_out = np.empty((B, H, A), dtype=dtype)
    w2a = _w(w, "enc_w2", dtype)[:, :D]
    for b in range(B):
        a = x[b] @ _w(w, "enc_w1", dtype).T + _w(w, "enc_b1", dtype)
        e = swish(a @ w2a.T + atb_k)
        tok = e @ _w(w, "enc_w3", dtype).T + _w(w, "enc_b3", dtype)
        h = np.concatenate([state[b].astype(dtype), tok], axis=0) if Ns else tok
        T = h.shape[0]
        if trace is not None:
            trace.setdefault("h_in", []).append(h.copy())
        for i in range(L):
            row = mod_k[b, i].astype(dtype)
            scale, shift = row[:D], row[D:2 * D]
            n = layer_norm(h, eps) * (1.0 + scale) + shift
            o = np.empty((T, Hq * Dh), dtype=dtype)
            if i % 2 == 0:
                q = (n @ _w(w, f"qkv_w.{i}", dtype).T).reshape(T, Hq, Dh)
                m = text_mask if i % 4 == 0 else image_mask
                vis = None if m is None else m[b].astype(bool)
                for hd in range(Hq):
                    o[:, hd * Dh:(hd + 1) * Dh] = attention(
                        q[:, hd], K[i][b, :, hd].astype(dtype), V[i][b, :, hd].astype(dtype), vis)
            else:
                qkv = n @ _w(w, f"qkv_w.{i}", dtype).T
                q = qkv[:, :Hq * Dh].reshape(T, Hq, Dh)
                k = qkv[:, Hq * Dh:2 * Hq * Dh].reshape(T, Hq, Dh)
                v = qkv[:, 2 * Hq * Dh:3 * Hq * Dh].reshape(T, Hq, Dh)
                for hd in range(Hq):
                    o[:, hd * Dh:(hd + 1) * Dh] = attention(q[:, hd], k[:, hd], v[:, hd])
            h = h + o @ _w(w, f"o_w.{i}", dtype).T
            f = gelu_tanh(layer_norm(h, eps) @ _w(w, f"up_w.{i}", dtype).T)
            h = h + f @ _w(w, f"down_w.{i}", dtype).T
            if trace is not None:
                trace.setdefault(f"h.{i}", []).append(h.copy())
        row = mod_k[b, L].astype(dtype)
        shift, scale = row[:D], row[D:2 * D]
        n = layer_norm(h, eps) * (1.0 + scale) + shift
        v_out[b] = n[Ns:] @ _w(w, "action_out_w", dtype).T + _w(w, "action_out_b", dtype)
    return v_out


def dit_denoise(g, w, x_noise, K, V, steps, text_mask=None, image_mask=None, state=None,
                dtype=np.float64, record=False):
    """Euler loop of vla.cpp Eq. (1) over the DiT velocity, tables hoisted once."""
    B = x_noise.shape[0]
    mod = modulation_table(g, w, steps, B, dtype)
    atb = action_time_bias(g, w, steps, dtype)
    x, vs = euler(x_noise.astype(dtype),
                  lambda x, k, tau: dit_velocity(g, w, x, mod[k * B:(k + 1) * B], atb[k], K, V,
                                                 text_mask, image_mask, state, dtype),
                  g["direction"], steps, record)
    return (x, vs) if record else x
