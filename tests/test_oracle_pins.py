"""Pins for the CPU oracle: closed forms, invariants, library routines, brute force.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
swapped split, a wrong sign or index, a transposed operand) fails it.  None
of them compares the oracle with itself.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle.dit import dit_velocity
from oracle.expert import ada_rms, expert_velocity

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def t64(a):
    return torch.from_numpy(np.asarray(a, np.float64))


# ---------------------------------------------------------------------------
# elementwise and normalisation ops vs torch library routines
# ---------------------------------------------------------------------------

def test_swish_and_gelu_match_torch():
    x = rng.standard_normal(1000) * 4
    np.testing.assert_allclose(oracle.swish(x), F.silu(t64(x)).numpy(), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(oracle.gelu_tanh(x), F.gelu(t64(x), approximate="tanh").numpy(),
                               rtol=1e-14, atol=1e-15)


def test_rms_norm_matches_torch():
    h = rng.standard_normal((7, 96)) * 3
    ref = F.rms_norm(t64(h), (96,), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(h, 1e-6), ref, rtol=1e-13, atol=1e-14)


def test_layer_norm_matches_torch():
    h = rng.standard_normal((7, 96)) * 3 + 1.5
    ref = F.layer_norm(t64(h), (96,), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.layer_norm(h, 1e-6), ref, rtol=1e-12, atol=1e-13)


def test_ada_rms_packing_scale_shift_gate():
    # scale = -1 collapses the normalised value: the output is exactly the shift
    D = 32
    h = rng.standard_normal((5, D))
    shift = rng.standard_normal(D)
    gate = rng.standard_normal(D)
    row = np.concatenate([-np.ones(D), shift, gate])
    y, g = ada_rms(h, row, 1e-6)
    np.testing.assert_array_equal(y, np.broadcast_to(shift, y.shape))
    np.testing.assert_array_equal(g, gate)
    # scale = shift = 0 is the plain RMSNorm
    y0, _ = ada_rms(h, np.concatenate([np.zeros(2 * D), gate]), 1e-6)
    np.testing.assert_allclose(y0, F.rms_norm(t64(h), (D,), eps=1e-6).numpy(), rtol=1e-13)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def test_rope_equals_complex_rotation():
    # rotate-half RoPE is multiplication of z_i = x_i + i x_{i+d/2} by exp(i pos w_i)
    d, T = 64, 9
    x = rng.standard_normal((T, d))
    pos = rng.integers(0, 5000, T)
    z = x[:, :d // 2] + 1j * x[:, d // 2:]
    w = 10000.0 ** (-np.arange(d // 2) * 2.0 / d)
    zr = z * np.exp(1j * pos[:, None] * w[None, :])
    ref = np.concatenate([zr.real, zr.imag], axis=-1)
    np.testing.assert_allclose(oracle.rope_rotate_half(x, pos, 10000.0), ref, rtol=1e-12, atol=1e-12)


def test_rope_identity_at_zero_and_relative_position():
    d = 32
    x = rng.standard_normal((4, d))
    np.testing.assert_array_equal(oracle.rope_rotate_half(x, np.zeros(4), 10000.0), x)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    def dot(m, n):
        return float(oracle.rope_rotate_half(q[None], [m], 1e4)[0] @ oracle.rope_rotate_half(k[None], [n], 1e4)[0])
    assert abs(dot(3, 11) - dot(103, 111)) < 1e-10
    assert abs(dot(3, 11) - dot(11, 3)) > 1e-6   # not symmetric: the sign of m - n matters


# ---------------------------------------------------------------------------
# attention, Eq. (2)
# ---------------------------------------------------------------------------

def test_attention_matches_torch_sdpa():
    q = rng.standard_normal((6, 48))
    k = rng.standard_normal((30, 48))
    v = rng.standard_normal((30, 48))
    ref = F.scaled_dot_product_attention(t64(q)[None], t64(k)[None], t64(v)[None])[0].numpy()
    np.testing.assert_allclose(oracle.attention(q, k, v), ref, rtol=1e-12, atol=1e-13)
    vis = rng.random(30) < 0.5
    vis[3] = True
    ref = F.scaled_dot_product_attention(t64(q)[None], t64(k)[None], t64(v)[None],
                                         attn_mask=torch.from_numpy(vis)[None, None, :])[0].numpy()
    np.testing.assert_allclose(oracle.attention(q, k, v, vis), ref, rtol=1e-12, atol=1e-13)


def test_attention_bruteforce_scalar_loops():
    q = rng.standard_normal((2, 3))
    k = rng.standard_normal((4, 3))
    v = rng.standard_normal((4, 2))
    out = np.zeros((2, 2))
    for i in range(2):
        s = [sum(q[i, c] * k[j, c] for c in range(3)) / math.sqrt(3) for j in range(4)]
        e = [math.exp(x) for x in s]
        z = sum(e)
        for c in range(2):
            out[i, c] = sum(e[j] / z * v[j, c] for j in range(4))
    np.testing.assert_allclose(oracle.attention(q, k, v), out, rtol=1e-13)


def test_attention_special_cases():
    v = rng.standard_normal((1, 16))
    q = rng.standard_normal((3, 16)) * 10
    k = rng.standard_normal((1, 16))
    # one key: the softmax of a single score is 1, the output is that value row
    np.testing.assert_allclose(oracle.attention(q, k, v), np.repeat(v, 3, 0), rtol=1e-15)
    # all keys equal: uniform weights, the output is the mean of V
    V = rng.standard_normal((7, 16))
    K = np.repeat(k, 7, 0)
    np.testing.assert_allclose(oracle.attention(q, K, V), np.repeat(V.mean(0, keepdims=True), 3, 0),
                               rtol=1e-12, atol=1e-14)
    # masked keys do not contribute
    Kr = rng.standard_normal((7, 16))
    vis = np.array([1, 0, 1, 1, 0, 0, 1], bool)
    np.testing.assert_allclose(oracle.attention(q, Kr, V, vis), oracle.attention(q, Kr[vis], V[vis]),
                               rtol=1e-13)
    # every key masked: zeros (reading S8), no NaN
    assert np.all(oracle.attention(q, Kr, V, np.zeros(7, bool)) == 0)


def test_error_metrics_closed_form():
    e_inf, e_rel = oracle.error_metrics([1.0, 2.0], [1.0, 1.0])
    assert e_inf == 1.0 and abs(e_rel - 1 / math.sqrt(2)) < 1e-15
    e_inf, e_rel = oracle.error_metrics([3.0, 4.0], [0.0, 0.0])
    assert e_inf == 4.0 and e_rel == 5.0   # zero reference: absolute error, Eq. (5)


# ---------------------------------------------------------------------------
# schedule, time embedding, hoist
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 2, 3, 4, 8, 10])
def test_schedule_endpoints(T):
    taus, dts = oracle.schedule(-1, T)
    assert taus[0] == 1.0 and taus[-1] == 0.0 and len(dts) == T
    assert abs(dts.sum() + 1.0) < 1e-15 and np.all(dts < 0)
    taus2, dts2 = oracle.schedule(+1, T)
    assert taus2[0] == 0.0 and taus2[-1] == 1.0 and np.all(dts2 > 0)


def test_time_embedding_closed_form():
    E = 64
    t0 = oracle.time_embedding(0.0, E)
    np.testing.assert_array_equal(t0, np.concatenate([np.zeros(32), np.ones(32)]))
    # the slowest frequency has period max_period = 4: at tau = 1 its angle is pi/2
    t1 = oracle.time_embedding(1.0, E)
    assert abs(t1[31] - 1.0) < 1e-15 and abs(t1[63]) < 1e-15
    # the fastest has period min_period = 4e-3: angle 2 pi tau / 4e-3
    assert abs(t1[0] - math.sin(2 * math.pi / 4e-3)) < 1e-12
    tx = oracle.time_embedding(0.37, E)
    np.testing.assert_allclose(tx[:32] ** 2 + tx[32:] ** 2, 1.0, rtol=1e-15)


@pytest.mark.parametrize("name", ["small_bf16", "small_dit"])
def test_hoisted_table_equals_per_step_evaluation(name):
    c = synth.make_case(name)
    g, w = c["geom"], c["weights"]
    T, B = 3, 2
    tab = oracle.modulation_table(g, w, T, B)
    taus, _ = oracle.schedule(g["direction"], T)
    from oracle.schedule import modulation_row
    for k, b, s in itertools.product(range(T), range(B), range(synth.norm_sites(g))):
        np.testing.assert_array_equal(tab[k * B + b, s], modulation_row(g, w, taus[k], s))
    # time MLP: c = swish(W_out swish(W_in temb + b_in) + b_out), checked through torch
    temb = t64(oracle.time_embedding(taus[1], g["time_dim"]))
    c1 = F.silu(F.linear(F.silu(F.linear(temb, t64(w["time_mlp_in_w"]), t64(w["time_mlp_in_b"]))),
                         t64(w["time_mlp_out_w"]), t64(w["time_mlp_out_b"])))
    ref = F.linear(c1, t64(w["cond_w"][2]), t64(w["cond_b"][2])).numpy()
    np.testing.assert_allclose(tab[1 * B, 2], ref, rtol=1e-12, atol=1e-14)


def test_action_time_bias_is_time_half_of_w2():
    # the hoisted bias is W2's time columns applied to the sinusoid, plus W2's bias
    c = synth.make_case("small_dit")
    g, w = c["geom"], c["weights"]
    D = g["hidden"]
    T = 4
    atb = oracle.action_time_bias(g, w, T)
    taus, _ = oracle.schedule(g["direction"], T)
    a = rng.standard_normal((5, D))
    for k in range(T):
        cat = np.concatenate([a, np.repeat(oracle.time_embedding(taus[k], g["time_dim"])[None], 5, 0)], 1)
        full = F.linear(t64(cat), t64(w["enc_w2"]), t64(w["enc_b2"])).numpy()
        np.testing.assert_allclose(a @ w["enc_w2"][:, :D].astype(np.float64).T + atb[k], full,
                                   rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Euler integration, Eq. (1)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 2, 4, 8])
@pytest.mark.parametrize("direction", [-1, +1])
def test_euler_constant_velocity_is_exact(T, direction):
    x0 = rng.integers(-64, 64, (3, 5)) / 8.0
    c = rng.integers(-64, 64, (3, 5)) / 16.0
    xT, _ = oracle.euler(x0, lambda x, k, tau: c, direction, T)
    np.testing.assert_array_equal(xT, x0 + direction * c)


def test_euler_linear_field_closed_form():
    # v = a x: each step multiplies by (1 + a dt); uses X^k, not X^{k+1}
    x0 = rng.standard_normal(6)
    a, T = 0.7, 5
    xT, _ = oracle.euler(x0, lambda x, k, tau: a * x, -1, T)
    np.testing.assert_allclose(xT, x0 * (1 - a / T) ** T, rtol=1e-14)
    # tau enters as tau_k: v = tau gives sum_k tau_k dt_k
    xT, _ = oracle.euler(np.zeros(1), lambda x, k, tau: np.full(1, tau), -1, 4)
    assert abs(xT[0] - (-(1 + 0.75 + 0.5 + 0.25) / 4)) < 1e-15


def test_reverse_time_with_velocity_sign_change():
    # vla.cpp III-A: reversing the time coordinate requires the velocity sign change
    f = lambda x, k, tau: np.sin(3 * x) * (1 + tau) - tau ** 2
    x0 = rng.standard_normal(8)
    xa, ta = oracle.euler(x0, f, +1, 4, record=True)
    xb, tb = oracle.euler(x0, lambda x, k, tau: -f(x, k, 1.0 - tau), -1, 4, record=True)
    np.testing.assert_array_equal(xa, xb)
    for u, v in zip(ta, tb):   # recorded velocities differ exactly by the sign
        np.testing.assert_array_equal(u, -v)


# ---------------------------------------------------------------------------
# whole expert: structural invariants and a torch-composed cross-check
# ---------------------------------------------------------------------------

def _expert_case(name="small_bf16", **kw):
    c = synth.make_case(name, **kw)
    for k in list(c["weights"]):
        c["weights"][k] = c["weights"][k].astype(np.float64)
    return c


def _rows(c, k=1):
    g = c["geom"]
    T, B = g["steps"], g["batch"]
    return oracle.modulation_table(g, c["weights"], T, B)[k * B:(k + 1) * B]


def torch_expert_velocity(g, w, x, rows, K, V):
    """The expert velocity composed from torch.nn.functional routines (fp64).

    RoPE in complex form, attention through scaled_dot_product_attention with
    the single KV head broadcast to every query head.
    """
    D, L, Hq, Dh, F_ = g["hidden"], g["layers"], g["q_heads"], g["head_dim"], g["mlp_dim"]
    B, H, A = x.shape
    P = K[0].shape[1]
    W = {k: t64(v) for k, v in w.items()}
    pos = torch.arange(P, P + H, dtype=torch.float64)
    ang = pos[:, None] * (g["rope_theta"] ** (-torch.arange(Dh // 2, dtype=torch.float64) * 2 / Dh))[None]
    rot = torch.polar(torch.ones_like(ang), ang)

    def rope(t):  # [..., H, Dh]
        z = torch.complex(t[..., :Dh // 2], t[..., Dh // 2:]) * rot
        return torch.cat([z.real, z.imag], -1)

    out = []
    for b in range(B):
        r = t64(rows[b])
        h = F.linear(t64(x[b]), W["action_in_w"], W["action_in_b"])
        for l in range(L):
            sc, sh, gt = r[2 * l].chunk(3)
            n = F.rms_norm(h, (D,), eps=g["norm_eps"]) * (1 + sc) + sh
            q, k, v = F.linear(n, W[f"qkv_w.{l}"]).split([Hq * Dh, Dh, Dh], -1)
            q = rope(q.view(H, Hq, Dh).transpose(0, 1))
            keys = torch.cat([t64(K[l][b, :, 0]), rope(k)], 0).expand(Hq, -1, -1)
            vals = torch.cat([t64(V[l][b, :, 0]), v], 0).expand(Hq, -1, -1)
            o = F.scaled_dot_product_attention(q, keys, vals).transpose(0, 1).reshape(H, Hq * Dh)
            h = h + gt * F.linear(o, W[f"o_w.{l}"])
            sc, sh, gt = r[2 * l + 1].chunk(3)
            n = F.rms_norm(h, (D,), eps=g["norm_eps"]) * (1 + sc) + sh
            up = F.linear(n, W[f"up_w.{l}"])
            u = F.gelu(up[:, :F_], approximate="tanh") * up[:, F_:] if up.shape[-1] == 2 * F_ \
                else F.gelu(up, approximate="tanh")
            h = h + gt * F.linear(u, W[f"down_w.{l}"])
        sc, sh, _ = r[2 * L].chunk(3)
        n = F.rms_norm(h, (D,), eps=g["norm_eps"]) * (1 + sc) + sh
        out.append(F.linear(n, W["action_out_w"], W["action_out_b"]))
    return torch.stack(out).numpy()


@pytest.mark.parametrize("name", ["small_bf16", "tiny"])
def test_expert_velocity_matches_torch_composition(name):
    c = _expert_case(name)
    g = c["geom"]
    rows = _rows(c)
    v = expert_velocity(g, c["weights"], c["x_noise"], rows, c["K"], c["V"])
    ref = torch_expert_velocity(g, c["weights"], c["x_noise"], rows, c["K"], c["V"])
    np.testing.assert_allclose(v, ref, rtol=1e-10, atol=1e-12)


def test_expert_zero_gates_drop_every_branch():
    c = _expert_case()
    g, w = c["geom"], c["weights"]
    D = g["hidden"]
    w["cond_w"][:, 2 * D:] = 0.0
    w["cond_b"][:, 2 * D:] = 0.0
    rows = _rows(c)
    v = expert_velocity(g, w, c["x_noise"], rows, c["K"], c["V"])
    K2 = [k * 0.5 + 1.0 for k in c["K"]]
    np.testing.assert_array_equal(v, expert_velocity(g, w, c["x_noise"], rows, K2, c["V"]))
    # equals the network with no layers: final AdaRMS of the input projection
    h = c["x_noise"].astype(np.float64) @ w["action_in_w"].T + w["action_in_b"]
    n, _ = ada_rms(h, rows[0, 2 * g["layers"]], g["norm_eps"])
    np.testing.assert_allclose(v[0], n[0] @ w["action_out_w"].T + w["action_out_b"], rtol=1e-13)


def test_expert_modulation_rows_select_branches():
    # row 2l gates layer l's attention branch, row 2l+1 its MLP branch
    c = _expert_case()
    g, w = c["geom"], c["weights"]
    D = g["hidden"]
    w["cond_w"][:, 2 * D:] = 0.0
    w["cond_b"][:, 2 * D:] = 0.0
    w["cond_b"][0, 2 * D:] = 1.0      # only layer 0's attention gate is open
    rows = _rows(c)
    base = expert_velocity(g, w, c["x_noise"], rows, c["K"], c["V"])
    w2 = dict(w)
    w2["down_w.0"] = w["down_w.0"] * 3.0
    np.testing.assert_array_equal(base, expert_velocity(g, w2, c["x_noise"], rows, c["K"], c["V"]))
    w3 = dict(w)
    w3["o_w.0"] = w["o_w.0"] * 3.0
    assert np.abs(expert_velocity(g, w3, c["x_noise"], rows, c["K"], c["V"]) - base).max() > 1e-6
    K2 = [k[:, ::-1].copy() * 0.9 for k in c["K"]]
    assert np.abs(expert_velocity(g, w, c["x_noise"], rows, K2, c["V"]) - base).max() > 1e-6


def test_expert_prefix_permutation_invariance():
    c = _expert_case()
    g = c["geom"]
    rows = _rows(c)
    v = expert_velocity(g, c["weights"], c["x_noise"], rows, c["K"], c["V"])
    perm = rng.permutation(g["prefix"])
    K2 = [k[:, perm] for k in c["K"]]
    V2 = [x[:, perm] for x in c["V"]]
    np.testing.assert_allclose(expert_velocity(g, c["weights"], c["x_noise"], rows, K2, V2), v,
                               rtol=1e-11, atol=1e-13)


def test_expert_empty_prefix_single_query_reads_own_value():
    # P = 0 and one action token: softmax over one key is 1, so q and k do not matter
    c = _expert_case("small_bf16", prefix=0, horizon=1, batch=1)
    g, w = c["geom"], c["weights"]
    rows = _rows(c)
    v = expert_velocity(g, w, c["x_noise"], rows, c["K"], c["V"])
    w2 = dict(w)
    qk = g["q_heads"] * g["head_dim"] + g["head_dim"]
    for l in range(g["layers"]):
        m = w[f"qkv_w.{l}"].copy()
        m[:qk] = rng.standard_normal(m[:qk].shape)
        w2[f"qkv_w.{l}"] = m
    np.testing.assert_allclose(expert_velocity(g, w2, c["x_noise"], rows, c["K"], c["V"]), v,
                               rtol=1e-12, atol=1e-14)


def test_expert_batch_samples_are_independent():
    c = _expert_case()
    g = c["geom"]
    rows = _rows(c)
    v = expert_velocity(g, c["weights"], c["x_noise"], rows, c["K"], c["V"])
    for b in range(g["batch"]):
        vb = expert_velocity(g, c["weights"], c["x_noise"][b:b + 1], rows[b:b + 1],
                             [k[b:b + 1] for k in c["K"]], [x[b:b + 1] for x in c["V"]])
        np.testing.assert_allclose(vb[0], v[b], rtol=1e-14, atol=1e-15)


def test_expert_fp32_instantiation_tracks_fp64():
    c = synth.make_case("tiny")
    x64 = oracle.denoise(c)
    x32 = oracle.denoise(c, dtype=np.float32)
    assert x32.dtype == np.float32
    assert oracle.error_metrics(x32, x64)[1] < 1e-6


# ---------------------------------------------------------------------------
# whole DiT head
# ---------------------------------------------------------------------------

def torch_dit_velocity(g, w, x, rows, atb, K, V, tm, im, state):
    D, L, Hq, Dh = g["hidden"], g["layers"], g["q_heads"], g["head_dim"]
    B, H, A = x.shape
    Ns = g["state_tokens"]
    W = {k: t64(v) for k, v in w.items()}
    out = []
    for b in range(B):
        r = t64(rows[b])
        a = F.linear(t64(x[b]), W["enc_w1"], W["enc_b1"])
        e = F.silu(F.linear(a, W["enc_w2"][:, :D]) + t64(atb))
        h = torch.cat([t64(state[b]), F.linear(e, W["enc_w3"], W["enc_b3"])], 0)
        T = h.shape[0]
        for i in range(L):
            sc, sh = r[i][:2 * D].chunk(2)
            n = F.layer_norm(h, (D,), eps=g["norm_eps"]) * (1 + sc) + sh
            if i % 2 == 0:
                q = F.linear(n, W[f"qkv_w.{i}"]).view(T, Hq, Dh).transpose(0, 1)
                k = t64(K[i][b]).transpose(0, 1)
                v = t64(V[i][b]).transpose(0, 1)
                m = torch.from_numpy((tm if i % 4 == 0 else im)[b].astype(bool))[None, None]
                o = F.scaled_dot_product_attention(q, k, v, attn_mask=m)
            else:
                q, k, v = F.linear(n, W[f"qkv_w.{i}"]).view(T, 3, Hq, Dh).permute(1, 2, 0, 3)
                o = F.scaled_dot_product_attention(q, k, v)
            h = h + F.linear(o.transpose(0, 1).reshape(T, Hq * Dh), W[f"o_w.{i}"])
            f = F.gelu(F.linear(F.layer_norm(h, (D,), eps=g["norm_eps"]), W[f"up_w.{i}"]), approximate="tanh")
            h = h + F.linear(f, W[f"down_w.{i}"])
        sh, sc = r[L][:2 * D].chunk(2)
        n = F.layer_norm(h, (D,), eps=g["norm_eps"]) * (1 + sc) + sh
        out.append(F.linear(n[Ns:], W["action_out_w"], W["action_out_b"]))
    return torch.stack(out).numpy()


@pytest.mark.parametrize("masks", ["ones", "random"])
def test_dit_velocity_matches_torch_composition(masks):
    c = _expert_case("small_dit")
    g, w = c["geom"], c["weights"]
    tm, im = synth.make_masks(g, 0, kind=masks)
    rows = _rows(c, 2)
    atb = oracle.action_time_bias(g, w, g["steps"])[2]
    v = dit_velocity(g, w, c["x_noise"], rows, atb, c["K"], c["V"], tm, im, c["state"])
    ref = torch_dit_velocity(g, w, c["x_noise"], rows, atb, c["K"], c["V"], tm, im, c["state"])
    np.testing.assert_allclose(v, ref, rtol=1e-10, atol=1e-12)


def test_dit_mask_selection_by_block_index():
    # text mask on blocks with i % 4 == 0, image mask on the other cross blocks
    c = _expert_case("small_dit", layers=2)
    g, w = c["geom"], c["weights"]
    rows = _rows(c)
    atb = oracle.action_time_bias(g, w, g["steps"])[1]
    tm, im = synth.make_masks(g, 0, kind="random")
    ones = np.ones_like(tm)
    base = dit_velocity(g, w, c["x_noise"], rows, atb, c["K"], c["V"], ones, ones, c["state"])
    np.testing.assert_array_equal(
        dit_velocity(g, w, c["x_noise"], rows, atb, c["K"], c["V"], ones, im, c["state"]), base)
    assert np.abs(dit_velocity(g, w, c["x_noise"], rows, atb, c["K"], c["V"], tm, ones, c["state"])
                  - base).max() > 1e-6


def test_dit_final_row_is_shift_then_scale():
    # the last row splits (shift, scale): scale = -1 leaves v = W_out shift + b_out for every token
    c = _expert_case("small_dit")
    g, w = c["geom"], c["weights"]
    D, L = g["hidden"], g["layers"]
    w["cond_w"][L] = 0.0
    shift = rng.standard_normal(D)
    w["cond_b"][L] = np.concatenate([shift, -np.ones(D)])
    rows = _rows(c)
    atb = oracle.action_time_bias(g, w, g["steps"])[1]
    v = dit_velocity(g, w, c["x_noise"], rows, atb, c["K"], c["V"], None, None, c["state"])
    np.testing.assert_allclose(v, np.broadcast_to(shift @ w["action_out_w"].T + w["action_out_b"], v.shape),
                               rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# geometry figures the pages print
# ---------------------------------------------------------------------------

def test_page_geometry_golden():
    gold = json.load(open(os.path.join(GOLDEN, "page_geometry.json")))
    g = synth.config("pi05")
    sh = synth.weight_shapes(g)
    layer_params = sum(int(np.prod(s)) for k, s in sh.items() if "." in k)
    cond = int(np.prod(sh["cond_w"]))
    assert round((layer_params + cond) / 1e6) == gold["pi05_expert_params_millions"]["value"]
    assert g["layers"] == gold["pi05_layers"]["value"] and g["hidden"] == gold["pi05_hidden"]["value"]
    assert g["head_dim"] == gold["pi05_head_dim"]["value"] and g["kv_heads"] == gold["pi05_kv_heads"]["value"]
    assert list(sh["cond_w"]) == gold["pi05_cond_denses"]["value"]
    assert round(cond * 2 / 1e6, 1) == gold["pi05_cond_fp16_megabytes"]["value"]
    assert [synth.norm_sites(g), synth.row_width(g)] == gold["pi05_modulation_entry"]["value"]
    d = synth.config("gr00t")
    shd = synth.weight_shapes(d)
    assert [synth.norm_sites(d), synth.row_width(d)] == gold["gr00t_adaln_table_entry"]["value"]
    assert sorted(shd["cond_w"][1:]) == sorted(gold["gr00t_adaln_projection"]["value"])
    assert round(int(np.prod(shd["cond_w"])) * 2 / 1e6) == gold["gr00t_adaln_fp16_megabytes"]["value"]
    assert d["hidden"] == gold["gr00t_action_time_bias"]["value"]
    assert [d["kv_heads"], d["head_dim"]] == gold["gr00t_cross_kv_heads_dim"]["value"]
    assert d["layers"] == gold["gr00t_blocks"]["value"] and d["steps"] == gold["gr00t_steps"]["value"]


def test_modulation_table_shape_matches_contract():
    # adarms_modulation is [num_steps * batch, 37, 3072] for the pi0.5 expert
    g = synth.config("pi05")
    w = {k: np.zeros(s, np.float32) for k, s in synth.weight_shapes(g).items()
         if k.startswith(("cond", "time"))}
    assert oracle.modulation_table(g, w, 2, 3).shape == (6, 37, 3072)


# ---------------------------------------------------------------------------
# FP8 (E4M3) weights: decode, row scales, and the oracle's use of them
# ---------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_decode_closed_forms():
    d = lambda c: float(oracle.e4m3_decode(np.uint8(c)))
    assert d(0x38) == 1.0 and d(0xB8) == -1.0
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0        # largest finite magnitude
    assert d(0x08) == 2.0 ** -6 and d(0x01) == 2.0 ** -9   # smallest normal / subnormal
    assert d(0x07) == 7 * 2.0 ** -9 and d(0x0F) == 1.875 * 2.0 ** -6
    assert d(0x00) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)   # finite codes are ordered by magnitude


def test_dequantize_rows_scales_each_output_row():
    codes = np.full((3, 5), 0x38, np.uint8)    # 1.0
    codes[1, 2] = 0xC0                          # -2.0
    sc = np.array([0.5, 2.0, 3.0], np.float32)
    W = oracle.dequantize_rows(codes, sc)
    ref = np.repeat(sc[:, None].astype(np.float64), 5, axis=1)
    ref[1, 2] = -4.0
    np.testing.assert_array_equal(W, ref)


def _dequantized(w8):
    wd = {k: v for k, v in w8.items() if not k.endswith(".scale")}
    for k in list(wd):
        if k + ".scale" in w8:
            wd[k] = oracle.dequantize_rows(w8[k], w8[k + ".scale"])
        else:
            wd[k] = wd[k].astype(np.float64)
    return wd


def test_fp8_expert_case_runs_on_the_dequantized_matrices():
    c = synth.make_case("small_fp8", batch=2)
    g, w8 = c["geom"], c["weights"]
    assert w8["qkv_w.0"].dtype == np.uint8 and w8["qkv_w.0.scale"].dtype == np.float32
    wd = _dequantized(w8)
    B = g["batch"]
    rows = oracle.modulation_table(g, wd, g["steps"], B)[B:2 * B]
    v8 = expert_velocity(g, w8, c["x_noise"], rows, c["K"], c["V"])
    vd = expert_velocity(g, wd, c["x_noise"], rows, c["K"], c["V"])
    assert np.array_equal(v8, vd)
    ref = torch_expert_velocity(g, wd, c["x_noise"], rows, c["K"], c["V"])
    np.testing.assert_allclose(v8, ref, rtol=1e-10, atol=1e-12)


def test_fp8_dit_case_runs_on_the_dequantized_matrices():
    c = synth.make_case("small_dit_fp8")
    g, w8 = c["geom"], c["weights"]
    wd = _dequantized(w8)
    B = g["batch"]
    rows = oracle.modulation_table(g, wd, g["steps"], B)[2 * B:3 * B]
    atb = oracle.action_time_bias(g, wd, g["steps"])[2]
    args = (c["x_noise"], rows, atb, c["K"], c["V"], c["text_mask"], c["image_mask"], c["state"])
    v8 = dit_velocity(g, w8, *args)
    assert np.array_equal(v8, dit_velocity(g, wd, *args))
    np.testing.assert_allclose(v8, torch_dit_velocity(g, wd, *args), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
# bind-time cross K/V projection (DiT with VL features)
# ---------------------------------------------------------------------------

def test_project_context_matches_torch_linear():
    c = synth.make_case("small_dit_ctx")
    g, w = c["geom"], c["weights"]
    K, V = oracle.project_context(g, w, c["features"])
    f = t64(c["features"])
    B, P = c["features"].shape[:2]
    for l in range(g["layers"]):
        if l % 2:
            assert K[l] is None and V[l] is None
            continue
        for M, name in ((K[l], "cross_k_w"), (V[l], "cross_v_w")):
            ref = F.linear(f, t64(w[f"{name}.{l}"])).reshape(B, P, g["kv_heads"], g["head_dim"]).numpy()
            np.testing.assert_allclose(M, ref, rtol=1e-12, atol=1e-12)


def test_context_case_equals_bound_projections():
    c = synth.make_case("small_dit_ctx")
    K, V = oracle.project_context(c["geom"], c["weights"], c["features"])
    bound = dict(c, features=None, K=K, V=V)
    assert np.array_equal(oracle.denoise(c), oracle.denoise(bound))


# ---------------------------------------------------------------------------
# bind-time state encoder (DiT with a raw robot state)
# ---------------------------------------------------------------------------

def test_encode_state_matches_torch_mlp():
    c = synth.make_case("small_dit_state")
    g, w = c["geom"], c["weights"]
    s = c["state_raw"]
    assert s.shape == (g["batch"], g["state_tokens"], g["state_dim"])
    got = oracle.encode_state(g, w, s)
    ref = F.linear(F.silu(F.linear(t64(s), t64(w["state_w1"]), t64(w["state_b1"]))),
                   t64(w["state_w2"]), t64(w["state_b2"])).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_encode_state_closed_forms():
    # zero first layer: every state maps to W_s2 swish(b_s1) + b_s2; zero second
    # layer: the bias alone; and the first layer sees the state, not its transpose
    c = synth.make_case("small_dit_state")
    g, w = c["geom"], dict(c["weights"])
    D = g["hidden"]
    w0 = dict(w, state_w1=np.zeros_like(w["state_w1"]))
    const = w["state_w2"].astype(np.float64) @ oracle.swish(w["state_b1"].astype(np.float64)) + w["state_b2"]
    got = oracle.encode_state(g, w0, c["state_raw"])
    np.testing.assert_allclose(got, np.broadcast_to(const, got.shape), rtol=1e-13, atol=1e-13)
    wz = dict(w, state_w2=np.zeros_like(w["state_w2"]))
    np.testing.assert_array_equal(oracle.encode_state(g, wz, c["state_raw"]),
                                  np.broadcast_to(w["state_b2"].astype(np.float64), (g["batch"], 1, D)))
    # a one-hot state picks one column of W_s1
    e = np.zeros((1, 1, g["state_dim"]))
    e[0, 0, 5] = 1.0
    wi = dict(w, state_w2=np.eye(D), state_b2=np.zeros(D), state_b1=np.zeros(D))
    np.testing.assert_allclose(oracle.encode_state(g, wi, e)[0, 0],
                               oracle.swish(w["state_w1"][:, 5].astype(np.float64)), rtol=1e-14, atol=1e-15)


def test_state_case_equals_bound_state_tokens():
    c = synth.make_case("small_dit_state")
    assert c["state"] is None and c["state_raw"] is not None
    tokens = oracle.encode_state(c["geom"], c["weights"], c["state_raw"])
    bound = dict(c, state_raw=None, state=tokens)
    assert np.array_equal(oracle.denoise(c), oracle.denoise(bound))


def test_residual_traces_end_in_the_velocity():
    # the last traced residual, through the final norm and output projection, is the
    # velocity; the first is the step's input embedding (the debug-dump reference)
    for name in ("small_bf16", "small_dit"):
        c = synth.make_case(name)
        g, w = c["geom"], c["weights"]
        B, L, D, k = g["batch"], g["layers"], g["hidden"], 1
        mod = oracle.modulation_table(g, w, g["steps"], B)[k * B:(k + 1) * B]
        tr = {}
        if g["family"] == synth.FAMILY_EXPERT:
            v = expert_velocity(g, w, c["x_noise"], mod, c["K"], c["V"], trace=tr)
            for b in range(B):
                n, _ = ada_rms(tr[f"h.{L - 1}"][b], mod[b, 2 * L].astype(np.float64), g["norm_eps"])
                np.testing.assert_allclose(n @ w["action_out_w"].astype(np.float64).T + w["action_out_b"], v[b],
                                           rtol=1e-12, atol=1e-12)
                h0 = c["x_noise"][b].astype(np.float64) @ w["action_in_w"].astype(np.float64).T + w["action_in_b"]
                np.testing.assert_allclose(tr["h_in"][b], h0, rtol=1e-13, atol=1e-13)
        else:
            atb = oracle.action_time_bias(g, w, g["steps"])[k]
            v = dit_velocity(g, w, c["x_noise"], mod, atb, c["K"], c["V"], c["text_mask"], c["image_mask"],
                             c["state"], trace=tr)
            Ns = g["state_tokens"]
            for b in range(B):
                row = mod[b, L].astype(np.float64)
                n = oracle.layer_norm(tr[f"h.{L - 1}"][b], g["norm_eps"]) * (1 + row[D:2 * D]) + row[:D]
                np.testing.assert_allclose(n[Ns:] @ w["action_out_w"].astype(np.float64).T + w["action_out_b"],
                                           v[b], rtol=1e-12, atol=1e-12)
                np.testing.assert_array_equal(tr["h_in"][b][:Ns], c["state"][b])
        assert len([k_ for k_ in tr if k_.startswith("h.")]) == L
