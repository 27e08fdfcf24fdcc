"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Gates: fp32 workloads rel-L2 <= 1e-4 (velocity per step and final chunk);
bf16 workloads per-step velocity rel-L2 <= 1e-2 (teacher forced: both sides
step from the oracle's x_k) and final chunk max-abs <= 2e-2 (free running).
Errors are vla.cpp Eq. (5).
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

FP32_REL = 1e-4
BF16_VEL_REL = 1e-2
BF16_CHUNK_ABS = 2e-2


def _fmv():
    import flow_matching_vla_gb300 as fmv
    return fmv


def _trajectory(case, steps=None):
    """Oracle x_k (fp64) and v_k for k = 0..T-1, plus x_T."""
    g = case["geom"]
    T = steps or g["steps"]
    xT, vs = oracle.denoise(case, steps=T, record=True)
    _, dts = oracle.schedule(g["direction"], T)
    xs = [case["x_noise"].astype(np.float64)]
    for k in range(T - 1):
        xs.append(xs[-1] + dts[k] * vs[k])
    return xs, vs, xT


def _gates(case):
    bf16 = case["geom"]["dtype"] == synth.DTYPE_BF16
    return (BF16_VEL_REL, None) if bf16 else (FP32_REL, FP32_REL)


def check_case(case, steps=None, samples=None, options=()):
    """Run the GPU loop on ``case`` and compare with the oracle.

    ``samples``: only compare these batch entries (the oracle runs them as
    batch-1 problems on their own inputs); None compares all of them.
    """
    fmv = _fmv()
    g = case["geom"]
    T = steps or g["steps"]
    loop, held = fmv.from_case(case, steps=T)
    for opt, val in options:
        loop.set_option(opt, val)
    x0 = torch.from_numpy(case["x_noise"]).cuda()
    out = loop.denoise(x0)
    # teacher-forced velocities need the oracle trajectory of the compared samples
    idx = list(range(g["batch"])) if samples is None else list(samples)
    sub = case if samples is None else _subcase(case, idx)
    xs, vs, xT = _trajectory(sub, T)
    vel_tol, chunk_rel = _gates(case)
    worst = 0.0
    for k in range(T):
        xk = np.zeros(case["x_noise"].shape, np.float32)
        xk[idx] = xs[k].astype(np.float32)
        v = loop.denoise_step(k, torch.from_numpy(xk).cuda()).cpu().numpy()[idx]
        e_inf, e_rel = oracle.error_metrics(v, vs[k])
        worst = max(worst, e_rel)
        assert e_rel <= vel_tol, f"step {k}: velocity rel-L2 {e_rel:.3e} > {vel_tol}"
    torch.cuda.synchronize()
    got = out.cpu().numpy()[idx]
    e_inf, e_rel = oracle.error_metrics(got, xT)
    # the margins, for the log: worst per-step velocity rel-L2 and the chunk errors
    print(f"parity {g.get('name', '?')} B={g['batch']} P={g['prefix']} T={T} samples={len(idx)}: "
          f"worst step rel-L2 {worst:.3e} (gate {vel_tol:g}), chunk max-abs {e_inf:.3e}, chunk rel-L2 {e_rel:.3e}")
    if chunk_rel is not None:
        assert e_rel <= chunk_rel, f"final chunk rel-L2 {e_rel:.3e}"
    else:
        assert e_inf <= BF16_CHUNK_ABS, f"final chunk max-abs {e_inf:.3e}"
    assert np.all(np.isfinite(out.cpu().numpy()))
    return loop, worst, e_inf, e_rel


def _subcase(case, idx):
    c = dict(case)
    c["x_noise"] = case["x_noise"][idx]
    c["K"] = [None if k is None else k[idx] for k in case["K"]]
    c["V"] = [None if v is None else v[idx] for v in case["V"]]
    for key in ("text_mask", "image_mask", "state", "state_raw", "features"):
        if case.get(key) is not None:
            c[key] = case[key][idx]
    c["geom"] = dict(case["geom"], batch=len(idx))
    return c


@pytest.mark.parametrize("name", ["tiny", "small_fp32", "small_dit_fp32"])
def test_fp32_parity(name):
    check_case(synth.make_case(name))


@pytest.mark.parametrize("name", ["small_bf16", "small_dit"])
def test_bf16_parity_small(name):
    check_case(synth.make_case(name))


def test_dit_random_masks():
    c = synth.make_case("small_dit")
    c["text_mask"], c["image_mask"] = synth.make_masks(c["geom"], 0, kind="random")
    check_case(c)


def test_dit_long_context_ring_and_fully_masked_rows():
    # 1000 context tokens: 16 key tiles through the attention's 6-slot TMA ring; sample 0
    # sees no text token at all, so the text-mask blocks' rows of that sample are 0
    c = synth.make_case("small_dit", prefix=1000)
    tm, im = synth.make_masks(c["geom"], 0, kind="random")
    tm[0] = 0
    c["text_mask"], c["image_mask"] = tm, im
    check_case(c)


def test_expert_empty_prefix_and_single_token():
    check_case(synth.make_case("small_bf16", prefix=0, horizon=1, batch=2))


def test_expert_fp32_empty_prefix():
    check_case(synth.make_case("small_fp32", prefix=0))


@pytest.mark.parametrize("steps", [1, 2, 5, 16])
def test_step_counts(steps):
    check_case(synth.make_case("small_bf16", steps=steps))


# horizon variants: LIBERO-style 10 actions, and 50 actions (ALOHA) at the full
# pi0.5 width with a short prefix
@pytest.mark.parametrize("horizon", [10, 50])
def test_horizon_variants(horizon):
    check_case(synth.make_case("small_bf16", horizon=horizon, batch=2))


def test_pi05_width_horizon_10():
    check_case(synth.make_case("pi05", horizon=10, prefix=256, layers=4))


def test_pi05_full_size():
    check_case(synth.make_case("pi05"))


def test_gr00t_full_size():
    check_case(synth.make_case("gr00t"))


def _straddling_samples(B, H, tiles=(128, 256)):
    """Samples whose token rows [b H, (b + 1) H) cross a 128- or 256-row tile
    boundary of the GEMMs, plus the first and the last sample."""
    out = {0, B - 1}
    for b in range(B):
        lo, hi = b * H, (b + 1) * H
        if any((lo // t) != ((hi - 1) // t) for t in tiles):
            out.add(b)
    return sorted(out)


def test_straddling_sample_choice():
    # pi0.5 at batch 32: rows of sample 2 (100..149) cross 128, sample 5 (250..299) crosses 256
    s = _straddling_samples(32, 50)
    assert {0, 2, 5, 7, 10, 12, 15, 17, 20, 23, 25, 28, 30, 31} <= set(s)


def test_pi05_batch32_straddling_samples():
    g = synth.config("pi05_b32")
    check_case(synth.make_case("pi05_b32"), samples=_straddling_samples(g["batch"], g["horizon"]))


def test_pi05_long_prefix_every_sample():
    check_case(synth.make_case("pi05_long"))


# every attention kernel of the expert family on the same small cases: 1 = CUDA
# cores, 2 = mma.sync head-folded, 3 = tcgen05/TMEM (several 128-row tiles,
# ragged key tiles, key splits combined across a cluster)
@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("kw", [dict(), dict(prefix=0, batch=1), dict(prefix=700, batch=2, horizon=30)])
def test_expert_attention_paths(path, kw):
    fmv = _fmv()
    check_case(synth.make_case("small_bf16", **kw), options=[(fmv.OPT_ATTN_PATH, path)])


# key tiles shared by the row tiles of a sample through cluster multicast: 2 row tiles
# (2 heads x 100 tokens) and 4 (4 heads x 100 tokens); the data movement must not change
# a single bit of the result
@pytest.mark.parametrize("kw", [dict(q_heads=2, horizon=100, batch=2, prefix=300),
                                dict(q_heads=4, horizon=100, batch=2, prefix=700)])
def test_attention_key_tile_multicast(kw):
    fmv = _fmv()
    case = synth.make_case("small_bf16", **kw)
    loop, _, _, _ = check_case(case, options=[(fmv.OPT_ATTN_MULTICAST, 1)])
    x0 = torch.from_numpy(case["x_noise"]).cuda()
    a = loop.denoise(x0).clone()
    loop.set_option(fmv.OPT_ATTN_MULTICAST, 0)
    b = loop.denoise(x0).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# the tensor-store epilogues (outputs staged in shared memory, written by tensor
# stores) against per-lane stores: the persistent GEMM's RoPE (head_dim 256 and 64),
# GeGLU and plain/GELU outputs, one and several tiles per CTA, a ragged last token
# tile; and the split GEMMs' fp32 residual partials (64- and 256-token tiles, 2 to 8
# splits, tokens past M clipped within each split).  Checked against the oracle with
# the tensor stores on (the default), then bit for bit against the per-lane stores.
@pytest.mark.parametrize("name,kw,split_cap", [
    ("small_bf16", dict(batch=8), 1),
    ("small_bf16", dict(batch=32, mlp_dim=2048), 4),
    ("small_bf16", dict(q_heads=4, head_dim=64, batch=6, prefix=150), 1),
    ("small_dit", dict(batch=16, prefix=120), 1),
    ("small_bf16", dict(), 4),
    ("small_dit", dict(), 4),
])
def test_gemm_tensor_store_epilogue(name, kw, split_cap):
    fmv = _fmv()
    case = synth.make_case(name, **kw)
    loop, _, _, _ = check_case(case, options=[(fmv.OPT_SPLIT_CAP, split_cap)])
    x0 = torch.from_numpy(case["x_noise"]).cuda()
    a = loop.denoise(x0).clone()
    loop.set_option(fmv.OPT_GEMM_TSTORE, 0)
    b = loop.denoise(x0).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# persistent GEMM tiles of two CTAs sharing each activation tile by multicast (one and
# several tiles per CTA, a ragged last token tile) against one CTA per tile stream
@pytest.mark.parametrize("kw", [dict(batch=8), dict(batch=32, mlp_dim=2048)])
def test_gemm_activation_multicast(kw):
    fmv = _fmv()
    case = synth.make_case("small_bf16", **kw)
    loop, _, _, _ = check_case(case, options=[(fmv.OPT_SPLIT_CAP, 1), (fmv.OPT_GEMM_MULTICAST, 1)])
    x0 = torch.from_numpy(case["x_noise"]).cuda()
    a = loop.denoise(x0).clone()
    loop.set_option(fmv.OPT_GEMM_MULTICAST, 0)
    b = loop.denoise(x0).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_tcgen05_attention_head_dim_64():
    fmv = _fmv()
    c = synth.make_case("small_bf16", q_heads=4, head_dim=64, batch=4, prefix=150)
    check_case(c, options=[(fmv.OPT_ATTN_PATH, 3)])


# many token rows (>= 256): the warp-per-row norms, the multi-row step head and
# the step tail; the residual split cap selects how many split-K partials the
# norms fold (1: none, 2: the unrolled pair, 16: the general loop)
@pytest.mark.parametrize("cap", [1, 2, 16])
def test_many_rows_expert_bf16(cap):
    fmv = _fmv()
    check_case(synth.make_case("small_bf16", batch=8), options=[(fmv.OPT_RESID_SPLIT_CAP, cap)])


def test_many_rows_expert_fp32():
    check_case(synth.make_case("small_fp32", batch=6))


def test_many_rows_dit_layer_norm():
    check_case(synth.make_case("small_dit", batch=16, prefix=120))


def test_single_token_horizon_unsplit_epilogue():
    # one token per sample and no split-K: the RoPE epilogue walks several
    # samples' rows per thread with a token index that wraps every column
    fmv = _fmv()
    check_case(synth.make_case("small_bf16", prefix=0, horizon=1, batch=5),
               options=[(fmv.OPT_SPLIT_CAP, 1)])


# split-K reduced on chip (partial tiles exchanged between the CTAs of a
# cluster): 128-token tiles with 2- and 4-way splits, and 8-way splits of the
# full-size DiT projections
@pytest.mark.parametrize("cap", [2, 4])
def test_onchip_split_k_small(cap):
    fmv = _fmv()
    check_case(synth.make_case("small_bf16", batch=2, prefix=120), options=[(fmv.OPT_SPLIT_CAP, cap)])


def test_onchip_split_k_dit_8way():
    fmv = _fmv()
    check_case(synth.make_case("gr00t"), options=[(fmv.OPT_SPLIT_CAP, 8)])


# FP8 weight streaming: per-layer projections as E4M3 codes + row scales (the
# oracle runs on the same codes, dequantized); several tiles, split-K reduced
# on chip and as partials, both families, then the full-size workloads
@pytest.mark.parametrize("name", ["small_fp8", "small_dit_fp8"])
def test_fp8_weights_parity_small(name):
    check_case(synth.make_case(name))


def test_fp8_weights_many_rows_and_caps():
    fmv = _fmv()
    check_case(synth.make_case("small_fp8", batch=8), options=[(fmv.OPT_SPLIT_CAP, 1)])
    check_case(synth.make_case("small_fp8", batch=2, prefix=120), options=[(fmv.OPT_SPLIT_CAP, 4)])


def test_pi05_fp8_full_size():
    check_case(synth.make_case("pi05_fp8"))


def test_gr00t_fp8_full_size():
    check_case(synth.make_case("gr00t_fp8"))


def test_pi05_fp8_batch32_sampled():
    check_case(synth.make_case("pi05_fp8", batch=32), samples=[0, 31])


# DiT cross K/V projected from VL features at bind time (gr00t_bind_context):
# the oracle projects in fp64, the GPU on the tensor cores into bf16 K/V
def test_dit_context_projection_small():
    check_case(synth.make_case("small_dit_ctx"))


def test_gr00t_context_projection_full_size():
    check_case(synth.make_case("gr00t_ctx"))


# DiT robot state embedded at bind time by the state encoder (raw state [B, Ns, state_dim],
# state_dim 40 and the pages' 132, padded to the tensor cores' K on the device)
def test_dit_state_encoder_small():
    check_case(synth.make_case("small_dit_state"))


def test_gr00t_state_encoder_full_size():
    check_case(synth.make_case("gr00t_state"))


def test_gr00t_state_encoder_with_context_projection():
    check_case(synth.make_case("small_dit_state", context_dim=256, batch=3))


def test_bind_context_refused_without_context_dim():
    fmv = _fmv()
    loop, held = fmv.from_case(synth.make_case("small_dit"))
    import torch
    f = torch.zeros((2, 300, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fmv.Gr00tError, match="ESTATE"):
        loop.bind_context(f)


# the pages' plane-major paged K/V pool bound directly: [2, B, capacity, 1, Dh]
# per layer, prefix in slot rows [0, P), every step's action K/V appended into
# rows [P, P + H); the filler rows must neither be read nor overwritten
def _pool_case(capacity=384, **kw):
    import torch
    case = synth.make_case("small_bf16", **dict(dict(batch=2, prefix=200), **kw))
    g = case["geom"]
    B, P, Dh = g["batch"], g["prefix"], g["head_dim"]
    pools = []
    for l in range(g["layers"]):
        pool = torch.full((2, B, capacity, 1, Dh), 1000.0, dtype=torch.bfloat16, device="cuda")
        pool[0, :, :P] = torch.from_numpy(case["K"][l]).to(torch.bfloat16).cuda()
        pool[1, :, :P] = torch.from_numpy(case["V"][l]).to(torch.bfloat16).cuda()
        pools.append(pool)
    return case, pools


# the second case runs the attention's row tiles as a 4-CTA multicast cluster (4 heads x
# 100 tokens), with the first row tile's CTA also storing the suffix K/V into the pool
@pytest.mark.parametrize("kw", [dict(), dict(q_heads=4, horizon=100)])
def test_expert_paged_kv_pool_parity(kw):
    import torch
    fmv = _fmv()
    case, pools = _pool_case(**kw)
    g = case["geom"]
    B, P, H = g["batch"], g["prefix"], g["horizon"]
    keep = [p.clone() for p in pools]
    loop = fmv.DenoiseLoop(g, case["weights"])
    loop.bind_kv_pool(pools, P)
    loop.set_schedule(g["steps"], B)
    out = loop.denoise(torch.from_numpy(case["x_noise"]).cuda())
    torch.cuda.synchronize()
    e_inf, _ = oracle.error_metrics(out.cpu().numpy(), oracle.denoise(case))
    assert e_inf <= BF16_CHUNK_ABS, f"final chunk max-abs {e_inf:.3e}"
    for p, p0 in zip(pools, keep):
        assert torch.equal(p[:, :, :P], p0[:, :, :P])                 # prefix untouched
        assert torch.equal(p[:, :, P + H:], p0[:, :, P + H:])         # past the suffix slots untouched
        assert float(p[:, :, P:P + H].float().abs().max()) < 100.0    # suffix slots written


def test_expert_paged_kv_pool_appends_the_step_suffix_kv():
    # one teacher-forced step from x: layer 0's slots [P, P + H) hold that step's
    # action-token K (RoPE at positions P + j) and V
    import torch
    from oracle.expert import ada_rms
    fmv = _fmv()
    case, pools = _pool_case()
    g = case["geom"]
    B, P, H, Hq, Dh = g["batch"], g["prefix"], g["horizon"], g["q_heads"], g["head_dim"]
    loop = fmv.DenoiseLoop(g, case["weights"])
    loop.bind_kv_pool(pools, P)
    loop.set_schedule(g["steps"], B)
    k = 1
    x = case["x_noise"]
    loop.denoise_step(k, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    w = case["weights"]
    mod = oracle.modulation_table(g, w, g["steps"], B)[k * B:(k + 1) * B]
    trace = {}
    oracle.expert_velocity(g, w, x, mod, case["K"], case["V"], trace=trace)
    for b in range(B):
        n, _ = ada_rms(trace["h_in"][b], mod[b, 0].astype(np.float64), g["norm_eps"])
        qkv = n @ w["qkv_w.0"].astype(np.float64).T
        k_ref = oracle.rope_rotate_half(qkv[:, Hq * Dh:Hq * Dh + Dh], P + np.arange(H), g["rope_theta"])
        v_ref = qkv[:, Hq * Dh + Dh:Hq * Dh + 2 * Dh]
        k_got = pools[0][0, b, P:P + H, 0].float().cpu().numpy()
        v_got = pools[0][1, b, P:P + H, 0].float().cpu().numpy()
        for got, ref in ((k_got, k_ref), (v_got, v_ref)):
            _, rel = oracle.error_metrics(got, ref)
            assert rel <= BF16_VEL_REL, f"sample {b}: suffix slot rel-L2 {rel:.3e}"


def test_paged_kv_pool_refusals():
    import torch
    fmv = _fmv()
    case, pools = _pool_case()
    g = case["geom"]
    loop = fmv.DenoiseLoop(g, case["weights"])
    small = [torch.zeros((2, 2, 200, 1, g["head_dim"]), dtype=torch.bfloat16, device="cuda")] * g["layers"]
    with pytest.raises(fmv.Gr00tError, match="capacity"):
        loop.bind_kv_pool(small, g["prefix"])   # 200 < prefix + horizon, not a multiple of 128
    loop.bind_kv_pool(pools, g["prefix"])
    loop.set_schedule(g["steps"], g["batch"])
    loop.set_option(fmv.OPT_ATTN_PATH, 1)
    with pytest.raises(fmv.Gr00tError, match="tcgen05 attention"):
        loop.denoise(torch.from_numpy(case["x_noise"]).cuda())
