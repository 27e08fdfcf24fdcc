"""Runtime behaviour of the C ABI on the GPU: graphs, determinism, rebinds, errors."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _fmv():
    import flow_matching_vla_gb300 as fmv
    return fmv


def test_graph_replay_matches_eager_and_is_deterministic():
    fmv = _fmv()
    c = synth.make_case("small_bf16")
    loop, held = fmv.from_case(c)
    x0 = torch.from_numpy(c["x_noise"]).cuda()
    a = loop.denoise(x0).clone()
    b = loop.denoise(x0).clone()
    loop.set_option(fmv.OPT_USE_GRAPH, 0)
    e = loop.denoise(x0).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b), "graph replays differ"
    assert torch.equal(a, e), "graph and eager differ"


def test_denoise_host_matches_device():
    fmv = _fmv()
    c = synth.make_case("small_bf16")
    loop, held = fmv.from_case(c)
    x0 = torch.from_numpy(c["x_noise"]).cuda()
    d = loop.denoise(x0).cpu()
    xh = torch.from_numpy(c["x_noise"]).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    loop.denoise_host(xh, oh)
    assert torch.equal(d, oh)


def test_aliasing_in_place():
    fmv = _fmv()
    c = synth.make_case("small_bf16")
    loop, held = fmv.from_case(c)
    x0 = torch.from_numpy(c["x_noise"]).cuda()
    ref = loop.denoise(x0).clone()
    x1 = x0.clone()
    loop.denoise(x1, out=x1)
    torch.cuda.synchronize()
    assert torch.equal(ref, x1)


def test_rebind_same_shape_uses_new_prefix():
    fmv = _fmv()
    c = synth.make_case("small_bf16")
    loop, held = fmv.from_case(c)
    x0 = torch.from_numpy(c["x_noise"]).cuda()
    first = loop.denoise(x0).cpu().numpy()
    c2 = synth.make_case("small_bf16", seed=0)
    K2, V2 = synth.make_prefix_kv(c2["geom"], seed=7)
    Kd = [torch.from_numpy(k).to("cuda", torch.bfloat16) for k in K2]
    Vd = [torch.from_numpy(v).to("cuda", torch.bfloat16) for v in V2]
    loop.bind_prefix_kv(Kd, Vd)
    second = loop.denoise(x0).cpu().numpy()
    c2["K"], c2["V"] = K2, V2
    ref = oracle.denoise(c2)
    assert oracle.error_metrics(second, ref)[0] <= 2e-2
    assert np.abs(second - first).max() > 1e-4


def test_hoist_is_noop_for_same_schedule_and_recomputes_on_change():
    fmv = _fmv()
    c = synth.make_case("small_bf16")
    loop, held = fmv.from_case(c)
    x0 = torch.from_numpy(c["x_noise"]).cuda()
    a = loop.denoise(x0).cpu()
    loop.set_schedule(3, 3)         # same (steps, batch): no-op
    b = loop.denoise(x0).cpu()
    assert torch.equal(a, b)
    loop.set_schedule(2, 3)
    c2 = loop.denoise(x0).cpu().numpy()
    ref = oracle.denoise(c, steps=2)
    assert oracle.error_metrics(c2, ref)[0] <= 2e-2


def test_errors_are_statuses_not_crashes():
    fmv = _fmv()
    c = synth.make_case("small_bf16")
    loop = fmv.DenoiseLoop(c["geom"], c["weights"])
    x0 = torch.from_numpy(c["x_noise"]).cuda()
    with pytest.raises(fmv.Gr00tError) as ei:
        loop.denoise(x0)
    assert ei.value.status == -4   # ESTATE: nothing bound
    with pytest.raises(fmv.Gr00tError) as ei:
        loop.set_schedule(c["geom"]["steps"] + 1, 1)
    assert ei.value.status == -1   # EINVAL: beyond max_steps
    g = dict(c["geom"])
    g["kv_heads"] = 2
    with pytest.raises(fmv.Gr00tError):
        fmv.DenoiseLoop(g, c["weights"])


def test_batch_mismatch_between_bind_and_schedule():
    fmv = _fmv()
    c = synth.make_case("small_bf16")
    loop, held = fmv.from_case(c)
    loop.set_schedule(3, 2)
    with pytest.raises(fmv.Gr00tError) as ei:
        loop.denoise(torch.from_numpy(c["x_noise"]).cuda())
    assert ei.value.status == -4


@pytest.mark.parametrize("name", ["small_bf16", "small_dit"])
def test_tensor_core_gemm_matches_cuda_core_gemm(name):
    """Same inputs through both GEMM paths: only the fp32 summation order differs."""
    fmv = _fmv()
    c = synth.make_case(name)
    loop, held = fmv.from_case(c)
    x0 = torch.from_numpy(c["x_noise"]).cuda()
    vs = []
    for path in (0, 1):
        loop.set_option(fmv.OPT_GEMM_PATH, path)
        vs.append(loop.denoise_step(0, x0).cpu().numpy())
    e_inf, e_rel = oracle.error_metrics(vs[0], vs[1])
    assert e_rel < 5e-3, e_rel
    assert loop.info(fmv.INFO_ERROR_FLAG) == 0


@pytest.mark.parametrize("name", ["pi05", "pi05_b32"])
def test_no_bounded_wait_timed_out(name):
    fmv = _fmv()
    c = synth.make_case(name)
    loop, held = fmv.from_case(c)
    x0 = torch.from_numpy(c["x_noise"]).cuda()
    loop.denoise(x0)
    assert loop.info(fmv.INFO_ERROR_FLAG) == 0


def test_launch_stamps_cover_every_launch_of_the_loop():
    """gr00t_kernel_times: one interval per launch of the captured loop, classes of
    every kind, intervals that add up to the loop's device time."""
    fmv = _fmv()
    c = synth.make_case("small_bf16")
    g = c["geom"]
    loop, held = fmv.from_case(c)
    x0 = torch.from_numpy(c["x_noise"]).cuda()
    ref = loop.denoise(x0).clone()
    per_step = loop.info(fmv.INFO_KERNELS_PER_STEP)
    loop.set_option(fmv.OPT_TIME_KERNELS, 1)
    got = loop.denoise(x0).clone()
    loop.denoise(x0)
    us, cls = loop.kernel_times()
    assert len(us) == per_step * g["steps"]
    assert set(cls) >= {fmv.KCLASS_QKV_GEMM, fmv.KCLASS_ATTENTION, fmv.KCLASS_O_GEMM, fmv.KCLASS_UP_GEMM,
                        fmv.KCLASS_DOWN_GEMM, fmv.KCLASS_NORM}
    assert all(u >= 0 for u in us) and sum(us) > 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    loop.denoise(x0)
    b.record()
    b.synchronize()
    loop_us = a.elapsed_time(b) * 1000.0
    us2, _ = loop.kernel_times()
    print(f"stamped loop {sum(us2):.1f} us, event-timed loop {loop_us:.1f} us")
    assert sum(us2) <= loop_us * 1.05 + 5.0
    assert torch.equal(got, ref), "the stamps changed the results"
    loop.set_option(fmv.OPT_TIME_KERNELS, 0)
    assert loop.kernel_times() == ([], [])


def test_bounded_wait_timeout_is_reported_and_the_context_recovers():
    """A bounded device wait that runs out (on a word nothing writes) sets the error
    word; the synchronous calls return GR00T_ETIMEOUT, clear it, and the next call
    runs clean with the same results as before."""
    fmv = _fmv()
    c = synth.make_case("small_bf16")
    loop, held = fmv.from_case(c)
    xh = torch.from_numpy(c["x_noise"]).pin_memory()
    clean = torch.empty_like(xh).pin_memory()
    loop.denoise_host(xh, clean)
    loop.set_option(fmv.OPT_TEST_STALL, 2000)
    oh = torch.empty_like(xh).pin_memory()
    with pytest.raises(fmv.Gr00tError) as ei:
        loop.denoise_host(xh, oh)
    assert ei.value.status == fmv.ETIMEOUT and "bounded device wait" in str(ei.value)
    assert loop.info(fmv.INFO_ERROR_FLAG) == 0          # cleared by the report
    loop.denoise_step(0, torch.from_numpy(c["x_noise"]).cuda())   # asynchronous: reported by sync
    with pytest.raises(fmv.Gr00tError) as ei:
        loop.sync()
    assert ei.value.status == fmv.ETIMEOUT
    loop.set_option(fmv.OPT_TEST_STALL, 0)
    loop.sync()
    again = torch.empty_like(xh).pin_memory()
    loop.denoise_host(xh, again)
    assert torch.equal(again, clean)


@pytest.mark.parametrize("name", ["small_bf16", "small_dit", "small_dit_state"])
def test_debug_dump_matches_the_oracle_trace(name):
    """gr00t_debug_dump: the residual stream after every block (and after the input
    projection, whose state rows are the bound -- or bind-time encoded -- state
    tokens) against the oracle's trace of the same velocity evaluation."""
    fmv = _fmv()
    c = synth.make_case(name)
    g, w = c["geom"], c["weights"]
    B, L, k = g["batch"], g["layers"], 1
    loop, held = fmv.from_case(c)
    x = c["x_noise"]
    mod = oracle.modulation_table(g, w, g["steps"], B)[k * B:(k + 1) * B]
    trace = {}
    if g["family"] == synth.FAMILY_EXPERT:
        oracle.expert_velocity(g, w, x, mod, c["K"], c["V"], trace=trace)
    else:
        atb = oracle.action_time_bias(g, w, g["steps"])[k]
        state = c["state"] if c.get("state_raw") is None else oracle.encode_state(g, w, c["state_raw"])
        oracle.dit_velocity(g, w, x, mod, atb, c["K"], c["V"], c["text_mask"], c["image_mask"], state,
                            trace=trace)
    xd = torch.from_numpy(x).cuda()
    worst = 0.0
    for layer in range(-1, L):
        h = loop.debug_dump(k, xd, layer).cpu().numpy()
        ref = np.stack(trace["h_in" if layer < 0 else f"h.{layer}"])
        _, rel = oracle.error_metrics(h, ref)
        worst = max(worst, rel)
        assert rel <= 1e-2, f"block {layer}: residual rel-L2 {rel:.3e}"
    print(f"debug dump {name}: worst residual rel-L2 {worst:.3e} over {L + 1} dumps")


def _bf16_ulp(x):
    # one unit in the last place of bf16 (8 significant bits) at |x|
    m, e = torch.frexp(x.abs().float())
    return torch.ldexp(torch.ones_like(m), (e - 8).clamp(min=-133))


@pytest.mark.parametrize("name,kw,exact", [
    ("small_bf16", dict(), True),          # steps x batch <= 64 rows: the same GEMM plan either way
    ("small_dit", dict(), True),
    ("pi05", dict(batch=8), False),        # 80 hoisted rows: 128-token tiles against 64-token ones
])
def test_hoisted_cond_equals_per_step_evaluation_on_gpu(name, kw, exact):
    """The hoist ("pi0.5 Design", cond component): for every step, the modulation rows that
    gr00t_set_schedule computed for all steps at once equal the same cond work evaluated for
    that step alone -- bit for bit where both run the same GEMM plan, else within one bf16 ulp
    (only the accumulation order of the GEMMs differs)."""
    fmv = _fmv()
    c = synth.make_case(name, **kw)
    g = c["geom"]
    loop, held = fmv.from_case(c)
    worst = 0.0
    for k in range(g["steps"]):
        h, p = loop.debug_cond_step(k, g["batch"])
        torch.cuda.synchronize()
        if exact:
            assert torch.equal(h, p), f"step {k}"
        d = (h.float() - p.float()).abs() / _bf16_ulp(torch.maximum(h.float().abs(), p.float().abs()))
        worst = max(worst, float(d.max()))
    print(f"hoist check {name}: worst difference {worst:.2f} bf16 ulp")
    assert worst <= 1.0
