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
