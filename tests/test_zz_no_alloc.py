"""The allocation-free step entry point, checked against gr00t_denoise_step.

Collected last on purpose (file name): a failure here comes after every other
test has run.  The entry point exists for callers that may not allocate device
memory when they run a step; it takes its scratch from a fixed array in the
library image instead of the context's workspace, so its results must match
the regular step's on the same inputs, call after call.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

VEL_REL = 1e-2     # bf16 per-step velocity gate used by the parity tests


def _fmv():
    import flow_matching_vla_gb300 as fmv
    return fmv


@pytest.mark.parametrize("name", ["small_bf16", "pi05", "small_fp8"])
def test_noalloc_step_matches_regular_step_twice(name):
    fmv = _fmv()
    c = synth.make_case(name)
    g = c["geom"]
    loop, held = fmv.from_case(c)
    x = torch.from_numpy(c["x_noise"]).cuda()
    mod = oracle.modulation_table(g, c["weights"], g["steps"], g["batch"])
    for k in (0, g["steps"] - 1):      # two calls in a row, different steps
        ref = loop.denoise_step(k, x).clone()
        got = torch.full_like(ref, float("nan"))
        loop.denoise_step_noalloc(k, x, got)
        torch.cuda.synchronize()
        # the same launch sequence with the same plans: bit for bit the regular step
        assert torch.equal(got, ref), (k, float((got - ref).abs().max()))
        v_ref = oracle.velocity(c, c["x_noise"].astype(np.float64), k, mod=mod)
        e_inf, e_rel = oracle.error_metrics(got.cpu().numpy(), v_ref)
        print(f"noalloc {name} k={k}: velocity rel-L2 vs oracle {e_rel:.3e}")
        assert e_rel <= VEL_REL, (k, e_rel)
    assert loop.info(fmv.INFO_ERROR_FLAG) == 0


def test_noalloc_rejects_a_step_larger_than_its_scratch():
    fmv = _fmv()
    # pi0.5 at batch 1: the residual GEMMs' split-K partials need ~0.4 M floats;
    # with the no-alloc bound lowered below that the step is refused (on a
    # 152-SM GPU no step needs the whole 3 * 2^20-float array)
    c = synth.make_case("small_bf16", hidden=1024, mlp_dim=1024, batch=1, layers=1, prefix=64, time_dim=256)
    loop, held = fmv.from_case(c)
    loop.set_option(fmv.OPT_NOALLOC_LIMIT, 1000)
    x = torch.from_numpy(c["x_noise"]).cuda()
    out = torch.empty_like(x)
    with pytest.raises(fmv.Gr00tError) as ei:
        loop.denoise_step_noalloc(0, x, out)
    assert ei.value.status == -1 and "fixed array" in str(ei.value)
    # the regular entry point still runs the same step, and so does the
    # allocation-free one once the whole array may be used again
    loop.denoise_step(0, x, out)
    loop.set_option(fmv.OPT_NOALLOC_LIMIT, 3 << 20)
    out2 = torch.empty_like(x)
    loop.denoise_step_noalloc(0, x, out2)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.allclose(out, out2, rtol=0, atol=0)
    with pytest.raises(fmv.Gr00tError):
        loop.set_option(fmv.OPT_NOALLOC_LIMIT, (3 << 20) + 1)
