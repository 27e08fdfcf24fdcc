"""Host-side checks that need no GPU: the library loads, exports what the
header declares, validates geometries, and refuses bad calls with statuses."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from flow_matching_vla_gb300 import build
    build.build()
    from flow_matching_vla_gb300 import _abi
    return _abi.load()


def test_every_declared_function_is_exported(lib):
    from flow_matching_vla_gb300 import _abi
    declared = _abi.header_functions()
    assert len(declared) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    for name in declared:
        assert name in exported, name
        assert name in _abi.SIGNATURES, name
        getattr(lib, name)


def test_library_is_sm103a_only(lib):
    from flow_matching_vla_gb300 import _abi
    out = subprocess.run(["cuobjdump", "--list-elf", _abi.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout
    assert all("sm_103" in l for l in out.stdout.splitlines() if ".cubin" in l)


@pytest.mark.parametrize("name", sorted(synth.CONFIGS))
def test_workload_geometries_validate(lib, name):
    import flow_matching_vla_gb300 as fmv
    rc, msg = fmv.validate_geometry(synth.config(name))
    assert rc == 0, msg


@pytest.mark.parametrize("field,value,needle", [
    ("kv_heads", 2, "kv_heads"),
    ("hidden", 100, "hidden"),
    ("direction", 0, "direction"),
    ("head_dim", 512, "head_dim"),
    ("max_steps", 0, "max_steps"),
    ("layers", 0, "layers"),
    ("mlp_kind", 7, "mlp_kind"),
    ("norm_eps", 0.0, "norm_eps"),
])
def test_bad_geometry_is_refused(lib, field, value, needle):
    import flow_matching_vla_gb300 as fmv
    g = synth.config("pi05")
    g[field] = value
    if field == "max_steps":
        g["steps"] = value
    rc, msg = fmv.validate_geometry(g)
    assert rc == -1 and needle in msg


def test_fp8_weight_geometry_rules(lib):
    import flow_matching_vla_gb300 as fmv
    assert fmv.validate_geometry(synth.config("pi05_fp8"))[0] == 0
    rc, msg = fmv.validate_geometry(synth.config("pi05_fp8", dtype=synth.DTYPE_FP32))
    assert rc == -1 and "BF16" in msg
    rc, msg = fmv.validate_geometry(synth.config("pi05_fp8", hidden=1088))   # 64 | 1088, 128 does not
    assert rc == -1 and "128" in msg
    rc, msg = fmv.validate_geometry(synth.config("pi05", weight_format=7))
    assert rc == -1 and "weight_format" in msg


def test_context_dim_rules(lib):
    import flow_matching_vla_gb300 as fmv
    assert fmv.validate_geometry(synth.config("gr00t_ctx"))[0] == 0
    rc, msg = fmv.validate_geometry(synth.config("pi05", context_dim=256))
    assert rc == -1 and "DiT" in msg
    rc, msg = fmv.validate_geometry(synth.config("gr00t_ctx", context_dim=100))
    assert rc == -1 and "context_dim" in msg


def test_state_dim_rules(lib):
    import flow_matching_vla_gb300 as fmv
    assert fmv.validate_geometry(synth.config("gr00t_state"))[0] == 0
    rc, msg = fmv.validate_geometry(synth.config("pi05", state_dim=32))
    assert rc == -1 and "state_dim" in msg
    rc, msg = fmv.validate_geometry(synth.config("gr00t_state", state_tokens=0))
    assert rc == -1 and "state_dim" in msg
    rc, msg = fmv.validate_geometry(synth.config("gr00t_state", state_dim=5000))
    assert rc == -1 and "state_dim" in msg


def test_dit_geometry_rules(lib):
    import flow_matching_vla_gb300 as fmv
    g = synth.config("gr00t")
    g["kv_heads"] = 1
    assert fmv.validate_geometry(g)[0] == -1
    g = synth.config("gr00t", prefix=0)
    assert fmv.validate_geometry(g)[0] == -1


def test_create_refuses_before_touching_cuda(lib):
    from flow_matching_vla_gb300 import _abi
    import flow_matching_vla_gb300 as fmv
    g = synth.config("pi05")
    g["kv_heads"] = 3
    geo = fmv._geometry(g)
    ctx = ctypes.c_void_p(1)
    w = _abi.Weights()
    rc = lib.gr00t_create(ctypes.byref(geo), ctypes.byref(w), None, ctypes.byref(ctx))
    assert rc == -1 and ctx.value is None
    assert b"kv_heads" in lib.gr00t_last_error(None)
    # NULL out pointer
    assert lib.gr00t_create(ctypes.byref(geo), ctypes.byref(w), None, None) == -1


def _dummy_weights(g, skip=()):
    """A gr00t_weights with every pointer the geometry needs set to a dummy
    non-NULL value (create checks presence before it touches the GPU)."""
    from flow_matching_vla_gb300 import _abi
    w = _abi.Weights()
    w.location = _abi.MEM_DEVICE
    one = ctypes.c_void_p(16)
    for name, _ in _abi.Weights._fields_[1:]:
        if name in skip:
            continue
        if name in ("qkv_w", "o_w", "up_w", "down_w", "qkv_s", "o_s", "up_s", "down_s", "cross_k_w", "cross_v_w"):
            arr = (ctypes.c_void_p * g["layers"])(*([16] * g["layers"]))
            setattr(w, name, ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)))
            w._keep = getattr(w, "_keep", []) + [arr]
        else:
            setattr(w, name, one)
    return w


@pytest.mark.parametrize("cfg,skip,needle", [
    ("pi05_fp8", ("qkv_s",), b"scale"),
    ("gr00t_ctx", ("cross_v_w",), b"cross"),
    ("pi05", ("cond_w",), b"cond_w"),
    ("gr00t_state", ("state_b2",), b"state encoder"),
])
def test_create_checks_weight_pointers_before_touching_cuda(lib, cfg, skip, needle):
    import flow_matching_vla_gb300 as fmv
    g = synth.config(cfg)
    ctx = ctypes.c_void_p(1)
    rc = lib.gr00t_create(ctypes.byref(fmv._geometry(g)), ctypes.byref(_dummy_weights(g, skip)), None,
                          ctypes.byref(ctx))
    assert rc == -1 and ctx.value is None
    assert needle in lib.gr00t_last_error(None)


def test_null_context_calls_are_einval(lib):
    assert lib.gr00t_set_schedule(None, 1, 1) == -1
    assert lib.gr00t_denoise(None, None, None) == -1
    assert lib.gr00t_destroy(None) == -1
    v = ctypes.c_int64()
    assert lib.gr00t_get_info(None, 1, ctypes.byref(v)) == -1


def test_binding_fails_loudly_without_library(tmp_path):
    code = ("import flow_matching_vla_gb300._abi as a; a.LIB_PATH='" + str(tmp_path / "nope.so") + "'\n"
            "try:\n    a.load()\nexcept RuntimeError as e:\n    print('raised', e)\n")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT)
    assert "raised" in out.stdout and "no CPU fallback" in out.stdout


def test_bench_work_accounting_matches_weight_shapes():
    """The bench's algorithmic bytes are the weights, the prefix K/V and the modulation
    rows read once per denoise step (641.1 MB for the pi0.5 expert at batch 1)."""
    import bench
    g = synth.config("pi05")
    w = bench.kernel_work(g, 1, 968)
    gemm_weight_bytes = sum(2 * int(np.prod(s)) for k, s in synth.weight_shapes(g).items() if "." in k)
    for name in ("qkv_gemm", "o_gemm", "up_gemm", "down_gemm", "attention"):
        assert w[name][0] == 18
    total_w = sum(w[k][0] * w[k][1] for k in ("qkv_gemm", "o_gemm", "up_gemm", "down_gemm"))
    assert total_w == gemm_weight_bytes
    assert w["attention"][0] * w["attention"][1] == 18 * 968 * 256 * 2 * 2
    by, fl = bench.step_work(g, 1, 968)
    assert abs(by / 1e6 - 641.1) < 0.2, by
    assert abs(fl / 1e9 - 38.65) < 0.1, fl
    by32, fl32 = bench.step_work(synth.config("pi05_b32"), 32, 968)
    assert abs(by32 / 1e9 - 1.201) < 0.002 and abs(fl32 / 1e9 - 1237) < 2, (by32, fl32)


def test_bench_traffic_needs_unchanged_sources(monkeypatch, tmp_path):
    import bench
    f = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic("pi05_b32", "attention") is None      # nothing recorded
    csv = tmp_path / "cap.csv"
    csv.write_text('"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
                   '"0","k","dram__bytes_read.sum","Mbyte","10.5"\n'
                   '"0","k","dram__bytes_write.sum","Mbyte","1.5"\n'
                   '"1","k","dram__bytes_read.sum","Mbyte","11.5"\n'
                   '"1","k","dram__bytes_write.sum","Mbyte","0.5"\n')
    bench.record_traffic(str(csv), "pi05_b32", "attention", "ncu ...")
    assert bench.measured_traffic("pi05_b32", "attention") == pytest.approx(12e6)
    # a digest that no longer matches the kernel sources hides the number
    monkeypatch.setattr(bench, "source_digest", lambda kernel="attention": "0" * 16)
    assert bench.measured_traffic("pi05_b32", "attention") is None


def test_bench_traffic_digest_is_per_kernel_class(monkeypatch, tmp_path):
    # a change to the GEMM sources leaves the attention's recorded traffic valid, and a
    # record for one class never vouches for another
    import bench
    f = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    csv = tmp_path / "cap.csv"
    csv.write_text('"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
                   '"0","k","dram__bytes_read.sum","Mbyte","8.0"\n'
                   '"0","k","dram__bytes_write.sum","Mbyte","2.0"\n')
    bench.record_traffic(str(csv), "pi05_b32", "attention", "ncu ...")
    assert bench.measured_traffic("pi05_b32", "attention") == pytest.approx(10e6)
    assert bench.measured_traffic("pi05_b32", "up_gemm") is None
    real = bench.source_digest
    monkeypatch.setattr(bench, "source_digest",
                        lambda kernel="attention": "f" * 16 if bench.source_group(kernel) == "gemm" else real(kernel))
    assert bench.measured_traffic("pi05_b32", "attention") == pytest.approx(10e6)
    assert bench.source_group("qkv_gemm") == "gemm" and bench.source_group("norm") == "norm"
