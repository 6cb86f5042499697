"""CPU-only checks of the C ABI: the library builds, loads and exports every declared
symbol; the host planner and argument validation behave as documented.  No
compute call is made (there is no GPU here)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dp():
    import __graft_entry__
    __graft_entry__.build()
    import example_gradient_clipping_gb300 as m
    return m


def _declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(dp_[a-z0-9_]+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol(dp):
    lib = ctypes.CDLL(dp.LIB_PATH)
    names = _declared_symbols()
    assert {"dp_layer_sqnorms", "dp_clip_factors", "dp_clipped_sum", "dp_add_noise",
            "dp_adaptive_bound", "dp_adaptive_bounds"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert dp.dp_abi_version() == 3


def test_planner_matches_golden_vgg11_decisions(dp):
    import workloads
    path = os.path.join(ROOT, "tests", "golden", "vgg11_cifar_decisions.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    wl = workloads.get_workload("vgg11_cifar_b1024")
    from helpers import desc_for
    names = {dp.DP_NORM_GHOST: "ghost", dp.DP_NORM_INSTANTIATE: "instantiate", dp.DP_NORM_T1: "t1"}
    for spec, row in zip(wl.layers, rows):
        m, T, D = dp.dp_plan(desc_for(dp, spec, wl.B, "bf16"))
        assert (names[m], T, D) == (row[6], int(row[1]), int(row[2]))


@pytest.mark.parametrize("name,mode", [("t1_linear_b32", "t1"), ("seq_linear_b64_t128", "ghost"),
                                       ("conv3x3_b256", "instantiate"), ("vit_mlp_b4096_t197", "ghost")])
def test_planner_on_workloads(dp, name, mode):
    import workloads
    from helpers import desc_for
    wl = workloads.get_workload(name)
    for spec in wl.layers:
        m, T, D = dp.dp_plan(desc_for(dp, spec, wl.B, wl.dtype))
        assert dp.MODE_NAMES[m] == mode and T == spec.rows and D == spec.D
        assert dp.dp_workspace_size(desc_for(dp, spec, wl.B, wl.dtype)) > 0


@pytest.mark.parametrize("name", ["t1_linear_b32", "seq_linear_b64_t128", "conv3x3_b256", "vgg11_cifar_b1024",
                                  "vit_mlp_b4096_t197"])
def test_speed_priority_plan_matches_oracle(dp, name):
    import oracle
    import workloads
    from helpers import desc_for
    wl = workloads.get_workload(name)
    for spec in wl.layers:
        m, T, D = dp.dp_plan(desc_for(dp, spec, wl.B, wl.dtype), dp.DP_NORM_AUTO_TIME)
        assert dp.MODE_NAMES[m] == oracle.dpsgd.norm_mode_plan_time(spec) and (T, D) == (spec.rows, spec.D)
        assert dp.dp_workspace_size(desc_for(dp, spec, wl.B, wl.dtype), dp.DP_NORM_AUTO_TIME) > 0


def test_speed_and_space_priority_part_ways(dp):
    d = dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=2, p=256, T=150, d=256)
    assert dp.dp_plan(d)[0] == dp.DP_NORM_GHOST
    assert dp.dp_plan(d, dp.DP_NORM_AUTO_TIME)[0] == dp.DP_NORM_INSTANTIATE


def test_ties_instantiate(dp):
    # 2T^2 == p*D: T=4 -> 32 = p*D with p=4, d=8
    d = dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=2, p=4, T=4, d=8)
    assert dp.dp_plan(d)[0] == dp.DP_NORM_INSTANTIATE
    d = dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=2, p=5, T=4, d=8)
    assert dp.dp_plan(d)[0] == dp.DP_NORM_GHOST


def test_conv_output_size(dp):
    d = dp.layer_desc(dp.DP_CONV2D, dp.DP_BF16, B=2, p=3, Cin=2, H=9, W=7, k=3, stride=2, pad=1, dil=2)
    _, T, D = dp.dp_plan(d, dp.DP_NORM_INSTANTIATE)
    Ho = (9 + 2 - 2 * 2 - 1) // 2 + 1
    Wo = (7 + 2 - 2 * 2 - 1) // 2 + 1
    assert (T, D) == (Ho * Wo, 2 * 9)


@pytest.mark.parametrize("kw", [
    dict(kind=0, dtype=0, B=0, p=4, T=2, d=3), dict(kind=0, dtype=0, B=2, p=0, T=2, d=3),
    dict(kind=0, dtype=7, B=2, p=4, T=2, d=3), dict(kind=5, dtype=0, B=2, p=4, T=2, d=3),
    dict(kind=0, dtype=0, B=2, p=4, T=0, d=3), dict(kind=1, dtype=0, B=2, p=4, Cin=2, H=2, W=2, k=5),
    dict(kind=1, dtype=0, B=2, p=4, Cin=2, H=8, W=8, k=3, stride=0),
    dict(kind=1, dtype=0, B=2, p=4, Cin=2, H=8, W=8, k=3, layout=2)])
def test_invalid_descriptors_rejected(dp, kw):
    d = dp.layer_desc(**kw)
    with pytest.raises(dp.DPError) as e:
        dp.dp_plan(d)
    assert e.value.status == dp.DP_ERR_INVALID_ARG
    assert dp.dp_workspace_size(d) == 0


def test_invalid_calls_launch_nothing(dp):
    d = dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=4, p=8, T=3, d=8)
    with pytest.raises(dp.DPError) as e:
        dp.dp_layer_sqnorms(d, 0, 0, 0, None, 0, stream=0)
    assert e.value.status == dp.DP_ERR_INVALID_ARG and "non-NULL" in str(e.value)
    d32 = dp.layer_desc(dp.DP_LINEAR, dp.DP_FP32, B=4, p=8, T=3, d=8)
    with pytest.raises(dp.DPError) as e:   # workspace too small (fp32 runs on the SIMT path)
        dp.dp_layer_sqnorms(d32, 16, 16, 16, 16, 1, mode=dp.DP_NORM_GHOST, stream=0)
    assert e.value.status == dp.DP_ERR_INVALID_ARG and "workspace" in str(e.value)
    with pytest.raises(dp.DPError) as e:
        dp.dp_plan(d, dp.DP_NORM_T1)
    assert e.value.status == dp.DP_ERR_INVALID_ARG
    nb = dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=4, p=8, T=3, d=8, has_bias=False)
    with pytest.raises(dp.DPError) as e:
        dp.dp_clipped_sum(nb, 16, 16, 16, 16, db=16, workspace=16, ws_bytes=1 << 30, stream=0)
    assert e.value.status == dp.DP_ERR_INVALID_ARG
    for C in ([0.0], [-1.0], [float("inf")]):
        with pytest.raises(dp.DPError) as e:
            dp.dp_clip_factors(16, 4, 1, False, C, 16, stream=0)
        assert e.value.status == dp.DP_ERR_INVALID_ARG
    with pytest.raises(dp.DPError):
        dp.dp_add_noise(16, 1.0, 1.0, 0, 0, 0, n=10, stream=0)
    with pytest.raises(dp.DPError):
        dp.dp_add_noise(16, -1.0, 1.0, 4, 0, 0, n=10, stream=0)
    dp.dp_add_noise(0, 1.0, 1.0, 4, 0, 0, n=0, stream=0)   # empty: no-op
    with pytest.raises(dp.DPError):
        dp.dp_adaptive_bound(16, 4, 0.0, 1.1, 2.0, 2.5, 0, 0, 16, stream=0)
    for kw in (dict(C_l2=[]), dict(C_l2=[1.0] * 65), dict(C_l2=[1.0, 0.0]), dict(C_l2=[float("nan")]),
               dict(C_l2=[1.0], layer0=-1)):
        with pytest.raises(dp.DPError) as e:
            dp.dp_adaptive_bounds(16, 4, kw.pop("C_l2"), 1.1, 2.0, 2.5, 0, 16, stream=0, **kw)
        assert e.value.status == dp.DP_ERR_INVALID_ARG


def test_invalid_noise_of_fused_sums_launches_nothing(dp):
    """The fused sum+noise calls check the noise descriptor before anything launches."""
    import ctypes
    d = dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=4, p=8, T=3, d=8)
    for nd in (dp.noise_desc(1.0, 1.0, 0), dp.noise_desc(-1.0, 1.0, 4), dp.noise_desc(1.0, float("nan"), 4),
               dp.noise_desc(float("inf"), 1.0, 4), dp.noise_desc(1.0, 1.0, 4, offset=2 ** 64 - 8)):
        with pytest.raises(dp.DPError) as e:
            dp.dp_clipped_sum_noised(d, 16, 16, 16, 16, 16, nd, workspace=16, ws_bytes=1 << 30, stream=0)
        assert e.value.status == dp.DP_ERR_INVALID_ARG
        with pytest.raises(dp.DPError) as e:
            dp.dp_clipped_sum_kept_noised(d, 16, 16, 16, 16, nd, workspace=16, ws_bytes=1 << 30, stream=0)
        assert e.value.status in (dp.DP_ERR_INVALID_ARG, dp.DP_ERR_UNSUPPORTED)
    ok = dp.noise_desc(1.0, 1.0, 4)
    with pytest.raises(dp.DPError) as e:
        dp.dp_clipped_sum_noised(d, 16, 16, 16, 16, 16, ok, workspace=16, ws_bytes=1 << 30, norm_mode=9, stream=0)
    assert e.value.status == dp.DP_ERR_INVALID_ARG
    st = dp._lib.dp_clipped_sum_noised(ctypes.byref(d), -1, 16, 16, 16, 16, 16, 0, None, 16, 1 << 30, None)
    assert st == dp.DP_ERR_INVALID_ARG and b"noise" in dp._lib.dp_last_error()


def test_invalid_noise_blocks_launch_nothing(dp):
    for blocks in ([], [(0, 10, 1.0)] * 65, [(0, 10, 1.0), (5, 10, 1.0)], [(0, 10, -1.0)],
                   [(0, 10, float("nan"))], [(2 ** 64 - 4, 8, 1.0)]):
        with pytest.raises(dp.DPError) as e:
            dp.dp_add_noise_blocks(16, blocks, 1.0, 4, stream=0)
        assert e.value.status == dp.DP_ERR_INVALID_ARG
    with pytest.raises(dp.DPError):
        dp.dp_add_noise_blocks(16, [(0, 10, 1.0)], 1.0, 0, stream=0)
    with pytest.raises(dp.DPError):
        dp.dp_add_noise_blocks(16, [(0, 10, 1.0)], -1.0, 4, stream=0)


def test_package_refuses_to_import_without_library(tmp_path):
    """The binding fails loudly when the compiled library is absent (no fallback)."""
    import shutil
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "example_gradient_clipping_gb300")
    dst = tmp_path / "example_gradient_clipping_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import example_gradient_clipping_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "not built" in r.stderr


def test_bench_step_work_counts():
    """bench.py's algorithmic counts (host only) for every workload and each conv kind."""
    import bench
    from workloads import WORKLOADS, LayerSpec, Workload
    for wl in WORKLOADS.values():
        for modes in (["ghost"] * len(wl.layers), ["instantiate"] * len(wl.layers)):
            w = bench.step_work(wl, modes)
            assert w["flop_sum"] == sum(wl.B * 2.0 * s.rows * s.p * s.D for s in wl.layers)
            assert w["in_bytes"] > 0 and w["bytes_total"] > w["in_bytes"]
    specs = (LayerSpec("c1", "conv1d", p=8, Cin=4, W=20, k=3, pad=1),
             LayerSpec("c3", "conv3d", p=8, Cin=2, Z=4, H=5, W=6, k=3, pad=1))
    wl = Workload(name="mixed", B=3, layers=specs, dtype="bf16", C=1.0, sigma=1.0)
    w = bench.step_work(wl, ["instantiate", "ghost"], kept=[True, False])
    assert w["in_bytes"] == 3 * 2 * (4 * 20 + 8 * 20 + 2 * 4 * 5 * 6 + 8 * 4 * 5 * 6)
    assert w["kept_bytes"] == 3 * (8 * 12 + 8) * 4
