"""bench.py as the driver runs it: one JSON line with the keys the measurement contract names.

The reference arm (the float64 oracle on the host cores) runs here without a GPU; our arm
runs on the GPU with a short step count.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config", "e2e"}


def _run(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--steps", "1", "--warmup", "3", "--workload", "t1_linear_b32"], 300)
    assert BASE_KEYS <= set(d) and d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "examples/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "t1_linear_b32" and d["warmup"] >= 3
    assert d["e2e"] == {"value": d["value"], "unit": "examples/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]


@pytest.mark.gpu
def test_bench_line_keys():
    """The default run: the ViT-Base MLP pair at B=4096 as the headline, the other
    workloads under per_config."""
    d = _run(["--steps", "3", "--warmup", "3", "--no-cpu-baseline"], 1200)
    assert BASE_KEYS <= set(d) and {"roofline", "clocks", "gpu_launches", "per_config"} <= set(d)
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] >= 3
    assert d["config"]["workload"] == "vit_mlp_b4096_t197" and d["data"] == "synthetic"
    r = d["roofline"]
    assert r["bound"] == "tensor" and 0 < r["frac"] < 1.5 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    # the dominant call's achieved rate recomputes from its FLOP count and its mean time
    flop = {"dp_clipped_sum": 2 * 4096 * 197 * 3072 * 768 * 2}.get(r["kernel"])
    if flop is not None:
        assert abs(flop / (d["calls_ms"]["sums"] * 1e-3) / 1e12 - r["achieved"]) <= 1e-3 * r["achieved"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 4096 * 197 * (768 + 3072) * 2 * 2
    assert e["d2h_bytes_per_step"] == 4 * (3072 * 768 + 3072 + 768 * 3072 + 768)
    assert d["gpu_launches"] == 3 * d["kernels_per_step"] > 0
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    pc = d["per_config"]
    assert set(pc) == {"t1_linear_b32", "seq_linear_b64_t128", "conv3x3_b256", "vgg11_cifar_b1024",
                       "vgg11_cifar_b1024_flat", "conv3x3_b256/channels_last", "vgg11_cifar_b1024/channels_last"}
    for name, c in pc.items():
        assert c["value"] > 0 and c["ms_per_step"] > 0 and c["roofline"]["frac"] > 0, name
        assert c["conv_layout"] == ("channels last" if name.endswith("/channels_last") else "channels first"), name
    assert pc["vgg11_cifar_b1024"]["kernels_per_step"] > pc["vgg11_cifar_b1024_flat"]["kernels_per_step"]


@pytest.mark.gpu
def test_bench_line_small_workload():
    d = _run(["--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--workload", "seq_linear_b64_t128"], 600)
    assert d["config"]["workload"] == "seq_linear_b64_t128" and "per_config" not in d
    assert d["e2e"]["h2d_bytes_per_step"] == 2 * 64 * 128 * 768 * 2


def test_traffic_records_match_call_kernel_batch_and_source(tmp_path, monkeypatch):
    """roofline.traffic comes from a record only for the dominant call's kernel at the batch
    the record states, while the kernel's source is the one captured; else it is null."""
    sys.path.insert(0, ROOT)
    import bench
    src_dir = tmp_path / "example_gradient_clipping_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (src_dir / "k.cu").write_bytes(b"kernel source")
    import hashlib
    h = hashlib.sha256(b"kernel source").hexdigest()[:16]
    rec = dict(workload="w", call="sums", kernel="kern", source="k.cu", source_sha256_16=h, B=64,
               dram_bytes_per_launch=1234)
    (tmp_path / "traffic.json").write_text(json.dumps({"records": [rec]}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "traffic.json"))
    assert bench._profiled_traffic("w", "sums", ["kern"], 64) == 1234
    assert bench._profiled_traffic("w", "norms", ["kern"], 64) is None      # another call
    assert bench._profiled_traffic("w", "sums", ["other"], 64) is None      # another kernel
    assert bench._profiled_traffic("w", "sums", ["kern"], 128) is None      # another batch
    assert bench._profiled_traffic("v", "sums", ["kern"], 64) is None       # another workload
    (src_dir / "k.cu").write_bytes(b"kernel source, edited")
    assert bench._profiled_traffic("w", "sums", ["kern"], 64) is None      # the source changed
