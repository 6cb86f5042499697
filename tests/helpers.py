"""Shared test helpers: descriptors from workload specs, tolerances, error measures."""
import numpy as np

import workloads

# Tolerances stated for this path: relative 1e-5 for fp32 inputs, 2e-2 for bf16
# inputs with fp32 accumulation (norms and factors per element; sums per vector).
TOL = {"fp32": 1e-5, "bf16": 2e-2}
# Normal draws: libm/CUDA transcendentals differ in the last bits.
Z_RTOL, Z_ATOL = 1e-5, 1e-6


def desc_for(dp, spec, B, dtype, layout=0):
    dt = dp.DP_BF16 if dtype == "bf16" else dp.DP_FP32
    if spec.kind == "linear":
        return dp.layer_desc(dp.DP_LINEAR, dt, B=B, p=spec.p, T=spec.T, d=spec.d, has_bias=spec.has_bias)
    if spec.kind == "conv3d":
        return dp.layer_desc(dp.DP_CONV3D, dt, B=B, p=spec.p, Cin=spec.Cin, Z=spec.Z, H=spec.H, W=spec.W, k=spec.k,
                             stride=spec.stride, pad=spec.pad, dil=spec.dil, has_bias=spec.has_bias, layout=layout)
    if spec.kind == "conv1d":
        return dp.layer_desc(dp.DP_CONV1D, dt, B=B, p=spec.p, Cin=spec.Cin, H=1, W=spec.W, k=spec.k,
                             stride=spec.stride, pad=spec.pad, dil=spec.dil, has_bias=spec.has_bias, layout=layout)
    return dp.layer_desc(dp.DP_CONV2D, dt, B=B, p=spec.p, Cin=spec.Cin, H=spec.H, W=spec.W, k=spec.k,
                         stride=spec.stride, pad=spec.pad, dil=spec.dil, has_bias=spec.has_bias, layout=layout)


def to_dev(x, dtype):
    return workloads.to_torch(x, dtype, "cuda")


def to_dev_channels_last(x, dtype):
    """A channels-first array [B, C, ...] as a contiguous channels-last device tensor [B, ..., C]."""
    return to_dev(x, dtype).movedim(1, -1).contiguous()


def rel_vec(x, ref):
    x = np.asarray(x, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def rel_elem(x, ref):
    x = np.asarray(x, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    return float(np.max(np.abs(x - ref) / np.maximum(np.abs(ref), 1e-30))) if ref.size else 0.0
