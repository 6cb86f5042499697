"""Shared test helpers: descriptors from workload specs, tolerances, error measures."""
import numpy as np

import workloads

# Tolerances stated for this path: relative 1e-5 for fp32 inputs, 2e-2 for bf16
# inputs with fp32 accumulation.  Norms and factors: per element, relative to the
# element.  Sums: per element, relative to |ref| + rms of the reference over the
# element's row (a row of the weight gradient, or the whole bias vector), so that an
# entry near zero is held to the row's scale rather than to its own.
TOL = {"fp32": 1e-5, "bf16": 2e-2}
# Normal draws against the oracle's float64 Box-Muller: the kernels take the angle's sine and
# cosine from the fp32 hardware approximations (absolute error about 2^-21.4 on [-pi, pi], plus
# ~2e-7 from rounding the fp32 argument), times a radius below sqrt(-2 ln 2^-24) = 5.8: under
# 4e-6 absolute; the radius itself is within a few ulp (relative).
Z_RTOL, Z_ATOL = 1e-5, 4e-6


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


def rel_rows(x, ref, row_len=None):
    """Largest element-wise error max_k |x_k - ref_k| / (|ref_k| + rms_k), rms_k the root
    mean square of ref over the row (row_len consecutive elements) holding k, or over the
    whole vector when row_len is None."""
    x = np.asarray(x, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    if not np.all(np.isfinite(x)):
        return float("inf")
    n = row_len if row_len else ref.size
    X, R = x.reshape(-1, n), ref.reshape(-1, n)
    rms = np.sqrt(np.mean(R * R, axis=1, keepdims=True))
    den = np.abs(R) + rms
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.abs(X - R) / den))


def rel_flat(g, ref, specs):
    """rel_rows over a flat gradient [W_0, b_0, W_1, b_1, ...] of layers `specs`: the rows of
    each weight block ([p, D]) and each bias block, each against its own rms."""
    g = np.asarray(g, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    assert g.shape == ref.shape
    worst, o = 0.0, 0
    for s in specs:
        n = s.p * s.D
        worst = max(worst, rel_rows(g[o:o + n], ref[o:o + n], s.D))
        o += n
        if s.has_bias:
            worst = max(worst, rel_rows(g[o:o + s.p], ref[o:o + s.p]))
            o += s.p
    assert o == g.size
    return worst


def rel_elem(x, ref):
    x = np.asarray(x, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    return float(np.max(np.abs(x - ref) / np.maximum(np.abs(ref), 1e-30))) if ref.size else 0.0
