"""GPU parity of conv layers whose A and G arrive channels last (DP_NHWC).

The oracle works on the channels-first arrays; the device gets the same values as
contiguous channels-last tensors ([B, H, W, C], [B, L, C], [B, Z, H, W, C]) with a
descriptor saying so.  Cases cover every conv path: the TMA im2col kernels (ghost norm,
per-example instantiation with the output gradient transposed back to [p, T], the
row-scaled sum with the output-gradient rows scaled in place), the row layout (the
shared-memory and the global unfold, padded widths), the FFMA kernels, 1-D and 3-D
convolutions, kept per-example gradients and a whole step.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import TOL, desc_for, rel_elem, rel_flat, rel_rows, to_dev_channels_last
from workloads import LayerSpec, Workload

pytestmark = pytest.mark.gpu

CASES = [
    ("im2col_T144", LayerSpec("e", "conv2d", p=72, Cin=64, H=12, W=12, k=3, pad=1), 3, "bf16"),
    ("im2col_T64_rowscaled", LayerSpec("e", "conv2d", p=64, Cin=64, H=8, W=8, k=3, pad=1), 4, "bf16"),
    ("im2col_s2_dil2_nobias", LayerSpec("e", "conv2d", p=136, Cin=128, H=23, W=23, k=3, stride=2, pad=2, dil=2,
                                        has_bias=False), 2, "bf16"),
    ("rows_smem", LayerSpec("e", "conv2d", p=64, Cin=16, H=12, W=12, k=3, pad=1), 4, "bf16"),
    ("rows_padD", LayerSpec("e", "conv2d", p=64, Cin=9, H=12, W=12, k=3, pad=1), 4, "bf16"),
    ("unfold_on_chip", LayerSpec("e", "conv2d", p=64, Cin=3, H=12, W=12, k=3, pad=1), 4, "bf16"),
    ("rows_global_unfold", LayerSpec("e", "conv2d", p=16, Cin=48, H=48, W=48, k=3, pad=1), 2, "bf16"),
    ("ffma_bf16", LayerSpec("e", "conv2d", p=6, Cin=5, H=9, W=8, k=3, stride=2, pad=1), 3, "bf16"),
    ("ffma_fp32", LayerSpec("e", "conv2d", p=4, Cin=3, H=10, W=10, k=3, pad=2, dil=2), 2, "fp32"),
    ("conv1d_rows", LayerSpec("e", "conv1d", p=16, Cin=8, W=50, k=5, stride=2, pad=2), 4, "bf16"),
    ("conv3d_rows", LayerSpec("e", "conv3d", p=16, Cin=4, Z=6, H=7, W=8, k=3, pad=1), 3, "bf16"),
]


def _inputs(tag, spec, B, dtype):
    wl = Workload(name=tag, B=B, layers=(spec,), dtype=dtype, C=1.0, sigma=1.0, seed=23)
    A, G = workloads.layer_inputs(wl, 0)
    return wl, A, G


@pytest.mark.parametrize("tag,spec,B,dtype", CASES, ids=[c[0] for c in CASES])
def test_channels_last_norms_and_sums(lib, tag, spec, B, dtype):
    import torch
    dp = lib
    wl, A, G = _inputs(tag, spec, B, dtype)
    desc = desc_for(dp, spec, B, dtype, layout=dp.DP_NHWC)
    Ad, Gd = to_dev_channels_last(A, dtype), to_dev_channels_last(G, dtype)
    fac = workloads.factor_inputs(wl, B, 0.1, 1.0)
    f = torch.tensor(fac, device="cuda")
    s_ref = oracle.layer_sqnorms(spec, A, G)
    S, Sb = oracle.clipped_sum(spec, A, G, fac.astype(np.float64))
    tol = TOL[dtype]
    for mode in (dp.DP_NORM_AUTO, dp.DP_NORM_GHOST, dp.DP_NORM_INSTANTIATE):
        ws = torch.empty(max(dp.dp_workspace_size(desc, mode), 16), dtype=torch.uint8, device="cuda")
        sq = torch.empty(B, dtype=torch.float32, device="cuda")
        dp.dp_layer_sqnorms(desc, Ad, Gd, sq, ws, mode=mode)
        dW = torch.full((spec.p * spec.D,), float("nan"), device="cuda")
        db = torch.full((spec.p,), float("nan"), device="cuda") if spec.has_bias else None
        dp.dp_clipped_sum(desc, Ad, Gd, f, dW, db, ws)
        torch.cuda.synchronize()
        assert rel_elem(sq.cpu().numpy(), s_ref) <= tol, mode
        assert rel_rows(dW.cpu().numpy(), S, spec.D) <= tol, mode
        if spec.has_bias:
            assert rel_rows(db.cpu().numpy(), Sb) <= tol, mode
    # nothing to share between the norm and sum calls: no layout copy is made
    assert dp.dp_layout_reused(desc, dp.DP_NORM_AUTO) == 0


@pytest.mark.parametrize("tag,spec,B", [
    ("im2col_T144", LayerSpec("e", "conv2d", p=72, Cin=64, H=12, W=12, k=3, pad=1), 3),
    ("rows_padD", LayerSpec("e", "conv2d", p=64, Cin=9, H=12, W=12, k=3, pad=1), 4),
    ("unfold_on_chip", LayerSpec("e", "conv2d", p=64, Cin=3, H=12, W=12, k=3, pad=1), 4)])
def test_channels_last_kept_gradients(lib, tag, spec, B):
    import torch
    dp = lib
    wl, A, G = _inputs(tag, spec, B, "bf16")
    desc = desc_for(dp, spec, B, "bf16", layout=dp.DP_NHWC)
    Ad, Gd = to_dev_channels_last(A, "bf16"), to_dev_channels_last(G, "bf16")
    nbytes = dp.dp_grads_size(desc)
    assert nbytes > 0
    grads = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    ws = torch.empty(dp.dp_workspace_size(desc, dp.DP_NORM_INSTANTIATE), dtype=torch.uint8, device="cuda")
    sq = torch.empty(B, dtype=torch.float32, device="cuda")
    dp.dp_layer_sqnorms_keep(desc, Ad, Gd, sq, grads, ws)
    fac = workloads.factor_inputs(wl, B, 0.1, 1.0)
    dW = torch.empty(spec.p * spec.D, device="cuda")
    db = torch.empty(spec.p, device="cuda")
    dp.dp_clipped_sum_kept(desc, grads, torch.tensor(fac, device="cuda"), dW, db, ws)
    torch.cuda.synchronize()
    assert rel_elem(sq.cpu().numpy(), oracle.layer_sqnorms(spec, A, G)) <= TOL["bf16"]
    S, Sb = oracle.clipped_sum(spec, A, G, fac.astype(np.float64))
    assert rel_rows(dW.cpu().numpy(), S, spec.D) <= TOL["bf16"]
    assert rel_rows(db.cpu().numpy(), Sb) <= TOL["bf16"]


def test_channels_last_step_equals_channels_first(lib):
    """A three-layer step (im2col ghost, im2col instantiation, row layout) through ClipStep:
    channels-last inputs give the oracle's step, and the channels-first step within tolerance."""
    import torch
    dp = lib
    specs = (LayerSpec("a", "conv2d", p=64, Cin=64, H=8, W=8, k=3, pad=1),
             LayerSpec("b", "conv2d", p=72, Cin=64, H=12, W=12, k=3, pad=1),
             LayerSpec("c", "conv2d", p=64, Cin=3, H=12, W=12, k=3, pad=1))
    wl = Workload(name="cl", B=4, layers=specs, dtype="bf16", C=1.0, sigma=0.7, seed=29)
    inputs = [workloads.layer_inputs(wl, l) for l in range(3)]
    grads = []
    for layout in (dp.DP_NCHW, dp.DP_NHWC):
        descs = [desc_for(dp, s, wl.B, "bf16", layout=layout) for s in specs]
        conv = (lambda x: workloads.to_torch(x, "bf16", "cuda")) if layout == dp.DP_NCHW else \
            (lambda x: to_dev_channels_last(x, "bf16"))
        dev = [(conv(A), conv(G)) for A, G in inputs]
        st = dp.ClipStep(descs, C=wl.C, sigma=wl.sigma)
        grads.append(st.run(dev, seed=5).double().cpu().numpy())
    ref = oracle.dp_step(wl, inputs, seed=5)
    assert rel_flat(grads[1], ref["noisy"], specs) <= TOL["bf16"]
    assert rel_flat(grads[1], grads[0], specs) <= TOL["bf16"]
