"""GPU parity of narrow conv layers (unfolded width plus bias at most 64) whose unfold the
kernel forms on chip from the example's input, reading the output gradient as it lies.

Cases: 3x3 over three channels (the first layer of VGG-11 on CIFAR, 8-pixel windows read
from padded input rows), 5x5 filling all 64 columns with the bias, stride 2 and dilation
(per-element gathers), odd widths (scalar input loads), more than 128 outputs (two output
tiles), ragged pixel chunks, many examples (ragged example splits), conv1d, no bias, and
channels-last inputs.  Every case meets the float64 oracle element by element: the norms in
both the automatic and the forced instantiated mode, the clipped sum with dense factors,
its accumulation, the kept per-example gradients and the clipped sum formed from them.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import TOL, desc_for, rel_elem, rel_rows, to_dev, to_dev_channels_last
from workloads import LayerSpec, Workload

pytestmark = pytest.mark.gpu

CASES = [
    ("rgb3x3_p64_B5", LayerSpec("e", "conv2d", p=64, Cin=3, H=32, W=32, k=3, pad=1), 5, False),
    ("rgb3x3_nobias", LayerSpec("e", "conv2d", p=64, Cin=3, H=16, W=16, k=3, pad=1, has_bias=False), 3, False),
    ("c2_5x5_full64", LayerSpec("e", "conv2d", p=24, Cin=2, H=16, W=16, k=5, pad=2), 4, False),
    ("s2_gather", LayerSpec("e", "conv2d", p=40, Cin=3, H=15, W=15, k=3, stride=2, pad=1), 3, False),
    ("dil2_oddW", LayerSpec("e", "conv2d", p=16, Cin=2, H=8, W=13, k=3, pad=2, dil=2), 3, False),
    ("p200_two_tiles", LayerSpec("e", "conv2d", p=200, Cin=3, H=8, W=8, k=3, pad=1), 3, False),
    ("T160_ragged_chunk", LayerSpec("e", "conv2d", p=16, Cin=3, H=10, W=16, k=3, pad=1), 7, False),
    ("B301_splits", LayerSpec("e", "conv2d", p=64, Cin=3, H=8, W=8, k=3, pad=1), 301, False),
    ("conv1d_k5", LayerSpec("e", "conv1d", p=32, Cin=4, W=64, k=5, pad=2), 4, False),
    ("nhwc_rgb3x3", LayerSpec("e", "conv2d", p=64, Cin=3, H=16, W=16, k=3, pad=1), 4, True),
    ("nhwc_p72_s2", LayerSpec("e", "conv2d", p=72, Cin=3, H=11, W=11, k=3, stride=2, pad=1, has_bias=False), 3,
     True),
]


@pytest.mark.parametrize("tag,spec,B,nhwc", CASES, ids=[c[0] for c in CASES])
def test_unfold_norms_sums_and_kept(lib, tag, spec, B, nhwc):
    import torch
    dp = lib
    wl = Workload(name=tag, B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=29)
    A, G = workloads.layer_inputs(wl, 0)
    fac = workloads.factor_inputs(wl, B, 0.1, 1.0)
    desc = desc_for(dp, spec, B, "bf16", layout=dp.DP_NHWC if nhwc else 0)
    move = to_dev_channels_last if nhwc else to_dev
    Ad, Gd = move(A, "bf16"), move(G, "bf16")
    f = torch.tensor(fac, device="cuda")
    tol = TOL["bf16"]
    s_ref = oracle.layer_sqnorms(spec, A, G)
    S, Sb = oracle.clipped_sum(spec, A, G, fac.astype(np.float64))

    for mode in (dp.DP_NORM_AUTO, dp.DP_NORM_INSTANTIATE):
        ws = torch.empty(max(dp.dp_workspace_size(desc, mode), 16), dtype=torch.uint8, device="cuda")
        sq = torch.full((B,), float("nan"), device="cuda")
        dp.dp_layer_sqnorms(desc, Ad, Gd, sq, ws, mode=mode)
        torch.cuda.synchronize()
        assert rel_elem(sq.cpu().numpy(), s_ref) <= tol, mode

    ws = torch.empty(max(dp.dp_workspace_size(desc, dp.DP_NORM_INSTANTIATE), 16), dtype=torch.uint8, device="cuda")
    dW = torch.full((spec.p * spec.D,), float("nan"), device="cuda")
    db = torch.full((spec.p,), float("nan"), device="cuda") if spec.has_bias else None
    dp.dp_clipped_sum(desc, Ad, Gd, f, dW, db, ws)
    torch.cuda.synchronize()
    assert rel_rows(dW.cpu().numpy(), S, spec.D) <= tol
    if spec.has_bias:
        assert rel_rows(db.cpu().numpy(), Sb) <= tol
    dp.dp_clipped_sum(desc, Ad, Gd, f, dW, db, ws, accumulate=True)
    torch.cuda.synchronize()
    assert rel_rows(dW.cpu().numpy(), 2 * S, spec.D) <= tol
    if spec.has_bias:
        assert rel_rows(db.cpu().numpy(), 2 * Sb) <= tol

    # kept gradients: the weight layout [p, D] (no padded columns) and the bias [p]
    nbytes = dp.dp_grads_size(desc)
    assert nbytes == 4 * B * spec.p * spec.D + (4 * B * spec.p if spec.has_bias else 0)
    grads = torch.full((nbytes // 4,), float("nan"), device="cuda")
    sq = torch.full((B,), float("nan"), device="cuda")
    dp.dp_layer_sqnorms_keep(desc, Ad, Gd, sq, grads, ws)
    torch.cuda.synchronize()
    assert rel_elem(sq.cpu().numpy(), s_ref) <= tol
    kept = grads[: B * spec.p * spec.D].view(B, spec.p, spec.D).cpu().numpy()
    kb = grads[B * spec.p * spec.D:].view(B, spec.p).cpu().numpy() if spec.has_bias else None
    for i in range(0, B, max(1, B // 8)):      # a spread of examples (all of them when B <= 8)
        gw, gb = oracle.per_example_grad(spec, A[i], G[i])
        assert rel_rows(kept[i], gw, spec.D) <= tol, i
        if spec.has_bias:
            assert rel_rows(kb[i], gb) <= tol, i
    dW2 = torch.full((spec.p * spec.D,), float("nan"), device="cuda")
    db2 = torch.full((spec.p,), float("nan"), device="cuda") if spec.has_bias else None
    dp.dp_clipped_sum_kept(desc, grads, f, dW2, db2, ws)
    torch.cuda.synchronize()
    assert rel_rows(dW2.cpu().numpy(), S, spec.D) <= tol
    if spec.has_bias:
        assert rel_rows(db2.cpu().numpy(), Sb) <= tol


def test_unfold_noised_sum_matches_sum_then_noise(lib):
    """The noised clipped sum (noise drawn in the split reduction) against the clipped sum
    followed by the separate noise pass over the same flat offsets."""
    import torch
    dp = lib
    spec = LayerSpec("e", "conv2d", p=64, Cin=3, H=16, W=16, k=3, pad=1)
    B = 200
    wl = Workload(name="unf_noise", B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=31)
    A, G = workloads.layer_inputs(wl, 0)
    desc = desc_for(dp, spec, B, "bf16")
    Ad, Gd = to_dev(A, "bf16"), to_dev(G, "bf16")
    f = torch.tensor(workloads.factor_inputs(wl, B, 0.1, 1.0), device="cuda")
    ws = torch.empty(max(dp.dp_workspace_size(desc), 16), dtype=torch.uint8, device="cuda")
    flat = torch.empty(spec.p * spec.D + spec.p, device="cuda")
    dW, db = flat[: spec.p * spec.D], flat[spec.p * spec.D:]
    nd = dp.noise_desc(0.8, 1.5, B, seed=1234, offset=96)
    dp.dp_clipped_sum_noised(desc, Ad, Gd, f, dW, db, nd, ws)
    ref = torch.empty_like(flat)
    dp.dp_clipped_sum(desc, Ad, Gd, f, ref[: spec.p * spec.D], ref[spec.p * spec.D:], ws)
    dp.dp_add_noise(ref, 0.8, 1.5, B, 1234, offset=96)
    torch.cuda.synchronize()
    assert torch.equal(flat, ref)
