"""GPU parity of stride-1 "same" conv layers over 64 input channels with at most 64 outputs
(k = 1 or 3), whose instantiated norm forms each example's gradient from shifted views of one
output-gradient tile (the filter rows, paired on M) and one input tile (the filter columns, on
N), over the output pixels laid out in padded rows.

Cases: the 3x3 workload's layer (32x32, 64 outputs), outputs not a multiple of 32 (p = 40, 56)
or below 32, dilation 2, a 1x1 kernel, odd image widths, tiny images, no bias, many examples,
channels-last inputs, and a 128-output layer (the im2col kernels).  Every case meets the float64
oracle element by element: the norms, the kept per-example gradients (the conv tile column
order: tap * 64 + channel), the clipped sum formed from them, and a clipped sum that reuses the
norm call's NHWC copy.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import TOL, desc_for, rel_elem, rel_rows, to_dev, to_dev_channels_last
from workloads import LayerSpec, Workload

pytestmark = pytest.mark.gpu

CASES = [
    ("conv3x3_p64_32x32", LayerSpec("e", "conv2d", p=64, Cin=64, H=32, W=32, k=3, pad=1), 3, False),
    ("p16_nobias", LayerSpec("e", "conv2d", p=16, Cin=64, H=8, W=8, k=3, pad=1, has_bias=False), 5, False),
    ("p40_5x7", LayerSpec("e", "conv2d", p=40, Cin=64, H=5, W=7, k=3, pad=1), 3, False),
    ("p56_12x10", LayerSpec("e", "conv2d", p=56, Cin=64, H=12, W=10, k=3, pad=1), 4, False),
    ("p24_dil2", LayerSpec("e", "conv2d", p=24, Cin=64, H=14, W=13, k=3, pad=2, dil=2), 2, False),
    ("p64_dil2", LayerSpec("e", "conv2d", p=64, Cin=64, H=9, W=11, k=3, pad=2, dil=2), 2, False),
    ("k1_pointwise", LayerSpec("e", "conv2d", p=64, Cin=64, H=9, W=14, k=1, pad=0), 3, False),
    ("tiny_2x3", LayerSpec("e", "conv2d", p=32, Cin=64, H=2, W=3, k=3, pad=1), 4, False),
    ("B301", LayerSpec("e", "conv2d", p=64, Cin=64, H=6, W=6, k=3, pad=1), 301, False),
    ("nhwc_p64", LayerSpec("e", "conv2d", p=64, Cin=64, H=16, W=16, k=3, pad=1), 3, True),
    ("nhwc_p48_nobias", LayerSpec("e", "conv2d", p=48, Cin=64, H=10, W=11, k=3, pad=1, has_bias=False), 2, True),
    ("p128_im2col", LayerSpec("e", "conv2d", p=128, Cin=64, H=16, W=16, k=3, pad=1), 2, False),
]


def _tile_to_weight(kept, spec, quad):
    """Kept rows -> the weight layout [B, p, 64 * k*k]: tile columns col = tap * 64 + c, stored
    [B, p, col] or, with `quad` (the shifted-tile kernel), column-quad major [B, col / 4, p, 4]."""
    B, kk = kept.shape[0], spec.k * spec.k
    if quad:
        kept = kept.reshape(B, kk * 16, spec.p, 4).transpose(0, 2, 1, 3)
    return kept.reshape(B, spec.p, kk, spec.Cin).transpose(0, 1, 3, 2).reshape(B, spec.p, -1)


@pytest.mark.parametrize("tag,spec,B,nhwc", CASES, ids=[c[0] for c in CASES])
def test_shifted_tile_norms_kept_and_sum(lib, tag, spec, B, nhwc):
    import torch
    dp = lib
    wl = Workload(name=tag, B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=37)
    A, G = workloads.layer_inputs(wl, 0)
    fac = workloads.factor_inputs(wl, B, 0.1, 1.0)
    desc = desc_for(dp, spec, B, "bf16", layout=dp.DP_NHWC if nhwc else 0)
    move = to_dev_channels_last if nhwc else to_dev
    Ad, Gd = move(A, "bf16"), move(G, "bf16")
    f = torch.tensor(fac, device="cuda")
    tol = TOL["bf16"]
    s_ref = oracle.layer_sqnorms(spec, A, G)
    S, Sb = oracle.clipped_sum(spec, A, G, fac.astype(np.float64))
    ws = torch.empty(max(dp.dp_workspace_size(desc, dp.DP_NORM_INSTANTIATE), 16), dtype=torch.uint8, device="cuda")

    sq = torch.full((B,), float("nan"), device="cuda")
    dp.dp_layer_sqnorms(desc, Ad, Gd, sq, ws, mode=dp.DP_NORM_INSTANTIATE)
    torch.cuda.synchronize()
    assert rel_elem(sq.cpu().numpy(), s_ref) <= tol

    # the clipped sum that reuses the norm call's NHWC copy
    dW = torch.full((spec.p * spec.D,), float("nan"), device="cuda")
    db = torch.full((spec.p,), float("nan"), device="cuda") if spec.has_bias else None
    dp.dp_clipped_sum_reuse(desc, dp.DP_NORM_INSTANTIATE, Ad, Gd, f, dW, db, ws)
    torch.cuda.synchronize()
    assert rel_rows(dW.cpu().numpy(), S, spec.D) <= tol
    if spec.has_bias:
        assert rel_rows(db.cpu().numpy(), Sb) <= tol

    # kept gradients (tile column order) and the clipped sum from them
    nbytes = dp.dp_grads_size(desc)
    assert nbytes == 4 * B * spec.p * spec.D + (4 * B * spec.p if spec.has_bias else 0)
    grads = torch.full((nbytes // 4,), float("nan"), device="cuda")
    sq = torch.full((B,), float("nan"), device="cuda")
    dp.dp_layer_sqnorms_keep(desc, Ad, Gd, sq, grads, ws)
    torch.cuda.synchronize()
    assert rel_elem(sq.cpu().numpy(), s_ref) <= tol
    kept = _tile_to_weight(grads[: B * spec.p * spec.D].view(B, -1).cpu().numpy(), spec, quad=spec.p <= 64)
    kb = grads[B * spec.p * spec.D:].view(B, spec.p).cpu().numpy() if spec.has_bias else None
    for i in range(0, B, max(1, B // 6)):
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


def test_shifted_tile_and_im2col_kernels_agree(lib, monkeypatch):
    """The 3x3 workload's layer: norms of the shifted-tile kernel and of the im2col kernel
    (DPCLIP_CONV=im2col) agree with each other and with the oracle."""
    import torch
    dp = lib
    wl = workloads.get_workload("conv3x3_b256").with_batch(6)
    spec = wl.layers[0]
    A, G = workloads.layer_inputs(wl, 0)
    desc = desc_for(dp, spec, wl.B, "bf16")
    Ad, Gd = to_dev(A, "bf16"), to_dev(G, "bf16")
    out = []
    for pin in ("", "im2col"):
        if pin:
            monkeypatch.setenv("DPCLIP_CONV", pin)
        ws = torch.empty(dp.dp_workspace_size(desc, dp.DP_NORM_INSTANTIATE), dtype=torch.uint8, device="cuda")
        sq = torch.empty(wl.B, device="cuda")
        dp.dp_layer_sqnorms(desc, Ad, Gd, sq, ws, mode=dp.DP_NORM_INSTANTIATE)
        torch.cuda.synchronize()
        out.append(sq.cpu().numpy())
    s_ref = oracle.layer_sqnorms(spec, A, G)
    for o in out:
        assert rel_elem(o, s_ref) <= TOL["bf16"]
