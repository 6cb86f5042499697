"""The clipped sum and the noise in one call (dp_clipped_sum_noised and its kept form).

The fused call must equal the clipped sum followed by dp_add_noise on the layer's blocks
bit for bit: the noise of element e is drawn at its flat index e in both, and the final
pass applies the same (x + sigma C z_e) / B.  Cases cover the sum paths that end in a
reduction of example splits (the noise then rides in that pass: no extra launch) and those
that do not (a noise pass follows inside the call), a misaligned flat offset, no bias
output, accumulation, the device-side seed, and whole steps through ClipStep and its graph.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import TOL, desc_for, rel_flat, to_dev, to_dev_channels_last
from workloads import LayerSpec, Workload

pytestmark = pytest.mark.gpu

CASES = [
    # (name, spec, B, dtype, channels last, fused into the sum's final reductions)
    ("seq_linear_b64_t128", None, 64, "bf16", False, True),
    ("t1_fp32_splits", LayerSpec("e", "linear", p=40, d=36, T=1), 100, "fp32", False, True),
    ("lin_rowscaled", LayerSpec("e", "linear", p=128, d=64, T=40), 5, "bf16", False, True),
    ("conv_rows", LayerSpec("e", "conv2d", p=64, Cin=16, H=12, W=12, k=3, pad=1), 5, "bf16", False, True),
    # im2col conv sums: the bias gets its noise in its reduction, the weights in a noise pass
    ("conv_im2col", LayerSpec("e", "conv2d", p=72, Cin=64, H=12, W=12, k=3, pad=1), 3, "bf16", False, False),
    ("conv_im2col_rowscaled", LayerSpec("e", "conv2d", p=64, Cin=64, H=8, W=8, k=3, pad=1), 4, "bf16", False, False),
    ("conv_im2col_rowscaled_cl", LayerSpec("e", "conv2d", p=64, Cin=64, H=8, W=8, k=3, pad=1), 4, "bf16", True,
     False),
    # padded unfolded width: the weights get their noise after the compaction
    ("conv_rows_padD", LayerSpec("e", "conv2d", p=64, Cin=9, H=12, W=12, k=3, pad=1), 4, "bf16", False, False),
    # on-chip unfold of a narrow conv layer: fused with example splits, a noise pass with one
    ("conv_unfold", LayerSpec("e", "conv2d", p=64, Cin=3, H=12, W=12, k=3, pad=1), 4, "bf16", False, True),
    ("conv_unfold_one_split", LayerSpec("e", "conv2d", p=64, Cin=3, H=16, W=16, k=3, pad=1), 1, "bf16", False,
     False),
    ("ffma_small", LayerSpec("e", "linear", p=6, d=10, T=5), 4, "fp32", False, False),
]


def _case(name, spec, B, dtype):
    if spec is None:
        wl = workloads.get_workload(name)
    else:
        wl = Workload(name=name, B=B, layers=(spec,), dtype=dtype, C=1.0, sigma=1.0, seed=17)
    spec = wl.layers[0]
    A, G = workloads.layer_inputs(wl, 0)
    fac = workloads.factor_inputs(wl, wl.B, 0.2, 1.0)
    return wl, spec, A, G, fac


@pytest.mark.parametrize("name,spec,B,dtype,cl,fused", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("offset,accumulate,with_db", [(0, 0, True), (3, 1, True), (6, 0, False)])
def test_fused_equals_sum_then_noise(lib, name, spec, B, dtype, cl, fused, offset, accumulate, with_db):
    import torch
    dp = lib
    wl, spec, A, G, fac = _case(name, spec, B, dtype)
    desc = desc_for(dp, spec, wl.B, wl.dtype, layout=dp.DP_NHWC if cl else dp.DP_NCHW)
    p, D = spec.p, spec.D
    conv = to_dev_channels_last if cl else to_dev
    dA, dG = conv(A, wl.dtype), conv(G, wl.dtype)
    f = torch.tensor(fac, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(dp.dp_workspace_size(desc, dp.DP_NORM_AUTO), 16), dtype=torch.uint8, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    init = torch.randn(p * D + p, generator=gen, device="cuda") if accumulate else None
    sigma, C, Bdiv, seed = 0.7, 1.3, wl.B + 3, 0xC0FFEE + offset
    outs = []
    for mode in ("two_calls", "fused"):
        flat = init.clone() if accumulate else torch.full((p * D + p,), float("nan"), device="cuda")
        dW, db = flat[:p * D], (flat[p * D:] if (with_db and spec.has_bias) else None)
        n0 = dp.dp_launch_count()
        if mode == "two_calls":
            dp.dp_clipped_sum(desc, dA, dG, f, dW, db, ws, accumulate=bool(accumulate))
            n_sum = dp.dp_launch_count() - n0
            dp.dp_add_noise(dW, sigma, C, Bdiv, seed, offset)
            if db is not None:
                dp.dp_add_noise(db, sigma, C, Bdiv, seed, offset + p * D)
        else:
            nd = dp.noise_desc(sigma, C, Bdiv, seed=seed, offset=offset)
            dp.dp_clipped_sum_noised(desc, dA, dG, f, dW, db, nd, ws, accumulate=bool(accumulate))
            n_fused = dp.dp_launch_count() - n0
        torch.cuda.synchronize()
        outs.append(flat[:p * D + (p if db is not None else 0)].cpu())
    assert torch.equal(outs[0], outs[1])
    if fused:
        assert n_fused == n_sum          # the noise rode in the sum's final reductions
    else:
        assert n_fused > n_sum


def test_fused_devseed_and_kept(lib):
    """Device-side seed, and the kept-gradient sum with its fused noise."""
    import torch
    dp = lib
    spec = LayerSpec("e", "linear", p=136, d=200, T=70)
    wl = Workload(name="kept", B=6, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=3)
    A, G = workloads.layer_inputs(wl, 0)
    desc = desc_for(dp, spec, wl.B, wl.dtype)
    dA, dG = to_dev(A, "bf16"), to_dev(G, "bf16")
    fac = torch.tensor(workloads.factor_inputs(wl, wl.B, 0.2, 1.0), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(dp.dp_workspace_size(desc, dp.DP_NORM_INSTANTIATE), 16), dtype=torch.uint8, device="cuda")
    nbytes = dp.dp_grads_size(desc)
    assert nbytes > 0
    grads = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    sq = torch.empty(wl.B, dtype=torch.float32, device="cuda")
    dp.dp_layer_sqnorms_keep(desc, dA, dG, sq, grads, ws)
    seed_dev = torch.tensor([0x1234_5678_9ABC], dtype=torch.int64, device="cuda")
    n = spec.p * spec.D + spec.p
    a = torch.empty(n, device="cuda")
    b = torch.empty(n, device="cuda")
    dp.dp_clipped_sum_kept(desc, grads, fac, a[:-spec.p], a[-spec.p:], ws)
    dp.dp_add_noise(a, 0.9, 1.1, wl.B, 0x1234_5678_9ABC, 5)
    nd = dp.noise_desc(0.9, 1.1, wl.B, seed=0, seed_dev=seed_dev, offset=5)
    dp.dp_clipped_sum_kept_noised(desc, grads, fac, b[:-spec.p], b[-spec.p:], nd, ws)
    torch.cuda.synchronize()
    assert torch.equal(a.cpu(), b.cpu())
    c = torch.empty(n, device="cuda")
    dp.dp_clipped_sum_noised(desc, dA, dG, fac, c[:-spec.p], c[-spec.p:], nd, ws)
    torch.cuda.synchronize()
    # the contraction and the kept gradients round differently: same noise, sums within tolerance
    assert rel_flat(c.cpu().numpy(), a.cpu().numpy(), [spec]) <= TOL["bf16"]


@pytest.mark.parametrize("per_layer", [False, True])
def test_clip_step_fused_matches_unfused_and_oracle(lib, per_layer):
    """A three-layer step: fused and unfused ClipStep agree bit for bit, eagerly and as a
    captured graph; both match the oracle's step."""
    import torch
    dp = lib
    # a linear layer (noise fused into its sum), a conv layer on the row layout and a conv layer
    # that keeps its per-example gradients (T = 576): the conv layers' noise is one launch
    specs = (LayerSpec("a", "linear", p=136, d=200, T=100),
             LayerSpec("b", "conv2d", p=64, Cin=16, H=10, W=10, k=3, pad=1),
             LayerSpec("c", "conv2d", p=64, Cin=64, H=24, W=24, k=3, pad=1))
    wl = Workload(name="three", B=12, layers=specs, dtype="bf16", C=1.0, sigma=0.6, seed=21, per_layer=per_layer)
    inputs = [workloads.layer_inputs(wl, l) for l in range(3)]
    dev = [(to_dev(A, "bf16"), to_dev(G, "bf16")) for A, G in inputs]
    descs = [desc_for(dp, s, wl.B, "bf16") for s in specs]
    C = [0.5, 0.8, 0.3] if per_layer else 1.0
    got = []
    for fuse in (False, True):
        st = dp.ClipStep(descs, C=C, sigma=wl.sigma, per_layer=per_layer, fuse_noise=fuse)
        assert [k is not None for k in st.kept] == [False, False, True]
        eager = st.run(dev, seed=99).clone()
        st.capture(dev)
        replayed = st.replay(99).clone()
        torch.cuda.synchronize()
        assert torch.equal(eager.cpu(), replayed.cpu())
        got.append(eager.cpu())
    assert torch.equal(got[0], got[1])
    ref = oracle.dp_step(wl, inputs, seed=99, C=C)
    assert rel_flat(got[1].numpy(), ref["noisy"], specs) <= TOL["bf16"]


def test_captured_step_draws_adaptive_bound_noise_from_replay_seed(lib):
    """A per-layer step with the adaptive bound: a graph replay with seed s gives the bounds
    (and the gradient) of an eager run with seed s, for two seeds, and the bounds are the
    oracle's for that seed."""
    import torch
    dp = lib
    specs = (LayerSpec("a", "linear", p=40, d=72, T=30),
             LayerSpec("b", "conv2d", p=16, Cin=8, H=6, W=6, k=3, pad=1))
    wl = Workload(name="adaptive", B=20, layers=specs, dtype="bf16", C=1.0, sigma=0.6, seed=3, per_layer=True)
    inputs = [workloads.layer_inputs(wl, l) for l in range(2)]
    dev = [(to_dev(A, "bf16"), to_dev(G, "bf16")) for A, G in inputs]
    descs = [desc_for(dp, s, wl.B, "bf16") for s in specs]
    ad = dict(alpha=1.1, beta=2.0, sigma_l2=2.5, C_l2=[0.7, 1.3])
    st = dp.ClipStep(descs, C=[0.5, 0.8], sigma=wl.sigma, per_layer=True, adaptive=ad)
    eager = {}
    for seed in (99, 7):
        g = st.run(dev, seed=seed).clone()
        eager[seed] = (g, st.bounds_next.clone())
    st.capture(dev)
    sq = st.sqnorms.cpu().numpy().astype(np.float64)
    for seed in (99, 7):
        g = st.replay(seed).clone()
        torch.cuda.synchronize()
        assert torch.equal(g, eager[seed][0])
        assert torch.equal(st.bounds_next, eager[seed][1])
        for l in range(2):
            rc, rcl2 = oracle.adaptive_bound(sq[l], ad["C_l2"][l], 1.1, 2.0, 2.5, seed, l)
            c, cl2 = st.bounds_next[l].cpu().numpy()
            assert c == pytest.approx(rc, rel=1e-5, abs=1e-6) and cl2 == pytest.approx(rcl2, rel=1e-5, abs=1e-6)
    assert not torch.equal(eager[99][1], eager[7][1])


def test_noise_blocks_equal_one_pass_per_block(lib):
    """dp_add_noise_blocks over blocks with their own bounds (misaligned offsets, neighbours
    sharing a Philox block, an empty block, a gap) equals one dp_add_noise per block, bit for
    bit; with the device-side seed too."""
    import torch
    dp = lib
    n = 5000
    blocks = [(0, 1001, 0.5), (1001, 3, 2.0), (1004, 0, 1.0), (1004, 998, 1.0), (2100, 2900, 0.25)]
    gen = torch.Generator(device="cuda").manual_seed(11)
    base = torch.randn(n, generator=gen, device="cuda")
    for use_dev in (False, True):
        a, b = base.clone(), base.clone()
        seed = 0xDEADBEEF12
        for o, m, C in blocks:
            if m:
                dp.dp_add_noise(a[o:o + m], 0.8, C, 7, seed, o)
        sd = torch.tensor([seed], dtype=torch.int64, device="cuda") if use_dev else None
        dp.dp_add_noise_blocks(b, blocks, 0.8, 7, seed=0 if use_dev else seed, seed_dev=sd)
        torch.cuda.synchronize()
        assert torch.equal(a.cpu(), b.cpu())
        assert torch.equal(b[2002:2100].cpu(), base[2002:2100].cpu())     # the gap is untouched

