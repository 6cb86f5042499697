"""GPU parity: the CUDA path through the C ABI against the float64 CPU oracle.

Every workload's shapes are covered: in full where the oracle finishes in seconds,
else on a smaller batch in full plus sampled examples at the full batch.  Edge
cases: one example, ragged rows and widths, strides/dilation, no bias,
accumulation, per-layer bounds, non-finite inputs, noise windows.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from helpers import TOL, Z_ATOL, Z_RTOL, desc_for, rel_elem, rel_flat, rel_rows, to_dev
from workloads import LayerSpec, Workload

pytestmark = pytest.mark.gpu


def _run_layer(dp, spec, wl, A, G, mode=None, factors=None):
    """GPU sqnorms (and, with factors, the clipped sum) for one layer."""
    import torch
    B = A.shape[0]
    desc = desc_for(dp, spec, B, wl.dtype)
    mode = dp.DP_NORM_AUTO if mode is None else mode
    ws = torch.empty(max(dp.dp_workspace_size(desc, mode), 16), dtype=torch.uint8, device="cuda")
    Ad, Gd = to_dev(A, wl.dtype), to_dev(G, wl.dtype)
    sq = torch.empty(B, dtype=torch.float32, device="cuda")
    chosen = dp.dp_layer_sqnorms(desc, Ad, Gd, sq, ws, mode=mode)
    out = dict(sq=sq, chosen=chosen)
    if factors is not None:
        f = torch.tensor(np.asarray(factors, dtype=np.float32), device="cuda")
        dW = torch.empty(spec.p * spec.D, dtype=torch.float32, device="cuda")
        db = torch.empty(spec.p, dtype=torch.float32, device="cuda") if spec.has_bias else None
        dp.dp_clipped_sum(desc, Ad, Gd, f, dW, db, ws)
        out.update(dW=dW, db=db)
    torch.cuda.synchronize()
    return out


def _check_layer(dp, spec, wl, examples=None, mode=None, factor_range=(0.0, 1.0)):
    A, G = workloads.layer_inputs(wl, list(wl.layers).index(spec), examples)
    fac = workloads.factor_inputs(wl, A.shape[0], *factor_range)
    got = _run_layer(dp, spec, wl, A, G, mode, fac)
    s_ref = oracle.layer_sqnorms(spec, A, G)
    tol = TOL[wl.dtype]
    assert rel_elem(got["sq"].cpu().numpy(), s_ref) <= tol
    S, Sb = oracle.clipped_sum(spec, A, G, fac.astype(np.float64))
    assert rel_rows(got["dW"].cpu().numpy(), S, spec.D) <= tol
    if spec.has_bias:
        assert rel_rows(got["db"].cpu().numpy(), Sb) <= tol
    return got


# ----------------------------------------------------------------- workloads in full

def test_t1_linear_full_step(lib):
    """One-row fp32 layer: norms, factors, clipped sum, noise -- the whole step."""
    import torch
    dp = lib
    wl = workloads.get_workload("t1_linear_b32")
    inputs = [workloads.layer_inputs(wl, 0)]
    ref = oracle.dp_step(wl, inputs)
    desc = desc_for(dp, wl.layers[0], wl.B, wl.dtype)
    step = dp.ClipStep([desc], C=wl.C, sigma=wl.sigma)
    dev = [(to_dev(A, wl.dtype), to_dev(G, wl.dtype)) for A, G in inputs]
    step.norms(dev)
    step.factors_()
    step.sums(dev)
    torch.cuda.synchronize()
    assert step.chosen == [dp.DP_NORM_T1]
    assert rel_elem(step.sqnorms.cpu().numpy(), ref["sqnorms"]) <= TOL["fp32"]
    assert rel_elem(step.factors.cpu().numpy()[0], ref["factors"]) <= TOL["fp32"]
    S, Sb = ref["sums"][0]
    pre = np.concatenate([S.ravel(), Sb])
    assert rel_flat(step.grad.cpu().numpy(), pre, wl.layers) <= TOL["fp32"]
    step.noise(wl.seed)
    torch.cuda.synchronize()
    assert rel_flat(step.grad.cpu().numpy(), ref["noisy"], wl.layers) <= TOL["fp32"]


def test_seq_linear_full_step(lib):
    import torch
    dp = lib
    wl = workloads.get_workload("seq_linear_b64_t128")
    inputs = [workloads.layer_inputs(wl, 0)]
    ref = oracle.dp_step(wl, inputs)
    desc = desc_for(dp, wl.layers[0], wl.B, wl.dtype)
    step = dp.ClipStep([desc], C=wl.C, sigma=wl.sigma)
    dev = [(to_dev(A, wl.dtype), to_dev(G, wl.dtype)) for A, G in inputs]
    step.norms(dev)
    step.factors_()
    step.sums(dev)
    torch.cuda.synchronize()
    assert step.chosen == [dp.DP_NORM_GHOST]
    tol = TOL["bf16"]
    assert rel_elem(step.sqnorms.cpu().numpy(), ref["sqnorms"]) <= tol
    assert rel_elem(step.factors.cpu().numpy()[0], ref["factors"]) <= tol
    S, Sb = ref["sums"][0]
    assert rel_flat(step.grad.cpu().numpy(), np.concatenate([S.ravel(), Sb]), wl.layers) <= tol
    step.noise(wl.seed)
    torch.cuda.synchronize()
    assert rel_flat(step.grad.cpu().numpy(), ref["noisy"], wl.layers) <= tol


def test_conv3x3_full_batch(lib):
    wl = workloads.get_workload("conv3x3_b256")
    got = _check_layer(lib, wl.layers[0], wl)
    assert got["chosen"] == lib.DP_NORM_INSTANTIATE


def test_vgg11_stack_small_batch_flat_and_per_layer(lib):
    """Every VGG-11 layer (mixed ghost/instantiate/one-row), whole step, flat and per-layer."""
    import torch
    dp = lib
    wl = workloads.get_workload("vgg11_cifar_b1024").with_batch(12)
    inputs = [workloads.layer_inputs(wl, l) for l in range(len(wl.layers))]
    descs = [desc_for(dp, s, wl.B, wl.dtype) for s in wl.layers]
    dev = [(to_dev(A, wl.dtype), to_dev(G, wl.dtype)) for A, G in inputs]
    # scale so that some examples clip and some do not
    for per_layer in (False, True):
        ref = oracle.dp_step(wl, inputs, per_layer=per_layer)
        step = dp.ClipStep(descs, C=wl.C, sigma=wl.sigma, per_layer=per_layer)
        step.norms(dev)
        step.factors_()
        step.sums(dev)
        torch.cuda.synchronize()
        assert rel_elem(step.sqnorms.cpu().numpy(), ref["sqnorms"]) <= TOL["bf16"]
        fac = step.factors.cpu().numpy()
        assert rel_elem(fac if per_layer else fac[0], ref["factors"]) <= TOL["bf16"]
        pre = np.concatenate([np.concatenate([S.ravel(), Sb]) for S, Sb in ref["sums"]])
        g = step.grad.cpu().numpy()
        for l in range(len(wl.layers)):
            o, n = wl.param_offsets()[l], wl.layers[l].n_params
            assert rel_flat(g[o:o + n], pre[o:o + n], [wl.layers[l]]) <= TOL["bf16"], wl.layers[l].name
        step.noise(wl.seed)
        torch.cuda.synchronize()
        assert rel_flat(step.grad.cpu().numpy(), ref["noisy"], wl.layers) <= TOL["bf16"]


def test_vit_mlp_small_batch(lib):
    wl = workloads.get_workload("vit_mlp_b4096_t197").with_batch(6)
    for spec in wl.layers:
        got = _check_layer(lib, spec, wl)
        assert got["chosen"] == lib.DP_NORM_GHOST


# ----------------------------------------------------------------- forced modes agree

@pytest.mark.parametrize("name,layer", [("seq_linear_b64_t128", 0), ("conv3x3_b256", 0),
                                        ("vgg11_cifar_b1024", 2), ("vgg11_cifar_b1024", 1),
                                        ("vgg11_cifar_b1024", 6)])
def test_ghost_and_instantiation_agree(lib, name, layer):
    wl = workloads.get_workload(name).with_batch(5)
    spec = wl.layers[layer]
    A, G = workloads.layer_inputs(wl, layer)
    ref = oracle.layer_sqnorms(spec, A, G)
    for mode in (lib.DP_NORM_GHOST, lib.DP_NORM_INSTANTIATE):
        got = _run_layer(lib, spec, wl, A, G, mode)
        assert got["chosen"] == mode
        assert rel_elem(got["sq"].cpu().numpy(), ref) <= TOL[wl.dtype]


# ----------------------------------------------------------------- edge shapes

EDGE = [
    ("lin_B1", LayerSpec("e", "linear", p=24, d=40, T=7), 1, "bf16"),
    ("lin_ragged", LayerSpec("e", "linear", p=50, d=100, T=37), 5, "bf16"),
    ("lin_ragged_fp32", LayerSpec("e", "linear", p=33, d=65, T=19), 4, "fp32"),
    ("lin_nobias", LayerSpec("e", "linear", p=64, d=96, T=130, has_bias=False), 3, "bf16"),
    ("lin_t1_odd", LayerSpec("e", "linear", p=10, d=13, T=1), 9, "bf16"),
    ("lin_t1_fp32_odd", LayerSpec("e", "linear", p=7, d=5, T=1), 3, "fp32"),
    ("lin_tc_ragged", LayerSpec("e", "linear", p=72, d=200, T=33), 5, "bf16"),
    ("lin_tc_T256", LayerSpec("e", "linear", p=128, d=64, T=256), 3, "bf16"),
    ("lin_tc_splits", LayerSpec("e", "linear", p=128, d=256, T=50), 37, "bf16"),
    ("lin_tc_B1", LayerSpec("e", "linear", p=64, d=64, T=64), 1, "bf16"),
    ("lin_tc_T300", LayerSpec("e", "linear", p=64, d=136, T=300, has_bias=False), 2, "bf16"),
    ("conv_s2", LayerSpec("e", "conv2d", p=6, Cin=5, H=11, W=9, k=3, stride=2, pad=1), 3, "bf16"),
    ("conv_dil", LayerSpec("e", "conv2d", p=4, Cin=3, H=10, W=10, k=3, stride=1, pad=2, dil=2), 2, "fp32"),
    ("conv_k1", LayerSpec("e", "conv2d", p=8, Cin=16, H=6, W=6, k=1), 3, "bf16"),
    ("conv_k5_nopad", LayerSpec("e", "conv2d", p=5, Cin=2, H=9, W=8, k=5, a_dist="abs_normal"), 2, "bf16"),
    # conv layers through their row layout on the tensor cores (D and p multiples of 8)
    ("conv_rows_3x3", LayerSpec("e", "conv2d", p=72, Cin=16, H=12, W=12, k=3, pad=1), 5, "bf16"),
    ("conv_rows_s2_dil", LayerSpec("e", "conv2d", p=64, Cin=8, H=17, W=17, k=3, stride=2, pad=2, dil=2), 3,
     "bf16"),
    ("conv_rows_T16", LayerSpec("e", "conv2d", p=128, Cin=64, H=4, W=4, k=3, pad=1, a_dist="abs_normal"), 7,
     "bf16"),
    ("conv_rows_k1_nobias", LayerSpec("e", "conv2d", p=64, Cin=64, H=8, W=8, k=1, has_bias=False), 4, "bf16"),
    ("conv_rows_p8", LayerSpec("e", "conv2d", p=8, Cin=8, H=5, W=7, k=3, pad=1), 3, "bf16"),
    # output-gradient row copies of every pixel count class: T = 4 and 6 (one thread per
    # 8 x T block), 8 (a warp tile of 256 rows x 8 pixels), 24 (128 x 16, ragged), 12 (T % 8 != 0)
    ("conv_rows_T4", LayerSpec("e", "conv2d", p=16, Cin=8, H=2, W=2, k=3, pad=1), 5, "bf16"),
    ("conv_rows_T6_p136", LayerSpec("e", "conv2d", p=136, Cin=8, H=2, W=3, k=3, pad=1), 3, "bf16"),
    ("conv_rows_T8_p40", LayerSpec("e", "conv2d", p=40, Cin=8, H=2, W=4, k=3, pad=1), 4, "bf16"),
    ("conv_rows_T24", LayerSpec("e", "conv2d", p=24, Cin=8, H=4, W=6, k=3, pad=1), 3, "bf16"),
    ("conv_rows_T12", LayerSpec("e", "conv2d", p=24, Cin=8, H=3, W=4, k=3, pad=1), 3, "bf16"),
    ("conv_c64_2x2", LayerSpec("e", "conv2d", p=64, Cin=64, H=2, W=2, k=3, pad=1), 5, "bf16"),
    ("conv_c128_4x4_p72", LayerSpec("e", "conv2d", p=72, Cin=128, H=4, W=4, k=3, pad=1), 3, "bf16"),
    # D = 27 padded to 32 columns in the row layout (the first VGG-11 layer's shape)
    ("conv_rows_padD", LayerSpec("e", "conv2d", p=64, Cin=9, H=12, W=12, k=3, pad=1), 4, "bf16"),
    # narrow conv layers: the unfold formed on chip (per-element gathers: Wout % 8 != 0)
    ("conv_unfold_12x12", LayerSpec("e", "conv2d", p=64, Cin=3, H=12, W=12, k=3, pad=1), 4, "bf16"),
    ("conv_rows_padD_s2", LayerSpec("e", "conv2d", p=24, Cin=5, H=13, W=11, k=3, stride=2, pad=1), 3, "bf16"),
    # conv layers whose unfold is done by TMA im2col loads (Cin % 64 == 0, T % 8 == 0, T >= 64)
    ("conv_im2col_3x3", LayerSpec("e", "conv2d", p=72, Cin=64, H=12, W=12, k=3, pad=1), 3, "bf16"),
    ("conv_im2col_s2_dil2", LayerSpec("e", "conv2d", p=136, Cin=128, H=23, W=23, k=3, stride=2, pad=2, dil=2),
     2, "bf16"),
    ("conv_im2col_k5_nobias", LayerSpec("e", "conv2d", p=64, Cin=64, H=12, W=12, k=5, has_bias=False,
                                        a_dist="abs_normal"), 3, "bf16"),
    # one row block (64 < T <= 128): the ghost norm with single-block pairs
    ("lin_ghost_split", LayerSpec("e", "linear", p=136, d=200, T=100), 3, "bf16"),
    ("conv_im2col_ghost_split", LayerSpec("e", "conv2d", p=72, Cin=64, H=10, W=10, k=3, pad=1), 2, "bf16"),
    # conv1d: the row layout on the tensor cores (p % 8 == 0), else the FFMA kernels
    ("conv1d_rows", LayerSpec("e", "conv1d", p=16, Cin=8, W=50, k=5, stride=2, pad=2), 4, "bf16"),
    ("conv1d_rows_dil_nobias", LayerSpec("e", "conv1d", p=24, Cin=3, W=70, k=3, dil=2, has_bias=False), 3, "bf16"),
    ("conv1d_long", LayerSpec("e", "conv1d", p=64, Cin=32, W=300, k=3, pad=1), 2, "bf16"),
    ("conv1d_fp32", LayerSpec("e", "conv1d", p=6, Cin=5, W=21, k=3, pad=1), 3, "fp32"),
    ("conv1d_k1", LayerSpec("e", "conv1d", p=8, Cin=64, W=40, k=1), 3, "bf16"),
    # conv3d: cubic kernels through the gathered row layout (p % 8 == 0), else the FFMA kernels
    ("conv3d_rows", LayerSpec("e", "conv3d", p=16, Cin=4, Z=6, H=7, W=8, k=3, pad=1), 3, "bf16"),
    ("conv3d_s2_dil2", LayerSpec("e", "conv3d", p=24, Cin=2, Z=9, H=9, W=10, k=3, stride=2, pad=2, dil=2), 3,
     "bf16"),
    ("conv3d_k2_nobias", LayerSpec("e", "conv3d", p=16, Cin=8, Z=5, H=6, W=7, k=2, has_bias=False), 2, "bf16"),
    ("conv3d_k1", LayerSpec("e", "conv3d", p=32, Cin=32, Z=4, H=4, W=4, k=1), 4, "bf16"),
    # a shape the 2-D im2col kernels would take (Cin % 64 == 0, T % 8 == 0): depth must keep it off them
    ("conv3d_k1_c64", LayerSpec("e", "conv3d", p=64, Cin=64, Z=3, H=8, W=8, k=1), 3, "bf16"),
    ("conv3d_c64_pad", LayerSpec("e", "conv3d", p=64, Cin=64, Z=2, H=8, W=8, k=3, pad=1), 2, "bf16"),
    ("conv3d_fp32", LayerSpec("e", "conv3d", p=6, Cin=3, Z=5, H=5, W=5, k=3, pad=1), 3, "fp32"),
    # two row blocks (128 < T <= 256): block 1 loaded as its valid rows rounded to 16 (N = r1 on the B side)
    ("lin_ghost_dual_T129", LayerSpec("e", "linear", p=64, d=64, T=129), 2, "bf16"),
    ("lin_ghost_dual_T150", LayerSpec("e", "linear", p=72, d=200, T=150), 3, "bf16"),
    ("lin_ghost_dual_T241_wide_p", LayerSpec("e", "linear", p=264, d=96, T=241, has_bias=False), 2, "bf16"),
    # the second row block loaded as 64 rows (T - 128 = 52): its Gram columns end at a 32-column chunk
    ("lin_ghost_dual_T180_r64", LayerSpec("e", "linear", p=96, d=64, T=180), 3, "bf16"),
    # more examples than SMs: each two-block CTA takes two or three examples in turn
    ("lin_ghost_dual_B400", LayerSpec("e", "linear", p=64, d=72, T=150), 400, "bf16"),
    # one row block: T just above the packed limit, batches of about half the SM count
    ("lin_ghost_slab_T65", LayerSpec("e", "linear", p=40, d=48, T=65), 5, "bf16"),
    ("lin_ghost_slab_B76", LayerSpec("e", "linear", p=64, d=72, T=128), 76, "bf16"),
    ("lin_ghost_B77", LayerSpec("e", "linear", p=64, d=72, T=128, has_bias=False), 77, "bf16"),
]


@pytest.mark.parametrize("tag,spec,B,dtype", EDGE, ids=[e[0] for e in EDGE])
def test_edge_shapes(lib, tag, spec, B, dtype):
    wl = Workload(name=tag, B=B, layers=(spec,), dtype=dtype, C=1.0, sigma=1.0, seed=11)
    for mode in (None, lib.DP_NORM_GHOST, lib.DP_NORM_INSTANTIATE):
        _check_layer(lib, spec, wl, mode=mode)


@pytest.mark.parametrize("B,d,p", [(25001, 64, 48), (19457, 40, 24)], ids=["B25001", "B19457_short_rows"])
def test_t1_norm_many_examples(lib, B, d, p):
    """One-row norms over more examples than the capped grid has warps (each warp takes two
    examples per pass; an odd count leaves the last pass with one)."""
    import torch
    spec = LayerSpec("e", "linear", p=p, d=d, T=1)
    wl = Workload(name="t1_many", B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=43)
    A, G = workloads.layer_inputs(wl, 0, threads=8)
    desc = desc_for(lib, spec, B, "bf16")
    sq = torch.full((B,), float("nan"), device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert lib.dp_layer_sqnorms(desc, to_dev(A, "bf16"), to_dev(G, "bf16"), sq, ws) == lib.DP_NORM_T1
    torch.cuda.synchronize()
    assert rel_elem(sq.cpu().numpy(), oracle.layer_sqnorms(spec, A, G)) <= TOL["bf16"]


@pytest.mark.parametrize("B,accumulate", [(300, False), (257, True)], ids=["B300", "B257_accumulate"])
def test_bias_shared_across_column_tiles(lib, B, accumulate):
    """A layer whose examples split over clusters with B >= 256: every column tile sums the
    bias over its share of the examples and the partial biases are added after the kernel.
    The whole bias and sampled weight entries against the oracle's entry-wise sum."""
    import torch
    dp = lib
    spec = LayerSpec("e", "linear", p=768, d=1280, T=64)
    wl = Workload(name="bias_shared", B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=37)
    A, G = workloads.layer_inputs(wl, 0)
    fac = workloads.factor_inputs(wl, B)
    desc = desc_for(dp, spec, B, "bf16")
    ws = torch.empty(dp.dp_workspace_size(desc), dtype=torch.uint8, device="cuda")
    dW = torch.full((spec.p * spec.D,), 0.5, device="cuda")
    db = torch.full((spec.p,), -0.25, device="cuda")
    dp.dp_clipped_sum(desc, to_dev(A, "bf16"), to_dev(G, "bf16"), torch.tensor(fac, device="cuda"), dW, db, ws,
                      accumulate=accumulate)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    rows = np.unique(np.r_[0, 127, 128, 255, 256, 767, rng.choice(spec.p, 20, replace=False)])
    cols = np.unique(np.r_[0, 255, 256, 511, 512, 1023, 1024, 1279, rng.choice(spec.D, 20, replace=False)])
    S, _ = oracle.clipped_sum_elements(spec, A, G, fac.astype(np.float64), rows, cols)
    _, Sb = oracle.clipped_sum_elements(spec, A, G, fac.astype(np.float64), np.arange(spec.p), [0])
    base_w, base_b = (0.5, -0.25) if accumulate else (0.0, 0.0)
    got = dW.view(spec.p, spec.D).cpu().numpy()[np.ix_(rows, cols)] - base_w
    assert rel_rows(got, S, cols.size) <= TOL["bf16"]
    assert rel_rows(db.cpu().numpy() - base_b, Sb) <= TOL["bf16"]


@pytest.mark.parametrize("conv_pin", ["", "rows"], ids=["im2col", "rows"])
def test_conv3x3_im2col_and_row_layout(lib, conv_pin, monkeypatch):
    """The 3x3 conv workload's layer (small batch): im2col kernels and the row layout."""
    if conv_pin:
        monkeypatch.setenv("DPCLIP_CONV", conv_pin)
    wl = workloads.get_workload("conv3x3_b256").with_batch(5)
    spec = wl.layers[0]
    for mode in (None, lib.DP_NORM_INSTANTIATE, lib.DP_NORM_GHOST):
        _check_layer(lib, spec, wl, mode=mode)


@pytest.mark.parametrize("pin", ["rows", "example"])
def test_conv_rows_sum_kernels(lib, pin, monkeypatch):
    """Both tensor-core clipped-sum kernels on a conv layer's row layout (ragged tiles)."""
    monkeypatch.setenv("DPCLIP_SUM_KERNEL", pin)
    spec = LayerSpec("e", "conv2d", p=136, Cin=32, H=10, W=9, k=3, pad=1, a_dist="abs_normal")
    wl = Workload(name="conv_pin", B=6, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=4)
    _check_layer(lib, spec, wl)


@pytest.mark.parametrize("p,has_bias", [(320, True), (448, False)], ids=["p320_one_acc_tail", "p448_three_boxes"])
def test_conv_rowscaled_wide_tiles(lib, p, has_bias):
    """The row-scaled conv GEMM with 256-output tiles (two TMEM accumulators sharing each
    stage's unfolded columns): enough batch rows per CTA to take them, a last output tile
    with one accumulator (320 = 256 + 64) or with three of its four G boxes (448)."""
    import torch
    dp = lib
    spec = LayerSpec("e", "conv2d", p=p, Cin=64, H=8, W=8, k=3, pad=1, has_bias=has_bias, a_dist="abs_normal")
    B = 640
    wl = Workload(name="wide", B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=41)
    A, G = workloads.layer_inputs(wl, 0)
    fac = workloads.factor_inputs(wl, B, 0.1, 1.0)
    desc = desc_for(dp, spec, B, "bf16")
    ws = torch.empty(dp.dp_workspace_size(desc), dtype=torch.uint8, device="cuda")
    Ad, Gd = to_dev(A, "bf16"), to_dev(G, "bf16")
    dW = torch.full((spec.p * spec.D,), float("nan"), device="cuda")
    db = torch.full((spec.p,), float("nan"), device="cuda") if has_bias else None
    dp.dp_clipped_sum(desc, Ad, Gd, torch.tensor(fac, device="cuda"), dW, db, ws)
    torch.cuda.synchronize()
    S, Sb = oracle.clipped_sum(spec, A, G, fac.astype(np.float64))
    assert rel_rows(dW.cpu().numpy(), S, spec.D) <= TOL["bf16"]
    if has_bias:
        assert rel_rows(db.cpu().numpy(), Sb) <= TOL["bf16"]


ACC = [(LayerSpec("e", "linear", p=42, d=72, T=9), 6),          # SIMT (p not a multiple of 8)
       (LayerSpec("e", "linear", p=128, d=64, T=40), 5),         # row-scaled tensor-core GEMM
       (LayerSpec("e", "linear", p=128, d=128, T=64), 4),        # per-example, several splits
       (LayerSpec("e", "linear", p=64, d=256, T=80), 1),         # per-example, one split
       (LayerSpec("e", "conv2d", p=16, Cin=9, H=8, W=8, k=3, pad=1), 3),   # conv, padded columns
       (LayerSpec("e", "conv2d", p=64, Cin=3, H=8, W=8, k=3, pad=1), 1),   # conv, on-chip unfold, one split
       (LayerSpec("e", "conv2d", p=64, Cin=64, H=8, W=8, k=3, pad=1), 3),  # conv, im2col row-scaled
       (LayerSpec("e", "conv2d", p=72, Cin=64, H=12, W=12, k=3, pad=1), 2),  # conv, im2col per example
       (LayerSpec("e", "linear", p=10, d=13, T=1), 300),                   # one row, 3 example splits
       (LayerSpec("e", "linear", p=136, d=264, T=70), 11),                 # per-example, grid splits
       (LayerSpec("e", "linear", p=256, d=256, T=64), 1),                  # per-example, bias, one split
       (LayerSpec("e", "linear", p=512, d=256, T=70), 11)]                 # per-example, bias, splits


ACC_PIN = ["", "rows", "example", "example", "", "", "", "", "", "example", "example", "example"]


@pytest.mark.parametrize("spec,B,pin", [(s, b, p) for (s, b), p in zip(ACC, ACC_PIN)],
                         ids=["simt", "tc_rows", "tc_ex_splits", "tc_ex_single", "conv_padded", "conv_unfold_direct",
                              "conv_im2col_rows", "conv_im2col_example", "t1_splits", "tc_ex_grid",
                              "tc_ex_256_single", "tc_ex_tail_splits"])
def test_accumulate_adds_to_existing_sum(lib, spec, B, pin, monkeypatch):
    if pin:
        monkeypatch.setenv("DPCLIP_SUM_KERNEL", pin)
    import torch
    dp = lib
    wl = Workload(name="acc", B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=2)
    A, G = workloads.layer_inputs(wl, 0)
    fac = workloads.factor_inputs(wl, B)
    desc = desc_for(dp, spec, B, "bf16")
    ws = torch.empty(dp.dp_workspace_size(desc), dtype=torch.uint8, device="cuda")
    Ad, Gd = to_dev(A, "bf16"), to_dev(G, "bf16")
    f = torch.tensor(fac, device="cuda")
    dW = torch.full((spec.p * spec.D,), 0.25, device="cuda")
    db = torch.full((spec.p,), -0.5, device="cuda")
    dp.dp_clipped_sum(desc, Ad, Gd, f, dW, db, ws, accumulate=True)
    dp.dp_clipped_sum(desc, Ad, Gd, f, dW, db, ws, accumulate=True)
    S, Sb = oracle.clipped_sum(spec, A, G, fac.astype(np.float64))
    assert rel_rows(dW.cpu().numpy() - 0.25, 2 * S.ravel(), spec.D) <= TOL["bf16"]
    assert rel_rows(db.cpu().numpy() + 0.5, 2 * Sb) <= TOL["bf16"]


def test_speed_priority_mode(lib):
    """DP_NORM_AUTO_TIME resolves by the time counts (here: instantiate, where the space
    rule would take the ghost norm) and gives the oracle's norms."""
    spec = LayerSpec("e", "linear", p=256, d=256, T=150)
    wl = Workload(name="speed", B=3, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=21)
    got = _check_layer(lib, spec, wl, mode=lib.DP_NORM_AUTO_TIME)
    assert got["chosen"] == lib.DP_NORM_INSTANTIATE


@pytest.mark.parametrize("per_layer", [False, True], ids=["flat", "per_layer"])
def test_virtual_step_matches_one_batch(lib, per_layer):
    """Gradient accumulation: micro-batches of 3 and 5 examples added into one step, then
    noise and 1/B once, equal the step over the logical batch of 8."""
    l1 = LayerSpec("a", "linear", p=32, d=48, T=16)
    l2 = LayerSpec("b", "conv2d", p=8, Cin=4, H=6, W=6, k=3, pad=1)
    wl = Workload(name="virtual", B=8, layers=(l1, l2), dtype="bf16", C=1.0, sigma=0.5, seed=9,
                  per_layer=per_layer)
    Cs = [1.0, 0.5]
    inputs = [workloads.layer_inputs(wl, l) for l in range(2)]
    ref = oracle.dp_step(wl, inputs, C=Cs if per_layer else None)
    vs = lib.VirtualStep([desc_for(lib, s, 5, "bf16") for s in wl.layers], C=Cs if per_layer else 1.0,
                         sigma=0.5, per_layer=per_layer)
    for _ in range(2):          # a second logical batch after zero() gives the same result
        vs.zero()
        for lo, hi in ((0, 3), (3, 8)):
            dev = [(to_dev(A[lo:hi], "bf16"), to_dev(G[lo:hi], "bf16")) for A, G in inputs]
            vs.add(dev, hi - lo)
        grad = vs.finish(wl.seed)
        assert vs.examples == 8
        assert rel_flat(grad.cpu().numpy(), ref["noisy"], wl.layers) <= TOL["bf16"]


def test_device_wait_timeout_reported_and_context_usable(lib):
    """Failure detection without a fault: a kernel whose bounded mbarrier wait has nothing
    to wait for gives up after the 2 s limit, the host reads DP_ERR_TIMEOUT, and the next
    step on the same context still matches the oracle."""
    import torch
    assert lib.dp_check_status() == lib.DP_OK
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    lib.dp_selftest_wait_timeout(waited)
    assert lib.dp_check_status() == lib.DP_ERR_TIMEOUT
    assert 1.9e9 <= waited.item() <= 10e9
    assert lib.dp_check_status() == lib.DP_OK            # cleared
    spec = LayerSpec("a", "linear", p=32, d=48, T=16)
    wl = Workload(name="after_timeout", B=6, layers=(spec,), dtype="bf16", C=1.0, sigma=0.5, seed=4)
    inputs = [workloads.layer_inputs(wl, 0)]
    ref = oracle.dp_step(wl, inputs)
    step = lib.ClipStep([desc_for(lib, spec, wl.B, "bf16")], C=1.0, sigma=0.5)
    grad = step.run([(to_dev(A, "bf16"), to_dev(G, "bf16")) for A, G in inputs], seed=wl.seed)
    assert lib.dp_check_status() == lib.DP_OK
    assert rel_flat(grad.cpu().numpy(), ref["noisy"], wl.layers) <= TOL["bf16"]


# Kept per-example gradients: the instantiated norm stores g_i and b_i, the clipped sum
# reads them back (conv through TMA im2col, linear per-example products, a conv layer on
# its padded row layout).
KEPT = [
    ("conv_im2col", LayerSpec("e", "conv2d", p=72, Cin=64, H=12, W=12, k=3, pad=1), 3),
    ("conv_im2col_s2_dil2_nobias", LayerSpec("e", "conv2d", p=136, Cin=128, H=23, W=23, k=3, stride=2, pad=2, dil=2,
                                             has_bias=False), 2),
    ("linear", LayerSpec("e", "linear", p=136, d=200, T=70), 5),
    ("conv_rows_padD", LayerSpec("e", "conv2d", p=64, Cin=9, H=12, W=12, k=3, pad=1), 4),
]


@pytest.mark.parametrize("tag,spec,B", KEPT, ids=[e[0] for e in KEPT])
def test_kept_gradients_norm_and_sum(lib, tag, spec, B):
    import torch
    dp = lib
    wl = Workload(name=tag, B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=17)
    A, G = workloads.layer_inputs(wl, 0)
    fac = workloads.factor_inputs(wl, B)
    desc = desc_for(dp, spec, B, "bf16")
    nbytes = dp.dp_grads_size(desc)
    width = 88 if tag == "conv_rows_padD" else spec.D      # the padded row layout keeps 81 -> 88 columns
    assert nbytes == 4 * B * spec.p * width + (4 * B * spec.p if spec.has_bias else 0)
    grads = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    ws = torch.empty(dp.dp_workspace_size(desc, dp.DP_NORM_INSTANTIATE), dtype=torch.uint8, device="cuda")
    Ad, Gd = to_dev(A, "bf16"), to_dev(G, "bf16")
    sq = torch.empty(B, dtype=torch.float32, device="cuda")
    dp.dp_layer_sqnorms_keep(desc, Ad, Gd, sq, grads, ws)
    f = torch.tensor(fac, device="cuda")
    dW = torch.empty(spec.p * spec.D, dtype=torch.float32, device="cuda")
    db = torch.empty(spec.p, dtype=torch.float32, device="cuda") if spec.has_bias else None
    dp.dp_clipped_sum_kept(desc, grads, f, dW, db, ws)
    torch.cuda.synchronize()
    assert rel_elem(sq.cpu().numpy(), oracle.layer_sqnorms(spec, A, G)) <= TOL["bf16"]
    S, Sb = oracle.clipped_sum(spec, A, G, fac.astype(np.float64))
    assert rel_rows(dW.cpu().numpy(), S, spec.D) <= TOL["bf16"]
    if spec.has_bias:
        assert rel_rows(db.cpu().numpy(), Sb) <= TOL["bf16"]
    # accumulate: a second call adds the same sum
    dp.dp_clipped_sum_kept(desc, grads, f, dW, db, ws, accumulate=True)
    torch.cuda.synchronize()
    assert rel_rows(dW.cpu().numpy(), 2 * S, spec.D) <= TOL["bf16"]


def test_kept_gradients_unsupported_layers(lib):
    dp = lib
    assert dp.dp_grads_size(dp.layer_desc(dp.DP_LINEAR, dp.DP_FP32, B=4, p=8, T=80, d=16)) == 0    # fp32
    assert dp.dp_grads_size(dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=4, p=8, T=1, d=16)) == 0     # one row
    assert dp.dp_grads_size(dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=4, p=12, T=80, d=16)) == 0   # p % 8


def test_clip_step_with_kept_gradients(lib):
    """A two-layer step with every instantiated layer keeping its gradients equals the oracle."""
    l1 = LayerSpec("a", "conv2d", p=72, Cin=64, H=12, W=12, k=3, pad=1)
    l2 = LayerSpec("b", "linear", p=136, d=200, T=70)
    wl = Workload(name="kept_step", B=4, layers=(l1, l2), dtype="bf16", C=1.0, sigma=0.5, seed=23)
    inputs = [workloads.layer_inputs(wl, l) for l in range(2)]
    ref = oracle.dp_step(wl, inputs)
    step = lib.ClipStep([desc_for(lib, s, wl.B, "bf16") for s in wl.layers], C=1.0, sigma=0.5,
                        norm_modes=[lib.DP_NORM_INSTANTIATE] * 2, keep_grads=True)
    assert all(k is not None for k in step.kept)
    grad = step.run([(to_dev(A, "bf16"), to_dev(G, "bf16")) for A, G in inputs], seed=wl.seed)
    assert rel_flat(grad.cpu().numpy(), ref["noisy"], wl.layers) <= TOL["bf16"]


# The clipped sum reading the NHWC input copy its layer's norm call left in the workspace:
# after a ghost norm (the row-scaled GEMM) and after an instantiated norm (the per-example
# conv kernel); a layer with no such copy (one-row fc) takes the plain path.
REUSE = [
    ("ghost_rows", LayerSpec("e", "conv2d", p=72, Cin=64, H=10, W=10, k=3, pad=1), 3, "GHOST", 1),
    ("ghost_rows_s2_nobias", LayerSpec("e", "conv2d", p=136, Cin=128, H=15, W=15, k=3, stride=2, pad=1,
                                       has_bias=False), 2, "GHOST", 1),
    ("inst_nhwc", LayerSpec("e", "conv2d", p=72, Cin=64, H=12, W=12, k=3, pad=1), 3, "INSTANTIATE", 1),
    ("linear_plain", LayerSpec("e", "linear", p=64, d=96, T=40), 3, "GHOST", 0),
]


@pytest.mark.parametrize("tag,spec,B,mode,level", REUSE, ids=[e[0] for e in REUSE])
def test_clipped_sum_reuses_norm_layouts(lib, tag, spec, B, mode, level):
    import torch
    dp = lib
    m = getattr(dp, "DP_NORM_" + mode)
    wl = Workload(name=tag, B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=29)
    A, G = workloads.layer_inputs(wl, 0)
    fac = workloads.factor_inputs(wl, B)
    desc = desc_for(dp, spec, B, "bf16")
    assert dp.dp_layout_reused(desc, m) == level
    ws = torch.empty(dp.dp_workspace_size(desc, m), dtype=torch.uint8, device="cuda")
    Ad, Gd = to_dev(A, "bf16"), to_dev(G, "bf16")
    sq = torch.empty(B, dtype=torch.float32, device="cuda")
    dp.dp_layer_sqnorms(desc, Ad, Gd, sq, ws, mode=m)
    f = torch.tensor(fac, device="cuda")
    dW = torch.full((spec.p * spec.D,), 0.5, dtype=torch.float32, device="cuda")
    db = torch.full((spec.p,), -1.0, dtype=torch.float32, device="cuda") if spec.has_bias else None
    dp.dp_clipped_sum_reuse(desc, m, Ad, Gd, f, dW, db, ws, accumulate=True)
    torch.cuda.synchronize()
    S, Sb = oracle.clipped_sum(spec, A, G, fac.astype(np.float64))
    assert rel_rows(dW.cpu().numpy() - 0.5, S, spec.D) <= TOL["bf16"]
    if spec.has_bias:
        assert rel_rows(db.cpu().numpy() + 1.0, Sb) <= TOL["bf16"]


def test_mixed_scale_factors_straddle_bound(lib):
    """Some examples under C (factor exactly 1), some over; flat clipping over two layers."""
    import torch
    dp = lib
    l1 = LayerSpec("a", "linear", p=32, d=48, T=16, g_std=0.01)
    l2 = LayerSpec("b", "conv2d", p=8, Cin=4, H=6, W=6, k=3, pad=1, g_std=0.01)
    wl = Workload(name="mixed", B=24, layers=(l1, l2), dtype="bf16", C=1.0, sigma=0.5, seed=5,
                  g_scale="mixed")
    inputs = [workloads.layer_inputs(wl, l) for l in range(2)]
    ref = oracle.dp_step(wl, inputs)
    n = np.sqrt(ref["sqnorms"].sum(0))
    assert (n < 1).sum() >= 3 and (n > 1).sum() >= 3
    step = dp.ClipStep([desc_for(dp, s, wl.B, "bf16") for s in wl.layers], C=1.0, sigma=0.5)
    dev = [(to_dev(A, "bf16"), to_dev(G, "bf16")) for A, G in inputs]
    grad = step.run(dev, seed=wl.seed)
    torch.cuda.synchronize()
    fac = step.factors.cpu().numpy()[0]
    under = n < 1 - 1e-3
    assert np.all(fac[under] == 1.0)
    assert rel_elem(fac, ref["factors"]) <= TOL["bf16"]
    assert rel_flat(grad.cpu().numpy(), ref["noisy"], wl.layers) <= TOL["bf16"]


def test_nonfinite_norm_zeroes_factor_and_raises_status(lib):
    import torch
    dp = lib
    spec = LayerSpec("e", "linear", p=16, d=16, T=4)
    wl = Workload(name="nf", B=4, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=1)
    A, G = workloads.layer_inputs(wl, 0)
    G[2, 1, 3] = np.inf
    assert dp.dp_check_status() == dp.DP_OK
    got = _run_layer(dp, spec, wl, A, G)
    sq = got["sq"]
    fac = torch.empty(4, device="cuda")
    dp.dp_clip_factors(sq.view(1, 4), 4, 1, False, [1.0], fac)
    assert dp.dp_check_status() == dp.DP_ERR_NONFINITE
    assert dp.dp_check_status() == dp.DP_OK      # cleared
    f = fac.cpu().numpy()
    assert f[2] == 0.0 and np.all(np.isfinite(f))


@pytest.mark.parametrize("pin", ["", "rows", "example"], ids=["auto", "rows_gemm", "per_example"])
def test_nonfinite_example_with_factor_zero_in_the_sum(lib, pin, monkeypatch):
    """An example whose G holds inf gets factor 0; in the clipped sum it still meets the
    contraction, so exactly the outputs it touches through the inf become NaN (0 * inf): row
    j of dW and db[j] for G_i[t, j] = inf.  Every other entry equals the sum over the finite
    examples."""
    import torch
    if pin:
        monkeypatch.setenv("DPCLIP_SUM_KERNEL", pin)
    dp = lib
    spec = LayerSpec("e", "linear", p=64, d=128, T=64)
    B = 4
    wl = Workload(name="nf_sum", B=B, layers=(spec,), dtype="bf16", C=1.0, sigma=1.0, seed=3)
    A, G = workloads.layer_inputs(wl, 0)
    G[2, 1, 3] = np.inf
    fac = np.array([0.5, 0.8, 0.0, 1.0], dtype=np.float32)
    desc = desc_for(dp, spec, B, "bf16")
    ws = torch.empty(max(dp.dp_workspace_size(desc), 16), dtype=torch.uint8, device="cuda")
    dW = torch.empty(spec.p * spec.D, device="cuda")
    db = torch.empty(spec.p, device="cuda")
    dp.dp_clipped_sum(desc, to_dev(A, "bf16"), to_dev(G, "bf16"), torch.tensor(fac, device="cuda"), dW, db, ws)
    torch.cuda.synchronize()
    W = dW.cpu().numpy().reshape(spec.p, spec.D)
    b = db.cpu().numpy()
    assert np.all(np.isnan(W[3])) and np.isnan(b[3])
    keep = [i for i in range(B) if i != 2]
    S, Sb = oracle.clipped_sum(spec, A[keep], G[keep], fac[keep].astype(np.float64))
    rows = [j for j in range(spec.p) if j != 3]
    assert rel_rows(W[rows], S.reshape(spec.p, spec.D)[rows], spec.D) <= TOL["bf16"]
    assert rel_rows(b[rows], Sb[rows]) <= TOL["bf16"]


# ----------------------------------------------------------------- noise and adaptive bound

@pytest.mark.parametrize("n,offset", [(1, 0), (3, 5), (7, 2), (1000, 0), (1001, 13), (1 << 20, 3), (1002, 8),
                                      (3 << 20, 4), ((3 << 20) + 3, 12)])
def test_noise_matches_oracle_definition(lib, n, offset):
    import torch
    seed = 0x1234_5678_9ABC
    buf = torch.zeros(n + 1, device="cuda")[1:] if offset % 2 else torch.zeros(n, device="cuda")
    lib.dp_add_noise(buf, 1.0, 1.0, 1, seed, offset)
    z = buf.cpu().numpy().astype(np.float64)
    ref = oracle.normal_noise(n, seed, offset)
    assert np.all(np.abs(z - ref) <= Z_RTOL * np.abs(ref) + Z_ATOL)


def test_noise_scale_and_moments(lib):
    import torch
    n = 1 << 22
    x = torch.zeros(n, device="cuda")
    lib.dp_add_noise(x, 0.7225, 2.0, 16, 99, 0)
    y = x.double().cpu().numpy()
    sd = 0.7225 * 2.0 / 16
    assert abs(y.mean()) < 5 * sd / math.sqrt(n)
    assert y.var() == pytest.approx(sd ** 2, rel=0.01)
    base = torch.linspace(-1, 1, 1000, device="cuda")
    b2 = base.clone()
    lib.dp_add_noise(b2, 0.0, 1.0, 8, 1, 0)
    assert torch.allclose(b2, base / 8, rtol=1e-7, atol=0)


def test_adaptive_bound_matches_oracle(lib):
    import torch
    rng = np.random.default_rng(3)
    s = (rng.random(1024) * 9.0).astype(np.float32)
    sd = torch.tensor(s, device="cuda")
    out = torch.empty(2, device="cuda")
    for layer, C_l2 in ((0, 1.5), (5, 0.8), (8, 10.0)):
        lib.dp_adaptive_bound(sd, 1024, C_l2, 1.1, 2.0, 2.5, 7, layer, out)
        c, cl2 = out.cpu().numpy()
        rc, rcl2 = oracle.adaptive_bound(s.astype(np.float64), C_l2, 1.1, 2.0, 2.5, 7, layer)
        assert c == pytest.approx(rc, rel=1e-5, abs=1e-6)
        assert cl2 == pytest.approx(rcl2, rel=1e-5, abs=1e-6)


def test_adaptive_bounds_of_all_layers_in_one_launch(lib):
    """dp_adaptive_bounds over nine layers (and over layers 64 .. 66) equals one
    dp_adaptive_bound call per layer bit for bit and the oracle per layer; the seed read from
    device memory gives the same values as the seed passed by value."""
    import torch
    rng = np.random.default_rng(5)
    L, B = 9, 1000
    s = (rng.random((L, B)) * rng.uniform(0.5, 20.0, (L, 1))).astype(np.float32)
    C_l2 = [float(c) for c in rng.uniform(0.5, 4.0, L)]
    sd = torch.tensor(s, device="cuda")
    for layer0 in (0, 64):
        n = L if layer0 == 0 else 3
        out = torch.full((n, 2), float("nan"), device="cuda")
        lib.dp_adaptive_bounds(sd[:n], B, C_l2[:n], 1.1, 2.0, 2.5, 11, out, layer0=layer0)
        seed_dev = torch.tensor([11], dtype=torch.int64, device="cuda")
        out_dev = torch.full((n, 2), float("nan"), device="cuda")
        lib.dp_adaptive_bounds(sd[:n], B, C_l2[:n], 1.1, 2.0, 2.5, 999, out_dev, layer0=layer0, seed_dev=seed_dev)
        one = torch.full((2,), float("nan"), device="cuda")
        for k in range(n):
            lib.dp_adaptive_bound(sd[k], B, C_l2[k], 1.1, 2.0, 2.5, 11, layer0 + k, one)
            assert torch.equal(out[k], one), k
            assert torch.equal(out_dev[k], one), k
            rc, rcl2 = oracle.adaptive_bound(s[k].astype(np.float64), C_l2[k], 1.1, 2.0, 2.5, 11, layer0 + k)
            c, cl2 = one.cpu().numpy()
            assert c == pytest.approx(rc, rel=1e-5, abs=1e-6) and cl2 == pytest.approx(rcl2, rel=1e-5, abs=1e-6)


def test_adaptive_bound_nonfinite_norm_raises_status(lib):
    """A non-finite norm raises DP_ERR_NONFINITE and enters the noisy mean at the bound
    (min(inf, C_l2) = C_l2): the oracle's value with that norm set to the bound."""
    import torch
    rng = np.random.default_rng(4)
    s = (rng.random(300) * 4.0).astype(np.float32)
    C_l2 = 1.2
    for bad in (np.inf, np.nan):
        t = s.copy()
        t[17] = bad
        assert lib.dp_check_status() == lib.DP_OK
        out = torch.empty(2, device="cuda")
        lib.dp_adaptive_bound(torch.tensor(t, device="cuda"), 300, C_l2, 1.1, 2.0, 2.5, 5, 3, out)
        assert lib.dp_check_status() == lib.DP_ERR_NONFINITE
        ref = s.astype(np.float64)
        ref[17] = C_l2 * C_l2
        rc, rcl2 = oracle.adaptive_bound(ref, C_l2, 1.1, 2.0, 2.5, 5, 3)
        c, cl2 = out.cpu().numpy()
        assert c == pytest.approx(rc, rel=1e-5, abs=1e-6) and cl2 == pytest.approx(rcl2, rel=1e-5, abs=1e-6)


def test_pipeline_matches_step(lib):
    """ClipPipeline (one graph per step, next batch copied alongside) gives ClipStep.run's result."""
    import torch
    dp = lib
    spec = LayerSpec("e", "linear", p=96, d=80, T=70)
    spec2 = LayerSpec("f", "linear", p=40, d=24, T=1)
    wls = [Workload(name=f"pipe{k}", B=6, layers=(spec, spec2), dtype="bf16", C=1.0, sigma=0.8, seed=20 + k)
           for k in range(4)]
    descs = [desc_for(dp, s_, 6, "bf16") for s_ in (spec, spec2)]
    host = []
    for wl in wls:
        host.append([tuple(workloads.to_torch(x, "bf16") for x in workloads.layer_inputs(wl, l)) for l in range(2)])
    shapes = [(tuple(a.shape), tuple(g.shape)) for a, g in host[0]]
    pipe = dp.ClipPipeline(descs, shapes, "bf16", C=1.0, sigma=0.8)

    def fill(k):
        for (ha, hg), (a, g) in zip(pipe.host_inputs(k), host[k]):
            ha.copy_(a)
            hg.copy_(g)
    fill(0)
    pipe.start()
    got = []
    for k in range(3):
        fill(k + 1)                 # the step copies batch k+1 while it computes batch k
        out = pipe.step(k, 1000 + k)
        torch.cuda.synchronize()
        got.append(out.clone())
    ref = dp.ClipStep(descs, C=1.0, sigma=0.8)
    for k in range(3):
        want = ref.run([(a.cuda(), g.cuda()) for a, g in host[k]], seed=1000 + k).cpu()
        torch.cuda.synchronize()
        assert torch.equal(got[k], want), k
