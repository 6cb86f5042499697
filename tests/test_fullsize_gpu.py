"""Full-size workloads on the GPU, checked on what the oracle can compute.

Inputs are drawn on the device by a seeded generator (host generation of the
multi-GB batches would take minutes); sampled examples are copied back for the
oracle.  Norms: sampled examples against the oracle.  Clipped sum: the full-size
launch with dense factors (every example contributes) against the oracle's
entry-wise sum on sampled entries, among them every tile edge of the output and its
ragged last rows and columns; the full-size launch with factors that are zero except
for a sample of examples, against the oracle's whole sum over those examples; and
additivity in the factors over the whole batch.  Flat and per-layer factors of the whole step are checked against the
factor rule applied to the GPU's own norms (the rule alone is what is checked
there; the norms are checked against the oracle).
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import TOL, desc_for, rel_elem, rel_rows

pytestmark = pytest.mark.gpu

SAMPLE = [0, 1, 777, 2049, 4095]


def _sample(B):
    return sorted({i for i in SAMPLE if i < B} | {B - 1})


def _host(x, i):
    return x[i].float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name,cl", [("vit_mlp_b4096_t197", False), ("vgg11_cifar_b1024", False),
                                     ("conv3x3_b256", False), ("seq_linear_b64_t128", False),
                                     ("vgg11_cifar_b1024", True), ("conv3x3_b256", True)],
                         ids=["vit", "vgg", "conv3x3", "seq", "vgg_channels_last", "conv3x3_channels_last"])
def test_full_size_norms_and_sparse_sums(lib, name, cl):
    import torch
    dp = lib
    wl = workloads.get_workload(name)
    idx = _sample(wl.B)
    for l, spec in enumerate(wl.layers):
        A, G = workloads.device_layer_inputs(wl, l)
        lay = dp.DP_NHWC if (cl and spec.kind != "linear") else dp.DP_NCHW
        desc = desc_for(dp, spec, wl.B, wl.dtype, layout=lay)
        if lay == dp.DP_NHWC:       # the same values channels last; the oracle reads channels first
            A, G = A.movedim(1, -1).contiguous(), G.movedim(1, -1).contiguous()
        ws = torch.empty(max(dp.dp_workspace_size(desc), 16), dtype=torch.uint8, device="cuda")
        sq = torch.empty(wl.B, device="cuda")
        dp.dp_layer_sqnorms(desc, A, G, sq, ws)
        # sparse factors: only the sampled examples contribute
        fac = np.zeros(wl.B, dtype=np.float32)
        fac[idx] = np.linspace(0.3, 1.0, len(idx), dtype=np.float32)
        f = torch.tensor(fac, device="cuda")
        dW = torch.empty(spec.p * spec.D, device="cuda")
        db = torch.empty(spec.p, device="cuda")
        dp.dp_clipped_sum(desc, A, G, f, dW, db, ws)
        torch.cuda.synchronize()
        a_s = np.stack([_host(A, i) for i in idx])
        g_s = np.stack([_host(G, i) for i in idx])
        if lay == dp.DP_NHWC:
            a_s, g_s = np.moveaxis(a_s, -1, 1), np.moveaxis(g_s, -1, 1)
        ref_sq = oracle.layer_sqnorms(spec, a_s, g_s)
        assert rel_elem(sq.cpu().numpy()[idx], ref_sq) <= TOL[wl.dtype], (name, spec.name)
        S, Sb = oracle.clipped_sum(spec, a_s, g_s, fac[idx].astype(np.float64))
        assert rel_rows(dW.cpu().numpy(), S, spec.D) <= TOL[wl.dtype], (name, spec.name)
        assert rel_rows(db.cpu().numpy(), Sb) <= TOL[wl.dtype], (name, spec.name)
        assert np.all(np.isfinite(sq.cpu().numpy())) and np.all(sq.cpu().numpy() > 0)
        del A, G


def _edge_indices(n, rng, k=12):
    """Indices of one output dimension: both ends, both sides of every 64-wide tile edge
    (the kernels' tiles are 64, 128 or 256 wide), the ragged tail, and k random ones."""
    idx = {0, 1, n - 2, n - 1}
    for e in range(64, n, 64):
        idx |= {e - 1, e}
    idx = sorted(i for i in idx if 0 <= i < n)
    if len(idx) > 40:           # wide layers: keep every 256-edge, sample the rest
        keep = [i for i in idx if i < 2 or i >= n - 2 or (i + 1) % 256 in (0, 1)]
        rest = sorted(set(idx) - set(keep))
        idx = sorted(set(keep) | set(rng.choice(rest, 40 - min(len(keep), 40), replace=False).tolist()))
    extra = rng.choice(n, min(k, n), replace=False)
    return np.array(sorted(set(idx) | set(extra.tolist())), dtype=np.int64)


DENSE = [("vit_mlp_b4096_t197", False), ("seq_linear_b64_t128", False), ("conv3x3_b256", False),
         ("conv3x3_b256", True), ("vgg11_cifar_b1024", False)]


@pytest.mark.parametrize("name,cl", DENSE, ids=["vit", "seq", "conv3x3", "conv3x3_channels_last", "vgg"])
def test_full_size_dense_sum_entries(lib, name, cl):
    """Every example contributes (dense factors in [0, 1)): sampled entries of dW and db of
    every layer against the oracle's entry-wise sum, element by element."""
    import torch
    dp = lib
    wl = workloads.get_workload(name)
    rng = np.random.default_rng(7)
    fac = workloads.factor_inputs(wl, wl.B, 0.0, 1.0)
    f = torch.tensor(fac, device="cuda")
    for l, spec in enumerate(wl.layers):
        A, G = workloads.device_layer_inputs(wl, l)
        lay = dp.DP_NHWC if (cl and spec.kind != "linear") else dp.DP_NCHW
        desc = desc_for(dp, spec, wl.B, wl.dtype, layout=lay)
        Ad, Gd = (A.movedim(1, -1).contiguous(), G.movedim(1, -1).contiguous()) if lay == dp.DP_NHWC else (A, G)
        ws = torch.empty(max(dp.dp_workspace_size(desc), 16), dtype=torch.uint8, device="cuda")
        dW = torch.full((spec.p * spec.D,), float("nan"), device="cuda")
        db = torch.full((spec.p,), float("nan"), device="cuda")
        dp.dp_clipped_sum(desc, Ad, Gd, f, dW, db, ws)
        torch.cuda.synchronize()
        del Ad, Gd
        rows, cols = _edge_indices(spec.p, rng), _edge_indices(spec.D, rng)
        if spec.kind == "linear":
            # entry (j, m) of a linear layer's sum reads G's column j and A's column m only:
            # the oracle gets those columns (a layer of width len(cols) -> len(rows))
            sub = workloads.LayerSpec("sub", "linear", p=rows.size, d=cols.size, T=spec.T)
            a_h = A[:, :, torch.tensor(cols, device="cuda")].float().cpu().numpy()
            g_h = G[:, :, torch.tensor(rows, device="cuda")].float().cpu().numpy()
            S, Sb = oracle.clipped_sum_elements(sub, a_h, g_h, fac.astype(np.float64),
                                                np.arange(rows.size), np.arange(cols.size))
        else:
            S, Sb = oracle.clipped_sum_elements(spec, A.float().cpu().numpy(), G.float().cpu().numpy(),
                                                fac.astype(np.float64), rows, cols)
        got = dW.view(spec.p, spec.D).cpu().numpy()[np.ix_(rows, cols)]
        tol = TOL[wl.dtype]
        assert rel_rows(got, S, cols.size) <= tol, (name, spec.name)
        assert rel_rows(db.cpu().numpy()[rows], Sb) <= tol, (name, spec.name)
        # the whole output was written (no entry left at the NaN fill)
        assert bool(torch.isfinite(dW).all()) and bool(torch.isfinite(db).all()), (name, spec.name)
        del A, G


# The per-example kernel scales each example's fp32 product, so linearity holds to fp32
# rounding; the row-scaled kernel rounds the scaled rows c_i G_i to bf16 before the
# MMA (2^-9 relative per element, which over 262,144 terms leaves a few 1e-3 of the
# row's scale on a typical entry and about 1e-2 on the worst of 36,864), so it holds
# to the bf16 path's tolerance.
ADDITIVE = [("vit_mlp_b4096_t197", "", 1e-4), ("conv3x3_b256", "", 1e-4),
            ("conv3x3_b256", "example", 1e-4), ("conv3x3_b256", "rows", 2e-2)]


@pytest.mark.parametrize("name,pin,tol", ADDITIVE, ids=["vit", "conv_im2col", "conv_example", "conv_rows"])
def test_full_size_sum_is_additive_in_factors(lib, name, pin, tol, monkeypatch):
    """sum(c1) + sum(c2) = sum(c1 + c2) over the whole batch (the reweighting is linear)."""
    import torch
    dp = lib
    if pin:
        monkeypatch.setenv("DPCLIP_SUM_KERNEL", pin)
    wl = workloads.get_workload(name)
    spec = wl.layers[0]
    A, G = workloads.device_layer_inputs(wl, 0)
    desc = desc_for(dp, spec, wl.B, wl.dtype)
    ws = torch.empty(max(dp.dp_workspace_size(desc), 16), dtype=torch.uint8, device="cuda")
    c1 = torch.tensor(workloads.factor_inputs(wl, wl.B, 0.0, 0.5), device="cuda")
    c2 = torch.flip(c1, [0]) * 0.7
    outs = []
    for f in (c1, c2, c1 + c2):
        dW = torch.empty(spec.p * spec.D, device="cuda")
        db = torch.empty(spec.p, device="cuda")
        dp.dp_clipped_sum(desc, A, G, f, dW, db, ws)
        outs.append((dW.double(), db.double()))
    torch.cuda.synchronize()
    lhs = (outs[0][0] + outs[1][0]).cpu().numpy()
    assert rel_rows(lhs, outs[2][0].cpu().numpy(), spec.D) <= tol
    lhs_b = (outs[0][1] + outs[1][1]).cpu().numpy()
    assert rel_rows(lhs_b, outs[2][1].cpu().numpy()) <= tol


def test_full_size_vgg_step_flat_and_per_layer_factors(lib):
    """The whole VGG-11 step at B=1024: factors follow the rule on the GPU norms."""
    import torch
    dp = lib
    wl = workloads.get_workload("vgg11_cifar_b1024")
    descs = [desc_for(dp, s, wl.B, wl.dtype) for s in wl.layers]
    inputs = [workloads.device_layer_inputs(wl, l) for l in range(len(wl.layers))]
    for per_layer in (False, True):
        step = dp.ClipStep(descs, C=wl.C, sigma=wl.sigma, per_layer=per_layer)
        g = step.run(inputs, seed=3)
        torch.cuda.synchronize()
        sq = step.sqnorms.double().cpu().numpy()
        want, _ = oracle.clip_factors(sq, wl.C if not per_layer else [wl.C] * len(wl.layers), per_layer)
        got = step.factors.double().cpu().numpy()
        assert rel_elem(got if per_layer else got[0], want) <= 1e-6
        assert np.all(np.isfinite(g.cpu().numpy()))


def test_full_size_conv3x3_kept_gradients_match_recomputed(lib):
    """The 3x3 conv workload at B=256: norms and clipped sum from kept per-example gradients
    equal the instantiated norms and the recomputing clipped sum (both fp32-accumulated)."""
    import torch
    dp = lib
    wl = workloads.get_workload("conv3x3_b256")
    spec = wl.layers[0]
    desc = desc_for(dp, spec, wl.B, wl.dtype)
    A, G = workloads.device_layer_inputs(wl, 0)
    ws = torch.empty(dp.dp_workspace_size(desc, dp.DP_NORM_INSTANTIATE), dtype=torch.uint8, device="cuda")
    grads = torch.empty(dp.dp_grads_size(desc) // 4, dtype=torch.float32, device="cuda")
    sq_k = torch.empty(wl.B, device="cuda")
    sq_r = torch.empty(wl.B, device="cuda")
    dp.dp_layer_sqnorms_keep(desc, A, G, sq_k, grads, ws)
    dp.dp_layer_sqnorms(desc, A, G, sq_r, ws, mode=dp.DP_NORM_INSTANTIATE)
    f = torch.rand(wl.B, device="cuda", generator=torch.Generator("cuda").manual_seed(5))
    outs = []
    for kept in (True, False):
        dW = torch.empty(spec.p * spec.D, device="cuda")
        db = torch.empty(spec.p, device="cuda")
        if kept:
            dp.dp_clipped_sum_kept(desc, grads, f, dW, db, ws)
        else:
            dp.dp_clipped_sum(desc, A, G, f, dW, db, ws)
        outs.append((dW, db))
    torch.cuda.synchronize()
    assert ((sq_k - sq_r).abs() / sq_r.abs()).max().item() <= 1e-5
    assert rel_rows(outs[0][0].cpu().numpy(), outs[1][0].cpu().numpy(), spec.D) <= 1e-5
    assert rel_rows(outs[0][1].cpu().numpy(), outs[1][1].cpu().numpy()) <= 1e-5
