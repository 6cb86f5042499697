"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each check compares the oracle with something other than itself: a library
routine (torch autograd, torch.nn.functional.unfold, torch.nn.grad.conv2d_weight,
numpy's Philox4x64-10, scipy's normal CDF), brute force on tiny inputs, a closed
form, or an invariant of the clip rule.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import dpsgd, philox
from workloads import LayerSpec, Workload, example_inputs, layer_inputs, get_workload

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _lin(T, d, p, bias=True):
    return LayerSpec(name="l", kind="linear", p=p, d=d, T=T, has_bias=bias)


def _conv(Cin, H, W, p, k, stride=1, pad=0, dil=1, bias=True):
    return LayerSpec(name="c", kind="conv2d", p=p, Cin=Cin, H=H, W=W, k=k, stride=stride,
                     pad=pad, dil=dil, has_bias=bias)


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- per-example gradients

def _torch_linear_grad(a, g, bias=True):
    """Per-example gradient by autograd of loss = <G, A W^T + b>."""
    A = torch.tensor(a, dtype=torch.float64)
    G = torch.tensor(g, dtype=torch.float64)
    W = torch.zeros(G.shape[-1], A.shape[-1], dtype=torch.float64, requires_grad=True)
    b = torch.zeros(G.shape[-1], dtype=torch.float64, requires_grad=True)
    out = A @ W.T + (b if bias else 0.0)
    (out * G).sum().backward()
    return W.grad.numpy(), b.grad.numpy()


def _torch_conv_grad(a, g, k, stride, pad, dil):
    x = torch.tensor(a, dtype=torch.float64)
    G = torch.tensor(g, dtype=torch.float64)
    if x.dim() == 3:
        x, G = x[None], G[None]
    W = torch.zeros(G.shape[1], x.shape[1], k, k, dtype=torch.float64, requires_grad=True)
    b = torch.zeros(G.shape[1], dtype=torch.float64, requires_grad=True)
    out = torch.nn.functional.conv2d(x, W, b, stride=stride, padding=pad, dilation=dil)
    assert out.shape == G.shape
    (out * G).sum().backward()
    return W.grad.reshape(G.shape[1], -1).numpy(), b.grad.numpy()


@pytest.mark.parametrize("T,d,p", [(1, 5, 3), (4, 7, 6), (9, 16, 5)])
def test_linear_per_example_grad_matches_autograd(T, d, p):
    rng = np.random.default_rng(1)
    spec = _lin(T, d, p)
    a, g = _rand(rng, T, d), _rand(rng, T, p)
    gw, gb = dpsgd.per_example_grad(spec, a, g)
    tw, tb = _torch_linear_grad(a, g)
    np.testing.assert_allclose(gw, tw, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(gb, tb, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("Cin,H,W,p,k,stride,pad,dil", [
    (3, 8, 8, 4, 3, 1, 1, 1), (2, 7, 9, 3, 3, 2, 1, 1), (4, 6, 6, 5, 1, 1, 0, 1),
    (2, 9, 7, 3, 3, 1, 2, 2), (3, 5, 5, 2, 5, 1, 2, 1)])
def test_conv_per_example_grad_matches_autograd(Cin, H, W, p, k, stride, pad, dil):
    rng = np.random.default_rng(2)
    spec = _conv(Cin, H, W, p, k, stride, pad, dil)
    a = _rand(rng, Cin, H, W)
    g = _rand(rng, p, spec.Hout, spec.Wout)
    gw, gb = dpsgd.per_example_grad(spec, a, g)
    tw, tb = _torch_conv_grad(a, g, k, stride, pad, dil)
    np.testing.assert_allclose(gw, tw, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gb, tb, rtol=1e-12, atol=1e-12)
    # the library's own weight-gradient routine, example by example
    cw = torch.nn.grad.conv2d_weight(torch.tensor(a)[None], (p, Cin, k, k), torch.tensor(g)[None],
                                     stride=stride, padding=pad, dilation=dil)
    np.testing.assert_allclose(gw, cw.reshape(p, -1).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("Cin,L,p,k,stride,pad,dil", [
    (3, 20, 4, 3, 1, 1, 1), (2, 17, 3, 5, 2, 2, 1), (4, 9, 5, 1, 1, 0, 1), (2, 15, 3, 3, 1, 2, 2)])
def test_conv1d_per_example_grad_matches_autograd(Cin, L, p, k, stride, pad, dil):
    rng = np.random.default_rng(5)
    spec = LayerSpec("c1", "conv1d", p=p, Cin=Cin, W=L, k=k, stride=stride, pad=pad, dil=dil)
    a = _rand(rng, Cin, L)
    g = _rand(rng, p, spec.Wout)
    gw, gb = dpsgd.per_example_grad(spec, a, g)
    x = torch.tensor(a)[None]
    W = torch.zeros(p, Cin, k, dtype=torch.float64, requires_grad=True)
    b = torch.zeros(p, dtype=torch.float64, requires_grad=True)
    out = torch.nn.functional.conv1d(x, W, b, stride=stride, padding=pad, dilation=dil)
    assert out.shape[1:] == g.shape
    (out[0] * torch.tensor(g)).sum().backward()
    np.testing.assert_allclose(gw, W.grad.reshape(p, -1).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gb, b.grad.numpy(), rtol=1e-12, atol=1e-12)
    # a conv1d is the conv2d of one input row with a 1 x k kernel
    U1 = dpsgd.unfold1d(a, k, stride, pad, dil)
    tu = torch.nn.functional.unfold(torch.tensor(a)[:, None, :][None], (1, k), dilation=(1, dil),
                                    padding=(0, pad), stride=(1, stride))
    np.testing.assert_array_equal(U1, tu[0].T.numpy())


@pytest.mark.parametrize("Cin,Z,H,W,p,k,stride,pad,dil", [
    (2, 5, 6, 4, 3, 3, 1, 1, 1), (3, 7, 5, 6, 2, 3, 2, 1, 1), (2, 4, 4, 5, 3, 1, 1, 0, 1),
    (1, 6, 7, 6, 2, 2, 1, 1, 2)])
def test_conv3d_per_example_grad_matches_autograd(Cin, Z, H, W, p, k, stride, pad, dil):
    rng = np.random.default_rng(6)
    spec = LayerSpec("c3", "conv3d", p=p, Cin=Cin, Z=Z, H=H, W=W, k=k, stride=stride, pad=pad, dil=dil)
    a = _rand(rng, Cin, Z, H, W)
    g = _rand(rng, p, spec.Zout, spec.Hout, spec.Wout)
    gw, gb = dpsgd.per_example_grad(spec, a, g)
    x = torch.tensor(a)[None]
    Wt = torch.zeros(p, Cin, k, k, k, dtype=torch.float64, requires_grad=True)
    b = torch.zeros(p, dtype=torch.float64, requires_grad=True)
    out = torch.nn.functional.conv3d(x, Wt, b, stride=stride, padding=pad, dilation=dil)
    assert out.shape[1:] == g.shape
    (out[0] * torch.tensor(g)).sum().backward()
    np.testing.assert_allclose(gw, Wt.grad.reshape(p, -1).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gb, b.grad.numpy(), rtol=1e-12, atol=1e-12)
    # each depth tap kd of the 3-D unfold is the 2-D unfold of input slice zo*stride - pad + kd*dil
    U3 = dpsgd.unfold3d(a, k, stride, pad, dil).reshape(spec.Zout, spec.Hout * spec.Wout, Cin, k, k * k)
    for zo in range(spec.Zout):
        for kd in range(k):
            z = zo * stride - pad + kd * dil
            sl = a[:, z] if 0 <= z < Z else np.zeros((Cin, H, W))
            U2 = dpsgd.unfold2d(sl, k, stride, pad, dil).reshape(spec.Hout * spec.Wout, Cin, k * k)
            np.testing.assert_array_equal(U3[zo, :, :, kd], U2)


@pytest.mark.parametrize("k,stride,pad,dil", [(3, 1, 1, 1), (3, 2, 0, 1), (2, 1, 1, 2), (1, 1, 0, 1)])
def test_unfold_matches_torch_unfold(k, stride, pad, dil):
    rng = np.random.default_rng(3)
    x = _rand(rng, 3, 7, 6)
    U = dpsgd.unfold2d(x, k, stride, pad, dil)
    tu = torch.nn.functional.unfold(torch.tensor(x)[None], k, dilation=dil, padding=pad, stride=stride)
    np.testing.assert_array_equal(U, tu[0].T.numpy())


# ---------------------------------------------------------------- norms

def test_sqnorm_brute_force_tiny():
    """s_i = sum_{j,k} (sum_t G[t,j] A[t,k])^2 + sum_j (sum_t G[t,j])^2, by plain loops."""
    rng = np.random.default_rng(4)
    T, d, p, B = 3, 4, 5, 3
    spec = _lin(T, d, p)
    A, G = _rand(rng, B, T, d), _rand(rng, B, T, p)
    s = dpsgd.layer_sqnorms(spec, A, G)
    for i in range(B):
        tot = 0.0
        for j in range(p):
            for kk in range(d):
                v = 0.0
                for t in range(T):
                    v += G[i, t, j] * A[i, t, kk]
                tot += v * v
        for j in range(p):
            v = sum(G[i, t, j] for t in range(T))
            tot += v * v
        assert s[i] == pytest.approx(tot, rel=1e-13)


@pytest.mark.parametrize("T,d,p", [(2, 3, 4), (5, 6, 3), (4, 2, 6)])
def test_ghost_identity_brute_force(T, d, p):
    """||G^T A||_F^2 = sum_{t,s} (a_t . a_s)(g_t . g_s) (the ghost norm, [MixGhost] eq. 2.7)."""
    rng = np.random.default_rng(5)
    spec = _lin(T, d, p, bias=False)
    A, G = _rand(rng, 1, T, d), _rand(rng, 1, T, p)
    ghost = 0.0
    for t in range(T):
        for s_ in range(T):
            aa = sum(A[0, t, k] * A[0, s_, k] for k in range(d))
            gg = sum(G[0, t, j] * G[0, s_, j] for j in range(p))
            ghost += aa * gg
    assert dpsgd.layer_sqnorms(spec, A, G)[0] == pytest.approx(ghost, rel=1e-12)


def test_ghost_identity_conv_brute_force():
    """Conv ghost norm: Grams of the unfolded input and of the flattened output grad."""
    rng = np.random.default_rng(6)
    spec = _conv(2, 4, 4, 3, 3, 1, 1, 1, bias=False)
    a, g = _rand(rng, 2, 4, 4), _rand(rng, 3, 4, 4)
    # unfold by the library, ghost sum by loops
    U = torch.nn.functional.unfold(torch.tensor(a)[None], 3, padding=1)[0].T.numpy()
    Gm = g.reshape(3, 16).T
    ghost = 0.0
    for t in range(16):
        for s_ in range(16):
            ghost += float(U[t] @ U[s_]) * float(Gm[t] @ Gm[s_])
    assert dpsgd.layer_sqnorms(spec, a[None], g[None])[0] == pytest.approx(ghost, rel=1e-12)


def test_t1_closed_form():
    """One row: ||g a^T||_F^2 = ||a||^2 ||g||^2, plus ||g||^2 for the bias ([FastClip] eq. 6)."""
    rng = np.random.default_rng(7)
    spec = _lin(1, 9, 4)
    A, G = _rand(rng, 6, 1, 9), _rand(rng, 6, 1, 4)
    s = dpsgd.layer_sqnorms(spec, A, G)
    for i in range(6):
        na, ng = np.linalg.norm(A[i, 0]), np.linalg.norm(G[i, 0])
        assert s[i] == pytest.approx(na ** 2 * ng ** 2 + ng ** 2, rel=1e-13)


def test_sqnorm_against_torch_vmap_norm():
    """Per-example norms equal those of autograd gradients taken one example at a time."""
    rng = np.random.default_rng(8)
    spec = _conv(3, 6, 6, 4, 3, 1, 1, 1)
    A, G = _rand(rng, 4, 3, 6, 6), _rand(rng, 4, 4, 6, 6)
    s = dpsgd.layer_sqnorms(spec, A, G)
    for i in range(4):
        tw, tb = _torch_conv_grad(A[i], G[i], 3, 1, 1, 1)
        assert s[i] == pytest.approx(np.sum(tw ** 2) + np.sum(tb ** 2), rel=1e-12)


# ---------------------------------------------------------------- clip factors

def _mixed_workload():
    spec = _lin(5, 12, 7)
    return Workload(name="mixed", B=40, layers=(spec,), dtype="fp32", C=1.0, sigma=1.0,
                    g_scale="mixed", seed=3)


def test_clip_invariants_mixed_scale():
    """clip_c keeps ||.|| <= c, is the identity below c and keeps the direction ([FastClip] section 2)."""
    wl = _mixed_workload()
    spec = wl.layers[0]
    A, G = layer_inputs(wl, 0)
    # make the scales straddle C
    G = G * 6.0
    s = dpsgd.layer_sqnorms(spec, A, G)
    n = np.sqrt(s)
    assert (n < 1.0).sum() >= 5 and (n > 1.0).sum() >= 5
    c, flags = dpsgd.clip_factors(s[None], 1.0, per_layer=False)
    assert not flags
    for i in range(wl.B):
        gw, gb = dpsgd.per_example_grad(spec, A[i], G[i])
        v = np.concatenate([gw.ravel(), gb])
        cv = c[i] * v
        assert np.linalg.norm(cv) <= 1.0 * (1 + 1e-12)
        if n[i] <= 1.0:
            assert c[i] == 1.0
        else:
            assert c[i] < 1.0
            assert np.linalg.norm(cv) == pytest.approx(1.0, rel=1e-12)
        cosang = float(cv @ v) / (np.linalg.norm(cv) * np.linalg.norm(v))
        assert cosang == pytest.approx(1.0, abs=1e-12)


def test_clip_factor_special_values():
    s = np.array([[0.0, 1.0, 4.0, 0.25, np.inf, np.nan]])
    c, flags = dpsgd.clip_factors(s, 1.0, per_layer=False)
    assert list(c) == [1.0, 1.0, 0.5, 1.0, 0.0, 0.0]
    assert oracle.NONFINITE in flags


def test_flat_sums_layers_per_layer_does_not():
    s = np.array([[0.64, 9.0], [0.36, 16.0]])
    flat, _ = dpsgd.clip_factors(s, 1.0, per_layer=False)
    np.testing.assert_allclose(flat, [1.0, 1.0 / 5.0])
    per, _ = dpsgd.clip_factors(s, [1.0, 2.0], per_layer=True)
    np.testing.assert_allclose(per, [[1.0, 1.0 / 3.0], [1.0, 2.0 / 4.0]])


# ---------------------------------------------------------------- clipped sum

def test_unclipped_sum_is_batch_gradient_linear():
    """With c_i = 1 the clipped sum is the ordinary batch gradient (autograd over the batch)."""
    rng = np.random.default_rng(9)
    spec = _lin(6, 10, 7)
    A, G = _rand(rng, 5, 6, 10), _rand(rng, 5, 6, 7)
    S, Sb = dpsgd.clipped_sum(spec, A, G, np.ones(5))
    tw, tb = _torch_linear_grad(A.reshape(-1, 10), G.reshape(-1, 7))
    np.testing.assert_allclose(S, tw, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Sb, tb, rtol=1e-12, atol=1e-12)


def test_unclipped_sum_is_batch_gradient_conv():
    rng = np.random.default_rng(10)
    spec = _conv(3, 8, 8, 4, 3, 1, 1, 1)
    A, G = _rand(rng, 4, 3, 8, 8), _rand(rng, 4, 4, 8, 8)
    S, Sb = dpsgd.clipped_sum(spec, A, G, np.ones(4))
    cw = torch.nn.grad.conv2d_weight(torch.tensor(A), (4, 3, 3, 3), torch.tensor(G), padding=1)
    np.testing.assert_allclose(S, cw.reshape(4, -1).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Sb, G.sum(axis=(0, 2, 3)), rtol=1e-12, atol=1e-12)


def test_clipped_sum_linear_in_factors_and_additive_over_batch():
    """Reweighting is linear in c and the sum splits over disjoint halves of the batch."""
    rng = np.random.default_rng(11)
    spec = _lin(4, 6, 5)
    A, G = _rand(rng, 8, 4, 6), _rand(rng, 8, 4, 5)
    c1, c2 = rng.random(8), rng.random(8)
    S1, b1 = dpsgd.clipped_sum(spec, A, G, c1)
    S2, b2 = dpsgd.clipped_sum(spec, A, G, c2)
    S3, b3 = dpsgd.clipped_sum(spec, A, G, 2.0 * c1 - 0.5 * c2)
    np.testing.assert_allclose(S3, 2.0 * S1 - 0.5 * S2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b3, 2.0 * b1 - 0.5 * b2, rtol=1e-12, atol=1e-12)
    Sa, ba = dpsgd.clipped_sum(spec, A[:3], G[:3], c1[:3])
    Sb_, bb = dpsgd.clipped_sum(spec, A[3:], G[3:], c1[3:])
    np.testing.assert_allclose(Sa + Sb_, S1, rtol=1e-12, atol=1e-12)
    # one example with factor c contributes c * its own autograd gradient
    tw, tb = _torch_linear_grad(A[2], G[2])
    S, b = dpsgd.clipped_sum(spec, A[2:3], G[2:3], np.array([0.3]))
    np.testing.assert_allclose(S, 0.3 * tw, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("spec", [
    _lin(7, 19, 11), _lin(1, 9, 6, bias=False),
    _conv(5, 9, 7, 6, 3, 2, 1, 1), _conv(3, 8, 8, 4, 3, 1, 2, 2, bias=False),
    LayerSpec(name="c1", kind="conv1d", p=5, Cin=4, W=17, k=3, stride=2, pad=1),
    LayerSpec(name="c3", kind="conv3d", p=3, Cin=3, Z=5, H=4, W=6, k=2, stride=1, pad=1, dil=2)],
    ids=["linear", "linear_t1_nobias", "conv2d_s2", "conv2d_dil_nobias", "conv1d", "conv3d"])
def test_clipped_sum_elements_match_the_full_sum(spec):
    """Entry-wise clipped sum = the selected entries of the materialised sum, for every
    entry and for scattered, repeated and unordered index lists."""
    rng = np.random.default_rng(31)
    B = 4
    A = _rand(rng, B, *spec.a_example_shape())
    G = _rand(rng, B, *spec.g_example_shape())
    c = rng.random(B)
    c[1] = 0.0
    S, Sb = dpsgd.clipped_sum(spec, A, G, c)
    Se, Sbe = dpsgd.clipped_sum_elements(spec, A, G, c, np.arange(spec.p), np.arange(spec.D))
    np.testing.assert_allclose(Se, S, rtol=1e-12, atol=1e-12)
    if spec.has_bias:
        np.testing.assert_allclose(Sbe, Sb, rtol=1e-12, atol=1e-12)
    else:
        assert Sbe is None
    rows = [spec.p - 1, 0, spec.p // 2, spec.p - 1]
    cols = [spec.D - 1, 3, 0, spec.D // 2, 3]
    Se, Sbe = dpsgd.clipped_sum_elements(spec, A, G, c, rows, cols)
    np.testing.assert_allclose(Se, S[np.ix_(rows, cols)], rtol=1e-12, atol=1e-12)
    if spec.has_bias:
        np.testing.assert_allclose(Sbe, Sb[rows], rtol=1e-12, atol=1e-12)


def test_clipped_sum_elements_linear_entry_by_brute_force():
    """One entry of a linear layer's clipped sum by plain loops over examples and rows."""
    rng = np.random.default_rng(32)
    spec = _lin(5, 4, 3)
    A, G, c = _rand(rng, 3, 5, 4), _rand(rng, 3, 5, 3), rng.random(3)
    j, m = 2, 1
    want = sum(c[i] * sum(G[i, t, j] * A[i, t, m] for t in range(5)) for i in range(3))
    Se, Sbe = dpsgd.clipped_sum_elements(spec, A, G, c, [j], [m])
    assert Se[0, 0] == pytest.approx(want, rel=1e-13)
    assert Sbe[0] == pytest.approx(sum(c[i] * G[i, :, j].sum() for i in range(3)), rel=1e-13)


# ---------------------------------------------------------------- noise

def test_philox4x64_matches_numpy():
    """The shared round function, at W=64, equals numpy's Philox4x64-10 bit for bit."""
    rng = np.random.default_rng(12)
    for _ in range(20):
        ctr = [int(x) for x in rng.integers(0, 2 ** 63, size=4, dtype=np.uint64)]
        key = [int(x) for x in rng.integers(0, 2 ** 63, size=2, dtype=np.uint64)]
        key[1] |= 1 << 63
        out = [int(v) for v in philox.philox4(ctr, key, width=64)]
        # numpy advances its counter before each block
        prev = (ctr[0] + (ctr[1] << 64) + (ctr[2] << 128) + (ctr[3] << 192) - 1) % (1 << 256)
        bg = np.random.Philox(counter=np.array([(prev >> (64 * j)) & (2 ** 64 - 1) for j in range(4)],
                                               dtype=np.uint64),
                              key=np.array(key, dtype=np.uint64))
        ref = [int(v) for v in bg.random_raw(4)]
        assert out == ref


def test_philox4x32_avalanche_and_uniformity():
    """At W=32: one flipped counter bit flips half the output bits; output bytes are uniform."""
    rng = np.random.default_rng(13)
    n = 4096
    ctr = [rng.integers(0, 2 ** 32, size=n, dtype=np.uint64) for _ in range(4)]
    key = (0x243F6A88, 0x85A308D3)
    base = np.stack(philox.philox4(ctr, key, 32), axis=1)
    frac = []
    for word in range(4):
        for bit in (0, 7, 19, 31):
            c2 = [c.copy() for c in ctr]
            c2[word] ^= np.uint64(1 << bit)
            o = np.stack(philox.philox4(c2, key, 32), axis=1)
            x = base ^ o
            flips = sum(int(bin(int(v)).count("1")) for v in x[:256].ravel())
            frac.append(flips / (256 * 128))
    assert 0.47 < np.mean(frac) < 0.53 and min(frac) > 0.45
    q = np.arange(1 << 18, dtype=np.uint64)
    words = np.stack(philox.philox4((q, q * 0, q * 0, q * 0), (1, 2), 32), axis=1).ravel()
    counts = np.bincount((words >> np.uint64(24)).astype(np.int64), minlength=256)
    exp = words.size / 256
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 400  # 255 dof: mean 255, sd ~22.6


def test_noise_is_standard_normal():
    """Box-Muller output passes a KS test against the normal CDF; moments match."""
    from scipy import stats
    z = philox.normal_noise(1 << 20, seed=0)
    assert abs(z.mean()) < 5 / math.sqrt(z.size)
    assert z.var() == pytest.approx(1.0, rel=0.01)
    assert stats.kstest(z, "norm").pvalue > 1e-3
    # pairs from the same block are uncorrelated
    zz = z[: (z.size // 4) * 4].reshape(-1, 4)
    assert abs(np.corrcoef(zz[:, 0], zz[:, 1])[0, 1]) < 0.01


def test_noise_offsets_are_windows_of_one_stream():
    z = philox.normal_noise(1000, seed=7)
    np.testing.assert_array_equal(philox.normal_noise(13, seed=7, offset=501), z[501:514])
    assert not np.allclose(philox.normal_noise(100, seed=8), z[:100])
    assert not np.allclose(philox.normal_noise(100, seed=7, stream=1), z[:100])


def test_box_muller_special_points():
    """u1 = 1/4 puts the pair at angle pi/2: z0 = 0 and z1 = sqrt(-2 ln u0)."""
    words = np.array([[0x80000000, 0x40000000, 0xFFFFFFFF, 0]], dtype=np.uint64)
    u = philox.uniform_from_word(words)[0]
    assert u[0] == (2 ** 22 + 0.5) / 2 ** 23 and u[2] == ((2 ** 23 - 1) + 0.5) / 2 ** 23
    assert 0 < u.min() and u.max() < 1


def test_add_noise_scale_and_variance():
    """(x + sigma C z)/B: sigma = 0 gives x/B; the noise alone has variance (sigma C / B)^2."""
    x = np.linspace(-1, 1, 200_000)
    np.testing.assert_allclose(dpsgd.add_noise(x, 0.0, 1.0, 8, seed=1), x / 8, rtol=0, atol=0)
    y = dpsgd.add_noise(np.zeros(400_000), 0.7225, 2.0, 16, seed=5)
    assert y.std() == pytest.approx(0.7225 * 2.0 / 16, rel=0.01)
    assert abs(y.mean()) < 5 * 0.7225 * 2.0 / 16 / math.sqrt(y.size)


# ---------------------------------------------------------------- adaptive bound

def test_adaptive_bound_special_cases():
    rng = np.random.default_rng(14)
    spec = _lin(3, 5, 4)
    A, G = _rand(rng, 10, 3, 5), _rand(rng, 10, 3, 4)
    s = dpsgd.layer_sqnorms(spec, A, G)
    norms = [np.linalg.norm(np.concatenate([w.ravel(), b])) for w, b in
             (_torch_linear_grad(A[i], G[i]) for i in range(10))]
    # no clipping, no noise: alpha times the mean norm
    c, cl2 = dpsgd.adaptive_bound(s, 1e30, 1.1, 2.0, 0.0, seed=0, layer=0)
    assert c == pytest.approx(1.1 * np.mean(norms), rel=1e-12)
    assert cl2 == pytest.approx(2.0 * c, rel=1e-15)
    # everything clipped: alpha times the bound
    c, _ = dpsgd.adaptive_bound(s, 1e-3, 1.1, 2.0, 0.0, seed=0, layer=0)
    assert c == pytest.approx(1.1e-3, rel=1e-12)
    # the noise term has standard deviation alpha sigma_l2 C_l2 / B
    draws = [dpsgd.adaptive_bound(s, 1e-3, 1.1, 2.0, 2.5, seed=sd, layer=3)[0] for sd in range(3000)]
    assert np.std(draws) == pytest.approx(1.1 * 2.5 * 1e-3 / 10, rel=0.06)


# ---------------------------------------------------------------- whole step

def test_dp_step_flat_equals_per_layer_for_one_layer():
    wl = Workload(name="one", B=6, layers=(_lin(3, 4, 5),), dtype="fp32", C=0.5, sigma=1.0, seed=2)
    inp = [layer_inputs(wl, 0)]
    a = dpsgd.dp_step(wl, inp, per_layer=False)
    b = dpsgd.dp_step(wl, inp, per_layer=True)
    np.testing.assert_array_equal(a["factors"], b["factors"][0])
    np.testing.assert_array_equal(a["noisy"], b["noisy"])


def test_dp_step_noise_only_when_grads_vanish():
    spec = _lin(2, 3, 4)
    wl = Workload(name="z", B=4, layers=(spec, spec), dtype="fp32", C=2.0, sigma=0.5, seed=9)
    zeros = (np.zeros((4, 2, 3)), np.zeros((4, 2, 4)))
    out = dpsgd.dp_step(wl, [zeros, zeros])
    assert np.all(out["factors"] == 1.0)
    z = philox.normal_noise(wl.n_params, seed=9)
    np.testing.assert_allclose(out["noisy"], 0.5 * 2.0 * z / 4, rtol=1e-15)


def test_layerwise_decision_golden():
    """Ghost vs instantiation for the VGG-11 CIFAR stack, against the hand-derived table."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "vgg11_cifar_decisions.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    wl = get_workload("vgg11_cifar_b1024")
    assert len(rows) == len(wl.layers)
    for spec, row in zip(wl.layers, rows):
        name, T, D, p, ghost_space, inst_space, mode = row
        assert (spec.name, spec.rows, spec.D, spec.p) == (name, int(T), int(D), int(p))
        assert 2 * spec.rows ** 2 == int(ghost_space) and spec.p * spec.D == int(inst_space)
        assert dpsgd.norm_mode_plan(spec) == mode


def test_speed_priority_counts_match_loop_nests():
    """The speed-priority plan's per-example counts, pinned by counting the arithmetic of
    the two algorithms as plain loop nests on tiny shapes (multiply and add = 2 flop)."""
    T, p, D = 3, 2, 4
    ghost = 0
    for _ in range(T):
        for _ in range(T):
            ghost += 2 * D          # (U U^T)_{ts}: D multiply-adds
            ghost += 2 * p          # (G G^T)_{ts}: p multiply-adds
            ghost += 2              # Hadamard product term, accumulated
    inst = 0
    for _ in range(p):
        for _ in range(D):
            inst += 2 * T           # g[a, b] = sum_t G[t, a] U[t, b]
            inst += 2               # g[a, b]^2, accumulated
    spec = LayerSpec("x", "linear", p=p, d=D, T=T)
    want = "ghost" if ghost < inst else "instantiate"
    assert dpsgd.norm_mode_plan_time(spec) == want
    # the space and speed rules part ways: T=150, p=D=256 -> space 2T^2 = 45000 < 65536
    # (ghost); time 23,085,000 flop (ghost) > 19,791,872 flop (instantiate)
    spec = LayerSpec("y", "linear", p=256, d=256, T=150)
    assert dpsgd.norm_mode_plan(spec) == "ghost"
    assert dpsgd.norm_mode_plan_time(spec) == "instantiate"
    assert dpsgd.norm_mode_plan_time(LayerSpec("z", "linear", p=8, d=8, T=1)) == "t1"


def test_micro_batch_sums_add_up():
    """Gradient accumulation ([MixGhost] section 5, Appendix E): per-example clipping makes
    the clipped sum additive over any split of the batch, and the noise and 1/B of the
    logical batch are applied once to the total."""
    wl = Workload(name="acc", B=7, layers=(LayerSpec("a", "linear", p=5, d=6, T=4),), dtype="fp32",
                  C=0.5, sigma=0.0, seed=3)
    spec = wl.layers[0]
    A, G = layer_inputs(wl, 0)
    sq = dpsgd.layer_sqnorms(spec, A, G)
    fac, _ = dpsgd.clip_factors(sq[None, :], 0.5, False)
    S, Sb = dpsgd.clipped_sum(spec, A, G, fac)
    S1, Sb1 = dpsgd.clipped_sum(spec, A[:3], G[:3], fac[:3])
    S2, Sb2 = dpsgd.clipped_sum(spec, A[3:], G[3:], fac[3:])
    np.testing.assert_allclose(S1 + S2, S, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(Sb1 + Sb2, Sb, rtol=1e-12, atol=1e-15)
    step = dpsgd.dp_step(wl, [(A, G)])
    np.testing.assert_allclose(step["noisy"], np.concatenate([S.ravel(), Sb]) / 7, rtol=1e-12, atol=1e-15)
