"""Plain float64 definition of DP-SGD per-example clipping (oracle).

TEST INFRASTRUCTURE ONLY (see the package header).

Pages cited (by title):
  [FastClip]  "Scaling up Differentially Private Deep Learning with Fast
              Per-Example Gradient Clipping" (arXiv 2009.03106)
  [ThreeTools] "Three Tools for Practical Differential Privacy" (arXiv 1812.02890)
  [MixGhost]  "Scalable and Efficient Training of Large Convolutional Neural
              Networks with Differential Privacy" (arXiv 2205.10683)
  [Blog]      "Privacy-Preserving Deep Learning: A Deep Dive into DP-SGD"

Layouts: linear A [B,T,d], G [B,T,p]; conv2d A [B,Cin,H,W], G [B,p,Hout,Wout].
Per-example weight gradient [p, D] (D = d, or Cin*k*k in (c, kh, kw) order, the
layout of a PyTorch weight), bias gradient [p].
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Union

import numpy as np

from .philox import normal_noise

NONFINITE = "nonfinite"


def unfold2d(x: np.ndarray, k: int, stride: int = 1, pad: int = 0, dil: int = 1) -> np.ndarray:
    """U(a_i): explicit im2col of one example x [Cin, H, W] -> [T, D].

    [MixGhost] section 2.3 and Appendix B (the unfold U and the PyTorch Unfold
    ordering); [FastClip] section 4, convolutional layers (im2col turns the
    per-example convolution into one GEMM).  Row t = h_out*Wout + w_out, column
    c*k*k + kh*k + kw; out-of-image taps read the zero padding.
    """
    x = np.asarray(x, dtype=np.float64)
    Cin, H, W = x.shape
    Hout = (H + 2 * pad - dil * (k - 1) - 1) // stride + 1
    Wout = (W + 2 * pad - dil * (k - 1) - 1) // stride + 1
    xp = np.zeros((Cin, H + 2 * pad, W + 2 * pad))
    xp[:, pad:pad + H, pad:pad + W] = x
    U = np.empty((Hout * Wout, Cin * k * k))
    for c in range(Cin):
        for kh in range(k):
            for kw in range(k):
                h0, w0 = kh * dil, kw * dil
                patch = xp[c, h0:h0 + stride * (Hout - 1) + 1:stride,
                           w0:w0 + stride * (Wout - 1) + 1:stride]
                U[:, c * k * k + kh * k + kw] = patch.reshape(-1)
    return U


def unfold1d(x: np.ndarray, k: int, stride: int = 1, pad: int = 0, dil: int = 1) -> np.ndarray:
    """U(a_i) of a 1-D convolution: one example x [Cin, L] -> [Lout, Cin*k].

    The 1-D case of the unfold ([MixGhost] section 2.3 and Appendix B treat 1D to 3D
    convolutions alike): row t = output position, column c*k + kw (the order of a
    PyTorch Conv1d weight [p, Cin, k]); taps outside the input read the zero padding.
    """
    x = np.asarray(x, dtype=np.float64)
    Cin, L = x.shape
    Lout = (L + 2 * pad - dil * (k - 1) - 1) // stride + 1
    U = np.zeros((Lout, Cin * k))
    for t in range(Lout):
        for c in range(Cin):
            for kw in range(k):
                pos = t * stride - pad + kw * dil
                if 0 <= pos < L:
                    U[t, c * k + kw] = x[c, pos]
    return U


def unfold3d(x: np.ndarray, k: int, stride: int = 1, pad: int = 0, dil: int = 1) -> np.ndarray:
    """U(a_i) of a 3-D convolution: one example x [Cin, Z, H, W] -> [Zout*Hout*Wout, Cin*k^3].

    The 3-D case of the unfold ([MixGhost] section 2.3 and Appendix B): row
    t = (zo*Hout + ho)*Wout + wo, column ((c*k + kd)*k + kh)*k + kw (the order of a
    PyTorch Conv3d weight [p, Cin, k, k, k]); taps outside the input read the padding.
    """
    x = np.asarray(x, dtype=np.float64)
    Cin, Z, H, W = x.shape
    o = lambda n: (n + 2 * pad - dil * (k - 1) - 1) // stride + 1
    Zo, Ho, Wo = o(Z), o(H), o(W)
    xp = np.zeros((Cin, Z + 2 * pad, H + 2 * pad, W + 2 * pad))
    xp[:, pad:pad + Z, pad:pad + H, pad:pad + W] = x
    U = np.empty((Zo * Ho * Wo, Cin * k ** 3))
    for c in range(Cin):
        for kd in range(k):
            for kh in range(k):
                for kw in range(k):
                    z0, h0, w0 = kd * dil, kh * dil, kw * dil
                    patch = xp[c, z0:z0 + stride * (Zo - 1) + 1:stride, h0:h0 + stride * (Ho - 1) + 1:stride,
                               w0:w0 + stride * (Wo - 1) + 1:stride]
                    U[:, ((c * k + kd) * k + kh) * k + kw] = patch.reshape(-1)
    return U


def per_example_grad(spec, a_i: np.ndarray, g_i: np.ndarray):
    """Materialised per-example gradient of one layer: (weight [p, D], bias [p]).

    Linear: dL_i/dW = sum_t g_{i,t} a_{i,t}^T = G_i^T A_i ([MixGhost] section 2.2,
    eq. 2.4; for one row the outer product of [FastClip] section 4, eq. 6).
    Conv: dL_i/dW = F^{-1}(dL/ds_i)^T U(a_i) ([MixGhost] section 2.3, eq. 2.6;
    [FastClip] Algorithm 3 via im2col).  Bias: dL_i/db = sum over rows of the
    output gradient ([FastClip] section 4, the bias-term derivative).
    """
    g = np.asarray(g_i, dtype=np.float64)
    if spec.kind == "linear":
        A = np.asarray(a_i, dtype=np.float64).reshape(spec.T, spec.d)
        Gm = g.reshape(spec.T, spec.p)
        gw = Gm.T @ A
        gb = Gm.sum(axis=0)
    elif spec.kind == "conv2d":
        U = unfold2d(a_i, spec.k, spec.stride, spec.pad, spec.dil)
        Gm = g.reshape(spec.p, spec.Hout * spec.Wout)      # F^{-1}: flatten the output map
        gw = Gm @ U
        gb = Gm.sum(axis=1)
    elif spec.kind == "conv3d":
        U = unfold3d(a_i, spec.k, spec.stride, spec.pad, spec.dil)
        Gm = g.reshape(spec.p, spec.Zout * spec.Hout * spec.Wout)
        gw = Gm @ U
        gb = Gm.sum(axis=1)
    elif spec.kind == "conv1d":
        U = unfold1d(a_i, spec.k, spec.stride, spec.pad, spec.dil)
        Gm = g.reshape(spec.p, spec.Wout)
        gw = Gm @ U
        gb = Gm.sum(axis=1)
    else:
        raise ValueError(spec.kind)
    return gw, gb


def layer_sqnorms(spec, A: np.ndarray, G: np.ndarray) -> np.ndarray:
    """s_i = ||dL_i/dW||_F^2 + ||dL_i/db||^2 for every example of one layer.

    The squared Frobenius norm of the materialised per-example gradient, the
    quantity [MixGhost] section 3.1 and Appendix C.4 compute by instantiation
    (and the ghost norm of eq. 2.7 reproduces).  The bias joins the layer's norm
    (the per-example norm covers all parameters: [Blog], the norm over all
    parameter gradients of one example).
    """
    B = A.shape[0]
    s = np.empty(B)
    for i in range(B):
        gw, gb = per_example_grad(spec, A[i], G[i])
        s[i] = np.sum(gw * gw) + (np.sum(gb * gb) if spec.has_bias else 0.0)
    return s


def _factor(n: float, C: float) -> float:
    # clip_c(z) = z if ||z|| <= c, else c z/||z||  ([FastClip] section 2; the factor
    # min(R/||g||, 1) of [MixGhost] Appendix C).  No epsilon in the denominator.
    if not np.isfinite(n):
        return 0.0
    return 1.0 if n <= C else C / n


def clip_factors(sqnorms: np.ndarray, C: Union[float, Sequence[float]], per_layer: bool):
    """Clip factors from per-(layer, example) squared norms [L, B].

    Flat: n_i = sqrt(sum_l s_{l,i}), c_i = min(1, C/n_i) -> [B].
    Per-layer ([ThreeTools] section 2: layers clipped independently with their
    own bound): c_{l,i} = min(1, C_l/sqrt(s_{l,i})) -> [L, B].
    A non-finite norm gives factor 0 and the flag NONFINITE in the returned set.
    """
    s = np.atleast_2d(np.asarray(sqnorms, dtype=np.float64))
    L, B = s.shape
    flags = set()
    if not per_layer:
        C0 = float(np.ravel([C])[0])
        n = np.sqrt(s.sum(axis=0))
        out = np.array([_factor(n[i], C0) for i in range(B)])
    else:
        Cl = np.broadcast_to(np.asarray(C, dtype=np.float64), (L,))
        n = np.sqrt(s)
        out = np.array([[_factor(n[l, i], Cl[l]) for i in range(B)] for l in range(L)])
    if not np.all(np.isfinite(n)):
        flags.add(NONFINITE)
    return out, flags


def clipped_sum(spec, A: np.ndarray, G: np.ndarray, factors: np.ndarray):
    """S = sum_i c_i dL_i/dW and Sb = sum_i c_i dL_i/db, summed explicitly.

    The clipped sum of [FastClip] section 2 (the sum of clip_c of each term) and
    the weighted gradient sum_i C_i g_i of [MixGhost] eq. 2.1 / Appendix C.5,
    formed here by materialising each g_i, scaling it and adding (not by the
    reweighted contraction the CUDA path uses).
    """
    S = np.zeros((spec.p, spec.D))
    Sb = np.zeros(spec.p)
    for i in range(A.shape[0]):
        c = float(factors[i])
        if c == 0.0:
            continue
        gw, gb = per_example_grad(spec, A[i], G[i])
        S += c * gw
        Sb += c * gb
    return S, (Sb if spec.has_bias else None)


def clipped_sum_elements(spec, A: np.ndarray, G: np.ndarray, factors: np.ndarray, rows, cols):
    """Selected entries of the clipped sum: S[j, m] for j in rows, m in cols, and Sb[j].

    The quantity of clipped_sum (sum_i c_i g_i: [FastClip] section 2, [MixGhost] eq. 2.1
    and Appendix C.5) written entry by entry from the per-example gradient's definition
    g_i[j, m] = sum_t G_i[t, j] U(A_i)[t, m] and b_i[j] = sum_t G_i[t, j] ([MixGhost]
    eq. 2.4 for linear layers, eq. 2.6 for convolutions), so that a few entries of a large
    layer cost O(B T) each.  Column m of a convolution's unfold, m = c*k^n + (tap), reads
    input channel c alone (Appendix B), so each example is unfolded over just the channels
    the requested columns read.  Examples with factor 0 are skipped, as in clipped_sum.
    Returns (S_sel [len(rows), len(cols)], Sb_sel [len(rows)] or None without a bias).
    """
    rows = np.asarray(rows, dtype=np.int64).ravel()
    cols = np.asarray(cols, dtype=np.int64).ravel()
    S = np.zeros((rows.size, cols.size))
    Sb = np.zeros(rows.size)
    if spec.kind != "linear":
        taps = spec.k ** {"conv1d": 1, "conv2d": 2, "conv3d": 3}[spec.kind]
        chans = np.unique(cols // taps)                       # input channels the columns read
        sub_col = np.searchsorted(chans, cols // taps) * taps + cols % taps
        unfold = {"conv1d": unfold1d, "conv2d": unfold2d, "conv3d": unfold3d}[spec.kind]
    for i in range(A.shape[0]):
        c = float(factors[i])
        if c == 0.0:
            continue
        if spec.kind == "linear":
            U = np.asarray(np.asarray(A[i]).reshape(spec.T, spec.d)[:, cols], dtype=np.float64)
            Gt = np.asarray(np.asarray(G[i]).reshape(spec.T, spec.p)[:, rows], dtype=np.float64)
        else:
            U = unfold(np.asarray(A[i])[chans], spec.k, spec.stride, spec.pad, spec.dil)[:, sub_col]
            Gt = np.asarray(np.asarray(G[i]).reshape(spec.p, -1)[rows], dtype=np.float64).T
        S += c * (Gt.T @ U)
        Sb += c * Gt.sum(axis=0)
    return S, (Sb if spec.has_bias else None)


def add_noise(x: np.ndarray, sigma: float, C: float, B: int, seed: int, offset: int = 0,
              stream: int = 0) -> np.ndarray:
    """(x + sigma*C*z) / B with z the seeded standard normals of elements offset.. .

    The Gaussian mechanism on the clipped sum, then the 1/B average ([FastClip]
    section 2; [MixGhost] eq. 2.1; the noise N(0, sigma^2 C^2 I) of [Blog]).  The
    noise enters before the 1/B scale (the reading of eq. 2.1 and of
    [ThreeTools]' bracket; the blog's code adds it after averaging).
    """
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    z = normal_noise(x.size, seed, offset, stream)
    return (x + sigma * C * z) / B


def adaptive_bound(sqnorms_l: np.ndarray, C_l2: float, alpha: float, beta: float,
                   sigma_l2: float, seed: int, layer: int):
    """Noisy-mean adaptive clipping bound of one layer ([ThreeTools] section 3).

    C_next = alpha/|L| * (sum_i clip(||g_i||) + N(0, sigma_l2^2 C_l2^2)),
    clip(y) = y / max(1, y/C_l2), and the next norm bound C_l2' = beta*C_next.
    The normal draw is element `layer` of noise stream 1 under `seed`.
    """
    n = np.sqrt(np.asarray(sqnorms_l, dtype=np.float64))
    B = n.size
    clipped = np.array([v / max(1.0, v / C_l2) for v in n])
    z = normal_noise(1, seed, offset=layer, stream=1)[0]
    C_next = alpha / B * (clipped.sum() + sigma_l2 * C_l2 * z)
    return C_next, beta * C_next


def norm_mode_plan(spec) -> str:
    """Layerwise choice of how the norm is formed ([MixGhost] section 4, eq. 4.1).

    The pages choose the more memory-efficient of the ghost norm (space 2T^2)
    and instantiation (space p*D).  Our reading: ghost iff 2T^2 < p*D, strict;
    ties instantiate.  One row (T=1) uses the outer-product closed form.
    The result does not depend on the choice; only the cost does.
    """
    T = spec.rows
    if T == 1:
        return "t1"
    return "ghost" if 2 * T * T < spec.p * spec.D else "instantiate"


def norm_mode_plan_time(spec) -> str:
    """Speed-priority variant of the layerwise choice ([MixGhost] section 4, the
    version that compares time complexities; the counts are its Table 1 / Appendix C).

    Per example: the ghost norm forms two T x T Grams (2T^2 D + 2T^2 p flop) and their
    Hadamard sum (2T^2); instantiation forms the p x D gradient (2TpD) and squares
    and sums it (2pD).  Ghost iff its count is strictly smaller; ties instantiate.
    One row (T=1) uses the outer-product closed form.
    """
    T, p, D = spec.rows, spec.p, spec.D
    if T == 1:
        return "t1"
    ghost = 2 * T * T * D + 2 * T * T * p + 2 * T * T
    inst = 2 * T * p * D + 2 * p * D
    return "ghost" if ghost < inst else "instantiate"


def dp_step(wl, inputs: List, seed: Optional[int] = None, C: Optional[Sequence[float]] = None,
            per_layer: Optional[bool] = None) -> Dict:
    """One privatised gradient: norms -> factors -> clipped sums -> noise, 1/B.

    inputs: list of (A, G) per layer.  Flat clipping uses one bound C; per-layer
    clipping uses C_l per layer and adds N(0, sigma^2 C_l^2) to that layer's
    sums.  Returns sqnorms [L,B], factors, pre-noise sums per layer and the
    noisy flat parameter vector (weight then bias for each layer).
    """
    seed = wl.seed if seed is None else seed
    per_layer = wl.per_layer if per_layer is None else per_layer
    L = len(wl.layers)
    if C is None:
        C = [wl.C] * L
    C = list(np.broadcast_to(np.asarray(C, dtype=np.float64), (L,)))
    sq = np.stack([layer_sqnorms(spec, *inputs[l]) for l, spec in enumerate(wl.layers)])
    fac, flags = clip_factors(sq, C if per_layer else C[0], per_layer)
    sums, noisy = [], []
    offs = wl.param_offsets()
    for l, spec in enumerate(wl.layers):
        f = fac[l] if per_layer else fac
        S, Sb = clipped_sum(spec, *inputs[l], f)
        sums.append((S, Sb))
        flat = S.reshape(-1) if Sb is None else np.concatenate([S.reshape(-1), Sb])
        Cl = C[l] if per_layer else C[0]
        noisy.append(add_noise(flat, wl.sigma, Cl, inputs[l][0].shape[0], seed, offs[l]))
    return dict(sqnorms=sq, factors=fac, flags=flags, sums=sums, noisy=np.concatenate(noisy))
