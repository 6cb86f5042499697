"""Seeded synthetic inputs for the per-example gradient clipping workloads.

This module holds shapes, value distributions and random draws only.  None of
the clipping method's arithmetic (norms, factors, sums, noise) lives here: the
CPU oracle and the CUDA library both take their inputs from it, and it imports
neither of them.

Every tensor is drawn one example at a time from numpy's Philox4x64-10 bit
generator keyed by (seed, tensor id, example index), so any single example can
be regenerated on its own (the oracle checks sampled examples of the large
workloads that way) and the full batch is the concatenation of the examples.

Layer layouts follow PyTorch conventions:
  linear  A [B, T, d]  (layer inputs a_{i,t}),  G [B, T, p]  (output grads)
  conv2d  A [B, Cin, H, W] (NCHW input),        G [B, p, Hout, Wout]
  conv1d  A [B, Cin, W] (NCL input),              G [B, p, Wout]
  conv3d  A [B, Cin, Z, H, W] (NCDHW input),       G [B, p, Zout, Hout, Wout]
bf16 workloads draw fp32 values and round them to bf16 (round to nearest
even); both sides read the rounded values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "LayerSpec", "Workload", "WORKLOADS", "get_workload", "example_inputs",
    "layer_inputs", "factor_inputs", "round_to_dtype", "to_torch",
]


@dataclass(frozen=True)
class LayerSpec:
    """One layer's shapes and the distribution of its captured tensors."""
    name: str
    kind: str                 # "linear", "conv1d", "conv2d" or "conv3d"
    p: int                    # output features / output channels
    d: int = 0                # linear: input features
    T: int = 1                # linear: rows (tokens) per example
    Cin: int = 0              # conv: input channels
    H: int = 0                # conv2d / conv3d
    W: int = 0                # conv2d / conv3d width, conv1d length
    k: int = 1
    stride: int = 1
    pad: int = 0
    dil: int = 1
    has_bias: bool = True
    a_dist: str = "normal"    # "normal" (N(0, a_std^2)) or "abs_normal" (|N(0, a_std^2)|)
    a_std: float = 1.0
    g_std: float = 0.01       # output grads ~ N(0, g_std^2)
    Z: int = 1                # conv3d: input depth

    @property
    def Zout(self) -> int:
        if self.kind != "conv3d":
            return 1
        return (self.Z + 2 * self.pad - self.dil * (self.k - 1) - 1) // self.stride + 1

    @property
    def Hout(self) -> int:
        if self.kind not in ("conv2d", "conv3d"):
            return 1
        return (self.H + 2 * self.pad - self.dil * (self.k - 1) - 1) // self.stride + 1

    @property
    def Wout(self) -> int:
        if self.kind == "linear":
            return 1
        return (self.W + 2 * self.pad - self.dil * (self.k - 1) - 1) // self.stride + 1

    @property
    def rows(self) -> int:
        """T: rows of the per-example contraction (tokens, or Hout*Wout)."""
        return self.T if self.kind == "linear" else self.Zout * self.Hout * self.Wout

    @property
    def D(self) -> int:
        """Width of the (unfolded) input: d, or Cin*k*k."""
        if self.kind == "linear":
            return self.d
        return self.Cin * self.k ** {"conv1d": 1, "conv2d": 2, "conv3d": 3}[self.kind]

    @property
    def n_weight(self) -> int:
        return self.p * self.D

    @property
    def n_params(self) -> int:
        return self.n_weight + (self.p if self.has_bias else 0)

    def a_example_shape(self) -> Tuple[int, ...]:
        if self.kind == "linear":
            return (self.T, self.d)
        if self.kind == "conv3d":
            return (self.Cin, self.Z, self.H, self.W)
        return (self.Cin, self.H, self.W) if self.kind == "conv2d" else (self.Cin, self.W)

    def g_example_shape(self) -> Tuple[int, ...]:
        if self.kind == "linear":
            return (self.T, self.p)
        if self.kind == "conv3d":
            return (self.p, self.Zout, self.Hout, self.Wout)
        return (self.p, self.Hout, self.Wout) if self.kind == "conv2d" else (self.p, self.Wout)


@dataclass(frozen=True)
class Workload:
    """A batch of layers processed by one clipping step."""
    name: str
    B: int
    layers: Tuple[LayerSpec, ...]
    dtype: str                # "fp32" or "bf16"
    C: float                  # flat bound, or the per-layer bound used for every layer
    sigma: float
    per_layer: bool = False
    seed: int = 0
    alpha: Optional[float] = None     # adaptive bound parameters, when used
    beta: Optional[float] = None
    sigma_l2: Optional[float] = None
    g_scale: str = "fixed"    # "fixed", or "mixed": per-example grad multiplier 10^U(-1,1)
    description: str = ""

    @property
    def n_params(self) -> int:
        return sum(l.n_params for l in self.layers)

    def param_offsets(self) -> List[int]:
        """First index of each layer's block (weight, then bias) in the flat parameter vector."""
        offs, o = [], 0
        for l in self.layers:
            offs.append(o)
            o += l.n_params
        return offs

    def with_batch(self, B: int) -> "Workload":
        return replace(self, B=B)


def _vgg11_cifar_layers() -> Tuple[LayerSpec, ...]:
    # VGG-11 (configuration "A"): conv widths 64-128-256-256-512-512-512-512 with
    # 2x2 max-pools after convs 1, 2, 4, 6 and 8, on 3x32x32 CIFAR images, then a
    # 512->10 classifier.  Spatial size per conv: 32, 16, 8, 8, 4, 4, 2, 2.
    widths = [64, 128, 256, 256, 512, 512, 512, 512]
    sizes = [32, 16, 8, 8, 4, 4, 2, 2]
    layers, cin = [], 3
    for j, (w, s) in enumerate(zip(widths, sizes)):
        layers.append(LayerSpec(name=f"conv{j + 1}", kind="conv2d", p=w, Cin=cin, H=s, W=s,
                                k=3, stride=1, pad=1, a_dist="abs_normal", g_std=0.01))
        cin = w
    layers.append(LayerSpec(name="fc", kind="linear", p=10, d=512, T=1,
                            a_dist="abs_normal", g_std=0.01))
    return tuple(layers)


WORKLOADS: Dict[str, Workload] = {
    # Single linear layer, one row per example.
    "t1_linear_b32": Workload(
        name="t1_linear_b32", B=32, dtype="fp32", C=1.0, sigma=1.0, seed=0,
        layers=(LayerSpec(name="fc", kind="linear", p=128, d=256, T=1, g_std=0.01),),
        description="single linear layer, T=1: B=32, d=256, p=128, fp32, flat C=1, sigma=1"),
    # Transformer-shaped sequence linear layer (ghost-norm regime, 2T^2 << p*d).
    "seq_linear_b64_t128": Workload(
        name="seq_linear_b64_t128", B=64, dtype="bf16", C=1.0, sigma=1.0, seed=0,
        layers=(LayerSpec(name="proj", kind="linear", p=768, d=768, T=128, g_std=0.01),),
        description="sequence linear layer: B=64, T=128, d=768, p=768, bf16, C=1, sigma=1"),
    # conv2d 3x3 s1 p1 on 64x32x32 (instantiation regime, 2T^2 > p*D).
    "conv3x3_b256": Workload(
        name="conv3x3_b256", B=256, dtype="bf16", C=1.0, sigma=1.0, seed=0,
        layers=(LayerSpec(name="conv", kind="conv2d", p=64, Cin=64, H=32, W=32, k=3,
                          stride=1, pad=1, a_dist="abs_normal", g_std=0.01),),
        description="conv2d 3x3 s1 p1: B=256, 64x32x32 -> 64 ch (T=1024, D=576), bf16, C=1"),
    # Whole VGG-11 CIFAR stack, per-layer bounds and the adaptive bound.
    "vgg11_cifar_b1024": Workload(
        name="vgg11_cifar_b1024", B=1024, dtype="bf16", C=2.0, sigma=0.7225, seed=0,
        per_layer=True, alpha=1.1, beta=2.0, sigma_l2=2.5, layers=_vgg11_cifar_layers(),
        description="VGG-11 CIFAR stack (8 conv + fc): B=1024, bf16, per-layer C=2, "
                    "sigma=0.7225, adaptive alpha=1.1 beta=2 sigma_l2=2.5"),
    # The same stack clipped flat (one bound over all layers).
    "vgg11_cifar_b1024_flat": Workload(
        name="vgg11_cifar_b1024_flat", B=1024, dtype="bf16", C=2.0, sigma=0.7225, seed=0,
        per_layer=False, layers=_vgg11_cifar_layers(),
        description="VGG-11 CIFAR stack (8 conv + fc): B=1024, bf16, flat C=2, sigma=0.7225"),
    # ViT-Base MLP pair at large batch.
    "vit_mlp_b4096_t197": Workload(
        name="vit_mlp_b4096_t197", B=4096, dtype="bf16", C=1.0, sigma=1.0, seed=0,
        layers=(LayerSpec(name="fc1", kind="linear", p=3072, d=768, T=197, g_std=0.01),
                LayerSpec(name="fc2", kind="linear", p=768, d=3072, T=197, g_std=0.01)),
        description="ViT-Base MLP: B=4096, T=197, 768->3072 and 3072->768, bf16, flat C=1"),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


# Tensor ids: layer l's A is 2l+1, its G is 2l+2; per-example grad multipliers
# (mixed-scale variant) and externally supplied factors have ids of their own.
_TID_SCALE = 1_000_001
_TID_FACTORS = 1_000_002


def _gen(seed: int, tensor_id: int, example: int) -> np.random.Generator:
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF,
                    ((tensor_id & 0xFFFFFFFF) << 32) | (example & 0xFFFFFFFF)], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to the workload dtype, returned as fp32 (exactly representable)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "fp32":
        return x
    if dtype != "bf16":
        raise ValueError(dtype)
    import torch
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()


def _grad_multiplier(wl: Workload, i: int) -> float:
    if wl.g_scale == "fixed":
        return 1.0
    u = _gen(wl.seed, _TID_SCALE, i).random()
    return float(10.0 ** (2.0 * u - 1.0))


def example_inputs(wl: Workload, layer: int, i: int) -> Tuple[np.ndarray, np.ndarray]:
    """(A_i, G_i) of example i at layer `layer`, fp32, already rounded to the workload dtype."""
    spec = wl.layers[layer]
    ga = _gen(wl.seed, 2 * layer + 1, i)
    a = ga.standard_normal(spec.a_example_shape(), dtype=np.float32)
    if spec.a_dist == "abs_normal":
        np.abs(a, out=a)
    elif spec.a_dist != "normal":
        raise ValueError(spec.a_dist)
    if spec.a_std != 1.0:
        a *= np.float32(spec.a_std)
    gg = _gen(wl.seed, 2 * layer + 2, i)
    g = gg.standard_normal(spec.g_example_shape(), dtype=np.float32)
    g *= np.float32(spec.g_std * _grad_multiplier(wl, i))
    return round_to_dtype(a, wl.dtype), round_to_dtype(g, wl.dtype)


def layer_inputs(wl: Workload, layer: int, examples: Optional[Sequence[int]] = None,
                 threads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Stacked (A, G) for the given examples (default: the whole batch), fp32 arrays."""
    spec = wl.layers[layer]
    idx = list(range(wl.B)) if examples is None else list(examples)
    A = np.empty((len(idx),) + spec.a_example_shape(), dtype=np.float32)
    G = np.empty((len(idx),) + spec.g_example_shape(), dtype=np.float32)

    def fill(j: int) -> None:
        A[j], G[j] = example_inputs(wl, layer, idx[j])

    if threads and len(idx) > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(len(idx))))
    else:
        for j in range(len(idx)):
            fill(j)
    return A, G


def device_layer_inputs(wl: Workload, layer: int, device: str = "cuda"):
    """(A, G) of the whole batch drawn on `device` by torch's seeded generator.

    For the full-size workloads, whose host-side generation would take minutes.
    Same shapes and distributions as layer_inputs (the values differ); the tests
    copy sampled examples back to the host for the oracle, so both sides still read
    the same numbers.  Returned in the workload dtype.
    """
    import torch
    spec = wl.layers[layer]
    gen = torch.Generator(device=device)
    gen.manual_seed((wl.seed * 1_000_003 + 2 * layer + 1) & 0x7FFFFFFFFFFFFFFF)
    A = torch.randn((wl.B,) + spec.a_example_shape(), generator=gen, device=device, dtype=torch.float32)
    if spec.a_dist == "abs_normal":
        A.abs_()
    if spec.a_std != 1.0:
        A.mul_(spec.a_std)
    gen.manual_seed((wl.seed * 1_000_003 + 2 * layer + 2) & 0x7FFFFFFFFFFFFFFF)
    G = torch.randn((wl.B,) + spec.g_example_shape(), generator=gen, device=device, dtype=torch.float32)
    G.mul_(spec.g_std)
    if wl.dtype == "bf16":
        A, G = A.to(torch.bfloat16), G.to(torch.bfloat16)
    return A, G


def factor_inputs(wl: Workload, n: int, low: float = 0.0, high: float = 1.0) -> np.ndarray:
    """Externally supplied clip factors in [low, high) (for testing the clipped sum alone)."""
    return _gen(wl.seed, _TID_FACTORS, 0).uniform(low, high, size=n).astype(np.float32)


def to_torch(x: np.ndarray, dtype: str, device: str = "cpu"):
    """Torch tensor of the workload dtype holding x (x already rounded)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.to(device)
