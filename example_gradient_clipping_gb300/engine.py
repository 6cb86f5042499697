"""Privatised gradients for a PyTorch model: A and G captured by autograd hooks.

The pages' privacy engine ([MixGhost] Appendix E; [FastClip] section 2) wraps a model so
that per-example clipping needs a few lines of code: the layer inputs A and the output
gradients G are taken from the ordinary forward and backward passes, the per-example
norms are formed from them (ghost norm or instantiation, [MixGhost] section 4), and the
clipped sum replaces the second back-propagation of the reweighted loss ([MixGhost] section
3.2) with one contraction per layer in this library.

Use (with a summed loss G_i is example i's own gradient; loss_reduction="mean" undoes the
1/B of an averaged loss):

    engine = PrivacyEngine(model, C=1.0, sigma=1.0)
    loss = criterion(model(x), y)          # reduction="sum"
    loss.backward()
    engine.privatise(seed)                 # param.grad <- (sum_i c_i g_i + sigma C z) / B
    optimizer.step()

Layers: nn.Linear (inputs [B, ..., d]; the middle dimensions are the rows T), nn.Conv1d,
nn.Conv2d and nn.Conv3d (square or cubic kernels, equal stride / padding / dilation in every
dimension), the conv layers with groups 1 and zero padding.  Conv2d/Conv3d layers whose input
arrives in PyTorch's channels_last memory format are handed over channels last (no layout
copy); their output gradients are brought to the same format.  Every trainable parameter of
the model must belong to such a layer.
Activations right after them must not be in-place (the backward hook reads the layer's
output gradient).  PyTorch warns that the hook fires on output gradients when the model
input needs no gradient; that gradient is the one wanted here.
"""
from __future__ import annotations

from typing import List, Optional

from . import DP_BF16, DP_CONV1D, DP_CONV2D, DP_CONV3D, DP_FP32, DP_LINEAR, DP_NCHW, DP_NHWC, DP_NORM_AUTO, layer_desc
from .step import ClipStep


class PrivacyEngine:
    def __init__(self, model, C=1.0, sigma: float = 1.0, per_layer: bool = False, norm_mode: int = DP_NORM_AUTO,
                 keep_grads="auto", loss_reduction: str = "sum"):
        """loss_reduction: "sum" (G_i as captured) or "mean" (the captured output gradients
        carry a 1/B factor, undone before the norms)."""
        import torch.nn as nn
        convs = (nn.Conv1d, nn.Conv2d, nn.Conv3d)
        if loss_reduction not in ("sum", "mean"):
            raise ValueError("loss_reduction is 'sum' or 'mean'")
        self.loss_reduction = loss_reduction
        self.model = model
        self.C, self.sigma, self.per_layer = C, float(sigma), bool(per_layer)
        self.norm_mode, self.keep_grads = norm_mode, keep_grads
        self.layers: List = []
        owned = set()
        for m in model.modules():
            if isinstance(m, (nn.Linear,) + convs) and m.weight.requires_grad:
                if isinstance(m, convs):
                    self._check_conv(m)
                if m.bias is not None and not m.bias.requires_grad:
                    raise ValueError(f"{m}: a bias must be trainable with its weight")
                self.layers.append(m)
                owned.add(id(m.weight))
                if m.bias is not None:
                    owned.add(id(m.bias))
        for name, prm in model.named_parameters():
            if prm.requires_grad and id(prm) not in owned:
                raise ValueError(f"parameter {name}: only nn.Linear and nn.Conv1d/2d/3d layers have per-example "
                                 "clipping here; freeze it or leave it out of the model")
        if not self.layers:
            raise ValueError("the model has no trainable nn.Linear or nn.Conv1d/2d/3d layer")
        self._acts: List = [None] * len(self.layers)
        self._grads: List = [None] * len(self.layers)
        self._handles = []
        for i, m in enumerate(self.layers):
            self._handles.append(m.register_forward_hook(self._fwd_hook(i)))
            self._handles.append(m.register_full_backward_pre_hook(self._bwd_hook(i)))
        self._step: Optional[ClipStep] = None
        self._key = None

    @staticmethod
    def _check_conv(m) -> None:
        k, s, p, d = m.kernel_size, m.stride, m.padding, m.dilation
        if isinstance(p, str) or m.groups != 1 or m.padding_mode != "zeros":
            raise ValueError(f"{m}: groups=1 and zero padding given as numbers only")
        if any(len(set(v)) != 1 for v in (k, s, p, d)):
            raise ValueError(f"{m}: square or cubic kernels with equal stride/padding/dilation in every dimension only")

    def _fwd_hook(self, i):
        def hook(module, inputs, output):
            self._acts[i] = inputs[0].detach()
        return hook

    def _bwd_hook(self, i):
        def hook(module, grad_output):       # the gradient of the loss w.r.t. the layer output
            self._grads[i] = grad_output[0].detach()
        return hook

    def detach(self) -> None:
        """Remove the hooks."""
        for h in self._handles:
            h.remove()
        self._handles = []

    @staticmethod
    def _layout(m, a) -> int:
        import torch
        import torch.nn as nn
        if isinstance(m, nn.Conv2d) and a.dim() == 4 and not a.is_contiguous() and \
                a.is_contiguous(memory_format=torch.channels_last):
            return DP_NHWC
        if isinstance(m, nn.Conv3d) and a.dim() == 5 and not a.is_contiguous() and \
                a.is_contiguous(memory_format=torch.channels_last_3d):
            return DP_NHWC
        return DP_NCHW

    @staticmethod
    def _as_layout(x, layout: int, dtype):
        import torch
        x = x.to(dtype)
        if layout == DP_NHWC:
            return x.contiguous(memory_format=torch.channels_last if x.dim() == 4 else torch.channels_last_3d)
        return x.contiguous()

    def _descs(self, B: int, dtype: int, layouts):
        import torch.nn as nn
        out = []
        for m, a, lay in zip(self.layers, self._acts, layouts):
            hb = m.bias is not None
            if isinstance(m, nn.Linear):
                T = a.numel() // (B * m.in_features)
                out.append(layer_desc(DP_LINEAR, dtype, B=B, p=m.out_features, T=T, d=m.in_features, has_bias=hb))
            elif isinstance(m, nn.Conv1d):
                out.append(layer_desc(DP_CONV1D, dtype, B=B, p=m.out_channels, Cin=m.in_channels, H=1, W=a.shape[2],
                                      k=m.kernel_size[0], stride=m.stride[0], pad=m.padding[0], dil=m.dilation[0],
                                      has_bias=hb))
            elif isinstance(m, nn.Conv3d):
                out.append(layer_desc(DP_CONV3D, dtype, B=B, p=m.out_channels, Cin=m.in_channels, Z=a.shape[2],
                                      H=a.shape[3], W=a.shape[4], k=m.kernel_size[0], stride=m.stride[0],
                                      pad=m.padding[0], dil=m.dilation[0], has_bias=hb, layout=lay))
            else:
                out.append(layer_desc(DP_CONV2D, dtype, B=B, p=m.out_channels, Cin=m.in_channels, H=a.shape[2],
                                      W=a.shape[3], k=m.kernel_size[0], stride=m.stride[0], pad=m.padding[0],
                                      dil=m.dilation[0], has_bias=hb, layout=lay))
        return out

    def privatise(self, seed: int, stream=None):
        """Replace every layer's .grad by its privatised gradient; returns the flat vector."""
        import torch
        if any(a is None for a in self._acts) or any(g is None for g in self._grads):
            raise RuntimeError("run the forward pass and loss.backward() first")
        B = self._acts[0].shape[0]
        dt = self._acts[0].dtype
        if dt not in (torch.bfloat16, torch.float32):
            raise ValueError(f"inputs of dtype {dt}: bf16 or fp32 only")
        dtype = DP_BF16 if dt == torch.bfloat16 else DP_FP32
        layouts = [self._layout(m, a) for m, a in zip(self.layers, self._acts)]
        key = (B, dtype, tuple(tuple(a.shape) for a in self._acts), tuple(layouts))
        if self._key != key:
            self._step = ClipStep(self._descs(B, dtype, layouts), C=self.C, sigma=self.sigma, per_layer=self.per_layer,
                                  norm_modes=[self.norm_mode] * len(self.layers), device=str(self._acts[0].device),
                                  keep_grads=self.keep_grads)
            self._key = key
        scale = float(B) if self.loss_reduction == "mean" else 1.0
        inputs = [(self._as_layout(a, lay, dt), self._as_layout(g * scale if scale != 1.0 else g, lay, dt))
                  for a, g, lay in zip(self._acts, self._grads, layouts)]
        flat = self._step.run(inputs, seed=seed, stream=stream)
        for l, m in enumerate(self.layers):
            dW, db = self._step.layer_views(l)
            m.weight.grad = dW.view_as(m.weight).to(m.weight.dtype).clone()
            if m.bias is not None:
                m.bias.grad = db.to(m.bias.dtype).clone()
        self._acts = [None] * len(self.layers)
        self._grads = [None] * len(self.layers)
        return flat
