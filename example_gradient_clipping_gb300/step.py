"""One privatised-gradient step over a list of layers, through the C ABI.

Per step: dp_layer_sqnorms for every layer (ghost norm, instantiation or the
one-row form, layer by layer), dp_clip_factors (flat or per-layer), then for every
layer the clipped sum into one flat fp32 gradient vector [W_0, b_0, W_1, b_1, ...]
with the noise and 1/B added by the same call for linear layers (dp_clipped_sum_noised)
and by one multi-block pass after the sums for conv layers (dp_add_noise_blocks); each
layer's noise is drawn at its flat offset, with its own bound when clipping per layer.
fuse_noise=False runs dp_clipped_sum per layer and dp_add_noise over the vector
instead; the result is bit-identical.  Torch supplies device memory and the stream only.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

from . import (DP_LINEAR, DP_NORM_AUTO, DP_NORM_INSTANTIATE, LayerDesc, dp_adaptive_bounds, dp_add_noise,
               dp_add_noise_blocks, dp_add_noise_devseed, dp_clip_factors,
               dp_clipped_sum, dp_clipped_sum_kept, dp_clipped_sum_kept_noised, dp_clipped_sum_noised,
               dp_clipped_sum_reuse, dp_grads_size, dp_launch_count, dp_layer_sqnorms, dp_layer_sqnorms_keep,
               dp_layout_reused, dp_plan, dp_workspace_size, noise_desc)

# Instantiated layers with at least this many rows per example keep their per-example
# gradients by default (the clipped sum then reads them once instead of recomputing a
# contraction over the rows).
KEEP_MIN_ROWS = 512


class ClipStep:
    """keep_grads: "auto" keeps the per-example gradients of instantiated layers with at
    least KEEP_MIN_ROWS rows (where the library supports it), True keeps them wherever it
    does, False never.

    adaptive: None, or dict(alpha, beta, sigma_l2, C_l2) -- the noisy-mean adaptive bound
    of [ThreeTools] section 3, run per layer on the step's norms right after they are
    formed (dp_adaptive_bounds: every layer in one launch; C_l2 one value or one per layer;
    a captured step reads the noise seed from the same device buffer as the gradient noise).
    Layer l's next bound and next norm bound land in bounds_next[l] = (C_next, C_l2_next) on
    the device; the step's own factors use the bounds it was built with."""

    def __init__(self, descs: Sequence[LayerDesc], C, sigma: float, per_layer: bool = False,
                 norm_modes: Optional[Sequence[int]] = None, device: str = "cuda", keep_grads="auto",
                 fuse_noise: bool = True, adaptive: Optional[dict] = None):
        import torch
        self.fuse_noise = bool(fuse_noise)
        self.descs = list(descs)
        L = len(self.descs)
        self.B = self.descs[0].B
        if any(d.B != self.B for d in self.descs):
            raise ValueError("all layers of a step share the batch size B")
        self.per_layer = bool(per_layer)
        self.C = [float(c) for c in (C if isinstance(C, (list, tuple)) else [C] * L)]
        self.sigma = float(sigma)
        self.modes = list(norm_modes) if norm_modes is not None else [DP_NORM_AUTO] * L
        self.plan = [dp_plan(d, m) for d, m in zip(self.descs, self.modes)]
        self.offsets, o = [], 0
        self.shapes = []
        for d, (_, T, D) in zip(self.descs, self.plan):
            self.offsets.append(o)
            self.shapes.append((d.p, D))
            o += d.p * D + (d.p if d.has_bias else 0)
        self.n_params = o
        ws = max(dp_workspace_size(d, m) for d, m in zip(self.descs, self.modes))
        dev = torch.device(device)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self.sqnorms = torch.empty(L, self.B, dtype=torch.float32, device=dev)
        self.factors = torch.empty((L if self.per_layer else 1), self.B, dtype=torch.float32, device=dev)
        self.grad = torch.empty(self.n_params, dtype=torch.float32, device=dev)
        self.seed_buf = torch.zeros(1, dtype=torch.int64, device=dev)
        self.adaptive = None
        if adaptive is not None:
            cl2 = adaptive["C_l2"]
            cl2 = [float(c) for c in (cl2 if isinstance(cl2, (list, tuple)) else [cl2] * L)]
            self.adaptive = dict(alpha=float(adaptive["alpha"]), beta=float(adaptive["beta"]),
                                 sigma_l2=float(adaptive["sigma_l2"]), C_l2=cl2)
            self.bounds_next = torch.empty(L, 2, dtype=torch.float32, device=dev)
        self.chosen: List[int] = [m for m, _, _ in self.plan]
        self.graph = None
        self.graph_kernels = 0
        self.kept = []
        for d, (m, T, _) in zip(self.descs, self.plan):
            want = keep_grads is True or (keep_grads == "auto" and T >= KEEP_MIN_ROWS)
            nbytes = dp_grads_size(d) if (want and m == DP_NORM_INSTANTIATE) else 0
            self.kept.append(torch.empty(nbytes // 4, dtype=torch.float32, device=dev) if nbytes else None)
        # conv layers whose clipped sum reuses the layouts their norm call wrote get a
        # workspace of their own, so the layouts survive the other layers' calls
        self.own_ws = []
        for l, (d, m) in enumerate(zip(self.descs, self.modes)):
            reuse = self.kept[l] is None and dp_layout_reused(d, m) > 0
            self.own_ws.append(torch.empty(max(dp_workspace_size(d, m), 16), dtype=torch.uint8, device=dev)
                               if reuse else None)

    def layer_views(self, l: int) -> Tuple:
        p, D = self.shapes[l]
        o = self.offsets[l]
        dW = self.grad[o:o + p * D]
        db = self.grad[o + p * D:o + p * D + p] if self.descs[l].has_bias else None
        return dW, db

    def norms(self, inputs, stream=None) -> None:
        for l, (d, (A, G)) in enumerate(zip(self.descs, inputs)):
            if self.kept[l] is not None:
                dp_layer_sqnorms_keep(d, A, G, self.sqnorms[l], self.kept[l], self.workspace, stream=stream)
                self.chosen[l] = DP_NORM_INSTANTIATE
            else:
                ws = self.own_ws[l] if self.own_ws[l] is not None else self.workspace
                self.chosen[l] = dp_layer_sqnorms(d, A, G, self.sqnorms[l], ws, mode=self.modes[l], stream=stream)

    def adaptive_(self, seed: int = 0, seed_dev=None, stream=None) -> None:
        """The adaptive bound of every layer from the norms just formed, all layers in one
        launch (no-op without one); with seed_dev the seed is read from that device buffer."""
        a = self.adaptive
        if a is None:
            return
        for l0 in range(0, len(self.descs), 64):
            l1 = min(len(self.descs), l0 + 64)
            dp_adaptive_bounds(self.sqnorms[l0:l1], self.B, a["C_l2"][l0:l1], a["alpha"], a["beta"], a["sigma_l2"],
                               seed, self.bounds_next[l0:l1], layer0=l0, seed_dev=seed_dev, stream=stream)

    def factors_(self, stream=None) -> None:
        L = len(self.descs)
        dp_clip_factors(self.sqnorms, self.B, L, self.per_layer, self.C if self.per_layer else self.C[:1],
                        self.factors, stream=stream)

    def sums(self, inputs, stream=None) -> None:
        for l, (d, (A, G)) in enumerate(zip(self.descs, inputs)):
            dW, db = self.layer_views(l)
            fac = self.factors[l] if self.per_layer else self.factors[0]
            if self.kept[l] is not None:
                dp_clipped_sum_kept(d, self.kept[l], fac, dW, db, self.workspace, stream=stream)
            elif self.own_ws[l] is not None:
                dp_clipped_sum_reuse(d, self.modes[l], A, G, fac, dW, db, self.own_ws[l], stream=stream)
            else:
                dp_clipped_sum(d, A, G, fac, dW, db, self.workspace, stream=stream)

    def sums_noised(self, inputs, seed: int = 0, seed_dev=None, stream=None) -> None:
        """sums() and noise() together.  Linear layers' clipped sum calls and every layer's
        sum from kept gradients add their blocks' noise and the 1/B scale in the sum's final
        pass (dp_clipped_sum_noised, dp_clipped_sum_kept_noised); the other conv layers'
        weight sums end in a column-mapping pass that does not draw noise, so their blocks get
        theirs from one multi-block noise launch after the sums (dp_add_noise_blocks) instead
        of one noise pass per layer."""
        blocks = []
        for l, (d, (A, G)) in enumerate(zip(self.descs, inputs)):
            dW, db = self.layer_views(l)
            fac = self.factors[l] if self.per_layer else self.factors[0]
            C = self.C[l] if self.per_layer else self.C[0]
            if d.kind != DP_LINEAR and self.kept[l] is None:
                p, D = self.shapes[l]
                blocks.append((self.offsets[l], p * D + (p if d.has_bias else 0), C))
                if self.own_ws[l] is not None:
                    dp_clipped_sum_reuse(d, self.modes[l], A, G, fac, dW, db, self.own_ws[l], stream=stream)
                else:
                    dp_clipped_sum(d, A, G, fac, dW, db, self.workspace, stream=stream)
                continue
            nd = noise_desc(self.sigma, C, self.B, seed, seed_dev, self.offsets[l])
            if self.kept[l] is not None:
                dp_clipped_sum_kept_noised(d, self.kept[l], fac, dW, db, nd, self.workspace, stream=stream)
            else:
                dp_clipped_sum_noised(d, A, G, fac, dW, db, nd, self.workspace, stream=stream)
        if blocks:
            dp_add_noise_blocks(self.grad, blocks, self.sigma, self.B, seed=seed, seed_dev=seed_dev, stream=stream)

    def noise(self, seed: int, stream=None) -> None:
        if not self.per_layer:
            dp_add_noise(self.grad, self.sigma, self.C[0], self.B, seed, 0, stream=stream)
            return
        for l, d in enumerate(self.descs):
            p, D = self.shapes[l]
            n = p * D + (p if d.has_bias else 0)
            o = self.offsets[l]
            dp_add_noise(self.grad[o:o + n], self.sigma, self.C[l], self.B, seed, o, stream=stream)

    def noise_devseed(self, stream=None) -> None:
        """Noise with the seed read from self.seed_buf when the kernels run."""
        if not self.per_layer:
            dp_add_noise_devseed(self.grad, self.sigma, self.C[0], self.B, self.seed_buf, 0, stream=stream)
            return
        for l, d in enumerate(self.descs):
            p, D = self.shapes[l]
            n = p * D + (p if d.has_bias else 0)
            o = self.offsets[l]
            dp_add_noise_devseed(self.grad[o:o + n], self.sigma, self.C[l], self.B, self.seed_buf, o,
                                 stream=stream)

    def sums_and_noise_devseed(self, inputs, stream=None) -> None:
        """The clipped sums and the noise with the seed read from self.seed_buf when the
        kernels run (fused unless fuse_noise is False)."""
        if self.fuse_noise:
            self.sums_noised(inputs, seed_dev=self.seed_buf, stream=stream)
        else:
            self.sums(inputs, stream)
            self.noise_devseed(stream)

    def capture(self, inputs) -> None:
        """Capture one whole step over the device buffers `inputs` in a CUDA graph.

        replay(seed) reruns it (one launch for the step) with noise drawn from `seed`;
        refill the same input buffers between replays to process new batches.
        """
        import torch
        self.run(inputs, seed=0)           # first calls resolve per-device state outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        n0 = dp_launch_count()
        with torch.cuda.graph(g):
            self.norms(inputs)
            self.adaptive_(seed_dev=self.seed_buf)
            self.factors_()
            self.sums_and_noise_devseed(inputs)
        self.graph_kernels = dp_launch_count() - n0
        self.graph = g

    def replay(self, seed: int):
        self.seed_buf.fill_(int(seed))
        self.graph.replay()
        return self.grad

    def run(self, inputs, seed: int, stream=None):
        """Norms (and the adaptive bound) -> factors -> clipped sums -> noise and 1/B; returns
        the flat gradient."""
        self.norms(inputs, stream)
        self.adaptive_(seed, stream)
        self.factors_(stream)
        if self.fuse_noise:
            self.sums_noised(inputs, seed=seed, stream=stream)
        else:
            self.sums(inputs, stream)
            self.noise(seed, stream)
        return self.grad


class VirtualStep:
    """One logical batch processed as physical micro-batches (gradient accumulation, the
    virtual step of [MixGhost] section 5 and Appendix E).

    add(inputs, B) runs one micro-batch of B examples through the same calls as ClipStep
    (norms, factors, clipped sums) and ADDS its clipped sums to the flat gradient; the clip
    factor of an example depends on that example alone, so the split changes nothing.
    finish(seed) then adds the noise N(0, sigma^2 C^2) once and scales by 1/B with B the
    logical batch (every example added since zero()).  `descs` give the layer shapes; their
    B is the largest micro-batch the step will see.
    """

    def __init__(self, descs: Sequence[LayerDesc], C, sigma: float, per_layer: bool = False,
                 norm_modes: Optional[Sequence[int]] = None, device: str = "cuda"):
        import torch
        self.base = ClipStep(descs, C, sigma, per_layer=per_layer, norm_modes=norm_modes, device=device,
                             keep_grads=False)
        b = self.base
        self.grad = b.grad
        L = len(b.descs)
        self.sq_flat = torch.empty(L * b.B, dtype=torch.float32, device=b.grad.device)
        self.fac_flat = torch.empty((L if b.per_layer else 1) * b.B, dtype=torch.float32, device=b.grad.device)
        self.examples = 0
        self.zero()

    def zero(self) -> None:
        self.grad.zero_()
        self.examples = 0

    def add(self, inputs, B: int, stream=None) -> None:
        import torch
        b = self.base
        if not 1 <= B <= b.B:
            raise ValueError(f"micro-batch of {B} examples; this step takes 1..{b.B}")
        L = len(b.descs)
        descs = []
        for d in b.descs:
            dm = type(d).from_buffer_copy(d)
            dm.B = B
            descs.append(dm)
        need = max(dp_workspace_size(d, m) for d, m in zip(descs, b.modes))
        if need > b.workspace.numel():
            b.workspace = torch.empty(need, dtype=torch.uint8, device=b.grad.device)
        sq = self.sq_flat[:L * B].view(L, B)
        fac = self.fac_flat[:(L if b.per_layer else 1) * B].view(-1, B)
        for l, (d, (A, G)) in enumerate(zip(descs, inputs)):
            b.chosen[l] = dp_layer_sqnorms(d, A, G, sq[l], b.workspace, mode=b.modes[l], stream=stream)
        dp_clip_factors(sq, B, L, b.per_layer, b.C if b.per_layer else b.C[:1], fac, stream=stream)
        for l, (d, (A, G)) in enumerate(zip(descs, inputs)):
            dW, db = b.layer_views(l)
            dp_clipped_sum(d, A, G, fac[l] if b.per_layer else fac[0], dW, db, b.workspace, accumulate=True,
                           stream=stream)
        self.examples += B

    def finish(self, seed: int, stream=None):
        """Noise once and 1/B over the logical batch; returns the flat gradient."""
        if self.examples == 0:
            raise ValueError("no micro-batch was added")
        b = self.base
        if not b.per_layer:
            dp_add_noise(self.grad, b.sigma, b.C[0], self.examples, seed, 0, stream=stream)
        else:
            # every layer's block with its own bound, up to 64 blocks a launch (bit-identical to
            # one dp_add_noise per layer)
            blocks = []
            for l, d in enumerate(b.descs):
                p, D = b.shapes[l]
                blocks.append((b.offsets[l], p * D + (p if d.has_bias else 0), b.C[l]))
            for k in range(0, len(blocks), 64):
                dp_add_noise_blocks(self.grad, blocks[k:k + 64], b.sigma, self.examples, seed=seed, stream=stream)
        return self.grad


class ClipPipeline:
    """Privatised-gradient steps over batches that arrive in pinned host memory.

    Two ClipSteps with their own device input buffers alternate.  The step for batch k
    is one CUDA graph: norms, factors, clipped sums and noise on buffer set k % 2, the
    gradient copied back to pinned host memory, and, on a forked stream inside the same
    graph, the copy of batch k+1 from host_inputs(k+1) into the other buffer set, which
    overlaps the compute.  So one graph launch per step drives copies and kernels.

    Use: fill host_inputs(0), call start(); then for each k fill host_inputs(k+1) and
    call step(k, seed); the gradient of batch k is in the returned pinned tensor once
    the stream reaches that point (it is reused by step k+2).  Results are exactly those
    of ClipStep.run on the same batches and seeds.
    """

    kCopyLanes = 1

    def __init__(self, descs, shapes, dtype, C, sigma: float, per_layer: bool = False, device: str = "cuda"):
        import torch
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        dev = torch.device(device)
        self.steps = [ClipStep(descs, C=C, sigma=sigma, per_layer=per_layer, device=str(dev)) for _ in range(2)]
        self.dev_in = [[(torch.zeros(a, dtype=tdt, device=dev), torch.zeros(g, dtype=tdt, device=dev))
                        for a, g in shapes] for _ in range(2)]
        self.host_in = [[(torch.zeros(a, dtype=tdt).pin_memory(), torch.zeros(g, dtype=tdt).pin_memory())
                         for a, g in shapes] for _ in range(2)]
        self.n_params = self.steps[0].n_params
        self.out_host = [torch.empty(self.n_params, dtype=torch.float32).pin_memory() for _ in range(2)]
        n0 = dp_launch_count()
        for st, inp in zip(self.steps, self.dev_in):
            st.run(inp, seed=0)                 # per-device state resolved outside capture
        torch.cuda.synchronize()
        # the next batch's copy runs on kCopyLanes forked streams, each taking a slice of
        # every tensor (one lane measured fastest on GB300: four lanes lowered the rate)
        self.side = [torch.cuda.Stream(dev) for _ in range(self.kCopyLanes)]
        self.graphs = []
        for b in range(2):
            st, cur, nxt = self.steps[b], self.dev_in[b], 1 - b
            g = torch.cuda.CUDAGraph()
            n0 = dp_launch_count()
            with torch.cuda.graph(g):
                cap = torch.cuda.current_stream()
                for lane, sd in enumerate(self.side):
                    sd.wait_stream(cap)
                    with torch.cuda.stream(sd):
                        for (ha, hg), (da, dg) in zip(self.host_in[nxt], self.dev_in[nxt]):
                            for h, d_ in ((ha, da), (hg, dg)):
                                n = h.numel()
                                lo, hi = n * lane // self.kCopyLanes, n * (lane + 1) // self.kCopyLanes
                                if hi > lo:
                                    d_.view(-1)[lo:hi].copy_(h.view(-1)[lo:hi], non_blocking=True)
                st.norms(cur)
                st.factors_()
                st.sums_and_noise_devseed(cur)
                self.out_host[b].copy_(st.grad, non_blocking=True)
                for sd in self.side:
                    cap.wait_stream(sd)
            self.graph_kernels = dp_launch_count() - n0
            self.graphs.append(g)

    def host_inputs(self, k: int):
        """The pinned (A, G) buffers per layer that batch k is read from."""
        return self.host_in[k & 1]

    def start(self) -> None:
        """Copy batch 0 from host_inputs(0) to the device (the graphs copy every later one)."""
        for (ha, hg), (da, dg) in zip(self.host_in[0], self.dev_in[0]):
            da.copy_(ha, non_blocking=True)
            dg.copy_(hg, non_blocking=True)

    def step(self, k: int, seed: int):
        """Batch k's step on the current stream; prefetches batch k+1 from host_inputs(k+1)."""
        b = k & 1
        self.steps[b].seed_buf.fill_(int(seed))
        self.graphs[b].replay()
        return self.out_host[b]
