"""Throughput of the DP-SGD clipping path: per-example norms -> clip factors ->
clipped sum -> Gaussian noise and 1/B, on synthetic inputs resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline]

Prints ONE JSON line on rank 0.  A step is one pass of the whole path over one
batch.  N > 1 (under torchrun) runs independent replicas, one per GPU, each on
its own batch: the path has no data exchange between replicas, so scaling is
weak and there is no collective in the timed work (a barrier brackets it).
`--impl reference` times the float64 CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "examples/sec through norm+clip+noisy-sum per config; % of TC/HBM roofline"
DEFAULT_WORKLOAD = "vit_mlp_b4096_t197"
L2_FLUSH_BYTES = 256 << 20


# inputs with more elements than this are drawn on the device rather than the host
HOST_GEN_LIMIT = 1 << 27


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def layer_desc(dp, spec, B, dtype, layout=0):
    dt = dp.DP_BF16 if dtype == "bf16" else dp.DP_FP32
    if spec.kind == "linear":
        return dp.layer_desc(dp.DP_LINEAR, dt, B=B, p=spec.p, T=spec.T, d=spec.d, has_bias=spec.has_bias)
    if spec.kind == "conv3d":
        return dp.layer_desc(dp.DP_CONV3D, dt, B=B, p=spec.p, Cin=spec.Cin, Z=spec.Z, H=spec.H, W=spec.W, k=spec.k,
                             stride=spec.stride, pad=spec.pad, dil=spec.dil, has_bias=spec.has_bias, layout=layout)
    if spec.kind == "conv1d":
        return dp.layer_desc(dp.DP_CONV1D, dt, B=B, p=spec.p, Cin=spec.Cin, H=1, W=spec.W, k=spec.k,
                             stride=spec.stride, pad=spec.pad, dil=spec.dil, has_bias=spec.has_bias, layout=layout)
    return dp.layer_desc(dp.DP_CONV2D, dt, B=B, p=spec.p, Cin=spec.Cin, H=spec.H, W=spec.W, k=spec.k,
                         stride=spec.stride, pad=spec.pad, dil=spec.dil, has_bias=spec.has_bias, layout=layout)


def step_work(wl, modes, kept=None):
    """Algorithmic FLOPs and bytes of one step, from the per-module complexity counts
    of the mixed-ghost paper (Appendix C): ghost norm 2T^2(D+p) + 2T^2 per example,
    instantiation 2TpD + 2pD, one-row norm 2(D+p), clipped sum 2TpD -- or, for a layer
    that keeps its per-example gradients, the weighted sum 2pD of the kept gradients.
    Bytes: the inputs read once by the norm pass and once by the sum pass (a kept layer:
    its fp32 gradients written by the norm pass and read by the sum pass instead), the
    fp32 gradient written once, and the noise pass reading and writing it."""
    es = 2 if wl.dtype == "bf16" else 4
    kept = kept or [False] * len(wl.layers)
    flop_norm = flop_sum = 0.0
    in_bytes = input_reads = kept_bytes = 0
    for spec, m, kp in zip(wl.layers, modes, kept):
        T, D, p = spec.rows, spec.D, spec.p
        if m == "ghost":
            flop_norm += wl.B * (2.0 * T * T * (D + p) + 2.0 * T * T)
        elif m == "instantiate":
            flop_norm += wl.B * (2.0 * T * p * D + 2.0 * p * D)
        else:
            flop_norm += wl.B * 2.0 * (D + p)
        a_el = math.prod(spec.a_example_shape())
        g_el = math.prod(spec.g_example_shape())
        layer_in = wl.B * (a_el + g_el) * es
        in_bytes += layer_in
        if kp:
            flop_sum += wl.B * 2.0 * p * D
            kept_bytes += wl.B * (p * D + p) * 4
            input_reads += layer_in              # the norm pass only
        else:
            flop_sum += wl.B * 2.0 * T * p * D
            input_reads += 2 * layer_in          # the norm pass and the sum pass
    n = wl.n_params
    return dict(flop_norm=flop_norm, flop_sum=flop_sum, in_bytes=in_bytes, kept_bytes=kept_bytes,
                bytes_total=input_reads + 2 * kept_bytes + 4 * n + 8 * n, n_params=n)


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# Kernels that serve each call on the tensor-core paths (for the DRAM traffic record).
_DOMINANT_KERNELS = {"sums": ["tc_sumx_kernel", "tc_sum_kernel", "tc_conv_kernel", "kept_wsum_direct_kernel"],
                     "norms": ["tc_ghost_kernel", "tc_conv_kernel", "tc_halo_kernel", "tc_unfold_kernel",
                               "tc_sumx_kernel"],
                     "noise": ["add_noise_kernel"], "factors": ["clip_factors_kernel"]}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def _profiled_traffic(workload, call, kernels, B):
    """DRAM bytes (read + write) per launch of the dominant call's kernel from one ncu
    capture, recorded in profiles/dram_traffic.json with the call, the hash of the kernel's
    source file at capture time and the batch the bytes are stated for; None when there is no
    record, the source has changed since or the batch differs."""
    import hashlib
    try:
        with open(TRAFFIC_FILE) as f:
            recs = json.load(f)["records"]
    except (OSError, ValueError, KeyError):
        return None
    for r in recs:
        if (r.get("workload") != workload or r.get("call") != call or r.get("kernel") not in kernels
                or r.get("B") != B):
            continue
        src = os.path.join(ROOT, "example_gradient_clipping_gb300", "csrc", r["source"])
        try:
            cur = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        except OSError:
            return None
        return int(r["dram_bytes_per_launch"]) if cur == r["source_sha256_16"] else None
    return None


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _oracle_batch_size(wl, sample_inputs, per_step_s: float) -> int:
    """Largest sub-batch (doubling from 1, at most B) whose oracle step takes about per_step_s."""
    import oracle
    b = 1
    while b < wl.B:
        t0 = time.perf_counter()
        oracle.dp_step(wl.with_batch(b), sample_inputs(b), seed=wl.seed)
        if time.perf_counter() - t0 >= per_step_s / 2:
            break
        b = min(2 * b, wl.B)
    return b


def cpu_baseline(wl, sample_inputs, budget_s: float = 12.0):
    """Time the float64 CPU oracle (as it stands) on a bounded sample of the workload.

    sample_inputs(b) returns the first b examples' (A, G) per layer as host arrays.
    Full batches when one takes well under the budget, else a sub-batch of the
    same layers; the value is examples per second either way.
    """
    import oracle
    b = _oracle_batch_size(wl, sample_inputs, budget_s / 4)
    sub, inputs = wl.with_batch(b), sample_inputs(b)
    t0 = time.perf_counter()
    runs = 0
    while True:
        oracle.dp_step(sub, inputs, seed=wl.seed + runs)
        runs += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    what = "full batch(es)" if b == wl.B else f"sub-batches of the first {b} examples"
    return dict(value=b * runs / dt, unit="examples/s", cores=_cores(), kind="oracle",
                sample=f"{runs} {what} of {wl.name} (B={wl.B}), float64 numpy, {dt:.1f} s")


def _cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"), default=0)
        if n:
            return n
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, wl):
    import workloads
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    import oracle

    def sample_inputs(b):
        return [workloads.layer_inputs(wl.with_batch(b), l, threads=8) for l in range(len(wl.layers))]

    # each step one bounded sample: the whole run stays within a few minutes
    per_step_s = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    b = _oracle_batch_size(wl, sample_inputs, per_step_s)
    sub, inputs = wl.with_batch(b), sample_inputs(b)
    for w in range(args.warmup):
        oracle.dp_step(sub, inputs, seed=wl.seed + w)
    times = []
    for k in range(args.steps):
        t0 = time.perf_counter()
        oracle.dp_step(sub, inputs, seed=wl.seed + 1000 + k)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = b * args.steps / tot
    what = "full batches" if b == wl.B else f"sub-batches of the first {b} examples"
    cores = _cores()
    line = dict(metric=METRIC, value=value, unit="examples/s", n_gpus=args.gpus, steps=args.steps,
                warmup=args.warmup, ms_per_step=1e3 * tot / args.steps, higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic", impl="reference",
                config=_config(wl), e2e={"value": value, "unit": "examples/s", "h2d_bytes_per_step": 0,
                                         "d2h_bytes_per_step": 0},
                cpu_baseline=dict(value=value, unit="examples/s", cores=cores, kind="oracle",
                                  sample=f"{args.steps} {what} of {wl.name} (B={wl.B}), float64 numpy"))
    print(json.dumps(line), flush=True)


def _config(wl, extra=None):
    c = dict(workload=wl.name, B=wl.B, dtype=wl.dtype, C=wl.C, sigma=wl.sigma,
             clipping="per-layer" if wl.per_layer else "flat",
             layers=[dict(kind=s.kind, T=s.rows, D=s.D, p=s.p) for s in wl.layers],
             l2="flushed between timed steps (256 MiB write)", description=wl.description)
    if extra:
        c.update(extra)
    return c


def max_over_ranks(v: float, device) -> float:
    """The slowest replica's time: MAX all-reduce of one float64 (identity on one process)."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()) \
            or torch.distributed.get_world_size() == 1:
        return float(v)
    t = torch.tensor([float(v)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# The smaller workloads of the metric, each timed on the device after the headline one
# (step time, examples/s and the dominant call's roofline fraction): the one-row layer,
# the sequence layer, the 3x3 conv layer, and the VGG-11 stack clipped per layer (with
# the adaptive bound) and flat.
PER_CONFIG = ("t1_linear_b32", "seq_linear_b64_t128", "conv3x3_b256", "vgg11_cifar_b1024",
              "vgg11_cifar_b1024_flat")
# ... and the conv workloads once more with channels-last conv inputs (DP_NHWC: no layout
# copies), under "<name>/channels_last".
PER_CONFIG_CHANNELS_LAST = ("conv3x3_b256", "vgg11_cifar_b1024")
# FP32 FFMA peak for the fp32 one-row layer's FFMA kernels: 152 SMs x 128 FP32 lanes x
# 2 flop x 2.07 GHz.
FP32_FFMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def roofline(wl, work, means, pk, peak_kind="burst"):
    """Roofline object of the step's dominant call (largest per-call mean)."""
    dom = max(("norms", "factors", "sums", "noise"), key=means.get)   # sums_noised: the step's fused form
    if not means[dom] > 0:   # the per-call timing gave nothing (e.g. under a profiler): no figure
        return dict(bound=None, achieved=None, peak=None, unit=None, frac=None, traffic=None, kernel=None,
                    peak_source=None)
    tc_peak = pk["bf16"] if peak_kind == "burst" else pk["bf16_sus"]
    sum_bytes = work["kept_bytes"] + 4 * work["n_params"]     # kept gradients read, sums written
    if dom in ("sums", "norms") and wl.dtype == "fp32":
        flop = work["flop_sum"] if dom == "sums" else work["flop_norm"]
        roof = dict(bound="alu", achieved=flop / (means[dom] * 1e-3) / 1e12, peak=FP32_FFMA_TFLOPS,
                    unit="TFLOP/s")
    elif dom == "sums" and sum_bytes / (pk["hbm"] * 1e9) > work["flop_sum"] / (tc_peak * 1e12):
        # mostly kept per-example gradients: a read-bound weighted sum
        roof = dict(bound="hbm", achieved=sum_bytes / (means["sums"] * 1e-3) / 1e9, peak=pk["hbm"], unit="GB/s")
    elif dom == "sums":
        roof = dict(bound="tensor", achieved=work["flop_sum"] / (means["sums"] * 1e-3) / 1e12,
                    peak=tc_peak, unit="TFLOP/s")
    elif dom == "norms":
        roof = dict(bound="tensor", achieved=work["flop_norm"] / (means["norms"] * 1e-3) / 1e12,
                    peak=tc_peak, unit="TFLOP/s")
    else:
        nb = 8 * work["n_params"]
        roof = dict(bound="hbm", achieved=nb / (means[dom] * 1e-3) / 1e9, peak=pk["hbm"], unit="GB/s")
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = _profiled_traffic(wl.name, dom, _DOMINANT_KERNELS[dom], wl.B)
    roof["kernel"] = {"sums": "dp_clipped_sum", "norms": "dp_layer_sqnorms", "noise": "dp_add_noise",
                      "factors": "dp_clip_factors"}[dom]
    roof["peak_source"] = (f"{pk['src']} ({peak_kind})" if roof["bound"] == "tensor" else
                           pk["src"] if roof["bound"] == "hbm" else "derived: 152 SMs x 128 lanes x 2 x 2.07 GHz")
    return roof


class StepBench:
    """One workload's step on the device: inputs, the captured step graph, per-call graphs."""

    REPS = 20

    def __init__(self, dp, wl, dev, channels_last=False, host_inputs=False):
        import torch
        import workloads
        self.wl, self.dev = wl, dev
        cl = [bool(channels_last) and s.kind != "linear" for s in wl.layers]
        self.cl = cl
        self.descs = [layer_desc(dp, s, wl.B, wl.dtype, layout=int(c)) for s, c in zip(wl.layers, cl)]

        def to_layout(pair, c):
            return tuple(x.movedim(1, -1).contiguous() for x in pair) if c else pair

        n_elem = wl.B * sum(math.prod(s.a_example_shape()) + math.prod(s.g_example_shape()) for s in wl.layers)
        self.host_in = None
        if host_inputs and n_elem <= HOST_GEN_LIMIT:
            self.host_in = [workloads.layer_inputs(wl, l, threads=8) for l in range(len(wl.layers))]
            self.dev_in = [to_layout((workloads.to_torch(A, wl.dtype, str(dev)),
                                      workloads.to_torch(G, wl.dtype, str(dev))), c)
                           for (A, G), c in zip(self.host_in, cl)]
        else:
            # full-size inputs drawn on the device (host generation would take minutes)
            self.dev_in = [to_layout(workloads.device_layer_inputs(wl, l, str(dev)), c) for l, c in enumerate(cl)]
        adaptive = None
        if wl.per_layer and wl.alpha is not None:
            # C_l2 of the first step: the mean unclipped per-layer norm of a batch of random
            # noise ([ThreeTools] section 3), which the synthetic batch is
            probe = dp.ClipStep(self.descs, C=wl.C, sigma=wl.sigma, per_layer=True, device=str(dev))
            probe.norms(self.dev_in)
            c_l2 = probe.sqnorms.double().sqrt().mean(dim=1).tolist()
            del probe
            adaptive = dict(alpha=wl.alpha, beta=wl.beta, sigma_l2=wl.sigma_l2, C_l2=c_l2)
        self.step = dp.ClipStep(self.descs, C=wl.C, sigma=wl.sigma, per_layer=wl.per_layer, device=str(dev),
                                adaptive=adaptive)
        step = self.step
        self.modes = [dp.MODE_NAMES[m] for m, _, _ in step.plan]
        self.kept = [k is not None for k in step.kept]
        self.work = step_work(wl, self.modes, self.kept)
        # The whole step is one CUDA graph (norms -> [adaptive bound] -> factors -> clipped
        # sums -> noise), replayed once per step; every kernel in it is a library kernel.
        step.capture(self.dev_in)
        # per-call graphs for the per-kernel roofline: each holds REPS calls, so graph launch
        # latency is amortised (the first call finds a flushed L2; in the step the clipped sum
        # likewise runs right after the norm pass read the inputs).  Each call is followed by
        # a one-element PyTorch kernel, which takes no part in programmatic launch, so no call
        # overlaps the next; a graph of REPS such separators is timed too and subtracted.
        self.sep_buf = torch.zeros(1, dtype=torch.float32, device=dev)
        self.call_graphs = {}
        dev_in = self.dev_in
        for name, fn in (("norms", lambda: step.norms(dev_in)), ("factors", lambda: step.factors_()),
                         ("sums", lambda: step.sums(dev_in)), ("noise", lambda: step.noise_devseed()),
                         ("sums_noised", lambda: step.sums_and_noise_devseed(dev_in)), ("_sep", None)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(self.REPS):
                    if fn is not None:
                        fn()
                    self.sep_buf.add_(1.0)
            self.call_graphs[name] = g

    def timed(self, replay, k_steps, seed_base, flush, stream):
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k_steps)]
        for k in range(k_steps):
            flush.zero_()                              # L2 flush, outside the events
            self.step.seed_buf.fill_(seed_base + k)    # fresh noise seed, outside the events
            evs[k][0].record(stream)
            replay()
            evs[k][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def per_call_means(self, n_rep, seed0, flush, stream):
        sep_ms = statistics.mean(self.timed(self.call_graphs["_sep"].replay, n_rep, seed0, flush, stream))
        per_call = {n: [max(t - sep_ms, 0.0) / self.REPS for t in self.timed(g.replay, n_rep, seed0, flush, stream)]
                    for n, g in self.call_graphs.items() if n != "_sep"}
        return {n: statistics.mean(v) for n, v in per_call.items()}

    def free(self):
        import torch
        self.call_graphs = {}
        self.step = None
        self.dev_in = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def run_ours(args, wl):
    import torch
    import example_gradient_clipping_gb300 as dp
    world, rank, local = _dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    pk = _peaks()

    sb = StepBench(dp, wl, dev, channels_last=args.channels_last, host_inputs=True)
    step = sb.step
    W = max(args.warmup, 3)
    seed0 = wl.seed + 1_000_003 * (rank + 1)
    sb.timed(step.graph.replay, W, seed0, flush, stream)      # warm-up
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        step_ms = sb.timed(step.graph.replay, args.steps, seed0, flush, stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    launches = step.graph_kernels * args.steps
    total_ms = max_over_ranks(sum(step_ms), dev)
    value = world * wl.B * args.steps / (total_ms / 1e3)
    means = sb.per_call_means(max(5, min(args.steps // 4, 12)), seed0, flush, stream)
    clocks = clk.summary()
    # the tensor-core peak for the dominant call: the sustained figure (a seconds-long GEMM
    # loop under the power cap) when its timing graph keeps the tensor cores busy for a long
    # stretch (REPS back-to-back calls of 50 ms or more in all), else the burst figure;
    # the fraction of the other beside it
    dom = max(("norms", "factors", "sums", "noise"), key=means.get)
    long_run = StepBench.REPS * means[dom] >= 50.0
    roof = roofline(wl, sb.work, means, pk, "sustained" if long_run else "burst")
    if roof["bound"] == "tensor":
        other = pk["bf16"] if long_run else pk["bf16_sus"]
        roof["frac_of_burst" if long_run else "frac_of_sustained"] = roof["achieved"] / other
    roof["timing"] = (f"CUDA events around a graph of {StepBench.REPS} calls after an L2 flush, each call followed "
                      "by a one-element PyTorch kernel (no overlap between calls; the separators' own graph time "
                      "subtracted); per-call mean")

    # end to end through the public API: every step copies a batch from pinned host memory
    # and its gradient back (ClipPipeline: one graph per step, the copy of batch k+1 on a
    # forked stream alongside the compute of batch k); events around K graph launches
    shapes = [(tuple(a.shape), tuple(g.shape)) for a, g in sb.dev_in]
    pipe = dp.ClipPipeline(sb.descs, shapes, wl.dtype, C=wl.C, sigma=wl.sigma, per_layer=wl.per_layer,
                           device=str(dev))
    for hset in (pipe.host_inputs(0), pipe.host_inputs(1)):     # the same batch every step
        for (ha, hg), (da, dg) in zip(hset, sb.dev_in):
            ha.copy_(da)
            hg.copy_(dg)
    h2d = sum(a.numel() * a.element_size() + g.numel() * g.element_size() for a, g in pipe.host_inputs(0))
    d2h = pipe.n_params * 4
    host_in, cl = sb.host_in, sb.cl
    hin0 = pipe.host_inputs(0)

    def sample_inputs(b):
        if host_in is not None:
            return [(A[:b], G[:b]) for A, G in host_in]
        return [tuple((x[:b].movedim(-1, 1) if c else x[:b]).float().numpy() for x in pair)   # channels first
                for pair, c in zip(hin0, cl)]

    sb.free()
    pipe.start()
    for k in range(W):
        pipe.step(k, wl.seed + 7 * k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(W, W + args.steps):
        pipe.step(k, wl.seed + 7 * k)
    e1.record(stream)
    e1.synchronize()
    e2e_tot = max_over_ranks(e0.elapsed_time(e1), dev)
    e2e_value = world * wl.B * args.steps / (e2e_tot / 1e3)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, sample_inputs)
    del pipe
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # the other workloads of the metric, device step time only
    per_config = {}
    if not args.no_per_config and wl.name == DEFAULT_WORKLOAD:
        k_steps = max(3, min(args.steps, 20))
        runs = [(n, False) for n in PER_CONFIG] + [(n, True) for n in PER_CONFIG_CHANNELS_LAST]
        for name, cl2 in runs:
            import workloads
            w2 = workloads.get_workload(name)
            b2 = StepBench(dp, w2, dev, channels_last=cl2)
            b2.timed(b2.step.graph.replay, W, seed0, flush, stream)
            ms = b2.timed(b2.step.graph.replay, k_steps, seed0, flush, stream)
            m2 = b2.per_call_means(5, seed0, flush, stream)
            r2 = roofline(w2, b2.work, m2, pk, "burst")
            tot = max_over_ranks(sum(ms), dev)
            per_config[name + ("/channels_last" if cl2 else "")] = dict(
                value=world * w2.B * k_steps / (tot / 1e3), unit="examples/s", ms_per_step=tot / k_steps,
                steps=k_steps, dtype=w2.dtype, norm_modes=b2.modes, kernels_per_step=b2.step.graph_kernels,
                step_flop=b2.work["flop_norm"] + b2.work["flop_sum"], step_bytes=b2.work["bytes_total"],
                calls_ms={n: round(v, 5) for n, v in m2.items()},
                roofline={k: r2[k] for k in ("bound", "kernel", "achieved", "peak", "unit", "frac", "traffic")},
                conv_layout="channels last" if cl2 else "channels first", description=w2.description)
            b2.free()
            del b2

    line = None
    if rank == 0:
        line = dict(metric=METRIC, value=value, unit="examples/s", n_gpus=world, steps=args.steps,
                    warmup=W, ms_per_step=total_ms / args.steps, higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype=wl.dtype, data="synthetic",
                    config=_config(wl),
                    e2e=dict(value=e2e_value, unit="examples/s", h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                             pipeline="ClipPipeline: one CUDA graph per step runs the step on one of two "
                                      "device buffer sets, copies its gradient to pinned host memory and, on a "
                                      "forked stream, copies the next batch from pinned host memory into the other "
                                      "set"),
                    gpu_launches=int(launches), roofline=roof, clocks=clocks,
                    calls_ms={n: round(v, 5) for n, v in means.items()},
                    kernels_per_step=step.graph_kernels, norm_modes=sb.modes,
                    parallelism=f"replicas x{world}",
                    conv_layout="channels last" if any(cl) else "channels first",
                    step_flop=sb.work["flop_norm"] + sb.work["flop_sum"], step_bytes=sb.work["bytes_total"])
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if per_config:
            line["per_config"] = per_config
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_hbm_sweep(args):
    """Supplementary steady-state bandwidth of the HBM-bound kernels on large inputs (not
    the bench line): the noise/scale pass over a >= 256 MB parameter vector and the one-row
    norm over a >= 512 MB batch, each timed with CUDA events over back-to-back calls after
    an L2 flush.  Bytes are algorithmic: noise reads and writes each fp32 element once;
    the one-row norm reads A and G once."""
    import torch
    import example_gradient_clipping_gb300 as dp
    pk = _peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    out = []

    def timed(fn, reps=10):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(ts)

    for n in (64 << 20, 256 << 20):                     # 256 MB and 1 GB of fp32
        g = torch.randn(n, device="cuda")
        sec = timed(lambda: dp.dp_add_noise(g, 1.0, 1.0, 64, 7, 0))
        gbs = 8 * n / sec / 1e9
        out.append(dict(kernel="add_noise_kernel", elements=n, bytes=8 * n, us=sec * 1e6, gbs=gbs,
                        frac=gbs / pk["hbm"]))
        del g
    for B, d, p in ((262144, 512, 512), (65536, 4096, 4096)):   # 512 MB and 2 GB of bf16 rows
        A = torch.randn(B, d, device="cuda").to(torch.bfloat16)
        G = torch.randn(B, p, device="cuda").to(torch.bfloat16)
        desc = dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=B, p=p, T=1, d=d, has_bias=True)
        sq = torch.empty(B, device="cuda")
        ws = torch.empty(16, dtype=torch.uint8, device="cuda")
        sec = timed(lambda: dp.dp_layer_sqnorms(desc, A, G, sq, ws, mode=dp.DP_NORM_T1))
        nb = 2 * B * (d + p)
        gbs = nb / sec / 1e9
        out.append(dict(kernel="t1_norm_kernel", B=B, d=d, p=p, bytes=nb, us=sec * 1e6, gbs=gbs,
                        frac=gbs / pk["hbm"]))
        del A, G
    print(json.dumps(dict(supplementary="hbm_sweep", peak_gbs=pk["hbm"], peak_source=pk["src"], results=out)),
          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the smaller workloads' device timings after the headline workload")
    ap.add_argument("--hbm-sweep", action="store_true",
                    help="supplementary steady-state bandwidth of the noise and one-row norm kernels")
    ap.add_argument("--channels-last", action="store_true",
                    help="hand conv layers' A and G over channels last (DP_NHWC); same values")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (profiling and sweeps; not the bench line)")
    args = ap.parse_args()
    import workloads
    wl = workloads.get_workload(args.workload)
    if args.batch:
        wl = wl.with_batch(args.batch)
    if args.hbm_sweep:
        run_hbm_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
