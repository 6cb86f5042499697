"""Data-parallel sharding of one clipping step, on two CPU ranks over gloo.

The step shards by example: every per-example norm and clip factor is local to
the rank that holds the example (flat clipping needs all of an example's layers
on one rank, which a split of the batch keeps), each rank forms the partial
clipped sum over its examples, one SUM all-reduce adds the partials, and the
Gaussian noise and the 1/B scale of the global batch are applied once to the
reduced sum ([FastClip] section 2: the sum over the batch, then the noise).  The
adaptive bound needs one all-reduce of sum_i min(||g_i||, C_l2) per layer
([ThreeTools] section 3).  These tests run that algebra with the oracle on a
ragged split (3 + 2 examples) and check it against the single-process step;
they also check the slowest-rank reduction that bench.py applies to replica
timings.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import dpsgd
from workloads import LayerSpec, Workload, layer_inputs

WORLD = 2


def _workload(per_layer: bool) -> Workload:
    layers = (
        LayerSpec(name="seq", kind="linear", p=6, d=5, T=4, has_bias=True),
        LayerSpec(name="conv", kind="conv2d", p=4, Cin=3, H=6, W=5, k=3, stride=1, pad=1, has_bias=True),
        LayerSpec(name="head", kind="linear", p=3, d=7, T=1, has_bias=False),
    )
    return Workload(name="shard_test", B=5, layers=layers, dtype="fp32", C=0.5, sigma=0.9,
                    per_layer=per_layer, seed=11, alpha=1.1, beta=2.0, sigma_l2=2.5,
                    g_scale="mixed")


def _shard(B: int, rank: int, world: int):
    """Contiguous, ragged split of the batch: the first B % world ranks take one more."""
    q, r = divmod(B, world)
    lo = rank * q + min(rank, r)
    return list(range(lo, lo + q + (1 if rank < r else 0)))


def _allreduce_sum(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return t.numpy()


def _sharded_step(wl: Workload, rank: int):
    mine = _shard(wl.B, rank, WORLD)
    L = len(wl.layers)
    inputs = [layer_inputs(wl, l, mine) for l in range(L)]
    sq = np.stack([dpsgd.layer_sqnorms(spec, *inputs[l]) for l, spec in enumerate(wl.layers)])
    C = [wl.C] * L
    fac, _ = dpsgd.clip_factors(sq, C if wl.per_layer else C[0], wl.per_layer)
    partial = []
    for l, spec in enumerate(wl.layers):
        f = fac[l] if wl.per_layer else fac
        S, Sb = dpsgd.clipped_sum(spec, *inputs[l], f)
        partial.append(S.reshape(-1) if Sb is None else np.concatenate([S.reshape(-1), Sb]))
    total = _allreduce_sum(np.concatenate(partial))
    # noise once on the reduced sum, 1/B of the global batch, layer by layer
    noisy, offs = [], wl.param_offsets()
    for l, spec in enumerate(wl.layers):
        seg = total[offs[l]:offs[l] + spec.n_params]
        noisy.append(dpsgd.add_noise(seg, wl.sigma, C[l], wl.B, wl.seed, offs[l]))
    # adaptive bound: per-layer partial of sum_i min(n_i, C_l2), one all-reduce
    C_l2 = 0.3
    clipped = np.array([np.minimum(np.sqrt(sq[l]), C_l2).sum() for l in range(L)])
    clipped = _allreduce_sum(clipped)
    return dict(total=total, noisy=np.concatenate(noisy), clipped=clipped, C_l2=C_l2)


def _worker(rank: int, port: int, per_layer: bool, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        wl = _workload(per_layer)
        res = _sharded_step(wl, rank)
        import bench
        slowest = bench.max_over_ranks(1.5 + rank, torch.device("cpu"))
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), slowest=slowest, **res)
    finally:
        dist.destroy_process_group()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(per_layer: bool, tmp_path):
    mp.spawn(_worker, args=(_free_port(), per_layer, str(tmp_path)), nprocs=WORLD, join=True)
    return [dict(np.load(tmp_path / f"rank{r}.npz")) for r in range(WORLD)]


def test_shard_split_covers_batch():
    for B in (1, 2, 5, 64, 4097):
        parts = [_shard(B, r, WORLD) for r in range(WORLD)]
        assert sum(parts, []) == list(range(B))
        assert max(map(len, parts)) - min(map(len, parts)) <= 1


@pytest.mark.parametrize("per_layer", [False, True], ids=["flat", "per_layer"])
def test_sharded_step_equals_single_process(per_layer, tmp_path):
    wl = _workload(per_layer)
    ranks = _run(per_layer, tmp_path)
    L = len(wl.layers)
    full_in = [layer_inputs(wl, l) for l in range(L)]
    ref = dpsgd.dp_step(wl, full_in)
    ref_sum = np.concatenate([S.reshape(-1) if Sb is None else np.concatenate([S.reshape(-1), Sb])
                              for S, Sb in ref["sums"]])
    # the split must clip something and leave something unclipped, or it tests little
    f = np.asarray(ref["factors"])
    assert (f < 1).any() and (f == 1).any()
    for r in ranks:
        np.testing.assert_allclose(r["total"], ref_sum, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(r["noisy"], ref["noisy"], rtol=1e-12, atol=1e-15)
    # every rank holds the same privatised gradient (the noise is drawn once, from one seed)
    np.testing.assert_array_equal(ranks[0]["noisy"], ranks[1]["noisy"])
    # adaptive bound from the reduced partials equals the oracle's on the full batch
    for l in range(L):
        n_full = np.asarray(ref["sqnorms"][l])
        want = dpsgd.adaptive_bound(n_full, ranks[0]["C_l2"], wl.alpha, wl.beta, wl.sigma_l2, wl.seed, l)
        z = dpsgd.normal_noise(1, wl.seed, offset=l, stream=1)[0]
        got = wl.alpha / wl.B * (ranks[0]["clipped"][l] + wl.sigma_l2 * ranks[0]["C_l2"] * z)
        assert got == pytest.approx(want[0], rel=1e-12)
        assert wl.beta * got == pytest.approx(want[1], rel=1e-12)


def test_replica_timing_takes_slowest_rank(tmp_path):
    ranks = _run(False, tmp_path)
    assert [float(r["slowest"]) for r in ranks] == [2.5, 2.5]
