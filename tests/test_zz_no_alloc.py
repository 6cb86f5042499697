"""dp_layer_sqnorms_noalloc: the per-example norm entry point for callers that cannot
allocate device memory (for instance code inside another framework's hook that
has no handle on that framework's allocator, or a loop that cannot afford the
device-wide synchronization of cudaMalloc/cudaFree).  It keeps its partial sums in
a library-owned static array instead of a caller workspace.

Checked through the C ABI against dp_layer_sqnorms (the workspace entry point),
within the tolerances the other parity tests use, on two calls in a row (the
second call reuses the array the first one left behind).  This file sorts last so
that a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

import workloads
from helpers import TOL, desc_for, rel_elem, to_dev
from workloads import LayerSpec, Workload

pytestmark = pytest.mark.gpu

CASES = [
    ("seq_linear_b64_t128", 0, None),            # ghost norm, full batch
    ("conv3x3_b256", 0, 32),                     # instantiation, 32 examples
    ("vgg11_cifar_b1024", 1, 16),                # instantiation (conv2)
    ("vgg11_cifar_b1024", 4, 16),                # ghost (conv5, T=16)
    ("vgg11_cifar_b1024", 8, 64),                # one-row fc layer
    ("vit_mlp_b4096_t197", 0, 8),                # ghost with a ragged 197-row tile
]


@pytest.mark.parametrize("name,layer,B", CASES, ids=[f"{c[0]}-{c[1]}" for c in CASES])
def test_noalloc_matches_workspace_entry_point(lib, name, layer, B):
    import torch
    dp = lib
    wl = workloads.get_workload(name)
    if B is not None:
        wl = wl.with_batch(B)
    spec = wl.layers[layer]
    A, G = workloads.layer_inputs(wl, layer)
    desc = desc_for(dp, spec, wl.B, wl.dtype)
    Ad, Gd = to_dev(A, wl.dtype), to_dev(G, wl.dtype)
    ws = torch.empty(max(dp.dp_workspace_size(desc), 16), dtype=torch.uint8, device="cuda")
    ref = torch.empty(wl.B, dtype=torch.float32, device="cuda")
    mode_ref = dp.dp_layer_sqnorms(desc, Ad, Gd, ref, ws)
    ref_np = ref.cpu().numpy()
    for call in range(2):
        out = torch.full((wl.B,), float("nan"), dtype=torch.float32, device="cuda")
        mode = dp.dp_layer_sqnorms_noalloc(desc, Ad, Gd, out)
        torch.cuda.synchronize()
        assert mode == mode_ref
        assert rel_elem(out.cpu().numpy(), ref_np) <= TOL[wl.dtype], f"call {call}"


def test_noalloc_rejects_layers_beyond_its_scratch(lib):
    import torch
    dp = lib
    # ghost partials for B=1024, T=1024: 2 * 1024 * 528 floats, above the 4 MiB array
    desc = dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=1024, p=8, T=1024, d=8)
    A = torch.zeros(1024 * 1024 * 8, dtype=torch.bfloat16, device="cuda")
    G = torch.zeros_like(A)
    out = torch.zeros(1024, dtype=torch.float32, device="cuda")
    with pytest.raises(dp.DPError) as e:
        dp.dp_layer_sqnorms_noalloc(desc, A, G, out, mode=dp.DP_NORM_GHOST)
    assert e.value.status == dp.DP_ERR_UNSUPPORTED and "static maximum" in str(e.value)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
