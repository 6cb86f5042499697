"""dp_layer_sqnorms_noalloc: the per-example norm entry point for callers that cannot
allocate device memory (for instance code inside another framework's hook that
has no handle on that framework's allocator, or a loop that cannot afford the
device-wide synchronization of cudaMalloc/cudaFree).  It keeps its partial sums in
a library-owned static array instead of a caller workspace.

Checked through the C ABI against the oracle and against dp_layer_sqnorms (the
workspace entry point), within the tolerances the other parity tests use, on two
calls in a row.  Between the two, calls on larger layers whose inputs are NaN fill
the shared array with NaN partials, so the second call passes only if it writes every
partial it reads.  This file sorts last so that a run stopping at the first failure
has already run every other test.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import TOL, desc_for, rel_elem, to_dev, to_dev_channels_last
from workloads import LayerSpec, Workload

pytestmark = pytest.mark.gpu

CASES = [
    ("seq_linear_b64_t128", 0, None, False),           # ghost norm, full batch
    ("conv3x3_b256", 0, 32, False),                    # instantiation, 32 examples
    ("conv3x3_b256", 0, 16, True),                     # instantiation, channels last
    ("vgg11_cifar_b1024", 1, 16, False),               # instantiation (conv2)
    ("vgg11_cifar_b1024", 4, 16, False),               # ghost (conv5, T=16)
    ("vgg11_cifar_b1024", 4, 8, True),                 # ghost, channels last
    ("vgg11_cifar_b1024", 8, 64, False),               # one-row fc layer
    ("vit_mlp_b4096_t197", 0, 8, False),               # ghost with a ragged 197-row tile
    ("fp32_linear", 0, 5, False),                      # fp32 inputs, ghost
    ("fp32_conv", 0, 4, False),                        # fp32 inputs, instantiation
]

_FP32 = {
    "fp32_linear": Workload(name="fp32_linear", B=5, dtype="fp32", C=1.0, sigma=1.0, seed=41,
                            layers=(LayerSpec("l", "linear", p=40, d=72, T=33),)),
    "fp32_conv": Workload(name="fp32_conv", B=4, dtype="fp32", C=1.0, sigma=1.0, seed=42,
                          layers=(LayerSpec("c", "conv2d", p=12, Cin=6, H=9, W=9, k=3, pad=1),)),
}


def _fill_scratch_with_nan(dp):
    """Calls on larger layers (ghost and instantiation) whose inputs are all NaN: they
    leave NaN partials across much of the shared array."""
    import torch
    for mode, desc in ((dp.DP_NORM_GHOST, dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=512, p=16, T=512, d=16)),
                       (dp.DP_NORM_INSTANTIATE, dp.layer_desc(dp.DP_LINEAR, dp.DP_BF16, B=64, p=1024, T=4,
                                                              d=1024))):
        n = desc.B * desc.T * max(desc.d, desc.p)
        X = torch.full((n,), float("nan"), dtype=torch.bfloat16, device="cuda")
        out = torch.empty(desc.B, dtype=torch.float32, device="cuda")
        dp.dp_layer_sqnorms_noalloc(desc, X, X, out, mode=mode)
        torch.cuda.synchronize()
        assert bool(torch.isnan(out).all())


@pytest.mark.parametrize("name,layer,B,cl", CASES,
                         ids=[f"{c[0]}-{c[1]}" + ("-channels_last" if c[3] else "") for c in CASES])
def test_noalloc_matches_oracle_and_workspace_entry_point(lib, name, layer, B, cl):
    import torch
    dp = lib
    wl = _FP32[name] if name in _FP32 else workloads.get_workload(name)
    if B is not None:
        wl = wl.with_batch(B)
    spec = wl.layers[layer]
    A, G = workloads.layer_inputs(wl, layer)
    s_ref = oracle.layer_sqnorms(spec, A, G)
    lay = dp.DP_NHWC if cl else dp.DP_NCHW
    desc = desc_for(dp, spec, wl.B, wl.dtype, layout=lay)
    put = (lambda x: to_dev_channels_last(x, wl.dtype)) if cl else (lambda x: to_dev(x, wl.dtype))
    Ad, Gd = put(A), put(G)
    ws = torch.empty(max(dp.dp_workspace_size(desc), 16), dtype=torch.uint8, device="cuda")
    ref = torch.empty(wl.B, dtype=torch.float32, device="cuda")
    mode_ref = dp.dp_layer_sqnorms(desc, Ad, Gd, ref, ws)
    ref_np = ref.cpu().numpy()
    tol = TOL[wl.dtype]
    assert rel_elem(ref_np, s_ref) <= tol
    for call in range(2):
        if call == 1:
            _fill_scratch_with_nan(dp)
        out = torch.full((wl.B,), float("nan"), dtype=torch.float32, device="cuda")
        mode = dp.dp_layer_sqnorms_noalloc(desc, Ad, Gd, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert mode == mode_ref
        assert rel_elem(got, s_ref) <= tol, f"call {call}: against the oracle"
        assert rel_elem(got, ref_np) <= tol, f"call {call}: against dp_layer_sqnorms"


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
