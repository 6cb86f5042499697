"""PrivacyEngine: A and G captured by autograd hooks, the step through the C ABI.

CPU: which models are accepted.  GPU: the privatised gradient equals the naive per-example
loop of the pages (batch size 1, autograd per example) clipped and noised by the oracle.
"""
import numpy as np
import pytest
import torch
import torch.nn as nn

import oracle
from helpers import rel_flat

# PyTorch notes that a layer hook fires on output gradients when the model input needs no
# gradient (the first layer here); that is exactly the gradient the engine reads.
pytestmark = pytest.mark.filterwarnings("ignore:Full backward hook is firing")


def _model(dtype=torch.float32):
    torch.manual_seed(0)
    return nn.Sequential(nn.Conv2d(3, 8, 3, padding=1), nn.ReLU(), nn.Conv2d(8, 8, 3, stride=2, padding=1),
                         nn.ReLU(), nn.Flatten(), nn.Linear(8 * 3 * 3, 16), nn.ReLU(), nn.Linear(16, 5)).to(dtype)


def test_engine_accepts_linear_and_conv_only():
    import example_gradient_clipping_gb300 as lib      # host only: hooks, no kernels
    eng = lib.PrivacyEngine(_model())
    assert len(eng.layers) == 4
    eng.detach()
    with pytest.raises(ValueError):
        lib.PrivacyEngine(nn.Sequential(nn.Linear(4, 4), nn.LayerNorm(4)))
    with pytest.raises(ValueError):
        lib.PrivacyEngine(nn.Sequential(nn.Conv2d(4, 4, 3, groups=2)))
    with pytest.raises(ValueError):
        lib.PrivacyEngine(nn.Sequential(nn.Conv2d(4, 4, (3, 1))))
    with pytest.raises(ValueError):
        lib.PrivacyEngine(nn.Sequential(nn.Conv3d(4, 4, 3, stride=(1, 2, 1))))
    lib.PrivacyEngine(nn.Sequential(nn.Conv3d(4, 4, 3, padding=1))).detach()
    frozen = nn.Sequential(nn.Linear(4, 4), nn.LayerNorm(4))
    for q in frozen[1].parameters():
        q.requires_grad_(False)
    lib.PrivacyEngine(frozen).detach()


class _Block:
    """p, D and has_bias of one layer's block in the flat gradient."""

    def __init__(self, m):
        self.p = m.weight.shape[0]
        self.D = m.weight[0].numel()
        self.has_bias = m.bias is not None


def _rel(got, want, model):
    """Element-wise error of a flat gradient over the model's layers (helpers.rel_flat)."""
    layers = [m for m in model.modules() if isinstance(m, (nn.Linear, nn.Conv1d, nn.Conv2d, nn.Conv3d))]
    return rel_flat(got, want, [_Block(m) for m in layers])


def _naive_reference(model, x, y, C, sigma, seed):
    """The pages' naive method: one example at a time through autograd, then the oracle's
    clip, sum and noise over the flat parameter vector [W_0, b_0, W_1, b_1, ...]."""
    layers = [m for m in model.modules() if isinstance(m, (nn.Linear, nn.Conv1d, nn.Conv2d, nn.Conv3d))]
    B = x.shape[0]
    g = []
    for i in range(B):
        model.zero_grad()
        loss = nn.functional.cross_entropy(model(x[i:i + 1]).float(), y[i:i + 1], reduction="sum")
        loss.backward()
        g.append(np.concatenate([np.concatenate([m.weight.grad.double().cpu().numpy().ravel(),
                                                 m.bias.grad.double().cpu().numpy()]) for m in layers]))
    g = np.stack(g)
    n = np.sqrt((g * g).sum(1))
    c = np.minimum(1.0, C / n)
    return oracle.add_noise((c[:, None] * g).sum(0), sigma, C, B, seed)


@pytest.fixture
def no_tf32():
    """fp32 convolutions and matmuls in full fp32 (cuDNN's TF32 default would round them)."""
    saved = torch.backends.cudnn.allow_tf32, torch.backends.cuda.matmul.allow_tf32
    torch.backends.cudnn.allow_tf32 = torch.backends.cuda.matmul.allow_tf32 = False
    yield
    torch.backends.cudnn.allow_tf32, torch.backends.cuda.matmul.allow_tf32 = saved


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,tol", [(torch.float32, 1e-5), (torch.bfloat16, 2e-2)], ids=["fp32", "bf16"])
def test_engine_matches_naive_per_example_loop(lib, no_tf32, dtype, tol):
    model = _model(dtype).cuda()
    gen = torch.Generator().manual_seed(1)
    x = torch.randn(6, 3, 6, 6, generator=gen).to(dtype).cuda()
    y = torch.randint(0, 5, (6,), generator=gen).cuda()
    want = _naive_reference(model, x, y, C=0.5, sigma=0.3, seed=77)
    eng = lib.PrivacyEngine(model, C=0.5, sigma=0.3)
    model.zero_grad()
    nn.functional.cross_entropy(model(x).float(), y, reduction="sum").backward()
    flat = eng.privatise(seed=77)
    got = flat.double().cpu().numpy()
    assert _rel(got, want, model) <= tol
    layers = [m for m in model.modules() if isinstance(m, (nn.Linear, nn.Conv2d))]
    from_grads = np.concatenate([np.concatenate([m.weight.grad.double().cpu().numpy().ravel(),
                                                 m.bias.grad.double().cpu().numpy()]) for m in layers])
    if dtype == torch.float32:
        np.testing.assert_array_equal(from_grads, got)       # .grad holds the privatised gradient
    else:
        assert _rel(from_grads, got, model) <= 1e-2   # rounded to bf16
    eng.detach()


@pytest.mark.gpu
def test_engine_channels_last_model(lib):
    """A channels_last model: its conv layers are handed over channels last (no layout copy)
    and give the naive per-example loop's result."""
    model = _model(torch.bfloat16).cuda().to(memory_format=torch.channels_last)
    gen = torch.Generator().manual_seed(9)
    x = torch.randn(6, 3, 6, 6, generator=gen).to(torch.bfloat16).cuda().to(memory_format=torch.channels_last)
    y = torch.randint(0, 5, (6,), generator=gen).cuda()
    want = _naive_reference(model, x, y, C=0.5, sigma=0.3, seed=21)
    eng = lib.PrivacyEngine(model, C=0.5, sigma=0.3)
    model.zero_grad()
    nn.functional.cross_entropy(model(x).float(), y, reduction="sum").backward()
    got = eng.privatise(seed=21).double().cpu().numpy()
    convs = [m for m in eng.layers if isinstance(m, nn.Conv2d)]
    assert [d.layout for d, m in zip(eng._step.descs, eng.layers) if isinstance(m, nn.Conv2d)] == \
        [lib.DP_NHWC] * len(convs)
    eng.detach()
    assert _rel(got, want, model) <= 2e-2


@pytest.mark.gpu
def test_engine_conv1d_model(lib, no_tf32):
    torch.manual_seed(3)
    model = nn.Sequential(nn.Conv1d(4, 8, 3, padding=1), nn.ReLU(), nn.Conv1d(8, 8, 5, stride=2, padding=2),
                          nn.ReLU(), nn.Flatten(), nn.Linear(8 * 10, 5)).cuda()
    gen = torch.Generator().manual_seed(4)
    x = torch.randn(6, 4, 20, generator=gen).cuda()
    y = torch.randint(0, 5, (6,), generator=gen).cuda()
    want = _naive_reference(model, x, y, C=0.5, sigma=0.3, seed=8)
    eng = lib.PrivacyEngine(model, C=0.5, sigma=0.3)
    model.zero_grad()
    nn.functional.cross_entropy(model(x), y, reduction="sum").backward()
    got = eng.privatise(seed=8).double().cpu().numpy()
    eng.detach()
    assert _rel(got, want, model) <= 1e-5


@pytest.mark.gpu
def test_engine_conv3d_model(lib, no_tf32):
    torch.manual_seed(5)
    model = nn.Sequential(nn.Conv3d(2, 8, 3, padding=1), nn.ReLU(), nn.Conv3d(8, 8, 2, stride=2),
                          nn.ReLU(), nn.Flatten(), nn.Linear(8 * 2 * 3 * 2, 4)).cuda()
    gen = torch.Generator().manual_seed(6)
    x = torch.randn(5, 2, 4, 6, 5, generator=gen).cuda()
    y = torch.randint(0, 4, (5,), generator=gen).cuda()
    want = _naive_reference(model, x, y, C=0.5, sigma=0.3, seed=9)
    eng = lib.PrivacyEngine(model, C=0.5, sigma=0.3)
    model.zero_grad()
    nn.functional.cross_entropy(model(x), y, reduction="sum").backward()
    got = eng.privatise(seed=9).double().cpu().numpy()
    eng.detach()
    assert _rel(got, want, model) <= 1e-5


@pytest.mark.gpu
def test_engine_mean_loss_equals_sum_loss(lib, no_tf32):
    model = _model().cuda()
    gen = torch.Generator().manual_seed(2)
    x = torch.randn(5, 3, 6, 6, generator=gen).cuda()
    y = torch.randint(0, 5, (5,), generator=gen).cuda()
    outs = []
    for red in ("sum", "mean"):
        eng = lib.PrivacyEngine(model, C=0.5, sigma=0.3, loss_reduction=red)
        model.zero_grad()
        nn.functional.cross_entropy(model(x), y, reduction=red).backward()
        outs.append(eng.privatise(seed=5).double().cpu().numpy())
        eng.detach()
    assert _rel(outs[1], outs[0], model) <= 1e-5
