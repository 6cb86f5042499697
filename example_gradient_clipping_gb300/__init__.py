"""Python binding of libdpclip, DP-SGD per-example gradient clipping on GB300.

Argument marshalling only: every function calls the C entry point of the same
name (declared in include/dpclip.h) with raw device pointers and the current CUDA
stream.  Tensors may be torch tensors (their data_ptr() is passed) or integer
device addresses.  There is no fallback: importing this package fails if the
compiled library is missing, and every non-DP_OK status raises DPError.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdpclip.so")

DP_OK, DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED, DP_ERR_CUDA, DP_ERR_NONFINITE, DP_ERR_TIMEOUT = range(6)
DP_BF16, DP_FP32 = 0, 1
DP_LINEAR, DP_CONV2D, DP_CONV1D, DP_CONV3D = 0, 1, 2, 3
DP_NCHW, DP_NHWC = 0, 1
DP_NORM_AUTO, DP_NORM_GHOST, DP_NORM_INSTANTIATE, DP_NORM_T1, DP_NORM_AUTO_TIME = 0, 1, 2, 3, 4
MODE_NAMES = {DP_NORM_GHOST: "ghost", DP_NORM_INSTANTIATE: "instantiate", DP_NORM_T1: "t1"}


class DPError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dpclip status {status}: {message}")
        self.status = status


class NoiseDesc(ctypes.Structure):
    """dp_noise_desc: noise N(0, (sigma C)^2) and 1/B for a fused clipped sum."""
    _fields_ = [("sigma", ctypes.c_float), ("C", ctypes.c_float), ("B", ctypes.c_int),
                ("seed", ctypes.c_uint64), ("seed_dev", ctypes.c_void_p), ("offset", ctypes.c_uint64)]


class NoiseBlock(ctypes.Structure):
    """dp_noise_block: one block of the flat gradient with its bound."""
    _fields_ = [("offset", ctypes.c_uint64), ("n", ctypes.c_uint64), ("C", ctypes.c_float)]


class LayerDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("kind", "dtype", "B", "T", "d", "p", "Cin", "H", "W", "k", "stride", "pad", "dil",
                 "has_bias", "Z", "layout")]


def layer_desc(kind: int, dtype: int, B: int, p: int, T: int = 1, d: int = 0, Cin: int = 0,
               H: int = 0, W: int = 0, k: int = 1, stride: int = 1, pad: int = 0, dil: int = 1,
               has_bias: bool = True, Z: int = 0, layout: int = 0) -> LayerDesc:
    """layout: DP_NCHW (channels first, PyTorch's default) or DP_NHWC (channels last) for
    the A and G of conv layers."""
    return LayerDesc(kind, dtype, B, T, d, p, Cin, H, W, k, stride, pad, dil, int(bool(has_bias)), Z, layout)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built (run example_gradient_clipping_gb300.build.build())")
    lib = ctypes.CDLL(LIB_PATH)
    c_int, c_size, c_void, c_f, c_u64 = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float, ctypes.c_uint64
    PD = ctypes.POINTER(LayerDesc)
    PI = ctypes.POINTER(c_int)
    sig = {
        "dp_abi_version": (c_int, []),
        "dp_launch_count": (ctypes.c_ulonglong, []),
        "dp_last_error": (ctypes.c_char_p, []),
        "dp_plan": (c_int, [PD, c_int, PI, PI, PI]),
        "dp_workspace_size": (c_size, [PD, c_int]),
        "dp_layer_sqnorms": (c_int, [PD, c_void, c_void, c_int, c_void, PI, c_void, c_size, c_void]),
        "dp_layer_sqnorms_noalloc": (c_int, [PD, c_void, c_void, c_int, c_void, PI, c_void]),
        "dp_clip_factors": (c_int, [c_void, c_int, c_int, c_int, ctypes.POINTER(c_f), c_void, c_void]),
        "dp_clipped_sum": (c_int, [PD, c_void, c_void, c_void, c_void, c_void, c_int, c_void, c_size, c_void]),
        "dp_add_noise": (c_int, [c_void, c_size, c_f, c_f, c_int, c_u64, c_u64, c_void]),
        "dp_add_noise_devseed": (c_int, [c_void, c_size, c_f, c_f, c_int, c_void, c_u64, c_void]),
        "dp_adaptive_bound": (c_int, [c_void, c_int, c_f, c_f, c_f, c_f, c_u64, c_int, c_void, c_void]),
        "dp_adaptive_bounds": (c_int, [c_void, c_int, c_int, c_int, ctypes.POINTER(c_f), c_f, c_f, c_f, c_u64,
                                       c_void, c_void, c_void]),
        "dp_check_status": (c_int, [c_void]),
        "dp_selftest_wait_timeout": (c_int, [c_void, c_void]),
        "dp_grads_size": (c_size, [PD]),
        "dp_clipped_sum_reuse": (c_int, [PD, c_int, c_void, c_void, c_void, c_void, c_void, c_int, c_void, c_size,
                                         c_void]),
        "dp_layout_reused": (c_int, [PD, c_int]),
        "dp_layer_sqnorms_keep": (c_int, [PD, c_void, c_void, c_void, c_void, c_void, c_size, c_void]),
        "dp_clipped_sum_kept": (c_int, [PD, c_void, c_void, c_void, c_void, c_int, c_void, c_size, c_void]),
        "dp_clipped_sum_noised": (c_int, [PD, c_int, c_void, c_void, c_void, c_void, c_void, c_int,
                                          ctypes.POINTER(NoiseDesc), c_void, c_size, c_void]),
        "dp_clipped_sum_kept_noised": (c_int, [PD, c_void, c_void, c_void, c_void, c_int, ctypes.POINTER(NoiseDesc),
                                               c_void, c_size, c_void]),
        "dp_add_noise_blocks": (c_int, [c_void, ctypes.POINTER(NoiseBlock), c_int, c_f, c_int, c_u64, c_void,
                                        c_void]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


_lib = _load()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _check(status: int) -> None:
    if status != DP_OK:
        raise DPError(status, _lib.dp_last_error().decode())


def dp_abi_version() -> int:
    return _lib.dp_abi_version()


def dp_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return _lib.dp_launch_count()


def dp_plan(desc: LayerDesc, requested: int = DP_NORM_AUTO):
    """(chosen_mode, T, D) for a layer (host only)."""
    m, T, D = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(_lib.dp_plan(ctypes.byref(desc), requested, ctypes.byref(m), ctypes.byref(T), ctypes.byref(D)))
    return m.value, T.value, D.value


def dp_workspace_size(desc: LayerDesc, mode: int = DP_NORM_AUTO) -> int:
    return _lib.dp_workspace_size(ctypes.byref(desc), mode)


def dp_layer_sqnorms(desc: LayerDesc, A, G, sqnorm_out, workspace=None, ws_bytes: Optional[int] = None,
                     mode: int = DP_NORM_AUTO, stream=None) -> int:
    chosen = ctypes.c_int(-1)
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None and not isinstance(workspace, int) else 0
    _check(_lib.dp_layer_sqnorms(ctypes.byref(desc), _ptr(A), _ptr(G), mode, _ptr(sqnorm_out),
                                 ctypes.byref(chosen), _ptr(workspace), ws_bytes, _stream(stream)))
    return chosen.value


def dp_layer_sqnorms_noalloc(desc: LayerDesc, A, G, sqnorm_out, mode: int = DP_NORM_AUTO,
                             stream=None) -> int:
    """dp_layer_sqnorms for callers that cannot allocate: the scratch is library-owned."""
    chosen = ctypes.c_int(-1)
    _check(_lib.dp_layer_sqnorms_noalloc(ctypes.byref(desc), _ptr(A), _ptr(G), mode, _ptr(sqnorm_out),
                                         ctypes.byref(chosen), _stream(stream)))
    return chosen.value


def dp_clip_factors(sqnorms, B: int, L: int, per_layer: bool, C: Sequence[float], factors_out,
                    stream=None) -> None:
    Cs = list(C) if isinstance(C, (list, tuple)) else [float(C)]
    arr = (ctypes.c_float * len(Cs))(*Cs)
    _check(_lib.dp_clip_factors(_ptr(sqnorms), B, L, int(bool(per_layer)), arr, _ptr(factors_out),
                                _stream(stream)))


def dp_clipped_sum(desc: LayerDesc, A, G, factors, dW, db=None, workspace=None,
                   ws_bytes: Optional[int] = None, accumulate: bool = False, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None and not isinstance(workspace, int) else 0
    _check(_lib.dp_clipped_sum(ctypes.byref(desc), _ptr(A), _ptr(G), _ptr(factors), _ptr(dW), _ptr(db),
                               int(bool(accumulate)), _ptr(workspace), ws_bytes, _stream(stream)))


def dp_add_noise(grad, sigma: float, C: float, B: int, seed: int, offset: int = 0,
                 n: Optional[int] = None, stream=None) -> None:
    if n is None:
        n = grad.numel()
    _check(_lib.dp_add_noise(_ptr(grad), n, sigma, C, B, seed, offset, _stream(stream)))


def dp_add_noise_devseed(grad, sigma: float, C: float, B: int, seed_dev, offset: int = 0,
                         n: Optional[int] = None, stream=None) -> None:
    """dp_add_noise reading the 64-bit seed from device memory (for CUDA-graph replays)."""
    if n is None:
        n = grad.numel()
    _check(_lib.dp_add_noise_devseed(_ptr(grad), n, sigma, C, B, _ptr(seed_dev), offset, _stream(stream)))


def dp_adaptive_bound(sqnorms, B: int, C_l2: float, alpha: float, beta: float, sigma_l2: float,
                      seed: int, layer: int, out, stream=None) -> None:
    _check(_lib.dp_adaptive_bound(_ptr(sqnorms), B, C_l2, alpha, beta, sigma_l2, seed, layer, _ptr(out),
                                  _stream(stream)))


def dp_adaptive_bounds(sqnorms, B: int, C_l2: Sequence[float], alpha: float, beta: float, sigma_l2: float,
                       seed: int, out, layer0: int = 0, seed_dev=None, stream=None) -> None:
    """dp_adaptive_bound of layers layer0 .. layer0 + len(C_l2) - 1 in one launch: sqnorms
    [L, B], out [L, 2]; with seed_dev the seed is read from that device buffer."""
    Cs = [float(c) for c in C_l2]
    arr = (ctypes.c_float * max(1, len(Cs)))(*Cs)
    _check(_lib.dp_adaptive_bounds(_ptr(sqnorms), B, layer0, len(Cs), arr, alpha, beta, sigma_l2, seed,
                                   _ptr(seed_dev), _ptr(out), _stream(stream)))


def dp_clipped_sum_reuse(desc: LayerDesc, norm_mode: int, A, G, factors, dW, db=None, workspace=None,
                         ws_bytes: Optional[int] = None, accumulate: bool = False, stream=None) -> None:
    """dp_clipped_sum reading the layouts this layer's norm call left in `workspace`."""
    _check(_lib.dp_clipped_sum_reuse(ctypes.byref(desc), norm_mode, _ptr(A), _ptr(G), _ptr(factors), _ptr(dW),
                                     _ptr(db), int(bool(accumulate)), _ptr(workspace),
                                     _ws_len(workspace) if ws_bytes is None else ws_bytes, _stream(stream)))


def dp_layout_reused(desc: LayerDesc, norm_mode: int = DP_NORM_AUTO) -> int:
    return int(_lib.dp_layout_reused(ctypes.byref(desc), norm_mode))


def dp_grads_size(desc: LayerDesc) -> int:
    """Bytes of the kept per-example gradients of `desc` (0: the layer cannot keep them)."""
    return int(_lib.dp_grads_size(ctypes.byref(desc)))


def _ws_len(workspace) -> int:
    return workspace.numel() * workspace.element_size() if workspace is not None and not isinstance(workspace, int) else 0


def dp_layer_sqnorms_keep(desc: LayerDesc, A, G, sqnorm_out, grads, workspace=None, ws_bytes: Optional[int] = None,
                          stream=None) -> None:
    _check(_lib.dp_layer_sqnorms_keep(ctypes.byref(desc), _ptr(A), _ptr(G), _ptr(sqnorm_out), _ptr(grads),
                                      _ptr(workspace), _ws_len(workspace) if ws_bytes is None else ws_bytes,
                                      _stream(stream)))


def dp_clipped_sum_kept(desc: LayerDesc, grads, factors, dW, db=None, workspace=None, ws_bytes: Optional[int] = None,
                        accumulate: bool = False, stream=None) -> None:
    _check(_lib.dp_clipped_sum_kept(ctypes.byref(desc), _ptr(grads), _ptr(factors), _ptr(dW), _ptr(db),
                                    int(bool(accumulate)), _ptr(workspace),
                                    _ws_len(workspace) if ws_bytes is None else ws_bytes, _stream(stream)))


def noise_desc(sigma: float, C: float, B: int, seed: int = 0, seed_dev=None, offset: int = 0) -> NoiseDesc:
    return NoiseDesc(float(sigma), float(C), int(B), int(seed) & (2 ** 64 - 1), _ptr(seed_dev), int(offset))


def dp_clipped_sum_noised(desc: LayerDesc, A, G, factors, dW, db, noise: NoiseDesc, workspace=None,
                          ws_bytes: Optional[int] = None, norm_mode: int = -1, accumulate: bool = False,
                          stream=None) -> None:
    """The clipped sum (norm_mode -1: dp_clipped_sum; >= 0: dp_clipped_sum_reuse) and the
    noise of dp_add_noise on this layer's blocks in one call."""
    _check(_lib.dp_clipped_sum_noised(ctypes.byref(desc), norm_mode, _ptr(A), _ptr(G), _ptr(factors), _ptr(dW),
                                      _ptr(db), int(bool(accumulate)), ctypes.byref(noise), _ptr(workspace),
                                      _ws_len(workspace) if ws_bytes is None else ws_bytes, _stream(stream)))


def dp_clipped_sum_kept_noised(desc: LayerDesc, grads, factors, dW, db, noise: NoiseDesc, workspace=None,
                               ws_bytes: Optional[int] = None, accumulate: bool = False, stream=None) -> None:
    _check(_lib.dp_clipped_sum_kept_noised(ctypes.byref(desc), _ptr(grads), _ptr(factors), _ptr(dW), _ptr(db),
                                           int(bool(accumulate)), ctypes.byref(noise), _ptr(workspace),
                                           _ws_len(workspace) if ws_bytes is None else ws_bytes, _stream(stream)))


def dp_add_noise_blocks(grad, blocks, sigma: float, B: int, seed: int = 0, seed_dev=None, stream=None) -> None:
    """dp_add_noise over several (offset, n, C) blocks of the flat gradient `grad` in one launch."""
    arr = (NoiseBlock * len(blocks))(*[NoiseBlock(int(o), int(n), float(c)) for o, n, c in blocks])
    _check(_lib.dp_add_noise_blocks(_ptr(grad), arr, len(blocks), float(sigma), int(B), int(seed) & (2 ** 64 - 1),
                                    _ptr(seed_dev), _stream(stream)))


def dp_selftest_wait_timeout(waited_ns=None, stream=None) -> None:
    """Launch the diagnostic kernel whose bounded device wait runs out (see dpclip.h);
    dp_check_status then returns DP_ERR_TIMEOUT."""
    _check(_lib.dp_selftest_wait_timeout(_ptr(waited_ns), _stream(stream)))


def dp_check_status(stream=None) -> int:
    """Synchronizes and returns the device status (DP_OK or the raised code) without raising."""
    return _lib.dp_check_status(_stream(stream))


from .step import ClipPipeline, ClipStep, VirtualStep  # noqa: E402,F401
from .engine import PrivacyEngine  # noqa: E402,F401
