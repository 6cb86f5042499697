"""The oracle's Philox4x32-10 against a library implementation: cuRAND's device API.

The pages fix only N(0, sigma^2 C^2) for the privacy noise; the generator is this
build's reading, Philox4x32-10 (Salmon et al., SC'11).  cuRAND implements the same
generator, and its documented device API positions a stream by (seed, subsequence,
offset): key = the 64-bit seed, subsequence in the counter's high words, offset/4 in
its low words.  A small test kernel (tests/native/curand_philox_words.cu, built here)
draws curand4 at counter (q, stream); the oracle's raw words must equal them bit for
bit, for several seeds, streams and counters (including ones past 2^32).
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from oracle.philox import noise_words

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "native", "curand_philox_words.cu")
OUT = os.path.join(HERE, "_build", "libcurand_philox_words.so")


@pytest.fixture(scope="module")
def curand_words(lib):
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    if not os.path.exists(OUT) or os.path.getmtime(OUT) < os.path.getmtime(SRC):
        nvcc = "/usr/local/cuda/bin/nvcc"
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler",
                        "-fPIC", SRC, "-o", OUT], check=True)
    so = ctypes.CDLL(OUT)
    f = so.curand_philox_words
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_ulonglong, ctypes.c_ulonglong, ctypes.c_ulonglong, ctypes.c_int,
                  ctypes.POINTER(ctypes.c_uint)]

    def words(seed, stream, q0, n):
        buf = (ctypes.c_uint * (4 * n))()
        assert f(seed, stream, q0, n, buf) == 0
        return np.array(buf[:], dtype=np.uint64).reshape(n, 4)
    return words


@pytest.mark.parametrize("seed,stream,q0", [(0, 0, 0), (0x1234_5678_9ABC, 0, 0), (99, 1, 5),
                                            (2 ** 64 - 1, 0, 2 ** 32 - 3), (7, 1, 123_456_789_012)])
def test_oracle_philox_words_equal_curand(curand_words, seed, stream, q0):
    n = 4096
    want = curand_words(seed, stream, q0, n)
    got, first = noise_words(4 * n, seed, offset=4 * q0, stream=stream)
    assert first == q0
    np.testing.assert_array_equal(got, want)
