"""The allocation-free GEMM entry point, w12_gemm_noalloc.

It serves callers that cannot allocate device memory (a plug-in whose host framework hands out
no device memory, a serving loop that must not call cudaMalloc because it can synchronise the
device): its workspace is a fixed array inside the library. These tests call it through the C
ABI and check its output against w12_gemm's and against the oracle's fp64 product, within the
GEMM error bound the other tests use, on two calls in a row (the array keeps the previous call's
contents). The file name sorts last, so a run that stops at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from lossless_bit_weight_gb300 import synth
from w12_testutil import REL, ABS, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from lossless_bit_weight_gb300 import build, w12 as mod

    build.build()
    oracle.build()
    return mod


def _call(w12, t, x, y):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return w12.lib().w12_gemm_noalloc(ctypes.byref(t.c), ctypes.c_void_p(x.data_ptr()), x.shape[0],
                                      ctypes.c_void_p(y.data_ptr()), w12.OUT_F32, stream)


@pytest.mark.parametrize("N,K,M", [(2100, 1024, 1), (2100, 1024, 32), (17408, 5120, 8)])
def test_noalloc_matches_gemm_on_two_calls(w12, N, K, M):
    w = synth.weights(N, K, synth.PROJ, seed=N + M, device="cuda")
    t = w12.encode(w)
    x = synth.activations(M, K, seed=M, device="cuda")
    ref = w12.gemm(t, x)
    y_ref, absdot = oracle.gemm(to_np_u16(x), to_np_u16(w))
    tol = REL * absdot + ABS
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(w12, t, x, y) == w12.OK
        torch.cuda.synchronize()
        diff = (y - ref).abs().double().cpu().numpy()
        assert np.all(diff <= tol)
        assert np.all(np.abs(y.double().cpu().numpy() - y_ref) <= tol)


def test_noalloc_rejects_problems_beyond_its_array(w12):
    w = synth.weights(256, 256, synth.TINY, seed=1, device="cuda")
    t = w12.encode(w)
    x = synth.activations(33, 256, seed=2, device="cuda")
    y = torch.empty((33, 256), dtype=torch.float32, device="cuda")
    assert _call(w12, t, x, y) == w12.ERR_UNSUPPORTED_SHAPE
