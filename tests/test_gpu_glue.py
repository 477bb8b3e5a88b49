"""The synthetic layer stream's glue on the GPU against the oracle, and the GEMM's accumulate mode.

- the row normalisation bf16(h / rms(h)): the oracle's bits, up to one bf16 ulp where the fp64
  sums (added in another order) straddle a rounding boundary; zero, constant and scaled rows;
- the gate-up product bf16(fp32(g u)) bit for bit, from the two halves of one [M, 2N] output;
- y += x W^T (W12_LAUNCH_ACCUMULATE): bitwise equal to y0 + (x W^T) added in fp32, through each
  way y leaves the kernel (tensor stores with a reduce-add, plain stores, the split-tile reduce
  kernel), plain and overlapped, exact and Q view; invalid combinations rejected.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from lossless_bit_weight_gb300 import synth
from w12_testutil import to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from lossless_bit_weight_gb300 import build, w12 as mod

    build.build()
    oracle.build()
    return mod


def _ulps(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 steps between two arrays of finite bf16 bit patterns of equal sign."""
    ia = a.astype(np.int32)
    ib = b.astype(np.int32)
    ma = np.where(ia & 0x8000, -(ia & 0x7FFF), ia)
    mb = np.where(ib & 0x8000, -(ib & 0x7FFF), ib)
    return np.abs(ma - mb)


@pytest.mark.parametrize("M,K", [(1, 5120), (5, 6144), (32, 17408), (384, 72)])
def test_rms_bf16_matches_oracle(w12, M, K):
    g = torch.Generator(device="cuda").manual_seed(M * 1000 + K)
    h = torch.randn((M, K), generator=g, device="cuda") * 7
    if M >= 5:
        h[1] = 0.0                       # all-zero row
        h[2] = -3.25                     # constant row
        h[3] *= 2.0 ** 60                # scaled rows
        h[4] *= 2.0 ** -60
    x = w12.rms_bf16(h)
    xo = w12.rms_bf16(h, overlap=True)
    assert torch.equal(x, xo)
    ref = oracle.rms_bf16(h.cpu().numpy())
    got = to_np_u16(x)
    d = _ulps(got, ref)
    assert d.max() <= 1
    assert np.count_nonzero(d) <= max(1, got.size // 10000)
    if M >= 5:
        assert not np.any(got[1]) and np.all(got[2] == 0xBF80)


@pytest.mark.parametrize("M,N", [(1, 17408), (16, 17408), (32, 100), (384, 72)])
def test_mul_bf16_matches_oracle(w12, M, N):
    g = torch.Generator(device="cuda").manual_seed(M + N)
    gu = torch.randn((M, 2 * N), generator=g, device="cuda") * 3
    p = w12.mul_bf16(gu, N)
    assert torch.equal(p, w12.mul_bf16(gu, N, overlap=True))
    ref = oracle.mul_bf16(gu[:, :N].cpu().numpy(), gu[:, N:].cpu().numpy())
    assert np.array_equal(to_np_u16(p), ref)


# whole tiles with tensor stores (136 tiles on 152 SMs), whole tiles with plain stores (rows of
# y not a multiple of 16 bytes), split tiles summed by the reduce kernel (8 tiles)
@pytest.mark.parametrize("N,K,M", [(17408, 512, 32), (19454, 256, 16), (1000, 320, 33), (1000, 320, 1)])
@pytest.mark.parametrize("qview", [False, True])
def test_gemm_accumulate(w12, N, K, M, qview):
    w = synth.weights(N, K, synth.PROJ, seed=N + K, device="cuda")
    x = synth.activations(M, K, seed=M, device="cuda")
    t = w12.encode(w)
    y0 = torch.randn((M, N), device="cuda")
    plain = w12.gemm(t, x, qview=qview)
    y = y0.clone()
    w12.gemm(t, x, qview=qview, out=y, accumulate=True)
    assert torch.equal(y.view(torch.int32), (y0 + plain).view(torch.int32))
    y2 = y0.clone()
    w12.gemm(t, x, qview=qview, out=y2, accumulate=True, overlap=True)
    assert torch.equal(y2, y)
    w12.check(t)
    if not qview:
        y_ref, ad = oracle.gemm(to_np_u16(x), to_np_u16(w))
        y_ref = y_ref + y0.double().cpu().numpy()
        e = np.abs(y.double().cpu().numpy() - y_ref)
        assert np.all(e <= 2e-3 * ad + 1e-6 + np.abs(y_ref) * 2.0 ** -23)


def test_accumulate_rejects_bf16_and_argmax(w12):
    N, K, M = 256, 64, 2
    w = synth.weights(N, K, synth.PROJ, seed=5, device="cuda")
    t = w12.encode(w)
    x = synth.activations(M, K, seed=6, device="cuda")
    yb = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):  # the binding's own check
        w12.gemm(t, x, out=yb, accumulate=True)
    wg, ng = t.workspace(M, w12.OP_GEMM)
    st = w12.lib().w12_gemm_ex(ctypes.byref(t.c), w12._ptr(x), M, w12.OP_GEMM, w12._ptr(yb), w12.OUT_BF16, None,
                               None, None, w12.LAUNCH_ACCUMULATE, w12._ptr(wg), ng, w12._stream())
    assert st == w12.ERR_INVALID_ARG
    # an output buffer of the wrong type or shape never reaches the library
    with pytest.raises(ValueError):
        w12.gemm(t, x, out=torch.empty((M, N - 1), device="cuda"))
    ws, nb = t.workspace(M, w12.OP_ARGMAX)
    idx = torch.empty(M, dtype=torch.int32, device="cuda")
    val = torch.empty(M, dtype=torch.float32, device="cuda")
    st = w12.lib().w12_gemm_ex(ctypes.byref(t.c), w12._ptr(x), M, w12.OP_ARGMAX, None, 0,
                               w12._ptr(idx), w12._ptr(val), w12._ptr(val), w12.LAUNCH_ACCUMULATE, w12._ptr(ws), nb,
                               w12._stream())
    assert st == w12.ERR_INVALID_ARG


def test_carried_chain_in_cuda_graph_matches_eager(w12):
    """Two layers of the carried step as the benchmark runs them (overlapped GEMMs, q|k|v in one
    GEMM whose q columns feed the o projection in place, the residual adds accumulated into h,
    stream-ordered glue, all captured in one CUDA graph) give the eager stream-ordered chain's h
    and head argmax bit for bit, replay after replay."""
    K, NM = synth.HIDDEN, 2048
    shapes = (("qkv", K, 1536), ("o", 1024, K), ("gu", K, 2 * NM), ("down", NM, K))
    layers = []
    for layer in range(2):
        layers.append({n: w12.encode(synth.weights(no, ki, synth.PROJ, seed=97 * layer + i, device="cuda"))
                       for i, (n, ki, no) in enumerate(shapes)})
    th = w12.encode(synth.weights(4096, K, synth.HEAD, seed=99, device="cuda"))
    M = 16
    h0 = synth.activations(M, K, seed=98, device="cuda").float()
    h = torch.empty_like(h0)
    xa = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    qkv = torch.empty((M, 1536), dtype=torch.bfloat16, device="cuda")
    a = qkv[:, :1024]  # the o projection reads the q columns in place (rows 1536 apart)
    gu = torch.empty((M, 2 * NM), dtype=torch.float32, device="cuda")
    pz = torch.empty((M, NM), dtype=torch.bfloat16, device="cuda")

    def chain(overlap):
        h.copy_(h0)
        for L in layers:
            w12.rms_bf16(h, out=xa)
            w12.gemm(L["qkv"], xa, out=qkv, overlap=overlap)
            w12.gemm(L["o"], a, out=h, accumulate=True, overlap=overlap)
            w12.rms_bf16(h, out=xa)
            w12.gemm(L["gu"], xa, out=gu, overlap=overlap)
            w12.mul_bf16(gu, NM, out=pz)
            w12.gemm(L["down"], pz, out=h, accumulate=True, overlap=overlap)
        w12.rms_bf16(h, out=xa)
        return w12.lmhead_argmax(th, xa, overlap=overlap)

    ref_idx, ref_val, _ = chain(False)
    ref_h = h.clone()
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        chain(True)  # workspaces and kernel attributes before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            gi, gv, _ = chain(True)
        for _ in range(3):
            g.replay()
            st.synchronize()
            assert torch.equal(h.view(torch.int32), ref_h.view(torch.int32))
            assert torch.equal(gi, ref_idx) and torch.equal(gv, ref_val)
    for L in layers:
        for t in L.values():
            w12.check(t)
    w12.check(th)
