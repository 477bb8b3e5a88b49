"""The INT6 Q-pass copy (SpecPilot §5.3, App. C) on the GPU against the oracle.

- the copy: record bytes and row scales bit for bit against the oracle's quantisation and record
  packing, with zero, Inf, NaN, subnormal and ragged rows and columns;
- the Q-pass GEMM against the oracle's fp64 s_n (x . c_n): fp32 and bf16 outputs, whole-tile and
  split-tile (stream-K) layouts, 1 to 384 rows, plain and overlapped launches bitwise equal;
- the Q-pass argmax against the oracle's argmax of the same logits (near-ties counted);
- the LM-head workload (vocabulary 151936 x 5120, 64 rows): sampled logits against the oracle,
  the argmax against the GEMM's own output, and the agreement with the exact W12 argmax
  (reported, not pinned).
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_bit_weight_gb300 import synth
from w12_testutil import argmax_check, gemm_violations, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from lossless_bit_weight_gb300 import build, w12 as mod

    build.build()
    oracle.build()
    return mod


def _special(N, K, seed, recipe=synth.HEAD):
    w = synth.weights(N, K, recipe, seed=seed, device="cuda")
    bits = w.view(torch.int16)
    bits[3 % N] = 0                       # all-zero row
    if N > 8:
        bits[5, 7] = 0x7F80               # +Inf
        bits[6, 1] = 0x7FC1               # NaN
        bits[7] = 0x3F80                  # all 1.0
        bits[8, 0] = 0x0001               # a subnormal next to normal weights
    return w


@pytest.mark.parametrize("N,K", [(1000, 320), (256, 64), (300, 200), (129, 8)])
def test_q6_copy_matches_oracle(w12, N, K):
    w = _special(N, K, seed=N + 3 * K)
    c = w12.q6_build(w)
    torch.cuda.synchronize()
    ref = oracle.copy_q6(to_np_u16(w))
    assert np.array_equal(c.codes.cpu().numpy(), oracle.q6_pack(ref.q))
    scale = c.scale.cpu().numpy()
    assert np.array_equal(scale[:N], ref.scale)
    assert not np.any(scale[N:])


def _q6_ref(w, x):
    ref = oracle.copy_q6(to_np_u16(w))
    return oracle.gemm_q6(to_np_u16(x), ref)


@pytest.mark.parametrize("N,K,M", [(1000, 320, 1), (1000, 320, 33), (3000, 256, 16), (129, 64, 5),
                                   (640, 192, 192), (520, 128, 300), (384, 64, 384)])
def test_q6_gemm_matches_oracle(w12, N, K, M):
    w = _special(N, K, seed=7 * N + M, recipe=synth.PROJ)
    x = synth.activations(M, K, seed=M + 11, device="cuda")
    c = w12.q6_build(w)
    y = w12.q6_gemm(c, x)
    yo = w12.q6_gemm(c, x, overlap=True)
    yb = w12.q6_gemm(c, x, out_dtype=torch.bfloat16)
    assert torch.equal(y.view(torch.int32), yo.view(torch.int32))
    y_ref, ad = _q6_ref(w, x)
    assert gemm_violations(y.cpu().numpy(), y_ref, ad) == 0
    assert gemm_violations(yb.float().cpu().numpy(), y_ref, ad, bf16=True) == 0
    # the same call again: bitwise reproducible
    assert torch.equal(w12.q6_gemm(c, x).view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("N,K,M,seed", [(3000, 256, 8, 51), (20000, 192, 16, 52), (129, 64, 3, 53),
                                        (2000, 320, 64, 54)])
def test_q6_argmax_matches_oracle(w12, N, K, M, seed):
    """The argmax over the copy against the oracle's argmax of s_n (x . c_n), whole-tile and
    split-tile layouts; overlapped and plain launches agree bitwise; the index equals that of the
    copy's own GEMM output wherever its top two differ."""
    w = synth.weights(N, K, synth.HEAD, seed=seed, device="cuda")
    x = synth.activations(M, K, seed=seed + 1, device="cuda")
    c = w12.q6_build(w)
    idx, val, gap = w12.q6_argmax(c, x)
    io, vo, go = w12.q6_argmax(c, x, overlap=True)
    assert torch.equal(idx, io) and torch.equal(val.view(torch.int32), vo.view(torch.int32))
    y_ref, ad = _q6_ref(w, x)
    checked, near, wrong, det = argmax_check(idx.cpu().numpy(), val.cpu().numpy(), gap.cpu().numpy(), y_ref, ad)
    assert wrong == 0, det
    assert checked + near == M
    y = w12.q6_gemm(c, x)
    top = torch.topk(y, 2, dim=1)
    clear = (top.values[:, 0] - top.values[:, 1] > 1e-5 * top.values[:, 0].abs()).cpu().numpy()
    assert np.array_equal(idx.cpu().numpy()[clear], top.indices[:, 0].int().cpu().numpy()[clear])


def test_q6_lm_head_workload(w12):
    """Vocabulary 151936 x 5120 at 64 rows: sampled logits of the copy's GEMM against the oracle
    (computed on the sampled rows of the head only, since each row's copy depends on that row
    alone), the argmax against the GEMM's own logits, and the top-1 agreement with the exact W12
    argmax, printed."""
    V, K, M = 151936, 5120, 64
    w = synth.weights(V, K, synth.HEAD, seed=synth.seed_for(2, 0), device="cuda")
    x = synth.activations(M, K, seed=synth.seed_for(4, 64), device="cuda")
    c = w12.q6_build(w)
    y = w12.q6_gemm(c, x)
    idx, val, gap = w12.q6_argmax(c, x)
    rng = np.random.default_rng(61)
    ns = np.unique(rng.integers(0, V, 512))
    ref = oracle.copy_q6(to_np_u16(w[torch.as_tensor(ns, device="cuda")]))
    assert np.array_equal(c.scale.cpu().numpy()[ns], ref.scale)
    y_ref, ad = oracle.gemm_q6(to_np_u16(x), ref)
    assert gemm_violations(y.cpu().numpy()[:, ns], y_ref, ad) == 0
    top = torch.topk(y, 2, dim=1)
    clear = (top.values[:, 0] - top.values[:, 1] > 1e-5 * top.values[:, 0].abs()).cpu().numpy()
    assert clear.sum() >= M - 2
    assert np.array_equal(idx.cpu().numpy()[clear], top.indices[:, 0].int().cpu().numpy()[clear])
    assert torch.allclose(val, top.values[:, 0], rtol=1e-6, atol=0)
    t = w12.encode(w)
    ie, _, _ = w12.lmhead_argmax(t, x)
    w12.check(t)
    print(f"INT6 copy top-1 agreement with the exact W12 argmax on the LM head at M={M}: "
          f"{float((ie == idx).float().mean()):.3f}")
