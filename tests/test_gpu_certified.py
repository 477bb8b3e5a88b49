"""Certified LM head (SpecPilot §4.1 "Certified LM head") on the GPU against the oracle.

- the INT8 copy: codes and scales bit for bit, bounds at or above the oracle's residual norms
  and within the stated evaluation margin of them, padding and non-finite rows;
- the approximate logits of the INT8 pass against s_n (x . q_n) in fp64;
- the certified argmax against the oracle's full argmax (and the oracle's certified argmax),
  survivor counts at or above the oracle's;
- the fallback when a row has more survivors than the list holds, and that the next call runs
  without it;
- the full-size head (vocabulary 151936 x 5120, 32 rows) against the oracle's fp64 argmax;
- the INT8 Q pass's argmax against the oracle's INT8 logits.
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_bit_weight_gb300 import synth
from w12_testutil import argmax_check, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from lossless_bit_weight_gb300 import build, w12 as mod

    build.build()
    oracle.build()
    return mod


def codes_rowmajor(h, N, K):
    """The copy's sign-magnitude record bytes as a row-major int8 matrix [N, K]."""
    nt, kt = (N + 127) // 128, (K + 63) // 64
    b = h.codes.cpu().numpy().reshape(nt, kt, 4, 128, 16)          # [nt, kt, chunk, n_l, j]
    b = b.transpose(0, 3, 1, 2, 4).reshape(nt * 128, kt * 64)       # [n, k]
    v = (b & 0x7F).astype(np.int16) * np.where(b & 0x80, -1, 1).astype(np.int16)
    return v[:N, :K].astype(np.int8), b


def _special_head(N, K, seed):
    w = synth.weights(N, K, synth.HEAD, seed=seed, device="cuda")
    bits = w.view(torch.int16)
    bits[3] = 0                       # all-zero row
    bits[5, 7] = 0x7F80               # +Inf
    bits[6, 9] = 0x7FC1               # NaN
    bits[7] = 0x3F80                  # all 1.0
    bits[8, 0] = 0x0001               # a subnormal next to normal weights
    return w


@pytest.mark.parametrize("N,K", [(1000, 320), (256, 64), (300, 200)])
def test_q8_copy_matches_oracle(w12, N, K):
    w = _special_head(N, K, seed=N + K)
    h = w12.q8_build(w)
    torch.cuda.synchronize()
    ref = oracle.head_q8(to_np_u16(w))
    q, raw = codes_rowmajor(h, N, K)
    assert np.array_equal(q, ref.q)
    # padding rows and padding k hold code 0
    assert not np.any(raw[N:]) and not np.any(raw[:, K:])
    scale = h.scale.cpu().numpy()
    bound = h.bound.cpu().numpy().astype(np.float64)
    assert np.array_equal(scale[:N], ref.scale)
    assert not np.any(scale[N:]) and not np.any(bound[N:])
    fin = np.isfinite(ref.resid)
    assert np.array_equal(np.isinf(bound[:N]), ~fin)
    r, qn, s = ref.resid[fin], ref.qnorm[fin], ref.scale[fin].astype(np.float64)
    b = bound[:N][fin]
    assert np.all(b >= r)
    margin = s * qn * (K + 3) * 2.0 ** -21
    assert np.all(b <= (r + margin) * (1 + 2.0 ** -15) + 1e-30)


def test_q8_bound_covers_every_logit(w12):
    """The GPU's row bounds: every exact logit lies within s_n (x . q_n) -+ ||x|| bound[n] (the
    interval the certified argmax relies on), on a head with zero, Inf, NaN and subnormal rows
    left out of the check only where the bound is infinite."""
    N, K, M = 1000, 320, 8
    w = synth.weights(N, K, synth.HEAD, seed=21, device="cuda")
    x = synth.activations(M, K, seed=22, device="cuda")
    h = w12.q8_build(w)
    ref = oracle.head_q8(to_np_u16(w))
    xv = (to_np_u16(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    yh = (xv @ ref.q.astype(np.float64).T) * ref.scale.astype(np.float64)[None, :]
    y, _ = oracle.gemm(to_np_u16(x), to_np_u16(w))
    bound = h.bound.cpu().numpy()[:N].astype(np.float64)
    xn = np.linalg.norm(xv, axis=1)
    assert np.all(np.abs(y - yh) <= xn[:, None] * bound[None, :])


@pytest.mark.parametrize("rescore", ["w12", "bf16"])
@pytest.mark.parametrize("N,K,M,seed", [(3000, 256, 8, 1), (2000, 192, 5, 2), (1000, 320, 33, 3), (129, 64, 2, 4)])
def test_certified_argmax_matches_oracle(w12, N, K, M, seed, rescore):
    w = synth.weights(N, K, synth.HEAD, seed=seed, device="cuda")
    if seed == 3:  # escapes in every row: a zero and a weight 2^12 times larger
        bits = w.view(torch.int16)
        bits[:, 5] = 0
        bits[:, 300] = bits[:, 300] + (12 << 7)
    x = synth.activations(M, K, seed=seed + 100, device="cuda")
    t = w12.encode(w)
    h = w12.q8_build(w)
    idx, val, gap, surv = w12.lmhead_certified(t, h, x, w_bf16=w if rescore == "bf16" else None)
    w12.check(t)
    wn, xn = to_np_u16(w), to_np_u16(x)
    y_ref, ad = oracle.gemm(xn, wn)
    checked, near, wrong, det = argmax_check(idx.cpu().numpy(), val.cpu().numpy(), gap.cpu().numpy(), y_ref, ad)
    assert wrong == 0, det
    assert checked + near == M
    # the GPU's bound is the oracle's plus its evaluation margin: it keeps at least as many
    _, _, _, ocnt = oracle.certified_argmax(xn, wn, oracle.head_q8(wn))
    s = surv.cpu().numpy()
    assert np.all(s >= ocnt) and np.all(s <= N)
    # the same rows through the fused W12 argmax
    fidx, fval, fgap = w12.lmhead_argmax(t, x)
    c2, n2, w2, d2 = argmax_check(fidx.cpu().numpy(), fval.cpu().numpy(), fgap.cpu().numpy(), y_ref, ad)
    assert w2 == 0


def test_certified_fallback_and_recovery(w12):
    """Identical rows tie: every token survives, the list (4096) overflows and the full W12
    argmax gives every row's result (index 0, gap 0); the next call, on an ordinary head, runs
    without the fallback."""
    N, K, M = 5000, 128, 4
    row = synth.weights(1, K, synth.HEAD, seed=31, device="cuda")
    w = row.repeat(N, 1).contiguous()
    x = synth.activations(M, K, seed=32, device="cuda")
    t = w12.encode(w)
    h = w12.q8_build(w)
    idx, val, gap, surv = w12.lmhead_certified(t, h, x)
    w12.check(t)
    assert np.all(surv.cpu().numpy() == N)
    assert np.all(idx.cpu().numpy() == 0) and np.all(gap.cpu().numpy() == 0)
    fidx, fval, fgap = w12.lmhead_argmax(t, x)
    assert torch.equal(val, fval)
    # an ordinary head next, through the same certified path (its own workspace)
    w2 = synth.weights(3000, K, synth.HEAD, seed=33, device="cuda")
    t2, h2 = w12.encode(w2), w12.q8_build(w2)
    idx2, val2, gap2, surv2 = w12.lmhead_certified(t2, h2, x)
    w12.check(t2)
    y_ref, ad = oracle.gemm(to_np_u16(x), to_np_u16(w2))
    _, _, wrong, det = argmax_check(idx2.cpu().numpy(), val2.cpu().numpy(), gap2.cpu().numpy(), y_ref, ad)
    assert wrong == 0, det
    assert np.all(surv2.cpu().numpy() < 4096)


def test_certified_full_head(w12):
    """The LM head workload (vocabulary 151936, K=5120, 32 rows): the certified argmax, rescored
    from the W12 records and from a bf16 copy, against the oracle's fp64 argmax of the whole head
    (exact top-1 wherever the oracle's gap is clear of the near-tie band, value within the GEMM
    bound); the fused W12 argmax agrees with it."""
    V, K = 151936, 5120
    w = synth.weights(V, K, synth.HEAD, seed=synth.seed_for(2, 0), device="cuda")
    x = synth.activations(32, K, seed=synth.seed_for(2, 1), device="cuda")
    t = w12.encode(w)
    h = w12.q8_build(w)
    ib, vb, gb, sb = w12.lmhead_certified(t, h, x, w_bf16=w)
    idx, val, gap, surv = w12.lmhead_certified(t, h, x)
    fidx, fval, fgap = w12.lmhead_argmax(t, x)
    w12.check(t)
    y_ref, ad = oracle.gemm(to_np_u16(x), to_np_u16(w))
    for i, v, g in ((idx, val, gap), (ib, vb, gb), (fidx, fval, fgap)):
        checked, near, wrong, det = argmax_check(i.cpu().numpy(), v.cpu().numpy(), g.cpu().numpy(), y_ref, ad)
        assert wrong == 0, det
        assert checked + near == 32 and checked >= 30
    assert torch.equal(surv, sb)
    s = surv.cpu().numpy()
    assert np.all(s >= 2) and np.all(s <= 4096)


@pytest.mark.parametrize("N,K,M,seed", [(3000, 256, 8, 41), (20000, 192, 16, 42), (129, 64, 3, 43)])
def test_q8_argmax_matches_oracle(w12, N, K, M, seed):
    """The Q pass over the INT8 copy: its argmax against the oracle's argmax of s_n (x . q_n), both
    whole-tile and split-tile (stream-K) layouts; overlapped and plain launches agree bitwise."""
    w = synth.weights(N, K, synth.HEAD, seed=seed, device="cuda")
    x = synth.activations(M, K, seed=seed + 1, device="cuda")
    h = w12.q8_build(w)
    idx, val, gap = w12.q8_argmax(h, x)
    io, vo, go = w12.q8_argmax(h, x, overlap=True)
    assert torch.equal(idx, io) and torch.equal(val.view(torch.int32), vo.view(torch.int32))
    yh, ad = oracle.gemm_q8(to_np_u16(x), oracle.head_q8(to_np_u16(w)))
    checked, near, wrong, det = argmax_check(idx.cpu().numpy(), val.cpu().numpy(), gap.cpu().numpy(), yh, ad)
    assert wrong == 0, det
    assert checked + near == M
