"""GPU parity of the W12 CUDA path against the CPU oracle, through the C ABI.

- encode: byte-identical records, window bases and both escape lists (SpecPilot §4.1, Fig. 5a);
- decode / verify: bit-exact round trip, corruption detected (SpecPilot §4.1 load-time check);
- GEMM, Q-view GEMM (SpecPilot §4.3) and fused argmax (SpecPilot §2.1) within the stated
  bounds, on ragged shapes that span several tiles, at every row count class, and repeatably.
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


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


def _assert_same_encoding(t, e):
    R = t.n_tiles * t.k_tiles
    assert np.array_equal(t.records.cpu().numpy(), e.records)
    assert np.array_equal(t.base_exp.cpu().numpy(), e.base_exp)
    assert np.array_equal(_u32(t.esc_off), e.esc_off)
    assert t.n_esc == e.esc_k.size
    assert np.array_equal(_u32(t.esc_k)[: t.n_esc], e.esc_k)
    assert np.array_equal(t.esc_bits.cpu().numpy().view(np.uint16)[: t.n_esc], e.esc_bits)
    assert np.array_equal(_u32(t.rec_esc_off), e.rec_esc_off)
    assert t.n_rec_esc == e.rec_esc.size
    assert np.array_equal(_u32(t.rec_esc)[: t.n_rec_esc], e.rec_esc)
    assert t.rec_esc_off.numel() == R + 1


def _weights(kind, N, K, seed):
    if kind == "synthetic":
        return synth.weights(N, K, synth.TINY, seed=seed, device="cuda")
    if kind == "all_patterns":
        return synth.from_bits(synth.all_bf16_patterns(K), device="cuda")
    if kind == "shuffled_patterns":
        rng = np.random.default_rng(seed)
        return synth.from_bits(rng.permutation(synth.all_bf16_patterns(512).reshape(-1)).reshape(N, K), "cuda")
    if kind == "zero_heavy":  # > 256 escapes in some records: the kernel's overflow path
        w = synth.weights(N, K, synth.TINY, seed=seed, device="cuda")
        w[:64, :] = 0
        w[200:210, 64:128] = 0
        return w
    raise ValueError(kind)


ENCODE_CASES = [
    ("synthetic", 512, 256), ("synthetic", 300, 200), ("synthetic", 1, 8), ("synthetic", 129, 72),
    ("all_patterns", 256, 256), ("shuffled_patterns", 128, 512), ("zero_heavy", 384, 320),
]


@pytest.mark.parametrize("kind,N,K", ENCODE_CASES)
def test_encode_matches_oracle_bytes(w12, kind, N, K):
    w = _weights(kind, N, K, seed=N + K)
    t = w12.encode(w)
    e = oracle.encode(to_np_u16(w))
    _assert_same_encoding(t, e)


@pytest.mark.parametrize("kind,N,K", ENCODE_CASES)
def test_decode_and_verify_bit_exact(w12, kind, N, K):
    w = _weights(kind, N, K, seed=N + K)
    t = w12.encode(w)
    assert torch.equal(w12.decode(t).view(torch.int16), w.view(torch.int16))
    assert w12.verify(t, w) == 0


def test_verify_detects_corruption(w12):
    w = synth.weights(300, 200, synth.TINY, seed=21, device="cuda")
    t = w12.encode(w)
    assert t.n_esc > 0
    t.records[5000] ^= 0x10            # one view byte
    assert w12.verify(t, w) >= 1
    t.records[5000] ^= 0x10
    assert w12.verify(t, w) == 0
    t.records[12288 + 9000] ^= 0x01    # one plane-B nibble in record 1
    assert w12.verify(t, w) >= 1
    t.records[12288 + 9000] ^= 0x01
    old = int(t.rec_esc[0])
    t.rec_esc[0] = old ^ (1 << 16)     # the bits of one escape entry
    assert w12.verify(t, w) >= 1
    t.rec_esc[0] = old
    t.esc_bits[0] ^= 1                 # the canonical list too
    assert w12.verify(t, w) >= 1
    t.esc_bits[0] ^= 1
    assert w12.verify(t, w) == 0


def _gemm_case(w12, N, K, M, seed, recipe=synth.TINY, qview=False, out_dtype=torch.float32, w=None):
    if w is None:
        w = synth.weights(N, K, recipe, seed=seed, device="cuda")
    x = synth.activations(M, K, seed=seed + 1, device="cuda")
    t = w12.encode(w)
    y = w12.gemm(t, x, out_dtype=out_dtype, qview=qview)
    w12.check(t)
    wb = to_np_u16(w)
    if qview:
        wb = oracle.qview_weights(wb)
    y_ref, absdot = oracle.gemm(to_np_u16(x), wb)
    yv = y.float().cpu().numpy()
    return t, x, y, yv, y_ref, absdot


@pytest.mark.parametrize("M", [1, 2, 3, 8, 16, 17, 32, 33, 64, 100, 192, 256, 257, 300, 384])
def test_gemm_ragged_all_row_classes(w12, M):
    _, _, _, yv, y_ref, ad = _gemm_case(w12, 300, 200, M, seed=100 + M)
    assert gemm_violations(yv, y_ref, ad) == 0


@pytest.mark.parametrize("N,K,M", [(512, 256, 1), (1024, 1024, 4), (640, 5120, 32), (2176, 320, 8)])
def test_gemm_shapes(w12, N, K, M):
    _, _, _, yv, y_ref, ad = _gemm_case(w12, N, K, M, seed=N + K + M)
    assert gemm_violations(yv, y_ref, ad) == 0


@pytest.mark.parametrize("M", [1, 32, 192])
def test_gemm_bf16_output(w12, M):
    _, _, _, yv, y_ref, ad = _gemm_case(w12, 640, 512, M, seed=7 + M, out_dtype=torch.bfloat16)
    assert gemm_violations(yv, y_ref, ad, bf16=True) == 0


def test_gemm_escape_overflow_path(w12):
    w = _weights("zero_heavy", 384, 320, seed=3)
    _, _, _, yv, y_ref, ad = _gemm_case(w12, 384, 320, 16, seed=3, w=w)
    assert gemm_violations(yv, y_ref, ad) == 0


def test_gemm_special_weights(w12):
    """Inf, NaN, signed zeros, subnormals and extreme binades, all restored through escapes."""
    w = synth.weights(256, 128, synth.TINY, seed=5, device="cuda")
    bits = w.view(torch.int16)
    for (n, k, u) in [(0, 0, 0x7F80),    # +Inf
                      (1, 3, 0x8000),    # -0
                      (2, 5, 0x0001),    # subnormal
                      (3, 7, 0x7E00),    # 2^125: top binade, no fp32 overflow after the sum
                      (4, 9, 0x0080),    # smallest normal
                      (5, 11, 0xFF80)]:  # -Inf
        bits[n, k] = int(np.array(u, np.uint16).view(np.int16))
    x = synth.activations(4, 128, seed=6, device="cuda")
    t = w12.encode(w)
    y = w12.gemm(t, x).cpu().numpy()
    y_ref, ad = oracle.gemm(to_np_u16(x), to_np_u16(w))
    finite = np.isfinite(y_ref)
    assert np.array_equal(np.isinf(y), np.isinf(y_ref))
    assert np.array_equal(np.sign(y[~finite]), np.sign(y_ref[~finite]))
    assert gemm_violations(y[finite], y_ref[finite], ad[finite]) == 0


def test_gemm_bitwise_reproducible(w12):
    w = synth.weights(2048, 2048, synth.PROJ, seed=9, device="cuda")
    x = synth.activations(32, 2048, seed=10, device="cuda")
    t = w12.encode(w)
    a = w12.gemm(t, x)
    b = w12.gemm(t, x)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    ia, va, ga = w12.lmhead_argmax(t, x)
    ib, vb, gb = w12.lmhead_argmax(t, x)
    assert torch.equal(ia, ib) and torch.equal(va.view(torch.int32), vb.view(torch.int32))


@pytest.mark.parametrize("M", [1, 32, 48, 64, 96, 192, 256, 320, 384])
@pytest.mark.parametrize("qview", [False, True])
def test_gemm_repeat_stress(w12, M, qview):
    """Thirty launches on weights larger than L2 (with 0.1% zeros: many escapes), every result
    bitwise equal to the first. Covers
    the ring configurations where the pipeline's stage count is not a multiple of the decode
    groups (slots shared between groups) as well as those where it is."""
    w = synth.weights(17408, 5120, synth.PROJ, seed=13, device="cuda")
    t = w12.encode(w)
    del w
    copies = [t] + [t.clone_records() for _ in range(2)]
    x = synth.activations(M, 5120, seed=14 + M, device="cuda")
    first = w12.gemm(copies[0], x, qview=qview)
    for i in range(1, 30):
        y = w12.gemm(copies[i % 3], x, qview=qview)
        assert torch.equal(y.view(torch.int32), first.view(torch.int32)), i
    for c in copies:
        w12.check(c)


def test_workspace_counters_left_zeroed(w12):
    """Counters and the error word (the head of the workspace) are back at zero after a call, so
    the next call can reuse the workspace without clearing it; partial sums need no clearing."""
    w = synth.weights(1000, 640, synth.TINY, seed=11, device="cuda")
    x = synth.activations(8, 640, seed=12, device="cuda")
    t = w12.encode(w)
    for _ in range(2):
        w12.gemm(t, x)
        w12.lmhead_argmax(t, x)
    torch.cuda.synchronize()
    align = lambda v: (v + 255) // 256 * 256
    head = 256 + align(4 * t.n_tiles) + 256  # error word, per-tile counters, completion counter
    for ws, nb in t._ws.values():
        assert int(ws[:head].count_nonzero()) == 0


@pytest.mark.parametrize("M", [1, 16, 64, 192, 300])
def test_qview_gemm(w12, M):
    _, _, _, yv, y_ref, ad = _gemm_case(w12, 300, 200, M, seed=300 + M, qview=True)
    assert gemm_violations(yv, y_ref, ad) == 0


@pytest.mark.parametrize("N,K,M", [(1000, 448, 8), (2000, 320, 32), (4000, 192, 3), (640, 1344, 17)])
def test_qview_gemm_odd_record_counts(w12, N, K, M):
    """Q view where blocks hold odd numbers of records and tiles an odd number of k slices: a
    slot's view copy then spans a record the block does not decode, or one past the last."""
    _, _, _, yv, y_ref, ad = _gemm_case(w12, N, K, M, seed=N + K + M, qview=True)
    assert gemm_violations(yv, y_ref, ad) == 0


@pytest.mark.parametrize("N,K,M,qview", [(3000, 512, 32, False), (1000, 256, 1, False),
                                         (3000, 512, 64, True), (129, 64, 5, False), (2000, 256, 300, False)])
def test_lmhead_argmax(w12, N, K, M, qview):
    w = synth.weights(N, K, synth.HEAD, seed=N + M, device="cuda")
    x = synth.activations(M, K, seed=N + M + 1, device="cuda")
    t = w12.encode(w)
    idx, val, gap = w12.lmhead_argmax(t, x, qview=qview)
    w12.check(t)
    wb = to_np_u16(w)
    if qview:
        wb = oracle.qview_weights(wb)
    y_ref, ad = oracle.gemm(to_np_u16(x), wb)
    checked, near, wrong, details = argmax_check(idx.cpu().numpy(), val.cpu().numpy(),
                                                 gap.cpu().numpy(), y_ref, ad)
    assert wrong == 0, details
    # near-ties (gap under 1e-3 of the row's scale) are a property of the data: a few per 100 rows
    assert checked + near == M and checked >= M - max(2, M // 25)
    # the gap is the difference of two GEMM outputs: within their summed bounds
    ridx, rval, rgap, _ = oracle.argmax(y_ref)
    g = gap.cpu().numpy().astype(np.float64)
    for m in range(M):
        if int(idx[m]) == ridx[m]:
            assert abs(g[m] - rgap[m]) <= 2 * (2e-3 * ad[m].max() + 1e-6)


def test_overlap_launch_chain_matches_plain(w12):
    """W12_LAUNCH_OVERLAP: each GEMM reads the previous GEMM's output as its x, with
    the programmatic dependent launch. The results equal those of plain launches bit for bit, the
    argmax included. The same tensor and workspace are reused back to back."""
    w1 = synth.weights(1024, 2048, synth.PROJ, seed=21, device="cuda")
    w2 = synth.weights(2048, 1024, synth.PROJ, seed=22, device="cuda")
    t1, t2 = w12.encode(w1), w12.encode(w2)
    x = synth.activations(16, 2048, seed=23, device="cuda")

    def chain(overlap):
        outs = []
        h = x
        for _ in range(6):
            a = w12.gemm(t1, h, out_dtype=torch.bfloat16, overlap=overlap)
            h = w12.gemm(t2, a, out_dtype=torch.bfloat16, overlap=overlap)
            outs.append(h)
        outs.append(w12.lmhead_argmax(t1, h, overlap=overlap)[0])
        return outs

    plain = chain(False)
    over = chain(True)
    torch.cuda.synchronize()
    for a, b in zip(plain, over):
        assert torch.equal(a, b)
    w12.check(t1)
    w12.check(t2)


def test_bounded_wait_timeout_is_reported(w12):
    """The failure path, without a GPU fault: under the W12_LAUNCH_TEST_STALL hook each block's
    producer fills only its first pipeline slot, the waits on the next slot give up after about a
    second, every block stops, and w12_check reports W12_ERR_TIMEOUT. The context stays usable:
    once the workspace is zero-filled again a normal call gives the right result."""
    w = synth.weights(512, 256, synth.TINY, seed=31, device="cuda")
    x = synth.activations(4, 256, seed=32, device="cuda")
    t = w12.encode(w)
    w12.gemm(t, x, test_stall=True)
    with pytest.raises(w12.W12Error) as e:
        w12.check(t)
    assert e.value.status == w12.ERR_TIMEOUT
    for ws, _ in t._ws.values():
        ws.zero_()
    y = w12.gemm(t, x)
    y_ref, ad = oracle.gemm(to_np_u16(x), to_np_u16(w))
    assert gemm_violations(y.cpu().numpy(), y_ref, ad) == 0
    w12.check(t)


def test_overlap_chain_in_cuda_graph(w12):
    """GEMMs launched with W12_LAUNCH_OVERLAP inside a captured CUDA graph: a chain in which each
    GEMM reads the previous one's output, stream-K shapes included (their reduce kernels become
    graph nodes too). Replays give the eager plain-launch results bit for bit."""
    w1 = synth.weights(1024, 2048, synth.PROJ, seed=41, device="cuda")  # stream-K: 8 tiles
    w2 = synth.weights(2048, 1024, synth.PROJ, seed=42, device="cuda")
    t1, t2 = w12.encode(w1), w12.encode(w2)
    x = synth.activations(32, 2048, seed=43, device="cuda")

    def chain(overlap):
        a = w12.gemm(t1, x, out_dtype=torch.bfloat16, overlap=overlap)
        b = w12.gemm(t2, a, out_dtype=torch.bfloat16, overlap=overlap)
        c = w12.gemm(t1, b, overlap=overlap)
        return c, w12.lmhead_argmax(t1, b, overlap=overlap)[0]

    ref_y, ref_i = chain(False)
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        chain(True)  # workspaces and kernel attributes before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            gy, gi = chain(True)
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    assert torch.equal(gy.view(torch.int32), ref_y.view(torch.int32))
    assert torch.equal(gi, ref_i)
    w12.check(t1)
    w12.check(t2)


@pytest.mark.parametrize("M", [1, 16, 33, 192])
def test_strided_activations(w12, M):
    """x as a column slice of a wider bf16 tensor (w12_gemm_strided) gives the contiguous copy's
    results bit for bit, plain, overlapped and accumulated; row strides that are not a multiple
    of 8 elements never reach a kernel."""
    N, K, W = 2176, 320, 512
    w = synth.weights(N, K, synth.PROJ, seed=71 + M, device="cuda")
    t = w12.encode(w)
    big = synth.activations(M, W, seed=72 + M, device="cuda")
    xs = big[:, :K]
    xc = xs.contiguous()
    ref = w12.gemm(t, xc)
    assert torch.equal(w12.gemm(t, xs).view(torch.int32), ref.view(torch.int32))
    assert torch.equal(w12.gemm(t, xs, overlap=True).view(torch.int32), ref.view(torch.int32))
    assert torch.equal(w12.gemm(t, xs, qview=True).view(torch.int32), w12.gemm(t, xc, qview=True).view(torch.int32))
    y0 = torch.randn((M, N), device="cuda")
    y = y0.clone()
    w12.gemm(t, xs, out=y, accumulate=True)
    assert torch.equal(y.view(torch.int32), (y0 + ref).view(torch.int32))
    w12.check(t)
    odd = synth.activations(M, K + 4, seed=73, device="cuda")[:, :K]
    with pytest.raises(w12.W12Error):
        w12.gemm(t, odd)


def test_rows_above_limit_rejected(w12):
    """M = 385 is outside [1, 384]: the call reports an unsupported shape and launches nothing."""
    w = synth.weights(256, 128, synth.TINY, seed=61, device="cuda")
    t = w12.encode(w)
    x = synth.activations(385, 128, seed=62, device="cuda")
    with pytest.raises(w12.W12Error) as e:
        w12.gemm(t, x)
    assert "shape" in str(e.value).lower()
