"""The persistent cross-GEMM kernel of the layer stream (w12_stream_step) on the GPU.

- small layers (hidden 256, q 192, k|v 2 x 64, ffn 512), 3 layers, M in {1, 7, 32}: the step
  against the chain of separate launches (w12_rms_bf16, w12_gemm with its accumulate mode and
  strided input, w12_mul_bf16), and the last layer's intermediates (read from the workspace)
  against the oracle: x and x2 against the oracle's row normalisation of the GPU's own h, q|k|v,
  o, gate, up and down against the oracle's fp64 GEMMs of the GPU's own inputs, the gate-up
  product and the residual adds;
- the full 64-layer model (hidden 5120, q 6144, k|v 2 x 1024, ffn 17408) at M in {1, 16, 32}:
  the step against the chain of launches, the head's argmax of its output against the oracle,
  and the first and last layers' linears against the oracle on sampled outputs;
- rows wider than one normalisation unit holds (the multi-pass normalisation, ragged last tiles)
  against the chain and the oracle;
- repeated steps on one workspace give identical rows (its counters are left zeroed);
- the failure path: under the test-stall hook the bounded waits run out and are reported, and a
  step on the re-zeroed workspace is right;
- shapes the kernel does not take are refused on the host.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from lossless_bit_weight_gb300 import synth
from w12_testutil import REL, ABS, argmax_check, gemm_violations, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from lossless_bit_weight_gb300 import build, w12 as mod

    build.build()
    oracle.build()
    return mod


def make_layers(w12, L, H, nq, nkv, F, seed, keep=()):
    """L synthetic layers: encoded q|k|v, o, gate|up (concatenated for the chain, interleaved for
    the step) and down; the bf16 weights of the layers in `keep`."""
    chain, step, bf = [], [], {}
    for layer in range(L):
        s = seed + 100 * layer
        wqkv = synth.weights(nq + 2 * nkv, H, synth.PROJ, seed=s, device="cuda")
        wo = synth.weights(H, nq, synth.PROJ, seed=s + 1, device="cuda")
        wg = synth.weights(F, H, synth.PROJ, seed=s + 2, device="cuda")
        wu = synth.weights(F, H, synth.PROJ, seed=s + 3, device="cuda")
        wd = synth.weights(H, F, synth.PROJ, seed=s + 4, device="cuda")
        tqkv, to, td = w12.encode(wqkv), w12.encode(wo), w12.encode(wd)
        chain.append({"qkv": tqkv, "o": to, "gate_up": w12.encode(torch.cat([wg, wu])), "down": td})
        step.append({"qkv": tqkv, "o": to, "gate_up": w12.encode(w12.stream_interleave(wg, wu)), "down": td})
        if layer in keep:
            bf[layer] = {"qkv": wqkv, "o": wo, "gate": wg, "up": wu, "down": wd}
        del wqkv, wo, wg, wu, wd
    return chain, step, bf


def chain_step(w12, layers, h, nq, F):
    """The same step as a chain of separate launches (the reference the persistent kernel follows)."""
    for ly in layers:
        x = w12.rms_bf16(h)
        qkv = w12.gemm(ly["qkv"], x, out_dtype=torch.bfloat16)
        w12.gemm(ly["o"], qkv[:, :nq], out=h, accumulate=True)
        x2 = w12.rms_bf16(h)
        gu = w12.gemm(ly["gate_up"], x2)
        p = w12.mul_bf16(gu, F)
        w12.gemm(ly["down"], p, out=h, accumulate=True)
    return w12.rms_bf16(h)


def bf16_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_rms(x_gpu: torch.Tensor, h: torch.Tensor):
    """x = rms_bf16(h) against the oracle: one bf16 step where the two fp64 quotients straddle a
    rounding boundary, in at most 1 in 10,000 elements."""
    d = np.abs(to_np_u16(x_gpu).astype(np.int32) - oracle.rms_bf16(h.cpu().numpy()).astype(np.int32))
    assert d.max() <= 1
    assert np.count_nonzero(d) <= max(1, d.size // 10000)


def check_gate_up_product(p_gpu: torch.Tensor, x2: torch.Tensor, wg: torch.Tensor, wu: torch.Tensor):
    """p = bf16(g u) against the oracle's fp64 g and u of the GPU's own x2: the GEMM bound on each
    factor carried through the product, plus the bf16 rounding of the result."""
    g, adg = oracle.gemm(to_np_u16(x2), to_np_u16(wg))
    u, adu = oracle.gemm(to_np_u16(x2), to_np_u16(wu))
    tg, tu = REL * adg + ABS, REL * adu + ABS
    ref = g * u
    p = bf16_f64(to_np_u16(p_gpu))
    tol = np.abs(g) * tu + np.abs(u) * tg + tg * tu + np.abs(ref) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(p - ref) <= tol)


@pytest.mark.parametrize("M", [1, 7, 32])
def test_stream_small_matches_chain_and_oracle(w12, M):
    L, H, nq, nkv, F = 3, 256, 192, 64, 512
    chain, step_layers, bf = make_layers(w12, L, H, nq, nkv, F, seed=500 + M, keep=(L - 1,))
    h0 = synth.activations(M, H, seed=900 + M, device="cuda").float() * 4.0
    hc = h0.clone()
    xc = chain_step(w12, chain, hc, nq, F)
    step = w12.StreamStep(step_layers, M, nq)
    hs = h0.clone()
    xs = step(hs)
    step.check()
    # the chain and the step use the same work split, the same fp32 sums and the same roundings
    assert torch.equal(hs.view(torch.int32), hc.view(torch.int32))
    assert torch.equal(xs.view(torch.int16), xc.view(torch.int16))
    buf = {k: v.clone() for k, v in step.buffers().items()}
    # h entering the last layer: the step over the first L - 1 layers (deterministic)
    h_in = h0.clone()
    w12.StreamStep(step_layers[: L - 1], M, nq)(h_in)
    w = bf[L - 1]
    check_rms(buf["x"], h_in)
    y, ad = oracle.gemm(to_np_u16(buf["x"]), to_np_u16(w["qkv"]))
    assert gemm_violations(buf["qkv"].float().cpu().numpy(), y, ad, bf16=True) == 0
    a = buf["qkv"][:, :nq].contiguous()
    o = w12.gemm(step_layers[L - 1]["o"], a)
    yo, ado = oracle.gemm(to_np_u16(a), to_np_u16(w["o"]))
    assert gemm_violations(o.cpu().numpy(), yo, ado) == 0
    h_mid = h_in + o  # the accumulate mode is one fp32 addition per element
    check_rms(buf["x2"], h_mid)
    check_gate_up_product(buf["p"], buf["x2"], w["gate"], w["up"])
    d = w12.gemm(step_layers[L - 1]["down"], buf["p"])
    yd, add = oracle.gemm(to_np_u16(buf["p"]), to_np_u16(w["down"]))
    assert gemm_violations(d.cpu().numpy(), yd, add) == 0
    assert torch.equal(hs.view(torch.int32), (h_mid + d).view(torch.int32))
    check_rms(xs, hs)


@pytest.mark.parametrize("M", [1, 7])
def test_stream_wide_rows(w12, M):
    """Rows longer than one normalisation unit holds at once (hidden 5184 > 1280 16-byte words of
    128 threads x 10): the normalisation's multi-pass path and the o and down sums over a ragged
    last tile. With 81 k tiles the interleaved gate|up tensor splits its tiles' k ranges at other
    points than the chain's concatenated one, so the gate|up sums, p and h are checked against the
    oracle here; x, q|k|v and x2 against the chain bit for bit."""
    L, H, nq, nkv, F = 1, 5184, 192, 64, 512
    chain, step_layers, bf = make_layers(w12, L, H, nq, nkv, F, seed=700 + M, keep=(0,))
    h0 = synth.activations(M, H, seed=710 + M, device="cuda").float() * 3.0
    step = w12.StreamStep(step_layers, M, nq)
    hs = h0.clone()
    xs = step(hs)
    step.check()
    b = {k: v.clone() for k, v in step.buffers().items()}
    w = bf[0]
    x = w12.rms_bf16(h0)
    assert torch.equal(b["x"].view(torch.int16), x.view(torch.int16))
    check_rms(b["x"], h0)
    assert torch.equal(b["qkv"].view(torch.int16), w12.gemm(chain[0]["qkv"], x, out_dtype=torch.bfloat16).view(torch.int16))
    a = b["qkv"][:, :nq].contiguous()
    h_mid = h0 + w12.gemm(step_layers[0]["o"], a)
    assert torch.equal(b["x2"].view(torch.int16), w12.rms_bf16(h_mid).view(torch.int16))
    check_rms(b["x2"], h_mid)
    check_gate_up_product(b["p"], b["x2"], w["gate"], w["up"])
    d, ad = oracle.gemm(to_np_u16(b["p"]), to_np_u16(w["down"]))
    h_ref = h_mid.double().cpu().numpy() + d
    tol = REL * ad + ABS + np.abs(h_ref) * 2.0 ** -23
    assert np.all(np.abs(hs.double().cpu().numpy() - h_ref) <= tol)
    check_rms(xs, hs)


def test_stream_repeat_and_counters(w12):
    """Steps on one workspace, one after another, give identical rows: the kernel leaves its
    completion counters and split-tile counters zeroed."""
    chain, step_layers, _ = make_layers(w12, 2, 256, 192, 64, 512, seed=77)
    step = w12.StreamStep(step_layers, 16, 192)
    h0 = synth.activations(16, 256, seed=78, device="cuda").float()
    outs = []
    for _ in range(3):
        h = h0.clone()
        x = step(h)
        outs.append((h, x))
    step.check()
    for h, x in outs[1:]:
        assert torch.equal(h.view(torch.int32), outs[0][0].view(torch.int32))
        assert torch.equal(x.view(torch.int16), outs[0][1].view(torch.int16))
    ws = step.ws.cpu().numpy()
    assert not ws[:4].any()  # the error word


def test_stream_timeout_is_reported(w12):
    """The failure path of the persistent kernel, without a GPU fault: under the
    W12_LAUNCH_TEST_STALL hook each block's activation producer issues its first slot's copies
    only, the MMAs' wait on the next slot gives up after about a second, every block stops (the
    other blocks' waits on the phase counters run out too), and w12_check reports W12_ERR_TIMEOUT.
    The context stays usable: once the workspace is zero-filled again, a step gives the rows of
    the chain of separate launches."""
    chain, step_layers, _ = make_layers(w12, 2, 256, 192, 64, 512, seed=91)
    step = w12.StreamStep(step_layers, 8, 192)
    h0 = synth.activations(8, 256, seed=92, device="cuda").float()
    h = h0.clone()
    step(h, test_stall=True)
    with pytest.raises(w12.W12Error) as e:
        step.check()
    assert e.value.status == w12.ERR_TIMEOUT
    step.ws.zero_()
    h = h0.clone()
    x = step(h)
    step.check()
    hc = h0.clone()
    xc = chain_step(w12, chain, hc, 192, 512)
    assert torch.equal(h.view(torch.int32), hc.view(torch.int32))
    assert torch.equal(x.view(torch.int16), xc.view(torch.int16))
    L = w12.lib()
    assert L.w12_stream_step_ex(step.arr, step.n, step.M, step.n_q, w12._ptr(h), w12._ptr(x), w12._ptr(step.ws),
                                step.ws_bytes, 8, None) == w12.ERR_INVALID_ARG  # an unknown flag


def test_stream_refuses_shapes(w12):
    _, layers, _ = make_layers(w12, 1, 256, 192, 64, 512, seed=81)
    L = w12.lib()
    arr = (w12.CStreamLayer * 1)()
    arr[0] = w12.CStreamLayer(layers[0]["qkv"].c, layers[0]["o"].c, layers[0]["gate_up"].c, layers[0]["down"].c)
    nb = ctypes.c_size_t()
    assert L.w12_stream_workspace_size(arr, 1, 33, 192, ctypes.byref(nb)) == w12.ERR_UNSUPPORTED_SHAPE
    assert L.w12_stream_workspace_size(arr, 1, 8, 128, ctypes.byref(nb)) == w12.ERR_INVALID_ARG  # o.K != n_q
    assert L.w12_stream_workspace_size(arr, 0, 8, 192, ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    assert L.w12_stream_workspace_size(arr, 1, 8, 192, ctypes.byref(nb)) == w12.OK
    # layers of different shapes
    _, other, _ = make_layers(w12, 1, 256, 128, 64, 512, seed=82)
    arr2 = (w12.CStreamLayer * 2)()
    arr2[0] = arr[0]
    arr2[1] = w12.CStreamLayer(other[0]["qkv"].c, other[0]["o"].c, other[0]["gate_up"].c, other[0]["down"].c)
    assert L.w12_stream_workspace_size(arr2, 2, 8, 192, ctypes.byref(nb)) == w12.ERR_INVALID_ARG


def _check_linear_sampled(t_in, w, y, rng, n_samples=256):
    M, N = y.shape
    ms = rng.integers(0, M, n_samples)
    ns = rng.integers(0, N, n_samples)
    y_ref, ad = oracle.gemm_sampled(to_np_u16(t_in), to_np_u16(w), ms, ns)
    got = y.float().cpu().numpy()[ms, ns]
    assert gemm_violations(got, y_ref, ad, bf16=(y.dtype == torch.bfloat16)) == 0


def test_stream_full_model(w12):
    """The 64-layer model workload in one persistent launch per step, at M in {1, 16, 32}."""
    H, nq, nkv, F, L = synth.HIDDEN, 6144, 1024, synth.MLP, 64
    keep = (0, L - 1)
    chain, step_layers, bf = make_layers(w12, L, H, nq, nkv, F, seed=synth.seed_for(3, 0), keep=keep)
    wh = synth.weights(synth.VOCAB, H, synth.HEAD, seed=synth.seed_for(2, 0), device="cuda")
    th = w12.encode(wh)
    rng = np.random.default_rng(11)
    for M in (1, 16, 32):
        h0 = synth.activations(M, H, seed=synth.seed_for(3, M), device="cuda").float()
        hc = h0.clone()
        xc = chain_step(w12, chain, hc, nq, F)
        step = w12.StreamStep(step_layers, M, nq)
        hs = h0.clone()
        xs = step(hs)
        step.check()
        assert torch.equal(hs.view(torch.int32), hc.view(torch.int32))
        assert torch.equal(xs.view(torch.int16), xc.view(torch.int16))
        idx, val, gap = w12.lmhead_argmax(th, xs)
        y_ref, ad = oracle.gemm(to_np_u16(xs), to_np_u16(wh))
        checked, near, wrong, det = argmax_check(idx.cpu().numpy(), val.cpu().numpy(), gap.cpu().numpy(), y_ref, ad)
        assert wrong == 0, det
        # the first and the last layer's linears against the oracle on the GPU's own inputs
        for layer in keep:
            h_in = h0.clone()
            if layer > 0:
                w12.StreamStep(step_layers[:layer], M, nq)(h_in)
            one = w12.StreamStep(step_layers[layer: layer + 1], M, nq)
            h_out = h_in.clone()
            one(h_out)
            b = one.buffers()
            w = bf[layer]
            check_rms(b["x"], h_in)
            _check_linear_sampled(b["x"], w["qkv"], b["qkv"], rng)
            a = b["qkv"][:, :nq].contiguous()
            o = w12.gemm(step_layers[layer]["o"], a)
            _check_linear_sampled(a, w["o"], o, rng)
            h_mid = h_in + o
            check_rms(b["x2"], h_mid)
            g = w12.gemm(chain[layer]["gate_up"], b["x2"])
            _check_linear_sampled(b["x2"], torch.cat([w["gate"], w["up"]]), g, rng)
            ref_p = oracle.mul_bf16(g[:, :F].cpu().numpy(), g[:, F:].cpu().numpy())
            assert np.array_equal(to_np_u16(b["p"]), ref_p)
            d = w12.gemm(step_layers[layer]["down"], b["p"])
            _check_linear_sampled(b["p"], w["down"], d, rng)
            assert torch.equal(h_out.view(torch.int32), (h_mid + d).view(torch.int32))
    w12.check(th)
