"""CPU pins of the W12 oracle against facts that do not come from the oracle itself.

- the lossless invariant: decode(encode(W)) == W bit for bit (SpecPilot §4.1; Table A2 caption),
  over all 65,536 bf16 patterns and over synthetic tensors;
- the window rule against a brute-force count over every candidate base (SpecPilot §4.1);
- the escape set against its definition, evaluated with float arithmetic on the values;
- hand-derived bytes of a small ragged tensor (tests/golden/w12_layout_fixture.txt);
- the fp64 GEMM against exact rational sums; the argmax against Python's own max over rows;
- the Q view (SpecPilot §4.3) against value-level properties and against a second route through
  the encoded records;
- the certified LM head (SpecPilot §4.1): quantisation properties of the INT8 copy, the
  Cauchy-Schwarz bound against the exact GEMM, and the certified argmax against the brute-force
  argmax over the whole head (random heads, exact ties, Inf rows);
- the INT6 Q-pass copy (SpecPilot §5.3, App. C): quantisation properties, hand-derived record
  bytes, a record reader written from the bit layout, and the lossless case of its GEMM against
  the exact GEMM;
- the glue of the synthetic layer stream: bf16 rounding from fp64, the row normalisation's
  special cases and invariances, the gate-up product against numpy's fp32 multiply.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from lossless_bit_weight_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_values(u16: np.ndarray) -> np.ndarray:
    """Exact float64 values of bf16 patterns via numpy's float32 (independent of the oracle)."""
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- lossless round trip


def test_roundtrip_all_65536_patterns(orc):
    w = synth.all_bf16_patterns(256)  # 256 channels, each a contiguous run of 256 patterns
    e = orc.encode(w)
    assert np.array_equal(orc.decode(e), w)
    assert np.array_equal(orc.decode_csr(e), w)


def test_roundtrip_all_patterns_shuffled_rows(orc):
    rng = np.random.default_rng(7)
    w = synth.all_bf16_patterns(512).reshape(-1)
    w = rng.permutation(w).reshape(128, 512)  # every channel mixes NaN, Inf, ±0, subnormals
    e = orc.encode(w)
    assert np.array_equal(orc.decode(e), w)
    assert np.array_equal(orc.decode_csr(e), w)


@pytest.mark.parametrize("N,K", [(512, 256), (300, 200), (1, 8), (129, 65)])
def test_roundtrip_synthetic(orc, N, K):
    w = synth.bits(synth.weights(N, K, synth.TINY, seed=11 + N + K))
    e = orc.encode(w)
    assert np.array_equal(orc.decode(e), w)
    assert np.array_equal(orc.decode_csr(e), w)


# ---------------------------------------------------------------- window rule


def brute_force_window(vals: np.ndarray) -> int:
    """Largest coverage by direct counting over E in [16, 254]; ties -> smallest E.

    Works on values: a weight is normal when 2^-126 <= |v| < inf, its binade is floor(log2|v|)."""
    a = np.abs(vals)
    normal = np.isfinite(a) & (a >= 2.0 ** -126)
    binade = np.floor(np.log2(a[normal])).astype(np.int64) + 127  # biased exponent
    best_E, best = None, -1
    for E in range(16, 255):
        c = int(np.count_nonzero((binade >= E - 15) & (binade <= E)))
        if c > best:
            best, best_E = c, E
    return best_E


def test_window_vs_brute_force(orc):
    rng = np.random.default_rng(3)
    rows = [synth.bits(synth.weights(4, 512, synth.TINY, seed=s)) for s in range(3)]
    rows = [r for blk in rows for r in blk]
    # wide spreads so the window really has to choose
    for _ in range(12):
        ex = rng.integers(60, 200, size=300)
        v = np.ldexp(rng.uniform(1, 2, size=300), ex - 127) * rng.choice([-1, 1], size=300)
        rows.append(synth.bits(torch.tensor(v, dtype=torch.float32).to(torch.bfloat16)))
    rows.append(np.zeros(64, np.uint16))                       # no normal weight at all
    rows.append(np.full(64, 0x7FC0, np.uint16))                # all NaN
    rows.append(np.full(64, 0x0001, np.uint16))                # all subnormal
    rows.append(np.array([0x0080] * 10 + [0x7F7F] * 10, np.uint16))  # extreme binades, a tie
    for r in rows:
        assert orc.window(r) == brute_force_window(bf16_values(r)), r[:8]


def test_window_ties_take_smallest_base(orc):
    # all weights in binade 127: every E in [127, 142] covers them all -> E_n = 127
    assert orc.window(np.full(16, 0x3F80, np.uint16)) == 127
    # two equal groups 20 binades apart: both windows cover 8; the lower one wins
    row = np.array([0x3F80] * 8 + [0x4980] * 8, np.uint16)  # e=127 and e=147
    assert orc.window(row) == 127


# ---------------------------------------------------------------- escapes


def test_escape_set_matches_definition(orc):
    w = synth.bits(synth.weights(256, 320, synth.TINY, seed=5))
    w[3, :] = 0                      # an all-zero channel
    w[4, 10] = 0x7F80                # +Inf
    w[5, 11] = 0xFFC1                # NaN with payload and sign
    w[6, 12] = 0x0003                # subnormal
    e = orc.encode(w)
    vals = bf16_values(w)
    n_expected = 0
    for n in range(w.shape[0]):
        En = int(e.base_exp[n])
        a = np.abs(vals[n])
        with np.errstate(divide="ignore", invalid="ignore"):
            binade = np.floor(np.log2(a)) + 127
        inside = np.isfinite(a) & (a >= 2.0 ** -126) & (binade >= En - 15) & (binade <= En)
        ks = np.nonzero(~inside)[0]
        lo, hi = int(e.esc_off[n]), int(e.esc_off[n + 1])
        assert np.array_equal(e.esc_k[lo:hi], ks)
        assert np.array_equal(e.esc_bits[lo:hi], w[n, ks])
        n_expected += ks.size
    assert e.esc_k.size == n_expected
    assert int(e.base_exp[3]) == 16  # no normal weight: every window covers 0 -> smallest base


def test_per_record_index_is_a_regrouping_of_the_csr(orc):
    w = synth.bits(synth.weights(300, 200, synth.TINY, seed=9))
    w[130:200, 70:100] = 0  # escapes in several 32-row quarters of a record
    e = orc.encode(w)
    from_csr = set()
    for n in range(e.N):
        for i in range(e.esc_off[n], e.esc_off[n + 1]):
            from_csr.add((n, int(e.esc_k[i]), int(e.esc_bits[i])))
    from_rec = set()
    R = e.n_tiles * e.k_tiles
    for r in range(R):
        nt, kt = divmod(r, e.k_tiles)
        seg = e.rec_esc[e.rec_esc_off[r]:e.rec_esc_off[r + 1]]
        assert seg.size % 4 == 0
        if seg.size == 0:
            continue
        header, body = seg[:4], seg[4:]
        real = body[body != 0xFFFFFFFF]
        assert real.size > 0 and int(header[3]) == real.size
        pos = real & 0xFFFF
        assert np.all(np.diff(pos.astype(np.int64)) > 0)
        quarter = (pos >> 11).astype(np.int64)
        for q in range(4):
            assert int(header[q]) == int(np.count_nonzero(quarter <= q))
        for ent in real:
            p = int(ent) & 0xFFFF
            from_rec.add((nt * 128 + p // 64, kt * 64 + p % 64, int(ent) >> 16))
    assert from_csr == from_rec


# ---------------------------------------------------------------- golden bytes


def _parse_fixture(path):
    lines = []
    with open(path) as f:
        for ln in f:
            ln = ln.split("#", 1)[0].strip()
            if ln:
                lines.append(ln.split())
    return lines


def test_golden_layout_fixture(orc):
    lines = _parse_fixture(os.path.join(GOLDEN, "w12_layout_fixture.txt"))
    w = None
    for t in lines:
        if t[0] == "shape":
            w = np.zeros((int(t[1]), int(t[2])), np.uint16)
        elif t[0] == "fill":
            w[:] = int(t[1], 16)
        elif t[0] == "row":
            w[int(t[1]), :] = int(t[2], 16)
        elif t[0] == "set":
            w[int(t[1]), int(t[2])] = int(t[3], 16)
    e = orc.encode(w)
    rec = e.records.reshape(-1, orc.RECORD_BYTES)
    checked = 0
    for t in lines:
        k = t[0]
        if k == "expect":
            what, a = t[1], t[2:]
            if what == "base_exp":
                assert e.base_exp[int(a[0])] == int(a[1]), t
            elif what == "view":
                assert rec[int(a[0]), int(a[1])] == int(a[2], 16), t
            elif what == "bnib":
                off = int(a[1])
                word = int.from_bytes(bytes(rec[int(a[0]), off:off + 4]), "little")
                assert (word >> (4 * int(a[2]))) & 0xF == int(a[3], 16), t
            elif what == "n_esc":
                assert e.esc_k.size == int(a[0]), t
            elif what == "esc_off":
                assert e.esc_off[int(a[0])] == int(a[1]), t
            elif what == "csr":
                i = int(a[0])
                assert (e.esc_k[i], e.esc_bits[i]) == (int(a[1]), int(a[2], 16)), t
            elif what == "rec_esc_off":
                assert list(e.rec_esc_off) == [int(v) for v in a], t
            elif what == "rec_entry":
                assert e.rec_esc[int(a[0])] == int(a[1], 16), t
            else:
                raise AssertionError(t)
            checked += 1
    assert checked > 50
    assert np.array_equal(orc.decode(e), w)


# ---------------------------------------------------------------- GEMM


def _exact_dot(xr, wr):
    s = Fraction(0)
    for a, b in zip(xr, wr):
        s += Fraction(float(a)) * Fraction(float(b))
    return s


def test_gemm_vs_exact_rational(orc):
    rng = np.random.default_rng(1)
    M, N, K = 3, 5, 37
    x = synth.bits(torch.tensor(rng.standard_normal((M, K)), dtype=torch.float32).to(torch.bfloat16))
    w = synth.bits(synth.weights(N, K, synth.TINY, seed=2))
    w[0, 0] = 0x7F7F            # largest finite bf16
    w[1, :4] = [0x0001, 0x8001, 0x0080, 0x0000]  # subnormals, smallest normal, zero
    x[2, :] = x[1, ::-1]        # a row with a different summation profile
    y, a = orc.gemm(x, w)
    xv, wv = bf16_values(x), bf16_values(w)
    for m in range(M):
        for n in range(N):
            exact = _exact_dot(xv[m], wv[n])
            absexact = sum(abs(Fraction(float(p))) for p in xv[m] * wv[n])
            # K sequential fp64 additions of exact products: |err| <= K * 2^-53 * sum|p|
            assert abs(Fraction(y[m, n]) - exact) <= K * Fraction(1, 2 ** 53) * absexact
            assert a[m, n] == pytest.approx(float(absexact), rel=1e-12)


def test_gemm_sampled_matches_full(orc):
    x = synth.bits(synth.activations(4, 96, seed=4))
    w = synth.bits(synth.weights(40, 96, synth.TINY, seed=4))
    y, a = orc.gemm(x, w)
    ms = np.array([0, 3, 2, 1, 3], np.int32)
    ns = np.array([0, 39, 17, 5, 5], np.int32)
    ys, as_ = orc.gemm_sampled(x, w, ms, ns)
    assert np.array_equal(ys, y[ms, ns]) and np.array_equal(as_, a[ms, ns])


# ---------------------------------------------------------------- argmax


def test_argmax_vs_python_max(orc):
    rng = np.random.default_rng(8)
    y = rng.standard_normal((6, 50))
    y[1, 7] = y[1, 30] = 9.0          # exact tie for the maximum -> index 7, gap 0
    y[2, :] = -1.0                    # constant row
    y[3, 49] = 100.0                  # maximum at the end
    y[4, :] = -np.abs(y[4, :])        # all negative
    idx, val, gap, sc = orc.argmax(y)
    for m in range(y.shape[0]):
        row = list(y[m])
        best = max(range(len(row)), key=lambda n: (row[n], -n))
        rest = [row[n] for n in range(len(row)) if n != best]
        assert idx[m] == best
        assert val[m] == row[best]
        assert gap[m] == row[best] - max(rest)
        assert sc[m] == max(abs(v) for v in row)
    assert idx[1] == 7 and gap[1] == 0.0
    one = orc.argmax(np.array([[3.5]]))
    assert one[0][0] == 0 and math.isinf(one[2][0])


# ---------------------------------------------------------------- Q view


def test_qview_value_properties(orc):
    w = synth.bits(synth.weights(256, 256, synth.TINY, seed=12))
    wq = orc.qview_weights(w)
    e = orc.encode(w)
    v, vq = bf16_values(w), bf16_values(wq)
    for n in range(w.shape[0]):
        En = int(e.base_exp[n])
        lo_b, hi_b = 2.0 ** (En - 15 - 127), 2.0 ** (En - 127 + 1)
        a = np.abs(v[n])
        inside = (a >= lo_b) & (a < hi_b) & (a >= 2.0 ** -126)
        # in-window weights: same sign, same binade, |wq - w| <= half of the dropped 4-bit range
        assert np.all(np.sign(vq[n][inside]) == np.sign(v[n][inside]))
        bq = np.floor(np.log2(np.abs(vq[n][inside])))
        assert np.array_equal(bq, np.floor(np.log2(a[inside])))
        ulp7 = 2.0 ** (bq - 7)  # one unit of the 7-bit mantissa; the low 4 bits span 16 units
        assert np.all(np.abs(vq[n][inside] - v[n][inside]) <= 8 * ulp7)
        # every Q-view weight is a normal number inside the channel's window
        aq = np.abs(vq[n])
        assert np.all((aq >= lo_b) & (aq < hi_b))


def test_qview_equals_decode_of_truncated_records(orc):
    """Second route: set every B nibble of the encoded records to 8, drop the escapes, decode."""
    w = synth.bits(synth.weights(200, 136, synth.TINY, seed=13))
    e = orc.encode(w)
    rec = e.records.reshape(-1, orc.RECORD_BYTES).copy()
    rec[:, 8192:] = 0x88
    e2 = orc.Encoded(e.N, e.K, rec.reshape(-1), e.base_exp, e.esc_off, e.esc_k[:0],
                     e.esc_bits[:0], np.zeros_like(e.rec_esc_off), e.rec_esc[:0])
    assert np.array_equal(orc.decode(e2), orc.qview_weights(w))


# ---------------------------------------------------------------- certified LM head (SpecPilot §4.1)


def _head(N, K, seed):
    return synth.weights(N, K, synth.HEAD, seed=seed).view(torch.int16).numpy().view(np.uint16)


def test_head_q8_quantisation_properties(orc):
    """Codes lie in [-127, 127]; the largest |w| of a row codes to +-127; every in-range weight
    is within half a step of its code; the scale is the row maximum over 127 in fp32; zero rows
    and rows holding Inf/NaN get scale 0 (the latter with an infinite residual)."""
    w = _head(64, 96, seed=4)
    w[3] = 0                      # all-zero row
    w[5, 7] = 0x7F80              # +Inf
    w[6, 9] = 0x7FC1              # NaN
    w[7, :] = 0x3F80              # all 1.0
    h = orc.head_q8(w)
    v = bf16_values(w)
    assert np.all(np.abs(h.q.astype(np.int32)) <= 127)
    for n in range(64):
        if n in (5, 6):
            assert h.scale[n] == 0 and math.isinf(h.resid[n]) and not np.any(h.q[n])
            continue
        amax = np.abs(v[n]).max()
        if amax == 0:
            assert h.scale[n] == 0 and h.resid[n] == 0 and not np.any(h.q[n])
            continue
        assert h.scale[n] == np.float32(amax / 127.0)
        s = float(h.scale[n])
        e = v[n] - s * h.q[n].astype(np.float64)
        assert np.all(np.abs(e) <= s / 2 * (1 + 1e-12) + abs(amax - 127 * s))
        k = int(np.argmax(np.abs(v[n])))
        assert abs(int(h.q[n, k])) == 127
        assert h.resid[n] == pytest.approx(float(np.sqrt(np.sum(e * e))), rel=1e-12, abs=1e-300)
    # all 1.0: every code is 127 and the residual is the fp32 scale's own rounding error
    s7 = float(h.scale[7])
    assert np.all(h.q[7] == 127) and h.resid[7] == pytest.approx(math.sqrt(96) * abs(1 - 127 * s7), rel=1e-9)


def test_certified_bound_holds(orc):
    """|y - yh| <= ||x|| c_n for every logit: the exact fp64 GEMM on one side, s_n (x . q_n) on
    the other (numpy), the residual norm from the oracle."""
    w = _head(500, 256, seed=8)
    x = synth.activations(6, 256, seed=9).view(torch.int16).numpy().view(np.uint16)
    h = orc.head_q8(w)
    y, _ = orc.gemm(x, w)
    xv = bf16_values(x)
    yh = (xv @ h.q.astype(np.float64).T) * h.scale.astype(np.float64)[None, :]
    bound = np.linalg.norm(xv, axis=1)[:, None] * h.resid[None, :]
    assert np.all(np.abs(y - yh) <= bound * (1 + 1e-9))
    # and it is not vacuous: on these Gaussian rows it is under a tenth of the logits' spread
    assert np.median(bound) < 0.1 * np.std(y) * math.sqrt(256)


@pytest.mark.parametrize("N,K,M,seed", [(3000, 256, 8, 1), (2000, 192, 5, 2), (1, 64, 3, 3), (2, 64, 2, 4)])
def test_certified_argmax_equals_full_argmax(orc, N, K, M, seed):
    """The survivors always hold the exact top-1 and top-2, so the certified result equals the
    argmax and gap over the whole head (brute force over the fp64 GEMM)."""
    w = _head(N, K, seed=seed)
    x = synth.activations(M, K, seed=seed + 50).view(torch.int16).numpy().view(np.uint16)
    h = orc.head_q8(w)
    idx, val, gap, cnt = orc.certified_argmax(x, w, h)
    y, _ = orc.gemm(x, w)
    ridx, rval, rgap, _ = orc.argmax(y)
    assert np.array_equal(idx, ridx)
    assert np.array_equal(val, rval)
    if N > 1:
        assert np.array_equal(gap, rgap)
    assert np.all(cnt >= min(N, 2)) and np.all(cnt <= N)
    if N >= 1000:
        assert np.all(cnt < N // 10)  # the bound discards most of a Gaussian head


def test_certified_argmax_ties_and_special_rows(orc):
    """Duplicate rows tie exactly (the smaller index wins, gap 0); a row with +Inf wins where its
    logit is +Inf; an all-zero row is an ordinary candidate."""
    w = _head(400, 128, seed=11)
    w[17] = w[250]                 # exact duplicates
    w[30] = 0
    w[99, 5] = 0x7F80              # +Inf weight
    x = synth.activations(4, 128, seed=12).view(torch.int16).numpy().view(np.uint16)
    xv = bf16_values(x)
    # make row 250 (and 17) the winner of row 0 by aligning it with x[0]
    w[250] = np.where(xv[0] > 0, 0x3C00, 0xBC00).astype(np.uint16)  # +-2^-7
    w[17] = w[250]
    h = orc.head_q8(w)
    idx, val, gap, cnt = orc.certified_argmax(x, w, h)
    y, _ = orc.gemm(x, w)
    ridx, rval, rgap, _ = orc.argmax(y)
    assert idx[0] == 17 and gap[0] == 0.0
    for m in range(4):
        if math.isinf(rval[m]):
            assert idx[m] == 99 and val[m] == rval[m]
        else:
            assert idx[m] == ridx[m] and val[m] == rval[m] and gap[m] == rgap[m]


# ---------------------------------------------------------------- INT6 Q-pass copy

def test_copy_q6_quantisation_properties(orc):
    """Codes lie in [-31, 31]; the largest |w| of a row codes to +-31; every weight is within half
    a step of its code; the scale is the row maximum over 31 in fp32; zero rows and rows holding
    Inf/NaN get scale 0 and code 0."""
    w = _head(64, 96, seed=14)
    w[3] = 0                      # all-zero row
    w[5, 7] = 0x7F80              # +Inf
    w[6, 9] = 0x7FC1              # NaN
    w[7, :] = 0x3F80              # all 1.0
    c = orc.copy_q6(w)
    v = bf16_values(w)
    assert np.all(np.abs(c.q.astype(np.int32)) <= 31)
    for n in range(64):
        amax = np.abs(v[n]).max() if n not in (5, 6) else np.inf
        if n in (3, 5, 6):
            assert c.scale[n] == 0 and not np.any(c.q[n])
            continue
        assert c.scale[n] == np.float32(amax / 31.0)
        s = float(c.scale[n])
        e = v[n] - s * c.q[n].astype(np.float64)
        assert np.all(np.abs(e) <= s / 2 * (1 + 1e-12) + abs(amax - 31 * s))
        assert abs(int(c.q[n, int(np.argmax(np.abs(v[n])))])) == 31
    # ties go to the even code: a row whose maximum is 7.75 = 31 * 2^-2 has scale 2^-2
    row = np.zeros((1, 64), np.uint16)
    row[0, 0] = 0x40F8            # 7.75 -> 31
    row[0, 1] = 0x3F20            # 0.625 = 2.5 * 2^-2 -> 2
    row[0, 2] = 0x3F60            # 0.875 = 3.5 * 2^-2 -> 4
    row[0, 3] = 0xBFB0            # -1.375 = -5.5 * 2^-2 -> -6
    row[0, 4] = 0x3FE0            # 1.75 = 7 * 2^-2 -> 7
    c = orc.copy_q6(row)
    assert c.scale[0] == 0.25 and list(c.q[0, :5]) == [31, 2, 4, -6, 7]


def _q6_read_records(rec, N, K):
    """Codes [N, K] read back from INT6 records by the stated bit layout (independent of the
    oracle's packer): per 128-row, 64-column tile a 6144-byte record; per local row twelve 32-bit
    little-endian words, eight of low nibbles (words 0-3 at byte 16 n_l, words 4-7 at 2048 +
    16 n_l) and four of top bit pairs (at 4096 + 16 n_l); k_l = 16 g + 2 j + h."""
    nt, kt = (N + 127) // 128, (K + 63) // 64
    out = np.zeros((nt * 128, kt * 64), dtype=np.int16)
    b = rec.reshape(nt * kt, 6144)
    for r in range(nt * kt):
        t, k0 = divmod(r, kt)
        lo = np.concatenate([b[r, :2048].reshape(128, 16), b[r, 2048:4096].reshape(128, 16)], axis=1)
        lo = lo.view("<u4")                                   # [128, 8]
        hi = b[r, 4096:].reshape(128, 16).view("<u4")         # [128, 4]
        for kl in range(64):
            g, j, h = kl >> 4, (kl & 15) >> 1, kl & 1
            low = (lo[:, 2 * g + (j >> 2)] >> (4 * (j & 3) + 16 * h)) & 15
            top = (hi[:, g] >> (2 * j + 16 * h)) & 3
            out[t * 128:(t + 1) * 128, k0 * 64 + kl] = (low | (top << 4)).astype(np.int16) - 32
    return out


def test_q6_records_hand_fixture(orc):
    """One record whose only nonzero code is c = -3 at n_l = 5, k_l = 37. Every other position
    holds u = 32 (low nibble 0, top bits 10b): plane L is zero and every plane-T word is
    0xAAAAAAAA. u = 29 = 01 1101b; k_l = 37 is g 2, j 2, h 1: its low nibble 0xD goes to L word
    4 of row 5 (byte 2048 + 80), bits 24-27, i.e. byte 2131 = 0x0D; its top bits 01 go to T word
    2 of row 5 (byte 4096 + 80 + 8 = 4184), bits 20-21: the word becomes 0xAA9AAAAA, i.e. byte
    4186 = 0x9A."""
    q = np.zeros((128, 64), dtype=np.int8)
    q[5, 37] = -3
    rec = orc.q6_pack(q)
    want = np.zeros(6144, dtype=np.uint8)
    want[4096:] = 0xAA
    want[2131] = 0x0D
    want[4186] = 0x9A
    assert np.array_equal(rec, want)


@pytest.mark.parametrize("N,K", [(128, 64), (300, 200), (129, 8)])
def test_q6_records_round_trip(orc, N, K):
    """Random codes in [-31, 31] read back unchanged from the records, and padding holds code 0."""
    rng = np.random.default_rng(N + K)
    q = rng.integers(-31, 32, size=(N, K)).astype(np.int8)
    back = _q6_read_records(orc.q6_pack(q), N, K)
    assert np.array_equal(back[:N, :K], q)
    assert not np.any(back[N:]) and not np.any(back[:, K:])


def test_gemm_q6_lossless_case_is_the_exact_gemm(orc):
    """Rows whose weights are integers times 2^-e with a maximum of 31 * 2^-e quantise without
    loss (scale 2^-e, codes the integers), so the Q6 GEMM equals the exact fp64 GEMM bit for bit
    (scaling by a power of two commutes with every rounding)."""
    rng = np.random.default_rng(21)
    N, K, M = 40, 128, 5
    ints = rng.integers(-31, 32, size=(N, K))
    ints[:, 0] = 31
    e = rng.integers(2, 12, size=N)
    wv = (ints * (2.0 ** -e)[:, None]).astype(np.float32)
    w = (wv.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(bf16_values(w), wv.astype(np.float64))
    x = synth.activations(M, K, seed=22).view(torch.int16).numpy().view(np.uint16)
    c = orc.copy_q6(w)
    assert np.array_equal(c.scale.astype(np.float64), 2.0 ** -e)
    assert np.array_equal(c.q, ints.astype(np.int8))
    y, _ = orc.gemm(x, w)
    yq, adq = orc.gemm_q6(x, c)
    assert np.array_equal(yq, y)
    assert np.array_equal(adq, np.abs(bf16_values(x)) @ np.abs(wv.astype(np.float64)).T)


def test_gemm_q8_lossless_case_and_brute_force(orc):
    """The INT8 Q pass: rows whose weights are integers times 2^-e with a maximum of 127 * 2^-e
    quantise without loss (scale 2^-e, codes the integers), so its logits equal the exact fp64
    GEMM bit for bit; on an ordinary tiny head each logit equals s_n times the brute-force sum of
    x_k q_nk, written out with Python integers and fractions."""
    from fractions import Fraction

    rng = np.random.default_rng(23)
    N, K, M = 24, 192, 3
    ints = rng.integers(-127, 128, size=(N, K))
    ints[:, 5] = -127
    e = rng.integers(2, 10, size=N)
    wv = (ints * (2.0 ** -e)[:, None]).astype(np.float32)
    w = (wv.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(bf16_values(w), wv.astype(np.float64))
    x = synth.activations(M, K, seed=24).view(torch.int16).numpy().view(np.uint16)
    h = orc.head_q8(w)
    assert np.array_equal(h.scale.astype(np.float64), 2.0 ** -e)
    assert np.array_equal(h.q.astype(np.int64), ints)
    y, _ = orc.gemm(x, w)
    yq, adq = orc.gemm_q8(x, h)
    assert np.array_equal(yq, y)
    assert np.array_equal(adq, np.abs(bf16_values(x)) @ np.abs(wv.astype(np.float64)).T)
    # an ordinary head: compare with exact rational sums (the fp64 sum of at most 64 products of
    # a bf16 value and a 7-bit integer is exact, so equality is exact too)
    w2 = synth.weights(16, 64, synth.HEAD, seed=25).view(torch.int16).numpy().view(np.uint16)
    x2 = synth.activations(2, 64, seed=26).view(torch.int16).numpy().view(np.uint16)
    h2 = orc.head_q8(w2)
    yq2, _ = orc.gemm_q8(x2, h2)
    xv = bf16_values(x2)
    for m in range(2):
        for n in range(16):
            acc = sum(Fraction(float(xv[m, k])) * int(h2.q[n, k]) for k in range(64))
            assert yq2[m, n] == float(Fraction(float(h2.scale[n])) * acc)


# ---------------------------------------------------------------- glue of the synthetic layer stream

def _bf16_rne_from_f32(f: np.ndarray) -> np.ndarray:
    """bf16 bits of float32 values, round to nearest even (finite inputs), by integer arithmetic."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_double_to_bf16_rounding(orc):
    """Ties to even at both parities, the subnormal quantum 2^-133, overflow to Inf, and
    agreement with integer rounding of fp32 values (exact in fp64)."""
    assert orc.double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80            # tie, even below
    assert orc.double_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82        # tie, even above
    assert orc.double_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert orc.double_to_bf16(-27.4 * 2.0 ** -133) == 0x801B        # subnormal
    assert orc.double_to_bf16(2.0 ** -135) == 0x0000                # below half the quantum
    assert orc.double_to_bf16(3.3895e38) == 0x7F7F and orc.double_to_bf16(3.3962e38) == 0x7F80
    rng = np.random.default_rng(5)
    f = (rng.standard_normal(4000) * np.exp(rng.uniform(-60, 60, 4000))).astype(np.float32)
    want = _bf16_rne_from_f32(f)
    got = np.array([orc.double_to_bf16(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_rms_bf16_properties(orc):
    """Constant rows give +-1; a zero row gives zeros; scaling a row by a power of two changes
    nothing (fp64 rounding commutes with it); on random rows the result is within one bf16 ulp
    of numpy's fp64 h / sqrt(mean h^2) and the row's mean square is 1 within bf16 precision."""
    rng = np.random.default_rng(6)
    h = (rng.standard_normal((6, 640)) * 3).astype(np.float32)
    h[1] = 2.5
    h[2] = -0.75
    h[3] = 0.0
    x = orc.rms_bf16(h)
    assert np.all(x[1] == 0x3F80) and np.all(x[2] == 0xBF80) and np.all(x[3] == 0)
    assert np.array_equal(orc.rms_bf16(h * np.float32(2.0 ** 40)), x)
    assert np.array_equal(orc.rms_bf16(h * np.float32(2.0 ** -30)), x)
    v = h.astype(np.float64)
    with np.errstate(invalid="ignore"):
        ref = v / np.sqrt(np.mean(v * v, axis=1, keepdims=True))
    got = bf16_values(x)
    ok = np.isfinite(ref)
    ulp = np.exp2(np.floor(np.log2(np.abs(np.where(ref == 0, 1, ref)))) - 7)
    assert np.all(np.abs(got[ok] - ref[ok]) <= ulp[ok] / 2 * (1 + 1e-9))
    ms = np.mean(got[[0, 4, 5]] ** 2, axis=1)
    assert np.all(np.abs(ms - 1) < 2 ** -7)


def test_mul_bf16_is_rounded_fp32_product(orc):
    """p = bf16(fp32(g u)): against numpy's fp32 multiply and an integer round-to-nearest-even."""
    rng = np.random.default_rng(7)
    g = (rng.standard_normal((5, 300)) * 4).astype(np.float32)
    u = (rng.standard_normal((5, 300)) * 0.01).astype(np.float32)
    assert np.array_equal(orc.mul_bf16(g, u), _bf16_rne_from_f32(g * u))
