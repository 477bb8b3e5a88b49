"""W12 CPU oracle: ctypes wrapper around ``w12_oracle.c``.

TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check and the benchmark's CPU-baseline
leg import this package. The product path (the CUDA library and its Python binding) never does.

Every function takes and returns numpy arrays (bf16 data as raw ``uint16`` bit patterns) and
computes on the CPU in plain scalar code, fp64 where floating point is involved.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w12_oracle.c")
_LIB = os.path.join(_HERE, "libw12oracle.so")

TILE_N = 128
TILE_K = 64
RECORD_BYTES = 12288


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libw12oracle.so`` with gcc (OpenMP over channels)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.w12o_window.argtypes = [P, i32]
        lib.w12o_window.restype = i32
        lib.w12o_count.argtypes = [P, i32, i32, P, P]
        lib.w12o_encode.argtypes = [P, i32, i32, P, P, P, P, P, P, P]
        lib.w12o_decode.argtypes = [P, P, P, P, i32, i32, P]
        lib.w12o_decode_csr.argtypes = [P, P, P, P, P, i32, i32, P]
        lib.w12o_qview_weights.argtypes = [P, i32, i32, P]
        lib.w12o_gemm.argtypes = [P, i32, P, i32, i32, P, P]
        lib.w12o_gemm_sampled.argtypes = [P, P, i32, P, P, i64, P, P]
        lib.w12o_argmax.argtypes = [P, i32, i32, P, P, P, P]
        lib.w12o_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.w12o_bf16_to_double.restype = ctypes.c_double
        lib.w12o_threads.restype = i32
        lib.w12o_set_threads.argtypes = [i32]
        lib.w12o_head_q8.argtypes = [P, i32, i32, P, P, P, P]
        lib.w12o_certified_argmax.argtypes = [P, i32, P, i32, i32, P, P, P, P, P, P, P]
        lib.w12o_copy_q6.argtypes = [P, i32, i32, P, P]
        lib.w12o_q6_pack.argtypes = [P, i32, i32, P]
        lib.w12o_gemm_q6.argtypes = [P, i32, P, P, i32, i32, P, P]
        lib.w12o_double_to_bf16.argtypes = [ctypes.c_double]
        lib.w12o_double_to_bf16.restype = ctypes.c_uint16
        lib.w12o_rms_bf16.argtypes = [P, i32, i32, P]
        lib.w12o_mul_bf16.argtypes = [P, P, i32, i32, i32, P]
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected raw bf16 bits as uint16, got {a.dtype}")
    return a


@dataclass
class Encoded:
    """The W12 tensor as the oracle produces it (all numpy, host memory)."""

    N: int
    K: int
    records: np.ndarray      # uint8 [R * 12288]
    base_exp: np.ndarray     # uint8 [n_tiles * 128]
    esc_off: np.ndarray      # uint32 [N + 1]
    esc_k: np.ndarray        # uint32 [n_esc]
    esc_bits: np.ndarray     # uint16 [n_esc]
    rec_esc_off: np.ndarray  # uint32 [R + 1]
    rec_esc: np.ndarray      # uint32 [n_rec_esc]

    @property
    def n_tiles(self) -> int:
        return (self.N + TILE_N - 1) // TILE_N

    @property
    def k_tiles(self) -> int:
        return (self.K + TILE_K - 1) // TILE_K


def window(row) -> int:
    row = _u16(row)
    return int(_load().w12o_window(_p(row), row.shape[0]))


def count(w) -> tuple[int, int]:
    w = _u16(w)
    N, K = w.shape
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _load().w12o_count(_p(w), N, K, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def encode(w) -> Encoded:
    w = _u16(w)
    N, K = w.shape
    n_esc, n_rec = count(w)
    nt, kt = (N + TILE_N - 1) // TILE_N, (K + TILE_K - 1) // TILE_K
    R = nt * kt
    e = Encoded(
        N, K,
        records=np.zeros(R * RECORD_BYTES, np.uint8),
        base_exp=np.zeros(nt * TILE_N, np.uint8),
        esc_off=np.zeros(N + 1, np.uint32),
        esc_k=np.zeros(max(n_esc, 1), np.uint32),
        esc_bits=np.zeros(max(n_esc, 1), np.uint16),
        rec_esc_off=np.zeros(R + 1, np.uint32),
        rec_esc=np.zeros(max(n_rec, 1), np.uint32),
    )
    _load().w12o_encode(_p(w), N, K, _p(e.records), _p(e.base_exp), _p(e.esc_off), _p(e.esc_k),
                        _p(e.esc_bits), _p(e.rec_esc_off), _p(e.rec_esc))
    e.esc_k, e.esc_bits, e.rec_esc = e.esc_k[:n_esc], e.esc_bits[:n_esc], e.rec_esc[:n_rec]
    return e


def decode(e: Encoded) -> np.ndarray:
    out = np.zeros((e.N, e.K), np.uint16)
    rec = e.rec_esc if e.rec_esc.size else np.zeros(1, np.uint32)
    _load().w12o_decode(_p(e.records), _p(e.base_exp), _p(e.rec_esc_off), _p(rec), e.N, e.K, _p(out))
    return out


def decode_csr(e: Encoded) -> np.ndarray:
    out = np.zeros((e.N, e.K), np.uint16)
    ek = e.esc_k if e.esc_k.size else np.zeros(1, np.uint32)
    eb = e.esc_bits if e.esc_bits.size else np.zeros(1, np.uint16)
    _load().w12o_decode_csr(_p(e.records), _p(e.base_exp), _p(e.esc_off), _p(ek), _p(eb),
                            e.N, e.K, _p(out))
    return out


def qview_weights(w) -> np.ndarray:
    w = _u16(w)
    N, K = w.shape
    out = np.zeros((N, K), np.uint16)
    _load().w12o_qview_weights(_p(w), N, K, _p(out))
    return out


def gemm(x, w) -> tuple[np.ndarray, np.ndarray]:
    """fp64 y = x @ w.T over exact bf16 values, and sum_k |x w| (the error-bound scale)."""
    x, w = _u16(x), _u16(w)
    M, K = x.shape
    N, K2 = w.shape
    assert K == K2
    y = np.zeros((M, N), np.float64)
    a = np.zeros((M, N), np.float64)
    _load().w12o_gemm(_p(x), M, _p(w), N, K, _p(y), _p(a))
    return y, a


def gemm_sampled(x, w, ms, ns) -> tuple[np.ndarray, np.ndarray]:
    x, w = _u16(x), _u16(w)
    ms = np.ascontiguousarray(ms, np.int32)
    ns = np.ascontiguousarray(ns, np.int32)
    y = np.zeros(ms.shape[0], np.float64)
    a = np.zeros(ms.shape[0], np.float64)
    _load().w12o_gemm_sampled(_p(x), _p(w), x.shape[1], _p(ms), _p(ns), ms.shape[0], _p(y), _p(a))
    return y, a


def argmax(y) -> tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """(top1 index, top1 value, top1 - top2 gap, max |y|) per row of an fp64 [M, N] array."""
    y = np.ascontiguousarray(y, np.float64)
    M, N = y.shape
    idx = np.zeros(M, np.int32)
    val = np.zeros(M, np.float64)
    gap = np.zeros(M, np.float64)
    sc = np.zeros(M, np.float64)
    _load().w12o_argmax(_p(y), M, N, _p(idx), _p(val), _p(gap), _p(sc))
    return idx, val, gap, sc


def threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().w12o_threads())


def set_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on (timings on one core or on all)."""
    _load().w12o_set_threads(int(n))


def bf16_to_double(u: int) -> float:
    return float(_load().w12o_bf16_to_double(int(u)))


@dataclass
class HeadQ8:
    """The certified head's INT8 copy (SpecPilot §4.1 "Certified LM head"), row-major."""

    scale: np.ndarray  # float32 [N]: s_n
    q: np.ndarray      # int8 [N, K]: round-half-even(w / s_n), clamped to +-127
    resid: np.ndarray  # float64 [N]: ||w_n - s_n q_n||_2 (+inf for a row with Inf or NaN)
    qnorm: np.ndarray  # float64 [N]: ||q_n||_2


def head_q8(w) -> HeadQ8:
    """Per-row INT8 quantisation of the head with its residual norms."""
    w = _u16(w)
    N, K = w.shape
    scale = np.zeros(N, np.float32)
    q = np.zeros((N, K), np.int8)
    resid = np.zeros(N, np.float64)
    qnorm = np.zeros(N, np.float64)
    _load().w12o_head_q8(_p(w), N, K, _p(scale), _p(q), _p(resid), _p(qnorm))
    return HeadQ8(scale, q, resid, qnorm)


def certified_argmax(x, w, h: HeadQ8):
    """The certified argmax per row, fp64 from its definition: survivors of the Cauchy-Schwarz
    bound rescored exactly. Returns (idx int32[M], val f64[M], gap f64[M], survivors int64[M])."""
    x, w = _u16(x), _u16(w)
    M, K = x.shape
    N = w.shape[0]
    idx = np.zeros(M, np.int32)
    val = np.zeros(M, np.float64)
    gap = np.zeros(M, np.float64)
    cnt = np.zeros(M, np.int64)
    _load().w12o_certified_argmax(_p(x), M, _p(w), N, K, _p(h.scale), _p(np.ascontiguousarray(h.q)),
                                  _p(h.resid), _p(idx), _p(val), _p(gap), _p(cnt))
    return idx, val, gap, cnt


def gemm_q8(x, h: HeadQ8) -> tuple[np.ndarray, np.ndarray]:
    """(yq, ad) [M, N] of the Q pass over the INT8 copy (SpecPilot §5.3 and App. C: the Q pass
    reads a separate low-precision copy): yq = s_n (x . q_n) and ad = s_n sum_k |x_k q_nk|, in
    fp64. The scaled-code product is the same definition as the INT6 copy's; only the codes
    differ, so both go through one routine."""
    x = _u16(x)
    M, K = x.shape
    N = h.q.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    ad = np.zeros((M, N), dtype=np.float64)
    _load().w12o_gemm_q6(_p(x), M, _p(np.ascontiguousarray(h.q)), _p(h.scale), N, K, _p(y), _p(ad))
    return y, ad


@dataclass
class CopyQ6:
    """The INT6 Q-pass copy (SpecPilot §5.3, App. C): row scales and row-major codes."""

    scale: np.ndarray  # float32 [N]
    q: np.ndarray      # int8 [N, K], in [-31, 31]


def copy_q6(w) -> CopyQ6:
    w = _u16(w)
    N, K = w.shape
    scale = np.zeros(N, dtype=np.float32)
    q = np.zeros((N, K), dtype=np.int8)
    _load().w12o_copy_q6(_p(w), N, K, _p(scale), _p(q))
    return CopyQ6(scale, q)


def q6_pack(q: np.ndarray) -> np.ndarray:
    """The INT6 copy's 6144-byte records (uint8 [n_tiles * k_tiles * 6144]) from row-major codes."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    N, K = q.shape
    nt, kt = (N + TILE_N - 1) // TILE_N, (K + TILE_K - 1) // TILE_K
    rec = np.zeros(nt * kt * 6144, dtype=np.uint8)
    _load().w12o_q6_pack(_p(q), N, K, _p(rec))
    return rec


def gemm_q6(x, c: CopyQ6) -> tuple[np.ndarray, np.ndarray]:
    """(yq, ad) [M, N]: yq = s_n (x . c_n) and ad = s_n sum_k |x_k c_nk|, in fp64."""
    x = _u16(x)
    M, K = x.shape
    N = c.q.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    ad = np.zeros((M, N), dtype=np.float64)
    _load().w12o_gemm_q6(_p(x), M, _p(np.ascontiguousarray(c.q)), _p(c.scale), N, K, _p(y), _p(ad))
    return y, ad


def double_to_bf16(v: float) -> int:
    """bf16 bits of a double, rounded to nearest even."""
    return int(_load().w12o_double_to_bf16(float(v)))


def rms_bf16(h: np.ndarray) -> np.ndarray:
    """The synthetic stream's row normalisation: bf16 bits of h / sqrt(mean(h^2)), fp64."""
    h = np.ascontiguousarray(h, dtype=np.float32)
    M, K = h.shape
    x = np.zeros((M, K), dtype=np.uint16)
    _load().w12o_rms_bf16(_p(h), M, K, _p(x))
    return x


def mul_bf16(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """The synthetic stream's gate-up product: bf16 bits of the fp32 product g * u."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    M, N = g.shape
    p = np.zeros((M, N), dtype=np.uint16)
    _load().w12o_mul_bf16(_p(g), _p(u), M, N, N, _p(p))
    return p
