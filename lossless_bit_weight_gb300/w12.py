"""Thin Python binding of the W12 C ABI (``include/w12.h``, ``libw12.so``).

It only marshals torch CUDA tensors into the C calls: every step of encode, verify, decode and
the GEMMs runs in the library's CUDA kernels. torch provides device memory and the current
stream. There is no CPU or eager fallback: if the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libw12.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_WORKSPACE, ERR_CUDA, ERR_MISMATCH, ERR_TIMEOUT, \
    ERR_DEVICE = range(8)
OUT_F32, OUT_BF16 = 0, 1
LAUNCH_OVERLAP, LAUNCH_TEST_STALL, LAUNCH_ACCUMULATE = 1, 2, 4
OP_GEMM, OP_QVIEW_GEMM, OP_ARGMAX, OP_QVIEW_ARGMAX = range(4)
TILE_N, TILE_K, RECORD_BYTES, VIEW_BYTES, MAX_M = 128, 64, 12288, 8192, 384


class W12Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_str(status)}")
        self.status = status


class CTensor(ctypes.Structure):
    """Mirror of ``w12_tensor``."""

    _fields_ = [
        ("N", ctypes.c_int32), ("K", ctypes.c_int32),
        ("n_tiles", ctypes.c_int32), ("k_tiles", ctypes.c_int32),
        ("records", ctypes.c_void_p), ("base_exp", ctypes.c_void_p),
        ("esc_off", ctypes.c_void_p), ("esc_k", ctypes.c_void_p), ("esc_bits", ctypes.c_void_p),
        ("rec_esc_off", ctypes.c_void_p), ("rec_esc", ctypes.c_void_p),
        ("n_esc", ctypes.c_int64), ("n_rec_esc", ctypes.c_int64),
    ]


class CStreamLayer(ctypes.Structure):
    """Mirror of ``w12_stream_layer``."""

    _fields_ = [("qkv", CTensor), ("o", CTensor), ("gate_up", CTensor), ("down", CTensor)]


class CQ8Head(ctypes.Structure):
    """Mirror of ``w12_q8_head``."""

    _fields_ = [
        ("N", ctypes.c_int32), ("K", ctypes.c_int32),
        ("n_tiles", ctypes.c_int32), ("k_tiles", ctypes.c_int32),
        ("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bound", ctypes.c_void_p),
    ]


class CQ6Copy(ctypes.Structure):
    """Mirror of ``w12_q6_copy``."""

    _fields_ = [
        ("N", ctypes.c_int32), ("K", ctypes.c_int32),
        ("n_tiles", ctypes.c_int32), ("k_tiles", ctypes.c_int32),
        ("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load ``libw12.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"W12 CUDA library not built: {LIB_PATH} is missing "
                               "(run lossless_bit_weight_gb300.build.build())")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        T = ctypes.POINTER(CTensor)
        sig = {
            "w12_status_str": ([i32], ctypes.c_char_p),
            "w12_tensor_shape": ([i32, i32, T, ctypes.POINTER(sz), ctypes.POINTER(sz)], i32),
            "w12_encode_scratch_size": ([i32, i32, ctypes.POINTER(sz)], i32),
            "w12_encode_sizes": ([P, i32, i32, P, sz, ctypes.POINTER(i64), ctypes.POINTER(i64), P], i32),
            "w12_encode": ([P, i32, i32, P, sz, T, P], i32),
            "w12_decode": ([T, P, P], i32),
            "w12_verify_scratch_size": ([ctypes.POINTER(sz)], i32),
            "w12_verify": ([T, P, P, sz, ctypes.POINTER(ctypes.c_uint64), P], i32),
            "w12_workspace_size": ([T, i32, i32, ctypes.POINTER(sz)], i32),
            "w12_gemm": ([T, P, i32, P, i32, P, sz, P], i32),
            "w12_qview_gemm": ([T, P, i32, P, i32, P, sz, P], i32),
            "w12_lmhead_argmax": ([T, P, i32, P, P, P, i32, P, sz, P], i32),
            "w12_check": ([P, sz, P], i32),
            "w12_gemm_noalloc": ([T, P, i32, P, i32, P], i32),
            "w12_gemm_ex": ([T, P, i32, i32, P, i32, P, P, P, ctypes.c_uint, P, sz, P], i32),
            "w12_gemm_strided": ([T, P, i32, i32, i32, P, i32, P, P, P, ctypes.c_uint, P, sz, P], i32),
            "w12_gemm_config": ([T, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                 ctypes.POINTER(i32)], i32),
            "w12_q8_shape": ([i32, i32, ctypes.POINTER(CQ8Head), ctypes.POINTER(sz), ctypes.POINTER(sz)], i32),
            "w12_q8_build": ([P, ctypes.POINTER(CQ8Head), P], i32),
            "w12_certified_workspace_size": ([T, ctypes.POINTER(CQ8Head), i32, ctypes.POINTER(sz)], i32),
            "w12_lmhead_certified": ([T, ctypes.POINTER(CQ8Head), P, P, i32, P, P, P, P, P, sz, P], i32),
            "w12_q8_argmax_workspace_size": ([ctypes.POINTER(CQ8Head), i32, ctypes.POINTER(sz)], i32),
            "w12_q8_argmax": ([ctypes.POINTER(CQ8Head), P, i32, P, P, P, ctypes.c_uint, P, sz, P], i32),
            "w12_rms_bf16": ([P, i32, i32, P, ctypes.c_uint, P], i32),
            "w12_mul_bf16": ([P, P, i32, i32, i32, P, ctypes.c_uint, P], i32),
            "w12_q6_shape": ([i32, i32, ctypes.POINTER(CQ6Copy), ctypes.POINTER(sz), ctypes.POINTER(sz)], i32),
            "w12_q6_build": ([P, ctypes.POINTER(CQ6Copy), P], i32),
            "w12_q6_workspace_size": ([ctypes.POINTER(CQ6Copy), i32, i32, ctypes.POINTER(sz)], i32),
            "w12_q6_gemm": ([ctypes.POINTER(CQ6Copy), P, i32, P, i32, ctypes.c_uint, P, sz, P], i32),
            "w12_q6_argmax": ([ctypes.POINTER(CQ6Copy), P, i32, P, P, P, ctypes.c_uint, P, sz, P], i32),
            "w12_stream_workspace_size": ([ctypes.POINTER(CStreamLayer), i32, i32, i32, ctypes.POINTER(sz)], i32),
            "w12_stream_buffers": ([ctypes.POINTER(CStreamLayer), i32, i32, i32, ctypes.POINTER(sz)], i32),
            "w12_stream_step": ([ctypes.POINTER(CStreamLayer), i32, i32, i32, P, P, P, sz, P], i32),
            "w12_stream_step_ex": ([ctypes.POINTER(CStreamLayer), i32, i32, i32, P, P, P, sz, ctypes.c_uint, P], i32),
            "w12_stream_interleave": ([P, P, i32, i32, P, P], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().w12_status_str(status).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise W12Error(status, what)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check_out(out: torch.Tensor, M: int, N: int, dtypes=(torch.float32, torch.bfloat16)) -> None:
    """The output buffer must be a contiguous [M, N] tensor of an accepted type on a CUDA device:
    the library writes M * N elements of out's own type."""
    if out.dtype not in dtypes or tuple(out.shape) != (M, N) or not out.is_contiguous() or not out.is_cuda:
        raise ValueError(f"out must be a contiguous CUDA tensor of shape ({M}, {N}) and type in {dtypes}, "
                         f"got {tuple(out.shape)} {out.dtype}")


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bits(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous bf16 CUDA tensor")
    return t


def _rows(x: torch.Tensor) -> int:
    """Row stride of a 2-D bf16 CUDA tensor whose rows are contiguous (a column slice of a wider
    row-major tensor qualifies)."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("expected a bf16 CUDA tensor [M, K] with contiguous rows")
    return x.stride(0)


@dataclass
class W12Tensor:
    """An encoded weight matrix: the device buffers of ``w12_tensor`` plus its descriptor."""

    N: int
    K: int
    records: torch.Tensor
    base_exp: torch.Tensor
    esc_off: torch.Tensor
    esc_k: torch.Tensor
    esc_bits: torch.Tensor
    rec_esc_off: torch.Tensor
    rec_esc: torch.Tensor
    n_esc: int
    n_rec_esc: int
    c: CTensor = field(default=None, repr=False)
    _ws: dict = field(default_factory=dict, repr=False)

    def __post_init__(self):
        self.c = CTensor(self.N, self.K, (self.N + TILE_N - 1) // TILE_N, (self.K + TILE_K - 1) // TILE_K,
                         self.records.data_ptr(), self.base_exp.data_ptr(), self.esc_off.data_ptr(),
                         self.esc_k.data_ptr(), self.esc_bits.data_ptr(), self.rec_esc_off.data_ptr(),
                         self.rec_esc.data_ptr(), self.n_esc, self.n_rec_esc)

    @property
    def n_tiles(self) -> int:
        return self.c.n_tiles

    @property
    def k_tiles(self) -> int:
        return self.c.k_tiles

    @property
    def nbytes(self) -> int:
        """Bytes of the encoded tensor (records, bases, both escape lists and their offsets)."""
        return sum(t.numel() * t.element_size() for t in (
            self.records, self.base_exp, self.esc_off, self.esc_k, self.esc_bits,
            self.rec_esc_off, self.rec_esc))

    def gemm_bytes(self, qview: bool = False) -> int:
        """Encoded bytes one GEMM call streams: records (or their 8-bit views), bases, and the
        per-record escape index with its offsets (the exact GEMM only)."""
        R = self.n_tiles * self.k_tiles
        if qview:
            return R * VIEW_BYTES + self.base_exp.numel()
        return (R * RECORD_BYTES + self.base_exp.numel() + 4 * (R + 1) + 4 * self.n_rec_esc)

    def workspace(self, M: int, op: int) -> tuple[torch.Tensor, int]:
        """A zero-filled workspace for (M, op), cached on this tensor and reused across calls."""
        key = (M, op, torch.cuda.current_device())
        if key not in self._ws:
            nb = ctypes.c_size_t()
            _check(lib().w12_workspace_size(ctypes.byref(self.c), M, op, ctypes.byref(nb)), "w12_workspace_size")
            self._ws[key] = (torch.zeros(max(int(nb.value), 16), dtype=torch.uint8, device="cuda"), int(nb.value))
        return self._ws[key]

    def clone_records(self) -> "W12Tensor":
        """A second encoded tensor with copied buffers (to stream weights that are not in L2)."""
        return W12Tensor(self.N, self.K, self.records.clone(), self.base_exp.clone(), self.esc_off.clone(),
                         self.esc_k.clone(), self.esc_bits.clone(), self.rec_esc_off.clone(),
                         self.rec_esc.clone(), self.n_esc, self.n_rec_esc)


def encode(w: torch.Tensor, stream=None) -> W12Tensor:
    """Encode a bf16 [N, K] CUDA tensor (``w12_encode_sizes`` then ``w12_encode``)."""
    _bits(w)
    N, K = w.shape
    L = lib()
    nb = ctypes.c_size_t()
    _check(L.w12_encode_scratch_size(N, K, ctypes.byref(nb)), "w12_encode_scratch_size")
    scratch = torch.empty(int(nb.value), dtype=torch.uint8, device=w.device)
    n_esc, n_rec = ctypes.c_int64(), ctypes.c_int64()
    st = _stream(stream)
    _check(L.w12_encode_sizes(_ptr(w), N, K, _ptr(scratch), nb, ctypes.byref(n_esc), ctypes.byref(n_rec), st),
           "w12_encode_sizes")
    shape = CTensor()
    rb, bb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(L.w12_tensor_shape(N, K, ctypes.byref(shape), ctypes.byref(rb), ctypes.byref(bb)), "w12_tensor_shape")
    R = shape.n_tiles * shape.k_tiles
    dev = w.device
    t = W12Tensor(
        N, K,
        records=torch.empty(int(rb.value), dtype=torch.uint8, device=dev),
        base_exp=torch.empty(int(bb.value), dtype=torch.uint8, device=dev),
        esc_off=torch.empty(N + 1, dtype=torch.int32, device=dev),
        esc_k=torch.empty(max(n_esc.value, 4), dtype=torch.int32, device=dev),
        esc_bits=torch.empty(max(n_esc.value, 8), dtype=torch.int16, device=dev),
        rec_esc_off=torch.empty(R + 1, dtype=torch.int32, device=dev),
        rec_esc=torch.empty(max(n_rec.value, 4), dtype=torch.int32, device=dev),
        n_esc=n_esc.value, n_rec_esc=n_rec.value,
    )
    _check(L.w12_encode(_ptr(w), N, K, _ptr(scratch), nb, ctypes.byref(t.c), st), "w12_encode")
    return t


def decode(t: W12Tensor, stream=None) -> torch.Tensor:
    out = torch.empty((t.N, t.K), dtype=torch.bfloat16, device=t.records.device)
    _check(lib().w12_decode(ctypes.byref(t.c), _ptr(out), _stream(stream)), "w12_decode")
    return out


def verify(t: W12Tensor, w_ref: torch.Tensor, stream=None) -> int:
    """Number of weights/escape entries that do not decode to ``w_ref`` bit for bit (0 = lossless)."""
    _bits(w_ref)
    nb = ctypes.c_size_t()
    _check(lib().w12_verify_scratch_size(ctypes.byref(nb)), "w12_verify_scratch_size")
    scratch = torch.empty(int(nb.value), dtype=torch.uint8, device=w_ref.device)
    bad = ctypes.c_uint64()
    st = lib().w12_verify(ctypes.byref(t.c), _ptr(w_ref), _ptr(scratch), nb, ctypes.byref(bad), _stream(stream))
    if st not in (OK, ERR_MISMATCH):
        _check(st, "w12_verify")
    return int(bad.value)


def gemm(t: W12Tensor, x: torch.Tensor, out_dtype=torch.float32, qview: bool = False,
         out: torch.Tensor | None = None, stream=None, overlap: bool = False,
         test_stall: bool = False, accumulate: bool = False) -> torch.Tensor:
    """y = x @ W^T over the exact weights (or the 8-bit view when ``qview``).

    ``overlap`` launches with ``W12_LAUNCH_OVERLAP`` (``w12_gemm_ex``): the kernel may start, and
    fetch and decode its weights, while the previous kernel on the stream finishes; t's buffers
    must not be written by that kernel. ``test_stall`` sets the ``W12_LAUNCH_TEST_STALL`` test
    hook (the bounded waits run out; ``check`` then raises). x may be a column slice of a wider
    tensor (rows contiguous, row stride a multiple of 8): it then goes through
    ``w12_gemm_strided``. ``accumulate`` (fp32 ``out`` only,
    ``W12_LAUNCH_ACCUMULATE``) adds the result into ``out`` instead of overwriting it."""
    ldx = _rows(x)
    M = x.shape[0]
    if x.shape[1] != t.K:
        raise ValueError("x must be [M, K]")
    if accumulate and (out is None or out.dtype != torch.float32):
        raise ValueError("accumulate needs an fp32 out tensor")
    if out is None:
        out = torch.empty((M, t.N), dtype=out_dtype, device=x.device)
    _check_out(out, M, t.N)
    ydt = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    op = OP_QVIEW_GEMM if qview else OP_GEMM
    ws, nb = t.workspace(M, op)
    if ldx != t.K:
        flags = ((LAUNCH_OVERLAP if overlap else 0) | (LAUNCH_TEST_STALL if test_stall else 0)
                 | (LAUNCH_ACCUMULATE if accumulate else 0))
        _check(lib().w12_gemm_strided(ctypes.byref(t.c), _ptr(x), ldx, M, op, _ptr(out), ydt, None, None, None,
                                      flags, _ptr(ws), nb, _stream(stream)), "w12_gemm_strided")
        return out
    if overlap or test_stall or accumulate:
        flags = ((LAUNCH_OVERLAP if overlap else 0) | (LAUNCH_TEST_STALL if test_stall else 0)
                 | (LAUNCH_ACCUMULATE if accumulate else 0))
        _check(lib().w12_gemm_ex(ctypes.byref(t.c), _ptr(x), M, op, _ptr(out), ydt, None, None, None,
                                 flags, _ptr(ws), nb, _stream(stream)), "w12_gemm_ex")
        return out
    fn = lib().w12_qview_gemm if qview else lib().w12_gemm
    _check(fn(ctypes.byref(t.c), _ptr(x), M, _ptr(out), ydt, _ptr(ws), nb, _stream(stream)),
           "w12_qview_gemm" if qview else "w12_gemm")
    return out


def lmhead_argmax(t: W12Tensor, x: torch.Tensor, qview: bool = False, stream=None, overlap: bool = False):
    """(idx int32[M], val f32[M], gap f32[M]) of y = x @ W^T without materialising y."""
    _bits(x)
    M = x.shape[0]
    idx = torch.empty(M, dtype=torch.int32, device=x.device)
    val = torch.empty(M, dtype=torch.float32, device=x.device)
    gap = torch.empty(M, dtype=torch.float32, device=x.device)
    op = OP_QVIEW_ARGMAX if qview else OP_ARGMAX
    ws, nb = t.workspace(M, op)
    if overlap:
        _check(lib().w12_gemm_ex(ctypes.byref(t.c), _ptr(x), M, op, None, OUT_F32, _ptr(idx), _ptr(val),
                                 _ptr(gap), LAUNCH_OVERLAP, _ptr(ws), nb, _stream(stream)), "w12_gemm_ex")
        return idx, val, gap
    _check(lib().w12_lmhead_argmax(ctypes.byref(t.c), _ptr(x), M, _ptr(idx), _ptr(val), _ptr(gap),
                                   1 if qview else 0, _ptr(ws), nb, _stream(stream)), "w12_lmhead_argmax")
    return idx, val, gap


def gemm_noalloc(t: W12Tensor, x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 y = x @ W^T through ``w12_gemm_noalloc``: no workspace is allocated (the library's
    fixed device array serves as workspace; M <= 32)."""
    _bits(x)
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, t.N), dtype=torch.float32, device=x.device)
    _check_out(out, M, t.N, (torch.float32,))
    _check(lib().w12_gemm_noalloc(ctypes.byref(t.c), _ptr(x), M, _ptr(out), OUT_F32, _stream(stream)),
           "w12_gemm_noalloc")
    return out


def check(t: W12Tensor, stream=None) -> None:
    """Synchronise and raise if any GEMM kernel on one of t's workspaces gave up a bounded wait."""
    for ws, nb in t._ws.values():
        _check(lib().w12_check(_ptr(ws), nb, _stream(stream)), "w12_check")


def gemm_config(t: W12Tensor, M: int, op: int) -> dict:
    g, s, m = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().w12_gemm_config(ctypes.byref(t.c), M, op, ctypes.byref(g), ctypes.byref(s), ctypes.byref(m)),
           "w12_gemm_config")
    return {"grid": g.value, "stages": s.value, "smem_bytes": m.value}


class Q8Head:
    """The certified LM head's INT8 copy (``w12_q8_head``): codes, row scales and row bounds."""

    def __init__(self, N: int, K: int, device="cuda"):
        self.c = CQ8Head()
        cb, rb = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().w12_q8_shape(N, K, ctypes.byref(self.c), ctypes.byref(cb), ctypes.byref(rb)), "w12_q8_shape")
        self.N, self.K = N, K
        self.codes = torch.empty(int(cb.value), dtype=torch.uint8, device=device)
        self.scale = torch.empty(int(rb.value) // 4, dtype=torch.float32, device=device)
        self.bound = torch.empty(int(rb.value) // 4, dtype=torch.float32, device=device)
        self.c.codes, self.c.scale, self.c.bound = self.codes.data_ptr(), self.scale.data_ptr(), self.bound.data_ptr()
        self._ws = {}

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.codes, self.scale, self.bound))

    def gemm_bytes(self) -> int:
        """Bytes the approximate pass streams: the codes and the row scales."""
        return self.codes.numel() + self.scale.numel() * 4


def q8_build(w: torch.Tensor, stream=None) -> Q8Head:
    """The INT8 copy of a bf16 head [N, K] (device)."""
    _bits(w)
    N, K = w.shape
    h = Q8Head(N, K, device=w.device)
    _check(lib().w12_q8_build(_ptr(w), ctypes.byref(h.c), _stream(stream)), "w12_q8_build")
    return h


def lmhead_certified(t: W12Tensor, h: Q8Head, x: torch.Tensor, w_bf16: torch.Tensor | None = None, stream=None):
    """(idx int32[M], val f32[M], gap f32[M], survivors int32[M]) of x @ W^T through the certified
    head: the INT8 copy's bound discards tokens; the survivors are rescored from w_bf16 (the
    bf16 head, if given) or else from the W12 head t."""
    if w_bf16 is not None:
        _bits(w_bf16)
    _bits(x)
    M = x.shape[0]
    idx = torch.empty(M, dtype=torch.int32, device=x.device)
    val = torch.empty(M, dtype=torch.float32, device=x.device)
    gap = torch.empty(M, dtype=torch.float32, device=x.device)
    surv = torch.empty(M, dtype=torch.int32, device=x.device)
    key = (M, torch.cuda.current_device())
    if key not in h._ws:
        nb = ctypes.c_size_t()
        _check(lib().w12_certified_workspace_size(ctypes.byref(t.c), ctypes.byref(h.c), M, ctypes.byref(nb)),
               "w12_certified_workspace_size")
        h._ws[key] = (torch.zeros(max(int(nb.value), 16), dtype=torch.uint8, device=x.device), int(nb.value))
    ws, nb = h._ws[key]
    _check(lib().w12_lmhead_certified(ctypes.byref(t.c), ctypes.byref(h.c), _ptr(w_bf16), _ptr(x), M, _ptr(idx), _ptr(val),
                                      _ptr(gap), _ptr(surv), _ptr(ws), nb, _stream(stream)), "w12_lmhead_certified")
    return idx, val, gap, surv


def q8_argmax(h: Q8Head, x: torch.Tensor, stream=None, overlap: bool = False):
    """(idx int32[M], val f32[M], gap f32[M]) of the argmax over the INT8 copy alone: the Q pass
    through the separate copy (approximate; compare lmhead_certified for the exact argmax)."""
    _bits(x)
    M = x.shape[0]
    idx = torch.empty(M, dtype=torch.int32, device=x.device)
    val = torch.empty(M, dtype=torch.float32, device=x.device)
    gap = torch.empty(M, dtype=torch.float32, device=x.device)
    key = ("argmax", M, torch.cuda.current_device())
    if key not in h._ws:
        nb = ctypes.c_size_t()
        _check(lib().w12_q8_argmax_workspace_size(ctypes.byref(h.c), M, ctypes.byref(nb)),
               "w12_q8_argmax_workspace_size")
        h._ws[key] = (torch.zeros(max(int(nb.value), 16), dtype=torch.uint8, device=x.device), int(nb.value))
    ws, nb = h._ws[key]
    _check(lib().w12_q8_argmax(ctypes.byref(h.c), _ptr(x), M, _ptr(idx), _ptr(val), _ptr(gap),
                               LAUNCH_OVERLAP if overlap else 0, _ptr(ws), nb, _stream(stream)), "w12_q8_argmax")
    return idx, val, gap


class Q6Copy:
    """The INT6 Q-pass copy of a weight matrix (``w12_q6_copy``): 6 KB records and row scales."""

    def __init__(self, N: int, K: int, device="cuda"):
        self.c = CQ6Copy()
        cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().w12_q6_shape(N, K, ctypes.byref(self.c), ctypes.byref(cb), ctypes.byref(sb)), "w12_q6_shape")
        self.N, self.K = N, K
        self.codes = torch.empty(int(cb.value), dtype=torch.uint8, device=device)
        self.scale = torch.empty(int(sb.value) // 4, dtype=torch.float32, device=device)
        self.c.codes, self.c.scale = self.codes.data_ptr(), self.scale.data_ptr()
        self._ws = {}

    @property
    def nbytes(self) -> int:
        return self.codes.numel() + self.scale.numel() * 4

    def workspace(self, M: int, argmax: bool, device):
        key = (M, bool(argmax), torch.cuda.current_device())
        if key not in self._ws:
            nb = ctypes.c_size_t()
            _check(lib().w12_q6_workspace_size(ctypes.byref(self.c), M, 1 if argmax else 0, ctypes.byref(nb)),
                   "w12_q6_workspace_size")
            self._ws[key] = (torch.zeros(max(int(nb.value), 16), dtype=torch.uint8, device=device), int(nb.value))
        return self._ws[key]


def q6_build(w: torch.Tensor, stream=None) -> Q6Copy:
    """The INT6 Q-pass copy of a bf16 matrix [N, K] (device)."""
    _bits(w)
    N, K = w.shape
    c = Q6Copy(N, K, device=w.device)
    _check(lib().w12_q6_build(_ptr(w), ctypes.byref(c.c), _stream(stream)), "w12_q6_build")
    return c


def q6_gemm(c: Q6Copy, x: torch.Tensor, out_dtype=torch.float32, out: torch.Tensor | None = None, stream=None,
            overlap: bool = False) -> torch.Tensor:
    """yq = x @ (scale * codes)^T through the INT6 copy: fp32 or bf16 [M, N]."""
    _bits(x)
    M = x.shape[0]
    if out is None:
        out = torch.empty(M, c.N, dtype=out_dtype, device=x.device)
    _check_out(out, M, c.N)
    ydt = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    ws, nb = c.workspace(M, False, x.device)
    _check(lib().w12_q6_gemm(ctypes.byref(c.c), _ptr(x), M, _ptr(out), ydt, LAUNCH_OVERLAP if overlap else 0,
                             _ptr(ws), nb, _stream(stream)), "w12_q6_gemm")
    return out


def q6_argmax(c: Q6Copy, x: torch.Tensor, stream=None, overlap: bool = False):
    """(idx int32[M], val f32[M], gap f32[M]) of each row's argmax of the INT6 Q pass."""
    _bits(x)
    M = x.shape[0]
    idx = torch.empty(M, dtype=torch.int32, device=x.device)
    val = torch.empty(M, dtype=torch.float32, device=x.device)
    gap = torch.empty(M, dtype=torch.float32, device=x.device)
    ws, nb = c.workspace(M, True, x.device)
    _check(lib().w12_q6_argmax(ctypes.byref(c.c), _ptr(x), M, _ptr(idx), _ptr(val), _ptr(gap),
                               LAUNCH_OVERLAP if overlap else 0, _ptr(ws), nb, _stream(stream)), "w12_q6_argmax")
    return idx, val, gap


def rms_bf16(h: torch.Tensor, out: torch.Tensor | None = None, stream=None, overlap: bool = False) -> torch.Tensor:
    """The synthetic layer stream's row normalisation: bf16 h * (1 / sqrt(mean(h^2))) of fp32 h
    [M, K], in fp64 before the one rounding to bf16."""
    if h.dtype != torch.float32 or not h.is_contiguous() or h.dim() != 2:
        raise ValueError("h must be a contiguous fp32 [M, K] tensor")
    M, K = h.shape
    if out is None:
        out = torch.empty((M, K), dtype=torch.bfloat16, device=h.device)
    _check_out(out, M, K, (torch.bfloat16,))
    _check(lib().w12_rms_bf16(_ptr(h), M, K, _ptr(out), LAUNCH_OVERLAP if overlap else 0, _stream(stream)),
           "w12_rms_bf16")
    return out


def mul_bf16(gu: torch.Tensor, N: int, out: torch.Tensor | None = None, stream=None,
             overlap: bool = False) -> torch.Tensor:
    """The synthetic layer stream's gate-up product: bf16 g * u, where g = gu[:, :N] and
    u = gu[:, N:2N] of one fp32 [M, 2N] GEMM output (the gate and up weights concatenated)."""
    if gu.dtype != torch.float32 or not gu.is_contiguous() or gu.dim() != 2 or gu.shape[1] != 2 * N:
        raise ValueError("gu must be a contiguous fp32 [M, 2N] tensor")
    M = gu.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=gu.device)
    _check_out(out, M, N, (torch.bfloat16,))
    _check(lib().w12_mul_bf16(_ptr(gu), gu.data_ptr() + 4 * N, M, N, 2 * N, _ptr(out),
                              LAUNCH_OVERLAP if overlap else 0, _stream(stream)), "w12_mul_bf16")
    return out


STREAM_MAX_LAYERS, STREAM_MAX_M = 80, 32


def stream_interleave(gate: torch.Tensor, up: torch.Tensor, stream=None) -> torch.Tensor:
    """The gate|up matrix the layer-stream step reads (``w12_stream_interleave``): bf16 [2F, H]
    with gate rows 64i.. at rows 128i.. and the matching up rows at rows 128i+64..; gate and up
    are bf16 [F, H] CUDA tensors."""
    _bits(gate)
    _bits(up)
    if gate.shape != up.shape:
        raise ValueError("gate and up must have the same shape")
    F, H = gate.shape
    out = torch.empty((2 * F, H), dtype=torch.bfloat16, device=gate.device)
    _check(lib().w12_stream_interleave(_ptr(gate), _ptr(up), F, H, _ptr(out), _stream(stream)),
           "w12_stream_interleave")
    return out


class StreamStep:
    """One decoding step of the synthetic layer stream in one persistent launch
    (``w12_stream_step``): every layer's row normalisations, q|k|v, o (added into h), gate|up with
    the gate-up product, down (added into h), then the final row normalisation.

    ``layers`` is a list of dicts with encoded tensors under "qkv", "o", "gate_up" (interleaved by
    ``stream_interleave``) and "down"; the workspace is allocated here and kept."""

    def __init__(self, layers: list, M: int, n_q: int, device="cuda"):
        n = len(layers)
        if not 1 <= n <= STREAM_MAX_LAYERS:
            raise ValueError(f"1 to {STREAM_MAX_LAYERS} layers")
        self.tensors = layers  # keeps the device buffers alive
        self.arr = (CStreamLayer * n)()
        for i, ly in enumerate(layers):
            self.arr[i] = CStreamLayer(ly["qkv"].c, ly["o"].c, ly["gate_up"].c, ly["down"].c)
        self.n, self.M, self.n_q = n, M, n_q
        nb = ctypes.c_size_t()
        _check(lib().w12_stream_workspace_size(self.arr, n, M, n_q, ctypes.byref(nb)), "w12_stream_workspace_size")
        self.ws_bytes = int(nb.value)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        offs = (ctypes.c_size_t * 4)()
        _check(lib().w12_stream_buffers(self.arr, n, M, n_q, offs), "w12_stream_buffers")
        self.offsets = [int(o) for o in offs]
        self.hidden = layers[0]["qkv"].K
        self.n_qkv = layers[0]["qkv"].N
        self.ffn = layers[0]["down"].K

    def __call__(self, h: torch.Tensor, x_out: torch.Tensor | None = None, stream=None,
                 test_stall: bool = False) -> torch.Tensor:
        """Runs the step on fp32 h [M, hidden] (updated in place); returns x_out = rms_bf16(final h).
        ``test_stall`` sets the ``W12_LAUNCH_TEST_STALL`` test hook (the failure path: the step's
        bounded waits run out; ``check`` then raises and the workspace must be zeroed again)."""
        if h.dtype != torch.float32 or not h.is_contiguous() or tuple(h.shape) != (self.M, self.hidden):
            raise ValueError(f"h must be a contiguous fp32 tensor of shape ({self.M}, {self.hidden})")
        if x_out is None:
            x_out = torch.empty((self.M, self.hidden), dtype=torch.bfloat16, device=h.device)
        _check_out(x_out, self.M, self.hidden, (torch.bfloat16,))
        _check(lib().w12_stream_step_ex(self.arr, self.n, self.M, self.n_q, _ptr(h), _ptr(x_out), _ptr(self.ws),
                                        self.ws_bytes, LAUNCH_TEST_STALL if test_stall else 0, _stream(stream)),
               "w12_stream_step")
        return x_out

    def buffers(self) -> dict:
        """Views of the last layer's intermediates in the workspace (valid after a step): x, qkv,
        x2 (bf16 [M, hidden], [M, n_qkv], [M, hidden]) and p (bf16 [M, ffn])."""
        M = self.M

        def view(off, cols):
            return self.ws[off: off + 2 * M * cols].view(torch.bfloat16).view(M, cols)

        return {"x": view(self.offsets[0], self.hidden), "qkv": view(self.offsets[1], self.n_qkv),
                "x2": view(self.offsets[2], self.hidden), "p": view(self.offsets[3], self.ffn)}

    def check(self, stream=None) -> None:
        """Synchronise and raise if the step's kernel gave up a bounded wait."""
        _check(lib().w12_check(_ptr(self.ws), self.ws_bytes, _stream(stream)), "w12_check")
