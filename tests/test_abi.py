"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every function that
include/w12.h declares, and answers its host-only calls (status names, shapes, scratch sizes,
argument errors caught before any device work). No call here reaches a kernel."""
import ctypes
import os
import re

import pytest

from lossless_bit_weight_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w12.h")


def declared_functions() -> list[str]:
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(w12_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def w12():
    libbuild.build()
    from lossless_bit_weight_gb300 import w12 as mod

    mod.lib()
    return mod


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("w12_encode_sizes", "w12_encode", "w12_decode", "w12_verify", "w12_gemm",
              "w12_qview_gemm", "w12_lmhead_argmax", "w12_workspace_size", "w12_status_str"):
        assert n in names


def test_library_exports_every_declared_function(w12):
    raw = ctypes.CDLL(w12.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing
    # and the binding knows the signature of each
    L = w12.lib()
    for n in declared_functions():
        assert getattr(L, n).restype is not None or n == "w12_status_str"


def test_library_is_built_for_sm103a():
    objs = [os.path.join(libbuild.BUILD, s.replace(".cu", ".o")) for s in libbuild.SOURCES]
    assert all(os.path.exists(o) for o in objs)
    assert "arch=compute_103a,code=sm_103a" in libbuild.ARCH


def test_status_names(w12):
    names = [w12.status_str(i) for i in range(8)]
    assert names == ["W12_OK", "W12_ERR_INVALID_ARG", "W12_ERR_UNSUPPORTED_SHAPE", "W12_ERR_WORKSPACE",
                     "W12_ERR_CUDA", "W12_ERR_MISMATCH", "W12_ERR_TIMEOUT", "W12_ERR_DEVICE"]
    assert w12.status_str(99) == "W12_ERR_UNKNOWN"


@pytest.mark.parametrize("N,K", [(512, 256), (17408, 5120), (151936, 5120), (1, 8), (130, 72)])
def test_tensor_shape(w12, N, K):
    t = w12.CTensor()
    rb, bb = ctypes.c_size_t(), ctypes.c_size_t()
    assert w12.lib().w12_tensor_shape(N, K, ctypes.byref(t), ctypes.byref(rb), ctypes.byref(bb)) == w12.OK
    nt, kt = -(-N // 128), -(-K // 64)
    assert (t.N, t.K, t.n_tiles, t.k_tiles) == (N, K, nt, kt)
    assert rb.value == nt * kt * 12288 and bb.value == nt * 128


def test_shape_errors(w12):
    L = w12.lib()
    t = w12.CTensor()
    rb, bb = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.w12_tensor_shape(16, 12, ctypes.byref(t), ctypes.byref(rb), ctypes.byref(bb)) == w12.ERR_UNSUPPORTED_SHAPE
    assert L.w12_tensor_shape(0, 64, ctypes.byref(t), ctypes.byref(rb), ctypes.byref(bb)) == w12.ERR_INVALID_ARG
    # 2^31 + 1 weights would overflow the 32-bit escape offsets
    assert L.w12_tensor_shape(262145, 8192, ctypes.byref(t), None, None) == w12.ERR_UNSUPPORTED_SHAPE
    assert L.w12_tensor_shape(64, 64, None, None, None) == w12.ERR_INVALID_ARG


def test_scratch_sizes(w12):
    L = w12.lib()
    nb = ctypes.c_size_t()
    assert L.w12_encode_scratch_size(17408, 5120, ctypes.byref(nb)) == w12.OK
    # at least the per-(channel, k tile) escape counts and the per-record counts
    assert nb.value >= 4 * 17408 * 80
    assert L.w12_encode_scratch_size(17408, 5120, None) == w12.ERR_INVALID_ARG
    assert L.w12_verify_scratch_size(ctypes.byref(nb)) == w12.OK and nb.value == 32
    assert L.w12_verify_scratch_size(None) == w12.ERR_INVALID_ARG


def test_null_tensor_is_rejected_before_device_work(w12):
    L = w12.lib()
    nb = ctypes.c_size_t()
    assert L.w12_decode(None, None, None) == w12.ERR_INVALID_ARG
    assert L.w12_workspace_size(None, 1, 0, ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    assert L.w12_gemm(None, None, 1, None, 0, None, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_gemm_noalloc(None, None, 1, None, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_gemm_strided(None, None, 64, 1, 0, None, 0, None, None, None, 0, None, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_gemm_strided(None, None, 0, 1, 0, None, 0, None, None, None, 0, None, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_encode(None, 64, 64, None, 0, None, None) == w12.ERR_INVALID_ARG


@pytest.mark.parametrize("N,K", [(151936, 5120), (17408, 5120), (1, 8), (130, 72)])
def test_q6_copy_shape_and_argument_checks(w12, N, K):
    """The INT6 copy's sizes (6144-byte records, one fp32 scale per padded row) and its calls'
    argument checks, all on the host."""
    L = w12.lib()
    c = w12.CQ6Copy()
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.w12_q6_shape(N, K, ctypes.byref(c), ctypes.byref(cb), ctypes.byref(sb)) == w12.OK
    nt, kt = -(-N // 128), -(-K // 64)
    assert (c.N, c.K, c.n_tiles, c.k_tiles) == (N, K, nt, kt)
    assert cb.value == nt * kt * 6144 and sb.value == 4 * nt * 128
    assert L.w12_q6_shape(N, 12, ctypes.byref(c), None, None) == w12.ERR_UNSUPPORTED_SHAPE
    nb = ctypes.c_size_t()
    # no buffers yet: rejected before any device work
    assert L.w12_q6_build(None, ctypes.byref(c), None) == w12.ERR_INVALID_ARG
    assert L.w12_q6_workspace_size(ctypes.byref(c), 1, 0, ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    assert L.w12_q6_gemm(ctypes.byref(c), None, 1, None, 0, 0, None, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_q6_argmax(None, None, 1, None, None, None, 0, None, 0, None) == w12.ERR_INVALID_ARG


def test_glue_argument_checks(w12):
    """The layer-stream glue rejects null pointers, bad sizes and unknown flags on the host."""
    L = w12.lib()
    P = ctypes.c_void_p
    one = P(16)  # never dereferenced: every call below fails its argument check first
    assert L.w12_rms_bf16(None, 1, 64, one, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_rms_bf16(one, 0, 64, one, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_rms_bf16(one, 385, 64, one, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_mul_bf16(one, one, 1, 64, 63, one, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_mul_bf16(one, None, 1, 64, 128, one, 0, None) == w12.ERR_INVALID_ARG


def test_plain_c_caller(w12, tmp_path):
    """The header compiles as C99 with warnings as errors, a C program links against the library,
    and its host-only calls answer without a GPU."""
    import subprocess
    exe = tmp_path / "c_abi_check"
    libdir = os.path.dirname(w12.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_check.c"), "-L", libdir, "-l:libw12.so",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    nt, kt = 17408 // 128, 5120 // 64
    assert out == [str(nt), str(kt), str(nt * kt * 12288), str(nt * 128), str(1187 * kt * 8192),
                   str(1187 * kt * 6144), "W12_ERR_TIMEOUT"]


def test_binding_fails_loudly_without_the_library(w12, monkeypatch):
    monkeypatch.setattr(w12, "_lib", None)
    monkeypatch.setattr(w12, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libw12.so"))
    with pytest.raises(RuntimeError, match="not built"):
        w12.lib()


def test_stream_argument_checks(w12):
    """The persistent layer-stream calls reject null pointers, layer counts, row counts and shapes
    they do not take on the host, before any device work."""
    L = w12.lib()
    P = ctypes.c_void_p
    one = P(256)  # never dereferenced: every call below fails its argument check first
    nb = ctypes.c_size_t()
    offs = (ctypes.c_size_t * 4)()
    arr = (w12.CStreamLayer * 2)()  # zeroed descriptors: no buffers
    assert L.w12_stream_workspace_size(None, 1, 8, 192, ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    assert L.w12_stream_workspace_size(arr, 0, 8, 192, ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    assert L.w12_stream_workspace_size(arr, w12.STREAM_MAX_LAYERS + 1, 8, 192, ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    assert L.w12_stream_workspace_size(arr, 1, 0, 192, ctypes.byref(nb)) == w12.ERR_UNSUPPORTED_SHAPE
    assert L.w12_stream_workspace_size(arr, 1, w12.STREAM_MAX_M + 1, 192, ctypes.byref(nb)) == w12.ERR_UNSUPPORTED_SHAPE
    assert L.w12_stream_workspace_size(arr, 1, 8, 192, ctypes.byref(nb)) == w12.ERR_INVALID_ARG  # no buffers
    assert L.w12_stream_workspace_size(arr, 1, 8, 192, None) == w12.ERR_INVALID_ARG
    assert L.w12_stream_buffers(arr, 1, 8, 192, None) == w12.ERR_INVALID_ARG
    assert L.w12_stream_buffers(arr, 1, 8, 192, offs) == w12.ERR_INVALID_ARG
    assert L.w12_stream_step(arr, 1, 8, 192, None, one, one, 1 << 20, None) == w12.ERR_INVALID_ARG
    assert L.w12_stream_step(arr, 1, 8, 192, one, one, P(258), 1 << 20, None) == w12.ERR_INVALID_ARG  # misaligned
    assert L.w12_stream_step_ex(arr, 1, 8, 192, None, one, one, 1 << 20, 0, None) == w12.ERR_INVALID_ARG
    assert L.w12_stream_step_ex(arr, 1, 8, 192, one, one, one, 1 << 20, 8, None) == w12.ERR_INVALID_ARG  # flag
    assert L.w12_stream_interleave(None, one, 128, 64, one, None) == w12.ERR_INVALID_ARG
    assert L.w12_stream_interleave(one, one, 100, 64, one, None) == w12.ERR_UNSUPPORTED_SHAPE


def _fake_tensor(w12, N, K):
    """A descriptor with the right shape and aligned buffer addresses that no call below reads:
    each fails its argument check before any device work."""
    t = w12.CTensor()
    assert w12.lib().w12_tensor_shape(N, K, ctypes.byref(t), None, None) == w12.OK
    t.records, t.base_exp, t.esc_off, t.rec_esc_off = 0x10000, 0x20000, 0x30000, 0x40000
    return t


def _fake_q8(w12, N, K):
    h = w12.CQ8Head()
    assert w12.lib().w12_q8_shape(N, K, ctypes.byref(h), None, None) == w12.OK
    h.codes, h.scale, h.bound = 0x50000, 0x60000, 0x70000
    return h


@pytest.mark.parametrize("N,K", [(151936, 5120), (130, 72)])
def test_int8_head_shape_and_argument_checks(w12, N, K):
    """The certified head's INT8 copy: its sizes (8192-byte records, one fp32 scale and bound per
    padded row), and its calls' argument checks, all on the host."""
    L = w12.lib()
    P = ctypes.c_void_p
    one = P(0x80000)
    h = w12.CQ8Head()
    cb, rb, nb = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    assert L.w12_q8_shape(N, K, ctypes.byref(h), ctypes.byref(cb), ctypes.byref(rb)) == w12.OK
    nt, kt = -(-N // 128), -(-K // 64)
    assert (h.N, h.K, h.n_tiles, h.k_tiles) == (N, K, nt, kt)
    assert cb.value == nt * kt * 8192 and rb.value == 4 * nt * 128
    assert L.w12_q8_shape(N, 12, ctypes.byref(h), None, None) == w12.ERR_UNSUPPORTED_SHAPE
    assert L.w12_q8_shape(N, K, None, None, None) == w12.ERR_INVALID_ARG
    # no buffers in h yet
    assert L.w12_q8_build(one, ctypes.byref(h), None) == w12.ERR_INVALID_ARG
    assert L.w12_q8_argmax_workspace_size(ctypes.byref(h), 1, ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    hq = _fake_q8(w12, N, K)
    assert L.w12_q8_build(None, ctypes.byref(hq), None) == w12.ERR_INVALID_ARG
    assert L.w12_q8_argmax_workspace_size(ctypes.byref(hq), 1, None) == w12.ERR_INVALID_ARG
    # the Q pass over the copy takes W12_LAUNCH_OVERLAP only
    assert L.w12_q8_argmax(ctypes.byref(hq), one, 1, one, one, one, w12.LAUNCH_TEST_STALL, one, 1 << 20,
                           None) == w12.ERR_INVALID_ARG
    hq.n_tiles += 1  # a descriptor whose tile counts do not match its shape
    assert L.w12_q8_build(one, ctypes.byref(hq), None) == w12.ERR_INVALID_ARG


def test_certified_head_argument_checks(w12):
    """w12_certified_workspace_size and w12_lmhead_certified reject a W12 head and an INT8 copy of
    different shapes, and row counts outside [1, W12_MAX_M], before any device work."""
    L = w12.lib()
    P = ctypes.c_void_p
    one = P(0x80000)
    nb = ctypes.c_size_t()
    t = _fake_tensor(w12, 1024, 512)
    h = _fake_q8(w12, 1024, 512)
    other = _fake_q8(w12, 1152, 512)
    assert L.w12_certified_workspace_size(ctypes.byref(t), ctypes.byref(h), 1, None) == w12.ERR_INVALID_ARG
    assert L.w12_certified_workspace_size(None, ctypes.byref(h), 1, ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    assert L.w12_certified_workspace_size(ctypes.byref(t), ctypes.byref(other), 1,
                                          ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    assert L.w12_certified_workspace_size(ctypes.byref(t), ctypes.byref(h), 0,
                                          ctypes.byref(nb)) == w12.ERR_UNSUPPORTED_SHAPE
    assert L.w12_certified_workspace_size(ctypes.byref(t), ctypes.byref(h), w12.MAX_M + 1,
                                          ctypes.byref(nb)) == w12.ERR_UNSUPPORTED_SHAPE
    assert L.w12_lmhead_certified(ctypes.byref(t), ctypes.byref(other), None, one, 1, one, one, one, None, one,
                                  1 << 20, None) == w12.ERR_INVALID_ARG


def test_gemm_launch_options_and_config_checks(w12):
    """w12_gemm_ex: unknown ops, an argmax op given y, and a GEMM op given argmax outputs are
    rejected; w12_gemm_config and w12_workspace_size reject row counts and ops they do not take;
    w12_check rejects a missing or too small workspace. All before any device work."""
    L = w12.lib()
    P = ctypes.c_void_p
    one = P(0x80000)
    t = _fake_tensor(w12, 17408, 5120)
    g, s, m = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    for op in (-1, 4, 99):
        assert L.w12_gemm_ex(ctypes.byref(t), one, 1, op, one, 0, None, None, None, 0, one, 1 << 20,
                             None) == w12.ERR_INVALID_ARG
    assert L.w12_gemm_ex(ctypes.byref(t), one, 1, w12.OP_ARGMAX, one, 0, one, one, one, 0, one, 1 << 20,
                         None) == w12.ERR_INVALID_ARG
    assert L.w12_gemm_ex(ctypes.byref(t), one, 1, w12.OP_GEMM, one, 0, one, None, None, 0, one, 1 << 20,
                         None) == w12.ERR_INVALID_ARG
    assert L.w12_gemm_config(None, 1, w12.OP_GEMM, ctypes.byref(g), ctypes.byref(s),
                             ctypes.byref(m)) == w12.ERR_INVALID_ARG
    for M in (0, w12.MAX_M + 1):
        assert L.w12_gemm_config(ctypes.byref(t), M, w12.OP_GEMM, ctypes.byref(g), ctypes.byref(s),
                                 ctypes.byref(m)) == w12.ERR_UNSUPPORTED_SHAPE
    nb = ctypes.c_size_t()
    for op in (-1, 4, 99, 100, 103):  # only the four W12_OP_* codes
        assert L.w12_gemm_config(ctypes.byref(t), 1, op, ctypes.byref(g), ctypes.byref(s),
                                 ctypes.byref(m)) == w12.ERR_INVALID_ARG
        assert L.w12_workspace_size(ctypes.byref(t), 1, op, ctypes.byref(nb)) == w12.ERR_INVALID_ARG
    assert L.w12_check(None, 16, None) == w12.ERR_INVALID_ARG
    assert L.w12_check(one, 8, None) == w12.ERR_INVALID_ARG
