"""Host-side checks of the C ABI: the library builds, loads without a GPU, exports
every symbol include/dprc.h declares, and rejects bad arguments before any
device work.  No kernel runs here."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dprc.h")


@pytest.fixture(scope="session")
def lib():
    from randomized_norm_clipping_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dprc_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("dprc_norm_hutch", "dprc_norm_hutchpp", "dprc_exact_norm",
                     "dprc_clip_factors", "dprc_add_noise", "dprc_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    from randomized_norm_clipping_gb300 import binding
    assert set(binding.EXPORTED) == set(_declared())


def test_bounds_checked_build_exports_the_same_symbols(lib):
    # libdprc_debug.so: the same sources with every computed index checked
    from randomized_norm_clipping_gb300 import build
    if not os.path.exists(build.DEBUG_LIB_PATH):
        build.build(variants=("debug",))
    dbg = ctypes.CDLL(build.DEBUG_LIB_PATH)
    for name in _declared():
        assert hasattr(dbg, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.dprc_abi_version() == 1
    for code in range(9):
        s = lib.dprc_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.dprc_status_string(99) == b"unknown status"


def test_workspace_bytes_host_only(lib):
    from randomized_norm_clipping_gb300 import binding as b
    # tensor-core path (bf16, k = 32): sketch hi/lo planes + partial slots
    ws = b.dprc_workspace_bytes(b.DPRC_OP_HUTCH, b.DPRC_BF16, 8, 4096, 2048, 2048, 32)
    assert ws >= 8 * 64 * 4096 * 2
    assert ws < 64 << 20
    # float32 path
    ws32 = b.dprc_workspace_bytes(b.DPRC_OP_HUTCH, b.DPRC_F32, 4, 128, 64, 64, 8)
    assert ws32 >= 4 * 128 * 8 * 4
    assert b.dprc_workspace_bytes(b.DPRC_OP_HUTCHPP, b.DPRC_BF16, 8, 4096, 2048, 2048, 16) > 0
    # exact norm: bf16 with aligned widths runs both forms on tensor cores
    # (one fp32 partial per 128 x 256 tile of A^T G, or per 128-token row
    # block and span of the ghost form: T (T + 1) / 2 blocks of 128 for
    # single-block spans); fp32 or odd widths the ghost form on CUDA cores (one
    # partial per pair of 32-token tiles)
    assert b.dprc_workspace_bytes(b.DPRC_OP_EXACT, b.DPRC_BF16, 2, 4096, 2048, 2048, 0) >= 2 * 16 * 8 * 4
    assert b.dprc_workspace_bytes(b.DPRC_OP_EXACT, b.DPRC_BF16, 2, 4096, 2048, 2048, 0) >= 2 * 32 * 33 // 2 * 4
    assert b.dprc_workspace_bytes(b.DPRC_OP_EXACT, b.DPRC_BF16, 3, 1000, 64, 16, 0) >= 3 * 8 * 9 // 2 * 4
    assert b.dprc_workspace_bytes(b.DPRC_OP_EXACT, b.DPRC_F32, 2, 4096, 64, 64, 0) >= 2 * 128 * 128 * 4
    assert b.dprc_workspace_bytes(b.DPRC_OP_EXACT, b.DPRC_BF16, 2, 4096, 63, 64, 0) >= 2 * 128 * 128 * 4
    # host-input stage: a chunk's workspace, P and two slots of a chunk each (four
    # 33.5 MB samples make the 128 MB chunk)
    hs = b.dprc_workspace_bytes(b.DPRC_OP_HUTCH_HOST, b.DPRC_BF16, 8, 4096, 2048, 2048, 32)
    four = b.dprc_workspace_bytes(b.DPRC_OP_HUTCH, b.DPRC_BF16, 4, 4096, 2048, 2048, 32)
    assert hs >= four + 2 * 4 * 4096 * 4096 * 2 + 2048 * 32 * 2
    assert hs < four + 2 * 4 * 4096 * 4096 * 2 + (1 << 20)
    # small samples go 4 (or a multiple of 4) to a chunk
    assert (b.dprc_workspace_bytes(b.DPRC_OP_HUTCH_HOST, b.DPRC_BF16, 64, 128, 256, 256, 16)
            >= 2 * 64 * 128 * 512 * 2)
    # invalid sizes give 0
    assert b.dprc_workspace_bytes(b.DPRC_OP_HUTCH_HOST, b.DPRC_BF16, 8, 4096, 2048, 2048, 0) == 0
    assert b.dprc_workspace_bytes(b.DPRC_OP_HUTCH, b.DPRC_BF16, 0, 4096, 2048, 2048, 32) == 0
    assert b.dprc_workspace_bytes(b.DPRC_OP_HUTCH, b.DPRC_BF16, 1, 4096, 2048, 2048, 0) == 0
    assert b.dprc_workspace_bytes(b.DPRC_OP_HUTCH, b.DPRC_BF16, 1, 4096, 2048, 2048, 257) == 0
    assert b.dprc_workspace_bytes(b.DPRC_OP_HUTCHPP, b.DPRC_BF16, 1, 64, 64, 8, 16) == 0  # r > p
    assert b.dprc_workspace_bytes(b.DPRC_OP_HUTCH, 7, 1, 64, 64, 64, 8) == 0
    assert b.dprc_workspace_bytes(9, b.DPRC_BF16, 1, 64, 64, 64, 8) == 0


def _vp(x):
    return ctypes.c_void_p(x)


A16 = 0x10000  # fake, aligned, never dereferenced: every call below fails its checks first


def test_argument_errors_return_before_device_work(lib):
    f = lib.dprc_norm_hutch
    ws = 1 << 30
    # null pointers
    assert f(None, _vp(A16), _vp(A16), 1, 1, 1, 8, 8, 16, _vp(A16), 0, _vp(A16), ws, None) == 1
    assert f(_vp(A16), _vp(A16), _vp(A16), 1, 1, 1, 8, 8, 16, None, 0, _vp(A16), ws, None) == 1
    # bad dtype, bad shapes
    assert f(_vp(A16), _vp(A16), _vp(A16), 5, 1, 1, 8, 8, 16, _vp(A16), 0, _vp(A16), ws, None) == 3
    assert f(_vp(A16), _vp(A16), _vp(A16), 1, 0, 1, 8, 8, 16, _vp(A16), 0, _vp(A16), ws, None) == 2
    assert f(_vp(A16), _vp(A16), _vp(A16), 1, 1, -3, 8, 8, 16, _vp(A16), 0, _vp(A16), ws, None) == 2
    assert f(_vp(A16), _vp(A16), _vp(A16), 1, 1, 1, 8, 8, 0, _vp(A16), 0, _vp(A16), ws, None) == 2
    assert f(_vp(A16), _vp(A16), _vp(A16), 1, 1, 1, 8, 8, 300, _vp(A16), 0, _vp(A16), ws, None) == 2
    # misaligned pointer
    assert f(_vp(A16 + 2), _vp(A16), _vp(A16), 1, 1, 1, 8, 8, 16, _vp(A16), 0, _vp(A16), ws, None) == 4
    assert f(_vp(A16), _vp(A16), _vp(A16), 1, 1, 1, 8, 8, 16, _vp(A16), 0, _vp(A16 + 8), ws, None) == 4
    # missing workspace
    assert f(_vp(A16), _vp(A16), _vp(A16), 1, 1, 1, 8, 8, 16, _vp(A16), 0, None, ws, None) == 5
    g = lib.dprc_norm_hutchpp
    assert g(_vp(A16), _vp(A16), None, _vp(A16), 1, 1, 1, 8, 8, 4, _vp(A16), 0, _vp(A16), ws, None) == 1
    assert g(_vp(A16), _vp(A16), _vp(A16), _vp(A16), 1, 1, 1, 8, 8, 16, _vp(A16), 0, _vp(A16), ws, None) == 2
    e = lib.dprc_exact_norm
    assert e(_vp(A16), None, 1, 1, 1, 8, 8, _vp(A16), 0, _vp(A16), ws, None) == 1
    assert e(_vp(A16), _vp(A16), 1, 1, 1, 8, 8, _vp(A16), 0, _vp(A16), 0, None) == 5
    hc = lib.dprc_norm_hutch_clip
    f32 = ctypes.c_float
    assert hc(_vp(A16), _vp(A16), _vp(A16), 1, 1, 64, 8, 8, 8, _vp(A16), 0, f32(1.0), None, None,
              _vp(A16), ws, None) == 1  # no c
    assert hc(_vp(A16), _vp(A16), _vp(A16), 1, 1, 64, 8, 8, 8, _vp(A16), 0, f32(0.0), _vp(A16),
              None, _vp(A16), ws, None) == 2  # C <= 0
    assert hc(_vp(A16), _vp(A16), _vp(A16), 1, 1, 64, 8, 8, 8, _vp(A16), 0, f32(1.0), _vp(A16 + 4),
              None, _vp(A16), ws, None) == 4  # misaligned c
    ef = lib.dprc_exact_norm_form
    assert ef(_vp(A16), _vp(A16), 1, 1, 1, 8, 8, 5, _vp(A16), 0, _vp(A16), ws, None) == 2  # form
    assert ef(_vp(A16), _vp(A16), 0, 1, 1, 8, 8, 3, _vp(A16), 0, _vp(A16), ws, None) == 2
    # the direct form needs bf16 rows of 16-byte multiples
    assert ef(_vp(A16), _vp(A16), 0, 1, 1, 8, 8, 1, _vp(A16), 0, _vp(A16), ws, None) == 2
    assert ef(_vp(A16), _vp(A16), 1, 1, 1, 12, 8, 1, _vp(A16), 0, _vp(A16), ws, None) == 2
    # the tensor-core ghost form stops at T = 65536
    assert ef(_vp(A16), _vp(A16), 1, 1, 65537, 8, 8, 2, _vp(A16), 0, _vp(A16), ws, None) == 2
    assert ef(_vp(A16), _vp(A16), 1, 1, 64, 8, 8, 2, _vp(A16), 0, _vp(A16), 0, None) == 5
    assert lib.dprc_exact_norm_plan(1, 1, 64, 8, 8, 5) == 0
    c = lib.dprc_clip_factors
    assert c(None, 4, ctypes.c_float(1.0), _vp(A16), None, None) == 1
    assert c(_vp(A16), 4, ctypes.c_float(0.0), _vp(A16), None, None) == 2
    assert c(_vp(A16), 4, ctypes.c_float(float("nan")), _vp(A16), None, None) == 2
    assert c(_vp(A16), 0, ctypes.c_float(1.0), _vp(A16), None, None) == 2
    n = lib.dprc_add_noise
    assert n(None, 10, ctypes.c_float(1.0), ctypes.c_float(1.0), 1, 1, None) == 1
    assert n(_vp(A16), -1, ctypes.c_float(1.0), ctypes.c_float(1.0), 1, 1, None) == 2
    assert n(_vp(A16 + 4), 10, ctypes.c_float(1.0), ctypes.c_float(1.0), 1, 1, None) == 4
    assert n(_vp(A16), 10, ctypes.c_float(-1.0), ctypes.c_float(1.0), 1, 1, None) == 2
    assert n(None, 0, ctypes.c_float(1.0), ctypes.c_float(1.0), 1, 1, None) == 0  # empty: no-op
    L2 = ctypes.c_void_p * 2
    I2 = ctypes.c_int64 * 2
    ptrs, bad = L2(A16, A16), L2(A16, A16 + 2)
    sizes = I2(8, 8)
    hl = lib.dprc_norm_hutch_layers
    assert hl(2, None, ptrs, ptrs, sizes, sizes, 1, 1, 1, 16, _vp(A16), 0, _vp(A16), ws, None) == 1
    assert hl(0, ptrs, ptrs, ptrs, sizes, sizes, 1, 1, 1, 16, _vp(A16), 0, _vp(A16), ws, None) == 2
    assert hl(2, ptrs, bad, ptrs, sizes, sizes, 1, 1, 1, 16, _vp(A16), 0, _vp(A16), ws, None) == 4
    assert hl(2, ptrs, ptrs, ptrs, I2(8, 0), sizes, 1, 1, 1, 16, _vp(A16), 0, _vp(A16), ws, None) == 2
    assert hl(2, ptrs, ptrs, ptrs, sizes, sizes, 1, 1, 1, 16, _vp(A16), 0, _vp(A16), 16, None) == 5
    hh = lib.dprc_norm_hutch_clip_host
    big = 1 << 40
    assert hh(_vp(A16), None, _vp(A16), 1, 2, 64, 8, 8, 8, f32(1.0), _vp(A16), _vp(A16),
              _vp(A16), big, None) == 1  # no G
    assert hh(_vp(A16), _vp(A16), _vp(A16), 1, 2, 64, 8, 8, 8, f32(1.0), _vp(A16), None,
              _vp(A16), big, None) == 1  # no c
    assert hh(_vp(A16), _vp(A16), _vp(A16), 1, 2, 64, 8, 8, 0, f32(1.0), _vp(A16), _vp(A16),
              _vp(A16), big, None) == 2  # k = 0
    assert hh(_vp(A16), _vp(A16), _vp(A16), 1, 2, 64, 8, 8, 8, f32(float("inf")), _vp(A16),
              _vp(A16), _vp(A16), big, None) == 2  # C not finite
    assert hh(_vp(A16), _vp(A16), _vp(A16), 1, 2, 64, 8, 8, 8, f32(1.0), _vp(A16), _vp(A16),
              _vp(A16 + 8), big, None) == 4  # misaligned stage
    assert hh(_vp(A16), _vp(A16), _vp(A16), 1, 2, 64, 8, 8, 8, f32(1.0), _vp(A16), _vp(A16),
              None, big, None) == 5  # no stage
    assert hh(_vp(A16), _vp(A16), _vp(A16), 1, 2, 64, 8, 8, 8, f32(1.0), _vp(A16), _vp(A16),
              _vp(A16), 1024, None) == 5  # stage too small
    na_ = lib.dprc_add_noise_at
    one = ctypes.c_float(1.0)
    assert na_(_vp(A16), 5, 10, 0, one, one, 1, 1, None) == 3            # unknown dtype
    assert na_(None, 0, 10, 0, one, one, 1, 1, None) == 1                 # no gradient
    assert na_(_vp(A16 + 4), 1, 10, 0, one, one, 1, 1, None) == 4         # misaligned
    assert na_(_vp(A16), 0, 10, 2**64 - 5, one, one, 1, 1, None) == 2     # range wraps
    assert na_(_vp(A16), 0, 10, 0, ctypes.c_float(-1.0), one, 1, 1, None) == 2
    assert na_(None, 1, 0, 123, one, one, 1, 1, None) == 0                # empty: no-op
    w = lib.dprc_philox_words
    assert w(None, 4, 0, 1, 1, None) == 1
    assert w(None, 0, 0, 1, 1, None) == 0
    na = lib.dprc_norm_hutch_noalloc
    assert na(None, _vp(A16), _vp(A16), 1, 1, 64, 8, 8, 8, _vp(A16), 0, None) == 1
    assert na(_vp(A16), _vp(A16), _vp(A16), 1, 1, 64, 8, 8, 0, _vp(A16), 0, None) == 2
    assert na(_vp(A16), _vp(A16 + 2), _vp(A16), 1, 1, 64, 8, 8, 8, _vp(A16), 0, None) == 4
    # beyond the built-in scratch: refused before any device is needed
    assert na(_vp(A16), _vp(A16), _vp(A16), 1, 64, 32768, 8192, 8192, 32, _vp(A16), 0,
              None) == 9
    tf = lib.dprc_test_hutch_fault
    one = ctypes.c_void_p * 1
    p1, s1 = one(A16), (ctypes.c_int64 * 1)(256)
    args = (1, p1, p1, p1, s1, s1, 2, 256, 32, _vp(A16), _vp(A16), big, None)
    assert tf(0, 1000000, *args[:1], None, *args[2:]) == 1       # no A list
    assert tf(7, 1000000, *args) == 2                            # unknown mode
    assert tf(0, 10, *args) == 2                                 # wait limit too short
    assert tf(0, 3000000000, *args) == 2                         # beyond the kernels' own limit
    assert tf(0, 1000000, 57, *args[1:]) == 2                    # more layers than one launch
    assert tf(0, 1000000, *args[:8], 64, *args[9:]) == 2         # k not 16 or 32
    assert tf(0, 1000000, *args[:1], one(A16 + 2), *args[2:]) == 4  # misaligned A
    assert tf(0, 1000000, *args[:10], None, big, None) == 5      # no workspace


def test_valid_calls_without_a_gpu_fail_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = lib.dprc_norm_hutch(_vp(A16), _vp(A16), _vp(A16), 1, 1, 1, 8, 8, 16, _vp(A16), 0,
                             _vp(A16), 1 << 30, None)
    assert st == 8  # DPRC_ERR_DEVICE: nothing was launched
    st = lib.dprc_norm_hutch_noalloc(_vp(A16), _vp(A16), _vp(A16), 1, 1, 64, 8, 8, 8, _vp(A16),
                                     0, None)
    assert st == 8  # the device check comes before the scratch lookup
    # the launch-count query enqueues nothing and reports 0 without a device
    assert lib.dprc_norm_hutch_launches(1, 8, 4096, 2048, 2048, 32) == 0
    assert lib.dprc_norm_hutchpp_launches(1, 8, 4096, 2048, 2048, 16) == 0


def test_launch_count_query_rejects_bad_arguments(lib):
    q = lib.dprc_norm_hutch_launches
    assert q(5, 8, 4096, 2048, 2048, 32) == 0   # unknown dtype
    assert q(1, 0, 4096, 2048, 2048, 32) == 0   # empty batch
    assert q(1, 8, 4096, 2048, 2048, 0) == 0    # k = 0
    assert q(1, 8, 4096, 2048, 2048, 300) == 0  # k > 256
    q = lib.dprc_norm_hutchpp_launches
    assert q(5, 8, 4096, 2048, 2048, 16) == 0   # unknown dtype
    assert q(1, 8, 4096, 2048, 2048, 0) == 0    # r = 0
    assert q(1, 8, 4096, 2048, 2048, 65) == 0   # r > 64
    assert q(1, 8, 4096, 2048, 16, 32) == 0     # r > p


def test_binding_raises_when_library_missing(monkeypatch, tmp_path):
    from randomized_norm_clipping_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()
