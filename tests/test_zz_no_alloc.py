"""The allocation-free Hutchinson entry point (dprc_norm_hutch_noalloc).

It serves callers that cannot allocate device memory where they need the
norm; its scratch is a fixed array inside the library.  Checked through the C
ABI against dprc_norm_hutch on the same inputs, on calls in a row with other
sizes (larger after smaller and smaller after larger, so the array's leftover
contents must not matter) and with accumulate set on repeated calls.
This file is collected last so a failure here cannot hide another test.
"""

import ctypes
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

RTOL = 1e-3
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    from randomized_norm_clipping_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding.lib()


def _case(B, T, d, p, k, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    A = torch.randn(B, T, d, generator=g).to(torch.bfloat16).to(DEV)
    G = (torch.randn(B, T, p, generator=g) * 0.05).to(torch.bfloat16).to(DEV)
    P = (torch.randn(p, k, generator=g) / k ** 0.5).to(torch.bfloat16).to(DEV)
    return A, G, P


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, A, G, P, n, accumulate=0):
    B, T, d = A.shape
    p, k = P.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.dprc_norm_hutch_noalloc(_vp(A), _vp(G), _vp(P), 1, B, T, d, p, k, _vp(n),
                                       accumulate, stream)


def _with_workspace(lib, A, G, P, n):
    B, T, d = A.shape
    p, k = P.shape
    nbytes = lib.dprc_workspace_bytes(1, 1, B, T, d, p, k)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.dprc_norm_hutch(_vp(A), _vp(G), _vp(P), 1, B, T, d, p, k, _vp(n), 0, _vp(ws),
                             nbytes, stream)
    torch.cuda.synchronize()
    return st


def test_noalloc_matches_workspace_entry_on_two_calls(lib):
    for shape, seed in (((4, 1000, 512, 768, 32), 1), ((8, 4096, 2048, 2048, 32), 2)):
        A, G, P = _case(*shape, seed)
        n_ref = torch.zeros(shape[0], device=DEV)
        n_new = torch.full((shape[0],), -1.0, device=DEV)
        assert _with_workspace(lib, A, G, P, n_ref) == 0
        assert _noalloc(lib, A, G, P, n_new) == 0
        torch.cuda.synchronize()
        ref = n_ref.cpu().double().numpy()
        got = n_new.cpu().double().numpy()
        assert np.all(np.abs(got - ref) <= RTOL * np.abs(ref)), (got, ref)


def test_noalloc_small_after_large_and_accumulate(lib):
    # the array keeps the last call's contents: a smaller call after a larger
    # one (other sketch stride and offsets) must not see them, and two calls
    # in a row with accumulate = 1 must add on the caller's n
    big = (8, 4096, 2048, 2048, 32)
    Ab, Gb, Pb = _case(*big, 3)
    nb = torch.zeros(big[0], device=DEV)
    assert _noalloc(lib, Ab, Gb, Pb, nb) == 0
    small = (4, 1000, 512, 768, 32)
    A, G, P = _case(*small, 4)
    n_ref = torch.zeros(small[0], device=DEV)
    assert _with_workspace(lib, A, G, P, n_ref) == 0
    ref = n_ref.cpu().double().numpy()
    n_new = torch.full((small[0],), -1.0, device=DEV)
    assert _noalloc(lib, A, G, P, n_new, accumulate=0) == 0
    torch.cuda.synchronize()
    got = n_new.cpu().double().numpy()
    assert np.all(np.abs(got - ref) <= RTOL * np.abs(ref)), (got, ref)
    for times in (2, 3):
        assert _noalloc(lib, A, G, P, n_new, accumulate=1) == 0
        torch.cuda.synchronize()
        got = n_new.cpu().double().numpy()
        assert np.all(np.abs(got - times * ref) <= RTOL * times * np.abs(ref)), (times, got, ref)


def test_noalloc_rejects_calls_beyond_its_scratch(lib):
    # B = 64, T = 32768, d = p = 8192: the sketch alone needs 256 MiB
    A16 = ctypes.c_void_p(0x10000)
    st = lib.dprc_norm_hutch_noalloc(A16, A16, A16, 1, 64, 32768, 8192, 8192, 32, A16, 0, None)
    assert st == 9  # DPRC_ERR_TOO_LARGE, returned before any device work
