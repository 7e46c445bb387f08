"""ctypes binding of libdprc (include/dprc.h): argument marshalling only.

Every function here takes torch tensors for device memory, passes their data
pointers and the current CUDA stream to the C ABI of the same name, and raises
``DprcError`` on a non-zero status.  All arithmetic runs in the library's
kernels; there is no fallback of any kind: if libdprc.so is missing, loading
raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
# DPRC_LIBRARY=debug loads the bounds-checked build (libdprc_debug.so: every
# computed index checked before its access, failures recorded in the device
# error word as DPRC_DEVERR_BOUNDS); anything else, the release build.
LIB_PATH = os.path.join(
    PKG_DIR, "libdprc_debug.so" if os.environ.get("DPRC_LIBRARY") == "debug" else "libdprc.so")

DPRC_F32, DPRC_BF16 = 0, 1
(DPRC_OP_HUTCH, DPRC_OP_HUTCHPP, DPRC_OP_EXACT, DPRC_OP_HUTCH_LAYERS, DPRC_OP_HUTCH_PM1,
 DPRC_OP_HUTCH_HOST) = (1, 2, 3, 4, 5, 6)
(DPRC_EXACT_AUTO, DPRC_EXACT_DIRECT, DPRC_EXACT_GHOST, DPRC_EXACT_GHOST_N128,
 DPRC_EXACT_GHOST_N256) = (0, 1, 2, 3, 4)
STATUS = {0: "ok", 1: "null pointer", 2: "shape", 3: "dtype", 4: "alignment",
          5: "workspace", 6: "cuda", 7: "non-finite", 8: "device", 9: "too large"}

# The C prototypes of include/dprc.h, as (name, restype, argtypes).
_c = ctypes
_PROTOS = [
    ("dprc_abi_version", _c.c_int, []),
    ("dprc_status_string", _c.c_char_p, [_c.c_int]),
    ("dprc_workspace_bytes", _c.c_size_t,
     [_c.c_int, _c.c_int, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64]),
    ("dprc_norm_hutch", _c.c_int,
     [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64, _c.c_int64,
      _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    ("dprc_norm_hutchpp", _c.c_int,
     [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64,
      _c.c_int64, _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_size_t,
      _c.c_void_p]),
    ("dprc_exact_norm", _c.c_int,
     [_c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64,
      _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    ("dprc_clip_factors", _c.c_int,
     [_c.c_void_p, _c.c_int64, _c.c_float, _c.c_void_p, _c.c_void_p, _c.c_void_p]),
    ("dprc_add_noise", _c.c_int,
     [_c.c_void_p, _c.c_int64, _c.c_float, _c.c_float, _c.c_uint64, _c.c_uint64, _c.c_void_p]),
    ("dprc_add_noise_at", _c.c_int,
     [_c.c_void_p, _c.c_int, _c.c_int64, _c.c_uint64, _c.c_float, _c.c_float, _c.c_uint64,
      _c.c_uint64, _c.c_void_p]),
    ("dprc_philox_words", _c.c_int,
     [_c.c_void_p, _c.c_int64, _c.c_uint64, _c.c_uint64, _c.c_uint64, _c.c_void_p]),
    ("dprc_device_error", _c.c_int, [_c.c_void_p, _c.c_int]),
    ("dprc_set_phase_events", _c.c_int, [_c.c_void_p, _c.c_int]),
    ("dprc_norm_hutch_pm1", _c.c_int,
     [_c.c_void_p, _c.c_void_p, _c.c_uint64, _c.c_uint64, _c.c_int, _c.c_int64, _c.c_int64,
      _c.c_int64, _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_size_t,
      _c.c_void_p]),
    ("dprc_norm_hutch_layers", _c.c_int,
     [_c.c_int64, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int,
      _c.c_int64, _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_size_t,
      _c.c_void_p]),
    ("dprc_norm_hutch_layers_clip", _c.c_int,
     [_c.c_int64, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int,
      _c.c_int64, _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_int, _c.c_float, _c.c_void_p,
      _c.c_void_p, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    ("dprc_norm_hutch_launches", _c.c_int,
     [_c.c_int, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64]),
    ("dprc_norm_hutchpp_launches", _c.c_int,
     [_c.c_int, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64]),
    ("dprc_exact_norm_form", _c.c_int,
     [_c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64,
      _c.c_int, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    ("dprc_exact_norm_plan", _c.c_int,
     [_c.c_int, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int]),
    ("dprc_norm_hutch_clip_host", _c.c_int,
     [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64, _c.c_int64,
      _c.c_int64, _c.c_int64, _c.c_float, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_size_t,
      _c.c_void_p]),
    ("dprc_norm_hutch_clip", _c.c_int,
     [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64, _c.c_int64,
      _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_int, _c.c_float, _c.c_void_p, _c.c_void_p,
      _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    ("dprc_norm_hutch_noalloc", _c.c_int,
     [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64, _c.c_int64,
      _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_int, _c.c_void_p]),
    ("dprc_test_hutch_fault", _c.c_int,
     [_c.c_int, _c.c_uint64, _c.c_int64, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
      _c.c_void_p, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_void_p, _c.c_size_t,
      _c.c_void_p]),
]
EXPORTED = tuple(name for name, _, _ in _PROTOS)

_lib = None
_lock = threading.Lock()


class DprcError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed with status {status} ({STATUS.get(status, '?')})")
        self.status = status


def lib():
    """The loaded libdprc (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with `python -c "
                        "\"import __graft_entry__ as g; g.build()\"`")
                h = ctypes.CDLL(LIB_PATH)
                for name, res, args in _PROTOS:
                    f = getattr(h, name)
                    f.restype = res
                    f.argtypes = args
                _lib = h
    return _lib


def _dtype_code(t):
    if t.dtype == torch.float32:
        return DPRC_F32
    if t.dtype == torch.bfloat16:
        return DPRC_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t, stream):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)
    if _raw_stream is not None:  # the current stream's handle without a Stream object
        return ctypes.c_void_p(_raw_stream(t.device.index))
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check(fn, status):
    if status != 0:
        raise DprcError(fn, status)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libdprc takes device tensors")
        if t is not None and not t.is_contiguous():
            raise ValueError("libdprc takes contiguous tensors")


def dprc_abi_version():
    return lib().dprc_abi_version()


def dprc_workspace_bytes(op, dtype_code, B, T, d, p, k):
    return int(lib().dprc_workspace_bytes(op, dtype_code, B, T, d, p, k))


def workspace(op, like, B, T, d, p, k):
    """A zeroed device byte buffer of dprc_workspace_bytes(...) bytes (torch
    allocation).  Workspaces must be zero before their first use; calls leave
    their counter block zero again, so the buffer can be reused."""
    n = dprc_workspace_bytes(op, _dtype_code(like), B, T, d, p, k)
    if n == 0:
        raise DprcError("dprc_workspace_bytes", 2)
    return torch.zeros(n, dtype=torch.uint8, device=like.device)


def dprc_norm_hutch_clip(A, G, P, n, C, c, accumulate=False, nonfinite=None, ws=None,
                         stream=None):
    """n[i] (+)= ||A_i^T (G_i P)||_F^2, then c[i] = min(1, C / sqrt(n[i]))
    (see include/dprc.h)."""
    _need_cuda(A, G, P, n, c, nonfinite)
    B, T, d = A.shape
    p, k = P.shape
    if ws is None:
        ws = workspace(DPRC_OP_HUTCH, A, B, T, d, p, k)
    st = lib().dprc_norm_hutch_clip(_ptr(A), _ptr(G), _ptr(P), _dtype_code(A), B, T, d, p, k,
                                    _ptr(n), int(bool(accumulate)), float(C), _ptr(c),
                                    _ptr(nonfinite) if nonfinite is not None else None,
                                    _ptr(ws), ws.numel(), _stream(A, stream))
    _check("dprc_norm_hutch_clip", st)
    return n, c


def host_stage(A, T, d, p, k, B=None, device=None):
    """A zeroed device stage buffer for dprc_norm_hutch_clip_host with the
    sizes of host tensor A ([B][T][d]) and P [p][k]."""
    B = A.shape[0] if B is None else B
    n = dprc_workspace_bytes(DPRC_OP_HUTCH_HOST, _dtype_code(A), B, T, d, p, k)
    if n == 0:
        raise DprcError("dprc_workspace_bytes", 2)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def dprc_norm_hutch_clip_host(A, G, P, C, n, c, stage=None, stream=None):
    """Host tensors A [B][T][d], G [B][T][p], P [p][k] (pinned for asynchronous
    copies) -> host float32 n, c [B]: n[i] = ||A_i^T (G_i P)||_F^2 and
    c[i] = min(1, C / sqrt(n[i])), copied back at the end of the work enqueued
    on the stream (see include/dprc.h); n may be None.  Synchronise the
    stream before reading n and c."""
    ts = [t for t in (A, G, P, n, c) if t is not None]
    for t in ts:
        if t.is_cuda:
            raise ValueError("dprc_norm_hutch_clip_host takes host tensors")
        if not t.is_contiguous():
            raise ValueError("host tensors must be contiguous")
    if (n is not None and n.dtype != torch.float32) or c.dtype != torch.float32:
        raise ValueError("n and c must be float32")
    B, T, d = A.shape
    p, k = P.shape
    if stage is None:
        stage = host_stage(A, T, d, p, k)
    st = lib().dprc_norm_hutch_clip_host(_ptr(A), _ptr(G), _ptr(P), _dtype_code(A), B, T, d, p, k,
                                         float(C), _ptr(n), _ptr(c), _ptr(stage), stage.numel(),
                                         _stream(stage, stream))
    _check("dprc_norm_hutch_clip_host", st)
    return n, c


def dprc_norm_hutch_pm1(A, G, k, seed, step, n, accumulate=False, ws=None, stream=None):
    """n[i] (+)= (1/k) ||A_i^T (G_i S)||_F^2 with the +-1 projection S of
    (seed, step) (see include/dprc.h)."""
    _need_cuda(A, G, n)
    B, T, d = A.shape
    p = G.shape[2]
    if ws is None:
        ws = workspace(DPRC_OP_HUTCH_PM1, A, B, T, d, p, k)
    st = lib().dprc_norm_hutch_pm1(_ptr(A), _ptr(G), int(seed) & (2**64 - 1),
                                   int(step) & (2**64 - 1), _dtype_code(A), B, T, d, p, k,
                                   _ptr(n), int(bool(accumulate)), _ptr(ws), ws.numel(),
                                   _stream(A, stream))
    _check("dprc_norm_hutch_pm1", st)
    return n


def dprc_norm_hutch_layers(As, Gs, Ps, n, accumulate=False, ws=None, stream=None, C=None,
                           c=None, nonfinite=None):
    """n[i] (+)= sum_l ||A_l,i^T (G_l,i P_l)||_F^2 over the layers (see
    include/dprc.h); with C and c also c[i] = min(1, C / sqrt(n[i])) of the sum
    (dprc_norm_hutch_layers_clip)."""
    if (C is None) != (c is None):
        raise ValueError("give both C and c, or neither")
    L = len(As)
    if not (L == len(Gs) == len(Ps)) or L == 0:
        raise ValueError("As, Gs and Ps must be non-empty lists of the same length")
    _need_cuda(*As, *Gs, *Ps, n)
    B, T = As[0].shape[0], As[0].shape[1]
    k = Ps[0].shape[1]
    d = (ctypes.c_int64 * L)(*[a.shape[2] for a in As])
    p = (ctypes.c_int64 * L)(*[g.shape[2] for g in Gs])
    ap = (ctypes.c_void_p * L)(*[_ptr(a) for a in As])
    gp = (ctypes.c_void_p * L)(*[_ptr(g) for g in Gs])
    pp = (ctypes.c_void_p * L)(*[_ptr(x) for x in Ps])
    if ws is None:
        ws = workspace(DPRC_OP_HUTCH_LAYERS, As[0], B, T, max(d), max(p), k)
    if C is None:
        st = lib().dprc_norm_hutch_layers(L, ap, gp, pp, d, p, _dtype_code(As[0]), B, T, k,
                                          _ptr(n), int(bool(accumulate)), _ptr(ws), ws.numel(),
                                          _stream(As[0], stream))
        _check("dprc_norm_hutch_layers", st)
        return n
    _need_cuda(c, nonfinite)
    st = lib().dprc_norm_hutch_layers_clip(L, ap, gp, pp, d, p, _dtype_code(As[0]), B, T, k,
                                           _ptr(n), int(bool(accumulate)), float(C), _ptr(c),
                                           _ptr(nonfinite) if nonfinite is not None else None,
                                           _ptr(ws), ws.numel(), _stream(As[0], stream))
    _check("dprc_norm_hutch_layers_clip", st)
    return n, c


def dprc_norm_hutch_launches(dtype_code, B, T, d, p, k):
    """Kernels one dprc_norm_hutch call with these sizes enqueues on the
    current device (1 fused, 2 sketch + projection, 3 CUDA cores; 0 invalid)."""
    return int(lib().dprc_norm_hutch_launches(dtype_code, B, T, d, p, k))


def dprc_norm_hutchpp_launches(dtype_code, B, T, d, p, r):
    """Kernels one dprc_norm_hutchpp call with these sizes enqueues on the
    current device (5 with passes 1 and 2 fused, 7 or 8 otherwise; 0 invalid)."""
    return int(lib().dprc_norm_hutchpp_launches(dtype_code, B, T, d, p, r))


def dprc_norm_hutch(A, G, P, n, accumulate=False, ws=None, stream=None):
    """n[i] (+)= ||A_i^T (G_i P)||_F^2 (see include/dprc.h)."""
    _need_cuda(A, G, P, n)
    B, T, d = A.shape
    p, k = P.shape
    if ws is None:
        ws = workspace(DPRC_OP_HUTCH, A, B, T, d, p, k)
    st = lib().dprc_norm_hutch(_ptr(A), _ptr(G), _ptr(P), _dtype_code(A), B, T, d, p, k,
                               _ptr(n), int(bool(accumulate)), _ptr(ws), ws.numel(),
                               _stream(A, stream))
    _check("dprc_norm_hutch", st)
    return n


def dprc_norm_hutchpp(A, G, S, P, n, accumulate=False, ws=None, stream=None):
    """n[i] (+)= Hutch++ head + tail / r (see include/dprc.h)."""
    _need_cuda(A, G, S, P, n)
    B, T, d = A.shape
    p, r = P.shape
    if ws is None:
        ws = workspace(DPRC_OP_HUTCHPP, A, B, T, d, p, r)
    st = lib().dprc_norm_hutchpp(_ptr(A), _ptr(G), _ptr(S), _ptr(P), _dtype_code(A), B, T, d, p,
                                 r, _ptr(n), int(bool(accumulate)), _ptr(ws), ws.numel(),
                                 _stream(A, stream))
    _check("dprc_norm_hutchpp", st)
    return n


def dprc_norm_hutch_noalloc(A, G, P, n, accumulate=False, stream=None):
    """dprc_norm_hutch with the library's built-in scratch instead of a workspace,
    for callers that cannot allocate device memory (see include/dprc.h)."""
    _need_cuda(A, G, P, n)
    B, T, d = A.shape
    p, k = P.shape
    st = lib().dprc_norm_hutch_noalloc(_ptr(A), _ptr(G), _ptr(P), _dtype_code(A), B, T, d, p, k,
                                       _ptr(n), int(bool(accumulate)), _stream(A, stream))
    _check("dprc_norm_hutch_noalloc", st)
    return n


# Device error codes (DPRC_DEVERR_* of include/dprc.h).
(DPRC_DEVERR_PIPE_FULL, DPRC_DEVERR_PIPE_EMPTY, DPRC_DEVERR_ACCUM, DPRC_DEVERR_CLUSTER,
 DPRC_DEVERR_READY, DPRC_DEVERR_LAUNCH, DPRC_DEVERR_BOUNDS) = (1, 2, 3, 4, 5, 6, 7)
FAULT_READY_NEVER_MET, FAULT_CLUSTER_SHAPE = 0, 1


def dprc_test_hutch_fault(mode, wait_ns, As, Gs, Ps, n, ws, stream=None):
    """Failure-detection test of the one-launch Hutchinson kernel (see
    include/dprc.h): mode FAULT_READY_NEVER_MET makes every projection's wait
    for its sample's sketch run out after wait_ns; mode FAULT_CLUSTER_SHAPE
    launches a plan without clusters as clusters of 2.  Read the outcome with
    dprc_device_error(reset=True)."""
    L = len(As)
    if not (L == len(Gs) == len(Ps)) or L == 0:
        raise ValueError("As, Gs and Ps must be non-empty lists of the same length")
    _need_cuda(*As, *Gs, *Ps, n, ws)
    B, T = As[0].shape[0], As[0].shape[1]
    k = Ps[0].shape[1]
    d = (ctypes.c_int64 * L)(*[a.shape[2] for a in As])
    p = (ctypes.c_int64 * L)(*[g.shape[2] for g in Gs])
    ap = (ctypes.c_void_p * L)(*[_ptr(a) for a in As])
    gp = (ctypes.c_void_p * L)(*[_ptr(g) for g in Gs])
    pp = (ctypes.c_void_p * L)(*[_ptr(x) for x in Ps])
    st = lib().dprc_test_hutch_fault(int(mode), int(wait_ns), L, ap, gp, pp, d, p, B, T, k,
                                     _ptr(n), _ptr(ws), ws.numel(), _stream(As[0], stream))
    _check("dprc_test_hutch_fault", st)
    return n


def dprc_exact_norm(A, G, n, accumulate=False, ws=None, stream=None, form=DPRC_EXACT_AUTO):
    """n[i] (+)= ||A_i^T G_i||_F^2 exactly, by the direct form A_i^T G_i or the
    ghost form sum_{t,s} (A_i A_i^T)_{ts} (G_i G_i^T)_{ts} (form: one of
    DPRC_EXACT_*; AUTO takes the one with less work, see include/dprc.h)."""
    _need_cuda(A, G, n)
    B, T, d = A.shape
    p = G.shape[2]
    if ws is None:
        ws = workspace(DPRC_OP_EXACT, A, B, T, d, p, 0)
    if form == DPRC_EXACT_AUTO:
        st = lib().dprc_exact_norm(_ptr(A), _ptr(G), _dtype_code(A), B, T, d, p, _ptr(n),
                                   int(bool(accumulate)), _ptr(ws), ws.numel(),
                                   _stream(A, stream))
        _check("dprc_exact_norm", st)
    else:
        st = lib().dprc_exact_norm_form(_ptr(A), _ptr(G), _dtype_code(A), B, T, d, p, int(form),
                                        _ptr(n), int(bool(accumulate)), _ptr(ws), ws.numel(),
                                        _stream(A, stream))
        _check("dprc_exact_norm_form", st)
    return n


def dprc_exact_norm_plan(dtype, B, T, d, p, form=DPRC_EXACT_AUTO):
    """The form (DPRC_EXACT_DIRECT, _GHOST_N128 or _GHOST_N256 on tensor cores,
    _GHOST on CUDA cores) an exact-norm call with these sizes runs on the
    current device, 0 if it would be rejected."""
    code = dtype if isinstance(dtype, int) else _dtype_code(torch.empty(0, dtype=dtype))
    return lib().dprc_exact_norm_plan(code, B, T, d, p, int(form))


def dprc_clip_factors(n, C, c, nonfinite=None, stream=None):
    """c[i] = min(1, C / sqrt(n[i])); non-finite or negative n gives 0."""
    _need_cuda(n, c, nonfinite)
    st = lib().dprc_clip_factors(_ptr(n), n.numel(), float(C), _ptr(c), _ptr(nonfinite),
                                 _stream(n, stream))
    _check("dprc_clip_factors", st)
    return c


def dprc_add_noise(grad, sigma, C, seed, step, stream=None):
    """grad += sigma * C * z (Philox4x32-10 + Box-Muller), in place."""
    _need_cuda(grad)
    st = lib().dprc_add_noise(_ptr(grad), grad.numel(), float(sigma), float(C),
                              int(seed) & (2**64 - 1), int(step) & (2**64 - 1),
                              _stream(grad, stream))
    _check("dprc_add_noise", st)
    return grad


def dprc_add_noise_at(grad, first_element, sigma, C, seed, step, stream=None):
    """grad += sigma * C * z[first_element : first_element + grad.numel()], in
    place (float32 or bfloat16): the noise of one piece of a gradient kept in
    several buffers (see include/dprc.h)."""
    _need_cuda(grad)
    st = lib().dprc_add_noise_at(_ptr(grad), _dtype_code(grad), grad.numel(),
                                 int(first_element) & (2**64 - 1), float(sigma), float(C),
                                 int(seed) & (2**64 - 1), int(step) & (2**64 - 1),
                                 _stream(grad, stream))
    _check("dprc_add_noise_at", st)
    return grad


def dprc_philox_words(out, first_block, seed, step, stream=None):
    """Fills out (int32 [n, 4]) with Philox blocks first_block .. first_block + n - 1."""
    _need_cuda(out)
    n_blocks = out.numel() // 4
    st = lib().dprc_philox_words(_ptr(out), n_blocks, int(first_block), int(seed) & (2**64 - 1),
                                 int(step) & (2**64 - 1), _stream(out, stream))
    _check("dprc_philox_words", st)
    return out


def dprc_device_error(reset=False):
    v = ctypes.c_int32(0)
    st = lib().dprc_device_error(ctypes.byref(v), int(bool(reset)))
    _check("dprc_device_error", st)
    return v.value


_events_keepalive = None


def dprc_set_phase_events(events):
    """Record these torch.cuda.Event objects between the stages of later calls
    on this thread (None turns it off)."""
    global _events_keepalive
    if not events:
        _events_keepalive = None
        _check("dprc_set_phase_events", lib().dprc_set_phase_events(None, 0))
        return
    for e in events:
        if not e.cuda_event:  # torch creates the event on its first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _events_keepalive = (arr, events)
    _check("dprc_set_phase_events", lib().dprc_set_phase_events(arr, len(events)))
