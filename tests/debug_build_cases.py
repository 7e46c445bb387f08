"""Small odd shapes through every kernel family of the bounds-checked build.

Run as a child process by tests/test_gpu_debug_build.py with
DPRC_LIBRARY=debug, so the binding loads libdprc_debug.so (every computed
global or distributed-shared-memory index checked before its access; a failed
check is recorded as DPRC_DEVERR_BOUNDS with its source line, and the access
skipped).  Each case is compared with the float64 oracle; the last line
printed is a JSON object with the worst relative error per case and the
device error word at the end.
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from randomized_norm_clipping_gb300 import binding as rnc  # noqa: E402
from randomized_norm_clipping_gb300.workloads import to_f64  # noqa: E402

DEV = "cuda:0"


def _inputs(seed, B, T, d, p, dtype=torch.bfloat16):
    g = torch.Generator(device="cpu").manual_seed(seed)
    A = torch.randn(B, T, d, generator=g).to(dtype)
    G = (torch.randn(B, T, p, generator=g) * 0.1).to(dtype)
    return A, G


def _proj(seed, p, k, dtype=torch.bfloat16, scale=None):
    g = torch.Generator(device="cpu").manual_seed(seed)
    s = (1.0 / k ** 0.5) if scale is None else scale
    return (torch.randn(p, k, generator=g) * s).to(dtype)


def _rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-300)))


def main():
    assert rnc.LIB_PATH.endswith("libdprc_debug.so"), rnc.LIB_PATH
    rnc.dprc_device_error(reset=True)
    out = {}

    # one-launch Hutchinson: clusters of 2 (split blocks), and a ragged shape
    for name, (B, T, d, p) in {"fused_clusters": (3, 200, 320, 256),
                               "fused_ragged": (2, 130, 136, 264)}.items():
        A, G = _inputs(1, B, T, d, p)
        P = _proj(2, p, 32)
        n = torch.zeros(B, device=DEV)
        c = torch.empty(B, device=DEV)
        rnc.dprc_norm_hutch_clip(A.to(DEV), G.to(DEV), P.to(DEV), n, 1.0, c)
        ref = oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))
        out[name] = max(_rel(n.cpu(), ref), _rel(c.cpu(), oracle.clip_factors(ref, 1.0)))

    # many layers in one launch, mixed widths (clusters of 4 and whole blocks)
    dims = [(256, 512), (512, 256), (384, 384), (136, 72)]
    As, Gs, Ps, refs = [], [], [], []
    for j, (d, p) in enumerate(dims):
        A, G = _inputs(10 + j, 2, 260, d, p)
        P = _proj(20 + j, p, 32)
        As.append(A.to(DEV))
        Gs.append(G.to(DEV))
        Ps.append(P.to(DEV))
        refs.append(oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P)))
    n = torch.zeros(2, device=DEV)
    rnc.dprc_norm_hutch_layers(As, Gs, Ps, n)
    out["layers"] = _rel(n.cpu(), oracle.layer_sum(refs))

    # the two-kernel path (k = 64), the +-1 projection, Hutch++
    A, G = _inputs(3, 2, 333, 200, 152)
    P = _proj(4, 152, 64)
    n = torch.zeros(2, device=DEV)
    rnc.dprc_norm_hutch(A.to(DEV), G.to(DEV), P.to(DEV), n)
    out["two_kernel_k64"] = _rel(n.cpu(), oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P)))

    A, G = _inputs(5, 3, 200, 320, 256)
    n = torch.zeros(3, device=DEV)
    rnc.dprc_norm_hutch_pm1(A.to(DEV), G.to(DEV), 32, 7, 3, n)
    S = oracle.rademacher_signs(7, 3, 256, 32)
    out["pm1"] = _rel(n.cpu(), oracle.hutch_norm_rademacher(to_f64(A), to_f64(G), S))

    A, G = _inputs(6, 2, 257, 136, 264)
    S, P = _proj(7, 264, 16, scale=1.0), _proj(8, 264, 16, scale=1.0)
    n = torch.zeros(2, device=DEV)
    rnc.dprc_norm_hutchpp(A.to(DEV), G.to(DEV), S.to(DEV), P.to(DEV), n)
    out["hutchpp"] = _rel(n.cpu(), oracle.hutchpp_norm(to_f64(A), to_f64(G), to_f64(S),
                                                       to_f64(P)))

    # narrow layers in both orientations (estimate and exact norm)
    for name, (d, p) in {"narrow_p16": (520, 16), "narrow_d16": (16, 520)}.items():
        A, G = _inputs(9, 3, 270, d, p)
        P = _proj(10, p, 32)
        n = torch.zeros(3, device=DEV)
        rnc.dprc_norm_hutch(A.to(DEV), G.to(DEV), P.to(DEV), n)
        e = torch.zeros(3, device=DEV)
        rnc.dprc_exact_norm(A.to(DEV), G.to(DEV), e)
        out[name] = max(_rel(n.cpu(), oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))),
                        _rel(e.cpu(), oracle.exact_norm(to_f64(A), to_f64(G))))

    # the exact norm in its direct and ghost forms, and on CUDA cores (fp32)
    A, G = _inputs(11, 2, 300, 136, 200)
    ref = oracle.exact_norm(to_f64(A), to_f64(G))
    for name, form in (("exact_direct", rnc.DPRC_EXACT_DIRECT),
                       ("exact_ghost", rnc.DPRC_EXACT_GHOST_N256)):
        n = torch.zeros(2, device=DEV)
        rnc.dprc_exact_norm(A.to(DEV), G.to(DEV), n, form=form)
        out[name] = _rel(n.cpu(), ref)
    A, G = _inputs(12, 2, 77, 33, 19, dtype=torch.float32)
    P = _proj(13, 19, 5, dtype=torch.float32)
    n = torch.zeros(2, device=DEV)
    rnc.dprc_norm_hutch(A.to(DEV), G.to(DEV), P.to(DEV), n)
    out["fp32_odd"] = _rel(n.cpu(), oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P)))

    # the noise on a piece that starts inside a Philox block
    g = torch.zeros(1003, device=DEV)
    rnc.dprc_add_noise_at(g, 5, 1.0, 1.0, 3, 4)
    z = oracle.noise_normals(1003, 3, 4, first_element=5)
    out["noise_at"] = float(np.max(np.abs(g.cpu().double().numpy() - z)))

    torch.cuda.synchronize()
    word = rnc.dprc_device_error(reset=True)
    print(json.dumps({"errors": out, "device_error": word, "code": word & 0xFF,
                      "line": word >> 8}))


if __name__ == "__main__":
    main()
