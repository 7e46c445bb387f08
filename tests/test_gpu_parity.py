"""Parity of the CUDA path (through the C ABI) with the float64 oracle on the
same seeded inputs.

Tolerances: relative 1e-3 on every per-sample norm estimate and clip factor
(bf16 inputs, fp32 accumulation); bit-exact Philox words; each normal within
2e-6 + 1e-6 r (r its Box-Muller pair's radius; the kernel's fp32 hardware
log, sine and cosine against float64), scaled by sigma*C, plus 4 ulp of the
gradient.
"""

import hashlib
import os

import numpy as np
import pytest
import torch

import oracle
import randomized_norm_clipping_gb300 as rnc
from randomized_norm_clipping_gb300 import workloads as wl
from randomized_norm_clipping_gb300.workloads import to_f64

pytestmark = pytest.mark.gpu

RTOL = 1e-3
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from randomized_norm_clipping_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rnc.dprc_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert rnc.dprc_device_error() == 0, "a bounded in-kernel wait ran out"


def _rand(shape, seed, dtype, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(dtype)


def _relerr(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-300))


def _hutch_case(B, T, d, p, k, dtype, seed, gscale=1.0):
    A = _rand((B, T, d), seed, dtype)
    G = _rand((B, T, p), seed + 1, dtype, gscale)
    P = _rand((p, k), seed + 2, dtype, 1.0 / np.sqrt(k))
    return A, G, P


# ------------------------------------------------------------------ Hutchinson

HUTCH_SHAPES = [
    # tensor-core path: bf16, k in {16, 32, 64}, widths multiples of 8
    (2, 64, 256, 256, 32),
    (3, 200, 320, 256, 32),        # ragged T (not a multiple of 64), d not a multiple of 256
    (1, 1, 8, 8, 16),              # minimum sizes
    (2, 1000, 520, 136, 16),
    (4, 4097, 256, 512, 64),       # T one past a tile; k = 64
    (1, 130, 1024, 2048, 32),
    (5, 333, 264, 1032, 32),
    (1, 2048, 1024, 1024, 32),     # few blocks: both kernels split blocks over 8-CTA clusters
    (3, 4096, 1024, 512, 16),      # two-CTA clusters for the sketch, four for the projection
    (40, 256, 256, 128, 32),       # many blocks: whole blocks per CTA, several per CTA
    # LoRA adapters (rank r = 8 .. 64): d_in -> r and r -> d_out
    (4, 1000, 2048, 16, 32),
    (4, 1000, 16, 2048, 32),
    (2, 300, 8, 512, 16),
    (2, 300, 512, 64, 32),
    # float32 / CUDA-core path through the same entry point
    (4, 128, 64, 64, 8),
]


@pytest.mark.parametrize("B,T,d,p,k", HUTCH_SHAPES)
def test_hutch_bf16_matches_oracle(B, T, d, p, k):
    A, G, P = _hutch_case(B, T, d, p, k, torch.bfloat16, seed=B * 1000 + T)
    n = torch.full((B,), -1.0, device=DEV)
    rnc.dprc_norm_hutch(A.to(DEV), G.to(DEV), P.to(DEV), n)
    ref = oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))
    assert _relerr(n.cpu(), ref) < RTOL


# The norm call with the clip factors of the updated n: in the fused kernel's
# finishing step (one launch), or the clip kernel after the other paths; bit
# for bit the two-call sequence, both clip branches, a non-finite sample.
@pytest.mark.parametrize("B,T,d,p,k,dtype", [
    (6, 300, 256, 512, 32, torch.bfloat16),   # fused kernel: the clip in its finisher
    (4, 200, 256, 256, 64, torch.bfloat16),   # two kernels, then the clip kernel
    (4, 500, 1024, 16, 32, torch.bfloat16),   # narrow layer, then the clip kernel
    (4, 128, 64, 64, 8, torch.float32),       # CUDA cores, then the clip kernel
])
def test_norm_hutch_clip_equals_norm_then_clip(B, T, d, p, k, dtype):
    A, G, P = _hutch_case(B, T, d, p, k, dtype, seed=300 + T)
    Ad, Gd, Pd = A.to(DEV), G.to(DEV), P.to(DEV)
    ref = oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))
    C = float(np.median(np.sqrt(ref)))  # half the samples clip
    n1 = torch.full((B,), 0.5, device=DEV)
    c1 = torch.empty(B, device=DEV)
    rnc.dprc_norm_hutch(Ad, Gd, Pd, n1, accumulate=True)
    rnc.dprc_clip_factors(n1, C, c1)
    n2 = torch.full((B,), 0.5, device=DEV)
    c2 = torch.empty(B, device=DEV)
    rnc.dprc_norm_hutch_clip(Ad, Gd, Pd, n2, C, c2, accumulate=True)
    assert torch.equal(n1, n2) and torch.equal(c1, c2)
    tol = 1e-5 if dtype == torch.float32 else RTOL
    assert _relerr(n2.cpu(), ref + 0.5) < tol
    assert _relerr(c2.cpu(), oracle.clip_factors(ref + 0.5, C)) < tol


def test_norm_hutch_clip_zeroes_a_nonfinite_sample():
    A, G, P = _hutch_case(3, 300, 256, 512, 32, torch.bfloat16, seed=77)
    A[1, 5, 7] = float("nan")
    n = torch.zeros(3, device=DEV)
    c = torch.full((3,), 9.0, device=DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    rnc.dprc_norm_hutch_clip(A.to(DEV), G.to(DEV), P.to(DEV), n, 1.0, c, nonfinite=bad)
    assert torch.isnan(n[1]) and float(c[1]) == 0.0 and int(bad) == 1
    ref = oracle.hutch_norm(to_f64(A[[0, 2]]), to_f64(G[[0, 2]]), to_f64(P))
    assert _relerr(c[[0, 2]].cpu(), oracle.clip_factors(ref, 1.0)) < RTOL


@pytest.mark.parametrize("shapes,B,T,k", [
    ([(128, 64), (64, 128)] * 31, 2, 130, 16),        # 62 layers: two launches, clip in the second
    ([(256, 256), (256, 512), (512, 256)], 3, 200, 64),  # k = 64: one call per layer, then the clip
])
def test_norm_hutch_layers_clip_equals_layers_then_clip(shapes, B, T, k):
    As, Gs, Ps = [], [], []
    for j, (d, p) in enumerate(shapes):
        A, G, P = _hutch_case(B, T, d, p, k, torch.bfloat16, seed=900 + 3 * j)
        As.append(A.to(DEV))
        Gs.append(G.to(DEV))
        Ps.append(P.to(DEV))
    n1 = torch.zeros(B, device=DEV)
    c1 = torch.empty(B, device=DEV)
    rnc.dprc_norm_hutch_layers(As, Gs, Ps, n1)
    C = float(torch.sqrt(n1).median())
    rnc.dprc_clip_factors(n1, C, c1)
    n2 = torch.zeros(B, device=DEV)
    c2 = torch.empty(B, device=DEV)
    rnc.dprc_norm_hutch_layers(As, Gs, Ps, n2, C=C, c=c2)
    assert torch.equal(n1, n2) and torch.equal(c1, c2)
    assert float(c2.min()) < 1.0 <= float(c2.max())  # both branches


# Narrow layers (a width <= 64): X_i = A_i^T G_i in one tensor-core pass; the
# exact norm for both orientations (the wide operand A or G), the estimate
# ||X_i P||^2 from the rows of X_i when p <= 64, from per-tile parts of X_i P
# when d <= 32 < p and k <= 128 (other d-narrow maps take the sketch path).  Both widths narrow, narrow widths padded to 16, 32 and 64
# columns, ragged T, k from 8 to 256 (P up to 64 x 256 in shared memory).
# With p <= 16 and k rounded up to 16, 32 or 64, the rows of X_i P come from
# the tensor cores (X as bf16 hi/lo against P).
NARROW_SHAPES = [
    (3, 1000, 2048, 16, 32),   # adapter down map: p narrow
    (3, 1000, 16, 2048, 32),   # adapter up map: d narrow, G is the wide operand
    (2, 1, 512, 8, 16),        # one token
    (2, 129, 24, 1000, 8),     # narrow width 24 (padded to 32), ragged wide width
    (2, 4097, 40, 136, 64),    # narrow width 40 (padded to 64), T one past a tile
    (4, 300, 64, 64, 256),     # both narrow; P 64 x 256 in shared memory
    (1, 640, 32, 16, 128),     # both narrow, d > p
    (5, 257, 1024, 64, 32),
    (2, 333, 32, 520, 128),    # d narrow: a 128 x 128 P tile per 128 p rows; last tile 8 rows
    (3, 200, 8, 4096, 24),     # d narrow, k not a multiple of 16
    (20, 64, 2048, 16, 32),    # 320 tiles: several per CTA (double-buffered accumulator)
    (20, 64, 16, 2048, 32),    # the same, d narrow (P tile restaged per tile)
    (2, 300, 256, 8, 64),      # p <= 16, kp = 64: rows of X P on the tensor cores
    (2, 300, 512, 16, 40),     # p <= 16, kp = 48: rows of X P on CUDA cores
]


@pytest.mark.parametrize("B,T,d,p,k", NARROW_SHAPES)
def test_hutch_narrow_matches_oracle(B, T, d, p, k):
    A, G, P = _hutch_case(B, T, d, p, k, torch.bfloat16, seed=B * 7 + T + d)
    n = torch.full((B,), 0.25, device=DEV)
    rnc.dprc_norm_hutch(A.to(DEV), G.to(DEV), P.to(DEV), n, accumulate=True)
    ref = oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))
    assert _relerr(n.cpu(), ref + 0.25) < RTOL
    e = torch.zeros(B, device=DEV)
    rnc.dprc_exact_norm(A.to(DEV), G.to(DEV), e)
    assert _relerr(e.cpu(), oracle.exact_norm(to_f64(A), to_f64(G))) < RTOL
    assert rnc.dprc_exact_norm_plan(rnc.DPRC_BF16, B, T, d, p) == rnc.DPRC_EXACT_DIRECT


def test_hutch_narrow_identity_projection_is_exact_and_repeats():
    # P = I_p turns ||X P||^2 into ||X||^2: the two narrow outputs agree with
    # each other and with the oracle's exact norm; a rerun is bitwise equal
    B, T, d, p = 3, 700, 1536, 32
    A, G, _ = _hutch_case(B, T, d, p, 32, torch.bfloat16, seed=91)
    Ad, Gd = A.to(DEV), G.to(DEV)
    eye = torch.eye(p, dtype=torch.bfloat16, device=DEV)
    n1, n2, e = (torch.zeros(B, device=DEV) for _ in range(3))
    rnc.dprc_norm_hutch(Ad, Gd, eye, n1)
    rnc.dprc_norm_hutch(Ad, Gd, eye, n2)
    rnc.dprc_exact_norm(Ad, Gd, e)
    assert torch.equal(n1, n2)
    ref = oracle.exact_norm(to_f64(A), to_f64(G))
    assert _relerr(n1.cpu(), ref) < RTOL and _relerr(e.cpu(), ref) < RTOL


@pytest.mark.parametrize("B,T,d,p,k", [(4, 128, 64, 64, 8), (2, 77, 30, 17, 5), (3, 64, 64, 64, 32)])
def test_hutch_fp32_matches_oracle(B, T, d, p, k):
    A, G, P = _hutch_case(B, T, d, p, k, torch.float32, seed=17 + T)
    n = torch.zeros(B, device=DEV)
    rnc.dprc_norm_hutch(A.to(DEV), G.to(DEV), P.to(DEV), n)
    ref = oracle.hutch_norm(A.double().numpy(), G.double().numpy(), P.double().numpy())
    assert _relerr(n.cpu(), ref) < 1e-5


def test_hutch_bf16_odd_widths_use_cuda_cores():
    # d, p not multiples of 8 and k = 24: served by the CUDA-core path
    A, G, P = _hutch_case(2, 90, 37, 45, 24, torch.bfloat16, seed=5)
    n = torch.zeros(2, device=DEV)
    rnc.dprc_norm_hutch(A.to(DEV), G.to(DEV), P.to(DEV), n)
    assert _relerr(n.cpu(), oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))) < RTOL


def test_every_tensor_core_variant_back_to_back():
    # all sketch/projection instantiations in one process, in an order where a
    # launch-attribute cache keyed on the wrong thing would fail
    A, G, _ = _hutch_case(2, 300, 256, 256, 16, torch.bfloat16, seed=77)
    Ad, Gd = A.to(DEV), G.to(DEV)
    g = torch.Generator(device="cpu").manual_seed(78)
    S = torch.randn(256, 16, generator=g).to(torch.bfloat16)
    Pp = torch.randn(256, 16, generator=g).to(torch.bfloat16)
    n = torch.zeros(2, device=DEV)
    rnc.dprc_norm_hutchpp(Ad, Gd, S.to(DEV), Pp.to(DEV), n)
    assert _relerr(n.cpu(), oracle.hutchpp_norm(to_f64(A), to_f64(G), to_f64(S), to_f64(Pp))) < RTOL
    for k in (64, 16, 32):
        P = _rand((256, k), 79 + k, torch.bfloat16, 1.0 / np.sqrt(k))
        rnc.dprc_norm_hutch(Ad, Gd, P.to(DEV), n)
        assert _relerr(n.cpu(), oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))) < RTOL, k


def test_hutch_accumulates_layerwise_sum():
    layers = [_hutch_case(3, 150, d, p, 32, torch.bfloat16, seed=100 + j)
              for j, (d, p) in enumerate([(256, 512), (512, 256), (128, 128)])]
    n = torch.zeros(3, device=DEV)
    for j, (A, G, P) in enumerate(layers):
        rnc.dprc_norm_hutch(A.to(DEV), G.to(DEV), P.to(DEV), n, accumulate=j > 0)
    ref = oracle.layer_sum([oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))
                            for A, G, P in layers])
    assert _relerr(n.cpu(), ref) < RTOL


def test_hutch_is_deterministic():
    A, G, P = _hutch_case(4, 1500, 768, 512, 32, torch.bfloat16, seed=9)
    A, G, P = A.to(DEV), G.to(DEV), P.to(DEV)
    n1 = torch.zeros(4, device=DEV)
    n2 = torch.zeros(4, device=DEV)
    rnc.dprc_norm_hutch(A, G, P, n1)
    rnc.dprc_norm_hutch(A, G, P, n2)
    assert torch.equal(n1, n2)


def test_launch_count_query_matches_the_path():
    from randomized_norm_clipping_gb300 import DPRC_BF16, DPRC_F32
    # bf16 k = 32 on the headline shape: one fused launch
    assert rnc.dprc_norm_hutch_launches(DPRC_BF16, 8, 4096, 2048, 2048, 32) == 1
    # k = 64: sketch and projection kernels
    assert rnc.dprc_norm_hutch_launches(DPRC_BF16, 8, 4096, 2048, 2048, 64) == 2
    # fp32 or widths that are not multiples of 8: the CUDA-core path
    assert rnc.dprc_norm_hutch_launches(DPRC_F32, 4, 128, 64, 64, 8) == 3
    assert rnc.dprc_norm_hutch_launches(DPRC_BF16, 2, 100, 97, 64, 32) == 3
    # a width <= 64: X = A^T G formed in one pass, times P in the epilogue, the
    # per-sample sum by the CTA that completes the sample's last tile
    assert rnc.dprc_norm_hutch_launches(DPRC_BF16, 8, 4096, 2048, 16, 32) == 1
    assert rnc.dprc_norm_hutch_launches(DPRC_BF16, 8, 4096, 64, 48, 256) == 1
    assert rnc.dprc_norm_hutch_launches(DPRC_BF16, 8, 4096, 16, 2048, 32) == 1


def test_hutchpp_launch_count_query_matches_the_path():
    from randomized_norm_clipping_gb300 import DPRC_BF16, DPRC_F32
    q = rnc.dprc_norm_hutchpp_launches
    # bf16 r = 16, p <= 4096: pack, passes 1 and 2 fused, cluster QR, pass 3
    assert q(DPRC_BF16, 8, 4096, 2048, 2048, 16) == 5
    assert q(DPRC_BF16, 3, 300, 136, 256, 16) == 5
    # p > 4096: three sketch and projection pairs and the one-CTA QR
    assert q(DPRC_BF16, 2, 256, 64, 8192, 16) == 7
    # fp32, r != 16 or widths that are not multiples of 8: the CUDA-core path
    assert q(DPRC_F32, 4, 128, 64, 64, 8) == 8
    assert q(DPRC_BF16, 4, 128, 64, 64, 8) == 8
    assert q(DPRC_BF16, 2, 100, 97, 64, 16) == 8
    assert q(DPRC_BF16, 8, 4096, 2048, 2048, 65) == 0


def test_one_workspace_serves_calls_with_different_batch_sizes():
    # a call with fewer samples must not leave scratch where a call with more
    # keeps its counters (they share one fixed counter block for B <= 256)
    T, d, p, k = 1024, 1024, 1024, 16
    ws = rnc.workspace(rnc.DPRC_OP_HUTCH, torch.empty(1, dtype=torch.bfloat16, device=DEV),
                       32, T, d, p, k)
    runs = []
    for B in (32, 6, 32, 6):
        A = _rand((B, T, d), 70 + B, torch.bfloat16).to(DEV)
        G = _rand((B, T, p), 71 + B, torch.bfloat16, 0.05).to(DEV)
        P = _rand((p, k), 72, torch.bfloat16, k ** -0.5).to(DEV)
        n = torch.zeros(B, device=DEV)
        c = torch.empty(B, device=DEV)
        rnc.dprc_norm_hutch_clip(A, G, P, n, 1.0, c, ws=ws)
        fresh = torch.zeros(B, device=DEV)
        rnc.dprc_norm_hutch(A, G, P, fresh)  # its own zeroed workspace
        runs.append((n, fresh))
        torch.cuda.synchronize()
        assert rnc.dprc_device_error() == 0
    for n, fresh in runs:
        assert torch.equal(n, fresh)


def _host_chunk(B, T, d, p, esize):
    # the chunk rule of dprc_norm_hutch_clip_host (include/dprc.h): the fewest
    # samples that make at least 128 MB of A and G
    sample = T * (d + p) * esize
    return min(B, -(-(128 << 20) // sample))


@pytest.mark.parametrize("B,T,d,p,k,dtype", [
    (9, 4096, 2048, 2048, 32, torch.bfloat16),   # chunks of 4, 4 and 1: a slot reused
    (70, 1024, 1024, 1024, 16, torch.bfloat16),  # chunks of 32, 32 and 6 samples
    (5, 100, 40, 24, 8, torch.float32),          # one chunk
])
def test_norm_hutch_clip_host_matches_device_calls_and_oracle(B, T, d, p, k, dtype):
    A = _rand((B, T, d), 60 + B, dtype)
    G = _rand((B, T, p), 61 + B, dtype, 0.05)
    P = _rand((p, k), 62 + B, dtype, k ** -0.5)
    Ah, Gh, Ph = (x.pin_memory() for x in (A, G, P))
    nh = torch.full((B,), -1.0).pin_memory()
    ch = torch.full((B,), -1.0).pin_memory()
    ref = oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))
    C = float(np.median(ref)) ** 0.5  # some samples clipped, some not
    stage = rnc.host_stage(Ah, T, d, p, k)
    rnc.dprc_norm_hutch_clip_host(Ah, Gh, Ph, C, nh, ch, stage=stage)
    torch.cuda.synchronize()
    assert _relerr(nh, ref) < (1e-5 if dtype == torch.float32 else RTOL)
    # the same chunks through the device entry: bit for bit
    step = _host_chunk(B, T, d, p, A.element_size())
    nd = torch.empty(B)
    cd = torch.empty(B)
    for i0 in range(0, B, step):
        sl = slice(i0, min(B, i0 + step))
        m = sl.stop - sl.start
        n1 = torch.zeros(m, device=DEV)
        c1 = torch.empty(m, device=DEV)
        rnc.dprc_norm_hutch_clip(A[sl].to(DEV), G[sl].to(DEV), P.to(DEV), n1, C, c1)
        nd[sl], cd[sl] = n1.cpu(), c1.cpu()
    assert torch.equal(nh, nd) and torch.equal(ch, cd)
    assert (ch < 1).any() and (ch == 1).any()  # both branches of the clip rule
    # a second call through the same stage buffer agrees; without n only c comes back
    ch2 = torch.zeros(B).pin_memory()
    rnc.dprc_norm_hutch_clip_host(Ah, Gh, Ph, C, None, ch2, stage=stage)
    torch.cuda.synchronize()
    assert torch.equal(ch, ch2)
    assert rnc.dprc_device_error() == 0


def test_hutch_identity_projection_gives_exact_norm():
    # P = I_p (k = p = 32) turns the estimate into the exact norm
    A, G, _ = _hutch_case(2, 300, 128, 32, 32, torch.bfloat16, seed=3)
    P = torch.eye(32, dtype=torch.bfloat16)
    n = torch.zeros(2, device=DEV)
    rnc.dprc_norm_hutch(A.to(DEV), G.to(DEV), P.to(DEV), n)
    assert _relerr(n.cpu(), oracle.exact_norm(to_f64(A), to_f64(G))) < RTOL


# ------------------------------------------------------------------ Hutch++

# the cluster QR with one row per thread (p <= 2048, 2040 with a ragged last
# CTA) and two (2056 .. 4096, up to its bound); past it (4200) the one-CTA QR
# and the three passes in sequence
@pytest.mark.parametrize("B,T,d,p", [(2, 200, 256, 256), (3, 77, 136, 64), (2, 1100, 512, 1024),
                                     (2, 300, 256, 3000), (2, 150, 136, 128), (2, 300, 128, 2040),
                                     (2, 300, 128, 2056), (1, 200, 128, 4096), (1, 120, 128, 4200),
                                     (1, 50, 8, 16), (2, 1, 16, 24)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_hutchpp_matches_oracle(B, T, d, p, dtype):
    r = 16
    A = _rand((B, T, d), 40 + T, dtype)
    g = torch.Generator(device="cpu").manual_seed(41 + T)
    U, V = torch.randn(B, T, 8, generator=g), torch.randn(B, p, 8, generator=g)
    G = (torch.bmm(U, V.transpose(1, 2)) / np.sqrt(8) + 0.05 * torch.randn(B, T, p, generator=g)).to(dtype)
    S = _rand((p, r), 42, dtype)
    P = _rand((p, r), 43, dtype)
    n = torch.zeros(B, device=DEV)
    rnc.dprc_norm_hutchpp(A.to(DEV), G.to(DEV), S.to(DEV), P.to(DEV), n)
    ref = oracle.hutchpp_norm(to_f64(A), to_f64(G), to_f64(S), to_f64(P))
    assert _relerr(n.cpu(), ref) < RTOL


@pytest.mark.parametrize("tail", [1e-2, 1e-3, 1e-5, 0.0])
def test_hutchpp_near_rank_deficient_sketch(tail):
    # G = rank 8 + a small tail: M = O S has 8 strong columns and 8 at the
    # tail's level, down to rounding noise (tail 0).  The combining step
    # forms X Q as (X M) R^-1 and drops columns of R at noise level; the
    # result must still be the oracle's (Householder Q) within RTOL
    B, T, d, p, r = 2, 300, 256, 512, 16
    A = _rand((B, T, d), 60, torch.bfloat16)
    g = torch.Generator(device="cpu").manual_seed(61)
    U, V = torch.randn(B, T, 8, generator=g), torch.randn(B, p, 8, generator=g)
    G = (torch.bmm(U, V.transpose(1, 2)) / np.sqrt(8) + tail * torch.randn(B, T, p, generator=g))
    G = G.to(torch.bfloat16)
    S, P = _rand((p, r), 62, torch.bfloat16), _rand((p, r), 63, torch.bfloat16)
    n = torch.zeros(B, device=DEV)
    rnc.dprc_norm_hutchpp(A.to(DEV), G.to(DEV), S.to(DEV), P.to(DEV), n)
    ref = oracle.hutchpp_norm(to_f64(A), to_f64(G), to_f64(S), to_f64(P))
    assert _relerr(n.cpu(), ref) < RTOL


def test_hutchpp_accumulates():
    # n (+)= the estimate: a second call with accumulate adds the same value
    B, T, d, p, r = 2, 200, 136, 256, 16
    A = _rand((B, T, d), 70, torch.bfloat16)
    G = _rand((B, T, p), 71, torch.bfloat16, 0.1)
    S, P = _rand((p, r), 72, torch.bfloat16), _rand((p, r), 73, torch.bfloat16)
    ref = oracle.hutchpp_norm(to_f64(A), to_f64(G), to_f64(S), to_f64(P))
    n = torch.full((B,), 5.0, device=DEV)
    rnc.dprc_norm_hutchpp(A.to(DEV), G.to(DEV), S.to(DEV), P.to(DEV), n)
    assert _relerr(n.cpu(), ref) < RTOL
    rnc.dprc_norm_hutchpp(A.to(DEV), G.to(DEV), S.to(DEV), P.to(DEV), n, accumulate=True)
    assert _relerr(n.cpu(), 2.0 * ref) < RTOL


def test_hutchpp_leaves_the_counter_block_zero_for_other_calls():
    # Hutch++ counts its sketch rows per sample in three rows of the counter
    # block that the fused Hutchinson kernel also uses (one row per layer);
    # the third pass zeroes them, so one workspace serves both calls in turn
    B, T, d, p, r, k = 3, 300, 136, 256, 16, 32
    A = _rand((B, T, d), 80, torch.bfloat16).to(DEV)
    G = _rand((B, T, p), 81, torch.bfloat16, 0.1).to(DEV)
    S, Pp = _rand((p, r), 82, torch.bfloat16).to(DEV), _rand((p, r), 83, torch.bfloat16).to(DEV)
    P = _rand((p, k), 84, torch.bfloat16).to(DEV)
    nbytes = max(rnc.workspace(rnc.DPRC_OP_HUTCHPP, A, B, T, d, p, r).numel(),
                 rnc.workspace(rnc.DPRC_OP_HUTCH_LAYERS, A, B, T, d, p, k).numel())
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    ref_pp = oracle.hutchpp_norm(to_f64(A.cpu()), to_f64(G.cpu()), to_f64(S.cpu()), to_f64(Pp.cpu()))
    ref_h = oracle.hutch_norm(to_f64(A.cpu()), to_f64(G.cpu()), to_f64(P.cpu()))
    for _ in range(2):
        n = torch.zeros(B, device=DEV)
        rnc.dprc_norm_hutchpp(A, G, S, Pp, n, ws=ws)
        assert _relerr(n.cpu(), ref_pp) < RTOL
        layers = [(A, G, P)] * 3
        n = torch.zeros(B, device=DEV)
        rnc.dprc_norm_hutch_layers([x[0] for x in layers], [x[1] for x in layers],
                                   [x[2] for x in layers], n, ws=ws)
        assert _relerr(n.cpu(), 3.0 * ref_h) < RTOL
    assert rnc.dprc_device_error(reset=True) == 0


def test_hutchpp_exact_on_low_rank_gradients():
    B, T, d, p, r = 2, 256, 256, 512, 16
    A = _rand((B, T, d), 50, torch.bfloat16)
    g = torch.Generator(device="cpu").manual_seed(51)
    G = torch.bmm(torch.randn(B, T, 4, generator=g), torch.randn(B, 4, p, generator=g)).to(torch.bfloat16)
    S, P = _rand((p, r), 52, torch.bfloat16), _rand((p, r), 53, torch.bfloat16)
    n = torch.zeros(B, device=DEV)
    rnc.dprc_norm_hutchpp(A.to(DEV), G.to(DEV), S.to(DEV), P.to(DEV), n)
    assert _relerr(n.cpu(), oracle.exact_norm(to_f64(A), to_f64(G))) < RTOL


# ------------------------------------------------------------------ exact norm

# The automatic choice: bf16 with d, p multiples of 8 takes a tensor-core form
# (direct A^T G in 128 x 256 tiles, or ghost for short T); fp32 or other widths
# take the ghost form on CUDA cores.
@pytest.mark.parametrize("B,T,d,p,dtype", [(4, 128, 64, 64, torch.float32),
                                           (2, 333, 96, 40, torch.bfloat16),
                                           (2, 333, 97, 41, torch.bfloat16),
                                           (1, 1, 8, 8, torch.bfloat16),
                                           (2, 1024, 512, 256, torch.bfloat16),
                                           (3, 1000, 392, 600, torch.bfloat16),
                                           (1, 4097, 128, 256, torch.bfloat16),
                                           (5, 64, 1024, 1536, torch.bfloat16),
                                           (4, 1000, 2048, 16, torch.bfloat16),   # LoRA down
                                           (4, 1000, 16, 2048, torch.bfloat16)])  # LoRA up
def test_exact_norm_matches_oracle(B, T, d, p, dtype):
    A = _rand((B, T, d), 60 + T, dtype)
    G = _rand((B, T, p), 61 + T, dtype, 0.05)
    n = torch.zeros(B, device=DEV)
    rnc.dprc_exact_norm(A.to(DEV), G.to(DEV), n)
    assert _relerr(n.cpu(), oracle.exact_norm(to_f64(A), to_f64(G))) < RTOL


def test_exact_norm_accumulates_and_repeats():
    A = _rand((3, 700, 264), 70, torch.bfloat16)
    G = _rand((3, 700, 520), 71, torch.bfloat16, 0.05)
    Ad, Gd = A.to(DEV), G.to(DEV)
    ref = oracle.exact_norm(to_f64(A), to_f64(G))
    n = torch.full((3,), 2.5, device=DEV)
    rnc.dprc_exact_norm(Ad, Gd, n, accumulate=True)
    assert _relerr(n.cpu(), ref + 2.5) < RTOL
    rnc.dprc_exact_norm(Ad, Gd, n, accumulate=False)
    once = n.clone()
    rnc.dprc_exact_norm(Ad, Gd, n, accumulate=False)
    assert torch.equal(n, once)  # fixed summation order: bitwise repeatable
    assert _relerr(n.cpu(), ref) < RTOL


def test_exact_norm_full_size_samples():
    # two samples of the q_proj workload (T = 4096, d = p = 2048), the launch
    # configuration the benchmark's exact-norm row times with B = 8
    wk = wl.WORKLOADS[wl.HEADLINE]
    A, G, _ = wl.layer_inputs(wk, 0, device=DEV, B=2)
    n = torch.zeros(2, device=DEV)
    rnc.dprc_exact_norm(A, G, n)
    assert _relerr(n.cpu(), oracle.exact_norm(to_f64(A), to_f64(G))) < RTOL


# Both exact forms on tensor cores at fixed forms and tile widths: T from one
# token to several 128-token blocks with ragged tails (odd and even block
# counts, so spans of two blocks end both full and half), ragged d and p, and
# LoRA-shaped widths.
EXACT_FORMS = [rnc.DPRC_EXACT_DIRECT, rnc.DPRC_EXACT_GHOST_N128, rnc.DPRC_EXACT_GHOST_N256]
EXACT_FORM_SHAPES = [(1, 1, 8, 8), (2, 100, 64, 72), (2, 129, 96, 40), (3, 257, 200, 136),
                     (2, 384, 64, 64), (2, 1000, 392, 600), (1, 2048, 128, 256),
                     (4, 640, 2048, 16), (4, 640, 16, 2048),
                     (2, 8192, 72, 64)]  # 64 blocks: 1056 ghost units per sample in the queue


@pytest.mark.parametrize("form", EXACT_FORMS)
@pytest.mark.parametrize("B,T,d,p", EXACT_FORM_SHAPES)
def test_exact_forms_match_oracle(B, T, d, p, form):
    A = _rand((B, T, d), 80 + T, torch.bfloat16)
    G = _rand((B, T, p), 81 + T, torch.bfloat16, 0.05)
    n = torch.zeros(B, device=DEV)
    rnc.dprc_exact_norm(A.to(DEV), G.to(DEV), n, form=form)
    assert _relerr(n.cpu(), oracle.exact_norm(to_f64(A), to_f64(G))) < RTOL


def test_exact_forms_agree_with_the_ghost_oracle_and_repeat():
    A = _rand((3, 700, 264), 90, torch.bfloat16)
    G = _rand((3, 700, 520), 91, torch.bfloat16, 0.05)
    Ad, Gd = A.to(DEV), G.to(DEV)
    ref = oracle.ghost_norm(to_f64(A), to_f64(G))
    for form in (rnc.DPRC_EXACT_GHOST_N128, rnc.DPRC_EXACT_GHOST_N256):
        n = torch.full((3,), 1.5, device=DEV)
        rnc.dprc_exact_norm(Ad, Gd, n, accumulate=True, form=form)
        assert _relerr(n.cpu(), ref + 1.5) < RTOL
        rnc.dprc_exact_norm(Ad, Gd, n, form=form)
        once = n.clone()
        rnc.dprc_exact_norm(Ad, Gd, n, form=form)
        assert torch.equal(n, once)  # fixed summation order: bitwise repeatable


def test_ghost_form_under_cancellation():
    # nearly collinear token rows and alternating-sign gradients: the T^2
    # Gram products are large and cancel, so n_i is small against them.  The
    # ghost form's error must stay within fp32 rounding of the scale
    # (sum_t ||a_t|| ||g_t||)^2 (each Gram entry is accurate to a few ulp of
    # ||a_t|| ||a_s||), its result must not be negative, and the direct form,
    # a sum of squares, stays accurate relative to n_i.
    B, T, d, p = 2, 512, 256, 128
    gen = torch.Generator().manual_seed(5)
    a = torch.randn(B, 1, d, generator=gen)
    g = torch.randn(B, 1, p, generator=gen)
    sign = (-1.0) ** torch.arange(T).reshape(1, T, 1)
    A = (a + 0.01 * torch.randn(B, T, d, generator=gen)).to(torch.bfloat16)
    G = (sign * g + 0.01 * torch.randn(B, T, p, generator=gen)).to(torch.bfloat16)
    ref = oracle.exact_norm(to_f64(A), to_f64(G))
    Af, Gf = to_f64(A), to_f64(G)
    scale = np.array([(np.linalg.norm(Af[i], axis=1) * np.linalg.norm(Gf[i], axis=1)).sum() ** 2
                      for i in range(B)])
    assert np.all(ref < 1e-3 * scale)  # the case really cancels
    for form in (rnc.DPRC_EXACT_GHOST_N128, rnc.DPRC_EXACT_GHOST_N256):
        n = torch.zeros(B, device=DEV)
        rnc.dprc_exact_norm(A.to(DEV), G.to(DEV), n, form=form)
        got = n.cpu().numpy().astype(np.float64)
        assert np.all(got >= 0)
        assert np.all(np.abs(got - ref) <= 1e-5 * scale)
    n = torch.zeros(B, device=DEV)
    rnc.dprc_exact_norm(A.to(DEV), G.to(DEV), n, form=rnc.DPRC_EXACT_DIRECT)
    assert _relerr(n.cpu(), ref) < RTOL


def test_exact_auto_takes_the_form_with_less_work():
    bf = rnc.DPRC_BF16
    # q_proj widths: ghost below T = 2 d p / (d + p) = 2048 when the batch has
    # enough 128-token blocks to fill the GPU, direct above
    assert rnc.dprc_exact_norm_plan(bf, 32, 512, 2048, 2048) in (rnc.DPRC_EXACT_GHOST_N128,
                                                                  rnc.DPRC_EXACT_GHOST_N256)
    assert rnc.dprc_exact_norm_plan(bf, 32, 1024, 2048, 2048) in (rnc.DPRC_EXACT_GHOST_N128,
                                                                   rnc.DPRC_EXACT_GHOST_N256)
    assert rnc.dprc_exact_norm_plan(bf, 8, 4096, 2048, 2048) == rnc.DPRC_EXACT_DIRECT
    # LoRA widths: the d x p product is tiny, always direct
    assert rnc.dprc_exact_norm_plan(bf, 8, 512, 2048, 16) == rnc.DPRC_EXACT_DIRECT
    # fixed forms are reported as asked; fp32 has only the CUDA-core ghost form
    assert rnc.dprc_exact_norm_plan(bf, 8, 512, 2048, 2048, rnc.DPRC_EXACT_DIRECT) == \
        rnc.DPRC_EXACT_DIRECT
    assert rnc.dprc_exact_norm_plan(bf, 8, 512, 64, 64, rnc.DPRC_EXACT_GHOST_N128) == \
        rnc.DPRC_EXACT_GHOST_N128
    assert rnc.dprc_exact_norm_plan(rnc.DPRC_F32, 2, 64, 64, 64) == rnc.DPRC_EXACT_GHOST
    assert rnc.dprc_exact_norm_plan(rnc.DPRC_F32, 2, 64, 64, 64, rnc.DPRC_EXACT_DIRECT) == 0
    # the automatic call is bitwise the call of the form it reports
    A = _rand((4, 300, 512), 95, torch.bfloat16).to(DEV)
    G = _rand((4, 300, 384), 96, torch.bfloat16, 0.05).to(DEV)
    form = rnc.dprc_exact_norm_plan(bf, 4, 300, 512, 384)
    n0, n1 = torch.zeros(4, device=DEV), torch.zeros(4, device=DEV)
    rnc.dprc_exact_norm(A, G, n0)
    rnc.dprc_exact_norm(A, G, n1, form=form)
    assert torch.equal(n0, n1)


# ------------------------------------------------------------------ clip

def test_clip_factors_match_oracle_including_edge_cases():
    vals = np.array([4.0, 0.25, 1.0, 0.0, 100.0, 3.7e-30, 2.5e30, np.nan, np.inf, -1.0, -np.inf,
                     1.0000001, 0.9999999], dtype=np.float32)
    n = torch.from_numpy(vals).to(DEV)
    c = torch.empty_like(n)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    rnc.dprc_clip_factors(n, 1.0, c, cnt)
    ref = oracle.clip_factors(vals.astype(np.float64), 1.0)
    got = c.cpu().double().numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-6, atol=0)
    assert int(cnt.item()) == 4
    c2 = torch.empty_like(n)
    rnc.dprc_clip_factors(n, 3.5, c2)
    np.testing.assert_allclose(c2.cpu().double().numpy(), oracle.clip_factors(vals.astype(np.float64), 3.5),
                               rtol=1e-6, atol=0)


# ------------------------------------------------------------------ Philox and noise

@pytest.mark.parametrize("first", [0, 12345, (1 << 32) - 7, (1 << 40) + 3])
def test_philox_words_bit_exact(first):
    seed, step = 0x0123456789ABCDEF, (5 << 32) | 77
    out = torch.empty(4096, 4, dtype=torch.int32, device=DEV)
    rnc.dprc_philox_words(out, first, seed, step)
    got = out.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, oracle.philox_words(seed, step, first, 4096))


def test_philox_long_stream_hash():
    n = 1 << 22
    out = torch.empty(n, 4, dtype=torch.int32, device=DEV)
    rnc.dprc_philox_words(out, 0, 2024, 9)
    got = out.cpu().numpy().view(np.uint32)
    ref = oracle.philox_words(2024, 9, 0, n)
    assert hashlib.sha256(got.tobytes()).hexdigest() == hashlib.sha256(ref.tobytes()).hexdigest()


def _pair_radius(z):
    """Radius sqrt(z_a^2 + z_b^2) of the Box-Muller pair each normal belongs to
    (elements 4j, 4j+1 and 4j+2, 4j+3), aligned with z."""
    zz = np.asarray(z, dtype=np.float64)
    n = zz.size
    pad = np.zeros((n + 1) // 2 * 2)
    pad[:n] = zz
    r = np.sqrt(pad[0::2] ** 2 + pad[1::2] ** 2)
    return np.repeat(r, 2)[:n]


def _noise_tol(z, g, sigma, C, r=None):
    # fp32 hardware log/sin/cos in the kernel: |dz| <= 2e-6 + 1e-6 r
    r = _pair_radius(z) if r is None else r
    return sigma * C * (2e-6 + 1e-6 * r) + 4 * np.finfo(np.float32).eps * np.abs(g)


@pytest.mark.parametrize("N", [1, 3, 4, 1001, 65536 + 3])
def test_noise_matches_oracle(N):
    grad = wl.gradient_buffer(N, seed=N)
    out = grad.to(DEV)
    sigma, C = 1.3, 0.7
    rnc.dprc_add_noise(out, sigma, C, seed=99, step=4)
    ref = oracle.add_noise(grad.double().numpy(), sigma, C, 99, 4)
    z = oracle.noise_normals(N, 99, 4)
    err = np.abs(out.cpu().double().numpy() - ref)
    assert np.all(err <= _noise_tol(z, grad.double().numpy(), sigma, C))


def _z_and_radius_at(first, N, seed, step):
    """z_e and its Box-Muller pair radius for e in [first, first + N)."""
    base = first & ~3
    z = oracle.noise_normals(first - base + N, seed, step, first_element=base)
    r = _pair_radius(z)  # pairs are (4j, 4j + 1), (4j + 2, 4j + 3): base is a multiple of 4
    return z[first - base:], r[first - base:]


@pytest.mark.parametrize("first,N", [(0, 1001), (4, 1003), (5, 4096), (6, 7), (7, 65539),
                                     ((1 << 33) + 1, 999), (1_235_814_397, 12)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noise_at_offset_matches_oracle(first, N, dtype):
    # a piece of a gradient kept in several buffers: element i gets z_{first + i}
    grad = wl.gradient_buffer(N, seed=N + 1).to(dtype)
    out = grad.to(DEV)
    sigma, C = 1.3, 0.7
    rnc.dprc_add_noise_at(out, first, sigma, C, seed=99, step=4)
    g = grad.double().numpy()
    z, r = _z_and_radius_at(first, N, 99, 4)
    ref = g + sigma * C * z
    got = out.cpu().double().numpy()
    tol = _noise_tol(z, g, sigma, C, r)
    if dtype == torch.bfloat16:
        # the fp32 sum is rounded once to bf16: one bf16 unit in the last place
        tol = tol + np.abs(ref) * 2.0 ** -7
    assert np.all(np.abs(got - ref) <= tol)


def test_noise_pieces_equal_the_whole_bitwise():
    # the training step's use: weight gradients laid end to end, each given
    # its stretch of the one stream, equal dprc_add_noise on the concatenation
    sizes = [4096, 1000, 3, 5, 8192, 12, 1]
    grad = wl.gradient_buffer(sum(sizes), seed=5).to(DEV)
    whole = grad.clone()
    rnc.dprc_add_noise(whole, 0.9, 1.1, seed=7, step=3)
    off, parts = 0, []
    for n in sizes:
        piece = grad[off:off + n].clone()  # its own (16-byte aligned) buffer
        rnc.dprc_add_noise_at(piece, off, 0.9, 1.1, seed=7, step=3)
        parts.append(piece)
        off += n
    assert torch.equal(torch.cat(parts), whole)


def test_noise_same_seed_step_reproduces_and_differs_otherwise():
    a = torch.zeros(10000, device=DEV)
    b = torch.zeros(10000, device=DEV)
    c = torch.zeros(10000, device=DEV)
    rnc.dprc_add_noise(a, 1.0, 1.0, seed=1, step=2)
    rnc.dprc_add_noise(b, 1.0, 1.0, seed=1, step=2)
    rnc.dprc_add_noise(c, 1.0, 1.0, seed=1, step=3)
    assert torch.equal(a, b)
    assert not torch.equal(a, c)


@pytest.mark.slow
def test_noise_full_gradient_buffer_sampled():
    # the whole Llama-3.2-1B gradient (1.24e9 fp32), checked at sampled elements
    N = wl.LLAMA32_1B_PARAMS
    grad = torch.zeros(N, device=DEV)
    rnc.dprc_add_noise(grad, 1.0, 1.0, seed=31337, step=1)
    rng = np.random.default_rng(0)
    idx = np.concatenate([rng.integers(0, N, 4000), np.arange(N - 7, N), np.arange(0, 8)])
    got = grad[torch.from_numpy(idx).to(DEV)].cpu().double().numpy()
    pairs = [oracle.noise_normals(2, 31337, 1, first_element=int(e) & ~1) for e in idx]
    ref = np.array([pr[e & 1] for pr, e in zip(pairs, idx)])
    rad = np.array([np.hypot(*pr) for pr in pairs])
    assert np.all(np.abs(got - ref) <= _noise_tol(ref, 0.0, 1.0, 1.0, rad))
    del grad
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ many layers in one call

def _layers(shapes, B, T, k, seed):
    As, Gs, Ps = [], [], []
    for j, (d, p) in enumerate(shapes):
        A, G, P = _hutch_case(B, T, d, p, k, torch.bfloat16, seed=seed + 7 * j, gscale=0.1)
        As.append(A)
        Gs.append(G)
        Ps.append(P)
    return As, Gs, Ps


@pytest.mark.parametrize("shapes,B,T,k", [
    ([(256, 512), (512, 256), (128, 128), (256, 1024), (1024, 256)], 3, 300, 32),  # one launch
    ([(128, 64), (64, 128)] * 31, 2, 130, 16),                                     # 62 layers: two launches
    ([(256, 256), (512, 128)], 2, 200, 64),                                        # k = 64: layer by layer
])
def test_hutch_layers_matches_layer_sum(shapes, B, T, k):
    As, Gs, Ps = _layers(shapes, B, T, k, seed=300 + T)
    n = torch.full((B,), 0.5, device=DEV)
    rnc.dprc_norm_hutch_layers([a.to(DEV) for a in As], [g.to(DEV) for g in Gs],
                               [p_.to(DEV) for p_ in Ps], n, accumulate=True)
    ref = oracle.layer_sum([oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))
                            for A, G, P in zip(As, Gs, Ps)])
    assert _relerr(n.cpu() - 0.5, ref) < RTOL
    assert rnc.dprc_device_error() == 0


def test_hutch_layers_repeats_bitwise_and_reuses_its_workspace():
    shapes = [(256, 512), (512, 512), (512, 256)] * 3
    As, Gs, Ps = _layers(shapes, 4, 1000, 32, seed=11)
    As, Gs, Ps = [a.to(DEV) for a in As], [g.to(DEV) for g in Gs], [p_.to(DEV) for p_ in Ps]
    ws = rnc.workspace(rnc.DPRC_OP_HUTCH_LAYERS, As[0], 4, 1000, 512, 512, 32)
    n1 = torch.zeros(4, device=DEV)
    n2 = torch.zeros(4, device=DEV)
    rnc.dprc_norm_hutch_layers(As, Gs, Ps, n1, ws=ws)
    rnc.dprc_norm_hutch(As[0], Gs[0], Ps[0], torch.zeros(4, device=DEV), ws=ws)  # same workspace
    rnc.dprc_norm_hutch_layers(As, Gs, Ps, n2, ws=ws)
    assert torch.equal(n1, n2)


# ------------------------------------------------------------------ +-1 projection

@pytest.mark.parametrize("B,T,d,p,k,dtype", [
    (3, 300, 256, 512, 32, torch.bfloat16),   # signs generated in the kernel (k = 32)
    (2, 1000, 520, 264, 16, torch.bfloat16),  # in the kernel, k = 16, ragged widths
    (8, 4096, 2048, 2048, 32, torch.bfloat16),  # the q_proj launch shape
    (2, 200, 256, 256, 64, torch.bfloat16),   # k = 64: signs in the workspace, two kernels
    (3, 77, 30, 17, 8, torch.float32),        # fp32: CUDA cores
    (2, 90, 37, 45, 24, torch.bfloat16),      # odd widths: CUDA cores
    (4, 1000, 2048, 16, 32, torch.bfloat16),  # adapter down map: X = A^T G, then X S
    (4, 1000, 16, 2048, 32, torch.bfloat16),  # adapter up map, d narrow: signs per P tile
    (2, 300, 8, 1000, 16, torch.bfloat16),    # d narrow, ragged last tile
])
def test_pm1_projection_matches_oracle(B, T, d, p, k, dtype):
    A = _rand((B, T, d), 500 + T, dtype)
    G = _rand((B, T, p), 501 + T, dtype, 0.1)
    seed, step = 0x1234_5678_9ABC, 17 + k
    n = torch.full((B,), 1.5, device=DEV)
    rnc.dprc_norm_hutch_pm1(A.to(DEV), G.to(DEV), k, seed, step, n, accumulate=True)
    S = oracle.rademacher_signs(seed, step, p, k)
    ref = oracle.hutch_norm_rademacher(to_f64(A), to_f64(G), S)
    tol = 1e-5 if dtype == torch.float32 else RTOL
    assert _relerr(n.cpu() - 1.5, ref) < tol
    assert rnc.dprc_device_error() == 0


def test_pm1_projection_is_deterministic_and_seeded():
    A = _rand((4, 700, 512), 5, torch.bfloat16).to(DEV)
    G = _rand((4, 700, 512), 6, torch.bfloat16, 0.1).to(DEV)
    n1, n2, n3 = (torch.zeros(4, device=DEV) for _ in range(3))
    rnc.dprc_norm_hutch_pm1(A, G, 32, 9, 1, n1)
    rnc.dprc_norm_hutch_pm1(A, G, 32, 9, 1, n2)
    rnc.dprc_norm_hutch_pm1(A, G, 32, 9, 2, n3)  # another step: other signs
    assert torch.equal(n1, n2)
    assert not torch.equal(n1, n3)
