"""Failure detection of the one-launch Hutchinson kernel, without a GPU fault.

The library promises that every wait inside a kernel is bounded: a wait that
runs out records a code in the device error word and the kernel unwinds and
returns, leaving the context usable.  These tests make that happen on purpose
through the C ABI's test hook (dprc_test_hutch_fault), with a short limit:

  - a launch whose sketch-ready targets can never be met: every projection
    block's wait for its sample's sketch runs out, the launch returns well
    within a second, the error word says DPRC_DEVERR_READY, n is not written,
    and a normal call on a re-zeroed workspace then matches the oracle;
  - a launch whose cluster shape differs from its plan: the kernel refuses it
    before touching memory (DPRC_DEVERR_LAUNCH), and a normal call on the same,
    untouched workspace matches the oracle.

Shapes cover the single-layer launch without clusters, with clusters of 2
(split sketch and projection blocks, exchanges through distributed shared
memory), and a multi-layer launch.
"""

import os
import time

import numpy as np
import pytest
import torch

import oracle
import randomized_norm_clipping_gb300 as rnc
from randomized_norm_clipping_gb300 import binding as bnd
from randomized_norm_clipping_gb300.workloads import to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
RTOL = 1e-3
WAIT_NS = 2_000_000   # 2 ms, against the 2 s the kernels use by default
SENTINEL = 12345.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not os.path.exists(bnd.LIB_PATH):
        from randomized_norm_clipping_gb300 import build
        build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rnc.dprc_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert rnc.dprc_device_error(reset=True) == 0


def _layers(seed, B, T, dims, k=32):
    g = torch.Generator(device="cpu").manual_seed(seed)
    As, Gs, Ps = [], [], []
    for d, p in dims:
        As.append(torch.randn(B, T, d, generator=g).to(torch.bfloat16))
        Gs.append((torch.randn(B, T, p, generator=g) * 0.1).to(torch.bfloat16))
        Ps.append((torch.randn(p, k, generator=g) / k ** 0.5).to(torch.bfloat16))
    return As, Gs, Ps


def _oracle_sum(As, Gs, Ps):
    return sum(oracle.hutch_norm(to_f64(a), to_f64(g), to_f64(p)) for a, g, p in zip(As, Gs, Ps))


def _workspace(As, Gs, Ps):
    B, T = As[0].shape[:2]
    k = Ps[0].shape[1]
    op = rnc.DPRC_OP_HUTCH_LAYERS if len(As) > 1 else rnc.DPRC_OP_HUTCH
    dmax = max(a.shape[2] for a in As)
    pmax = max(g.shape[2] for g in Gs)
    return rnc.workspace(op, As[0].to(DEV), B, T, dmax, pmax, k)


def _normal_call(Ad, Gd, Pd, n, ws):
    if len(Ad) == 1:
        rnc.dprc_norm_hutch(Ad[0], Gd[0], Pd[0], n, ws=ws)
    else:
        rnc.dprc_norm_hutch_layers(Ad, Gd, Pd, n, ws=ws)


# (name, B, T, [(d, p) per layer]); the first plans no clusters, the second
# clusters of 2 (both phases split), the third is a multi-layer launch
SHAPES = [
    ("single_no_clusters", 8, 2048, [(2048, 2048)]),
    ("single_clusters", 3, 200, [(320, 256)]),
    ("three_layers", 2, 512, [(256, 512), (512, 256), (384, 384)]),
]


@pytest.mark.parametrize("name,B,T,dims", SHAPES, ids=[s[0] for s in SHAPES])
def test_ready_wait_runs_out_and_the_launch_unwinds(name, B, T, dims):
    As, Gs, Ps = _layers(31, B, T, dims)
    Ad = [a.to(DEV) for a in As]
    Gd = [g.to(DEV) for g in Gs]
    Pd = [p.to(DEV) for p in Ps]
    k = Ps[0].shape[1]
    if len(dims) == 1:
        d, p = dims[0]
        assert rnc.dprc_norm_hutch_launches(rnc.DPRC_BF16, B, T, d, p, k) == 1
    ws = _workspace(As, Gs, Ps)
    n = torch.full((B,), SENTINEL, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rnc.dprc_test_hutch_fault(bnd.FAULT_READY_NEVER_MET, WAIT_NS, Ad, Gd, Pd, n, ws)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    # the limit given to the launch is the one that ended it, not the 2 s
    # default, and the unwinding adds no wait of its own
    assert elapsed < 0.5, elapsed
    assert rnc.dprc_device_error(reset=True) == bnd.DPRC_DEVERR_READY
    assert torch.all(n == SENTINEL), n  # no sample was finished
    # the context is usable: zero the workspace (its counters were left
    # mid-call) and run the same layers normally
    ws.zero_()
    n2 = torch.zeros(B, device=DEV)
    _normal_call(Ad, Gd, Pd, n2, ws)
    torch.cuda.synchronize()
    assert rnc.dprc_device_error(reset=True) == 0
    ref = _oracle_sum(As, Gs, Ps)
    np.testing.assert_allclose(n2.cpu().double().numpy(), ref, rtol=RTOL)


def test_a_launch_of_the_wrong_cluster_shape_is_refused():
    name, B, T, dims = SHAPES[0]
    As, Gs, Ps = _layers(32, B, T, dims)
    Ad = [a.to(DEV) for a in As]
    Gd = [g.to(DEV) for g in Gs]
    Pd = [p.to(DEV) for p in Ps]
    ws = _workspace(As, Gs, Ps)
    n = torch.full((B,), SENTINEL, device=DEV)
    rnc.dprc_test_hutch_fault(bnd.FAULT_CLUSTER_SHAPE, WAIT_NS, Ad, Gd, Pd, n, ws)
    torch.cuda.synchronize()
    assert rnc.dprc_device_error(reset=True) == bnd.DPRC_DEVERR_LAUNCH
    assert torch.all(n == SENTINEL), n
    assert int(ws.count_nonzero()) == 0  # nothing was touched
    # the same workspace, as it is, serves a normal call
    n2 = torch.zeros(B, device=DEV)
    _normal_call(Ad, Gd, Pd, n2, ws)
    torch.cuda.synchronize()
    assert rnc.dprc_device_error(reset=True) == 0
    np.testing.assert_allclose(n2.cpu().double().numpy(), _oracle_sum(As, Gs, Ps), rtol=RTOL)


def test_the_hook_rejects_a_plan_that_already_uses_clusters():
    name, B, T, dims = SHAPES[1]
    As, Gs, Ps = _layers(33, B, T, dims)
    ws = _workspace(As, Gs, Ps)
    n = torch.zeros(B, device=DEV)
    with pytest.raises(rnc.DprcError) as e:
        rnc.dprc_test_hutch_fault(bnd.FAULT_CLUSTER_SHAPE, WAIT_NS, [As[0].to(DEV)],
                                  [Gs[0].to(DEV)], [Ps[0].to(DEV)], n, ws)
    assert e.value.status == 2
