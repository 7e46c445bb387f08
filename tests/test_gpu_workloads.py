"""Parity at the benchmark's configurations, in the launch shapes it times.

Each configuration is drawn by `workloads.layer_inputs` on the GPU, run
through the C ABI with the full batch, and compared with the float64 oracle
on the same bytes: every sample where the oracle is quick, a sampled subset
(stated per test) where it is not.  Tolerance: relative 1e-3 on n and on the
clip factors (bf16 inputs, fp32 accumulation).
"""

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


def _relerr(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-300))


def _clip_both_branches(n_gpu, ref):
    # C = 1 (the workloads' value: every sample clips) and C = the median
    # sqrt(n), so both branches of min(1, C / sqrt(n)) are exercised
    for C in (1.0, float(np.median(np.sqrt(ref)))):
        c = torch.empty_like(n_gpu)
        rnc.dprc_clip_factors(n_gpu, C, c)
        assert _relerr(c.cpu(), oracle.clip_factors(ref, C)) < RTOL, C


def test_single_fp32_layer_b4_t128():
    wk = wl.WORKLOADS["hutch_b4_t128_64x64_k8_f32"]
    A, G, P = wl.layer_inputs(wk, 0, device=DEV)
    n = torch.zeros(wk.B, device=DEV)
    rnc.dprc_norm_hutch(A, G, P, n)
    ref = oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))
    assert _relerr(n.cpu(), ref) < 1e-5  # fp32 inputs, fp32 arithmetic
    e = torch.zeros(wk.B, device=DEV)
    rnc.dprc_exact_norm(A, G, e)
    assert _relerr(e.cpu(), oracle.exact_norm(to_f64(A), to_f64(G))) < 1e-5
    _clip_both_branches(n, ref)


def test_q_proj_b8_t4096_every_sample():
    wk = wl.WORKLOADS[wl.HEADLINE]
    A, G, P = wl.layer_inputs(wk, 0, device=DEV)
    n = torch.zeros(wk.B, device=DEV)
    rnc.dprc_norm_hutch(A, G, P, n)
    ref = oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P))
    assert _relerr(n.cpu(), ref) < RTOL
    _clip_both_branches(n, ref)
    assert rnc.dprc_device_error() == 0


def test_llama_block_layer_by_layer_sum_and_clip():
    # the first decoder block of the 112-layer workload (q, k, v, o, gate, up,
    # down at B = 4, T = 4096), accumulated into one n as the step does
    wk = wl.WORKLOADS["hutch_llama32_1b_112layers_b4_t4096_k32_bf16"]
    n = torch.zeros(wk.B, device=DEV)
    refs = []
    for j in range(len(wl.LLAMA32_1B_BLOCK)):
        A, G, P = wl.layer_inputs(wk, j, device=DEV)
        rnc.dprc_norm_hutch(A, G, P, n, accumulate=j > 0)
        refs.append(oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(P)))
        del A, G, P
    ref = oracle.layer_sum(refs)
    assert _relerr(n.cpu(), ref) < RTOL
    _clip_both_branches(n, ref)


def test_c3_112_layers_in_the_launches_the_benchmark_times():
    # The exact call bench.py times for the 112-layer step: one
    # dprc_norm_hutch_layers_clip over all 112 Llama-3.2-1B layers at B = 4,
    # T = 4096 (two persistent launches of 56 layers, clusters chosen by
    # shape), the layerwise sum and the clip factors in the launch that adds
    # the last layer, on one reused workspace.  The oracle runs every layer
    # and every sample, one sample at a time (a layer widened to float64 is
    # up to 2 GB).  Both branches of the clip rule: C = 1 (every sample clips)
    # and C = the median sqrt(n), each through the same launches.
    wk = wl.WORKLOADS["hutch_llama32_1b_112layers_b4_t4096_k32_bf16"]
    assert len(wk.layers) == 112
    layers = [wl.layer_inputs(wk, i, device=DEV) for i in range(len(wk.layers))]
    As = [x[0] for x in layers]
    Gs = [x[1] for x in layers]
    Ps = [x[2] for x in layers]
    wsz = rnc.dprc_workspace_bytes(rnc.DPRC_OP_HUTCH_LAYERS, rnc.DPRC_BF16, wk.B, wk.T,
                                   max(lay.d for lay in wk.layers),
                                   max(lay.p for lay in wk.layers), wk.k)
    wsbuf = torch.zeros(wsz, dtype=torch.uint8, device=DEV)
    n = torch.zeros(wk.B, device=DEV)
    c = torch.empty(wk.B, device=DEV)
    rnc.dprc_norm_hutch_layers(As, Gs, Ps, n, ws=wsbuf, C=wk.C, c=c)
    torch.cuda.synchronize()
    assert rnc.dprc_device_error() == 0
    per_layer = []
    for A, G, P in layers:
        Pf = to_f64(P)
        per_layer.append(np.concatenate(
            [oracle.hutch_norm(to_f64(A[i:i + 1]), to_f64(G[i:i + 1]), Pf)
             for i in range(wk.B)]))
    ref = oracle.layer_sum(per_layer)
    assert _relerr(n.cpu(), ref) < RTOL
    assert _relerr(c.cpu(), oracle.clip_factors(ref, wk.C)) < RTOL
    C2 = float(np.median(np.sqrt(ref)))
    c_ref2 = oracle.clip_factors(ref, C2)
    assert np.any(c_ref2 < 1) and np.any(c_ref2 == 1)
    n2 = torch.zeros(wk.B, device=DEV)
    c2 = torch.empty(wk.B, device=DEV)
    rnc.dprc_norm_hutch_layers(As, Gs, Ps, n2, ws=wsbuf, C=C2, c=c2)
    torch.cuda.synchronize()
    assert torch.equal(n2, n)  # the layer sum is added in a fixed order
    assert _relerr(c2.cpu(), c_ref2) < RTOL
    assert rnc.dprc_device_error() == 0


def test_hutchpp_q_proj_b8_t4096_every_sample():
    wk = wl.WORKLOADS["hutchpp_q_proj_b8_t4096_r16_bf16"]
    A, G, (S, P) = wl.layer_inputs(wk, 0, device=DEV)
    n = torch.zeros(wk.B, device=DEV)
    rnc.dprc_norm_hutchpp(A, G, S, P, n)
    ref = oracle.hutchpp_norm(to_f64(A), to_f64(G), to_f64(S), to_f64(P))
    assert _relerr(n.cpu(), ref) < RTOL
    assert rnc.dprc_device_error() == 0


def test_exact_both_forms_q_proj_b32_t1024_sampled():
    # the short-sequence exact-norm row of the benchmark: q_proj widths at
    # T = 1024, B = 32, where the ghost form does half the direct form's work;
    # every form on the full batch, the oracle on every fourth sample
    wk = wl.WORKLOADS[wl.HEADLINE]
    lay = wk.layers[0]
    B, T = 32, 1024
    A, G, _ = wl.layer_inputs(wk, 0, device=DEV, B=B, T=T)
    idx = list(range(0, B, 4))
    ref = oracle.exact_norm(to_f64(A[idx]), to_f64(G[idx]))
    assert rnc.dprc_exact_norm_plan(rnc.DPRC_BF16, B, T, lay.d, lay.p) != rnc.DPRC_EXACT_DIRECT
    for form in (rnc.DPRC_EXACT_AUTO, rnc.DPRC_EXACT_DIRECT, rnc.DPRC_EXACT_GHOST_N128,
                 rnc.DPRC_EXACT_GHOST_N256):
        n = torch.zeros(B, device=DEV)
        rnc.dprc_exact_norm(A, G, n, form=form)
        assert _relerr(n[idx].cpu(), ref) < RTOL, form
    assert rnc.dprc_device_error() == 0


@pytest.mark.parametrize("layer", [0, 1])
def test_long_context_b2_t32768_every_sample(layer):
    # the full B = 2 launch; the oracle checks both samples, one at a time
    # (one sample of T = 32768 widened to float64 is up to 2.7 GB)
    wk = wl.WORKLOADS["hutch_long_b2_t32768_up_down_k32_bf16"]
    A, G, P = wl.layer_inputs(wk, layer, device=DEV)
    n = torch.zeros(wk.B, device=DEV)
    rnc.dprc_norm_hutch(A, G, P, n)
    Pf = to_f64(P)
    ref = np.concatenate([oracle.hutch_norm(to_f64(A[i:i + 1]), to_f64(G[i:i + 1]), Pf)
                          for i in range(wk.B)])
    assert _relerr(n.cpu(), ref) < RTOL
    _clip_both_branches(n, ref)
