"""The CUDA path as an estimator: many independent projections through the C ABI.

Parity at fixed projections checks the arithmetic; these tests check that
what the kernels compute behaves as the method's estimator over 10^4 draws
("Efficient DP-SGD for LLMs with Randomized Clipping", papernotes.org, "Key
design > Hutchinson random projection": n_hat = trace(P^T O P) with P_uv ~
N(0, 1/k) is unbiased for trace(O) = ||A^T G||_F^2; the privacy analysis
("f-DP") uses its law, a chi^2 mixture sum_j lambda_j chi^2_j(k) / k, which
for a rank-one O is trace(O) chi^2(k) / k).  A stale or reused projection
tile, a wrong scale or a dropped column would pass a fixed-P parity check at
the tested seeds and fail these.

  - unbiasedness: the mean of 10^4 estimates is within 4 standard errors of
    the exact norm, with the closed-form variance 2 ||O||_F^2 / k (Gaussian P)
    or (2/k)(||O||_F^2 - sum_j O_jj^2) (the +-1 projection), and the sample
    variance matches that law;
  - the chi^2(k) law for a rank-one O (T = 1), by a Kolmogorov-Smirnov test,
    with chi^2(k - 1) and chi^2(2k) rejected;
  - Hutch++ over fresh P for a fixed S: the mean is trace(O) and the variance
    2 ||O_res||_F^2 / r, O_res the part of O outside the head's span.

Shapes: the single-layer fp32 configuration (B4 T128 d = p = 64, k = 8:
CUDA-core path) and a bf16 layer that takes the one-launch tensor-core kernel
(B2 T256 d = p = 256, k = 32).  The projections are drawn on the GPU from a
seeded generator; the exact norms and the laws come from the float64 oracle.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import randomized_norm_clipping_gb300 as rnc
from randomized_norm_clipping_gb300 import workloads as wl
from randomized_norm_clipping_gb300.workloads import to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DRAWS = 10_000


@pytest.fixture(scope="module", autouse=True)
def _built():
    from randomized_norm_clipping_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rnc.dprc_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert rnc.dprc_device_error() == 0


def _gram(A, G):
    """O_i = G_i^T A_i A_i^T G_i per sample (float64, from the exact inputs)."""
    Af, Gf = to_f64(A), to_f64(G)
    return [Gf[i].T @ Af[i] @ Af[i].T @ Gf[i] for i in range(Af.shape[0])]


def _gaussian_draws(A, G, k, seed):
    """[DRAWS][B] estimates, one fresh P ~ N(0, 1/k) per draw (rounded to the
    inputs' dtype, as the caller would store it)."""
    B, T, d = A.shape
    p = G.shape[2]
    g = torch.Generator(device=DEV).manual_seed(seed)
    Ps = (torch.randn(DRAWS, p, k, generator=g, device=DEV) / math.sqrt(k)).to(A.dtype)
    out = _rows(B)
    ws = rnc.workspace(rnc.DPRC_OP_HUTCH, A, B, T, d, p, k)
    for j in range(DRAWS):
        rnc.dprc_norm_hutch(A, G, Ps[j], out[j, :B], ws=ws)
    torch.cuda.synchronize()
    return out[:, :B].double().cpu().numpy(), Ps


def _rows(B):
    """[DRAWS][B] outputs, each row 16-byte aligned (the library's rule)."""
    return torch.zeros(DRAWS, (B + 3) // 4 * 4, device=DEV)


def _fp32_case(T=None, seed_shift=0):
    wk = wl.WORKLOADS["hutch_b4_t128_64x64_k8_f32"]
    wk = wl.Workload(**{**wk.__dict__, "seed": wk.seed + seed_shift})
    A, G, _ = wl.layer_inputs(wk, 0, device=DEV, T=T)
    return A, G, wk.k


def _bf16_case(B=2, T=256, d=256, p=256, seed=17):
    g = torch.Generator(device=DEV).manual_seed(seed)
    A = torch.randn(B, T, d, generator=g, device=DEV).to(torch.bfloat16)
    G = (torch.randn(B, T, p, generator=g, device=DEV) * 0.05).to(torch.bfloat16)
    return A, G


def _check_unbiased(x, O, var_of, var_tol=0.10):
    """Per sample: mean within 4 standard errors of trace(O), sample variance
    within var_tol of the closed form (its relative standard deviation over
    10^4 draws is 1 to 3 % for these laws)."""
    for i, Oi in enumerate(O):
        var = var_of(Oi)
        se = math.sqrt(var / x.shape[0])
        assert abs(x[:, i].mean() - np.trace(Oi)) < 4.0 * se, (i, x[:, i].mean(), np.trace(Oi), se)
        assert abs(x[:, i].var() / var - 1.0) < var_tol, (i, x[:, i].var(), var)


def test_gaussian_estimate_is_unbiased_fp32_path():
    A, G, k = _fp32_case()
    assert rnc.dprc_norm_hutch_launches(rnc.DPRC_F32, *A.shape, G.shape[2], k) == 3
    x, _ = _gaussian_draws(A, G, k, seed=101)
    _check_unbiased(x, _gram(A, G), lambda O: 2.0 * np.sum(O * O) / k)


def test_gaussian_estimate_is_unbiased_fused_tensor_core_path():
    A, G = _bf16_case()
    k = 32
    assert rnc.dprc_norm_hutch_launches(rnc.DPRC_BF16, *A.shape, G.shape[2], k) == 1
    x, _ = _gaussian_draws(A, G, k, seed=102)
    # the bf16-rounded P keeps E[P P^T] = I to rounding (relative 2^-9, either
    # sign), far inside four standard errors of 10^4 draws
    _check_unbiased(x, _gram(A, G), lambda O: 2.0 * np.sum(O * O) / k)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rank_one_law_is_chi2_k(dtype):
    # T = 1: O_i = (g_i g_i^T) ||a_i||^2 has rank one, and k n_hat_i / trace(O_i)
    # ~ chi^2(k) exactly for P ~ N(0, 1/k) (the single-chi^2 case of the
    # pages' chi^2-mixture law)
    if dtype == "f32":
        A, G, k = _fp32_case(T=1, seed_shift=5)
    else:
        A, G = _bf16_case(B=2, T=1, d=256, p=256, seed=23)
        k = 32
    x, _ = _gaussian_draws(A, G, k, seed=103)
    tr = np.array([np.trace(O) for O in _gram(A, G)])
    import scipy.stats as st
    for i in range(x.shape[1]):
        z = k * x[:, i] / tr[i]
        assert st.kstest(z, st.chi2(k).cdf).pvalue > 1e-3, i
        assert st.kstest(z, st.chi2(k - 1).cdf).pvalue < 1e-6, i
        assert st.kstest(z, st.chi2(2 * k).cdf).pvalue < 1e-6, i


@pytest.mark.parametrize("path", ["fp32", "fused"])
def test_plus_minus_one_estimate_is_unbiased_with_its_variance_law(path):
    # n_hat = (1/k) ||A^T G S||^2 with independent Rademacher columns: unbiased,
    # Var = (2/k) (||O||_F^2 - sum_j O_jj^2); the signs of draw j come from the
    # Philox stream of (seed, step = j)
    if path == "fp32":
        A, G, k = _fp32_case(seed_shift=9)
    else:
        A, G = _bf16_case(seed=29)
        k = 32
    B, T, d = A.shape
    p = G.shape[2]
    out = _rows(B)
    ws = rnc.workspace(rnc.DPRC_OP_HUTCH_PM1, A, B, T, d, p, k)
    for j in range(DRAWS):
        rnc.dprc_norm_hutch_pm1(A, G, k, 4242, j, out[j, :B], ws=ws)
    torch.cuda.synchronize()
    x = out[:, :B].double().cpu().numpy()
    _check_unbiased(x, _gram(A, G),
                    lambda O: 2.0 / k * (np.sum(O * O) - np.sum(np.diag(O) ** 2)), var_tol=0.15)


def test_draws_are_independent_of_each_other():
    # a projection tile reused across calls would correlate consecutive draws:
    # the lag-1 correlation of the Gaussian draws is within 4 / sqrt(n) of 0
    A, G = _bf16_case(seed=31)
    x, _ = _gaussian_draws(A, G, 32, seed=104)
    for i in range(x.shape[1]):
        c = np.corrcoef(x[:-1, i], x[1:, i])[0, 1]
        assert abs(c) < 4.0 / math.sqrt(DRAWS), (i, c)


def test_hutchpp_tail_is_unbiased_given_the_head():
    # Hutch++ (papernotes.org, "Key design > Hutch++ head-tail decomposition"):
    # for a fixed S the head ||X Q||^2 is exact and the tail (1/r)||X P'||^2,
    # P' = (I - Q Q^T) P with P ~ N(0, 1), is unbiased for trace(O_res),
    # O_res = (I - Q Q^T) O (I - Q Q^T), with variance 2 ||O_res||_F^2 / r.  So
    # over fresh P the estimates average to trace(O) = ||A^T G||_F^2 exactly.
    # Run through the tensor-core path whose third pass streams X M and forms
    # X Q = (X M) R^-1 in its epilogue: a wrong factor, scale or C in that
    # step would bias the mean or change the variance.
    B, T, d, p, r = 2, 256, 256, 256, 16
    g = torch.Generator(device=DEV).manual_seed(37)
    A = torch.randn(B, T, d, generator=g, device=DEV).to(torch.bfloat16)
    U = torch.randn(B, T, 8, generator=g, device=DEV)
    V = torch.randn(B, p, 8, generator=g, device=DEV)
    G = (torch.bmm(U, V.transpose(1, 2)) / math.sqrt(8)
         + 0.3 * torch.randn(B, T, p, generator=g, device=DEV)).to(torch.bfloat16)
    S = torch.randn(p, r, generator=g, device=DEV).to(torch.bfloat16)
    draws = 4000
    Ps = torch.randn(draws, p, r, generator=g, device=DEV).to(torch.bfloat16)
    out = _rows(B)[:draws]
    ws = rnc.workspace(rnc.DPRC_OP_HUTCHPP, A, B, T, d, p, r)
    for j in range(draws):
        rnc.dprc_norm_hutchpp(A, G, S, Ps[j], out[j, :B], ws=ws)
    torch.cuda.synchronize()
    x = out[:, :B].double().cpu().numpy()
    Af, Gf, Sf = to_f64(A), to_f64(G), to_f64(S)
    for i in range(B):
        X = Af[i].T @ Gf[i]
        O = X.T @ X
        Q, _ = np.linalg.qr(O @ Sf)
        Pr = np.eye(p) - Q @ Q.T
        Ores = Pr @ O @ Pr
        var = 2.0 * np.sum(Ores * Ores) / r
        se = math.sqrt(var / draws)
        assert abs(x[:, i].mean() - np.trace(O)) < 4.0 * se, (i, x[:, i].mean(), np.trace(O), se)
        assert abs(x[:, i].var() / var - 1.0) < 0.15, (i, x[:, i].var(), var)
