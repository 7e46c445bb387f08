"""Pins for the float64 oracle: each check ties it to something other than itself
(brute force, hand-worked values, distribution laws, the pages' printed ratios,
an independent Philox implementation).  CPU only."""

import json
import math
import os

import numpy as np
import pytest
import scipy.stats as st

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _int_case(rng, B, T, d, p, lo=-3, hi=3):
    A = rng.integers(lo, hi + 1, size=(B, T, d)).astype(np.float64)
    G = rng.integers(lo, hi + 1, size=(B, T, p)).astype(np.float64)
    return A, G


# --------------------------------------------------------------------------
# exact norm: identity ||A^T G||^2 = trace(G^T A A^T G) = sum (AA^T)(GG^T)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(3, 5, 4, 3), (2, 1, 6, 2), (2, 7, 1, 5), (1, 9, 3, 8)])
def test_exact_forms_equal_brute_force_on_integers(shape):
    rng = np.random.default_rng(11)
    A, G = _int_case(rng, *shape)
    brute = oracle.brute_force_norm(A.tolist(), G.tolist())
    # integer inputs: every form is exact in float64, so equality is exact
    assert np.array_equal(oracle.exact_norm(A, G), brute)
    assert np.array_equal(oracle.ghost_norm(A, G), brute)
    assert np.array_equal(oracle.trace_norm(A, G), brute)


def test_exact_norm_hand_cases():
    for case in _load("hand_norms.json")["exact"]:
        A = np.array([case["A"]], dtype=np.float64)
        G = np.array([case["G"]], dtype=np.float64)
        for f in (oracle.exact_norm, oracle.ghost_norm, oracle.trace_norm):
            assert f(A, G)[0] == case["n"], (f.__name__, case["why"])


def test_exact_norm_empty_sequence_is_zero():
    A = np.zeros((2, 0, 3))
    G = np.zeros((2, 0, 4))
    assert np.array_equal(oracle.exact_norm(A, G), [0.0, 0.0])
    assert np.array_equal(oracle.ghost_norm(A, G), [0.0, 0.0])


# --------------------------------------------------------------------------
# Hutchinson
# --------------------------------------------------------------------------

def test_hutch_hand_cases():
    for case in _load("hand_norms.json")["hutch"]:
        A = np.array([case["A"]], dtype=np.float64)
        G = np.array([case["G"]], dtype=np.float64)
        P = np.array(case["P"], dtype=np.float64)
        assert oracle.hutch_norm(A, G, P)[0] == case["n_hat"], case["why"]


@pytest.mark.parametrize("shape", [(3, 6, 5, 4), (2, 128, 64, 64)])
def test_hutch_with_identity_projection_is_exact(shape):
    # P = I_p (k = p): trace(P^T O P) = trace(O), exactly on integer inputs
    rng = np.random.default_rng(5)
    A, G = _int_case(rng, *shape)
    P = np.eye(shape[3])
    assert np.array_equal(oracle.hutch_norm(A, G, P), oracle.exact_norm(A, G))


def test_hutch_is_linear_in_column_blocks():
    # ||A^T G [P1 | P2]||^2 = ||A^T G P1||^2 + ||A^T G P2||^2 (sum over columns)
    rng = np.random.default_rng(6)
    A, G = _int_case(rng, 2, 7, 5, 6)
    P1 = rng.integers(-2, 3, size=(6, 3)).astype(np.float64)
    P2 = rng.integers(-2, 3, size=(6, 4)).astype(np.float64)
    both = oracle.hutch_norm(A, G, np.concatenate([P1, P2], axis=1))
    assert np.array_equal(both, oracle.hutch_norm(A, G, P1) + oracle.hutch_norm(A, G, P2))


def _hutch_draws(A, G, k, n_draws, seed):
    rng = np.random.default_rng(seed)
    p = G.shape[2]
    return np.array([oracle.hutch_norm(A, G, rng.normal(0.0, 1.0 / math.sqrt(k), size=(p, k)))[0]
                     for _ in range(n_draws)])


@pytest.mark.parametrize("which", ["T1", "d1"])
def test_hutch_rank_one_law_is_scaled_chi2(which):
    # rank-one O (T = 1, or d = 1 which is the DP-SGD-JL case):
    # k * n_hat / trace(O) ~ chi^2(k) exactly when P_uv ~ N(0, 1/k)
    rng = np.random.default_rng(21)
    k = 8
    if which == "T1":
        A, G = rng.normal(size=(1, 1, 6)), rng.normal(size=(1, 1, 5))
    else:
        A, G = rng.normal(size=(1, 9, 1)), rng.normal(size=(1, 9, 5))
    tr = oracle.trace_norm(A, G)[0]
    x = k * _hutch_draws(A, G, k, 10_000, seed=3) / tr
    assert st.kstest(x, st.chi2(k).cdf).pvalue > 1e-3
    # and a wrong law (k - 1 or 2k degrees of freedom) is rejected
    assert st.kstest(x, st.chi2(k - 1).cdf).pvalue < 1e-6
    assert st.kstest(x, st.chi2(2 * k).cdf).pvalue < 1e-6


def test_hutch_unbiased_and_variance_law():
    # E[n_hat] = trace(O); Var[n_hat] = 2 ||O||_F^2 / k for Gaussian P ~ N(0, 1/k)
    rng = np.random.default_rng(8)
    A, G = rng.normal(size=(1, 12, 7)), rng.normal(size=(1, 12, 6))
    k, n = 4, 10_000
    O = G[0].T @ A[0] @ A[0].T @ G[0]
    var = 2.0 * np.sum(O * O) / k
    x = _hutch_draws(A, G, k, n, seed=4)
    assert abs(x.mean() - np.trace(O)) < 4.0 * math.sqrt(var / n)
    # sample variance within 10% (its relative std here is ~3%)
    assert abs(x.var() / var - 1.0) < 0.10


# --------------------------------------------------------------------------
# Hutch++
# --------------------------------------------------------------------------

@pytest.mark.parametrize("rank", [1, 8, 16])
def test_hutchpp_exact_when_rank_at_most_r(rank):
    rng = np.random.default_rng(30 + rank)
    B, T, d, p, r = 2, 40, 24, 32, 16
    A = rng.normal(size=(B, T, d))
    G = np.stack([rng.normal(size=(T, rank)) @ rng.normal(size=(rank, p)) for _ in range(B)])
    S, P = rng.normal(size=(p, r)), rng.normal(size=(p, r))
    est = oracle.hutchpp_norm(A, G, S, P)
    np.testing.assert_allclose(est, oracle.exact_norm(A, G), rtol=1e-10)
    head, tail, _ = oracle.hutchpp_parts(A, G, S, P)
    assert np.all(tail <= 1e-12 * head)


@pytest.mark.parametrize("d", [1, 5, 16])
def test_hutchpp_exact_when_activations_limit_the_rank(d):
    # rank(O) = rank(G^T A A^T G) <= d: with d <= r the estimate is exact even
    # though G itself is full rank, so the sketch must be of O, not of G^T G.
    rng = np.random.default_rng(40 + d)
    B, T, p, r = 2, 48, 40, 16
    A = rng.normal(size=(B, T, d))
    G = rng.normal(size=(B, T, p))
    S, P = rng.normal(size=(p, r)), rng.normal(size=(p, r))
    np.testing.assert_allclose(oracle.hutchpp_norm(A, G, S, P), oracle.exact_norm(A, G), rtol=1e-9)


def test_hutchpp_full_width_sketch_has_no_tail():
    rng = np.random.default_rng(9)
    A, G = rng.normal(size=(2, 10, 5)), rng.normal(size=(2, 10, 6))
    S, P = rng.normal(size=(6, 6)), rng.normal(size=(6, 6))
    head, tail, _ = oracle.hutchpp_parts(A, G, S, P)
    np.testing.assert_allclose(head, oracle.exact_norm(A, G), rtol=1e-10)
    assert np.all(tail < 1e-18 * head)


def test_hutchpp_unbiased_given_the_sketch():
    # For a fixed S (hence Q), E_P[n_hat] = trace(Q^T O Q) + trace((I-QQ^T) O) = trace(O),
    # with Var = 2 ||(I-QQ^T) O (I-QQ^T)||_F^2 / r.
    rng = np.random.default_rng(12)
    T, d, p, r, n = 30, 9, 20, 4, 10_000
    A, G = rng.normal(size=(1, T, d)), rng.normal(size=(1, T, p))
    S = rng.normal(size=(p, r))
    _, _, Qs = oracle.hutchpp_parts(A, G, S, rng.normal(size=(p, r)))
    Q = Qs[0]
    O = G[0].T @ A[0] @ A[0].T @ G[0]
    R = np.eye(p) - Q @ Q.T
    var = 2.0 * np.sum((R @ O @ R) ** 2) / r
    draws = np.array([oracle.hutchpp_norm(A, G, S, rng.normal(size=(p, r)))[0] for _ in range(n)])
    assert abs(draws.mean() - np.trace(O)) < 4.0 * math.sqrt(var / n)


def test_hutchpp_invariant_to_orthonormal_basis():
    # n_hat depends on span(Q) only: modified Gram-Schmidt, or Q times a random
    # rotation and sign flips, give the same estimate as the Householder basis.
    rng = np.random.default_rng(13)
    A, G = rng.normal(size=(2, 25, 11)), rng.normal(size=(2, 25, 14))
    S, P = rng.normal(size=(14, 5)), rng.normal(size=(14, 5))

    def mgs(M):
        Q = np.array(M, dtype=np.float64)
        for j in range(Q.shape[1]):
            for i in range(j):
                Q[:, j] -= (Q[:, i] @ Q[:, j]) * Q[:, i]
            Q[:, j] /= np.linalg.norm(Q[:, j])
        return Q

    rot, _ = np.linalg.qr(rng.normal(size=(5, 5)))

    def rotated(M):
        Q, _ = np.linalg.qr(M)
        return Q @ rot

    ref = oracle.hutchpp_norm(A, G, S, P)
    np.testing.assert_allclose(oracle.hutchpp_norm(A, G, S, P, mgs), ref, rtol=1e-10)
    np.testing.assert_allclose(oracle.hutchpp_norm(A, G, S, P, rotated), ref, rtol=1e-10)


def test_hutchpp_matches_hutch_when_head_is_empty():
    # With a basis Q of directions G never touches (G Q = 0) the head is 0 and
    # G P' = G P, so the estimate reduces to Hutchinson with P, scaled by 1/r.
    rng = np.random.default_rng(14)
    T, d, p, r = 6, 4, 10, 2
    A = rng.normal(size=(1, T, d))
    G = np.zeros((1, T, p))
    G[0, :, :5] = rng.normal(size=(T, 5))        # G lives in the first 5 coordinates
    S = rng.normal(size=(p, r))
    P = rng.normal(size=(p, r))

    def outside(M):
        Q = np.zeros((p, r))
        Q[5, 0] = 1.0
        Q[6, 1] = 1.0                            # directions G never touches
        return Q

    est = oracle.hutchpp_norm(A, G, S, P, outside)[0]
    assert np.isclose(est, oracle.hutch_norm(A, G, P)[0] / r, rtol=1e-12)


# --------------------------------------------------------------------------
# layerwise sum and clip
# --------------------------------------------------------------------------

def test_layer_sum():
    per_layer = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0]])
    assert np.array_equal(oracle.layer_sum(per_layer), [111.0, 222.0])


def test_clip_hand_cases():
    for case in _load("hand_norms.json")["clip"]["cases"]:
        got = oracle.clip_factors(np.array([case["n"]]), case["C"])[0]
        assert got == pytest.approx(case["c"], rel=1e-15), case


def test_clip_nonfinite_and_negative_give_zero():
    n = np.array([np.nan, np.inf, -np.inf, -1.0, 0.0, 4.0])
    np.testing.assert_array_equal(oracle.clip_factors(n, 1.0), [0, 0, 0, 0, 1.0, 0.5])


def test_clip_is_monotone_and_bounded():
    n = np.logspace(-8, 8, 200)
    c = oracle.clip_factors(n, 3.0)
    assert np.all(np.diff(c) <= 0) and np.all(c <= 1) and np.all(c > 0)
    # the clipped norm sqrt(n) * c never exceeds C
    assert np.all(np.sqrt(n) * c <= 3.0 * (1 + 1e-15))


# --------------------------------------------------------------------------
# analytic cost model vs the pages' printed efficiency table
# --------------------------------------------------------------------------

def test_cost_model_reproduces_printed_savings():
    g = _load("efficiency_ablation.json")
    T, k = g["T"], g["k"]
    cost = oracle.cost
    for which in ("largest", "smallest"):
        d, p = g[f"{which}_layer"]
        fgc = cost.flops_fgc(T, d, p)
        hutch = 100.0 * (1 - cost.flops_hutch(T, d, p, k) / fgc)
        assert round(hutch, 2) == g["flops_saving_pct"]["hutch"][which]
        # Hutch++ ~ 4 Hutchinson-sized products; the printed value carries a small
        # extra term (QR) the pages do not spell out, so agree to 0.1 points
        hpp = 100.0 * (1 - cost.flops_hutchpp(T, d, p, k) / fgc)
        assert abs(hpp - g["flops_saving_pct"]["hutchpp"][which]) < 0.1
    d, p = g["largest_layer"]
    mem = 100.0 * (1 - cost.norm_memory_hutch(T, k) / cost.norm_memory_fgc(d, p))
    assert round(mem, 2) == g["peak_memory_saving_excluding_inputs_pct"]["hutch"]
    mempp = 100.0 * (1 - cost.norm_memory_hutchpp(T, k) / cost.norm_memory_fgc(d, p))
    assert abs(mempp - g["peak_memory_saving_excluding_inputs_pct"]["hutchpp"]) < 0.01
    gc = g["flop_reduction_vs_ghost_clipping"]
    # GC / DP-SGD-RC = 2T^2(p+d) / 2Tk(p+d) = T / k, any layer shape
    for d, p in ((2048, 2048), (8192, 2048), (2048, 512)):
        ratio = cost.flops_ghost(gc["T"], d, p) / cost.flops_hutch(gc["T"], d, p, gc["k"])
        assert ratio == gc["factor"]


# --------------------------------------------------------------------------
# Philox4x32-10 and the normal transform
# --------------------------------------------------------------------------

def _triton_philox(seed, c0, c1, c2, c3):
    """Words from triton's own Philox4x32 (run by its CPU interpreter): an
    implementation of the SC'11 generator independent of the oracle's."""
    os.environ["TRITON_INTERPRET"] = "1"
    triton = pytest.importorskip("triton")
    tl = pytest.importorskip("triton.language")
    import torch

    @triton.jit
    def kern(c_ptr, out_ptr, seed, N: tl.constexpr):
        i = tl.arange(0, N)
        a = tl.load(c_ptr + 4 * i + 0)
        b = tl.load(c_ptr + 4 * i + 1)
        c = tl.load(c_ptr + 4 * i + 2)
        d = tl.load(c_ptr + 4 * i + 3)
        w0, w1, w2, w3 = tl.philox(seed, a, b, c, d)
        tl.store(out_ptr + 4 * i + 0, w0)
        tl.store(out_ptr + 4 * i + 1, w1)
        tl.store(out_ptr + 4 * i + 2, w2)
        tl.store(out_ptr + 4 * i + 3, w3)

    n = len(c0)
    ctr = np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32).view(np.int32)
    cin = torch.from_numpy(ctr.reshape(-1).copy())
    out = torch.zeros(4 * n, dtype=torch.int32)
    kern[(1,)](cin, out, seed, N=n)
    return out.numpy().view(np.uint32).reshape(n, 4)


def test_philox_matches_independent_implementation():
    rng = np.random.default_rng(99)
    n = 64
    c = rng.integers(0, 2**32, size=(4, n), dtype=np.uint64)
    c[:, 0] = 0                          # the all-zero counter
    c[:, 1] = 0xFFFFFFFF                 # the all-ones counter
    for seed in (0, 1, 0x1234567890ABCDEF, 2**64 - 1):
        ref = _triton_philox(seed, *c)
        got = np.stack(oracle.philox4x32_10(*c, seed & 0xFFFFFFFF, seed >> 32), axis=1)
        assert np.array_equal(got, ref), hex(seed)


def test_philox_stream_layout_matches_independent_implementation():
    # block j of (seed, step) = Philox(counter = (j_lo, j_hi, step_lo, step_hi), key = seed)
    seed, step = 0xDEADBEEF12345678, (7 << 32) | 3
    first = (1 << 32) - 5                # crosses the j_lo carry into j_hi
    words = oracle.philox_words(seed, step, first, 16)
    j = np.arange(16, dtype=np.uint64) + np.uint64(first)
    ref = _triton_philox(seed, j & 0xFFFFFFFF, j >> 32,
                         np.full(16, step & 0xFFFFFFFF, np.uint64), np.full(16, step >> 32, np.uint64))
    assert np.array_equal(words, ref)


def test_philox_words_are_uniform_and_distinct():
    w = oracle.philox_words(42, 0, 0, 250_000).reshape(-1)
    u = w.astype(np.float64) / 2**32
    assert st.kstest(u, "uniform").pvalue > 1e-3
    assert len(np.unique(w)) > 0.9998 * w.size      # ~116 expected collisions of 1e6 draws
    # each bit is fair
    bits = ((w[:, None] >> np.arange(32, dtype=np.uint32)) & 1).mean(axis=0)
    assert np.all(np.abs(bits - 0.5) < 5 * 0.5 / math.sqrt(w.size))


def test_normals_are_standard_and_pairs_uncorrelated():
    z = oracle.noise_normals(1_000_000, seed=2024, step=5)
    assert abs(z.mean()) < 5.0 / 1000.0
    assert abs(z.var() - 1.0) < 5.0 * math.sqrt(2.0) / 1000.0
    assert st.kstest(z, "norm").pvalue > 1e-3
    zz = z.reshape(-1, 4)
    for a, b in ((0, 1), (2, 3), (0, 2), (1, 3)):
        assert abs(np.corrcoef(zz[:, a], zz[:, b])[0, 1]) < 5.0 / math.sqrt(len(zz))


def test_uniform_endpoints():
    # u1 in (0, 1] keeps log finite: the extreme words give the extreme normals
    w = np.array([[0, 0, 0xFFFFFFFF, 0xFFFFFFFF]], dtype=np.uint32)
    z = oracle.normals_from_words(w)[0]
    r_max = math.sqrt(-2.0 * math.log(2.0 ** -24))
    assert z[0] == pytest.approx(r_max, rel=1e-15)   # u1 = 2^-24, u2 = 0: cos = 1
    assert z[1] == 0.0
    assert z[2] == 0.0 and z[3] == 0.0               # u1 = 1: radius 0


def test_noise_stream_is_offset_consistent():
    full = oracle.noise_normals(1001, seed=3, step=9)
    part = oracle.noise_normals(500, seed=3, step=9, first_element=333)
    assert np.array_equal(full[333:833], part)
    g = np.linspace(-1, 1, 1001)
    out = oracle.add_noise(g, sigma=0.5, C=2.0, seed=3, step=9)
    np.testing.assert_allclose(out - g, 1.0 * full, rtol=0, atol=1e-15)
    # a different step or seed gives an independent stream
    other = oracle.noise_normals(1001, seed=3, step=10)
    assert abs(np.corrcoef(full, other)[0, 1]) < 0.15


# ---------------------------------------------------------------------------
# +-1 (Rademacher) projection variant
# ---------------------------------------------------------------------------

def test_rademacher_bit_layout_follows_the_philox_words():
    # k = 32: row u of S is word u of the stream, least significant bit first
    S = oracle.rademacher_signs(seed=5, step=3, p=8, k=32)
    w = oracle.philox_words(5, 3, 0, 2).reshape(-1)  # 8 words
    for u in range(8):
        bits = [(int(w[u]) >> b) & 1 for b in range(32)]
        assert list(S[u]) == [1.0 - 2.0 * b for b in bits]
    # k = 16: two rows per word, the even row in the low half
    S16 = oracle.rademacher_signs(seed=5, step=3, p=4, k=16)
    assert list(S16[1]) == [1.0 - 2.0 * ((int(w[0]) >> (16 + b)) & 1) for b in range(16)]


def test_rademacher_signs_are_balanced_and_plus_minus_one():
    S = oracle.rademacher_signs(seed=11, step=0, p=1024, k=1024)
    assert set(np.unique(S)) == {-1.0, 1.0}
    assert abs(S.mean()) < 4.0 / np.sqrt(S.size)


def test_rademacher_estimate_is_exact_when_o_is_diagonal():
    # G = I_p and A with orthogonal rows make O = A A^T diagonal; then
    # (1/k) sum_v s_v^T O s_v = trace(O) for any signs
    rng = np.random.default_rng(3)
    p, d, k = 12, 5, 8
    A = np.diag(rng.uniform(0.5, 2.0, size=p)) @ np.eye(p)[:, :d]  # T = p, A A^T diagonal
    G = np.eye(p)
    S = oracle.rademacher_signs(seed=1, step=1, p=p, k=k)
    got = oracle.hutch_norm_rademacher(A[None], G[None], S)[0]
    assert abs(got - oracle.exact_norm(A[None], G[None])[0]) <= 1e-12 * got


def test_rademacher_estimate_is_unbiased_with_its_variance_law():
    rng = np.random.default_rng(4)
    T, d, p, k, draws = 6, 5, 7, 4, 4000
    A = rng.standard_normal((1, T, d))
    G = rng.standard_normal((1, T, p))
    exact = oracle.exact_norm(A, G)[0]
    vals = np.array([oracle.hutch_norm_rademacher(A, G, oracle.rademacher_signs(s, 0, p, k))[0]
                     for s in range(draws)])
    var = oracle.rademacher_variance(A[0], G[0], k)
    assert abs(vals.mean() - exact) < 4.0 * np.sqrt(var / draws)
    assert abs(vals.var() / var - 1.0) < 0.15
    # smaller than the Gaussian law 2 ||O||_F^2 / k whenever O has a diagonal
    O = G[0].T @ A[0] @ A[0].T @ G[0]
    assert var < 2.0 / k * np.sum(O * O)
