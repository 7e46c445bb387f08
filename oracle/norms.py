"""Float64 oracle for the per-sample, per-layer gradient-norm path of DP-SGD-RC.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "Efficient DP-SGD for LLMs with Randomized Clipping" (ICML 2026), page
notes at papernotes.org, sections "Method > Overall framework" and
"Method > Key design" (Hutchinson random projection; Hutch++ head/tail split),
and the gist.science technical summary, section "Methodologie > Kernmechanisme".

Notation follows the pages.  For one linear-like layer and sample i:
  A_i in R^{T x d}   input activations (forward hook),
  G_i in R^{T x p}   output gradients (backward hook),
  the per-sample weight gradient is A_i^T G_i (d x p), and its squared
  Frobenius norm is n_i = ||A_i^T G_i||_F^2 = trace(G_i^T A_i A_i^T G_i)
  = trace(O_i) with O_i = G_i^T A_i A_i^T G_i (p x p).

Batched arrays are laid out [B][T][d] and [B][T][p]; projections are [p][k].
All arithmetic is float64; inputs of any float dtype are widened exactly.
"""

from __future__ import annotations

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Exact norm: three algebraically equal forms of ||A^T G||_F^2
# (papernotes, "Research background": the exact per-sample norm the method
#  replaces; "Key design > Hutchinson": the trace identity).
# ---------------------------------------------------------------------------

def exact_norm(A, G):
    """Direct form: n_i = sum_{a,b} (sum_t A_i[t,a] G_i[t,b])^2.

    Materialises the d x p per-sample gradient A_i^T G_i (the Fast Gradient
    Clipping route the pages contrast with) and sums its squares.
    Returns float64 [B].
    """
    A, G = _f64(A), _f64(G)
    out = np.empty(A.shape[0])
    for i in range(A.shape[0]):
        grad = A[i].T @ G[i]                     # d x p
        out[i] = np.sum(grad * grad)
    return out


def ghost_norm(A, G):
    """Ghost-clipping form: n_i = sum_{t,s} (A_i A_i^T)_{ts} (G_i G_i^T)_{ts}.

    The T x T Gram route whose O(T^2) memory the method avoids (papernotes,
    "Research background"; gist.science, "Complexiteitsreductie").  Only
    sensible for small T.  Returns float64 [B].
    """
    A, G = _f64(A), _f64(G)
    out = np.empty(A.shape[0])
    for i in range(A.shape[0]):
        out[i] = np.sum((A[i] @ A[i].T) * (G[i] @ G[i].T))
    return out


def trace_norm(A, G):
    """Trace form: n_i = trace(O_i), O_i = G_i^T A_i A_i^T G_i (p x p).

    The identity ||A^T G||_F^2 = trace(G^T A A^T G) is the starting point of
    the method (papernotes, "Key design > Hutchinson"; gist.science,
    "Kernmechanisme").  Returns float64 [B].
    """
    A, G = _f64(A), _f64(G)
    out = np.empty(A.shape[0])
    for i in range(A.shape[0]):
        O = G[i].T @ A[i] @ A[i].T @ G[i]
        out[i] = np.trace(O)
    return out


def brute_force_norm(A, G):
    """Pure-Python loops over every index: the per-sample gradient entry
    g[a][b] = sum_t A[t][a] * G[t][b], then sum of g^2.  Tiny inputs only."""
    out = []
    for Ai, Gi in zip(A, G):
        T, d, p = len(Ai), len(Ai[0]), len(Gi[0])
        total = 0.0
        for a in range(d):
            for b in range(p):
                g = 0.0
                for t in range(T):
                    g += float(Ai[t][a]) * float(Gi[t][b])
                total += g * g
        out.append(total)
    return np.array(out, dtype=np.float64)


# ---------------------------------------------------------------------------
# Hutchinson estimator (papernotes, "Key design > Hutchinson random projection";
# gist.science, "Kernmechanisme" item 1).
# ---------------------------------------------------------------------------

def hutch_norm(A, G, P):
    """Hutchinson estimate n_hat_i = trace(P^T O_i P) = ||A_i^T (G_i P)||_F^2.

    P in R^{p x k} is one projection shared by the whole batch (the memory term
    is O(BkT + kp), so P is not per-sample), with entries drawn N(0, 1/k) by the
    caller.  The pages' evaluation order: first the T x k sketch W = G_i P,
    then Y = A_i^T W (d x k), then ||Y||_F^2; neither the d x p gradient nor a
    T x T matrix is formed.  Returns float64 [B].
    """
    A, G, P = _f64(A), _f64(G), _f64(P)
    out = np.empty(A.shape[0])
    for i in range(A.shape[0]):
        W = G[i] @ P                  # T x k sketch
        Y = A[i].T @ W                # d x k
        out[i] = np.sum(Y * Y)
    return out


# ---------------------------------------------------------------------------
# Hutch++ head/tail estimator (papernotes, "Key design > Hutch++ head-tail
# decomposition"; gist.science, "Kernmechanisme" item 2).
# Reading: the sketch is taken on the p side, O_i = G_i^T A_i A_i^T G_i, with
# S, P in R^{p x r} ~ N(0, 1) and the tail scaled by 1/r (Hutch++'s own
# normalisation), i.e.
#   n_hat = ||A^T G Q||_F^2 + (1/r) ||A^T G (I - Q Q^T) P||_F^2,
#   Q = orthonormal basis of Col(O S).
# ---------------------------------------------------------------------------

def _householder_q(M):
    """Thin Q (p x r) of a Householder QR of M (library QR as one step)."""
    Q, _ = np.linalg.qr(M, mode="reduced")
    return Q


def hutchpp_parts(A, G, S, P, orthonormalize=_householder_q):
    """Per-sample (head, tail_sum, Q list) of Hutch++.

    Steps, in the order the pages give them:
      1. Z = A_i^T (G_i S)                    (d x r)
      2. M = G_i^T (A_i Z) = O_i S            (p x r)
      3. Q = orthonormal basis of Col(M)      (p x r, thin QR)
      4. head = ||A_i^T (G_i Q)||_F^2 = trace(Q^T O_i Q)
      5. P' = (I - Q Q^T) P = P - Q (Q^T P)
      6. tail_sum = ||A_i^T (G_i P')||_F^2
    ``orthonormalize`` may be replaced to check invariance to the basis choice.
    """
    A, G, S, P = _f64(A), _f64(G), _f64(S), _f64(P)
    heads, tails, Qs = [], [], []
    for i in range(A.shape[0]):
        Z = A[i].T @ (G[i] @ S)
        M = G[i].T @ (A[i] @ Z)
        Q = orthonormalize(M)
        Yh = A[i].T @ (G[i] @ Q)
        Pp = P - Q @ (Q.T @ P)
        Yt = A[i].T @ (G[i] @ Pp)
        heads.append(np.sum(Yh * Yh))
        tails.append(np.sum(Yt * Yt))
        Qs.append(Q)
    return np.array(heads), np.array(tails), Qs


def hutchpp_norm(A, G, S, P, orthonormalize=_householder_q):
    """Hutch++ estimate n_hat_i = head_i + tail_sum_i / r.  Returns float64 [B]."""
    r = np.shape(P)[1]
    head, tail, _ = hutchpp_parts(A, G, S, P, orthonormalize)
    return head + tail / r


# ---------------------------------------------------------------------------
# Layerwise sum and clip factors (papernotes, "Method > Overall framework").
# ---------------------------------------------------------------------------

def layer_sum(per_layer):
    """n_i = sum_l n_hat_i^(l) over the linear-like layers.  per_layer: [L][B]."""
    return np.sum(_f64(per_layer), axis=0)


def clip_factors(n, C):
    """c_i = min(1, C / sqrt(n_i)).

    Reading: n_i estimates the SQUARED norm, so the clip scale takes its square
    root (the overall-framework paragraph writes min(C/sqrt(n_i), 1)).
    n_i == 0 gives 1.  A non-finite or negative n_i gives 0: a sample whose
    norm is unknown contributes nothing rather than passing unclipped.
    """
    n = _f64(n)
    C = float(C)
    out = np.zeros_like(n)
    ok = np.isfinite(n) & (n >= 0)
    with np.errstate(divide="ignore"):
        scale = np.where(n[ok] > 0, C / np.sqrt(np.where(n[ok] > 0, n[ok], 1.0)), np.inf)
    out[ok] = np.minimum(1.0, scale)
    return out
