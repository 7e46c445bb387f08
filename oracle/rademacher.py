"""Oracle for the +-1 (Rademacher) projection variant of the Hutchinson estimate.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Efficient DP-SGD for LLMs with Randomized Clipping" (papernotes.org,
"Experiments > Ablation", on where the memory savings end) notes that the
projection P itself becomes the memory bottleneck as k grows, and names a
{-1, +1} one-bit projection in the style of Achlioptas as the way to shrink it
further, with the caveat that the privacy analysis would have to be redone.
The pages give no formula for it; this library's reading:

  n_hat_i = (1/k) || A_i^T (G_i S) ||_F^2,   S in {-1, +1}^{p x k},

with independent, equally likely signs, so E[S S^T] = k I and the estimate is
unbiased (the Gaussian P ~ N(0, 1/k) becomes S / sqrt(k); the 1/k is applied
to the squared norm, where it is exact for powers of two).

Signs come from the same Philox4x32-10 stream as the noise (oracle.philox):
entry (u, v) has linear index e = u * k + v; its bit is bit (e & 31) of word
((e >> 5) & 3) of block (e >> 7) of the stream of (seed, step); bit 0 gives +1,
bit 1 gives -1.  This layout is the library's convention, not the pages'.
"""

from __future__ import annotations

import numpy as np

from .norms import _f64
from .philox import philox_words


def rademacher_signs(seed, step, p, k):
    """S [p][k] in {-1, +1} (float64) from the Philox stream of (seed, step)."""
    n = p * k
    n_blocks = (n + 127) // 128
    words = philox_words(seed, step, 0, n_blocks).reshape(-1)  # word w = block w>>2, word w&3
    e = np.arange(n, dtype=np.int64)
    bits = (words[e >> 5].astype(np.uint64) >> (e & 31).astype(np.uint64)) & np.uint64(1)
    return (1.0 - 2.0 * bits.astype(np.float64)).reshape(p, k)


def hutch_norm_rademacher(A, G, S):
    """(1/k) ||A_i^T (G_i S)||_F^2 for a given sign matrix S [p][k]; float64 [B].

    Same evaluation order as the Gaussian estimate: the T x k sketch W = G_i S,
    then Y = A_i^T W, then the squared Frobenius norm, scaled by 1/k.
    """
    A, G, S = _f64(A), _f64(G), _f64(S)
    k = S.shape[1]
    out = np.empty(A.shape[0])
    for i in range(A.shape[0]):
        W = G[i] @ S
        Y = A[i].T @ W
        out[i] = np.sum(Y * Y) / k
    return out


def rademacher_variance(A, G, k):
    """Closed-form variance of the estimate for one sample pair (A, G):
    with O = G^T A A^T G and independent Rademacher columns,
    Var[n_hat] = (2/k) (||O||_F^2 - sum_j O_jj^2)."""
    A, G = _f64(A), _f64(G)
    O = G.T @ A @ A.T @ G
    return 2.0 / k * (np.sum(O * O) - np.sum(np.diag(O) ** 2))
