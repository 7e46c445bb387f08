"""Analytic FLOP and memory counts for the norm routines of DP-SGD-RC.

TEST INFRASTRUCTURE ONLY (see the package docstring).

These are the counts under which the pages' efficiency numbers come out; the
tests check them against the printed values.  Sources: "Efficient DP-SGD for
LLMs with Randomized Clipping", papernotes.org, "Experiments > Ablation"
(efficiency table for the 8192 x 2048 layer at T = 4096, k = 32), and the
gist.science summary, "Complexiteitsreductie" (FGC O(BTpd), GC O(BT^2(p+d)),
DP-SGD-RC O(BTk(p+d)); 128x fewer FLOPs than GC at T = 4096, k = 32).
All counts are per sample and per layer (the factor B cancels in every ratio).
"""

from __future__ import annotations


def flops_fgc(T, d, p):
    """Materialise A^T G (d x p, K = T): 2 T d p."""
    return 2 * T * d * p


def flops_ghost(T, d, p):
    """The two T x T Grams A A^T (K = d) and G G^T (K = p): 2 T^2 (d + p)."""
    return 2 * T * T * (d + p)


def flops_hutch(T, d, p, k):
    """W = G P (T x k, K = p) plus Y = A^T W (d x k, K = T): 2 T k (p + d)."""
    return 2 * T * k * (p + d)


def flops_hutchpp(T, d, p, k):
    """Four k-column Hutchinson-sized products (Z, M, and the head and tail
    blocks), each 2 T k (p + d), with the pages' k columns per block."""
    return 4 * flops_hutch(T, d, p, k)


def norm_memory_fgc(d, p):
    """Norm workspace of FGC: the d x p per-sample gradient."""
    return d * p


def norm_memory_hutch(T, k):
    """Norm workspace of Hutchinson: the T x k sketch G P."""
    return T * k


def norm_memory_hutchpp(T, k):
    """Norm workspace of Hutch++: three T x k sketches."""
    return 3 * T * k
