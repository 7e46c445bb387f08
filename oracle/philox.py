"""Oracle for the Gaussian noise step: Philox4x32-10, uniform -> normal, noise add.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The method adds isotropic Gaussian noise sigma*C*N(0, I) to the aggregated
clipped gradient before the optimizer step ("Efficient DP-SGD for LLMs with
Randomized Clipping", papernotes.org, "Method > Overall framework" and
"Loss / training strategy"; the generic DP-SGD tutorial at intelliparadigm.com,
section 1.1, states the same Gaussian mechanism with variance sigma^2 C^2).
The pages do not name a generator.  This library draws the noise from the
counter-based Philox4x32-10 generator of Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), written here from that
paper's definition:

  round:  (hi0, lo0) = M0 * x0,  (hi1, lo1) = M1 * x2   (32x32 -> 64-bit)
          x' = (hi1 ^ x1 ^ k0,  lo1,  hi0 ^ x3 ^ k1,  lo0)
  key:    after every round  k0 += W0,  k1 += W1
  M0 = 0xD2511F53, M1 = 0xCD9E8D57, W0 = 0x9E3779B9, W1 = 0xBB67AE85; 10 rounds.

Stream layout (this library's convention): element e of the gradient uses word
(e & 3) of block j = e >> 2, where block j is Philox4x32-10 applied to the
counter (j_lo, j_hi, step_lo, step_hi) under the key (seed_lo, seed_hi).
Words pair up as (x0, x1) and (x2, x3); each pair gives two normals by the
Box-Muller transform with 24-bit uniforms
  u1 = ((x_a >> 8) + 1) * 2^-24  in (0, 1],   u2 = (x_b >> 8) * 2^-24  in [0, 1)
  z_a = sqrt(-2 ln u1) cos(2 pi u2),          z_b = sqrt(-2 ln u1) sin(2 pi u2).
"""

from __future__ import annotations

import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0, k1, rounds=10):
    """Philox4x32 with ``rounds`` rounds on uint32 arrays (vectorised numpy).

    Returns four uint32 arrays.  Arithmetic is carried in uint64 so that the
    32x32 -> 64-bit products are exact.
    """
    x0 = np.asarray(c0, dtype=np.uint64) & MASK32
    x1 = np.asarray(c1, dtype=np.uint64) & MASK32
    x2 = np.asarray(c2, dtype=np.uint64) & MASK32
    x3 = np.asarray(c3, dtype=np.uint64) & MASK32
    k0 = np.uint64(int(k0) & MASK32)
    k1 = np.uint64(int(k1) & MASK32)
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    w0, w1 = np.uint64(PHILOX_W0), np.uint64(PHILOX_W1)
    m32, s32 = np.uint64(MASK32), np.uint64(32)
    for _ in range(rounds):
        p0 = m0 * x0
        p1 = m1 * x2
        hi0, lo0 = p0 >> s32, p0 & m32
        hi1, lo1 = p1 >> s32, p1 & m32
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
        k0 = (k0 + w0) & m32
        k1 = (k1 + w1) & m32
    return tuple(v.astype(np.uint32) for v in (x0, x1, x2, x3))


def philox_words(seed, step, first_block, n_blocks):
    """Words of blocks [first_block, first_block + n_blocks) as uint32 [n, 4]."""
    seed, step = int(seed), int(step)
    j = np.arange(n_blocks, dtype=np.uint64) + np.uint64(first_block)
    words = philox4x32_10(j & np.uint64(MASK32), j >> np.uint64(32),
                          np.full(n_blocks, step & MASK32, dtype=np.uint64),
                          np.full(n_blocks, (step >> 32) & MASK32, dtype=np.uint64),
                          seed & MASK32, (seed >> 32) & MASK32)
    return np.stack(words, axis=1)


def normals_from_words(words):
    """Box-Muller on word pairs (x0,x1), (x2,x3) -> float64 normals [n, 4]."""
    w = np.asarray(words, dtype=np.uint64)
    out = np.empty(w.shape, dtype=np.float64)
    two_m24 = 2.0 ** -24
    for a, b in ((0, 1), (2, 3)):
        u1 = ((w[:, a] >> np.uint64(8)).astype(np.float64) + 1.0) * two_m24
        u2 = (w[:, b] >> np.uint64(8)).astype(np.float64) * two_m24
        r = np.sqrt(-2.0 * np.log(u1))
        out[:, a] = r * np.cos(2.0 * np.pi * u2)
        out[:, b] = r * np.sin(2.0 * np.pi * u2)
    return out


def noise_normals(N, seed, step, first_element=0):
    """The normals z_e for elements [first_element, first_element + N)."""
    if N == 0:
        return np.zeros(0)
    e0 = int(first_element)
    b0, b1 = e0 >> 2, (e0 + N - 1) >> 2
    z = normals_from_words(philox_words(seed, step, b0, b1 - b0 + 1)).reshape(-1)
    off = e0 - 4 * b0
    return z[off:off + N]


def add_noise(grad, sigma, C, seed, step, first_element=0):
    """grad + sigma * C * z  (float64), z from the stream above."""
    g = np.asarray(grad, dtype=np.float64)
    z = noise_normals(g.size, seed, step, first_element)
    return g + float(sigma) * float(C) * z.reshape(g.shape)
