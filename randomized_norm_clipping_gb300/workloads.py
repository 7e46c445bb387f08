"""Seeded synthetic workloads for the norm-estimation path.

This module only draws inputs; it holds none of the method's arithmetic.  The
tests feed the same bytes to the CUDA library and to the float64 oracle, and
``bench.py`` times the library on them.

Shapes follow the pages' setting ("Efficient DP-SGD for LLMs with Randomized
Clipping": Llama-3.2-1B linear layers, context T = 4096, projection width
k = 32; the efficiency ablation uses the 8192 x 2048 and 2048 x 512 layers).
No dataset or trained weight is used: activations and gradients are Gaussian
stand-ins with the spectra stated per workload below.

Recipe (all draws from ``torch.Generator`` seeded as stated):
  A      ~ N(0, 1)                                       [B][T][d]
  G_i    = s_i * N(0, 1),  s_i = exp(-4 + z_i), z_i ~ N(0,1)  [B][T][p]
           (one s_i per sample, shared by every layer of a model)
  P      ~ N(0, 1/k)                                     [p][k]
  Hutch++: S, P ~ N(0, 1) [p][r];  G_i = U_i V_i^T / sqrt(8) + 0.05 E_i with
           U_i [T][8], V_i [p][8], E_i [T][p] all N(0, 1)  (rank-8 head).
Values are drawn in float32 and rounded once to the workload dtype.
"""

from __future__ import annotations

import dataclasses
import math

import torch

# Llama-3.2-1B linear layers per decoder block: (name, d_in, p_out).
LLAMA32_1B_BLOCK = (
    ("q_proj", 2048, 2048),
    ("k_proj", 2048, 512),
    ("v_proj", 2048, 512),
    ("o_proj", 2048, 2048),
    ("gate_proj", 2048, 8192),
    ("up_proj", 2048, 8192),
    ("down_proj", 8192, 2048),
)
LLAMA32_1B_BLOCKS = 16
# Parameter count of Llama-3.2-1B (tied embedding): the size of the aggregated
# gradient buffer the noise is added to.
LLAMA32_1B_PARAMS = 1_235_814_400


@dataclasses.dataclass(frozen=True)
class Layer:
    name: str
    d: int
    p: int


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    method: str                # "hutch" | "hutchpp"
    B: int
    T: int
    layers: tuple
    k: int
    dtype: str                 # "f32" | "bf16"
    C: float = 1.0
    sigma: float = 1.0
    noise_elems: int = 0       # 0: no noise step in this workload
    g_scale: str = "lognormal"  # "unit" | "lognormal" | "lowrank"
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self):
        return 4 if self.dtype == "f32" else 2


WORKLOADS = {
    # single linear layer, Hutchinson, fp32
    "hutch_b4_t128_64x64_k8_f32": Workload(
        "hutch_b4_t128_64x64_k8_f32", "hutch", 4, 128, (Layer("linear", 64, 64),), 8, "f32",
        g_scale="unit", seed=1000),
    # Llama-3.2-1B q_proj shape, Hutchinson
    "hutch_q_proj_b8_t4096_k32_bf16": Workload(
        "hutch_q_proj_b8_t4096_k32_bf16", "hutch", 8, 4096, (Layer("q_proj", 2048, 2048),), 32,
        "bf16", seed=2000),
    # full Llama-3.2-1B linear set, layerwise sum, clip, noise on the whole gradient
    "hutch_llama32_1b_112layers_b4_t4096_k32_bf16": Workload(
        "hutch_llama32_1b_112layers_b4_t4096_k32_bf16", "hutch", 4, 4096,
        tuple(Layer(f"l{b}.{n}", d, p) for b in range(LLAMA32_1B_BLOCKS)
              for (n, d, p) in LLAMA32_1B_BLOCK),
        32, "bf16", noise_elems=LLAMA32_1B_PARAMS, seed=3000),
    # Hutch++ on the q_proj shape, rank-8 head + 0.05 tail
    "hutchpp_q_proj_b8_t4096_r16_bf16": Workload(
        "hutchpp_q_proj_b8_t4096_r16_bf16", "hutchpp", 8, 4096, (Layer("q_proj", 2048, 2048),),
        16, "bf16", g_scale="lowrank", seed=4000),
    # long context, Hutchinson, up_proj and down_proj
    "hutch_long_b2_t32768_up_down_k32_bf16": Workload(
        "hutch_long_b2_t32768_up_down_k32_bf16", "hutch", 2, 32768,
        (Layer("up_proj", 2048, 8192), Layer("down_proj", 8192, 2048)), 32, "bf16", seed=5000),
}

# The workload the headline throughput is quoted on (q_proj, B=8, T=4096, k=32).
HEADLINE = "hutch_q_proj_b8_t4096_k32_bf16"


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def sample_scales(wl: Workload, device="cpu", B=None):
    """Per-sample gradient scales s_i (float32 [B], B = the workload's batch by
    default; a larger B appends draws from a second seed, so the first
    samples keep their scales)."""
    B = wl.B if B is None else B
    if wl.g_scale != "lognormal":
        return torch.ones(B, dtype=torch.float32, device=device)
    z = torch.randn(wl.B, generator=_gen(device, wl.seed + 7), device=device)
    if B > wl.B:
        extra = torch.randn(B - wl.B, generator=_gen(device, wl.seed + 8), device=device)
        z = torch.cat([z, extra])
    return torch.exp(-4.0 + z[:B])


def layer_inputs(wl: Workload, layer_index: int, device="cpu", B=None, T=None):
    """(A, G, proj) for one layer.  proj is P [p][k] for Hutchinson and the pair
    (S, P) [p][r] for Hutch++.  ``B``/``T`` override the workload's batch and
    sequence length (smaller cases with the same recipe)."""
    B = wl.B if B is None else B
    T = wl.T if T is None else T
    lay = wl.layers[layer_index]
    d, p, k = lay.d, lay.p, wl.k
    base = wl.seed + 10 * layer_index
    dt = wl.torch_dtype
    A = torch.randn(B, T, d, generator=_gen(device, base + 1), device=device).to(dt)
    if wl.g_scale == "lowrank":
        g = _gen(device, base + 2)
        U = torch.randn(B, T, 8, generator=g, device=device)
        V = torch.randn(B, p, 8, generator=g, device=device)
        E = torch.randn(B, T, p, generator=g, device=device)
        G = (torch.bmm(U, V.transpose(1, 2)) / math.sqrt(8.0) + 0.05 * E).to(dt)
        del U, V, E
    else:
        s = sample_scales(wl, device, B)
        G = (torch.randn(B, T, p, generator=_gen(device, base + 2), device=device)
             * s.view(B, 1, 1)).to(dt)
    if wl.method == "hutchpp":
        S = torch.randn(p, k, generator=_gen(device, base + 3), device=device).to(dt)
        P = torch.randn(p, k, generator=_gen(device, base + 4), device=device).to(dt)
        return A, G, (S, P)
    P = (torch.randn(p, k, generator=_gen(device, base + 3), device=device)
         / math.sqrt(k)).to(dt)
    return A, G, P


def gradient_buffer(n, seed=77, device="cpu"):
    """An fp32 stand-in for the aggregated clipped gradient (N(0, 1e-4))."""
    return torch.randn(n, generator=_gen(device, seed), device=device) * 1e-2


def to_f64(t):
    """Exact widening of a float tensor (any device) to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
