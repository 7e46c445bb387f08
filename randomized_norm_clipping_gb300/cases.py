"""Run one named case of the library a few times, for profilers.

    python -m randomized_norm_clipping_gb300.cases NAME [--reps R] [--warmup W]

Each case draws its seeded inputs on the current GPU, calls one entry point
W + R times on the current stream and prints the mean device time of the last
R calls.  The cases are the benchmark's configurations (or a stated smaller
slice of one, sized to stay above the 126 MB L2 so DRAM counters still mean
something), so a profiler run such as

    ncu --set full --clock-control none -k regex:colproj -s 2 -c 1 \\
        python -m randomized_norm_clipping_gb300.cases hutch_q_proj

captures one launch of the kernel on the workload the benchmark times.
"""

from __future__ import annotations

import argparse

import torch

from . import binding as rnc
from . import workloads as wl


def _hutch(name, layer=0, clip=False):
    wk = wl.WORKLOADS[name]
    lay = wk.layers[layer]
    A, G, P = wl.layer_inputs(wk, layer, device="cuda")
    n = torch.zeros(wk.B, device="cuda")
    c = torch.empty(wk.B, device="cuda")
    ws = rnc.workspace(rnc.DPRC_OP_HUTCH, A, wk.B, wk.T, lay.d, lay.p, wk.k)
    if clip:
        return lambda: rnc.dprc_norm_hutch_clip(A, G, P, n, wk.C, c, ws=ws)
    return lambda: rnc.dprc_norm_hutch(A, G, P, n, ws=ws)


def _lora(B, T, d, p, k, exact):
    g = torch.Generator(device="cuda").manual_seed(5)
    A = torch.randn(B, T, d, device="cuda", generator=g).to(torch.bfloat16)
    G = (torch.randn(B, T, p, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    P = (torch.randn(p, k, device="cuda", generator=g) / k ** 0.5).to(torch.bfloat16)
    n = torch.zeros(B, device="cuda")
    if exact:
        ws = rnc.workspace(rnc.DPRC_OP_EXACT, A, B, T, d, p, 0)
        return lambda: rnc.dprc_exact_norm(A, G, n, ws=ws)
    ws = rnc.workspace(rnc.DPRC_OP_HUTCH, A, B, T, d, p, k)
    return lambda: rnc.dprc_norm_hutch(A, G, P, n, ws=ws)


def _hutch_layers(B, T):
    wk = wl.WORKLOADS["hutch_llama32_1b_112layers_b4_t4096_k32_bf16"]
    nl = len(wl.LLAMA32_1B_BLOCK)
    layers = [wl.layer_inputs(wk, j, device="cuda", B=B, T=T) for j in range(nl)]
    As, Gs, Ps = [x[0] for x in layers], [x[1] for x in layers], [x[2] for x in layers]
    n = torch.zeros(B, device="cuda")
    ws = rnc.workspace(rnc.DPRC_OP_HUTCH_LAYERS, As[0], B, T, max(a.shape[2] for a in As),
                       max(g.shape[2] for g in Gs), wk.k)
    return lambda: rnc.dprc_norm_hutch_layers(As, Gs, Ps, n, ws=ws)


def _hutch_pm1(name):
    wk = wl.WORKLOADS[name]
    lay = wk.layers[0]
    A, G, _ = wl.layer_inputs(wk, 0, device="cuda")
    n = torch.zeros(wk.B, device="cuda")
    ws = rnc.workspace(rnc.DPRC_OP_HUTCH_PM1, A, wk.B, wk.T, lay.d, lay.p, wk.k)
    return lambda: rnc.dprc_norm_hutch_pm1(A, G, wk.k, 1234, 1, n, ws=ws)


def _hutchpp():
    wk = wl.WORKLOADS["hutchpp_q_proj_b8_t4096_r16_bf16"]
    lay = wk.layers[0]
    A, G, (S, P) = wl.layer_inputs(wk, 0, device="cuda")
    n = torch.zeros(wk.B, device="cuda")
    ws = rnc.workspace(rnc.DPRC_OP_HUTCHPP, A, wk.B, wk.T, lay.d, lay.p, wk.k)
    return lambda: rnc.dprc_norm_hutchpp(A, G, S, P, n, ws=ws)


def _noise(n_elems):
    grad = wl.gradient_buffer(n_elems, device="cuda")
    return lambda: rnc.dprc_add_noise(grad, 1.0, 1.0, 1234, 1)


def _exact(B, T, form=rnc.DPRC_EXACT_AUTO):
    wk = wl.WORKLOADS[wl.HEADLINE]
    lay = wk.layers[0]
    A, G, _ = wl.layer_inputs(wk, 0, device="cuda", B=B, T=T)
    n = torch.zeros(B, device="cuda")
    ws = rnc.workspace(rnc.DPRC_OP_EXACT, A, B, T, lay.d, lay.p, wk.k)
    return lambda: rnc.dprc_exact_norm(A, G, n, ws=ws, form=form)


def _clip():
    n = torch.rand(8, device="cuda") * 4.0
    c = torch.empty(8, device="cuda")
    return lambda: rnc.dprc_clip_factors(n, 1.0, c)


CASES = {
    # B8 T4096 d = p = 2048 k32 bf16 (268 MB of A and G)
    "hutch_q_proj": lambda: _hutch("hutch_q_proj_b8_t4096_k32_bf16"),
    # the same with the clip factors in the launch (the benchmark's step)
    "hutch_clip_q_proj": lambda: _hutch("hutch_q_proj_b8_t4096_k32_bf16", clip=True),
    # rank-16 adapter maps of the q_proj batch (B8 T4096; 135 MB of A and G)
    "lora_down_exact": lambda: _lora(8, 4096, 2048, 16, 32, True),
    "lora_down_hutch": lambda: _lora(8, 4096, 2048, 16, 32, False),
    "lora_up_exact": lambda: _lora(8, 4096, 16, 2048, 32, True),
    "lora_up_hutch": lambda: _lora(8, 4096, 16, 2048, 32, False),
    # B2 T32768 2048 -> 8192 and 8192 -> 2048, k32 bf16 (1.34 GB each)
    # the same batch with the +-1 projection generated in the kernel
    "hutch_pm1_q_proj": lambda: _hutch_pm1("hutch_q_proj_b8_t4096_k32_bf16"),
    "hutch_long_up": lambda: _hutch("hutch_long_b2_t32768_up_down_k32_bf16", 0),
    "hutch_long_down": lambda: _hutch("hutch_long_b2_t32768_up_down_k32_bf16", 1),
    # one Llama-3.2-1B decoder block (q, k, v, o, gate, up, down) in one
    # dprc_norm_hutch_layers call, B2 T2048 (0.37 GB of A and G)
    "hutch_layers_block_b2_t2048": lambda: _hutch_layers(2, 2048),
    # Hutch++ B8 T4096 d = p = 2048 r16 bf16
    "hutchpp_q_proj": _hutchpp,
    # the noise kernel on 2^27 fp32 elements (1.07 GB read + written), a slice of
    # the 1,235,814,400-element gradient: same per-element work, fewer elements
    "noise_2p27": lambda: _noise(1 << 27),
    "noise_llama32_1b": lambda: _noise(wl.LLAMA32_1B_PARAMS),
    # exact ghost norm on 2 samples of the q_proj batch, T = 1024
    "exact_q_proj_b2_t1024": lambda: _exact(2, 1024),
    # the ghost form on q_proj widths at T = 1024, B = 32 (268 MB of A and G),
    # Gram tiles 128 x 256 and 128 x 128
    "exact_ghost_n256_q_proj_b32_t1024": lambda: _exact(32, 1024, rnc.DPRC_EXACT_GHOST_N256),
    "exact_ghost_n128_q_proj_b32_t1024": lambda: _exact(32, 1024, rnc.DPRC_EXACT_GHOST_N128),
    "clip_b8": _clip,
}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    args = ap.parse_args(argv)
    fn = CASES[args.case]()
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    err = rnc.dprc_device_error()
    print(f"{args.case}: {e0.elapsed_time(e1) / max(args.reps, 1) * 1e3:.1f} us per call "
          f"(mean of {args.reps}), device error {err}")
    if err != 0:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
