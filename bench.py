"""Benchmark of the DP-SGD-RC norm-estimation hot path on GB300.

One step = one pass of the hot path over one batch of the headline workload
(Llama-3.2-1B q_proj shape: B = 8 per GPU, T = 4096, d = p = 2048, k = 32,
bf16): the Hutchinson estimate n_hat_i = ||A_i^T (G_i P)||_F^2 (sketch and
projection as two phases of one launch) and the clip factors
min(1, C / sqrt(n_i)) (in that launch's finishing step), one call of
dprc_norm_hutch_clip.

Metric: norm-estimation tokens/s (B*T per second per layer), whole job over
all ranks, plus the HBM roofline fraction of the dominant kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
  torchrun --nproc-per-node N bench.py --gpus N ...      (one rank per GPU)

After the headline, the other configurations of the path are timed the same
way and reported under "rows" (--rows all|none|c3,c4,c5,noise,exact): the
112-layer Llama-3.2-1B step with layerwise sum, clip and noise on the
1,235,814,400-element gradient; Hutch++; the T = 32768 up/down projections;
the noise kernel alone; and the exact ghost norm.

Ranks shard the batch (weak scaling: every rank runs its own B = 8 samples);
the norm path has no cross-rank exchange, so the only collectives are the
barriers and the max-over-ranks of the timed region.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from randomized_norm_clipping_gb300 import workloads as wl  # noqa: E402

METRIC = "norm-estimation tokens/s (B·T/s per layer) at k=32; % of HBM roofline"
UNIT = "tokens/s"


# ---------------------------------------------------------------- distributed

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device):
    """Max of a float across ranks (the job takes as long as its slowest rank)."""
    if ws == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_seed(base, rank):
    """Each rank draws its own batch (weak scaling)."""
    return base + 7919 * rank


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def ncu_traffic(kernel):
    """DRAM bytes per launch of the named headline kernel from the committed ncu
    capture, or None when the kernel's sources changed since it was taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic_hutch_q_proj.json")) as f:
            rec = json.load(f)["kernels"][kernel]
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        return int(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def measured_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


def headline_inputs(wk, rank, device):
    seeded = wl.Workload(**{**wk.__dict__, "seed": shard_seed(wk.seed, rank)})
    return wl.layer_inputs(seeded, 0, device=device)


def algorithmic_bytes(B, T, d, p, k, eb):
    """Bytes the method must move per launch: the sketch kernel reads G and P,
    the projection kernel reads A (the sketch it re-reads is the implementation's
    own intermediate, not counted)."""
    sketch = B * T * p * eb + p * k * eb
    project = B * T * d * eb
    return sketch, project


def cpu_oracle_rate(A, G, P, C, budget_s=12.0):
    """The float64 oracle on host cores, on whole samples of the same batch,
    repeated until ~budget_s of CPU work; returns (tokens/s, samples, seconds)."""
    import oracle
    B, T = A.shape[0], A.shape[1]
    Af = wl.to_f64(A)
    Gf = wl.to_f64(G)
    Pf = wl.to_f64(P)
    done, t0 = 0, time.perf_counter()
    while True:
        i = done % B
        n = oracle.hutch_norm(Af[i:i + 1], Gf[i:i + 1], Pf)
        oracle.clip_factors(n, C)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 20000:
            break
    return done * T / el, done, el


# ---------------------------------------------------------------- native arm

def run_native(args, rank, ws, local):
    import randomized_norm_clipping_gb300 as rnc

    device = torch.device("cuda", local)
    wk = wl.WORKLOADS[wl.HEADLINE]
    lay = wk.layers[0]
    B, T, d, p, k = wk.B, wk.T, lay.d, lay.p, wk.k
    A, G, P = headline_inputs(wk, rank, device)
    n = torch.zeros(B, device=device)
    c = torch.empty(B, device=device)
    wsbuf = rnc.workspace(rnc.DPRC_OP_HUTCH, A, B, T, d, p, k)
    stream = torch.cuda.current_stream(device)

    def step():
        # the layer's norms and the clip factors: one call
        rnc.dprc_norm_hutch_clip(A, G, P, n, wk.C, c, accumulate=False, ws=wsbuf)

    # kernels per step: one fused launch (the clip factors in its finishing
    # step), or sketch + projection + clip
    norm_launches = rnc.dprc_norm_hutch_launches(rnc.DPRC_BF16, B, T, d, p, k)
    launches_per_step = norm_launches if norm_launches == 1 else norm_launches + 1
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)

    # Eager rate: one Python call per kernel launch (host overhead included).
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(device)
    eager_ms = ev0.elapsed_time(ev1) / args.steps

    # The K timed steps captured as one CUDA graph (the way a training loop
    # captures its step): the GPU runs the K launches back to back, each a
    # programmatic dependent of the one before; one replay is the timed region.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(device)

    # keep the GPU loaded ~1.5 s so the clock samples cover a steady state
    with ClockSampler(local) as clk:
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 1.5:
            for _ in range(max(1, 500 // args.steps)):
                graph.replay()
            torch.cuda.synchronize(device)
        barrier(ws)
        torch.cuda.synchronize(device)
        torch.cuda._sleep(2_000_000)  # queue the replay behind ~1 ms of GPU work
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize(device)
        barrier(ws)
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, ws, device)
    ms_per_step = ms / args.steps
    value = ws * B * T / (ms_per_step * 1e-3)

    # Per-kernel durations: events between the two kernels of each call, with
    # the calls queued behind a GPU sleep so host launch gaps are not counted.
    reps = 20
    sets = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    for evs in sets:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize(device)
    torch.cuda._sleep(20_000_000)
    try:
        for evs in sets:
            rnc.dprc_set_phase_events(evs)
            rnc.dprc_norm_hutch(A, G, P, n, accumulate=False, ws=wsbuf)
    finally:
        rnc.dprc_set_phase_events(None)
    torch.cuda.synchronize(device)
    k1_ms = [evs[0].elapsed_time(evs[1]) for evs in sets]
    k2_ms = [evs[1].elapsed_time(evs[2]) for evs in sets]
    # whole call (both kernels, dependent launch active), queued the same way
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(20_000_000)
    e0.record(stream)
    for _ in range(reps):
        rnc.dprc_norm_hutch_clip(A, G, P, n, wk.C, c, accumulate=False, ws=wsbuf)
    e1.record(stream)
    torch.cuda.synchronize(device)
    call_ms = e0.elapsed_time(e1) / reps

    eb = wk.elem_bytes
    sk_bytes, pj_bytes = algorithmic_bytes(B, T, d, p, k, eb)
    k1 = float(np.mean(k1_ms))
    k2 = float(np.mean(k2_ms))
    peak, peak_kind = measured_peaks()
    if norm_launches == 1:
        # one kernel streams G, P and A, once per step: its average launch
        # duration is the timed region divided by the K launches in it
        dom, dom_ms, dom_bytes, dom_key = ("tc_hutch_kernel (sketch G P + projection "
                                           "A^T W, ||Y||^2, one launch)", ms_local / args.steps,
                                           sk_bytes + pj_bytes, "fused")
    elif k2 >= k1:
        dom, dom_ms, dom_bytes, dom_key = "colproj (A^T W, ||Y||^2)", k2, pj_bytes, "colproj"
    else:
        dom, dom_ms, dom_bytes, dom_key = "rowproj (G P)", k1, sk_bytes, "rowproj"
    traffic = ncu_traffic(dom_key)
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    op_achieved = (sk_bytes + pj_bytes) / (call_ms * 1e-3) / 1e9

    # end to end through the public API: pinned host inputs -> device -> call -> host result
    Ah = torch.empty(A.shape, dtype=A.dtype, pin_memory=True)
    Gh = torch.empty(G.shape, dtype=G.dtype, pin_memory=True)
    Ph = torch.empty(P.shape, dtype=P.dtype, pin_memory=True)
    Ah.copy_(A)
    Gh.copy_(G)
    Ph.copy_(P)
    ch = torch.empty(B, dtype=torch.float32, pin_memory=True)
    stage = rnc.host_stage(Ah, T, d, p, k, device=device)
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        # host tensors in, host n and c out: per-sample copies on the library's
        # copy stream, each sample's kernel under the next sample's copy
        rnc.dprc_norm_hutch_clip_host(Ah, Gh, Ph, wk.C, None, ch, stage=stage, stream=stream)

    e2e_step()
    torch.cuda.synchronize(device)
    barrier(ws)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, ws, device)
    h2d = (Ah.numel() + Gh.numel() + Ph.numel()) * eb
    d2h = ch.numel() * 4

    out = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded Gaussian activations/gradients, lognormal per-sample scale)",
        "config": {
            "workload": wk.name,
            "model": "Llama-3.2-1B q_proj shape",
            "global_batch": ws * B, "seq_len": T, "d": d, "p": p, "k": k,
            "parallelism": f"replicas x{ws} (samples sharded, no collective)",
            "l2": "inputs (268 MB per rank) larger than the 126 MB L2; no flush",
            "timed": "the K steps captured as one CUDA graph (one launch each), one replay",
            "eager_ms_per_step": eager_ms,
        },
        "roofline": {
            "bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "ms": dom_ms, "algorithmic_bytes": dom_bytes,
        },
        "roofline_op": {
            "what": "dprc_norm_hutch_clip called eagerly 20 times back to back (host launch "
                    "cost hidden behind a GPU sleep), algorithmic bytes A + G + P",
            "achieved": op_achieved, "peak": peak, "unit": "GB/s", "frac": op_achieved / peak,
            "ms": call_ms,
            "kernel_ms": ({"fused": k1} if norm_launches == 1 else {"rowproj": k1, "colproj": k2}),
        },
        "e2e": {"value": ws * B * T / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "dprc_norm_hutch_clip_host: pinned host A, G, P in, host clip factors out"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    which = set() if args.rows == "none" else (
        {"c3", "c4", "c5", "noise", "exact", "step", "pm1", "lora"} if args.rows == "all"
        else set(args.rows.split(",")))
    rows = measure_rows(which, device, peak, measured_tflops(), 7919 * rank) if which else {}
    if rank == 0 and not args.no_cpu_baseline:
        rate, done, el = cpu_oracle_rate(A.cpu(), G.cpu(), P.cpu(), wk.C)
        out["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": os.cpu_count(),
                               "kind": "oracle",
                               "sample": f"{done} whole samples (T={T}) of the same batch, "
                                         f"{el:.1f} s, float64 numpy (BLAS threads = cores)"}
        if rows:
            cpu_oracle_subsets(rows, device)
    if rows:
        # the full rows first; the line ends with a compact summary of them,
        # ordered so the 112-layer step, the noise, Hutch++ and the training
        # step come last (a reader of only the line's tail still sees them)
        out["rows_detail"] = rows
        out["rows"] = compact_rows(rows)
    return out


# ---------------------------------------------------------------- other rows

def _sig(x, digits=4):
    return float(f"{x:.{digits}g}") if isinstance(x, (int, float)) and x is not None else x


# compact summary: which fields of each row, in print order (the most
# important rows last)
_COMPACT = (
    ("exact_q_proj_b32_t1024", None),
    ("exact_c2", ("ms", "frac")),
    ("lora_down_r16", ("ms", "frac", "exact_ms", "exact_frac")),
    ("lora_up_r16", ("ms", "frac", "exact_ms", "exact_frac")),
    ("pm1_q_proj", ("ms", "frac")),
    ("c5_up_proj", ("ms", "frac", "tokens_per_s", "cpu_tokens_per_s")),
    ("c5_down_proj", ("ms", "frac", "tokens_per_s", "cpu_tokens_per_s")),
    ("c4_hutchpp", ("ms", "frac", "tokens_per_s", "cpu_tokens_per_s")),
    ("noise_1.24e9", ("ms", "frac", "cpu_ms")),
    ("dpsgd_rc_step_mlp", ("ms", "plain_backward_ms", "overhead")),
    ("c3_112layers", ("ms", "frac", "norms_ms", "norms_frac", "tokens_per_s_per_layer",
                      "cpu_tokens_per_s_per_layer", "clip_fraction")),
)


def compact_rows(rows):
    out = {}
    for name, fields in _COMPACT:
        if name not in rows:
            continue
        r = rows[name]
        if name == "exact_q_proj_b32_t1024":
            out[name] = {"auto": r["auto"], **{f"{k}_ms": _sig(v["ms"]) for k, v in r["forms"].items()},
                         **{f"{k}_frac": _sig(v["frac"], 3) for k, v in r["forms"].items()}}
            continue
        flat = dict(r)
        if "norms" in r:
            flat["norms_ms"] = r["norms"]["ms"]
            flat["norms_frac"] = r["norms"]["frac"]
        if "cpu_oracle" in r:
            flat.update({k: v for k, v in r["cpu_oracle"].items() if k != "sample"})
        out[name] = {k: _sig(flat[k], 3 if "frac" in k else 4) for k in fields if k in flat}
    return out


def cpu_oracle_subsets(rows, device):
    """The float64 oracle on the host cores on a stated subset of each row's
    workload, extrapolated linearly in samples and layers (the oracle's time
    per sample grows with T (d + p)); added to the rows as "cpu_oracle"."""
    import oracle

    def one_sample(wk, li):
        A, G, P = wl.layer_inputs(wk, li, device=device)
        if isinstance(P, tuple):
            args = (wl.to_f64(A[:1]), wl.to_f64(G[:1]), *[wl.to_f64(x) for x in P])
            fn = oracle.hutchpp_norm
        else:
            args = (wl.to_f64(A[:1]), wl.to_f64(G[:1]), wl.to_f64(P))
            fn = oracle.hutch_norm
        del A, G, P
        t0 = time.perf_counter()
        fn(*args)
        return time.perf_counter() - t0

    if "c4_hutchpp" in rows:
        wk = wl.WORKLOADS["hutchpp_q_proj_b8_t4096_r16_bf16"]
        t = one_sample(wk, 0)
        rows["c4_hutchpp"]["cpu_oracle"] = {
            "cpu_tokens_per_s": wk.T / t, "cores": os.cpu_count(),
            "sample": f"one sample (T={wk.T}) of the batch, {t:.2f} s"}
    for i, name in enumerate(("c5_up_proj", "c5_down_proj")):
        if name in rows:
            wk = wl.WORKLOADS["hutch_long_b2_t32768_up_down_k32_bf16"]
            t = one_sample(wk, i)
            rows[name]["cpu_oracle"] = {
                "cpu_tokens_per_s": wk.T / t, "cores": os.cpu_count(),
                "sample": f"one sample (T={wk.T}) of the B=2 batch, {t:.2f} s"}
    if "noise_1.24e9" in rows or "c3_112layers" in rows:
        wk = wl.WORKLOADS["hutch_llama32_1b_112layers_b4_t4096_k32_bf16"]
        sub = 1 << 20
        g = np.zeros(sub)
        t0 = time.perf_counter()
        oracle.add_noise(g, wk.sigma, wk.C, 1234, 1)
        t_noise = (time.perf_counter() - t0) * wk.noise_elems / sub
        if "noise_1.24e9" in rows:
            rows["noise_1.24e9"]["cpu_oracle"] = {
                "cpu_ms": 1e3 * t_noise, "cores": os.cpu_count(),
                "sample": f"{sub} elements, scaled to {wk.noise_elems}"}
        if "c3_112layers" in rows:
            nblock = len(wl.LLAMA32_1B_BLOCK)
            per_sample = sum(one_sample(wk, j) for j in range(nblock))
            t_norms = per_sample * wk.B * wl.LLAMA32_1B_BLOCKS
            rows["c3_112layers"]["cpu_oracle"] = {
                "cpu_tokens_per_s_per_layer": wk.B * wk.T * len(wk.layers) / t_norms,
                "cpu_step_ms": 1e3 * (t_norms + t_noise), "cores": os.cpu_count(),
                "sample": f"one sample of each of the {nblock} layer shapes of a block "
                          f"({per_sample:.2f} s), scaled by {wk.B} samples x "
                          f"{wl.LLAMA32_1B_BLOCKS} blocks; the noise on {sub} elements, "
                          f"scaled to {wk.noise_elems}"}

def graph_ms(fn, device, reps, warmup=3):
    """Mean device time of fn: reps calls captured as one CUDA graph, replayed
    once (queued behind a GPU sleep so host launch gaps are hidden)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize(device)
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(5_000_000)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize(device)
    del g
    return e0.elapsed_time(e1) / reps


def hbm_entry(ms, nbytes, peak, **extra):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": ms, "algorithmic_bytes": nbytes, "achieved_gbs": gbs, "frac": gbs / peak,
            **extra}


def hutch_bytes(B, T, d, p, k, eb):
    return B * T * (d + p) * eb + p * k * eb


def measure_rows(which, device, peak, tflops_peak, seed_shift):
    """Every other configuration of the path, each timed the same way as the
    headline (a CUDA graph of the whole row, inputs resident in HBM)."""
    import randomized_norm_clipping_gb300 as rnc

    rows = {}
    if "step" in which:
        # first: the eager step is sensitive to the allocator state the
        # multi-GB rows below leave behind
        rows["dpsgd_rc_step_mlp"] = measure_step(device)
        torch.cuda.empty_cache()

    def inputs(wk, i):
        seeded = wl.Workload(**{**wk.__dict__, "seed": wk.seed + seed_shift})
        return wl.layer_inputs(seeded, i, device=device)

    if "c3" in which or "noise" in which:
        wk = wl.WORKLOADS["hutch_llama32_1b_112layers_b4_t4096_k32_bf16"]
        grad = wl.gradient_buffer(wk.noise_elems, device=device)
        noise_bytes = 8 * wk.noise_elems
        t_noise = graph_ms(lambda: rnc.dprc_add_noise(grad, wk.sigma, wk.C, 1234, 1), device, 10)
        rows["noise_1.24e9"] = hbm_entry(t_noise, noise_bytes, peak,
                                         what="dprc_add_noise on the 1,235,814,400-element "
                                              "fp32 Llama-3.2-1B gradient (read + write)")
        if "c3" in which:
            layers = [inputs(wk, i) for i in range(len(wk.layers))]
            n = torch.zeros(wk.B, device=device)
            c = torch.empty(wk.B, device=device)
            wsz = rnc.dprc_workspace_bytes(rnc.DPRC_OP_HUTCH_LAYERS, rnc.DPRC_BF16, wk.B, wk.T,
                                           max(lay.d for lay in wk.layers),
                                           max(lay.p for lay in wk.layers), wk.k)
            wsbuf = torch.zeros(wsz, dtype=torch.uint8, device=device)

            As = [x[0] for x in layers]
            Gs = [x[1] for x in layers]
            Ps = [x[2] for x in layers]

            def norms():
                # one call for the whole layer list (two persistent launches)
                rnc.dprc_norm_hutch_layers(As, Gs, Ps, n, ws=wsbuf)

            def step():
                # the clip factors come with the launch that adds the last layer
                rnc.dprc_norm_hutch_layers(As, Gs, Ps, n, ws=wsbuf, C=wk.C, c=c)
                rnc.dprc_add_noise(grad, wk.sigma, wk.C, 1234, 1)

            norm_bytes = sum(hutch_bytes(wk.B, wk.T, lay.d, lay.p, wk.k, 2) for lay in wk.layers)
            t_norms = graph_ms(norms, device, 10)
            t_step = graph_ms(step, device, 10)
            rows["c3_112layers"] = hbm_entry(
                t_step, norm_bytes + noise_bytes, peak,
                what="dprc_norm_hutch_layers_clip over the 112 layers (layerwise sum and clip "
                     "factors) + noise, one graph",
                tokens_per_s_per_layer=wk.B * wk.T * len(wk.layers) / (t_norms * 1e-3),
                norms=hbm_entry(t_norms, norm_bytes, peak),
                clip_fraction=float((c < 1).float().mean().item()),
                launches=2 + 1)
            del layers, n, c, wsbuf
        del grad
        torch.cuda.empty_cache()

    if "c4" in which:
        wk = wl.WORKLOADS["hutchpp_q_proj_b8_t4096_r16_bf16"]
        lay = wk.layers[0]
        A, G, (S, P) = inputs(wk, 0)
        n = torch.zeros(wk.B, device=device)
        wsbuf = rnc.workspace(rnc.DPRC_OP_HUTCHPP, A, wk.B, wk.T, lay.d, lay.p, wk.k)
        t = graph_ms(lambda: rnc.dprc_norm_hutchpp(A, G, S, P, n, ws=wsbuf), device, 20)
        nb = 3 * wk.B * wk.T * (lay.d + lay.p) * 2 + 2 * lay.p * wk.k * 2
        rows["c4_hutchpp"] = hbm_entry(t, nb, peak, what="dprc_norm_hutchpp, three passes, the QR beside the third",
                                       tokens_per_s=wk.B * wk.T / (t * 1e-3))
        del A, G, S, P, n, wsbuf

    if "c5" in which:
        wk = wl.WORKLOADS["hutch_long_b2_t32768_up_down_k32_bf16"]
        n = torch.zeros(wk.B, device=device)
        for i, lay in enumerate(wk.layers):
            A, G, P = inputs(wk, i)
            wsbuf = rnc.workspace(rnc.DPRC_OP_HUTCH, A, wk.B, wk.T, lay.d, lay.p, wk.k)
            t = graph_ms(lambda: rnc.dprc_norm_hutch(A, G, P, n, ws=wsbuf), device, 20)
            rows[f"c5_{lay.name}"] = hbm_entry(
                t, hutch_bytes(wk.B, wk.T, lay.d, lay.p, wk.k, 2), peak,
                what=f"dprc_norm_hutch B2 T32768 {lay.d}->{lay.p}",
                tokens_per_s=wk.B * wk.T / (t * 1e-3))
            del A, G, P, wsbuf
        del n

    if "pm1" in which:
        wk = wl.WORKLOADS[wl.HEADLINE]
        lay = wk.layers[0]
        A, G, _ = inputs(wk, 0)
        n = torch.zeros(wk.B, device=device)
        wsbuf = rnc.workspace(rnc.DPRC_OP_HUTCH_PM1, A, wk.B, wk.T, lay.d, lay.p, wk.k)
        t = graph_ms(lambda: rnc.dprc_norm_hutch_pm1(A, G, wk.k, 99, 1, n, ws=wsbuf), device, 20)
        rows["pm1_q_proj"] = hbm_entry(
            t, wk.B * wk.T * (lay.d + lay.p) * 2, peak,
            what="dprc_norm_hutch_pm1 on the q_proj batch: +-1 projection generated in the "
                 "kernel (no P in memory), one launch",
            tokens_per_s=wk.B * wk.T / (t * 1e-3),
            ncu_traffic_bytes=ncu_traffic("pm1"))
        del A, G, n, wsbuf

    if "lora" in which:
        # LoRA adapters of the q_proj batch (B8 T4096, rank 16): the down map
        # 2048 -> 16 and the up map 16 -> 2048, by the estimate and the exact norm
        wk = wl.WORKLOADS[wl.HEADLINE]
        g = torch.Generator(device=device)
        g.manual_seed(4242 + seed_shift)
        r = 16
        for name, (d, p) in (("down", (2048, r)), ("up", (r, 2048))):
            A = torch.randn(wk.B, wk.T, d, generator=g, device=device).to(torch.bfloat16)
            G = (torch.randn(wk.B, wk.T, p, generator=g, device=device) * 0.02).to(torch.bfloat16)
            P = (torch.randn(p, wk.k, generator=g, device=device) / wk.k ** 0.5).to(torch.bfloat16)
            n = torch.zeros(wk.B, device=device)
            wsh = rnc.workspace(rnc.DPRC_OP_HUTCH, A, wk.B, wk.T, d, p, wk.k)
            wse = rnc.workspace(rnc.DPRC_OP_EXACT, A, wk.B, wk.T, d, p, wk.k)
            nbytes = wk.B * wk.T * (d + p) * 2
            th = graph_ms(lambda: rnc.dprc_norm_hutch(A, G, P, n, ws=wsh), device, 20)
            te = graph_ms(lambda: rnc.dprc_exact_norm(A, G, n, ws=wse), device, 20)
            rows[f"lora_{name}_r16"] = hbm_entry(
                th, nbytes, peak, exact_ms=te,
                exact_frac=nbytes / (te * 1e-3) / 1e9 / peak,
                what=f"LoRA {name} map {d} -> {p} on B8 T4096: dprc_norm_hutch (k=32) and "
                     "dprc_exact_norm; at rank <= k the exact norm moves the same bytes")
            del A, G, P, n, wsh, wse

    if "exact" in which:
        wk = wl.WORKLOADS[wl.HEADLINE]
        lay = wk.layers[0]
        A, G, _ = inputs(wk, 0)
        n = torch.zeros(wk.B, device=device)
        wsbuf = rnc.workspace(rnc.DPRC_OP_EXACT, A, wk.B, wk.T, lay.d, lay.p, wk.k)
        t = graph_ms(lambda: rnc.dprc_exact_norm(A, G, n, ws=wsbuf), device, 2, warmup=1)
        # bf16 q_proj shapes take the direct form A_i^T G_i on tensor cores:
        # 2 T d p flops per sample (the ghost form would need 2 T^2 (d + p))
        flops = wk.B * 2 * wk.T * lay.d * lay.p
        tf = flops / (t * 1e-3) / 1e12
        rows["exact_c2"] = {"ms": t, "algorithmic_flops": flops, "achieved_tflops": tf,
                            "bound": "tensor", "peak_tflops": tflops_peak,
                            "frac": tf / tflops_peak,
                            "ghost_form_flops": wk.B * 2 * wk.T * wk.T * (lay.d + lay.p),
                            "what": "dprc_exact_norm on the q_proj batch, direct form on "
                                    "tensor cores; flops 2 T d p per sample"}
        del A, G, n, wsbuf
        # short sequences: the q_proj widths at T = 1024 with B = 32 (the same
        # 268 MB of A and G), where the ghost form sum_{t,s} (A A^T)(G G^T) does
        # half the direct form's work; both forms timed, the automatic choice
        # named
        B, T = 32, 1024
        A, G, _ = wl.layer_inputs(wl.Workload(**{**wk.__dict__, "seed": wk.seed + seed_shift}),
                                  0, device=device, B=B, T=T)
        n = torch.zeros(B, device=device)
        wsbuf = rnc.workspace(rnc.DPRC_OP_EXACT, A, B, T, lay.d, lay.p, wk.k)
        auto = rnc.dprc_exact_norm_plan(rnc.DPRC_BF16, B, T, lay.d, lay.p)
        nt = (T + 127) // 128
        flops_ghost = B * T * (T + 1) * (lay.d + lay.p)  # Gram entries t <= s, 2 (d + p) each
        forms = {}
        for name, form in (("ghost_n128", rnc.DPRC_EXACT_GHOST_N128),
                           ("ghost_n256", rnc.DPRC_EXACT_GHOST_N256),
                           ("direct", rnc.DPRC_EXACT_DIRECT)):
            t = graph_ms(lambda: rnc.dprc_exact_norm(A, G, n, ws=wsbuf, form=form), device, 5,
                         warmup=2)
            fl = B * 2 * T * lay.d * lay.p if name == "direct" else flops_ghost
            mma = (B * 2 * T * lay.d * lay.p if name == "direct"
                   else B * nt * (nt + 1) // 2 * 2 * 128 * 128 * (lay.d + lay.p))
            forms[name] = {"ms": t, "algorithmic_flops": fl, "mma_flops": mma,
                           "achieved_tflops": fl / (t * 1e-3) / 1e12,
                           "frac": fl / (t * 1e-3) / 1e12 / tflops_peak}
        names = {rnc.DPRC_EXACT_DIRECT: "direct", rnc.DPRC_EXACT_GHOST_N128: "ghost_n128",
                 rnc.DPRC_EXACT_GHOST_N256: "ghost_n256"}
        best = min(forms, key=lambda k: forms[k]["ms"])
        rows["exact_q_proj_b32_t1024"] = {
            "forms": forms, "auto": names.get(auto, str(auto)), "fastest": best,
            "bound": "tensor", "peak_tflops": tflops_peak,
            "what": "dprc_exact_norm on q_proj widths at T = 1024, B = 32, each form; the "
                    "ghost form's algorithmic flops count the Gram entries t <= s, "
                    "T (T + 1) (d + p) per sample; mma_flops adds the diagonal blocks' "
                    "lower halves"}
        del A, G, n, wsbuf
    torch.cuda.empty_cache()
    return rows


def measure_step(device, B=4, T=4096):
    """One DP-SGD-RC step (randomized_norm_clipping_gb300.step) on a Llama-3.2-1B
    MLP-shaped bias-free block (2048 -> 8192 -> 2048, bf16, B x T tokens),
    against the same forward with an ordinary backward."""
    from randomized_norm_clipping_gb300.step import RandomizedClippingStep
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(2048, 8192, bias=False), torch.nn.SiLU(),
                                torch.nn.Linear(8192, 2048, bias=False)).to(device, torch.bfloat16)
    x = torch.randn(B, T, 2048, device=device).to(torch.bfloat16)

    def losses():
        return (model(x).float() ** 2).mean(dim=(1, 2))

    step = RandomizedClippingStep(model, C=1.0, sigma=1.0, k=32, seed=1)

    def dp():
        step(losses(), step=0)

    def plain():
        for m in model:
            if isinstance(m, torch.nn.Linear):
                m.weight.grad = None
        losses().sum().backward()

    def timed(fn, reps=10):
        for _ in range(5):
            fn()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / reps

    t_dp, t_plain = timed(dp), timed(plain)
    step.close()
    return {"ms": t_dp, "plain_backward_ms": t_plain, "overhead": t_dp / t_plain,
            "what": "forward + first backward to the layer outputs + dprc_norm_hutch per layer "
                    "+ clip + rescaled second backward + noise, B4 T4096 bf16 2048->8192->2048 "
                    "(eager, host launch time included), against forward + plain backward"}


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank, ws):
    """The float64 oracle on the host cores, same workload, one sample per step."""
    if rank != 0:
        return None
    import oracle
    wk = wl.WORKLOADS[wl.HEADLINE]
    lay = wk.layers[0]
    A, G, P = wl.layer_inputs(wk, 0, device="cpu", B=1)
    Af, Gf, Pf = wl.to_f64(A), wl.to_f64(G), wl.to_f64(P)

    def step():
        oracle.clip_factors(oracle.hutch_norm(Af, Gf, Pf), wk.C)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = args.steps * wk.T / el
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wk.name, "model": "Llama-3.2-1B q_proj shape",
                   "global_batch": 1, "seq_len": wk.T, "d": lay.d, "p": lay.p, "k": wk.k,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "one sample (T=4096) of the headline batch per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", default="all",
                    help="other configurations to time after the headline: all, none, or a "
                         "comma list of c3,c4,c5,noise,exact,step,pm1,lora")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, ws, local = dist_setup()
    if args.impl == "reference":
        out = run_reference(args, rank, ws)
    else:
        out = run_native(args, rank, ws, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
