"""The DP-SGD-RC step on a small model (randomized_norm_clipping_gb300.step).

With P = I_p the Hutchinson estimate equals the exact per-sample norm, so the
step must reproduce textbook per-sample clipping computed by a loop over
samples; with random projections it must match the float64 oracle on the
same activations, gradients and projections; the noise must be sigma*C*z
with z the library's Philox normals.
"""

import numpy as np
import pytest
import torch

import oracle
import randomized_norm_clipping_gb300 as rnc
from randomized_norm_clipping_gb300.step import RandomizedClippingStep
from randomized_norm_clipping_gb300.workloads import to_f64

DEV = "cuda:0"


def _model(dtype, widths=(64, 64, 64), seed=0):
    torch.manual_seed(seed)
    layers = []
    for a, b in zip(widths[:-1], widths[1:]):
        layers += [torch.nn.Linear(a, b, bias=False), torch.nn.Tanh()]
    return torch.nn.Sequential(*layers[:-1]).to(DEV, dtype)


def _losses(model, x):
    out = model(x)
    return (out.float() ** 2).mean(dim=tuple(range(1, out.dim())))


def _per_sample_reference(model, x, C):
    """Exact per-sample squared norms and sum_i c_i grad L_i by a loop."""
    ws = [m.weight for m in model if isinstance(m, torch.nn.Linear)]
    B = x.shape[0]
    norms, grads = [], []
    for i in range(B):
        gi = torch.autograd.grad(_losses(model, x[i:i + 1]).sum(), ws)
        norms.append(sum(float((g.double() ** 2).sum()) for g in gi))
        grads.append([g.double() for g in gi])
    n = np.array(norms)
    c = np.minimum(1.0, C / np.sqrt(n))
    agg = [sum(c[i] * grads[i][j] for i in range(B)) for j in range(len(ws))]
    return n, c, agg


def _capture(model, x):
    """(A_l, G_l) of every linear layer for the per-sample loss sum."""
    acts, outs = [], []

    def hook(module, inputs, output):  # returns None: the output is kept
        acts.append(inputs[0])
        outs.append(output)

    hs = [m.register_forward_hook(hook) for m in model if isinstance(m, torch.nn.Linear)]
    loss = _losses(model, x).sum()
    for h in hs:
        h.remove()
    gs = torch.autograd.grad(loss, outs)
    return [(a.detach(), g.detach().to(a.dtype)) for a, g in zip(acts, gs)]


@pytest.mark.gpu
def test_identity_projection_reproduces_per_sample_clipping():
    model = _model(torch.float32)
    x = torch.randn(4, 16, 64, device=DEV, generator=torch.Generator(DEV).manual_seed(1))
    n_ref, _, _ = _per_sample_reference(model, x, 1.0)
    C = float(np.median(np.sqrt(n_ref)))  # half the samples clip
    n_ref, c_ref, agg = _per_sample_reference(model, x, C)
    step = RandomizedClippingStep(model, C=C, sigma=0.0, k=64)
    eye = [torch.eye(64, device=DEV)] * 2
    out = step(_losses(model, x), step=0, projections=eye)
    assert np.allclose(out["n"].cpu().numpy(), n_ref, rtol=1e-4)
    assert np.allclose(out["c"].cpu().numpy(), c_ref, rtol=1e-4)
    ws = [m.weight for m in model if isinstance(m, torch.nn.Linear)]
    for w, ref in zip(ws, agg):
        assert torch.allclose(w.grad.double(), ref, rtol=1e-4, atol=1e-7 * float(ref.abs().max()))
    step.close()


class _Block(torch.nn.Module):
    """A pre-norm transformer block: causal self-attention (q, k, v, o) and a
    SiLU MLP (up, down), every projection a bias-free nn.Linear; the norms are
    frozen (their per-sample norms are outside the method)."""

    def __init__(self, dm=64, heads=4, hidden=128):
        super().__init__()
        self.heads = heads
        self.n1 = torch.nn.LayerNorm(dm, elementwise_affine=False)
        self.q = torch.nn.Linear(dm, dm, bias=False)
        self.k = torch.nn.Linear(dm, dm, bias=False)
        self.v = torch.nn.Linear(dm, dm, bias=False)
        self.o = torch.nn.Linear(dm, dm, bias=False)
        self.n2 = torch.nn.LayerNorm(dm, elementwise_affine=False)
        self.up = torch.nn.Linear(dm, hidden, bias=False)
        self.down = torch.nn.Linear(hidden, dm, bias=False)

    def forward(self, x):
        B, T, dm = x.shape
        h = self.n1(x)
        split = lambda t: t.view(B, T, self.heads, dm // self.heads).transpose(1, 2)  # noqa: E731
        att = torch.nn.functional.scaled_dot_product_attention(
            split(self.q(h)), split(self.k(h)), split(self.v(h)), is_causal=True)
        x = x + self.o(att.transpose(1, 2).reshape(B, T, dm))
        return x + self.down(torch.nn.functional.silu(self.up(self.n2(x))))


@pytest.mark.gpu
def test_transformer_block_step_reproduces_per_sample_clipping():
    # with P = I for every layer the estimate is exact, so the step must equal
    # per-sample clipping of the block's six projections computed by a loop
    torch.manual_seed(3)
    block = _Block().to(DEV)
    x = torch.randn(4, 24, 64, device=DEV, generator=torch.Generator(DEV).manual_seed(4))
    ws = [m.weight for m in (block.q, block.k, block.v, block.o, block.up, block.down)]

    def losses(inp):
        return (block(inp) ** 2).mean(dim=(1, 2))

    norms, grads = [], []
    for i in range(x.shape[0]):
        gi = torch.autograd.grad(losses(x[i:i + 1]).sum(), ws)
        norms.append(sum(float((g.double() ** 2).sum()) for g in gi))
        grads.append([g.double() for g in gi])
    n_ref = np.array(norms)
    C = float(np.median(np.sqrt(n_ref)))
    c_ref = np.minimum(1.0, C / np.sqrt(n_ref))
    step = RandomizedClippingStep(block, C=C, sigma=0.0, k=64)
    assert [m.weight for m in step.layers] == ws  # module order
    eye = [torch.eye(m.out_features, device=DEV) for m in step.layers]
    out = step(losses(x), step=0, projections=eye)
    assert np.allclose(out["n"].cpu().numpy(), n_ref, rtol=1e-4)
    assert np.allclose(out["c"].cpu().numpy(), c_ref, rtol=1e-4)
    for j, w in enumerate(ws):
        ref = sum(c_ref[i] * grads[i][j] for i in range(x.shape[0]))
        assert torch.allclose(w.grad.double(), ref, rtol=1e-4, atol=1e-7 * float(ref.abs().max()))
    step.close()


@pytest.mark.gpu
def test_bf16_transformer_block_step_matches_oracle():
    # bf16 block: q, k, v, o, down (p = 64) take the narrow kernel, up (64 -> 128)
    # the fused sketch kernel; the layer sum and clip factors against the oracle
    # on the same activations, gradients and projections
    torch.manual_seed(5)
    block = _Block().to(DEV, torch.bfloat16)
    x = torch.randn(3, 100, 64, device=DEV,
                    generator=torch.Generator(DEV).manual_seed(6)).to(torch.bfloat16)

    def losses(inp):
        return (block(inp).float() ** 2).mean(dim=(1, 2))

    step = RandomizedClippingStep(block, C=1.0, sigma=0.0, k=32, seed=2)
    out = step(losses(x), step=11)
    proj = step.projections(11)
    acts, outs = [], []
    hooks = [m.register_forward_hook(lambda mod, inp, o: (acts.append(inp[0]), outs.append(o))
                                     and None) for m in step.layers]
    loss = losses(x).sum()
    for h in hooks:
        h.remove()
    gs = torch.autograd.grad(loss, outs)
    ref = 0.0
    for a_, g_, pr in zip(acts, gs, proj):
        A = a_.detach().reshape(3, -1, a_.shape[-1])
        G = g_.detach().reshape(3, -1, g_.shape[-1]).to(A.dtype)
        ref = ref + oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(pr))
    got = out["n"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref) / ref) < 1e-3
    assert np.allclose(out["c"].cpu().numpy(), oracle.clip_factors(ref, 1.0), rtol=1e-3)
    step.close()


@pytest.mark.gpu
@pytest.mark.parametrize("method,k", [("hutch", 32), ("hutchpp", 16)])
def test_bf16_step_matches_oracle(method, k):
    model = _model(torch.bfloat16, widths=(256, 512, 128))
    x = torch.randn(3, 200, 256, device=DEV,
                    generator=torch.Generator(DEV).manual_seed(2)).to(torch.bfloat16)
    step = RandomizedClippingStep(model, C=1.0, sigma=0.0, k=k, method=method, seed=5)
    out = step(_losses(model, x), step=7)
    proj = step.projections(7)
    ref = 0.0
    for (A, G), pr in zip(_capture(model, x), proj):
        if method == "hutch":
            ref = ref + oracle.hutch_norm(to_f64(A), to_f64(G), to_f64(pr))
        else:
            ref = ref + oracle.hutchpp_norm(to_f64(A), to_f64(G), to_f64(pr[0]), to_f64(pr[1]))
    got = out["n"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref) / ref) < 1e-3
    assert np.allclose(out["c"].cpu().numpy(), oracle.clip_factors(ref, 1.0), rtol=1e-3)
    step.close()


@pytest.mark.gpu
def test_noise_is_sigma_c_times_the_philox_normals():
    x = torch.randn(4, 16, 64, device=DEV, generator=torch.Generator(DEV).manual_seed(3))
    grads = []
    for sigma in (0.0, 0.7):
        model = _model(torch.float32, seed=11)
        step = RandomizedClippingStep(model, C=2.0, sigma=sigma, k=64, seed=9)
        step(_losses(model, x), step=4)
        grads.append(torch.cat([m.weight.grad.reshape(-1) for m in model
                                if isinstance(m, torch.nn.Linear)]))
        step.close()
    z = torch.zeros_like(grads[0])
    rnc.dprc_add_noise(z, 1.0, 1.0, _noise_seed(9), 4)
    diff = grads[1] - grads[0]
    scale = 0.7 * 2.0
    tol = 1e-6 * float(grads[0].abs().max()) + 1e-6
    assert torch.allclose(diff, scale * z, atol=tol, rtol=1e-5)


@pytest.mark.gpu
def test_noise_in_place_on_bf16_weight_gradients():
    # the step adds the noise to each weight's bf16 gradient in place (its
    # stretch of the one stream); the result is the fp32 sum rounded once
    x = torch.randn(4, 16, 64, device=DEV,
                    generator=torch.Generator(DEV).manual_seed(5)).to(torch.bfloat16)
    grads = []
    for sigma in (0.0, 0.7):
        model = _model(torch.bfloat16, widths=(64, 96, 40), seed=12)
        step = RandomizedClippingStep(model, C=2.0, sigma=sigma, k=32, seed=9)
        step(_losses(model, x), step=6)
        grads.append(torch.cat([m.weight.grad.reshape(-1) for m in model
                                if isinstance(m, torch.nn.Linear)]).float())
        step.close()
    z = torch.zeros_like(grads[0])
    rnc.dprc_add_noise(z, 1.0, 1.0, _noise_seed(9), 6)
    want = grads[0] + 1.4 * z
    # one bf16 rounding of the sum (2^-8 relative), plus the normals' bound
    tol = (want.abs() * 2.0 ** -8 + 1.4 * 1e-5).to(want.dtype)
    assert torch.all((grads[1] - want).abs() <= tol)


def _noise_seed(seed):
    from randomized_norm_clipping_gb300.step import _seed
    return _seed(seed, 2)


def test_step_rejects_parameters_it_cannot_clip():
    m = torch.nn.Sequential(torch.nn.Linear(8, 8, bias=True))
    with pytest.raises(ValueError):
        RandomizedClippingStep(m, C=1.0, sigma=1.0)
    m = torch.nn.Sequential(torch.nn.Linear(8, 8, bias=False), torch.nn.LayerNorm(8))
    with pytest.raises(ValueError):
        RandomizedClippingStep(m, C=1.0, sigma=1.0)
    m = torch.nn.Sequential(torch.nn.Linear(8, 8, bias=False), torch.nn.LayerNorm(8))
    for prm in m[1].parameters():
        prm.requires_grad_(False)
    RandomizedClippingStep(m, C=1.0, sigma=1.0).close()  # frozen norms are fine
