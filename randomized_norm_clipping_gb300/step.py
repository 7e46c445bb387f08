"""One DP-SGD-RC step on a PyTorch model, with libdprc doing the work.

"Efficient DP-SGD for LLMs with Randomized Clipping" (papernotes.org,
"Method > Overall framework") lays the step out as:

  1. a forward pass that records, for every linear layer, its input
     activations A (B x T x d);
  2. a first backward pass that records the gradients G (B x T x p) with
     respect to each linear layer's output;
  3. per sample, per layer, the Hutchinson estimate of the squared norm of
     the weight gradient A_i^T G_i, summed over the layers;
  4. clip factors c_i = min(1, C / sqrt(n_i)) and a second backward pass of
     sum_i c_i L_i, which yields the clipped gradient sum sum_i c_i grad L_i;
  5. Gaussian noise sigma C N(0, I) added to that aggregated gradient.

`RandomizedClippingStep` does steps 2-5 around the caller's forward pass.
Steps 3-5 run in libdprc (Hutchinson: every layer and the clip factors of
the layer sum in one dprc_norm_hutch_layers_clip call; Hutch++: a
dprc_norm_hutchpp call per layer with accumulation, then dprc_clip_factors;
dprc_add_noise_at on each weight's gradient in place); PyTorch
provides the forward and backward passes and the memory.  The first backward
asks autograd only for the gradients with respect to the recorded layer
outputs, so no weight gradient is formed before the clip factors are known.

Scope: every trainable parameter must be the weight of an nn.Linear without
bias (per-sample norms of other parameter kinds need their own per-sample
gradients, which the method does not cover); each layer runs once per
forward pass on inputs (B, ..., d) (every position between the batch and the
feature axis counts as a token), and the per-sample losses must not couple
samples.  Projections are drawn fresh per (layer, step) from a seeded
generator (a reading of the pages, which do not say how often P is redrawn):
P ~ N(0, 1/k) for Hutchinson, S and P ~ N(0, 1) for Hutch++.  Dividing the
noisy sum by the batch size is left to the optimiser.
"""

from __future__ import annotations

import torch

from . import binding as rnc

_MIX = 0x9E3779B97F4A7C15


def _seed(*parts):
    """A 63-bit seed from integers (splitmix-style mixing)."""
    h = 0
    for x in parts:
        h = (h ^ (int(x) & 0xFFFFFFFFFFFFFFFF)) * _MIX & 0xFFFFFFFFFFFFFFFF
        h ^= h >> 31
    return h & 0x7FFFFFFFFFFFFFFF


class RandomizedClippingStep:
    """DP-SGD-RC gradient step for the nn.Linear weights of `model`.

    Args:
      model: the module; all its trainable parameters must be bias-free
        nn.Linear weights.
      C: clipping threshold.
      sigma: noise multiplier (0 disables the noise).
      k: projection width (Hutchinson) or r (Hutch++, k = 16).
      method: "hutch" or "hutchpp".
      seed: base seed of the projections and the noise.
    """

    def __init__(self, model, C, sigma, k=32, method="hutch", seed=0):
        if method not in ("hutch", "hutchpp"):
            raise ValueError("method must be 'hutch' or 'hutchpp'")
        self.model = model
        self.C = float(C)
        self.sigma = float(sigma)
        self.k = int(k)
        self.method = method
        self.seed = int(seed)
        self.layers = [m for m in model.modules()
                       if isinstance(m, torch.nn.Linear) and m.weight.requires_grad]
        covered = {id(m.weight) for m in self.layers}
        for name, prm in model.named_parameters():
            if prm.requires_grad and id(prm) not in covered:
                raise ValueError(f"trainable parameter {name!r} is not a bias-free "
                                 "nn.Linear weight; per-sample norms cover only those")
        for m in self.layers:
            if m.bias is not None and m.bias.requires_grad:
                raise ValueError("nn.Linear layers with a trainable bias are not supported")
        self._acts = {}
        self._outs = {}
        self._handles = [m.register_forward_hook(self._record) for m in self.layers]
        self._ws = {}

    def close(self):
        """Removes the hooks."""
        for h in self._handles:
            h.remove()
        self._handles = []

    def _record(self, module, inputs, output):
        if torch.is_grad_enabled():
            self._acts[module] = inputs[0]
            self._outs[module] = output

    def projections(self, step):
        """The projection(s) of every layer for `step`: P [p][k] (Hutchinson)
        or (S, P) [p][k] (Hutch++), in the layer's dtype, on its device."""
        out = []
        for j, m in enumerate(self.layers):
            p = m.out_features
            dev, dt = m.weight.device, m.weight.dtype
            g = torch.Generator(device=dev)
            g.manual_seed(_seed(self.seed, 1, j, step))
            if self.method == "hutch":
                P = (torch.randn(p, self.k, generator=g, device=dev) / self.k ** 0.5).to(dt)
                out.append(P)
            else:
                S = torch.randn(p, self.k, generator=g, device=dev).to(dt)
                P = torch.randn(p, self.k, generator=g, device=dev).to(dt)
                out.append((S, P))
        return out

    def _layers_workspace(self, As, Gs, proj):
        B, T = As[0].shape[0], As[0].shape[1]
        k = max(P.shape[1] for P in proj)
        need = rnc.dprc_workspace_bytes(rnc.DPRC_OP_HUTCH_LAYERS, rnc._dtype_code(As[0]), B, T,
                                        max(A.shape[2] for A in As), max(G.shape[2] for G in Gs),
                                        k)
        key = (As[0].device, rnc.DPRC_OP_HUTCH_LAYERS)
        ws = self._ws.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(need, dtype=torch.uint8, device=As[0].device)  # zeroed once
            self._ws[key] = ws
        return ws

    def _workspace(self, op, A, B, T, d, p, k):
        need = rnc.dprc_workspace_bytes(op, rnc._dtype_code(A), B, T, d, p, k)
        key = (A.device, op)
        ws = self._ws.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(need, dtype=torch.uint8, device=A.device)  # zeroed once
            self._ws[key] = ws
        return ws

    def __call__(self, per_sample_losses, step, projections=None):
        """Runs steps 2-5 for losses L_i = per_sample_losses [B] of the forward
        pass just made.  Leaves sum_i c_i grad L_i (+ noise) in the weights'
        .grad and returns {"n": n, "c": c} (fp32 [B] on the device)."""
        losses = per_sample_losses
        if losses.dim() != 1:
            raise ValueError("per_sample_losses must have shape [B]")
        B = losses.shape[0]
        missing = [m for m in self.layers if m not in self._outs]
        if missing:
            raise RuntimeError("no forward pass recorded for some linear layers")
        outs = [self._outs[m] for m in self.layers]
        # step 2: gradients with respect to the layer outputs only
        grads = torch.autograd.grad(losses.sum(), outs, retain_graph=True)
        proj = self.projections(step) if projections is None else projections
        # step 3: layerwise sum of the per-sample estimates
        n = torch.zeros(B, dtype=torch.float32, device=losses.device)
        c = torch.empty_like(n)
        As, Gs = [], []
        for m, G in zip(self.layers, grads):
            A = self._acts[m]
            # (B, ..., d): every position between batch and features is a token
            As.append(A.detach().reshape(B, -1, A.shape[-1]).contiguous())
            Gs.append(G.detach().reshape(B, -1, G.shape[-1]).to(A.dtype).contiguous())
        one_call = (self.method == "hutch" and len({A.shape[1] for A in As}) == 1
                    and len({P.shape[1] for P in proj}) == 1 and len({A.dtype for A in As}) == 1)
        if one_call:
            # every layer in one call (persistent launches of up to 56 layers),
            # the clip factors of the layer sum in the same call (step 4)
            ws = self._layers_workspace(As, Gs, proj)
            rnc.dprc_norm_hutch_layers(As, Gs, proj, n, ws=ws, C=self.C, c=c)
        else:
            last = len(self.layers) - 1
            for j, (A, G) in enumerate(zip(As, Gs)):
                Bt, T, d = A.shape
                p = G.shape[-1]
                if self.method == "hutch":
                    ws = self._workspace(rnc.DPRC_OP_HUTCH, A, Bt, T, d, p, proj[j].shape[1])
                    if j == last:  # step 4's clip factors come with the last layer's norms
                        rnc.dprc_norm_hutch_clip(A, G, proj[j], n, self.C, c, accumulate=j > 0,
                                                 ws=ws)
                    else:
                        rnc.dprc_norm_hutch(A, G, proj[j], n, accumulate=j > 0, ws=ws)
                else:
                    S, P = proj[j]
                    ws = self._workspace(rnc.DPRC_OP_HUTCHPP, A, Bt, T, d, p, S.shape[1])
                    rnc.dprc_norm_hutchpp(A, G, S, P, n, accumulate=j > 0, ws=ws)
        # step 4: clip factors (Hutch++: here) and the rescaled second backward
        if self.method != "hutch":
            rnc.dprc_clip_factors(n, self.C, c)
        for m in self.layers:
            m.weight.grad = None
        (c.to(losses.dtype) * losses).sum().backward()
        # step 5: noise on the aggregated gradient, in place: the weights'
        # gradients laid end to end in layer order are that gradient, and each
        # gets the stretch of the one noise stream its position there selects
        if self.sigma > 0.0:
            off = 0
            for m in self.layers:
                g = m.weight.grad
                if not g.is_contiguous():
                    raise RuntimeError("weight gradients must be contiguous")
                rnc.dprc_add_noise_at(g, off, self.sigma, self.C, _seed(self.seed, 2), step)
                off += g.numel()
        self._acts.clear()
        self._outs.clear()
        return {"n": n, "c": c}
