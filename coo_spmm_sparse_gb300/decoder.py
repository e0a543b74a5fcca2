"""GPT-2-small-shaped decoder whose attention and MLP projections are SNACK
sparse layers: the training harness of the paper's GPT-2 dynamic-sparse runs
("Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
GPU", §5 Tables 4-5; Appendix G "Sparsity schedule and DST"), on random
tokens instead of WikiText-103.

Every block's four projections (c_attn 768->2304, attention c_proj
768->768, c_fc 768->3072, MLP c_proj 3072->768) are ``SnackLinear`` layers
at the given sparsity: their forward and backward run in the library's
kernels.  Token and position embeddings, layer norms, the attention
arithmetic (softmax(QK^T / sqrt(d)) V, causal), GELU and the tied LM head
stay dense PyTorch: the paper makes only the Linear projections sparse.

The training step is plain SGD on every parameter (the sparse values are
updated in place through their Parameter views) and, every
``prune_every`` steps, a magnitude-prune / uniform-regrow of each sparse
layer (Appendix G) with a per-layer seed derived from the step.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch
import torch.nn.functional as F

from . import SnackLinear


def nnz_for(out: int, inp: int, sparsity_pct: float) -> int:
    """Stored entries of an out x in layer: (1 - sparsity) * out * in,
    rounded half up (256x256 at 90 % -> 6554)."""
    x = (100.0 - sparsity_pct) * out * inp
    return int(math.floor(x / 100.0 + 0.5))


@dataclass
class DecoderConfig:
    vocab: int = 50257
    ctx: int = 256
    d: int = 768
    heads: int = 12
    layers: int = 12
    mlp: int = 3072
    sparsity: float = 99.0
    std: float = 0.02
    seed: int = 0


class Block(torch.nn.Module):
    def __init__(self, cfg: DecoderConfig, index: int):
        super().__init__()
        d, m = cfg.d, cfg.mlp
        self.heads = cfg.heads
        self.ln_1 = torch.nn.LayerNorm(d)
        self.ln_2 = torch.nn.LayerNorm(d)

        def sparse(j, inp, out):
            return SnackLinear(inp, out, nnz_for(out, inp, cfg.sparsity),
                               seed=cfg.seed + 1000 * index + j, std=cfg.std)

        self.c_attn = sparse(0, d, 3 * d)
        self.attn_c_proj = sparse(1, d, d)
        self.c_fc = sparse(2, d, m)
        self.mlp_c_proj = sparse(3, m, d)

    def sparse_layers(self):
        return [self.c_attn, self.attn_c_proj, self.c_fc, self.mlp_c_proj]

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        B, T, d = x.shape
        h = self.heads
        q, k, v = self.c_attn(self.ln_1(x)).split(d, dim=2)
        q, k, v = (t.view(B, T, h, d // h).transpose(1, 2) for t in (q, k, v))
        a = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        x = x + self.attn_c_proj(a.transpose(1, 2).reshape(B, T, d))
        x = x + self.mlp_c_proj(F.gelu(self.c_fc(self.ln_2(x)), approximate="tanh"))
        return x


class SparseDecoder(torch.nn.Module):
    """GPT-2-small-shaped decoder with SNACK sparse projections."""

    def __init__(self, cfg: DecoderConfig = DecoderConfig(), device=None):
        super().__init__()
        self.cfg = cfg
        dev = device or torch.device("cuda", torch.cuda.current_device())
        g = torch.Generator(device="cpu").manual_seed(cfg.seed)
        self.wte = torch.nn.Embedding(cfg.vocab, cfg.d, device=dev)
        self.wpe = torch.nn.Embedding(cfg.ctx, cfg.d, device=dev)
        with torch.no_grad():
            self.wte.weight.copy_(torch.randn(cfg.vocab, cfg.d, generator=g) * cfg.std)
            self.wpe.weight.copy_(torch.randn(cfg.ctx, cfg.d, generator=g) * 0.01)
        self.blocks = torch.nn.ModuleList(Block(cfg, i) for i in range(cfg.layers))
        self.ln_f = torch.nn.LayerNorm(cfg.d, device=dev)
        self.to(dev)

    def sparse_layers(self):
        return [lin for b in self.blocks for lin in b.sparse_layers()]

    def forward(self, idx: torch.Tensor) -> torch.Tensor:
        B, T = idx.shape
        pos = torch.arange(T, device=idx.device)
        x = self.wte(idx) + self.wpe(pos)
        for b in self.blocks:
            x = b(x)
        return F.linear(self.ln_f(x), self.wte.weight)  # tied LM head

    def loss(self, idx: torch.Tensor) -> torch.Tensor:
        """Next-token cross-entropy of a [B][T] token batch."""
        logits = self.forward(idx)
        return F.cross_entropy(logits[:, :-1].reshape(-1, logits.shape[-1]),
                               idx[:, 1:].reshape(-1))

    @torch.no_grad()
    def prune_regrow(self, frac: float, step: int):
        """Magnitude-prune / uniform-regrow every sparse layer (Appendix G);
        layer i uses seed 7919 * step + i.  Returns [(pruned, trials)]."""
        return [lin.prune_regrow(frac, 7919 * step + i) for i, lin in
                enumerate(self.sparse_layers())]


class Trainer:
    """Plain SGD (no momentum) on every parameter, with prune/regrow of the
    sparse layers every ``prune_every`` steps."""

    def __init__(self, model: SparseDecoder, lr: float = 1e-2, prune_frac: float = 0.30,
                 prune_every: int = 100):
        self.model = model
        self.opt = torch.optim.SGD(model.parameters(), lr=lr, momentum=0.0)
        self.prune_frac, self.prune_every = prune_frac, prune_every
        self.step_no = 0

    def step(self, idx: torch.Tensor) -> torch.Tensor:
        """One training step on a token batch; returns the loss (on device)."""
        self.opt.zero_grad(set_to_none=True)
        loss = self.model.loss(idx)
        loss.backward()
        self.opt.step()
        self.step_no += 1
        if self.prune_every and self.step_no % self.prune_every == 0:
            self.model.prune_regrow(self.prune_frac, self.step_no)
        return loss.detach()
