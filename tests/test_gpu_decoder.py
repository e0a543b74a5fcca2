"""The GPT-2-small-shaped sparse decoder (12 blocks, d 768, 12 heads, MLP
3072, context 256, vocabulary 50257, tied LM head; all 48 attention / MLP
projections SNACK layers at 99 %) trained with SGD at lr 1e-2 for 301 steps
on one seeded batch of 256 random tokens, with a 30 % magnitude-prune /
uniform-regrow of every sparse layer every 100 steps (the paper's GPT-2
dynamic-sparse setting, §5 Tables 4-5, Appendix G, without WikiText).

Checked against the CPU oracle, layer by layer, on the first step and on the
first step after each regrow: every sparse layer's output Y (minus its dense
bias), its input gradient dX and its weight gradient at the stored entries,
for the inputs and output gradients the layer saw inside the model
(1e-5 * sum|terms| per element); and each regrow's topology, values and
trial count bit for bit.  The loss must stay finite and fall (the batch is
fixed, so the model can memorise it)."""

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_close

pytestmark = pytest.mark.gpu


class _Tap:
    """Forward / backward hooks recording a sparse layer's X, Y, dY and dX."""

    def __init__(self, lin):
        self.lin = lin
        self.on = False
        lin.register_forward_hook(self._fwd)
        lin.register_full_backward_hook(self._bwd)

    def _fwd(self, mod, inp, out):
        if self.on:
            self.X = inp[0].detach().reshape(-1, mod.in_features).clone()
            self.Y = out.detach().reshape(-1, mod.out_features).clone()

    def _bwd(self, mod, grad_in, grad_out):
        if self.on:
            self.dY = grad_out[0].detach().reshape(-1, mod.out_features).clone()
            self.dX = grad_in[0].detach().reshape(-1, mod.in_features).clone()

    def check(self, tag):
        lin = self.lin
        out, inp = lin.out_features, lin.in_features
        row, col, val = lin.export()
        X, dY = self.X.cpu().numpy(), self.dY.cpu().numpy()
        Yo, Sy = oracle.forward(out, inp, row, col, val, X)
        # the module adds its dense bias in fp32 after the sparse product:
        # one more rounding, at most an ulp of the result, on top of 1e-5 * S
        want = Yo.astype(np.float64) + lin.bias.detach().cpu().numpy().astype(np.float64)
        got = self.Y.cpu().numpy().astype(np.float64)
        bad = np.abs(got - want) > 1e-5 * Sy + np.abs(want) * 2.0 ** -23
        assert not bad.any(), (tag, int(bad.sum()))
        dXo, Sx = oracle.backward_input(out, inp, row, col, val, dY)
        assert_close(f"{tag} dX", self.dX, dXo, Sx)
        dWo, Sw = oracle.backward_weight(out, inp, row, col, X, dY)
        assert_close(f"{tag} dW", lin.weight_values.grad, dWo, Sw)


def test_sparse_decoder_trains_with_layer_parity_and_regrow():
    from coo_spmm_sparse_gb300.decoder import DecoderConfig, SparseDecoder
    cfg = DecoderConfig(seed=0)
    model = SparseDecoder(cfg)
    lins = model.sparse_layers()
    assert len(lins) == 48
    assert [l.nnz for l in lins[:4]] == [17695, 5898, 23593, 23593]
    taps = [_Tap(l) for l in lins]
    opt = torch.optim.SGD(model.parameters(), lr=1e-2)
    g = torch.Generator(device="cpu").manual_seed(1)
    idx = torch.randint(0, cfg.vocab, (1, cfg.ctx), generator=g).cuda()
    losses = []
    for step in range(1, 302):
        check = step in (1, 101, 201, 301)
        for t in taps:
            t.on = check
        opt.zero_grad(set_to_none=True)
        loss = model.loss(idx)
        loss.backward()
        if check:
            torch.cuda.synchronize()
            for i, t in enumerate(taps):
                t.check(f"step {step} layer {i}")
        opt.step()
        losses.append(loss.item())
        if step % 100 == 0:  # Appendix G topology step on every layer
            before = [l.export() for l in lins]
            res = model.prune_regrow(0.30, step)
            for i, (l, (r0, c0, v0), (p, tr)) in enumerate(zip(lins, before, res)):
                o = oracle.prune_regrow(l.out_features, l.in_features, r0, c0, v0, 0.30,
                                        7919 * step + i)
                assert (p, tr) == (o["pruned"], o["trials"]), (step, i)
                r1, c1, v1 = l.export()
                assert np.array_equal(r1, o["row"]) and np.array_equal(c1, o["col"]), (step, i)
                assert np.array_equal(v1.view(np.uint32), o["val"].view(np.uint32)), (step, i)
    assert np.all(np.isfinite(losses))
    assert losses[-1] < losses[0] - 0.5, (losses[0], losses[-1])
