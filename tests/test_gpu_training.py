"""The GPT-2-shaped decoder workload trained through the library: every step
runs the forward, the input gradient and an Adam step of each sparse
layer of one block; every 100 steps each layer is magnitude-pruned by 30 %
and regrown uniformly (Appendix G's schedule with the workload's fraction).

Checks: each prune/regrow gives, bit for bit, the oracle's topology and
values from the values the GPU trained; nnz never changes; optimizer state
survives for kept entries and is zero for regrown ones; after training the
products still match the oracle on the final topology."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import canonical, check_products, check_topology, dev, sn

pytestmark = pytest.mark.gpu


def test_decoder_block_training_with_prune_regrow():
    m = sn()
    wl = workloads.workload("gpt2_decoder")
    frac = wl.extra["prune_frac"]
    layers = wl.layers[:4]
    hs = []
    for L in layers:
        row, col, val = L.coo()
        hs.append(m.snack_create(L.out, L.inp, row, col, val))
    gen = torch.Generator(device=dev()).manual_seed(7)
    tokens = 256
    for step in range(1, 201):
        for L, h in zip(layers, hs):
            X = torch.randn(tokens, L.inp, device=dev(), generator=gen)
            dY = torch.randn(tokens, L.out, device=dev(), generator=gen) * 1e-2
            m.snack_forward(h, X)
            m.snack_backward_input(h, dY)
            m.snack_adam_step(h, X, dY, lr=1e-3, step=step)
        if step % 100:
            continue
        for L, h in zip(layers, hs):
            torch.cuda.synchronize()
            r0, c0, v0 = m.snack_export(h)
            m0 = m.snack_optimizer_state(h, 0).cpu().numpy().copy()
            before = {(int(r), int(c)): a for r, c, a in zip(r0, c0, m0)}
            seed = 1000 * step + L.seed
            pruned, trials = m.snack_prune_regrow(h, frac, seed)
            o = oracle.prune_regrow(L.out, L.inp, r0, c0, v0, frac, seed)
            assert (pruned, trials) == (o["pruned"], o["trials"])
            check_topology(h, canonical(L.out, L.inp, o["row"], o["col"], o["val"]))
            r1, c1, _ = m.snack_export(h)
            assert r1.size == r0.size
            m1 = m.snack_optimizer_state(h, 0).cpu().numpy()
            kept = 0
            for r, c, a in zip(r1, c1, m1):
                key = (int(r), int(c))
                if key in before and a == before[key]:
                    kept += 1
                else:
                    assert a == 0.0, key
            assert kept >= r0.size - pruned
    g = np.random.default_rng(8)
    for L, h in zip(layers, hs):
        r, c, v = m.snack_export(h)
        ref = canonical(L.out, L.inp, r, c, v)
        X = g.standard_normal((16, L.inp)).astype(np.float32)
        dY = g.standard_normal((16, L.out)).astype(np.float32)
        check_products(h, L.out, L.inp, ref, X, dY)
        assert m.snack_device_error(h) == 0


def test_decoder_block_sgd_training_with_prune_regrow():
    """The decoder workload's own recipe on its second block: plain SGD (no
    momentum, §4.2) at the workload's learning rate, 300 steps of 256 tokens,
    30 % magnitude prune / uniform regrow every 100 steps (three topology
    changes, each bit-exact against the oracle from the trained values)."""
    m = sn()
    wl = workloads.workload("gpt2_decoder")
    frac, lr, every = wl.extra["prune_frac"], wl.extra["lr"], wl.extra["prune_every"]
    layers = wl.layers[4:8]
    hs = []
    for L in layers:
        row, col, val = L.coo()
        hs.append(m.snack_create(L.out, L.inp, row, col, val))
    gen = torch.Generator(device=dev()).manual_seed(9)
    tokens = wl.extra["ctx"]
    events = 0
    for step in range(1, 301):
        for L, h in zip(layers, hs):
            X = torch.randn(tokens, L.inp, device=dev(), generator=gen)
            dY = torch.randn(tokens, L.out, device=dev(), generator=gen) * 1e-2
            m.snack_forward(h, X)
            m.snack_backward_input(h, dY)
            m.snack_sgd_step(h, X, dY, lr=lr)
        if step % every:
            continue
        events += 1
        for L, h in zip(layers, hs):
            torch.cuda.synchronize()
            r0, c0, v0 = m.snack_export(h)
            seed = 1000 * step + L.seed
            pruned, trials = m.snack_prune_regrow(h, frac, seed)
            o = oracle.prune_regrow(L.out, L.inp, r0, c0, v0, frac, seed)
            assert (pruned, trials) == (o["pruned"], o["trials"])
            check_topology(h, canonical(L.out, L.inp, o["row"], o["col"], o["val"]))
            assert h.nnz == L.nnz
    assert events == 3
    g = np.random.default_rng(10)
    for L, h in zip(layers, hs):
        r, c, v = m.snack_export(h)
        ref = canonical(L.out, L.inp, r, c, v)
        X = g.standard_normal((8, L.inp)).astype(np.float32)
        dY = g.standard_normal((8, L.out)).astype(np.float32)
        check_products(h, L.out, L.inp, ref, X, dY)
        assert m.snack_device_error(h) == 0
