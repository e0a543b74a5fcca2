"""SnackLinear and its autograd function against the CPU oracle.

The module's forward runs snack_forward, autograd's backward runs
snack_backward; the gradients autograd hands back must be the oracle's: the
input gradient dX = dY W (§3.4, W^T by swapped index arrays) and the weight
gradient at the stored entries, in the canonical order of ``weight_values``
(§3.4, Appendix F).  Then a torch.optim.SGD step writes the values in place
(the next forward must see them, and dX must not read a stale
column-ordered copy), and a prune/regrow (Appendix G) reorders them under the
live Parameter.  Tolerance: 1e-5 times the oracle's sum of |terms| per
element."""

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_close

pytestmark = pytest.mark.gpu


def _check_step(lin, X, G, tag):
    """One forward + backward through the module, checked against the oracle
    on the layer's exported (canonical) entries."""
    out, inp = lin.out_features, lin.in_features
    row, col, val = lin.export()
    assert np.array_equal(val, lin.weight_values.detach().cpu().numpy())
    Xt = torch.from_numpy(X).cuda().requires_grad_(True)
    lin.zero_grad(set_to_none=True)
    y = lin(Xt)
    y.backward(torch.from_numpy(G).cuda())
    torch.cuda.synchronize()
    Yo, Sy = oracle.forward(out, inp, row, col, val, X)
    # the module adds its dense bias in fp32 after the sparse product: one
    # more rounding, at most an ulp of the result, on top of 1e-5 * S
    want = Yo.astype(np.float64) + lin.bias.detach().cpu().numpy().astype(np.float64)
    got = y.detach().cpu().numpy().astype(np.float64)
    bad = np.abs(got - want) > 1e-5 * Sy + np.abs(want) * 2.0 ** -23
    assert not bad.any(), (tag, int(bad.sum()))
    dXo, Sx = oracle.backward_input(out, inp, row, col, val, G)
    assert_close(f"{tag} dX", Xt.grad, dXo, Sx)
    dWo, Sw = oracle.backward_weight(out, inp, row, col, X, G)
    assert lin.weight_values.grad.shape == (lin.nnz,)
    assert_close(f"{tag} dW (canonical order)", lin.weight_values.grad, dWo, Sw)
    np.testing.assert_allclose(lin.bias.grad.cpu().numpy(), G.sum(0), rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("out,inp,density,B", [(768, 3072, 0.05, 16), (3000, 2000, 0.02, 3)])
def test_snack_linear_autograd_step_and_regrow(out, inp, density, B):
    from coo_spmm_sparse_gb300 import SnackLinear
    nnz = int(round(density * out * inp))
    lin = SnackLinear(inp, out, nnz, seed=7, std=0.05)
    with torch.no_grad():
        lin.bias.copy_(torch.linspace(-1, 1, out))
    g = np.random.default_rng(out + B)
    X = g.standard_normal((B, inp)).astype(np.float32)
    G = g.standard_normal((B, out)).astype(np.float32)
    _check_step(lin, X, G, "initial")

    # torch's optimizer updates the values in place through the Parameter
    opt = torch.optim.SGD(lin.parameters(), lr=0.1)
    before = lin.weight_values.detach().clone()
    grad = lin.weight_values.grad.detach().clone()
    opt.step()
    torch.cuda.synchronize()
    # torch's own update arithmetic (fused or not) rounds within an ulp or so
    torch.testing.assert_close(lin.weight_values.detach(), before - 0.1 * grad, rtol=1e-5,
                               atol=1e-8)
    _check_step(lin, X, G, "after an SGD step")

    # prune/regrow under the live Parameter: the view follows the new order
    ptr = lin.weight_values.data_ptr()
    row0, col0, val0 = lin.export()
    pruned, trials = lin.prune_regrow(0.3, 99)
    o = oracle.prune_regrow(out, inp, row0, col0, val0, 0.3, 99)
    assert (pruned, trials) == (o["pruned"], o["trials"])
    row1, col1, val1 = lin.export()
    assert np.array_equal(row1, o["row"]) and np.array_equal(col1, o["col"])
    assert np.array_equal(val1, o["val"])
    assert lin.weight_values.data_ptr() == ptr
    _check_step(lin, X, G, "after prune/regrow")
    opt.step()
    _check_step(lin, X, G, "after a second SGD step")


def test_snack_linear_refuses_backward_after_inplace_write():
    from coo_spmm_sparse_gb300 import SnackLinear
    lin = SnackLinear(256, 128, 2000, seed=3)
    x = torch.randn(4, 256, device="cuda", requires_grad=True)
    y = lin(x)
    with torch.no_grad():
        lin.weight_values.mul_(2.0)
    with pytest.raises(RuntimeError):
        y.sum().backward()


def test_snack_linear_frozen_values_then_written():
    # Values unchanged from one forward to the next: the module has the
    # column-ordered copy re-derived and dX streams it.  A write afterwards
    # makes the copy stale before the next dX, which then reads through the
    # permutation.  dX must match the oracle on the current values each time.
    from coo_spmm_sparse_gb300 import SnackLinear
    lin = SnackLinear(1500, 900, 40000, seed=5, std=0.1)
    g = np.random.default_rng(5)
    X = g.standard_normal((8, 1500)).astype(np.float32)
    G = g.standard_normal((8, 900)).astype(np.float32)
    _check_step(lin, X, G, "first")
    assert not lin._copy_current
    _check_step(lin, X, G, "values unchanged (copy re-derived)")
    assert lin._copy_current
    _check_step(lin, X, G, "values unchanged (copy kept)")
    with torch.no_grad():
        lin.weight_values.mul_(-1.5)
    _check_step(lin, X, G, "after an in-place write")
    assert not lin._copy_current
