"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare with the CPU oracle on the same seeded inputs.

Tolerance (fp32 outputs): |gpu - oracle| <= 1e-5 * S per element, where S
is the oracle's sum of |term| for that element.  Topology / index results are
compared bit for bit."""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = 1e-5


def sn():
    import coo_spmm_sparse_gb300 as m
    return m


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def assert_close(name, got, want, S, tol=TOL):
    got = got.detach().cpu().numpy() if isinstance(got, torch.Tensor) else got
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    err = np.abs(got - want)
    bad = ~(err <= tol * S)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / np.maximum(S, 1e-300), 0)), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} elements outside 1e-5*S; worst at {i}: "
                             f"gpu={got[i]!r} oracle={want[i]!r} S={S[i]!r}")


def canonical(out, inp, row, col, val):
    return oracle.canonicalize(out, inp, row, col, val)


def check_topology(h, ref):
    m = sn()
    r, c, v = m.snack_export(h)
    assert np.array_equal(r, ref["row"])
    assert np.array_equal(c, ref["col"])
    # values compared bit for bit (NaN payloads and signed zeros included)
    assert np.array_equal(v.view(np.uint32), np.asarray(ref["val"], np.float32).view(np.uint32))
    seg = m.snack_export_segments(h)
    for k in ("row_ptr", "col_ptr", "csc_row", "csc_perm"):
        assert np.array_equal(seg[k], ref[k]), k


def check_products(h, out, inp, ref, X, dY, fused=True):
    """Forward, backward-input, backward-weight (and the fused backward) vs oracle."""
    m = sn()
    Xd, dYd = to_dev(X), to_dev(dY)
    Y = m.snack_forward(h, Xd)
    dX = m.snack_backward_input(h, dYd)
    dW = m.snack_backward_weight(h, Xd, dYd)
    torch.cuda.synchronize()
    Yo, Sy = oracle.forward(out, inp, ref["row"], ref["col"], ref["val"], X)
    dXo, Sx = oracle.backward_input(out, inp, ref["row"], ref["col"], ref["val"], dY)
    dWo, Sw = oracle.backward_weight(out, inp, ref["row"], ref["col"], X, dY)
    assert_close("Y", Y, Yo, Sy)
    assert_close("dX", dX, dXo, Sx)
    assert_close("dW", dW, dWo, Sw)
    if fused:
        dX2, dW2 = m.snack_backward(h, Xd, dYd)
        torch.cuda.synchronize()
        assert_close("dX(fused)", dX2, dXo, Sx)
        assert_close("dW(fused)", dW2, dWo, Sw)
    return Y, dX, dW
