"""Column-panel kernels (slices of 8-64 floats; the operand swept through
shared memory panel by panel) against the CPU oracle, full outputs.

Layers get a panel partition at creation when they hold at least
SNACK_PANEL_MIN_NNZ entries (2^21 by default); the tests lower the threshold
so that small layers take the panel path too, and cover its edge cases:
lines cut by warp boundaries (one line over many warps), CTAs with no lines,
warps with no entries, lines without entries, batches that are not a power of
two, dW accumulated over a second batch slice (batch 300 = 256 + 44), dX from
the column-ordered value copy and through the permutation, and a layer whose
warps would hold too many lines (it keeps the segment kernels).  Tolerance:
1e-5 times the oracle's sum of |terms| per element."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import assert_close, canonical, check_products, sn, to_dev

pytestmark = pytest.mark.gpu


def _layer(out, inp, row, col, val, monkeypatch, min_nnz=1):
    monkeypatch.setenv("SNACK_PANEL_MIN_NNZ", str(min_nnz))
    ref = canonical(out, inp, row, col, val)
    h = sn().snack_create(out, inp, row, col, val)
    return h, ref


def _uses_panel(h, B):
    return [sn().snack_plan(h, op, B, with_resident=True)[3] for op in (0, 1, 2)]


def test_panel_uniform_layer_all_widths(monkeypatch):
    out, inp = 3000, 2600
    nnz = workloads.nnz_for(out, inp, 95)
    row, col = workloads.uniform_pattern(out, inp, nnz, 21)
    val = workloads.normal(nnz, 0.05, 21, 0)
    h, ref = _layer(out, inp, row, col, val, monkeypatch)
    assert _uses_panel(h, 16) == [2, 2, 2]
    g = np.random.default_rng(22)
    for B in (8, 12, 16, 31, 32, 64, 300):
        X = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref, X, dY)
        # dX through the column permutation once a writable values view is out
        sn().snack_values(h)
        dX = sn().snack_backward_input(h, to_dev(dY))
        torch.cuda.synchronize()
        dXo, Sx = oracle.backward_input(out, inp, ref["row"], ref["col"], ref["val"], dY)
        assert_close(f"dX(perm) B={B}", dX, dXo, Sx)
        sn().snack_values_changed(h)
    assert sn().snack_device_error(h) == 0


def test_panel_long_lines_empty_lines_and_idle_ctas(monkeypatch):
    # 24 full rows of 4000 entries (each spans many warps, and the CTAs
    # between row-aligned shares get no lines), 900 rows of ~40 entries,
    # a few empty rows among them; columns 3999 and 0 both used.
    out, inp = 1200, 4000
    g = np.random.default_rng(31)
    rows, cols = [], []
    full = g.choice(out, 24, replace=False)
    empty = set(g.choice(out, 12, replace=False)) - set(full)
    for r in range(out):
        if r in full:
            c = np.arange(inp)
        elif r in empty:
            continue
        else:
            c = g.choice(inp, int(g.integers(20, 60)), replace=False)
        rows.append(np.full(c.size, r))
        cols.append(c)
    row = np.concatenate(rows).astype(np.int32)
    col = np.concatenate(cols).astype(np.int32)
    perm = g.permutation(row.size)
    row, col = row[perm], col[perm]
    val = g.standard_normal(row.size).astype(np.float32)
    h, ref = _layer(out, inp, row, col, val, monkeypatch)
    assert _uses_panel(h, 8)[0] == 2 and _uses_panel(h, 8)[2] == 2
    for B in (8, 17, 64):
        X = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref, X, dY)
    assert sn().snack_device_error(h) == 0


def test_panel_tiny_layer_most_warps_idle(monkeypatch):
    out, inp, nnz = 64, 48, 100
    row, col = workloads.uniform_pattern(out, inp, nnz, 41)
    val = workloads.normal(nnz, 1.0, 41, 0)
    h, ref = _layer(out, inp, row, col, val, monkeypatch)
    assert _uses_panel(h, 16) == [2, 2, 2]
    g = np.random.default_rng(42)
    for B in (8, 16, 32, 64):
        X = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref, X, dY)
    assert sn().snack_device_error(h) == 0


def test_panel_off_when_warps_would_hold_too_many_lines(monkeypatch):
    # 20000 rows of 1-2 entries: a warp's share covers many lines, more than
    # the panel kernels hold, so the layer keeps the segment kernels.
    out, inp = 20000, 500
    nnz = 30000
    row, col = workloads.uniform_pattern(out, inp, nnz, 51)
    val = workloads.normal(nnz, 1.0, 51, 0)
    h, ref = _layer(out, inp, row, col, val, monkeypatch)
    assert _uses_panel(h, 16)[0] == 0
    g = np.random.default_rng(52)
    X = g.standard_normal((16, inp)).astype(np.float32)
    dY = g.standard_normal((16, out)).astype(np.float32)
    check_products(h, out, inp, ref, X, dY)
