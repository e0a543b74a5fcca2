"""Column-panel SDDMM (the weight gradient with X^T swept through shared
memory panel by panel, slices of 8-64 floats) against the CPU oracle, full
outputs.

Layers get a panel partition at creation when they hold at least
SNACK_PANEL_MIN_NNZ entries (2^21 by default), and a backward-weight call
takes the sweep when the mean run of a row per panel is at least 64 entries.
The tests lower the size threshold and use layers with long rows so that the
sweep runs at every width, and cover its edge cases: a few full rows among
short ones (CTAs with no rows, rows spread over many warps), rows without
entries, warps with no entries, batches that are not a power of two, dW
accumulated over a second batch slice (batch 300 = 256 + 44), and a layer
whose warps would hold too many rows (it keeps the segment kernels).  The
other products of the same calls are checked too.  Tolerance: 1e-5 times
the oracle's sum of |terms| per element."""

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


def _sweeps(h, B):
    return sn().snack_plan(h, 2, B, with_resident=True)[3] == 2


def test_panel_sddmm_every_width(monkeypatch):
    out, inp = 600, 4000  # 30 % dense: 1200 entries per row
    nnz = workloads.nnz_for(out, inp, 70)
    row, col = workloads.uniform_pattern(out, inp, nnz, 21)
    val = workloads.normal(nnz, 0.05, 21, 0)
    h, ref = _layer(out, inp, row, col, val, monkeypatch)
    assert all(_sweeps(h, B) for B in (8, 16, 32, 64))
    g = np.random.default_rng(22)
    for B in (8, 12, 16, 31, 32, 64, 300):
        X = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref, X, dY)
    assert sn().snack_device_error(h) == 0


def test_panel_long_rows_empty_rows_and_idle_ctas(monkeypatch):
    # 24 full rows of 600 entries (each spans many warps, and the CTAs
    # between row-aligned shares get no rows), 900 rows of ~40 entries, a
    # few empty rows among them; columns 599 and 0 both used.
    out, inp = 1200, 600
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
    assert _sweeps(h, 8) and _sweeps(h, 16)
    for B in (8, 13, 16):
        X = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref, X, dY)
    assert sn().snack_device_error(h) == 0


def test_panel_tiny_layer_most_warps_idle(monkeypatch):
    out, inp, nnz = 64, 48, 100
    row, col = workloads.uniform_pattern(out, inp, nnz, 41)
    val = workloads.normal(nnz, 1.0, 41, 0)
    h, ref = _layer(out, inp, row, col, val, monkeypatch)
    assert _sweeps(h, 8)
    g = np.random.default_rng(42)
    for B in (5, 8):
        X = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref, X, dY)
    assert sn().snack_device_error(h) == 0


def test_panel_off_when_warps_would_hold_too_many_rows(monkeypatch):
    # 20000 rows of 1-2 entries: a warp's share covers many rows, more than
    # the sweep holds, so the layer keeps the segment kernels.
    out, inp = 20000, 500
    nnz = 30000
    row, col = workloads.uniform_pattern(out, inp, nnz, 51)
    val = workloads.normal(nnz, 1.0, 51, 0)
    h, ref = _layer(out, inp, row, col, val, monkeypatch)
    assert not _sweeps(h, 8)
    g = np.random.default_rng(52)
    X = g.standard_normal((16, inp)).astype(np.float32)
    dY = g.standard_normal((16, out)).astype(np.float32)
    check_products(h, out, inp, ref, X, dY)
