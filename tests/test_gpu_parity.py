"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Forward, backward-input and backward-weight are compared element by element
within 1e-5 * sum|terms|; canonical order, CSR/CSC segmentation,
Algorithm 2 draws and prune/regrow results bit for bit.  Sizes span several
segments and tiles with ragged tails; the full-size workloads are checked on
sampled outputs (rows, columns, entries) that the oracle computes on their
own."""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import (assert_close, canonical, check_products, check_topology, dev, sn,
                         to_dev)

pytestmark = pytest.mark.gpu

ALL_B = [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 130, 256, 300]


def _layer_case(out, inp, row, col, val, batches, seed=0, fused=True):
    ref = canonical(out, inp, row, col, val)
    h = sn().snack_create(out, inp, row, col, val)
    check_topology(h, ref)
    g = np.random.default_rng(seed)
    for B in batches:
        X = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref, X, dY, fused=fused)
    return h, ref


# ------------------------------------------------------------ worked example

def test_table7_example():
    row, col, val = [2, 0, 1], [1, 2, 0], np.array([5, 3, 4], np.float32)
    h, ref = _layer_case(3, 3, row, col, val, [1, 3, 8])
    eye = to_dev(np.eye(3, dtype=np.float32))
    Y = sn().snack_forward(h, eye).cpu().numpy()
    assert np.array_equal(Y, np.array([[0, 4, 0], [0, 0, 5], [3, 0, 0]], np.float32))


# ------------------------------------------------------------ workloads

def test_toy256_all_batch_widths():
    L = workloads.workload("toy256").layers[0]
    row, col, val = L.coo()
    _layer_case(L.out, L.inp, row, col, val, ALL_B, seed=1)


def test_slices_after_the_first_accumulate_at_every_group_size():
    """Batches past the widest slice (256) run further slices that add into
    dW: remainders of 2 / 8 / 16 / 32 / 74 / 256 rows take slices of 2, 8,
    16, 32, 128 and 256 floats, so every lane-group size of the weight
    product's reduction (1, 2, 4, 8, 16, 32 lanes per entry) stores
    through its accumulate path."""
    L = workloads.workload("toy256").layers[0]
    row, col, val = L.coo()
    _layer_case(L.out, L.inp, row, col, val, [258, 264, 272, 288, 330, 512], seed=11)


@pytest.mark.parametrize("which", [0, 1])
def test_gpt2_mlp_layers(which):
    L = workloads.workload("gpt2_mlp").layers[which]
    row, col, val = L.coo()
    h, ref = _layer_case(L.out, L.inp, row, col, val, [], seed=2)
    for B in (1, 8, 32):
        X, dY = L.activations(B)
        check_products(h, L.out, L.inp, ref, X, dY)


def test_skewed_zipf_rows_full_size():
    L = workloads.workload("skewed").layers[0]
    row, col, val = L.coo()
    h, ref = _layer_case(L.out, L.inp, row, col, val, [], seed=3)
    # long rows are cut into several segments (split-row path)
    _, _, segs = sn().snack_plan(h, 0, 16)
    assert segs > L.out
    for B in (1, 16):
        X, dY = L.activations(B)
        Y1, dX1, dW1 = check_products(h, L.out, L.inp, ref, X, dY)
        # the split-row tickets re-arm: a second call gives identical bits
        Y2 = sn().snack_forward(h, to_dev(X))
        dX2 = sn().snack_backward_input(h, to_dev(dY))
        torch.cuda.synchronize()
        assert torch.equal(Y1, Y2) and torch.equal(dX1, dX2)


def test_gpt2_decoder_block_layers_and_regrow():
    wl = workloads.workload("gpt2_decoder")
    for L in wl.layers[:4]:
        row, col, val = L.coo()
        h, ref = _layer_case(L.out, L.inp, row, col, val, [], seed=4)
        X, dY = L.activations(256)
        check_products(h, L.out, L.inp, ref, X, dY)
        frac, seed = wl.extra["prune_frac"], 100 + L.seed
        pruned, trials = sn().snack_prune_regrow(h, frac, seed)
        o = oracle.prune_regrow(L.out, L.inp, ref["row"], ref["col"], ref["val"], frac, seed)
        assert (pruned, trials) == (o["pruned"], o["trials"])
        ref2 = canonical(L.out, L.inp, o["row"], o["col"], o["val"])
        check_topology(h, ref2)
        check_products(h, L.out, L.inp, ref2, X, dY, fused=False)


def _sampled_large(sparsity, batches):
    L = workloads.workload(f"large{sparsity}").layers[0]
    row, col, val = L.coo()
    ref = canonical(L.out, L.inp, row, col, val)
    h = sn().snack_create(L.out, L.inp, row, col, val)
    check_topology(h, ref)
    g = np.random.default_rng(sparsity)
    rows = np.sort(g.choice(L.out, 384, replace=False))
    cols = np.sort(g.choice(L.inp, 384, replace=False))
    ents = np.sort(g.choice(L.nnz, 4096, replace=False))
    rp, cp = ref["row_ptr"], ref["col_ptr"]
    rk = np.concatenate([np.arange(rp[r], rp[r + 1]) for r in rows])
    ck = np.concatenate([ref["csc_perm"][cp[c]:cp[c + 1]] for c in cols])
    m = sn()
    for B in batches:
        X, dY = L.activations(B)
        Xd, dYd = to_dev(X), to_dev(dY)
        Yo, Sy = oracle.forward(L.out, L.inp, ref["row"][rk], ref["col"][rk], ref["val"][rk], X)
        dXo, Sx = oracle.backward_input(L.out, L.inp, ref["row"][ck], ref["col"][ck],
                                        ref["val"][ck], dY)
        dWo, Sw = oracle.backward_weight(L.out, L.inp, ref["row"][ents], ref["col"][ents], X, dY)

        def check_dx(dX, tag):
            assert_close(f"dX[{B}] {tag}", dX.cpu().numpy()[:, cols], dXo[:, cols], Sx[:, cols])

        def check_dw(dW, tag):
            assert_close(f"dW[{B}] {tag}", dW.cpu().numpy()[ents], dWo, Sw)

        Y = m.snack_forward(h, Xd)
        dX, dW = m.snack_backward(h, Xd, dYd)
        torch.cuda.synchronize()
        assert_close(f"Y[{B}]", Y.cpu().numpy()[:, rows], Yo[:, rows], Sy[:, rows])
        check_dx(dX, "fused")
        check_dw(dW, "fused")
        # the standalone calls, the ones timed per op: dX from the
        # column-ordered value copy, then through the column permutation once
        # a writable values pointer has made that copy stale
        check_dx(m.snack_backward_input(h, dYd), "column-ordered copy")
        check_dw(m.snack_backward_weight(h, Xd, dYd), "standalone")
        m.snack_values(h)
        check_dx(m.snack_backward_input(h, dYd), "through the permutation")
        check_dx(m.snack_backward(h, Xd, dYd)[0], "fused, through the permutation")
        m.snack_values_changed(h)


@pytest.mark.parametrize("sparsity", [99, 95, 90])
def test_large_layer_full_size_sampled(sparsity):
    # 33 and 65 on the 95 % layer: batches just above a power of two, cut into
    # a power-of-two slice and a small remainder on large layers
    _sampled_large(sparsity, [1, 4, 8, 16, 64] + ([33, 65] if sparsity == 95 else []))


def test_large99_full_oracle_b16():
    # every output of the full-size 10000x10000 @99% layer at batch 16
    L = workloads.workload("large99").layers[0]
    row, col, val = L.coo()
    h, ref = _layer_case(L.out, L.inp, row, col, val, [], seed=5)
    X, dY = L.activations(16)
    check_products(h, L.out, L.inp, ref, X, dY, fused=False)


# ------------------------------------------------------------ resident operand

def test_resident_operand_full_oracle():
    # 3000 x 3000 at 47 %: 4.23 M entries, enough for the kernels that stage
    # the whole transposed operand in shared memory (slices of 1-4); full
    # oracle for every product, fused backward included.
    out = inp = 3000
    nnz = workloads.nnz_for(out, inp, 53)
    row, col = workloads.uniform_pattern(out, inp, nnz, 13)
    val = workloads.normal(nnz, 0.05, 13, 0)
    ref = canonical(out, inp, row, col, val)
    h = sn().snack_create(out, inp, row, col, val)
    for op in (0, 1, 2):
        assert sn().snack_plan(h, op, 4, with_resident=True)[3] == 1
    g = np.random.default_rng(14)
    for B in (1, 2, 3, 4):
        X = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref, X, dY)
    assert sn().snack_device_error(h) == 0


# ------------------------------------------------------------ dense-ish layer

def test_dense_lines_full_oracle():
    # 3000 x 3000 at 15 %: 1.35M entries, 450 per row and per column, every
    # slice width, batch slices above 64 accumulating dW; full oracle.
    out = inp = 3000
    nnz = workloads.nnz_for(out, inp, 85)
    row, col = workloads.uniform_pattern(out, inp, nnz, 11)
    val = workloads.normal(nnz, 0.05, 11, 0)
    ref = canonical(out, inp, row, col, val)
    h = sn().snack_create(out, inp, row, col, val)
    g = np.random.default_rng(12)
    for B in (4, 8, 16, 33, 64, 70, 200, 260):
        X = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref, X, dY)
    assert sn().snack_device_error(h) == 0


def test_nonfinite_values_stay_in_their_lines():
    # Entries with +-inf / NaN values poison only the outputs that sum them;
    # neighbouring lines (whose 16-byte loads cover those entries) are exact.
    g = np.random.default_rng(13)
    for (out, inp, dens) in ((300, 200, 0.2), (3000, 3000, 0.15)):
        nnz = workloads.nnz_for(out, inp, round(100 * (1 - dens)))
        row, col = workloads.uniform_pattern(out, inp, nnz, 13)
        val = workloads.normal(nnz, 1.0, 13, 0)
        bad = g.choice(nnz, 5, replace=False)
        val[bad] = np.array([np.inf, -np.inf, np.nan, np.inf, np.nan], np.float32)
        ref = canonical(out, inp, row, col, val)
        h = sn().snack_create(out, inp, row, col, val)
        X = g.standard_normal((16, inp)).astype(np.float32)
        dY = g.standard_normal((16, out)).astype(np.float32)
        Y = sn().snack_forward(h, to_dev(X)).cpu().numpy()
        dX = sn().snack_backward_input(h, to_dev(dY)).cpu().numpy()
        Yo, Sy = oracle.forward(out, inp, ref["row"], ref["col"], ref["val"], X)
        dXo, Sx = oracle.backward_input(out, inp, ref["row"], ref["col"], ref["val"], dY)
        fin_r = np.isfinite(Sy).all(axis=0)
        fin_c = np.isfinite(Sx).all(axis=0)
        assert fin_r.sum() < out and fin_c.sum() < inp
        assert_close("Y finite rows", Y[:, fin_r], Yo[:, fin_r], Sy[:, fin_r])
        assert_close("dX finite cols", dX[:, fin_c], dXo[:, fin_c], Sx[:, fin_c])
        assert not np.isfinite(Y[:, ~fin_r]).any()


# ------------------------------------------------------------ edge cases

def test_empty_layer_and_empty_lines():
    m = sn()
    h = m.snack_create(7, 5, np.zeros(0, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float32))
    X = to_dev(np.ones((3, 5), np.float32))
    dY = to_dev(np.ones((3, 7), np.float32))
    Y = m.snack_forward(h, X)
    dX, dW = m.snack_backward(h, X, dY)
    torch.cuda.synchronize()
    assert torch.all(Y == 0) and torch.all(dX == 0) and dW.numel() == 0
    # some empty rows and columns
    row = np.array([0, 0, 4, 6], np.int32)
    col = np.array([1, 4, 4, 0], np.int32)
    val = np.array([1.5, -2.0, 3.0, 0.25], np.float32)
    _layer_case(7, 5, row, col, val, [1, 4, 33])


@pytest.mark.parametrize("shape", [(1, 1), (1, 3000), (3000, 1), (16, 16), (64, 300)])
def test_dense_patterns(shape):
    out, inp = shape
    row = np.repeat(np.arange(out), inp).astype(np.int32)
    col = np.tile(np.arange(inp), out).astype(np.int32)
    val = np.random.default_rng(6).standard_normal(out * inp).astype(np.float32)
    _layer_case(out, inp, row, col, val, [1, 5, 16, 64])


def test_long_rows_and_columns_split():
    # three full rows of 20000 entries (rows split into many segments) and a
    # matching skew in columns
    g = np.random.default_rng(7)
    out, inp = 40, 20000
    cells = [np.arange(inp) + r * inp for r in (3, 17, 39)]
    cells.append(g.choice(out * inp, 5000, replace=False))
    cells = np.unique(np.concatenate(cells))
    g.shuffle(cells)
    row = (cells // inp).astype(np.int32)
    col = (cells % inp).astype(np.int32)
    val = g.standard_normal(cells.size).astype(np.float32)
    h, _ = _layer_case(out, inp, row, col, val, [1, 8, 64, 70])
    _, _, segs = sn().snack_plan(h, 0, 8)
    assert segs > out


def _heavy_tailed(out, inp, full_rows, seed):
    """Rows of 0-30 entries (geometric, a tenth of them empty) plus a few full
    rows: a heavy-tailed table, its long rows cut into many parts."""
    g = np.random.default_rng(seed)
    lens = np.minimum(g.geometric(0.09, out) - 1, 30)
    lens[g.random(out) < 0.1] = 0
    lens[full_rows] = inp
    cells = np.concatenate([r * inp + g.choice(inp, n, replace=False)
                            for r, n in enumerate(lens) if n > 0])
    g.shuffle(cells)
    row = (cells // inp).astype(np.int32)
    col = (cells % inp).astype(np.int32)
    val = g.standard_normal(cells.size).astype(np.float32)
    return row, col, val


def test_heavy_tailed_rows_with_empty_rows():
    out, inp = 3000, 2000
    row, col, val = _heavy_tailed(out, inp, [5, 1234, 2999, 3000 // 2], seed=11)
    # every slice width (1-256), odd batches, and the slice split above 256
    h, ref = _layer_case(out, inp, row, col, val, [1, 2, 3, 5, 8, 16, 17, 33, 64, 100, 256, 300],
                         seed=12)
    _, _, segs = sn().snack_plan(h, 0, 16)
    assert segs > out  # the full rows are split
    # split-row tickets re-arm: identical bits on a second call
    X = to_dev(np.random.default_rng(13).standard_normal((16, inp)).astype(np.float32))
    Y1 = sn().snack_forward(h, X)
    Y2 = sn().snack_forward(h, X)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
    # the segment tables are rebuilt with the topology
    pruned, trials = sn().snack_prune_regrow(h, 0.3, 21)
    o = oracle.prune_regrow(out, inp, ref["row"], ref["col"], ref["val"], 0.3, 21)
    assert (pruned, trials) == (o["pruned"], o["trials"])
    ref2 = canonical(out, inp, o["row"], o["col"], o["val"])
    check_topology(h, ref2)
    g = np.random.default_rng(14)
    for B in (1, 16, 64):
        Xb = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref2, Xb, dY, fused=False)


def test_one_row_of_sixty_thousand_entries():
    """A 64 x 60000 layer whose row 0 holds every column, beside rows of 0-30
    entries: the heavy-tailed cut gives that row about 900 parts, so the
    second pass's threads each walk many parts in several rounds of eight
    loads (at every slice width from 8 floats), and the tickets sum them at
    slices of 1-4."""
    out, inp = 64, 60000
    row, col, val = _heavy_tailed(out, inp, [0], seed=31)
    h, ref = _layer_case(out, inp, row, col, val, [1, 3, 8, 16, 40, 64, 200], seed=32)
    _, _, segs = sn().snack_plan(h, 0, 16)
    assert segs > out + 500  # the full row alone is cut into hundreds of parts


def test_halved_lines_wide_slices():
    # 2.2 M entries over 4096 x 4096 (537 per row and column): 64-wide
    # slices walk every line in four parts, 32-wide slices of the weight
    # product and of the fused backward in two, combined by the split-line
    # path; every product, the fused backward included, against the oracle
    out = inp = 4096
    h0, _ = sn().snack_create_random(out, inp, 2_200_000, 31)
    row, col, _ = sn().snack_export(h0)
    val = np.random.default_rng(32).standard_normal(row.size).astype(np.float32)
    h, ref = _layer_case(out, inp, row, col, val, [64, 41, 100, 200, 32, 16], seed=33)
    assert sn().snack_plan(h, 0, 64)[2] == 4 * out
    assert sn().snack_plan(h, 1, 64)[2] == 4 * inp
    assert sn().snack_plan(h, 2, 32)[2] == 2 * out
    # the parts' partial sums are summed again from scratch: identical bits on
    # a second call
    X = to_dev(np.random.default_rng(34).standard_normal((64, inp)).astype(np.float32))
    Y1 = sn().snack_forward(h, X)
    Y2 = sn().snack_forward(h, X)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
    # the cut copies are rebuilt with the topology
    pruned, trials = sn().snack_prune_regrow(h, 0.2, 35)
    o = oracle.prune_regrow(out, inp, ref["row"], ref["col"], ref["val"], 0.2, 35)
    assert (pruned, trials) == (o["pruned"], o["trials"])
    ref2 = canonical(out, inp, o["row"], o["col"], o["val"])
    check_topology(h, ref2)
    assert sn().snack_plan(h, 0, 64)[2] == 4 * out
    g = np.random.default_rng(36)
    for B in (64, 32):
        Xb = g.standard_normal((B, inp)).astype(np.float32)
        dY = g.standard_normal((B, out)).astype(np.float32)
        check_products(h, out, inp, ref2, Xb, dY)


def test_identity_pattern_bit_exact():
    n = 4099
    idx = np.arange(n, dtype=np.int32)
    perm = np.random.default_rng(8).permutation(n)
    h = sn().snack_create(n, n, idx[perm], idx[perm], np.ones(n, np.float32))
    for B in (1, 3, 16, 64, 100):
        X = to_dev(np.random.default_rng(B).standard_normal((B, n)).astype(np.float32))
        Y = sn().snack_forward(h, X)
        dX = sn().snack_backward_input(h, X)
        torch.cuda.synchronize()
        assert torch.equal(Y, X) and torch.equal(dX, X)


def test_device_pointer_input_and_side_stream():
    L = workloads.workload("toy256").layers[0]
    row, col, val = L.coo()
    ref = canonical(L.out, L.inp, row, col, val)
    h = sn().snack_create(L.out, L.inp, to_dev(row), to_dev(col), to_dev(val))
    check_topology(h, ref)
    X, dY = L.activations(4)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Y = sn().snack_forward(h, to_dev(X))
    s.synchronize()
    Yo, Sy = oracle.forward(L.out, L.inp, ref["row"], ref["col"], ref["val"], X)
    assert_close("Y", Y, Yo, Sy)


def test_column_ordered_value_copy_follows_writes():
    # dX streams a column-ordered copy of the values while the library owns
    # every write; a writable view switches it to the permutation path until
    # snack_values_changed() re-derives the copy.  Resident (batch 1) and
    # segment (batch 16) kernels, standalone and fused backward.
    m = sn()
    L = workloads.workload("gpt2_mlp").layers[0]
    row, col, val = L.coo()
    ref = canonical(L.out, L.inp, row, col, val)
    h = m.snack_create(L.out, L.inp, row, col, val)

    def check(vals):
        for B in (1, 16):
            X, dY = L.activations(B)
            check_products(h, L.out, L.inp, dict(ref, val=vals), X, dY)
    check(ref["val"])                              # copy current since creation
    v = m.snack_values(h)
    v.mul_(-0.5)                                   # written through the view
    check(ref["val"] * np.float32(-0.5))           # permutation path
    m.snack_values_changed(h)
    check(ref["val"] * np.float32(-0.5))           # copy re-derived
    v.add_(1.0)                                    # a write the handle is not told of
    m.snack_values(h)                              # ... until the view is taken again
    check(ref["val"] * np.float32(-0.5) + np.float32(1.0))


def test_values_view_updates_in_place():
    L = workloads.workload("toy256").layers[0]
    row, col, val = L.coo()
    h = sn().snack_create(L.out, L.inp, row, col, val)
    v = sn().snack_values(h)
    ref = canonical(L.out, L.inp, row, col, val)
    assert np.array_equal(v.cpu().numpy(), ref["val"])
    v.mul_(2.0)
    X, dY = L.activations(4)
    check_products(h, L.out, L.inp, dict(ref, val=ref["val"] * 2), X, dY, fused=False)


# ------------------------------------------------------------ errors

def test_invalid_inputs_return_status():
    m = sn()
    with pytest.raises(m.SnackError) as e:
        m.snack_create(4, 4, [0, 4], [0, 1], [1.0, 2.0])
    assert e.value.status == 2
    with pytest.raises(m.SnackError) as e:
        m.snack_create(4, 4, [1, 2, 1], [3, 0, 3], [1.0, 2.0, 3.0])
    assert e.value.status == 3
    with pytest.raises(m.SnackError) as e:
        m.snack_create(4, 4, [0, -1], [0, 1])
    assert e.value.status == 2
    h = m.snack_create(4, 4, [0, 1], [0, 1], [1.0, 2.0])
    X = torch.zeros(3 * 4 + 1, device=dev())
    with pytest.raises(m.SnackError) as e:      # misaligned X
        m._check(m._lib.snack_forward(h.ptr, m._ptr(X[1:]), m._ptr(X[:12]), 3, m._stream(None)), h)
    assert e.value.status == 1
    with pytest.raises(m.SnackError) as e:      # batch 0
        m._check(m._lib.snack_forward(h.ptr, m._ptr(X), m._ptr(X), 0, m._stream(None)), h)
    assert e.value.status == 1
    # the handle is still usable after rejected calls
    Y = m.snack_forward(h, torch.ones(2, 4, device=dev()))
    torch.cuda.synchronize()
    assert Y.cpu().numpy().tolist() == [[1, 2, 0, 0], [1, 2, 0, 0]]


# ------------------------------------------------------------ kernel choice

def test_plan_follows_batch_and_row_length():
    L = workloads.workload("large99").layers[0]
    h, _ = sn().snack_create_random(L.out, L.inp, L.nnz, 1)
    for B, w in ((1, 1), (2, 2), (3, 4), (5, 8), (16, 16), (17, 32), (64, 64), (65, 128),
                 (129, 256), (300, 256)):
        assert sn().snack_plan(h, 0, B)[0] == w
    assert sn().snack_plan(h, 0, 16)[1] == 32            # 100 entries per row
    # a 1 M-entry layer gathers its operand from global memory at every
    # width; a 5 M-entry one stages the whole 10000-line operand in shared
    # memory while its copies (one per SM) stay within the value bytes
    assert sn().snack_plan(h, 0, 1, with_resident=True)[3] == 0
    h5, _ = sn().snack_create_random(L.out, L.inp, 5 * L.nnz, 2)
    assert sn().snack_plan(h5, 0, 1, with_resident=True)[3] == 1
    assert sn().snack_plan(h5, 1, 2, with_resident=True)[3] == 1
    assert sn().snack_plan(h5, 0, 4, with_resident=True)[3] == 0
    assert sn().snack_plan(h5, 0, 16, with_resident=True)[3] == 0
    # dW of the 5 M-entry layer sweeps its operand in column panels while a
    # row's run per panel is long (500 entries per row: batch 8, not 16)
    assert sn().snack_plan(h5, 2, 8, with_resident=True)[3] == 2
    assert sn().snack_plan(h5, 2, 16, with_resident=True)[3] == 0
    # on a large layer a batch just above a power of two w >= 32 starts
    # with a slice of w (the remainder follows as its own slice)
    for B, w in ((9, 16), (33, 32), (40, 32), (41, 64), (65, 64), (129, 128), (300, 256)):
        assert sn().snack_plan(h5, 0, B)[0] == w, B
    # 64-wide slices of a large layer of long lines walk its lines in four
    # parts (four segments per row or column), and so do the weight
    # product's wider slices; its 32-wide slices walk halves; other widths
    # and small layers walk whole lines
    for op in (0, 1, 2):
        assert sn().snack_plan(h5, op, 64)[2] == 4 * L.out
        assert sn().snack_plan(h5, op, 32)[2] == (2 * L.out if op == 2 else L.out)
        assert sn().snack_plan(h5, op, 16)[2] == L.out
        assert sn().snack_plan(h5, op, 128)[2] == (4 * L.out if op == 2 else L.out)
    assert sn().snack_plan(h, 0, 64)[2] == L.out
    small = workloads.workload("toy256").layers[0]
    r, c, v = small.coo()
    h2 = sn().snack_create(small.out, small.inp, r, c, v)
    assert sn().snack_plan(h2, 0, 4)[1] == 8             # ~26 entries per row


# ------------------------------------------------------------ Algorithm 2

@pytest.mark.parametrize("shape", [(7, 9, 40), (300, 200, 6000), (3072, 768, 117965),
                                   (1000, 1000, 990000)])
def test_create_random_matches_oracle(shape):
    out, inp, nnz = shape
    for seed in (0, 12345):
        h, trials = sn().snack_create_random(out, inp, nnz, seed)
        r, c, _ = sn().snack_export(h)
        orow, ocol, otrials = oracle.uniform_init(out, inp, nnz, seed)
        assert trials == otrials
        cells = np.sort(orow.astype(np.int64) * inp + ocol)
        assert np.array_equal(r.astype(np.int64) * inp + c, cells)


# ------------------------------------------------------------ prune / regrow

@pytest.mark.parametrize("frac", [0.0, 0.05, 0.3, 1.0])
def test_prune_regrow_matches_oracle(frac):
    L = workloads.workload("gpt2_mlp").layers[0]
    row, col, val = L.coo()
    g = np.random.default_rng(9)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-30, -1e-30], np.float32)
    pick = g.choice(val.size, 500, replace=False)
    val[pick] = special[g.integers(0, special.size, 500)]
    val[g.choice(val.size, 2000, replace=False)] = 0.5  # many ties
    ref = canonical(L.out, L.inp, row, col, val)
    h = sn().snack_create(L.out, L.inp, row, col, val)
    for step in range(3):
        seed = 77 + step
        p, t = sn().snack_prune_regrow(h, frac, seed)
        o = oracle.prune_regrow(L.out, L.inp, ref["row"], ref["col"], ref["val"], frac, seed)
        assert (p, t) == (o["pruned"], o["trials"])
        ref = canonical(L.out, L.inp, o["row"], o["col"], o["val"])
        check_topology(h, ref)


def test_prune_regrow_dense_layer_reuses_pruned_cells():
    out, inp = 8, 8
    row = np.repeat(np.arange(out), inp).astype(np.int32)
    col = np.tile(np.arange(inp), out).astype(np.int32)
    val = np.arange(1, 65, dtype=np.float32)
    ref = canonical(out, inp, row, col, val)
    h = sn().snack_create(out, inp, row, col, val)
    p, t = sn().snack_prune_regrow(h, 0.25, 5)
    o = oracle.prune_regrow(out, inp, ref["row"], ref["col"], ref["val"], 0.25, 5)
    assert (p, t) == (o["pruned"], o["trials"])
    check_topology(h, canonical(out, inp, o["row"], o["col"], o["val"]))


def test_prune_regrow_large_layer():
    L = workloads.workload("large99").layers[0]
    row, col, val = L.coo()
    ref = canonical(L.out, L.inp, row, col, val)
    h = sn().snack_create(L.out, L.inp, row, col, val)
    p, t = sn().snack_prune_regrow(h, 0.3, 2024)
    o = oracle.prune_regrow(L.out, L.inp, ref["row"], ref["col"], ref["val"], 0.3, 2024)
    assert (p, t) == (o["pruned"], o["trials"])
    assert p == math.floor(float(np.float32(0.3)) * L.nnz)
    check_topology(h, canonical(L.out, L.inp, o["row"], o["col"], o["val"]))


# ------------------------------------------------------------ failure path

def test_bounded_wait_gives_up_and_context_stays_usable():
    # a device barrier that nothing completes: the bounded wait gives up,
    # records it and returns; the GPU keeps working
    m = sn()
    assert m.snack_selftest_wait() == 1
    L = workloads.workload("toy256").layers[0]
    row, col, val = L.coo()
    h, ref = _layer_case(L.out, L.inp, row, col, val, [4], seed=9)
    assert m.snack_device_error(h) == 0
