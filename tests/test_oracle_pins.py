"""Pins for the CPU oracle against facts fixed outside the oracle itself.

Each test ties one oracle routine to the paper ("Beyond Masked Sparsity:
SNACK Enables Truly Sparse Neural Networks on GPU") or to mathematics that
does not depend on the oracle: the printed Table 7 example, dense matmul in
fp64 (numpy), scipy.sparse's CSR/CSC builders, the published SplitMix64
output sequence, the closed-form expected trial count of Algorithm 2, and
brute-force restatements on tiny inputs.  CPU only.
"""

import json
import math
import os
import struct

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U32 = 2.0 ** -24  # fp32 unit roundoff


def _table7():
    with open(os.path.join(GOLDEN, "table7_formats.json")) as f:
        return json.load(f)


def _dense(out, inp, row, col, val):
    W = np.zeros((out, inp), np.float64)
    W[row, col] = val
    return W


def _random_layer(g, out, inp, density):
    cells = np.flatnonzero(g.random(out * inp) < density)
    g.shuffle(cells)
    row = (cells // inp).astype(np.int32)
    col = (cells % inp).astype(np.int32)
    val = g.standard_normal(cells.size).astype(np.float32)
    return row, col, val


# --------------------------------------------------------------------------
# Appendix B, Table 7
# --------------------------------------------------------------------------

@pytest.mark.parametrize("order", [[0, 1, 2], [2, 0, 1], [1, 2, 0], [2, 1, 0]])
def test_table7_csr_csc(order):
    t = _table7()
    row = np.array(t["coo"]["row"])[order]
    col = np.array(t["coo"]["col"])[order]
    val = np.array(t["coo"]["data"], np.float32)[order]
    r = oracle.canonicalize(3, 3, row, col, val)
    assert r["row_ptr"].tolist() == t["csr"]["indptr"]
    assert r["col"].tolist() == t["csr"]["indices"]
    assert r["val"].tolist() == t["csr"]["data"]
    assert r["col_ptr"].tolist() == t["csc"]["indptr"]
    assert r["csc_row"].tolist() == t["csc"]["indices"]
    assert r["val"][r["csc_perm"]].tolist() == t["csc"]["data"]
    assert r["row"].tolist() == t["coo"]["row"]


def test_table7_products_reproduce_A():
    t = _table7()
    A = np.array(t["dense_A"], np.float64)
    r = oracle.canonicalize(3, 3, t["coo"]["row"], t["coo"]["col"], t["coo"]["data"])
    eye = np.eye(3, dtype=np.float32)
    Y, _ = oracle.forward(3, 3, r["row"], r["col"], r["val"], eye)
    assert np.array_equal(Y, A.T)            # Y = I W^T
    dX, _ = oracle.backward_input(3, 3, r["row"], r["col"], r["val"], eye)
    assert np.array_equal(dX, A)             # dX = I W
    X = np.arange(1, 7, dtype=np.float32).reshape(2, 3)
    dY = np.arange(7, 13, dtype=np.float32).reshape(2, 3)
    dW, _ = oracle.backward_weight(3, 3, r["row"], r["col"], X, dY)
    full = dY.astype(np.float64).T @ X.astype(np.float64)
    assert dW.tolist() == [full[0, 2], full[1, 0], full[2, 1]]


# --------------------------------------------------------------------------
# §3.1 Algorithm 1, §3.4, Appendix F: brute force against dense matmul
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(120))
def test_dense_bruteforce_all_three(seed):
    g = np.random.default_rng(seed)
    out, inp = int(g.integers(1, 17)), int(g.integers(1, 17))
    B = int(g.integers(1, 5))
    row, col, val = _random_layer(g, out, inp, float(g.uniform(0.05, 0.9)))
    X = g.standard_normal((B, inp)).astype(np.float32)
    dY = g.standard_normal((B, out)).astype(np.float32)
    W = _dense(out, inp, row, col, val)
    X64, dY64 = X.astype(np.float64), dY.astype(np.float64)

    Y, S = oracle.forward(out, inp, row, col, val, X)
    ref = X64 @ W.T
    assert np.all(np.abs(Y - ref) <= U32 * np.abs(ref) + 1e-12 * S + 1e-300)
    assert np.allclose(S, np.abs(X64) @ np.abs(W).T, rtol=1e-12, atol=0)

    dX, S = oracle.backward_input(out, inp, row, col, val, dY)
    ref = dY64 @ W
    assert np.all(np.abs(dX - ref) <= U32 * np.abs(ref) + 1e-12 * S + 1e-300)
    assert np.allclose(S, np.abs(dY64) @ np.abs(W), rtol=1e-12, atol=0)

    dW, S = oracle.backward_weight(out, inp, row, col, X, dY)
    full = dY64.T @ X64
    ref = full[row, col]
    assert dW.shape == (row.size,)          # exactly nnz entries, aligned
    assert np.all(np.abs(dW - ref) <= U32 * np.abs(ref) + 1e-12 * S + 1e-300)
    assert np.allclose(S, (np.abs(dY64).T @ np.abs(X64))[row, col], rtol=1e-12, atol=0)


def test_all_ones_pattern_is_dense_linear():
    g = np.random.default_rng(7)
    out, inp, B = 9, 13, 3
    row = np.repeat(np.arange(out), inp).astype(np.int32)
    col = np.tile(np.arange(inp), out).astype(np.int32)
    Wd = g.standard_normal((out, inp)).astype(np.float32)
    val = Wd.reshape(-1)
    X = g.standard_normal((B, inp)).astype(np.float32)
    Y, S = oracle.forward(out, inp, row, col, val, X)
    ref = X.astype(np.float64) @ Wd.astype(np.float64).T
    assert np.all(np.abs(Y - ref) <= U32 * np.abs(ref) + 1e-12 * S)


def test_identity_pattern_is_bit_exact():
    g = np.random.default_rng(3)
    n, B = 37, 5
    idx = np.arange(n, dtype=np.int32)
    one = np.ones(n, np.float32)
    X = g.standard_normal((B, n)).astype(np.float32)
    dY = g.standard_normal((B, n)).astype(np.float32)
    Y, _ = oracle.forward(n, n, idx, idx, one, X)
    assert np.array_equal(Y, X)
    dX, _ = oracle.backward_input(n, n, idx, idx, one, dY)
    assert np.array_equal(dX, dY)


def test_backward_input_is_forward_of_swapped_indices():
    g = np.random.default_rng(11)
    out, inp, B = 23, 31, 4
    row, col, val = _random_layer(g, out, inp, 0.2)
    dY = g.standard_normal((B, out)).astype(np.float32)
    dX, S1 = oracle.backward_input(out, inp, row, col, val, dY)
    dX2, S2 = oracle.forward(inp, out, col, row, val, dY)
    assert np.array_equal(dX, dX2) and np.array_equal(S1, S2)


def test_empty_rows_columns_and_nnz0():
    out, inp, B = 6, 5, 2
    row = np.array([1, 1, 4], np.int32)
    col = np.array([0, 3, 3], np.int32)
    val = np.array([2.0, -1.0, 0.5], np.float32)
    X = np.ones((B, inp), np.float32)
    Y, S = oracle.forward(out, inp, row, col, val, X)
    for r in (0, 2, 3, 5):
        assert np.all(Y[:, r] == 0.0) and np.all(S[:, r] == 0.0)
    dX, _ = oracle.backward_input(out, inp, row, col, val, np.ones((B, out), np.float32))
    for c in (1, 2, 4):
        assert np.all(dX[:, c] == 0.0)
    e = np.zeros(0, np.int32)
    Y, S = oracle.forward(out, inp, e, e, np.zeros(0, np.float32), X)
    assert np.all(Y == 0) and np.all(S == 0)
    dW, _ = oracle.backward_weight(out, inp, e, e, X, np.ones((B, out), np.float32))
    assert dW.size == 0


def test_linearity_in_values_and_input():
    g = np.random.default_rng(5)
    out, inp, B = 12, 10, 3
    row, col, v1 = _random_layer(g, out, inp, 0.4)
    v2 = g.standard_normal(row.size).astype(np.float32)
    X = g.standard_normal((B, inp)).astype(np.float32)
    Ya, Sa = oracle.forward(out, inp, row, col, v1, X)
    Yb, Sb = oracle.forward(out, inp, row, col, v2, X)
    Yc, _ = oracle.forward(out, inp, row, col, (v1.astype(np.float64) + v2).astype(np.float32), X)
    assert np.all(np.abs(Yc - (Ya.astype(np.float64) + Yb)) <= 4 * U32 * (Sa + Sb) + 1e-30)
    Yd, _ = oracle.forward(out, inp, row, col, v1, 2 * X)
    assert np.array_equal(Yd, 2 * Ya)  # scaling by 2 is exact


# --------------------------------------------------------------------------
# Canonicalisation against scipy.sparse
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(20))
def test_canonicalize_matches_scipy(seed):
    sp = pytest.importorskip("scipy.sparse")
    g = np.random.default_rng(100 + seed)
    out, inp = int(g.integers(1, 60)), int(g.integers(1, 60))
    row, col, val = _random_layer(g, out, inp, float(g.uniform(0.0, 0.5)))
    r = oracle.canonicalize(out, inp, row, col, val)
    csr = sp.csr_matrix((val, (row, col)), shape=(out, inp))
    csr.sort_indices()
    assert np.array_equal(r["row_ptr"], csr.indptr)
    assert np.array_equal(r["col"], csr.indices)
    assert np.array_equal(r["val"], csr.data)
    csc = sp.csc_matrix((val, (row, col)), shape=(out, inp))
    csc.sort_indices()
    assert np.array_equal(r["col_ptr"], csc.indptr)
    assert np.array_equal(r["csc_row"], csc.indices)
    assert np.array_equal(r["val"][r["csc_perm"]], csc.data)
    # src maps canonical entries back to the user's positions
    assert np.array_equal(row[r["src"]], r["row"]) and np.array_equal(col[r["src"]], r["col"])
    assert np.array_equal(np.sort(r["csc_perm"]), np.arange(row.size))


def test_canonicalize_rejects_bad_input():
    with pytest.raises(oracle.OracleError) as e:
        oracle.canonicalize(4, 4, [0, 4], [0, 0])
    assert e.value.code == oracle.ERR_RANGE and e.value.bad == 1
    with pytest.raises(oracle.OracleError) as e:
        oracle.canonicalize(4, 4, [0, 1], [0, -1])
    assert e.value.code == oracle.ERR_RANGE
    with pytest.raises(oracle.OracleError) as e:
        oracle.canonicalize(4, 4, [2, 1, 2], [3, 0, 3])
    assert e.value.code == oracle.ERR_DUPLICATE


# --------------------------------------------------------------------------
# getrand(): SplitMix64 and the cell reduction
# --------------------------------------------------------------------------

def test_splitmix64_published_sequence():
    # First outputs of SplitMix64 started from state 0 (Vigna's reference
    # splitmix64.c, the generator of Steele, Lea and Flood, OOPSLA 2014).
    expected = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F,
                0xF88BB8A8724C81EC]
    assert [oracle.splitmix64(0, t) for t in range(4)] == expected


def test_splitmix64_is_a_counter_stream():
    # draw t from seed s equals draw 0 from seed s + t*gamma (state advance)
    gamma = 0x9E3779B97F4A7C15
    for s in (0, 1, 12345, 2**63 + 7):
        for t in (0, 1, 5, 1000):
            assert oracle.splitmix64(s, t) == oracle.splitmix64((s + t * gamma) % 2**64, 0)


def test_cell_index_range_and_monotone():
    for n in (1, 2, 3, 100, 10**8, 2**40 + 3):
        xs = [0, 1, 2**63, 2**64 - 1, 0x123456789ABCDEF]
        idx = [oracle.cell_index(x, n) for x in xs]
        assert all(0 <= i < n for i in idx)
        assert idx == [(x * n) >> 64 for x in xs]
        assert oracle.cell_index(2**64 - 1, n) == n - 1
        assert oracle.cell_index(0, n) == 0


# --------------------------------------------------------------------------
# §3.3 Algorithm 2
# --------------------------------------------------------------------------

def test_alg2_invariants():
    out, inp = 300, 200
    nnz = workloads.nnz_for(out, inp, 90)
    row, col, trials = oracle.uniform_init(out, inp, nnz, seed=42)
    assert row.size == nnz and trials >= nnz
    assert row.min() >= 0 and row.max() < out and col.min() >= 0 and col.max() < inp
    cells = row.astype(np.int64) * inp + col
    assert np.unique(cells).size == nnz


def test_alg2_matches_python_restatement_tiny():
    # Same definition written out with Python integers and a Python set.
    gamma, M = 0x9E3779B97F4A7C15, 2**64 - 1

    def draw(seed, t):
        z = (seed + (t + 1) * gamma) & M
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
        return z ^ (z >> 31)

    for seed in (0, 1, 99):
        out, inp, count = 5, 7, 20
        seen, acc, t = set(), [], 0
        while len(acc) < count:
            p = (draw(seed, t) * out * inp) >> 64
            t += 1
            if p not in seen:
                seen.add(p)
                acc.append(p)
        row, col, trials = oracle.uniform_init(out, inp, count, seed)
        assert trials == t
        assert (row.astype(np.int64) * inp + col).tolist() == acc


def test_alg2_expected_trials_closed_form():
    # E[trials] = sum_{i<nnz} mk/(mk-i); each step is geometric with
    # success probability p_i = 1 - i/mk (§3.3, Appendix F).
    mk, nnz, seeds = 400, 300, 300
    p = 1.0 - np.arange(nnz) / mk
    mean = np.sum(1.0 / p)
    var = np.sum((1.0 - p) / p**2)
    got = np.array([oracle.uniform_init(20, 20, nnz, s)[2] for s in range(seeds)], float)
    assert abs(got.mean() - mean) <= 4.0 * math.sqrt(var / seeds)


def test_alg2_rejection_penalty_approximation():
    # zeta = E[trials]/nnz ~ -ln(eta)/(1-eta) for large mk (Appendix F).
    out, inp = 400, 500
    for eta in (0.5, 0.9):
        nnz = workloads.nnz_for(out, inp, eta * 100)
        tr = np.mean([oracle.uniform_init(out, inp, nnz, s)[2] for s in range(5)])
        zeta = -math.log(eta) / (1.0 - eta)
        assert abs(tr / nnz - zeta) / zeta < 0.01


def test_alg2_uniform_marginals_chi2():
    stats = pytest.importorskip("scipy.stats")
    out, inp, nnz = 40, 30, 120
    rc = np.zeros(out)
    cc = np.zeros(inp)
    for s in range(400):
        row, col, _ = oracle.uniform_init(out, inp, nnz, 1000 + s)
        rc += np.bincount(row, minlength=out)
        cc += np.bincount(col, minlength=inp)
    assert stats.chisquare(rc).pvalue > 1e-4
    assert stats.chisquare(cc).pvalue > 1e-4


# --------------------------------------------------------------------------
# Appendix G: magnitude prune + uniform regrow
# --------------------------------------------------------------------------

def _bits_abs(v):
    return struct.unpack("<I", struct.pack("<f", float(v)))[0] & 0x7FFFFFFF


def _prune_regrow_bruteforce(out, inp, row, col, val, frac, seed):
    nnz = len(row)
    P = int(math.floor(float(np.float32(frac)) * nnz)) if frac > 0 else 0
    order = sorted(range(nnz), key=lambda k: (_bits_abs(val[k]), k))
    gone = set(order[:P])
    surv = {int(row[k]) * inp + int(col[k]): float(val[k]) for k in range(nnz) if k not in gone}
    taken = set(surv)
    new, t = [], 0
    while len(new) < P:
        p = (oracle.splitmix64(seed, t) * out * inp) >> 64
        t += 1
        if p not in taken:
            taken.add(p)
            new.append(p)
    cells = sorted(list(surv) + new)
    return ([c // inp for c in cells], [c % inp for c in cells],
            [surv.get(c, 0.0) for c in cells], P, t)


@pytest.mark.parametrize("seed", range(25))
def test_prune_regrow_bruteforce_tiny(seed):
    g = np.random.default_rng(500 + seed)
    out, inp = int(g.integers(2, 9)), int(g.integers(2, 9))
    row, col, val = _random_layer(g, out, inp, float(g.uniform(0.2, 0.9)))
    if row.size == 0:
        return
    # ties, signed zeros, infinities and NaN in the magnitudes
    special = [0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan]
    for k in range(row.size):
        if g.random() < 0.3:
            val[k] = special[int(g.integers(0, len(special)))]
    r = oracle.canonicalize(out, inp, row, col, val)
    frac = float(g.choice([0.0, 0.05, 0.3, 0.5, 1.0]))
    res = oracle.prune_regrow(out, inp, r["row"], r["col"], r["val"], frac, seed)
    er, ec, ev, P, t = _prune_regrow_bruteforce(out, inp, r["row"], r["col"], r["val"],
                                                frac, seed)
    assert res["pruned"] == P and res["trials"] == t
    assert res["row"].tolist() == er and res["col"].tolist() == ec
    np.testing.assert_array_equal(res["val"], np.array(ev, np.float32))


def test_prune_regrow_invariants_and_count():
    out, inp = 200, 150
    nnz = workloads.nnz_for(out, inp, 95)
    row, col = workloads.uniform_pattern(out, inp, nnz, 3)
    val = workloads.normal(nnz, 0.02, 3, 0)
    r = oracle.canonicalize(out, inp, row, col, val)
    res = oracle.prune_regrow(out, inp, r["row"], r["col"], r["val"], 0.3, 77)
    assert res["pruned"] == int(math.floor(float(np.float32(0.3)) * nnz))
    cells = res["row"].astype(np.int64) * inp + res["col"]
    assert cells.size == nnz and np.all(np.diff(cells) > 0)   # canonical, unique
    old = dict(zip((r["row"].astype(np.int64) * inp + r["col"]).tolist(), r["val"].tolist()))
    mags = np.sort(np.abs(r["val"]))
    thresh = mags[res["pruned"] - 1]
    kept = 0
    for c, v in zip(cells.tolist(), res["val"].tolist()):
        if c in old and old[c] == v and abs(v) >= thresh:
            kept += 1
        else:
            assert v == 0.0                                   # regrown entries start at 0
    assert kept >= nnz - 2 * res["pruned"]


def test_prune_count_is_the_floor_of_the_float_fraction_times_nnz():
    """P = floor(f * nnz) for the float32 f the call takes: the exact product
    of the float's value and nnz (rational arithmetic here), so 0.7f * 10 is
    6 (0.7f is just below 0.7) while 0.3f * 10 is 3; no pruning for f <= 0
    or NaN, everything for f >= 1."""
    from fractions import Fraction
    for f in (0.3, 0.7, 0.05, 0.5, 0.25, 1e-7, 0.999999):
        for nnz in (1, 10, 6554, 117965, 1_000_000, 10_000_000, (1 << 28) + 3):
            want = math.floor(Fraction(float(np.float32(f))) * nnz)
            assert oracle.prune_count(f, nnz) == want, (f, nnz)
    assert oracle.prune_count(0.7, 10) == 6 and oracle.prune_count(0.3, 10) == 3
    for f in (0.0, -0.5, float("nan")):
        assert oracle.prune_count(f, 1000) == 0
    for f in (1.0, 1.5, float("inf")):
        assert oracle.prune_count(f, 1000) == 1000


def test_prune_zero_fraction_is_identity():
    out, inp = 20, 20
    row, col = workloads.uniform_pattern(out, inp, 50, 1)
    val = workloads.normal(50, 1.0, 1, 0)
    r = oracle.canonicalize(out, inp, row, col, val)
    res = oracle.prune_regrow(out, inp, r["row"], r["col"], r["val"], 0.0, 5)
    assert res["pruned"] == 0 and res["trials"] == 0
    assert np.array_equal(res["row"], r["row"]) and np.array_equal(res["val"], r["val"])


def test_just_pruned_cell_is_eligible_for_regrowth():
    # 3x3 with 8 stored cells: after pruning one, the only free cells are the
    # empty one and the pruned one; some seed must re-draw the pruned cell.
    out = inp = 3
    cells = [c for c in range(9) if c != 4]
    row = np.array([c // 3 for c in cells], np.int32)
    col = np.array([c % 3 for c in cells], np.int32)
    val = np.arange(1, 9, dtype=np.float32)        # cell 0 has the smallest |val|
    hit = None
    for seed in range(64):
        res = oracle.prune_regrow(out, inp, row, col, val, 0.125, seed)
        got = (res["row"].astype(int) * 3 + res["col"]).tolist()
        if got == cells:
            hit = res
            break
    assert hit is not None
    assert hit["val"][0] == 0.0 and hit["val"][1:].tolist() == val[1:].tolist()


def test_nnz_rounding():
    assert workloads.nnz_for(256, 256, 90) == 6554         # 6553.6 rounds up
    assert workloads.nnz_for(8192, 8192, 99) == 671089      # 671088.64
    assert workloads.nnz_for(3072, 768, 95) == 117965       # 117964.8
    assert workloads.nnz_for(10000, 10000, 95) == 5_000_000


# ------------------------------------------------------------ optimizer steps
# The update rules are the textbook ones; torch.optim's CPU implementations
# in float64 are the library routines they are pinned to, one step at a time
# from a given (float32) state.

def _torch_step(opt_cls, val, g, state, **kw):
    import torch
    p = torch.nn.Parameter(torch.from_numpy(np.asarray(val, np.float64).copy()))
    opt = opt_cls([p], **kw)
    if state:
        opt.state[p] = state(p)
    p.grad = torch.from_numpy(np.asarray(g, np.float64).copy())
    opt.step()
    return p.detach().numpy(), opt.state[p]


def test_weight_gradient64_matches_rounded_gradient():
    g = np.random.default_rng(40)
    out, inp, B = 9, 7, 5
    cells = g.choice(out * inp, 20, replace=False)
    row, col = (cells // inp).astype(np.int32), (cells % inp).astype(np.int32)
    X = g.standard_normal((B, inp)).astype(np.float32)
    dY = g.standard_normal((B, out)).astype(np.float32)
    g64, S = oracle.weight_gradient64(out, inp, row, col, X, dY)
    dense = dY.astype(np.float64).T @ X.astype(np.float64)
    assert np.allclose(g64, dense[row, col], rtol=1e-13, atol=1e-13)
    dW, S2 = oracle.backward_weight(out, inp, row, col, X, dY)
    assert np.array_equal(dW, g64.astype(np.float32)) and np.array_equal(S, S2)


@pytest.mark.parametrize("momentum,wd", [(0.0, 0.0), (0.0, 0.01), (0.9, 0.0), (0.9, 5e-4)])
def test_sgd_update_matches_torch(momentum, wd):
    import torch
    g = np.random.default_rng(41)
    n = 50
    val = g.standard_normal(n).astype(np.float32)
    grad = g.standard_normal(n)
    buf = g.standard_normal(n).astype(np.float32)
    lr = 0.05
    state = (lambda p: {"momentum_buffer": torch.from_numpy(buf.astype(np.float64))}) \
        if momentum else None
    want, st = _torch_step(torch.optim.SGD, val, grad, state, lr=lr, momentum=momentum,
                           weight_decay=wd)
    got, bout = oracle.sgd_update(val, grad, buf, lr, momentum, wd)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-15)
    if momentum:
        assert np.allclose(bout, st["momentum_buffer"].numpy(), rtol=1e-14, atol=1e-15)
    # torch's first momentum step (no buffer yet) equals ours from a zero buffer
    want0, _ = _torch_step(torch.optim.SGD, val, grad, None, lr=lr, momentum=momentum,
                           weight_decay=wd)
    got0, _ = oracle.sgd_update(val, grad, np.zeros(n, np.float32), lr, momentum, wd)
    assert np.allclose(got0, want0, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("t,wd", [(1, 0.0), (2, 0.0), (7, 0.01), (1000, 0.0)])
def test_adam_update_matches_torch(t, wd):
    import torch
    g = np.random.default_rng(42 + t)
    n = 50
    val = g.standard_normal(n).astype(np.float32)
    grad = g.standard_normal(n) * 1e-2
    m = (g.standard_normal(n) * 1e-2).astype(np.float32) if t > 1 else np.zeros(n, np.float32)
    v = (g.random(n) * 1e-4).astype(np.float32) if t > 1 else np.zeros(n, np.float32)
    kw = dict(lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=wd)

    def state(p):
        return {"step": torch.tensor(float(t - 1)),
                "exp_avg": torch.from_numpy(m.astype(np.float64)),
                "exp_avg_sq": torch.from_numpy(v.astype(np.float64))}
    want, st = _torch_step(torch.optim.Adam, val, grad, state, **kw)
    got, mo, vo = oracle.adam_update(val, grad, m, v, 1e-3, 0.9, 0.999, 1e-8, wd, t)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-16)
    assert np.allclose(mo, st["exp_avg"].numpy(), rtol=1e-13, atol=1e-20)
    assert np.allclose(vo, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=1e-24)


def test_adam_first_step_closed_form():
    # from zero moments the bias-corrected step is lr * g / (|g| + eps)
    g = np.array([3.0, -0.25, 1e-9, 0.0])
    val = np.array([1.0, 2.0, 3.0, 4.0], np.float32)
    z = np.zeros(4, np.float32)
    got, m, v = oracle.adam_update(val, g, z, z, 0.01, 0.9, 0.999, 1e-8, 0.0, 1)
    assert np.allclose(got, val - 0.01 * g / (np.abs(g) + 1e-8), rtol=1e-15, atol=0)
    assert np.allclose(m, 0.1 * g) and np.allclose(v, 0.001 * g * g)


# ------------------------------------------------------------ all-cores copy

@pytest.mark.parametrize("shape,sp,B", [((300, 200), 90, 5), ((64, 3000), 99, 1),
                                        ((2000, 1500), 97, 17)])
def test_omp_copy_is_bit_identical_to_the_oracle(shape, sp, B):
    # The CPU baseline's all-cores copy of the three product loops must give
    # the single-threaded oracle's bits (same terms, same order per output),
    # whatever the thread count.
    import workloads
    out, inp = shape
    nnz = workloads.nnz_for(out, inp, sp)
    row, col = workloads.uniform_pattern(out, inp, nnz, sp)
    val = workloads.normal(nnz, 0.1, sp, 0)
    ref = oracle.canonicalize(out, inp, row, col, val)
    g = np.random.default_rng(sp + B)
    X = g.standard_normal((B, inp)).astype(np.float32)
    dY = g.standard_normal((B, out)).astype(np.float32)
    want = (oracle.forward(out, inp, ref["row"], ref["col"], ref["val"], X),
            oracle.backward_input(out, inp, ref["row"], ref["col"], ref["val"], dY),
            oracle.backward_weight(out, inp, ref["row"], ref["col"], X, dY))
    for threads in (1, 3, oracle.host_cores()):
        got = (oracle.forward_omp(out, inp, ref, X, threads),
               oracle.backward_input_omp(out, inp, ref, dY, threads),
               oracle.backward_weight_omp(out, inp, ref, X, dY, threads))
        for (a, sa), (b, sb) in zip(got, want):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
            assert np.array_equal(sa, sb)
