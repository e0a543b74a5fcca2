"""GPU parity of the optimizer step (SGD / Adam on the stored entries; the
weight gradient is computed inside the step's kernel for batches of 1-4 and
through the handle's gradient buffer for larger ones, both covered here).

Each step is checked on its own against the oracle: the oracle takes the
GPU's values and state before the step (read back) and the float64 gradient
of the same inputs.  Tolerance: the GPU's gradient may differ from the
oracle's by the parity bound delta = 1e-5 * sum|terms| (plus a few ulp of
the weight-decay term), so the oracle is evaluated across g - delta ..
g + delta and the GPU result must lie in that range, widened by 1e-6 of the
magnitudes entering the float32 update (a handful of roundings)."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import canonical, dev, sn, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _f32(*xs):
    """Hyper-parameters as the C ABI receives them (float32), for the oracle."""
    return [float(np.float32(x)) for x in xs]


def _hull(fn, g, delta):
    """Elementwise min / max of fn(g + t * delta) over t in [-1, 1]; fn returns
    a tuple of arrays."""
    outs = [fn(g + t * delta) for t in (-1.0, -0.5, 0.0, 0.5, 1.0)]
    lo = [np.min(np.stack(o), axis=0) for o in zip(*outs)]
    hi = [np.max(np.stack(o), axis=0) for o in zip(*outs)]
    return lo, hi


def _within(name, got, lo, hi, scale):
    got = np.asarray(got, np.float64)
    slack = 1e-6 * scale + 1e-30
    bad = (got < lo - slack) | (got > hi + slack)
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{name}: {int(bad.sum())} outside; first at {i}: gpu={got[i]!r} "
                             f"oracle range=[{lo[i]!r}, {hi[i]!r}] slack={slack[i]!r}")


class Case:
    def __init__(self, out, inp, row, col, val, seed):
        self.out, self.inp = out, inp
        self.ref = canonical(out, inp, row, col, val)
        self.h = sn().snack_create(out, inp, row, col, val)
        self.g = np.random.default_rng(seed)

    def batch(self, B):
        X = self.g.standard_normal((B, self.inp)).astype(np.float32)
        dY = self.g.standard_normal((B, self.out)).astype(np.float32)
        g, S = oracle.weight_gradient64(self.out, self.inp, self.ref["row"], self.ref["col"],
                                        X, dY)
        return X, dY, g, S

    def values(self):
        # read-only copy (a snack_values() view would hand out a writable
        # pointer and stop the handle's column-ordered value copy)
        torch.cuda.synchronize()
        return sn().snack_export(self.h)[2]

    def check_dx(self, B):
        # after optimizer steps dX reads the values through the column permutation
        # (their column-ordered copy is stale); after snack_values_changed()
        # it streams the re-derived copy
        dY = self.g.standard_normal((B, self.out)).astype(np.float32)
        r = self.ref
        want, S = oracle.backward_input(self.out, self.inp, r["row"], r["col"], self.values(), dY)
        for refresh in (False, True):
            if refresh:
                sn().snack_values_changed(self.h)
            dX = sn().snack_backward_input(self.h, to_dev(dY))
            torch.cuda.synchronize()
            got = dX.cpu().numpy().astype(np.float64)
            assert np.all(np.abs(got - want) <= TOL * S + 1e-30), refresh

    def state(self, which):
        try:
            return sn().snack_optimizer_state(self.h, which).cpu().numpy().copy()
        except sn().SnackError:
            return np.zeros(self.ref["row"].size, np.float32)

    def sgd(self, B, lr, mom, wd):
        lr, mom, wd = _f32(lr, mom, wd)
        X, dY, g, S = self.batch(B)
        w0, b0 = self.values(), self.state(0)
        sn().snack_sgd_step(self.h, to_dev(X), to_dev(dY), lr, mom, wd)
        w1 = self.values()
        delta = TOL * S + 1e-6 * np.abs(wd * w0.astype(np.float64))

        def fn(gg):
            v, b = oracle.sgd_update(w0, gg, b0, lr, mom, wd)
            return (v,) if b is None else (v, b)
        lo, hi = _hull(fn, g, delta)
        d = np.abs(g) + S + np.abs(wd * w0) + (mom * np.abs(b0) if mom else 0)
        _within("val", w1, lo[0], hi[0], np.abs(w0) + lr * d)
        if mom:
            _within("momentum", self.state(0), lo[1], hi[1], mom * np.abs(b0) + d)

    def adam(self, B, t, lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=0.0, fresh=False):
        lr, b1, b2, eps, wd = _f32(lr, b1, b2, eps, wd)
        X, dY, g, S = self.batch(B)
        w0, m0, v0 = self.values(), self.state(0), self.state(1)
        if fresh:                      # state of another optimizer kind is zeroed first
            m0, v0 = np.zeros_like(m0), np.zeros_like(v0)
        sn().snack_adam_step(self.h, to_dev(X), to_dev(dY), lr, (b1, b2), eps, wd, t)
        w1, m1, v1 = self.values(), self.state(0), self.state(1)
        delta = TOL * S + 1e-6 * np.abs(wd * w0.astype(np.float64))
        lo, hi = _hull(lambda gg: oracle.adam_update(w0, gg, m0, v0, lr, b1, b2, eps, wd, t),
                       g, delta)
        step = np.abs(hi[0] - w0) + np.abs(lo[0] - w0)
        _within("val", w1, lo[0], hi[0], np.abs(w0) + step)
        d = np.abs(g) + S + np.abs(wd * w0)
        _within("m", m1, lo[1], hi[1], b1 * np.abs(m0) + (1 - b1) * d)
        _within("v", v1, lo[2], hi[2], b2 * np.abs(v0) + (1 - b2) * d * d)


def _uniform_case(out, inp, sparsity, seed):
    nnz = workloads.nnz_for(out, inp, sparsity)
    row, col = workloads.uniform_pattern(out, inp, nnz, seed)
    val = workloads.normal(nnz, 0.05, seed, 0)
    return Case(out, inp, row, col, val, seed + 1)


@pytest.mark.parametrize("B", [1, 4, 16, 130, 300])
def test_sgd_plain_and_momentum(B):
    c = _uniform_case(256, 256, 90, 30)
    c.sgd(B, 0.05, 0.0, 0.0)
    for _ in range(3):
        c.sgd(B, 0.05, 0.9, 1e-3)
    c.check_dx(B)
    assert sn().snack_device_error(c.h) == 0


@pytest.mark.parametrize("shape,B", [((256, 256, 90), 4), ((3072, 768, 95), 1),
                                     ((3072, 768, 95), 8), ((768, 3072, 95), 32),
                                     ((3000, 3000, 85), 64), ((700, 900, 80), 130),
                                     ((700, 900, 80), 300),
                                     # 2.3 M entries, 960 per line: the gradient of
                                     # 64- and 128-wide slices over lines cut in four
                                     ((2400, 2400, 60), 64), ((2400, 2400, 60), 130)])
def test_adam_steps(shape, B):
    c = _uniform_case(*shape, 31)
    for t in (1, 2, 3):
        c.adam(B, t, wd=1e-4 if t == 3 else 0.0)
    c.check_dx(min(B, 64))
    assert sn().snack_device_error(c.h) == 0


def test_optimizer_kind_switch_zeroes_state():
    c = _uniform_case(256, 256, 90, 32)
    c.sgd(8, 0.1, 0.9, 0.0)
    assert np.any(c.state(0) != 0)
    c.adam(8, 1, fresh=True)          # Adam starts from zero moments


def test_state_follows_entries_through_prune_regrow():
    c = _uniform_case(300, 200, 90, 33)
    for t in (1, 2):
        c.adam(16, t)
    r0, c0, _ = sn().snack_export(c.h)
    m0, v0 = c.state(0), c.state(1)
    before = {(int(r), int(q)): (a, b) for r, q, a, b in zip(r0, c0, m0, v0)}
    pruned, _ = sn().snack_prune_regrow(c.h, 0.3, 77)
    assert pruned == int(0.3 * r0.size)
    r1, c1, _ = sn().snack_export(c.h)
    m1, v1 = c.state(0), c.state(1)
    regrown = 0
    for r, q, a, b in zip(r1, c1, m1, v1):
        key = (int(r), int(q))
        if key in before and (a, b) == before[key]:
            continue
        assert a == 0.0 and b == 0.0, key      # a regrown entry starts from zero state
        regrown += 1
    assert regrown >= 1
    # and the next step runs on the new layout
    c.ref = canonical(c.out, c.inp, r1, c1, c.values())
    c.adam(16, 3)
    c.check_dx(16)


def test_invalid_optimizer_arguments():
    m = sn()
    c = _uniform_case(64, 64, 90, 34)
    X = torch.zeros(2, 64, device=dev())
    dY = torch.zeros(2, 64, device=dev())
    for kw in (dict(lr=float("nan")), dict(lr=0.1, momentum=-1.0)):
        with pytest.raises(m.SnackError) as e:
            m.snack_sgd_step(c.h, X, dY, **kw)
        assert e.value.status == 1
    for kw in (dict(step=0), dict(betas=(1.0, 0.999)), dict(eps=0.0)):
        with pytest.raises(m.SnackError) as e:
            m.snack_adam_step(c.h, X, dY, **kw)
        assert e.value.status == 1
    with pytest.raises(m.SnackError):
        m.snack_optimizer_state(c.h, 1)       # no Adam state yet
