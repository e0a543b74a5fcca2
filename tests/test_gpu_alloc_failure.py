"""Out-of-memory paths, driven by the library's allocation hook
(snack_debug_fail_alloc) instead of exhausting the device.

Every device allocation a layer creation makes is failed once in turn: each
failure returns SNACK_ERR_ALLOC and frees what the call had allocated (no
memory is lost over many failed creations), and the next creation works.
An optimizer step whose state or gradient buffer cannot be allocated, and a
prune/regrow that fails at any of its allocations, leave the handle as it
was: same topology, values and state, same products."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import canonical, check_products, check_topology, dev, sn

pytestmark = pytest.mark.gpu

SNACK_ERR_ALLOC = 4


def _fail_at(after, call):
    """Run `call` with the after-th next allocation failing; returns the
    SnackError it raised (None if it needed fewer allocations)."""
    m = sn()
    m.snack_debug_fail_alloc(after)
    try:
        call()
    except m.SnackError as e:
        return e
    finally:
        m.snack_debug_fail_alloc(-1)
    return None


def _allocation_points(call, limit=400):
    """Fail each allocation of `call` in turn until it succeeds; returns the
    number of allocation points (every failure must be SNACK_ERR_ALLOC)."""
    for after in range(limit):
        e = _fail_at(after, call)
        if e is None:
            return after
        assert e.status == SNACK_ERR_ALLOC, e
    pytest.fail(f"still failing after {limit} allocation points")


def test_create_fails_cleanly_at_every_allocation():
    m = sn()
    L = workloads.Layer("alloc", 900, 700, 95, seed=5)
    row, col, val = L.coo()
    made = []
    points = _allocation_points(lambda: made.append(m.snack_create(L.out, L.inp, row, col, val)))
    assert points >= 10 and len(made) == 1
    h = made[0]
    ref = canonical(L.out, L.inp, row, col, val)
    check_topology(h, ref)
    g = np.random.default_rng(1)
    X = g.standard_normal((8, L.inp)).astype(np.float32)
    dY = g.standard_normal((8, L.out)).astype(np.float32)
    check_products(h, L.out, L.inp, ref, X, dY)
    # and from device pointers, and the device initializer
    points_random = _allocation_points(lambda: m.snack_create_random(L.out, L.inp, L.nnz, 3))
    assert points_random >= 10


def test_failed_creations_leak_nothing():
    m = sn()
    L = workloads.Layer("alloc_big", 4000, 4000, 90, seed=6)   # 1.6 M entries, ~6.4 MB per array
    row, col, val = L.coo()
    create = lambda: m.snack_create(L.out, L.inp, row, col, val)
    points = _allocation_points(lambda: m.snack_destroy(create()))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(4):
        for after in range(points):
            e = _fail_at(after, create)
            assert e is not None and e.status == SNACK_ERR_ALLOC
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    # a leaked entry-sized array at any point would lose >= 4 x 6.4 MB
    assert free0 - free1 < 16 * 2**20, (free0, free1)


@pytest.mark.parametrize("B", [3, 16])   # fused step; gradient buffer + streaming update
def test_optimizer_allocation_failure_leaves_handle(B):
    m = sn()
    L = workloads.Layer("alloc_opt", 1500, 1200, 95, seed=7)
    row, col, val = L.coo()
    h = m.snack_create(L.out, L.inp, row, col, val)
    X = torch.randn(B, L.inp, device=dev())
    dY = torch.randn(B, L.out, device=dev())
    torch.cuda.synchronize()
    r0, c0, v0 = m.snack_export(h)
    bytes0 = m.snack_device_bytes(h)
    points = 0
    for after in range(8):
        e = _fail_at(after, lambda: m.snack_adam_step(h, X, dY, lr=1e-3, step=1))
        if e is None:
            break
        assert e.status == SNACK_ERR_ALLOC, e
        points += 1
        r, c, v = m.snack_export(h)
        assert np.array_equal(r, r0) and np.array_equal(c, c0)
        assert np.array_equal(v.view(np.uint32), v0.view(np.uint32))
        assert m.snack_device_bytes(h) == bytes0     # nothing kept from the failed call
    # two moments (and the gradient buffer from batch 5 on) before any launch
    assert points == (2 if B <= 4 else 3)
    # the step that finally ran is the first Adam step from zero state
    torch.cuda.synchronize()
    v1 = m.snack_export(h)[2]
    assert not np.array_equal(v1, v0)
    assert np.all(np.abs(v1 - v0) <= 1.0e-3 * 1.0001 + 1e-7)    # |first Adam update| <= lr
    ref = canonical(L.out, L.inp, r0, c0, v1)
    g = np.random.default_rng(2)
    check_products(h, L.out, L.inp, ref, g.standard_normal((4, L.inp)).astype(np.float32),
                   g.standard_normal((4, L.out)).astype(np.float32))
    assert m.snack_device_error(h) == 0


def test_prune_regrow_allocation_failure_leaves_handle():
    m = sn()
    L = workloads.Layer("alloc_prune", 1200, 1000, 95, seed=8)
    row, col, val = L.coo()
    h = m.snack_create(L.out, L.inp, row, col, val)
    X = torch.randn(16, L.inp, device=dev())
    dY = torch.randn(16, L.out, device=dev())
    m.snack_adam_step(h, X, dY, lr=1e-3, step=1)          # state to carry
    torch.cuda.synchronize()
    r0, c0, v0 = m.snack_export(h)
    m0 = m.snack_optimizer_state(h, 0).cpu().numpy().copy()
    ref0 = canonical(L.out, L.inp, r0, c0, v0)
    seed = 1234
    failures = 0
    for after in range(400):
        e = _fail_at(after, lambda: m.snack_prune_regrow(h, 0.3, seed))
        if e is None:
            break
        assert e.status == SNACK_ERR_ALLOC, e
        failures += 1
        check_topology(h, ref0)
        assert np.array_equal(m.snack_optimizer_state(h, 0).cpu().numpy(), m0)
    else:
        pytest.fail("prune/regrow still failing")
    assert failures >= 10
    # the call that went through is the oracle's prune/regrow of the same layer
    o = oracle.prune_regrow(L.out, L.inp, r0, c0, v0, 0.3, seed)
    check_topology(h, canonical(L.out, L.inp, o["row"], o["col"], o["val"]))
    g = np.random.default_rng(3)
    ref = canonical(L.out, L.inp, o["row"], o["col"], o["val"])
    check_products(h, L.out, L.inp, ref, g.standard_normal((8, L.inp)).astype(np.float32),
                   g.standard_normal((8, L.out)).astype(np.float32))
    assert m.snack_device_error(h) == 0
