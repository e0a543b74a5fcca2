"""snack_forward_csr_static: the forward pass for callers that cannot
allocate device memory when they run the layer (serving loops whose device
memory a pool reserved up front, latency-critical paths that cannot take an
allocation's device synchronisation, plug-ins inside a host framework that
owns all allocation).  It runs from caller-held CSR arrays and the library's
fixed device scratch.

Checked through the C ABI against the CPU oracle's Y element by element,
within the tolerance of the other parity tests (1e-5 times the oracle's sum
of |terms|), on two calls in a row (the shared scratch keeps the previous
call's contents); the regular entry point snack_forward is compared on the
same inputs.  That the call allocates nothing is checked twice: with the
library's allocation-failure hook armed for the very next allocation, the
call still succeeds and the hook is still armed afterwards (the next
allocating call meets it), and the device's free memory is unchanged.  This
file is collected last so that a run stopping at the first failure has run
every other test already; it also passes when run alone in a fresh
process."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import assert_close, canonical, to_dev

pytestmark = pytest.mark.gpu


def _csr_on_device(h):
    import coo_spmm_sparse_gb300 as sn
    seg = sn.snack_export_segments(h)
    _, col, val = sn.snack_export(h)
    return (to_dev(seg["row_ptr"]), to_dev(col), to_dev(val))


@pytest.mark.parametrize("name,idx,batches", [
    ("toy256", 0, [4, 1, 7]),
    ("gpt2_mlp", 0, [8, 32]),
    ("gpt2_mlp", 1, [1, 33]),
    ("skewed", 0, [16]),
    ("large99", 0, [64, 70]),
])
def test_static_scratch_forward_matches_oracle(name, idx, batches):
    import coo_spmm_sparse_gb300 as sn
    L = workloads.workload(name).layers[idx]
    row, col, val = L.coo()
    ref = canonical(L.out, L.inp, row, col, val)
    h = sn.snack_create(L.out, L.inp, row, col, val)
    row_ptr, dcol, dval = _csr_on_device(h)
    for B in batches:
        X, _ = L.activations(B)
        Xd = to_dev(X)
        Yo, S = oracle.forward(L.out, L.inp, ref["row"], ref["col"], ref["val"], X)
        want = sn.snack_forward(h, Xd)
        torch.cuda.synchronize()
        assert_close(f"{name} B={B} snack_forward", want, Yo, S)
        Y = torch.full((B, L.out), float("nan"), device=Xd.device)
        for call in range(2):  # two calls in a row share the scratch
            got = sn.snack_forward_csr_static(L.out, L.inp, row_ptr, dcol, dval, Xd, Y)
            torch.cuda.synchronize()
            assert_close(f"{name} B={B} call {call}", got, Yo, S)


def test_static_scratch_call_allocates_nothing():
    import coo_spmm_sparse_gb300 as sn
    L = workloads.workload("gpt2_mlp").layers[0]
    row, col, val = L.coo()
    ref = canonical(L.out, L.inp, row, col, val)
    h = sn.snack_create(L.out, L.inp, row, col, val)
    row_ptr, dcol, dval = _csr_on_device(h)
    X, _ = L.activations(8)
    Xd = to_dev(X)
    Y = torch.empty((8, L.out), device=Xd.device)
    # first call on this device: the scratch address is looked up
    sn.snack_forward_csr_static(L.out, L.inp, row_ptr, dcol, dval, Xd, Y)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    sn.snack_debug_fail_alloc(0)  # the library's next device allocation fails
    try:
        for _ in range(2):
            sn.snack_forward_csr_static(L.out, L.inp, row_ptr, dcol, dval, Xd, Y)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        # the hook is still armed: the next allocating call meets it
        with pytest.raises(sn.SnackError) as e:
            sn.snack_create(L.out, L.inp, row, col, val)
        assert e.value.status == 4  # SNACK_ERR_ALLOC
    finally:
        sn.snack_debug_fail_alloc(-1)
    assert free1 == free0
    Yo, S = oracle.forward(L.out, L.inp, ref["row"], ref["col"], ref["val"], X)
    assert_close("Y after the guarded calls", Y, Yo, S)


def test_static_scratch_rejects_oversized_slice_and_overlap():
    import coo_spmm_sparse_gb300 as sn
    inp, out = 40000, 8        # 40000 x 64 > 2^21 floats of scratch
    row_ptr = torch.zeros(out + 1, dtype=torch.int32, device="cuda")
    col = torch.zeros(4, dtype=torch.int32, device="cuda")
    val = torch.zeros(4, dtype=torch.float32, device="cuda")
    X = torch.zeros(64, inp, device="cuda")
    with pytest.raises(sn.SnackError) as e:
        sn.snack_forward_csr_static(out, inp, row_ptr, col[:0], val[:0], X)
    assert e.value.status == 6 and "static scratch" in str(e.value)
    # batch 1 needs no scratch and runs: an all-empty layer gives zeros
    Y = sn.snack_forward_csr_static(out, inp, row_ptr, col[:0], val[:0], X[:1].contiguous())
    torch.cuda.synchronize()
    assert torch.all(Y == 0)
    # Y overlapping X is refused
    buf = torch.zeros(2 * inp, device="cuda")
    with pytest.raises(sn.SnackError) as e:
        sn.snack_forward_csr_static(out, inp, row_ptr, col[:0], val[:0], buf[:inp].view(1, inp),
                                    buf[4:4 + out].view(1, out))
    assert e.value.status == 1 and "overlaps" in str(e.value)
