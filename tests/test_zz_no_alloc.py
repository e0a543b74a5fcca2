"""snack_forward_csr_static: the forward pass for callers that cannot
allocate device memory when they run the layer (code inside a CUDA graph
capture in global mode, serving loops whose device memory is reserved by
another allocator, latency-critical paths that cannot take an allocation's
device synchronisation).  It runs from caller-held CSR arrays and the
library's fixed device scratch.

Checked through the C ABI against snack_forward on the same layer and
inputs, twice in a row (the shared scratch keeps the previous call's
contents), within the parity tolerance of the other tests (1e-5 times the
sum of |terms| from the CPU oracle).  This file is collected last so that a
run stopping at the first failure has run every other test already; it also
passes when run alone in a fresh process."""

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
def test_static_scratch_forward_matches_snack_forward(name, idx, batches):
    import coo_spmm_sparse_gb300 as sn
    L = workloads.workload(name).layers[idx]
    row, col, val = L.coo()
    ref = canonical(L.out, L.inp, row, col, val)
    h = sn.snack_create(L.out, L.inp, row, col, val)
    row_ptr, dcol, dval = _csr_on_device(h)
    for B in batches:
        X, _ = L.activations(B)
        Xd = to_dev(X)
        want = sn.snack_forward(h, Xd)
        _, S = oracle.forward(L.out, L.inp, ref["row"], ref["col"], ref["val"], X)
        for call in range(2):  # two calls in a row share the scratch
            got = sn.snack_forward_csr_static(L.out, L.inp, row_ptr, dcol, dval, Xd)
            torch.cuda.synchronize()
            assert_close(f"{name} B={B} call {call}", got, want.cpu().numpy(), S)


def test_static_scratch_rejects_oversized_slice():
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
