"""Memory headroom (SNACK §4.4, Figure 4): a sparse layer's device footprint
follows its nonzeros, never the dense out x in matrix."""

import pytest
import torch

import workloads
from parity_util import sn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sparsity", [90, 99])
def test_handle_bytes_follow_nnz(sparsity):
    m = sn()
    out, inp = 10000, 15000
    nnz = workloads.nnz_for(out, inp, sparsity)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    h, _ = m.snack_create_random(out, inp, nnz, 3)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    acct = m.snack_device_bytes(h)
    # indices, values in both orders and both layouts: 24 B per stored
    # entry, plus per line an offset, a segment record and a 256-float row of
    # operand workspace, and on a large layer of long lines its copies cut
    # in 2 and 4 parts (6 segment records and 2 split records per line, the
    # quarters' partial sums of 64 floats each, two tickets)
    per_line = 4 + 16 + 256 * 4 + 6 * 16 + 2 * 16 + 4 * 64 * 4 + 2 * 4
    assert 24 * nnz <= acct <= 25 * nnz + per_line * (out + inp) + (1 << 20)
    # what the device really gave up (allocation granularity included)
    assert free0 - free1 <= acct + (64 << 20)
    # against the dense W alone (4 B per cell): ~0.6x at 90 %, ~0.1x at 99 %
    dense = 4 * out * inp
    assert acct < {90: 0.7, 99: 0.12}[sparsity] * dense
    del h
