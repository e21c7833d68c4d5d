"""Failure detection on the GPU without a fault: a bounded device wait runs out.

The self-check kernel waits, with the bounded wait every operator kernel uses,
for an mbarrier phase that nothing completes. The wait must give up after its
budget, record WQ_ERR_DEVICE_TIMEOUT and the place in the workspace status
word, and leave the CUDA context usable: the same workspace, zeroed again,
then serves an operator call whose result matches the oracle.
"""
import pytest
import torch

from parity_util import compare, run_oracle
from weight_only_bit_pack_b300 import inputs

pytestmark = pytest.mark.gpu

DEVICE_TIMEOUT = 8  # WQ_ERR_DEVICE_TIMEOUT


def test_bounded_wait_gives_up_and_context_stays_usable(wq):
    ws = torch.zeros(16 << 20, dtype=torch.uint8, device="cuda")
    wq.check_device_timeout(ws, budget_cycles=2_000_000)  # about a millisecond
    st = wq.read_device_status(ws)
    assert st & 0xFF == DEVICE_TIMEOUT
    assert (st >> 8) == wq.WHERE_SELF_CHECK
    torch.cuda.synchronize()

    ws.zero_()  # the header must be zero again before the next operator call
    p = inputs.decode("cuda")
    w = wq.pack_int4(p.x2)
    y = torch.empty_like(p.residual)
    no = torch.empty_like(p.residual)
    wq.matmul_add_rmsnorm(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma, p.eps, p.group,
                          y=y, normOut=no, workspace=ws)
    assert wq.read_device_status(ws) == 0
    rows = [0, 3, 7]
    ref = run_oracle(p, rows)
    compare(p, y, no, ref, rows)
