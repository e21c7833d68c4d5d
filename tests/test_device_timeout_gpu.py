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


GENERIC, DECODE, PREFILL = 1, 2, 3

OPERATOR_CASES = [
    # name, problem, kernel, place that must give up
    ("decode_grid", lambda: inputs.decode("cuda"), DECODE, 15),
    ("prefill_f16emu_row_block",
     lambda: inputs.make_problem(M_shape=(600,), K=512, N=1024, dtype=torch.bfloat16, wbits=4,
                                 mode="group", group=64, seed=21, device="cuda"), PREFILL, 5),
    ("prefill_rawq_row_block",
     lambda: inputs.make_problem(M_shape=(300,), K=256, N=768, dtype=torch.float16, wbits=8,
                                 mode="channel", seed=22, device="cuda"), PREFILL, 5),
]


@pytest.mark.parametrize("name,make,kernel,where", OPERATOR_CASES,
                         ids=[c[0] for c in OPERATOR_CASES])
def test_operator_wait_gives_up_and_context_stays_usable(wq, name, make, kernel, where):
    """An operator kernel whose wait for other thread blocks cannot complete (the
    test hook asks for one arrival more than the kernel makes, with a ~1 ms budget)
    must record WQ_ERR_DEVICE_TIMEOUT with its place, drain and exit; the same
    context and workspace, header zeroed, then serve a correct call."""
    p = make()
    w = wq.pack_int4(p.x2) if p.wbits == 4 else p.x2
    ws_bytes = wq.matmul_add_rmsnorm_get_workspace(p.x1, w, p.scale, p.offset, p.bias,
                                                   p.residual, p.gamma, p.eps, p.group,
                                                   kernel=kernel)
    ws = torch.zeros(max(ws_bytes, 2048), dtype=torch.uint8, device="cuda")
    wq.set_wait_limits_for_testing(2_000_000, 1)
    try:
        wq.matmul_add_rmsnorm(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma, p.eps,
                              p.group, workspace=ws, kernel=kernel)
        st = wq.read_device_status(ws)
    finally:
        wq.set_wait_limits_for_testing(0, 0)
    assert st & 0xFF == DEVICE_TIMEOUT, hex(st)
    assert st >> 8 == where, hex(st)

    ws[:2048].zero_()
    y, no = wq.matmul_add_rmsnorm(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma,
                                  p.eps, p.group, workspace=ws, kernel=kernel, check_status=True)
    torch.cuda.synchronize()
    rows = [0, 1, p.M // 2, p.M - 1]
    compare(p, y, no, run_oracle(p, rows), rows)


def test_binding_check_status_raises_and_rearms_the_workspace(wq):
    from weight_only_bit_pack_b300.binding import Status, WQError
    p = inputs.decode("cuda")
    w = wq.pack_int4(p.x2)
    ws = torch.zeros(16 << 20, dtype=torch.uint8, device="cuda")
    wq.set_wait_limits_for_testing(2_000_000, 1)
    try:
        with pytest.raises(WQError) as ei:
            wq.matmul_add_rmsnorm(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma,
                                  p.eps, p.group, workspace=ws, check_status=True)
    finally:
        wq.set_wait_limits_for_testing(0, 0)
    assert ei.value.status == Status.ERR_DEVICE_TIMEOUT
    assert int(ws[:2048].abs().sum()) == 0  # the binding zeroed the header again
    y, no = wq.matmul_add_rmsnorm(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma,
                                  p.eps, p.group, workspace=ws, check_status=True)
    torch.cuda.synchronize()
    compare(p, y, no, run_oracle(p))
