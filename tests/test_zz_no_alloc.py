"""The allocation-free entry point, wq_matmul_add_rmsnorm_noalloc (GPU).

It exists for callers that cannot allocate device memory or pass a workspace
(frameworks whose custom-op interface hands over only inputs and outputs,
runtimes that forbid allocations after start-up); its scratch is a fixed array
inside the library. It runs the same deterministic kernels as the workspace
entry point, so its outputs must equal that entry point's bit for bit, and
match the oracle, on calls in a row that share the array: two decode-kernel
problems and then a prefill-kernel problem, whose larger scratch layout lands
on the array the decode calls left dirty. This file is named so that pytest
collects it last.
"""
import ctypes

import pytest
import torch

from weight_only_bit_pack_b300 import inputs
from parity_util import compare, gpu_weight, run_oracle, sample_rows, to_device

pytestmark = pytest.mark.gpu

DEVICE_TIMEOUT = 8  # WQ_ERR_DEVICE_TIMEOUT


def _problems():
    prefill = inputs.make_problem(M_shape=(256,), K=4096, N=4096, dtype=torch.bfloat16, wbits=4,
                                  mode="group", group=128, offset=True, seed=41, device="cuda",
                                  name="noalloc_prefill_256x4096x4096")
    return [inputs.decode("cuda"), to_device(inputs.tiny()), prefill]


def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row(wq):
    probs = _problems()
    weights = [gpu_weight(wq, p) for p in probs]
    kernels = [int(wq.select_kernel(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma,
                                    p.eps, p.group)) for p, w in zip(probs, weights)]
    assert kernels == [wq.Kernel.DECODE, wq.Kernel.DECODE, wq.Kernel.PREFILL]
    for p, w in zip(probs, weights):
        need = wq.matmul_add_rmsnorm_get_workspace(p.x1, w, p.scale, p.offset, p.bias,
                                                   p.residual, p.gamma, p.eps, p.group)
        assert need <= wq.NOALLOC_SCRATCH_BYTES, (p.name, need)
    refs = [wq.matmul_add_rmsnorm(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma,
                                  p.eps, p.group) for p, w in zip(probs, weights)]
    torch.cuda.synchronize()
    outs = []
    for p, w in zip(probs, weights):  # calls in a row on the same static scratch
        outs.append(wq.matmul_add_rmsnorm_noalloc(p.x1, w, p.scale, p.offset, p.bias,
                                                  p.residual, p.gamma, p.eps, p.group))
        assert wq.noalloc_read_device_status() == 0, p.name
    torch.cuda.synchronize()
    for p, (yr, nr), (y, n) in zip(probs, refs, outs):
        assert torch.equal(y, yr) and torch.equal(n, nr), p.name
        rows = sample_rows(p.M, 64)
        compare(p, y, n, run_oracle(p, rows), rows)


def test_noalloc_device_status_is_observable(wq):
    """A bounded device wait of a no-alloc call that runs out (test hook: one more
    arrival than the kernel makes, ~1 ms budget) shows in the array's status word;
    the next no-alloc call clears it and computes correctly."""
    p = inputs.decode("cuda")
    w = gpu_weight(wq, p)
    wq.set_wait_limits_for_testing(2_000_000, 1)
    try:
        wq.matmul_add_rmsnorm_noalloc(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma,
                                      p.eps, p.group)
        st = wq.noalloc_read_device_status()
    finally:
        wq.set_wait_limits_for_testing(0, 0)
    assert st & 0xFF == DEVICE_TIMEOUT and st >> 8 == wq.WHERE_DECODE_GRID, hex(st)
    y, n = wq.matmul_add_rmsnorm_noalloc(p.x1, w, p.scale, p.offset, p.bias, p.residual,
                                         p.gamma, p.eps, p.group)
    assert wq.noalloc_read_device_status() == 0
    compare(p, y, n, run_oracle(p))


def test_noalloc_rejects_problems_larger_than_its_scratch(wq):
    """Descriptors with placeholder addresses: the call must be refused on the
    host (WQ_ERR_WORKSPACE) before anything is enqueued. The placeholders never
    reach a kernel because the first phase is checked to ask for more than the
    array holds before the entry point is called."""
    from weight_only_bit_pack_b300 import binding as B
    M, K, N = 1 << 20, 4096, 4096
    base = [0x10_0000_0000]

    def d(dt, shape):
        t = B.WqTensor()
        t.data = base[0]
        base[0] += 1 << 36
        t.dtype = int(dt); t.ndim = len(shape)
        for i, v in enumerate(shape):
            t.shape[i] = v
        return t

    args = [d(B.DType.BF16, (M, K)), d(B.DType.INT4, (K, N)), d(B.DType.BF16, (N,)), None, None,
            d(B.DType.BF16, (M, N)), d(B.DType.BF16, (N,))]
    y, no = d(B.DType.BF16, (M, N)), d(B.DType.BF16, (M, N))
    r = lambda t: None if t is None else ctypes.byref(t)
    need = ctypes.c_uint64(0)
    assert B.lib.wq_matmul_add_rmsnorm_get_workspace(*[r(a) for a in args], 1e-6, 0, r(y), r(no),
                                                     ctypes.byref(need)) == 0
    assert need.value > B.NOALLOC_SCRATCH_BYTES, need.value  # else stop: no launch on placeholders
    st = B.lib.wq_matmul_add_rmsnorm_noalloc(*[r(a) for a in args], 1e-6, 0, r(y), r(no), None)
    assert st == B.Status.ERR_WORKSPACE
    assert b"static scratch" in B.lib.wq_last_error()
