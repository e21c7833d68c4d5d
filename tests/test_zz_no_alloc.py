"""The allocation-free entry point, wq_matmul_add_rmsnorm_noalloc (GPU).

It exists for callers that cannot allocate device memory or pass a workspace
(frameworks whose custom-op interface hands over only inputs and outputs,
runtimes that forbid allocations after start-up); its scratch is a fixed array
inside the library. Its output must match the workspace entry point's within
the parity tolerance, on two calls in a row that share that array. This file is
named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from weight_only_bit_pack_b300 import inputs
from parity_util import TOL, gpu_weight, to_device

pytestmark = pytest.mark.gpu


def _close(a, b, tol):
    a = a.double(); b = b.double()
    return bool(((a - b).abs() <= tol * (1.0 + b.abs())).all())


def test_noalloc_matches_workspace_entry_point_on_two_calls(wq):
    probs = [inputs.decode("cuda"), to_device(inputs.tiny())]
    weights = [gpu_weight(wq, p) for p in probs]
    refs = []
    for p, w in zip(probs, weights):
        refs.append(wq.matmul_add_rmsnorm(p.x1, w, p.scale, p.offset, p.bias, p.residual,
                                          p.gamma, p.eps, p.group))
    torch.cuda.synchronize()
    outs = []
    for p, w in zip(probs, weights):  # two calls in a row on the same static scratch
        outs.append(wq.matmul_add_rmsnorm_noalloc(p.x1, w, p.scale, p.offset, p.bias,
                                                  p.residual, p.gamma, p.eps, p.group))
    torch.cuda.synchronize()
    for p, (yr, nr), (y, n) in zip(probs, refs, outs):
        tol = TOL[p.dtype]
        assert _close(y, yr, tol), p.name
        assert _close(n, nr, tol), p.name


def test_noalloc_rejects_problems_larger_than_its_scratch(wq):
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
    st = B.lib.wq_matmul_add_rmsnorm_noalloc(*[r(a) for a in args], 1e-6, 0, r(y), r(no), None)
    assert st == B.Status.ERR_WORKSPACE
    assert b"static scratch" in B.lib.wq_last_error()
