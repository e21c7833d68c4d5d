"""Parity over the whole range of the inputs (GPU): rows far from unit scale,
per-group scales that span many binades within one column, and rows holding
NaN, Inf or nothing but zeros.

The operator's inputs are fp16/bf16 over their whole range (the weight-quant
matmul page's constraints name dtypes, not magnitudes). These cases reach the
exponent handling that the N(0, 1) workloads never touch: the prefill kernel's
fp16-operand mode scales every row of x1 by a power of two that puts its
maximum in [2^13, 2^14) and every scale column by another; the decode and
generic kernels take the values as they are.

Rows scaled by 2^s (no bias) have y exactly 2^s times the unscaled row's y,
and the stated tolerance |d| <= tol * (1 + |ref|) is read on the unscaled
values: y of those rows is compared after multiplying both sides by 2^-s. (On
the raw values its absolute floor would be unreachable for 2^15-scale rows even
for exact weights: fp32 accumulation of K terms of that size errs by more than
1e-2 where the sum cancels to about 1.) normOut does not depend on the row's
scale, so it is compared as it is for every row.
"""
import zlib

import numpy as np
import pytest
import torch

from weight_only_bit_pack_b300 import inputs
from parity_util import TOL, compare, compare_nonfinite, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

AUTO, GENERIC, DECODE, PREFILL = 0, 1, 2, 3

# (row range, power of two applied to those rows of x1 and residual). The sum of
# y^2 is kept in fp32 (the kernels' stated precision), so rows whose y lies below
# about 2^-63 everywhere would underflow it; 2^-60 is the smallest scale used.
ROW_SCALES = [((0, 4), -20), ((4, 8), 15), ((8, 12), -60)]


def _scaled_rows_problem(M, eps, seed):
    prob = inputs.make_problem(M_shape=(M,), K=512, N=1024, dtype=torch.bfloat16, wbits=4,
                               mode="group", group=64, offset=True, bias=False, seed=seed,
                               eps=eps, device="cuda", name=f"row_scales_M{M}_eps{eps:g}")
    for (r0, r1), s in ROW_SCALES:
        prob.x1[r0:r1] *= 2.0 ** s  # exact in bf16: no value leaves the normal range
        prob.residual[r0:r1] *= 2.0 ** s
    return prob


@pytest.mark.parametrize("eps", [0.0, 1e-12])
@pytest.mark.parametrize("M,kernel", [(300, PREFILL), (300, GENERIC), (12, DECODE),
                                      (12, GENERIC), (12, PREFILL)])
def test_rows_far_from_unit_scale(wq, M, kernel, eps):
    prob = _scaled_rows_problem(M, eps, seed=M + int(eps > 0))
    y, no = run_gpu(wq, prob, kernel)
    _, ry, rn = run_oracle(prob)
    tol = TOL[prob.dtype]
    yg = y.double().cpu().numpy()
    ng = no.double().cpu().numpy()
    scale = np.ones((M, 1))
    for (r0, r1), s in ROW_SCALES:
        scale[r0:r1] = 2.0 ** -s
    for name, g, r in (("y", yg * scale, ry * scale), ("normOut", ng, rn)):
        err = np.abs(g - r) / (1.0 + np.abs(r))
        bad = np.argwhere(~(err <= tol))
        assert bad.size == 0, (f"{prob.name} {name}: {len(bad)} elements exceed {tol}; worst "
                               f"{err.max():.3e} at {tuple(bad[0])} (row scale 2^"
                               f"{-np.log2(scale[bad[0][0], 0]):g})")


@pytest.mark.parametrize("M,kernel", [(300, PREFILL), (300, GENERIC), (12, DECODE)])
def test_group_scales_spanning_2e20_in_one_column(wq, M, kernel):
    """Scale row r of every column is U[0.5, 1) * 2^(-20 r / (G - 1)): the groups of
    one column differ by up to 2^20 (offsets follow the same factor)."""
    K, N, g = 1024, 512, 64
    G = K // g
    prob = inputs.make_problem(M_shape=(M,), K=K, N=N, dtype=torch.bfloat16, wbits=4,
                               mode="group", group=g, offset=True, bias=True, seed=7 + M,
                               device="cuda", name=f"scale_spread_M{M}")
    gen = torch.Generator(device="cuda").manual_seed(99)
    fac = 2.0 ** (-20.0 * torch.arange(G, device="cuda", dtype=torch.float32) / (G - 1))
    u = 0.5 + 0.5 * torch.rand((G, N), generator=gen, device="cuda")
    prob.scale = (u * fac[:, None]).to(torch.bfloat16)
    prob.offset = ((torch.rand((G, N), generator=gen, device="cuda") - 0.5) * 0.04 *
                   fac[:, None]).to(torch.bfloat16)
    y, no = run_gpu(wq, prob, kernel)
    compare(prob, y, no, run_oracle(prob))


@pytest.mark.parametrize("eps", [0.0, 1e-6])
@pytest.mark.parametrize("M,kernel,dtype,mode", [
    (40, PREFILL, torch.bfloat16, "group"),     # fp16-operand mode
    (40, PREFILL, torch.float16, "channel"),    # raw-q mode
    (12, DECODE, torch.bfloat16, "group"),
    (40, GENERIC, torch.float16, "group"),
])
def test_nan_inf_and_zero_rows(wq, M, kernel, dtype, mode, eps):
    """Row 3 of x1 holds a NaN, row 5 a +Inf, row 7 of the residual a +Inf, and row 9
    of x1 and of the residual is all zeros (no bias, so y = 0 there: normOut is 0
    for eps > 0 and 0/0 = NaN for eps = 0). Every other row must be unaffected."""
    name = f"nonfinite_{kernel}_{mode}_{str(dtype)[6:]}_{eps:g}"
    prob = inputs.make_problem(M_shape=(M,), K=256, N=512, dtype=dtype, wbits=4, mode=mode,
                               group=64 if mode == "group" else 0, offset=True, bias=False,
                               seed=zlib.crc32(name.encode()) % 1000, eps=eps, device="cuda",
                               name=name)
    prob.x1[3, 17] = float("nan")
    prob.x1[5, 100] = float("inf")
    prob.residual[7, 33] = float("inf")
    prob.x1[9].zero_()
    prob.residual[9].zero_()
    y, no = run_gpu(wq, prob, kernel)
    ref = run_oracle(prob)
    compare_nonfinite(prob, y, no, ref)
    assert torch.isnan(y[3]).all() and torch.isnan(no[3]).all()
    assert bool((y[9] == 0).all())
    if eps > 0:
        assert bool((no[9] == 0).all())
    else:
        assert torch.isnan(no[9]).all()
