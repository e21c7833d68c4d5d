"""Per-token symmetric dynamic quantization on the GPU (aclnnDynamicQuant,
"Function description"): codes and scales must equal the oracle's bit for bit
(both sides take every floating-point step as the same IEEE fp32 operation, and
the code is the round-half-to-even integer of the quotient)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _check(wq, x, smooth, bits):
    y, s = wq.dynamic_quant(x, smooth, bits=bits)
    torch.cuda.synchronize()
    rq, rs = oracle.dynamic_quant(x.float().cpu(), None if smooth is None else smooth.float().cpu(),
                                  bits=bits)
    assert np.array_equal(s.cpu().numpy().reshape(rs.shape), rs)
    if bits == 8:
        assert np.array_equal(y.cpu().numpy(), rq)
    else:
        packed = oracle.pack_int4(rq.reshape(-1, rq.shape[-1]).astype(np.int32))
        assert np.array_equal(y.cpu().numpy().reshape(packed.shape), packed)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("shape", [(1, 8), (3, 200), (8192, 4096), (2, 5, 1024), (7, 65534),
                                   (33, 6), (300, 8192), (9, 6144), (5, 2056), (4, 8200)])
@pytest.mark.parametrize("smooth", [False, True])
def test_dynamic_quant_bit_exact(wq, dtype, bits, shape, smooth):
    g = torch.Generator(device="cuda").manual_seed(sum(shape) + bits)
    x = (torch.randn(shape, generator=g, device="cuda") *
         torch.empty(shape[:-1] + (1,), device="cuda").uniform_(0.01, 50, generator=g)).to(dtype)
    sm = (torch.rand(shape[-1], generator=g, device="cuda") * 1.5 + 0.25).to(dtype) if smooth else None
    _check(wq, x, sm, bits)


def test_dynamic_quant_ties_zero_and_nonfinite_rows(wq):
    rows = [[2.5, 127, -3.5, 0.5, 1.5, -0.5, 0, 100],   # scale exactly 1: ties to even
            [0] * 8,                                    # zero row: scale 0, codes 0
            [1, float("nan"), -2, 4, 0, 0, 0, 1],       # a NaN element
            [1, float("inf"), -2, 4, 0, 0, 0, 1],       # an Inf element
            [-127, 63.5, -63.5, 0.25, 126.5, -126.5, 1, 2]]
    for dt in (torch.float16, torch.bfloat16):
        x = torch.tensor(rows, dtype=dt, device="cuda")
        for bits in (8, 4):
            _check(wq, x, None, bits)


def test_dynamic_quant_tiny_and_huge_scales(wq):
    """bf16 keeps fp32's exponent range: a row maximum near 1e-38 gives a
    subnormal scale (codes from the IEEE quotient itself), near 1e-30 and 1e36
    normal scales with their reciprocals far from 1."""
    rows = [[1e-38, -5e-39, 3e-39, 0, 2.5e-39, -7.5e-39, 1e-40, 6e-39],
            [1e-30, -3.3e-31, 5e-31, 0, 2e-31, -7.9e-31, 1e-32, 6.1e-31],
            [1e36, -3.3e35, 5e35, 0, 2e35, -7.9e35, 1e34, 6.1e35]]
    x = torch.tensor(rows, dtype=torch.bfloat16, device="cuda")
    for bits in (8, 4):
        _check(wq, x, None, bits)
