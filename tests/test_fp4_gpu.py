"""FP4 E2M1 pack and the mx block-scaled matmul with in-place add on the GPU.

Pack (aclnnConvertWeightToINT4Pack, "Function description", FLOAT ->
FLOAT4_E2M1): codes must equal the oracle's bit for bit (nearest magnitude, ties
to the even code, saturating at 6, the sign of -0 and of negatives that round to
0 kept).

mx matmul (aclnnQuantBatchMatmulInplaceAdd, "Function description", mx
quantization): every slice sum is exact in fp32 and the scaled slices are added
in fp64 on both sides, so the kernel's y must equal the oracle's fp64 result
rounded once to fp32, bit for bit; an E8M0 byte of 255 is NaN.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

# every E2M1 magnitude, every midpoint between neighbours, and values around them
_EDGE = [0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0, 7.0,
         0.2499999, 0.2500001, 0.7499999, 0.7500001, 4.9999995, 5.0000005, 5.9999995, 6.0000005,
         1e-30, 1e30, 65504.0, float("inf"), 1e-45]


def _pack(wq, v):
    v = v.cuda().contiguous()
    out = wq.pack_fp4(v)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_pack_fp4_edges(wq):
    vals = _EDGE + [-x for x in _EDGE]
    vals += [0.0] * (len(vals) % 2)
    v = torch.tensor(vals, dtype=torch.float32).reshape(1, -1)
    assert np.array_equal(_pack(wq, v), oracle.pack_fp4(v))


def test_pack_fp4_golden(wq):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "fp4_literals.txt")
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        lhs, rhs = line.split("->")
        v = torch.tensor([[float(t) for t in lhs.split()]], dtype=torch.float32)
        want = np.array([[int(t, 16) for t in rhs.split()]], dtype=np.uint8)
        assert np.array_equal(_pack(wq, v), want), line


@pytest.mark.parametrize("shape", [(1, 2), (3, 10), (64, 130), (4096, 4096), (7, 65534), (0, 8)])
def test_pack_fp4_random(wq, shape):
    g = torch.Generator().manual_seed(shape[0] * 7 + shape[1])
    v = torch.randn(shape, generator=g) * 3
    # plant exact ties and out-of-range values across the tensor
    if v.numel():
        idx = torch.randint(0, v.numel(), (min(v.numel(), 1000),), generator=g)
        ties = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 9.0, -1e6, -0.0])
        v.view(-1)[idx] = ties[torch.randint(0, len(ties), (len(idx),), generator=g)]
    assert np.array_equal(_pack(wq, v), oracle.pack_fp4(v))


def test_pack_fp4_unaligned_views(wq):
    # a storage offset that breaks the 16-byte vector path takes the byte path
    g = torch.Generator().manual_seed(5)
    base = (torch.randn(1, 4 * 1026 + 1, generator=g) * 4).cuda()
    v = base[:, 1:].reshape(4, 1026)
    out = wq.pack_fp4(v)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.pack_fp4(v.cpu()))


def _rand_codes(g, rows, cols):
    return torch.randint(0, 256, (rows, cols // 2), generator=g, dtype=torch.uint8)


def _mx_case(M, K, N, seed, lo=117, hi=137, nan_at=None):
    g = torch.Generator().manual_seed(seed)
    J = (K + 31) // 32
    x1, x2 = _rand_codes(g, M, K), _rand_codes(g, K, N)
    s1 = torch.randint(lo, hi, (M, J), generator=g, dtype=torch.uint8)
    s2 = torch.randint(lo, hi, (J, N), generator=g, dtype=torch.uint8)
    if nan_at is not None:
        s1[nan_at] = 255
    y = torch.randn(M, N, generator=g) * 100
    return x1, s1, x2, s2, y


def _check_mx(wq, x1, s1, x2, s2, y):
    K = x1.shape[1] * 2
    with np.errstate(over="ignore"):  # products beyond fp32 range round to inf on both sides
        want = oracle.mx_matmul_add(x1, s1, x2, s2, y.double(), K).astype(np.float32)
    yd = y.cuda().contiguous()
    wq.mx_matmul_add(x1.cuda(), s1.cuda(), x2.cuda(), s2.cuda(), yd, kernel="exact")
    torch.cuda.synchronize()
    got = yd.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok].view(np.uint32), want[ok].view(np.uint32))


@pytest.mark.parametrize("M,K,N", [(1, 32, 2), (3, 70, 10), (8, 64, 128), (17, 256, 130),
                                   (64, 1024, 256), (9, 2, 4), (5, 34, 258)])
def test_mx_matmul_add_bit_exact(wq, M, K, N):
    _check_mx(wq, *_mx_case(M, K, N, seed=M * 1000 + K + N))


def test_mx_matmul_add_wide_scales(wq):
    # exponents from 2^-127 to 2^127 on each side: products reach 2^±254
    x1, s1, x2, s2, y = _mx_case(16, 128, 64, seed=3, lo=0, hi=255)
    y[:] = 0
    _check_mx(wq, x1, s1, x2, s2, y)


def test_mx_matmul_add_nan_scale(wq):
    _check_mx(wq, *_mx_case(12, 96, 66, seed=4, nan_at=(5, 1)))


def test_mx_matmul_add_large_sample(wq):
    # a decode-sized product checked on sampled outputs (rows against the oracle one by one)
    M, K, N = 16, 4096, 4096
    x1, s1, x2, s2, y = _mx_case(M, K, N, seed=11)
    yd = y.cuda()
    wq.mx_matmul_add(x1.cuda(), s1.cuda(), x2.cuda(), s2.cuda(), yd, kernel="exact")
    torch.cuda.synchronize()
    got = yd.cpu().numpy()
    g = np.random.default_rng(0)
    cols = np.sort(g.choice(N // 2, 64, replace=False))
    for m in (0, 7, 15):
        sub2 = x2[:, cols]                      # byte columns: output columns 2c, 2c+1
        s2sub = s2[:, np.stack([2 * cols, 2 * cols + 1], 1).reshape(-1)]
        ysub = y[m:m + 1, np.stack([2 * cols, 2 * cols + 1], 1).reshape(-1)].double()
        want = oracle.mx_matmul_add(x1[m:m + 1], s1[m:m + 1], sub2, s2sub, ysub, K).astype(np.float32)
        gsub = got[m:m + 1, np.stack([2 * cols, 2 * cols + 1], 1).reshape(-1)]
        assert np.array_equal(gsub.view(np.uint32), want.view(np.uint32))


def test_mx_matmul_add_accumulates_in_place(wq):
    # two calls add twice: y + 2P where P is exact in both orders at small scales
    x1, s1, x2, s2, y = _mx_case(4, 64, 8, seed=6, lo=127, hi=128)
    want = oracle.mx_matmul_add(x1, s1, x2, s2, y.double(), 64)
    want = oracle.mx_matmul_add(x1, s1, x2, s2, want.astype(np.float32).astype(np.float64), 64)
    yd = y.cuda()
    for _ in range(2):
        wq.mx_matmul_add(x1.cuda(), s1.cuda(), x2.cuda(), s2.cuda(), yd, kernel="exact")
    torch.cuda.synchronize()
    assert np.array_equal(yd.cpu().numpy().view(np.uint32), want.astype(np.float32).view(np.uint32))


def _codes_transposed(x1):
    """(M, K/2) codes packed along K -> the same codes of x1^T, (K, M/2) packed along M."""
    b = x1.to(torch.int32)
    codes = torch.stack([b & 15, b >> 4], dim=2).reshape(x1.shape[0], -1)  # (M, K)
    t = codes.t().contiguous()                                             # (K, M)
    return (t[:, 0::2] | (t[:, 1::2] << 4)).to(torch.uint8)


@pytest.mark.parametrize("M,K,N", [(2, 32, 2), (8, 70, 10), (64, 256, 130), (18, 96, 64)])
def test_mx_matmul_add_transposed_x1(wq, M, K, N):
    # the page's supported form: x1 given as (K, M) in memory, scale1 as (ceil(K/32), M)
    x1, s1, x2, s2, y = _mx_case(M, K, N, seed=77 + M + K)
    with np.errstate(over="ignore"):
        want = oracle.mx_matmul_add(x1, s1, x2, s2, y.double(), K).astype(np.float32)
    x1t = _codes_transposed(x1)
    assert x1t.shape == (K, M // 2)
    yd = y.cuda().contiguous()
    wq.mx_matmul_add(x1t.cuda(), s1.t().contiguous().cuda(), x2.cuda(), s2.cuda(), yd,
                     x1_transposed=True, kernel="exact")
    torch.cuda.synchronize()
    assert np.array_equal(yd.cpu().numpy().view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------- tensor-core kernel

def _abs_codes(x):
    return (x & 0x77).to(torch.uint8)  # both nibbles' sign bits cleared


def _check_tc(wq, x1, s1, x2, s2, y, x1_transposed=False):
    K = x1.shape[1] * 2
    J = (K + 31) // 32
    with np.errstate(over="ignore", invalid="ignore"):
        want = oracle.mx_matmul_add(x1, s1, x2, s2, y.double(), K)
        mag = oracle.mx_matmul_add(_abs_codes(x1), s1, _abs_codes(x2), s2, y.double().abs(), K)
    tol = (J + 3) * 2.0 ** -24 * mag + (J + 2) * 2.0 ** -149
    yd = y.cuda().contiguous()
    if x1_transposed:
        wq.mx_matmul_add(_codes_transposed(x1).cuda(), s1.t().contiguous().cuda(), x2.cuda(), s2.cuda(),
                         yd, x1_transposed=True)
    else:
        wq.mx_matmul_add(x1.cuda(), s1.cuda(), x2.cuda(), s2.cuda(), yd)
    torch.cuda.synchronize()
    got = yd.cpu().numpy().astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    ok = ~nan
    err = np.abs(got[ok] - want[ok])
    assert np.all(err <= tol[ok]), (err - tol[ok]).max()


@pytest.mark.parametrize("M,K,N", [(1, 32, 2), (3, 70, 10), (128, 128, 128), (130, 256, 258),
                                   (256, 1024, 384), (9, 2, 4), (5, 34, 258), (200, 96, 136)])
def test_mx_tensor_kernel_within_bound(wq, M, K, N):
    _check_tc(wq, *_mx_case(M, K, N, seed=5000 + M * 7 + K + N))


@pytest.mark.parametrize("M,K,N", [(2, 32, 2), (130, 70, 10), (128, 256, 130), (256, 512, 256),
                                   (128, 70, 128), (64, 1000, 96), (160, 2048, 352)])
def test_mx_tensor_kernel_transposed_x1(wq, M, K, N):
    # M and N multiples of 32 take the copy-ring kernel, the others the register-fetch one
    _check_tc(wq, *_mx_case(M, K, N, seed=6000 + M + K + N), x1_transposed=True)


def test_mx_tensor_kernel_wide_exponents(wq):
    # scales from 2^-127 to 2^53 on each side: products from 2^-254 to 2^106, no fp32 overflow
    x1, s1, x2, s2, y = _mx_case(160, 256, 136, seed=8, lo=0, hi=181)
    _check_tc(wq, x1, s1, x2, s2, y)


def test_mx_tensor_kernel_large_row_exponents(wq):
    # row scales 2^118 .. 2^127 with column scales 2^-127 .. 2^-108: the slices
    # take the two-step path (a row exponent alone could overflow acc * 2^e1)
    x1, s1, x2, s2, y = _mx_case(64, 128, 64, seed=9, lo=245, hi=255)
    s2[:] = torch.randint(0, 20, s2.shape, generator=torch.Generator().manual_seed(10), dtype=torch.uint8)
    _check_tc(wq, x1, s1, x2, s2, y)


def test_mx_tensor_kernel_nan_scale(wq):
    _check_tc(wq, *_mx_case(140, 96, 130, seed=11, nan_at=(133, 2)))


def test_mx_tensor_kernel_sampled_large(wq):
    # the bench's gradient-accumulation shape, x1 transposed, rows sampled
    M, K, N = 4096, 8192, 4096
    x1, s1, x2, s2, y = _mx_case(M, K, N, seed=12, lo=120, hi=134)
    yd = y.cuda()
    wq.mx_matmul_add(_codes_transposed(x1).cuda(), s1.t().contiguous().cuda(), x2.cuda(), s2.cuda(), yd,
                     x1_transposed=True)
    torch.cuda.synchronize()
    got = yd.cpu().numpy().astype(np.float64)
    J = K // 32
    for m in (0, 1, 127, 128, 2049, 4095):
        want = oracle.mx_matmul_add(x1[m:m + 1], s1[m:m + 1], x2, s2, y[m:m + 1].double(), K)
        mag = oracle.mx_matmul_add(_abs_codes(x1[m:m + 1]), s1[m:m + 1], _abs_codes(x2), s2,
                                   y[m:m + 1].double().abs(), K)
        tol = (J + 3) * 2.0 ** -24 * mag
        assert np.all(np.abs(got[m:m + 1] - want) <= tol), m
