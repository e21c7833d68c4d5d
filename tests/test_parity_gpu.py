"""CUDA path vs the fp64 oracle for the fused dequant-matmul + AddRmsNorm (GPU).

Every case draws seeded inputs (weight_only_bit_pack_b300.inputs), packs INT4
weights with the pack kernel, runs the operator through the C ABI, and checks y
and normOut against the oracle within |d| <= tol * (1 + |ref|) (1e-2 for bf16,
2e-3 for fp16). Large problems are checked on a seeded sample of rows plus the
first and last row; rows are independent, so each sampled row is checked in
full.
"""
import zlib

import numpy as np
import pytest
import torch

from weight_only_bit_pack_b300 import inputs
from parity_util import compare, gpu_weight, run_gpu, run_oracle, sample_rows, to_device

pytestmark = pytest.mark.gpu

GENERIC, DECODE, PREFILL = 1, 2, 3


# Oracle results of the large named workloads, kept for the test session so
# that each workload's oracle runs once for all the kernels checked on it.
_ORACLE_CACHE = {}


def _check(wq, prob, kernel, n_sample=None):
    y, no = run_gpu(wq, prob, kernel)
    rows = None if n_sample is None else sample_rows(prob.M, n_sample)
    key = (prob.name, None if rows is None else tuple(int(r) for r in rows))
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = run_oracle(prob, rows)
    return compare(prob, y, no, _ORACLE_CACHE[key], rows)


# rows compared on the large workloads: a seeded sample of 512 plus the first
# and the last row (rows are independent, so every sampled row is checked in full)
N_SAMPLE = 512


# ------------------------------------------------------------------ named workloads

def test_tiny_auto(wq):
    _check(wq, to_device(inputs.tiny()), 0)


@pytest.mark.parametrize("kernel", [GENERIC, DECODE])
def test_tiny_forced(wq, kernel):
    _check(wq, to_device(inputs.tiny()), kernel)


def test_prefill_rejects_fp16_per_group(wq):
    """fp16 activations with per-group scales have no exact single-operand tensor-core
    form; the prefill kernel refuses them instead of rounding W."""
    from weight_only_bit_pack_b300.binding import WQError, Status
    with pytest.raises(WQError) as ei:
        run_gpu(wq, to_device(inputs.tiny()), PREFILL)
    assert ei.value.status == Status.ERR_UNSUPPORTED


@pytest.mark.parametrize("kernel", [0, GENERIC, DECODE, PREFILL])
def test_decode(wq, kernel):
    _check(wq, inputs.decode("cuda"), kernel)


@pytest.mark.parametrize("kernel", [0, GENERIC, PREFILL])
def test_w8a16(wq, kernel):
    """Every element of the 2048 x 11008 output."""
    _check(wq, inputs.w8a16("cuda"), kernel)


@pytest.mark.parametrize("kernel", [0, PREFILL])
def test_prefill_workload(wq, kernel):
    _check(wq, inputs.prefill("cuda"), kernel, n_sample=N_SAMPLE)


@pytest.mark.parametrize("M", inputs.SWEEP_M)
def test_sweep(wq, M):
    _check(wq, inputs.sweep(M, device="cuda"), 0, n_sample=N_SAMPLE)


def test_sweep_per_tensor(wq):
    _check(wq, inputs.sweep(4096, per_tensor=True, device="cuda"), 0, n_sample=N_SAMPLE)


PREFILL_EDGE = [
    ("m_tail_k_tail", dict(M_shape=(300,), K=200, N=608, dtype=torch.bfloat16, wbits=4,
                           mode="group", group=64)),
    ("many_waves_bf16_g32", dict(M_shape=(1000,), K=512, N=2048, dtype=torch.bfloat16, wbits=4,
                                 mode="group", group=32)),
    ("many_waves_fp16_channel", dict(M_shape=(1000,), K=512, N=2048, dtype=torch.float16, wbits=4,
                                     mode="channel")),
    ("int8_bf16_group", dict(M_shape=(160,), K=256, N=272, dtype=torch.bfloat16, wbits=8,
                             mode="group", group=64)),
    ("int8_bf16_offset", dict(M_shape=(3, 70), K=136, N=208, dtype=torch.bfloat16, wbits=8,
                              mode="channel")),
    ("int8_fp16_tensor", dict(M_shape=(129,), K=64, N=272, dtype=torch.float16, wbits=8,
                              mode="tensor", bias=False)),
    ("int4_per_tensor_nobias", dict(M_shape=(256,), K=1024, N=512, dtype=torch.bfloat16, wbits=4,
                                    mode="tensor", bias=False, offset=False)),
    ("single_k_tile", dict(M_shape=(130,), K=64, N=256, dtype=torch.float16, wbits=4,
                           mode="channel")),
    ("wide_rows_79_ntiles", dict(M_shape=(200,), K=128, N=20000 + 224, dtype=torch.bfloat16,
                                 wbits=4, mode="group", group=32)),
    # enough n-tiles that 256-row tiles (two 128-row MMA halves) are chosen:
    # the last row block ends inside its first half, its second half is empty
    ("halves_m_tail_bf16_g64", dict(M_shape=(600,), K=128, N=148 * 256, dtype=torch.bfloat16,
                                    wbits=4, mode="group", group=64)),
    ("halves_fp16_channel_offset", dict(M_shape=(200,), K=192, N=79 * 256, dtype=torch.float16,
                                        wbits=4, mode="channel")),
    ("int8_bf16_tensor_79_ntiles", dict(M_shape=(200,), K=96, N=79 * 256, dtype=torch.bfloat16,
                                        wbits=8, mode="tensor", bias=False)),
    # INT8 weights over 79 n-tiles: per-group scales (fp16-operand form with
    # its offset k-steps) and per-channel scales with offsets, ragged last row block
    ("int8_halves_bf16_g64_offset", dict(M_shape=(250,), K=192, N=79 * 256,
                                         dtype=torch.bfloat16, wbits=8, mode="group", group=64)),
    ("int8_halves_fp16_channel_offset", dict(M_shape=(2, 100), K=128, N=79 * 256,
                                             dtype=torch.float16, wbits=8, mode="channel")),
]


@pytest.mark.parametrize("name,kw", PREFILL_EDGE, ids=[e[0] for e in PREFILL_EDGE])
def test_prefill_edge_shapes(wq, name, kw):
    prob = inputs.make_problem(**kw, seed=zlib.crc32(name.encode()) % 1000, device="cuda",
                               name=name)
    _check(wq, prob, PREFILL)


# ------------------------------------------------------------------ edge shapes

EDGE = [
    # name, kwargs of inputs.make_problem
    ("ragged_group", dict(M_shape=(5,), K=200, N=96, dtype=torch.bfloat16, wbits=4, mode="group",
                          group=64)),
    ("odd_k_per_channel", dict(M_shape=(3,), K=77, N=46, dtype=torch.float16, wbits=4,
                               mode="channel")),
    ("n2_per_tensor", dict(M_shape=(4,), K=64, N=2, dtype=torch.bfloat16, wbits=4, mode="tensor")),
    ("m1", dict(M_shape=(1,), K=512, N=384, dtype=torch.bfloat16, wbits=4, mode="group", group=128,
                offset=False)),
    ("int8_bf16_channel2d", dict(M_shape=(2, 9), K=160, N=200, dtype=torch.bfloat16, wbits=8,
                                 mode="channel2d")),
    ("int8_odd_n", dict(M_shape=(7,), K=96, N=33, dtype=torch.float16, wbits=8, mode="tensor",
                        bias=False)),
    ("n_not_mult_256", dict(M_shape=(33,), K=256, N=4104, dtype=torch.bfloat16, wbits=4,
                            mode="group", group=32)),
    ("wide_n", dict(M_shape=(2,), K=64, N=20000, dtype=torch.float16, wbits=4, mode="channel")),
]


@pytest.mark.parametrize("name,kw", EDGE, ids=[e[0] for e in EDGE])
@pytest.mark.parametrize("kernel", [0, GENERIC])
def test_edge_shapes(wq, name, kw, kernel):
    prob = inputs.make_problem(**kw, seed=zlib.crc32(name.encode()) % 1000, device="cuda", name=name)
    _check(wq, prob, kernel)


def test_empty_m_writes_nothing(wq):
    prob = inputs.make_problem(M_shape=(0,), K=64, N=32, dtype=torch.float16, wbits=4,
                               mode="channel", device="cuda")
    y = torch.full((0, 32), 7.0, dtype=torch.float16, device="cuda")
    y2, no = run_gpu(wq, prob, 0, y=y)
    assert y2.shape == (0, 32) and no.shape == (0, 32)


def test_in_place_y_into_residual(wq):
    prob = inputs.make_problem(M_shape=(4, 3), K=128, N=64, dtype=torch.bfloat16, wbits=4,
                               mode="group", group=64, device="cuda")
    ref = run_oracle(prob)
    res = prob.residual.clone()
    y, no = run_gpu(wq, prob, 0, y=res)
    prob_view = prob
    assert y.data_ptr() == res.data_ptr()
    compare(prob_view, y, no, ref)


def test_integer_inputs_bit_exact_y(wq):
    """Integer x1 in [-4, 4], scale 1, no offset/bias/residual: every fp32 partial
    sum is an exact integer below 2^24, so y = RNE_fp16(x1 @ q) bit for bit."""
    K, N, M = 96, 64, 8
    g = torch.Generator().manual_seed(11)
    x1 = torch.randint(-4, 5, (M, K), generator=g).to(torch.float16)
    q = torch.randint(-8, 8, (K, N), generator=g, dtype=torch.int32)
    prob = inputs.Problem("int_exact", torch.float16, 4, x1, q, torch.ones(1, dtype=torch.float16),
                          None, None, torch.zeros(M, N, dtype=torch.float16),
                          torch.ones(N, dtype=torch.float16), 1e-6, 0)
    to_device(prob)
    mm = (x1.double() @ q.double())
    assert mm.abs().max() <= 2048
    for kernel in (0, GENERIC, DECODE, PREFILL):
        y, _ = run_gpu(wq, prob, kernel)
        assert torch.equal(y.cpu(), mm.to(torch.float16)), kernel


def test_deterministic_across_runs(wq):
    prob = inputs.decode("cuda")
    w = gpu_weight(wq, prob)
    for kernel in (0, GENERIC, DECODE, PREFILL):
        a = run_gpu(wq, prob, kernel, w=w)
        b = run_gpu(wq, prob, kernel, w=w)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_row_permutation_equivariance(wq):
    prob = inputs.make_problem(M_shape=(12,), K=256, N=512, dtype=torch.bfloat16, wbits=4,
                               mode="group", group=128, device="cuda")
    w = gpu_weight(wq, prob)
    y, no = run_gpu(wq, prob, 0, w=w)
    perm = torch.randperm(12, generator=torch.Generator().manual_seed(3)).cuda()
    prob.x1 = prob.x1[perm].contiguous()
    prob.residual = prob.residual[perm].contiguous()
    yp, nop = run_gpu(wq, prob, 0, w=w)
    assert torch.equal(yp, y[perm]) and torch.equal(nop, no[perm])
