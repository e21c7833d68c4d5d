"""Transposed weights on the GPU (aclnnWeightQuantMatmulAllReduceAddRmsNorm,
"Constraints": x2 may be transposed): the operator with x2 stored as its (N, K)
transpose -- INT8, or INT4 packed two per byte along K -- against the fp64 oracle
on the untransposed weight, and the INT4 layout conversions (dense, transposed,
tiled) against the oracle's packings, bit for bit."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from weight_only_bit_pack_b300 import inputs
from parity_util import compare, run_oracle

pytestmark = pytest.mark.gpu


def _transposed(wq, prob):
    qt = prob.x2.to("cuda").t().contiguous()  # (N, K)
    if prob.wbits == 8:
        return wq.TransposedWeight(qt, 8)
    return wq.TransposedWeight(wq.pack_int4(qt.to(torch.int32)), 4)


CASES = [
    ("int4_group_m5", dict(M_shape=(5,), K=256, N=96, dtype=torch.bfloat16, wbits=4, mode="group",
                           group=64)),
    ("int4_channel_m40", dict(M_shape=(40,), K=130, N=66, dtype=torch.float16, wbits=4,
                              mode="channel")),
    ("int8_tensor_m3", dict(M_shape=(3,), K=77, N=33, dtype=torch.float16, wbits=8, mode="tensor")),
    ("int8_group_m300", dict(M_shape=(300,), K=512, N=256, dtype=torch.bfloat16, wbits=8,
                             mode="group", group=128)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_transposed_x2_vs_oracle(wq, name, kw):
    prob = inputs.make_problem(**kw, seed=zlib.crc32(name.encode()) % 1000, device="cuda", name=name)
    w = _transposed(wq, prob)
    assert wq.select_kernel(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                            prob.gamma, prob.eps, prob.group) == wq.Kernel.GENERIC
    y, no = wq.matmul_add_rmsnorm(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                                  prob.gamma, prob.eps, prob.group)
    torch.cuda.synchronize()
    compare(prob, y, no, run_oracle(prob))


@pytest.mark.parametrize("K,N", [(64, 16), (130, 48), (4096, 4096), (200, 1008)])
def test_int4_layout_conversions_bit_exact(wq, K, N):
    g = torch.Generator().manual_seed(K + N)
    v = torch.randint(-8, 8, (K, N), generator=g, dtype=torch.int32)
    nd_ref = oracle.pack_int4(v)                  # (K, N/2)
    t_ref = oracle.pack_int4(v.t().contiguous())  # (N, K/2): packed along K
    tiled_ref = oracle.pack_int4_tiled(v)
    nd = wq.pack_int4(v.cuda())
    tw = wq.TransposedWeight(wq.pack_int4(v.t().contiguous().cuda()), 4)
    assert np.array_equal(tw.data.cpu().numpy(), t_ref)
    outs = {
        ("dense", "transposed"): wq.convert_int4(nd, "transposed").data,
        ("transposed", "dense"): wq.convert_int4(tw, "dense"),
        ("transposed", "tiled"): wq.convert_int4(tw, "tiled").data,
        ("tiled", "transposed"): wq.convert_int4(wq.pack_int4_tiled(v.cuda()), "transposed").data,
    }
    torch.cuda.synchronize()
    refs = {"dense": nd_ref, "transposed": t_ref, "tiled": tiled_ref}
    for (a, b), out in outs.items():
        assert np.array_equal(out.cpu().numpy().reshape(refs[b].shape), refs[b]), (a, b)


def test_transposed_weight_converted_for_the_decode_kernel(wq):
    """An INT4_T weight converted once to the tiled layout runs on the tiled decode
    kernel and matches the oracle."""
    prob = inputs.decode("cuda")
    tiled = wq.convert_int4(_transposed(wq, prob), "tiled")
    assert wq.select_kernel(prob.x1, tiled, prob.scale, prob.offset, prob.bias, prob.residual,
                            prob.gamma, prob.eps, prob.group) == wq.Kernel.DECODE
    y, no = wq.matmul_add_rmsnorm(prob.x1, tiled, prob.scale, prob.offset, prob.bias,
                                  prob.residual, prob.gamma, prob.eps, prob.group)
    torch.cuda.synchronize()
    compare(prob, y, no, run_oracle(prob))


# ---------------------------------------------------------------- transposed large-M kernel

from parity_util import sample_rows  # noqa: E402

T_CASES = [
    ("t_256x512x512_g128", dict(M_shape=(256,), K=512, N=512, g=128)),
    ("t_300x256x288_g64", dict(M_shape=(300,), K=256, N=288, g=64)),   # ragged row block and n-tile
    ("t_17x128x32_g32", dict(M_shape=(17,), K=128, N=32, g=32)),      # one partial tile, two groups per k-step
    ("t_2x9x64_g64_3d", dict(M_shape=(2, 9), K=192, N=96, g=64)),     # 3-D x1, group ending mid-stage
]


@pytest.mark.parametrize("name,kw", T_CASES, ids=[c[0] for c in T_CASES])
def test_transposed_prefill_kernel_vs_oracle(wq, name, kw):
    """bf16 per-group, no offset: the transposed weight runs on the large-M kernel
    whose dequantized weight is the MMA's A operand in tensor memory."""
    prob = inputs.make_problem(M_shape=kw["M_shape"], K=kw["K"], N=kw["N"], dtype=torch.bfloat16,
                               wbits=4, mode="group", group=kw["g"], offset=False,
                               seed=zlib.crc32(name.encode()) % 1000, device="cuda", name=name)
    w = _transposed(wq, prob)
    assert wq.select_kernel(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                            prob.gamma, prob.eps, prob.group) == wq.Kernel.PREFILL
    y, no = wq.matmul_add_rmsnorm(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                                  prob.gamma, prob.eps, prob.group, check_status=True)
    torch.cuda.synchronize()
    compare(prob, y, no, run_oracle(prob))


def test_transposed_prefill_sweep_shape_sampled(wq):
    """The sweep's weight (8192 x 28672, g = 128) transposed, M = 1024: 512 seeded
    rows plus the first and last against the oracle."""
    prob = inputs.sweep(1024, device="cuda")
    w = _transposed(wq, prob)
    assert wq.select_kernel(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                            prob.gamma, prob.eps, prob.group) == wq.Kernel.PREFILL
    y, no = wq.matmul_add_rmsnorm(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                                  prob.gamma, prob.eps, prob.group, check_status=True)
    torch.cuda.synchronize()
    rows = sample_rows(prob.M, 512)
    compare(prob, y, no, run_oracle(prob, rows=rows), rows=rows)


def test_transposed_prefill_in_place_and_repeat(wq):
    """y written into residual, and two calls on one workspace give the same bits."""
    prob = inputs.make_problem(M_shape=(200,), K=256, N=256, dtype=torch.bfloat16, wbits=4,
                               mode="group", group=128, offset=False, seed=5, device="cuda",
                               name="t_inplace")
    w = _transposed(wq, prob)
    ref = run_oracle(prob)
    y1, n1 = wq.matmul_add_rmsnorm(prob.x1, w, prob.scale, None, prob.bias, prob.residual,
                                   prob.gamma, prob.eps, prob.group)
    y2, n2 = wq.matmul_add_rmsnorm(prob.x1, w, prob.scale, None, prob.bias, prob.residual,
                                   prob.gamma, prob.eps, prob.group)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(n1, n2)
    res = prob.residual.clone()
    y3, n3 = wq.matmul_add_rmsnorm(prob.x1, w, prob.scale, None, prob.bias, res, prob.gamma,
                                   prob.eps, prob.group, y=res)
    torch.cuda.synchronize()
    assert torch.equal(y3, y1) and torch.equal(n3, n1)
    compare(prob, y1, n1, ref)


def test_transposed_with_offset_stays_generic(wq):
    prob = inputs.make_problem(M_shape=(64,), K=256, N=64, dtype=torch.bfloat16, wbits=4,
                               mode="group", group=64, offset=True, seed=6, device="cuda",
                               name="t_offset")
    w = _transposed(wq, prob)
    assert wq.select_kernel(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                            prob.gamma, prob.eps, prob.group) == wq.Kernel.GENERIC
    y, no = wq.matmul_add_rmsnorm(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                                  prob.gamma, prob.eps, prob.group)
    torch.cuda.synchronize()
    compare(prob, y, no, run_oracle(prob))
