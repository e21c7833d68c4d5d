"""Kernel-native tiled INT4 layout on the GPU: the pack into it and the layout
conversions (bit-exact against the oracle's restatement of the layout), and the
tiled decode kernel (against the fp64 oracle, like every other kernel).

The layout is the library's analogue of the pack's matrix-unit output
(aclnnConvertWeightToINT4Pack, "Function description"), defined in
include/wq.h; the operator it feeds is the one of
aclnnWeightQuantMatmulAllReduceAddRmsNorm.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from weight_only_bit_pack_b300 import inputs
from parity_util import compare, run_oracle, sample_rows

pytestmark = pytest.mark.gpu

AUTO, GENERIC, DECODE, PREFILL = 0, 1, 2, 3


@pytest.mark.parametrize("K,N", [(64, 16), (100, 48), (256, 128), (4096, 4096), (8192, 28672),
                                 (33, 4112)])
def test_pack_tiled_bit_exact_and_conversions(wq, K, N):
    g = torch.Generator().manual_seed(K * 7 + N)
    v = torch.randint(-8, 8, (K, N), generator=g, dtype=torch.int32)
    if K * N < 1 << 20:  # out-of-range int32 keep their low four bits, as in the ND pack
        v[0, :4] = torch.tensor([100, -100, 2 ** 30, -(2 ** 31)], dtype=torch.int32)
    vd = v.cuda()
    t = wq.pack_int4_tiled(vd)
    ref = oracle.pack_int4_tiled(v)
    assert np.array_equal(t.data.cpu().numpy(), ref)
    nd = wq.pack_int4(vd)
    assert torch.equal(wq.int4_to_tiled(nd).data, t.data)          # ND -> tiled
    assert torch.equal(wq.tiled_to_int4(t), nd)                    # tiled -> ND
    torch.cuda.synchronize()


def _tiled_problem(prob):
    return prob, wq_tiled(prob)


def wq_tiled(prob):
    import weight_only_bit_pack_b300 as wq
    return wq.pack_int4_tiled(prob.x2.to("cuda").contiguous())


def _run(wq, prob, w, kernel, **kw):
    y, no = wq.matmul_add_rmsnorm(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                                  prob.gamma, prob.eps, prob.group, kernel=kernel, **kw)
    torch.cuda.synchronize()
    return y, no


@pytest.mark.parametrize("cfg", ["tiny", "decode", "sweep1", "sweep16"])
def test_named_workloads_tiled(wq, cfg):
    if cfg == "tiny":
        from parity_util import to_device
        prob = to_device(inputs.tiny())
    elif cfg == "decode":
        prob = inputs.decode("cuda")
    else:
        prob = inputs.sweep(int(cfg[5:]), device="cuda")
    w = wq_tiled(prob)
    assert wq.select_kernel(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                            prob.gamma, prob.eps, prob.group) == wq.Kernel.DECODE
    y, no = _run(wq, prob, w, AUTO)
    compare(prob, y, no, run_oracle(prob))


CASES = [
    ("m1_channel", dict(M_shape=(1,), K=512, N=256, dtype=torch.bfloat16, mode="channel")),
    ("m3_tensor_offset", dict(M_shape=(3,), K=192, N=48, dtype=torch.float16, mode="tensor")),
    ("m5_group32_ragged_k", dict(M_shape=(5,), K=200, N=96, dtype=torch.bfloat16, mode="group",
                                 group=32)),
    ("m7_group96", dict(M_shape=(7,), K=960, N=320, dtype=torch.bfloat16, mode="group",
                        group=96)),
    ("m8_group64_nooffset", dict(M_shape=(8,), K=1024, N=1024, dtype=torch.bfloat16,
                                 mode="group", group=64, offset=False)),
    ("m9_fp16_group128", dict(M_shape=(9,), K=2048, N=512, dtype=torch.float16, mode="group",
                              group=128)),
    ("m12_channel2d_nobias", dict(M_shape=(3, 4), K=1024, N=2064, dtype=torch.bfloat16,
                                  mode="channel2d", bias=False)),
    ("m16_group32", dict(M_shape=(2, 8), K=4096, N=768, dtype=torch.bfloat16, mode="group",
                         group=32)),
    ("k8_single_rows", dict(M_shape=(4,), K=8, N=16, dtype=torch.float16, mode="channel")),
    ("wide_n_20000", dict(M_shape=(6,), K=256, N=20000, dtype=torch.float16, mode="channel")),
    ("long_k_65528", dict(M_shape=(2,), K=65528, N=64, dtype=torch.bfloat16, mode="group",
                          group=256, offset=False)),
    ("max_n_65520", dict(M_shape=(1,), K=64, N=65520, dtype=torch.bfloat16, mode="group",
                         group=32)),
    # group-structured loop (K % 128 == 0, group % 128 == 0 or one scale row,
    # x1 staged in shared memory, >= 8 units of 128 k-rows per warp): groups
    # of several units with a short last group, per-channel with an odd unit
    # count, a per-tensor scale with offsets, one column group per CTA, eight
    # rows with per-group offsets, two row blocks (12 rows)
    ("m4_group256_short_last", dict(M_shape=(4,), K=16512, N=272, dtype=torch.bfloat16,
                                    mode="group", group=256)),
    ("m2_channel_odd_units", dict(M_shape=(2,), K=16256, N=4800, dtype=torch.float16,
                                  mode="channel")),
    ("m5_tensor_offset_k8192", dict(M_shape=(5,), K=8192, N=4096, dtype=torch.float16,
                                    mode="tensor")),
    ("m3_group384_one_group_per_cta", dict(M_shape=(3,), K=19200, N=96, dtype=torch.float16,
                                           mode="group", group=384)),
    ("m8_group128_offset_n8192", dict(M_shape=(8,), K=8192, N=8192, dtype=torch.bfloat16,
                                      mode="group", group=128)),
    ("m12_group128_two_row_blocks", dict(M_shape=(12,), K=4096, N=8192, dtype=torch.bfloat16,
                                         mode="group", group=128, offset=False)),
    # the general loop with 16 rows, offsets and x1 read from global memory
    ("m16_group128_offset_k8192", dict(M_shape=(16,), K=8192, N=512, dtype=torch.bfloat16,
                                       mode="group", group=128)),
    # the k-major kernel (9..64 rows, x1 staged per 128-row slice): 16 rows
    # with >= 8 column groups per CTA, 24 rows (four row blocks, rows past M
    # zero-filled by the copy) with few column groups, 32 rows fp16 with
    # offsets and 256-row groups, per-channel, per-tensor with 9 rows
    ("km_m16_group128", dict(M_shape=(16,), K=1024, N=20480, dtype=torch.bfloat16,
                             mode="group", group=128, offset=False)),
    ("km_m24_group128_offset", dict(M_shape=(4, 6), K=2048, N=4096, dtype=torch.bfloat16,
                                    mode="group", group=128)),
    ("km_m32_fp16_group256_offset", dict(M_shape=(32,), K=4096, N=2048, dtype=torch.float16,
                                         mode="group", group=256)),
    ("km_m20_channel", dict(M_shape=(20,), K=1024, N=20480, dtype=torch.bfloat16,
                            mode="channel")),
    ("km_m9_tensor_fp16", dict(M_shape=(9,), K=1280, N=20480, dtype=torch.float16,
                               mode="tensor")),
    # eight row blocks (two passes per slice): 64 rows, and 40 rows fp16 with offsets
    ("km_m64_group128", dict(M_shape=(64,), K=2048, N=4096, dtype=torch.bfloat16,
                             mode="group", group=128, offset=False)),
    ("km_m40_fp16_channel", dict(M_shape=(5, 8), K=1024, N=2048, dtype=torch.float16,
                                 mode="channel")),
    # one 128-row slice (fewer slices than the weight ring holds)
    ("km_m12_k128_channel", dict(M_shape=(12,), K=128, N=20480, dtype=torch.bfloat16,
                                 mode="channel")),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("kernel", [DECODE, GENERIC])
def test_tiled_kernels_vs_oracle(wq, name, kw, kernel):
    prob = inputs.make_problem(**kw, wbits=4, seed=zlib.crc32(name.encode()) % 1000,
                               device="cuda", name=name)
    w = wq_tiled(prob)
    y, no = _run(wq, prob, w, kernel)
    compare(prob, y, no, run_oracle(prob))


def test_tiled_auto_above_16_rows_runs_generic(wq):
    prob = inputs.make_problem(M_shape=(40,), K=256, N=128, dtype=torch.bfloat16, wbits=4,
                               mode="group", group=64, seed=3, device="cuda", name="tiled_m40")
    w = wq_tiled(prob)
    assert wq.select_kernel(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                            prob.gamma, prob.eps, prob.group) == wq.Kernel.GENERIC
    y, no = _run(wq, prob, w, AUTO)
    compare(prob, y, no, run_oracle(prob))


def test_tiled_decode_deterministic_and_reusable_workspace(wq):
    prob = inputs.sweep(16, device="cuda")
    w = wq_tiled(prob)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    a = _run(wq, prob, w, AUTO, workspace=ws)
    b = _run(wq, prob, w, AUTO, workspace=ws)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert wq.read_device_status(ws) == 0
    assert int(ws[:2048].sum()) == 0  # grid counters back at zero


def _timeout_problem(which):
    if which == "decode":  # the general loop
        return inputs.decode("cuda")
    if which == "sweep1":  # the group-structured loop
        return inputs.sweep(1, device="cuda")
    # the k-major kernel
    return inputs.make_problem(M_shape=(24,), K=2048, N=4096, dtype=torch.bfloat16, wbits=4,
                               mode="group", group=128, seed=5, device="cuda", name="km_timeout")


@pytest.mark.parametrize("which", ["decode", "sweep1", "kmajor"])
def test_tiled_decode_timeout_path(wq, which):
    prob = _timeout_problem(which)
    w = wq_tiled(prob)
    assert wq.select_kernel(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                            prob.gamma, prob.eps, prob.group) == wq.Kernel.DECODE
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    wq.set_wait_limits_for_testing(2_000_000, 1)
    try:
        _run(wq, prob, w, AUTO, workspace=ws)
        st = wq.read_device_status(ws)
    finally:
        wq.set_wait_limits_for_testing(0, 0)
    assert st & 0xFF == 8 and st >> 8 == wq.WHERE_DECODE_GRID, hex(st)
    ws[:2048].zero_()
    y, no = _run(wq, prob, w, AUTO, workspace=ws, check_status=True)
    compare(prob, y, no, run_oracle(prob))
