"""The small-M decode kernel (WQ_KERNEL_DECODE) vs the fp64 oracle (GPU).

The decode kernel cuts the (256-column tile, 64-row stage) units into one
equal run per CTA, finishes each tile in the CTA that completes its last
segment, and meets all CTAs at a grid-wide counter for the RMSNorm. These
cases aim at its edges: K that leaves a partial 64-row stage or a single
stage, runs that cover several tiles, group sizes that are not powers of two,
every scale mode with and without offset, one and two 8-row MMA tiles, and
repeated calls on one workspace whose grid changes between calls (the
counters in the workspace header must come back to zero after every call).
"""
import zlib

import pytest
import torch

from weight_only_bit_pack_b300 import inputs
from parity_util import compare, gpu_weight, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

DECODE = 2

CASES = [
    ("k64_one_stage", dict(M_shape=(3,), K=64, N=256, dtype=torch.bfloat16, wbits=4,
                           mode="channel")),
    ("k96_two_stages", dict(M_shape=(8,), K=96, N=64, dtype=torch.float16, wbits=4,
                            mode="group", group=32)),
    ("k200_partial_stage", dict(M_shape=(5,), K=200, N=96, dtype=torch.bfloat16, wbits=4,
                                mode="group", group=64)),
    ("g96_not_pow2", dict(M_shape=(7,), K=960, N=320, dtype=torch.bfloat16, wbits=4,
                          mode="group", group=96)),
    ("fp16_group_offset_m16", dict(M_shape=(2, 8), K=1024, N=512, dtype=torch.float16,
                                   wbits=4, mode="group", group=128)),
    ("bf16_tensor_m9", dict(M_shape=(9,), K=512, N=768, dtype=torch.bfloat16, wbits=4,
                            mode="tensor")),
    ("bf16_channel2d_nobias", dict(M_shape=(4,), K=2048, N=1024, dtype=torch.bfloat16, wbits=4,
                                   mode="channel2d", bias=False)),
    ("many_tiles_m1", dict(M_shape=(1,), K=1024, N=16384, dtype=torch.bfloat16, wbits=4,
                           mode="group", group=128, offset=False)),
    ("long_k_m12", dict(M_shape=(12,), K=16384, N=256, dtype=torch.bfloat16, wbits=4,
                        mode="group", group=256, offset=False)),
    ("ragged_n_tile", dict(M_shape=(6,), K=512, N=20000, dtype=torch.float16, wbits=4,
                           mode="channel")),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_decode_edge_cases(wq, name, kw):
    prob = inputs.make_problem(**kw, seed=zlib.crc32(name.encode()) % 1000, device="cuda",
                               name=name)
    y, no = run_gpu(wq, prob, DECODE)
    compare(prob, y, no, run_oracle(prob))


def test_decode_is_auto_choice_for_small_m(wq):
    for M in (1, 8, 16):
        p = inputs.make_problem(M_shape=(M,), K=256, N=256, dtype=torch.bfloat16, wbits=4,
                                mode="group", group=64, device="cuda")
        w = gpu_weight(wq, p)
        assert wq.select_kernel(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma,
                                p.eps, p.group) == wq.Kernel.DECODE


def test_decode_rejects_what_it_cannot_run(wq):
    from weight_only_bit_pack_b300.binding import Status, WQError
    bad = [dict(M_shape=(17,), K=256, N=256, wbits=4),       # M > 16
           dict(M_shape=(4,), K=256, N=96 + 2, wbits=4),      # n % 32 != 0
           dict(M_shape=(4,), K=77, N=256, wbits=4),          # k % 8 != 0
           dict(M_shape=(4,), K=256, N=256, wbits=8)]         # INT8
    for kw in bad:
        p = inputs.make_problem(**kw, dtype=torch.bfloat16, mode="channel", device="cuda")
        with pytest.raises(WQError) as ei:
            run_gpu(wq, p, DECODE)
        assert ei.value.status == Status.ERR_UNSUPPORTED


def test_workspace_reused_across_grids_and_status_stays_clear(wq):
    """One zeroed workspace, decode calls whose cluster counts differ (1 tile, many
    tiles, one stage of K): every call must see the grid counters at zero."""
    shapes = [(8, 4096, 256), (8, 4096, 8192), (3, 64, 512), (16, 2048, 4096), (1, 512, 256)]
    ws = torch.zeros(16 << 20, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for i, (M, K, N) in enumerate(shapes):
            p = inputs.make_problem(M_shape=(M,), K=K, N=N, dtype=torch.bfloat16, wbits=4,
                                    mode="group", group=128 if K > 128 else 32,
                                    seed=100 * rep + i, device="cuda",
                                    name=f"reuse_{M}x{K}x{N}")
            y, no = run_gpu(wq, p, DECODE, workspace=ws)
            compare(p, y, no, run_oracle(p))
            assert wq.read_device_status(ws) == 0
    assert int(ws[:2048].cpu().view(torch.int32).abs().sum()) == 0  # header back at zero


def test_decode_back_to_back_on_one_stream_in_a_graph(wq):
    """Captured calls launched with programmatic dependent launch: call i+1 may start
    while call i drains; the results must equal the eager ones bit for bit."""
    p = inputs.decode("cuda")
    w = gpu_weight(wq, p)
    ys = [torch.empty_like(p.residual) for _ in range(4)]
    ns = [torch.empty_like(p.residual) for _ in range(4)]
    ws = torch.zeros(16 << 20, dtype=torch.uint8, device="cuda")
    ey, en = run_gpu(wq, p, DECODE, w=w, workspace=ws)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(4):
                wq.matmul_add_rmsnorm(p.x1, w, p.scale, p.offset, p.bias, p.residual, p.gamma,
                                      p.eps, p.group, y=ys[i], normOut=ns[i], workspace=ws,
                                      kernel=DECODE, stream=s)
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    for i in range(4):
        assert torch.equal(ys[i], ey) and torch.equal(ns[i], en)
    assert wq.read_device_status(ws) == 0
