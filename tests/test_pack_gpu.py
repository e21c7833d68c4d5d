"""INT32 -> INT4 pack kernel vs the oracle pack: bit-exact (GPU)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _pack_both(wq, v_cpu):
    got = wq.pack_int4(v_cpu.cuda())
    torch.cuda.synchronize()
    return got.cpu().numpy(), oracle.pack_int4(v_cpu)


@pytest.mark.parametrize("K,N", [(1, 2), (3, 6), (7, 34), (256, 128), (255, 130), (4096, 4096),
                                 (8192, 8192), (1, 65534)])
def test_pack_matches_oracle(wq, K, N):
    g = torch.Generator().manual_seed(K * 131 + N)
    v = torch.randint(-8, 8, (K, N), generator=g, dtype=torch.int32)
    got, ref = _pack_both(wq, v)
    np.testing.assert_array_equal(got, ref)


def test_pack_full_size_sweep_weight(wq):
    """The 8192 x 28672 weight of the M-sweep, drawn as the workload draws it."""
    from weight_only_bit_pack_b300 import inputs
    g = torch.Generator().manual_seed(4)
    v = torch.randint(-8, 8, (8192, 28672), generator=g, dtype=torch.int32)
    got, ref = _pack_both(wq, v)
    assert np.array_equal(got, ref)
    del inputs


def test_pack_out_of_range_values_keep_low_nibble(wq):
    g = torch.Generator().manual_seed(99)
    v = torch.randint(-2**31, 2**31 - 1, (33, 66), generator=g, dtype=torch.int64).to(torch.int32)
    got, ref = _pack_both(wq, v)
    np.testing.assert_array_equal(got, ref)


def test_pack_unaligned_pointers_use_scalar_path(wq):
    K, N = 37, 50
    g = torch.Generator().manual_seed(5)
    v = torch.randint(-8, 8, (K, N), generator=g, dtype=torch.int32)
    src = torch.empty(K * N + 1, dtype=torch.int32, device="cuda")
    src[1:] = v.cuda().reshape(-1)
    dst = torch.zeros(K * N // 2 + 3, dtype=torch.uint8, device="cuda")
    out = dst[3:].view(K, N // 2)
    wq.pack_int4(src[1:].view(K, N), out=out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.pack_int4(v))
    assert dst[:3].sum().item() == 0  # nothing written before the output


def test_pack_deterministic_and_empty(wq):
    v = torch.randint(-8, 8, (512, 1024), dtype=torch.int32).cuda()
    a = wq.pack_int4(v); b = wq.pack_int4(v)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    e = wq.pack_int4(torch.empty((0, 64), dtype=torch.int32, device="cuda"))
    assert e.shape == (0, 32)
