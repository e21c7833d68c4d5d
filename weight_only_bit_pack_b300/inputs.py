"""Seeded synthetic inputs for the weight-only quantized matmul + AddRmsNorm.

This module only draws random tensors; it holds none of the operator's
arithmetic, so both the CUDA path (through the tests and the bench) and the
fp64 oracle can be fed from it. Nothing here packs, dequantizes or multiplies.

Recipe (one ``torch.Generator`` per problem, seeded as given, on the device the
tensors are made on):
  * continuous U[a, b] = a + (b - a) * rand, N(0, s) = s * randn, both drawn in
    fp32 and then cast (round to nearest even) to the problem's dtype;
  * integer weights uniform[lo, hi] = randint(lo, hi + 1); INT4 weights are
    returned unpacked as int32 (K, N) values in [-8, 7] -- the pack kernel turns
    them into bytes;
  * draw order x1, x2, scale, offset, bias, residual, gamma; the M-sweep draws
    the weight side (x2, scale, offset, bias, gamma) from a generator seeded
    ``seed`` so the weights are the same for every M, and the activation side
    (x1, residual) from a second generator seeded ``seed * 1000 + M``.

The named workloads are the ones the operator is measured on: a tiny fp16
case, a bf16 decode step (M = 8), an fp16 W8A16 per-channel layer, a bf16
prefill with per-group offsets and an M-sweep over a 8192 x 28672 INT4 layer.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class Problem:
    name: str
    dtype: torch.dtype          # activation dtype (x1, scale, offset, bias, residual, gamma)
    wbits: int                  # 4 or 8
    x1: torch.Tensor            # (M, K) or (b, s, K)
    x2: torch.Tensor            # int32 (K, N) values in [-8, 7] for INT4; int8 (K, N) for INT8
    scale: torch.Tensor         # (1) | (N) | (G, N)
    offset: Optional[torch.Tensor]
    bias: Optional[torch.Tensor]
    residual: torch.Tensor      # (M, N) or (b, s, N)
    gamma: torch.Tensor         # (N)
    eps: float
    group: int                  # 0 unless per-group
    meta: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        n = 1
        for d in self.x1.shape[:-1]:
            n *= d
        return n

    @property
    def K(self) -> int:
        return self.x1.shape[-1]

    @property
    def N(self) -> int:
        return self.x2.shape[1]


def _u(g, shape, a, b, dtype, device):
    return (a + (b - a) * torch.rand(shape, generator=g, device=device, dtype=torch.float32)).to(dtype)


def _n(g, shape, s, dtype, device):
    return (s * torch.randn(shape, generator=g, device=device, dtype=torch.float32)).to(dtype)


def _ri(g, shape, lo, hi, device, dtype=torch.int32):
    return torch.randint(lo, hi + 1, shape, generator=g, device=device, dtype=torch.int64).to(dtype)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_problem(*, M_shape, K, N, dtype, wbits, mode, group=0, offset=True, bias=True,
                 seed=0, eps=1e-6, device="cpu", x_sigma=1.0, scale_range=(0.002, 0.01),
                 offset_range=(-0.02, 0.02), bias_sigma=0.05, name="custom",
                 x_int_range=None) -> Problem:
    """General recipe. ``mode`` is 'tensor' (scale (1)), 'channel' (scale (N)),
    'channel2d' (scale (1, N)) or 'group' (scale (ceil(K/group), N)).
    ``x_int_range=(lo, hi)`` draws integer-valued x1 instead of N(0, x_sigma)."""
    g = _gen(seed, device)
    xs = tuple(M_shape) + (K,)
    if x_int_range is not None:
        x1 = _ri(g, xs, x_int_range[0], x_int_range[1], device).to(dtype)
    else:
        x1 = _n(g, xs, x_sigma, dtype, device)
    if wbits == 4:
        x2 = _ri(g, (K, N), -8, 7, device, torch.int32)
    else:
        x2 = _ri(g, (K, N), -128, 127, device, torch.int8)
    if mode == "tensor":
        sshape = (1,)
    elif mode == "channel":
        sshape = (N,)
    elif mode == "channel2d":
        sshape = (1, N)
    elif mode == "group":
        sshape = ((K + group - 1) // group, N)
    else:
        raise ValueError(mode)
    scale = _u(g, sshape, scale_range[0], scale_range[1], dtype, device)
    off = _u(g, sshape, offset_range[0], offset_range[1], dtype, device) if offset else None
    b = _n(g, (N,), bias_sigma, dtype, device) if bias else None
    residual = _n(g, tuple(M_shape) + (N,), 1.0, dtype, device)
    gamma = _u(g, (N,), 0.5, 1.5, dtype, device)
    return Problem(name, dtype, wbits, x1, x2, scale, off, b, residual, gamma, float(eps),
                   int(group) if mode == "group" else 0, {"seed": seed})


SWEEP_M = (1, 16, 64, 256, 1024, 4096, 16384)


def tiny(device="cpu") -> Problem:
    """16 x 256 x 128, fp16, INT4, per-group g=32 with offset and bias, seed 0."""
    return make_problem(M_shape=(16,), K=256, N=128, dtype=torch.float16, wbits=4, mode="group",
                        group=32, offset=True, bias=True, seed=0, eps=1e-6, device=device,
                        scale_range=(0.005, 0.02), offset_range=(-0.05, 0.05), bias_sigma=0.1,
                        name="tiny_fp16_w4_g32")


def decode(device="cpu") -> Problem:
    """M=8 (1 x 8) x 4096 x 4096, bf16, INT4, per-group g=128, no offset, seed 1."""
    return make_problem(M_shape=(1, 8), K=4096, N=4096, dtype=torch.bfloat16, wbits=4, mode="group",
                        group=128, offset=False, bias=True, seed=1, eps=1e-6, device=device,
                        scale_range=(0.002, 0.01), bias_sigma=0.05, name="decode_w4a16_bf16_g128")


def w8a16(device="cpu") -> Problem:
    """2048 x 4096 x 11008, fp16, INT8, per-channel scale + offset, no bias, seed 2."""
    return make_problem(M_shape=(2048,), K=4096, N=11008, dtype=torch.float16, wbits=8,
                        mode="channel", offset=True, bias=False, seed=2, eps=1e-5, device=device,
                        scale_range=(0.0005, 0.002), offset_range=(-0.01, 0.01),
                        name="w8a16_fp16_perchannel")


def prefill(device="cpu") -> Problem:
    """(4 x 2048) x 8192 x 8192, bf16, INT4, per-group g=64 with offset and bias, seed 3."""
    return make_problem(M_shape=(4, 2048), K=8192, N=8192, dtype=torch.bfloat16, wbits=4,
                        mode="group", group=64, offset=True, bias=True, seed=3, eps=1e-6,
                        device=device, scale_range=(0.002, 0.01), offset_range=(-0.02, 0.02),
                        bias_sigma=0.05, name="prefill_w4a16_bf16_g64_offset")


def sweep(M: int, per_tensor: bool = False, device="cpu") -> Problem:
    """M x 8192 x 28672, bf16, INT4, per-group g=128 (or per-tensor scale), no offset.
    Weight side seeded 4 (5 for the per-tensor variant), activations seeded seed*1000+M."""
    K, N = 8192, 28672
    seed = 5 if per_tensor else 4
    gw = _gen(seed, device)
    x2 = _ri(gw, (K, N), -8, 7, device, torch.int32)
    if per_tensor:
        scale = _u(gw, (1,), 0.002, 0.01, torch.bfloat16, device)
    else:
        scale = _u(gw, ((K + 127) // 128, N), 0.002, 0.01, torch.bfloat16, device)
    bias = _n(gw, (N,), 0.05, torch.bfloat16, device)
    gamma = _u(gw, (N,), 0.5, 1.5, torch.bfloat16, device)
    ga = _gen(seed * 1000 + M, device)
    x1 = _n(ga, (1, M, K), 1.0, torch.bfloat16, device)
    residual = _n(ga, (1, M, N), 1.0, torch.bfloat16, device)
    name = f"sweep_w4a16_bf16_{'pertensor' if per_tensor else 'g128'}_M{M}"
    return Problem(name, torch.bfloat16, 4, x1, x2, scale, None, bias, residual, gamma, 1e-6,
                   0 if per_tensor else 128, {"seed": seed, "M": M})


CONFIGS = {
    "tiny": tiny,
    "decode": decode,
    "w8a16": w8a16,
    "prefill": prefill,
}
