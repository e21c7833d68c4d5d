"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: byte literals and an
exhaustive nibble round trip for the pack, numpy's matmul for the plain-matmul
special case, closed forms for RMSNorm, identities between the antiquant modes,
and the hand-worked 2 x 32 x 2 case in tests/golden/. A plausible slip in the
oracle -- a swapped nibble, a wrong group index r(k), an offset added before
scaling, a dropped bias, 1/N replaced by 1/K, eps outside the sqrt, a transposed
operand -- fails at least one of them.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pack_literals():
    rows = []
    with open(os.path.join(GOLDEN, "pack_literals.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, rest = line.split(None, 1)
            vals, out = rest.split("->")
            rows.append((kind, [int(v) for v in vals.split()], out.split()))
    return rows


# --------------------------------------------------------------------------- pack

@pytest.mark.parametrize("kind,vals,out", _read_pack_literals())
def test_pack_literals(kind, vals, out):
    b = oracle.pack_int4(np.array([vals], dtype=np.int32))
    if kind == "bytes":
        assert [f"{x:02x}" for x in b[0]] == out
    else:
        assert b.shape == (1, 4)
        assert f"{int(b.view('<u4')[0, 0]):08x}" == out[0]


def test_pack_exhaustive_pairs_is_a_bijection():
    a, b = np.meshgrid(np.arange(-8, 8), np.arange(-8, 8), indexing="ij")
    v = np.stack([a.ravel(), b.ravel()], axis=1).astype(np.int32)  # 256 rows of (a, b)
    packed = oracle.pack_int4(v)
    assert packed.shape == (256, 1)
    assert sorted(packed[:, 0].tolist()) == list(range(256))  # every byte exactly once
    np.testing.assert_array_equal(oracle.unpack_int4(packed, 2), v)
    # the low nibble carries the even column: (a, 0) and (0, b) land in disjoint bits
    for x in range(-8, 8):
        assert oracle.pack_int4(np.array([[x, 0]], np.int32))[0, 0] < 16
        assert oracle.pack_int4(np.array([[0, x]], np.int32))[0, 0] % 16 == 0


def test_pack_roundtrip_random_and_int32_view():
    rng = np.random.default_rng(7)
    v = rng.integers(-8, 8, size=(37, 64), dtype=np.int32)
    b = oracle.pack_int4(v)
    assert b.shape == (37, 32)
    np.testing.assert_array_equal(oracle.unpack_int4(b, 64), v)
    # the (K, N/8) little-endian int32 view holds element 8i+t at bits 4t+3:4t
    u = b.view("<u4")
    for i in range(8):
        for t in range(8):
            nib = (u[:, i] >> (4 * t)) & 0xF
            expect = v[:, 8 * i + t] & 0xF
            np.testing.assert_array_equal(nib, expect)


def _read_tiled_literals():
    rows = []
    with open(os.path.join(GOLDEN, "tiled_literals.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            K, N, k, n, v = (int(x) for x in lhs.split())
            bi, bv = rhs.split()
            rows.append((K, N, k, n, v, int(bi), int(bv, 16)))
    return rows


@pytest.mark.parametrize("K,N,k,n,v,byte,value", _read_tiled_literals())
def test_tiled_pack_literals(K, N, k, n, v, byte, value):
    w = np.zeros((K, N), dtype=np.int32)
    w[k, n] = v
    b = oracle.pack_int4_tiled(w)
    assert b.size == (K + 63) // 64 * 64 * N // 2
    assert np.nonzero(b)[0].tolist() == [byte]
    assert int(b[byte]) == value


def test_tiled_roundtrip_and_same_nibbles_as_nd():
    rng = np.random.default_rng(11)
    for K, N in ((64, 16), (100, 48), (130, 32), (1, 16)):
        v = rng.integers(-8, 8, size=(K, N), dtype=np.int32)
        t = oracle.pack_int4_tiled(v)
        np.testing.assert_array_equal(oracle.unpack_int4_tiled(t, K, N), v)
        # a permutation of the ND pack's nibbles, padded with zero nibbles
        nd = oracle.pack_int4(v).reshape(-1)
        nib = lambda b: np.sort(np.concatenate([b & 0xF, b >> 4]))
        pad = t.size * 2 - nd.size * 2
        np.testing.assert_array_equal(nib(t), np.sort(np.concatenate([nib(nd), np.zeros(pad, np.uint8)])))


def test_tiled_layout_feeds_the_m16n8k16_fragments():
    """What the layout is for: lane l's word j of a tile is the A fragment
    (A = W^T, 16 columns x 16 k) of the tile's MMA j, in the PTX ISA's m16n8k16
    register map -- a0 = A[g][2t..2t+1], a1 = A[g+8][2t..], a2 = A[g][2t+8..],
    a3 = A[g+8][2t+8..], register i holding nibble i (low half) and nibble i+4
    (high half) -- when MMA j's k index kk maps to k-row 32(j/2) + 4(j%2) + 8t +
    e with e = kk % 2 (kk < 8) or 2 + kk % 2 (kk >= 8). Summing the four MMAs of
    a tile must then give W_tile^T @ x for any x."""
    rng = np.random.default_rng(5)
    K, N = 64, 32
    v = rng.integers(-8, 8, size=(K, N), dtype=np.int32)
    x = rng.standard_normal((K, 8))
    tb = oracle.pack_int4_tiled(v)
    for c in range(N // 16):
        tile = tb[c * 512:(c + 1) * 512].reshape(32, 4, 4)  # lane, word, byte
        out = np.zeros((16, 8))
        for j in range(4):
            A = np.zeros((16, 16))
            Bm = np.zeros((16, 8))
            for lane in range(32):
                g, t = lane // 4, lane % 4
                w = int.from_bytes(bytes(tile[lane, j]), "little")
                nib = [(w >> (4 * i)) & 0xF for i in range(8)]
                sv = [q - 16 if q >= 8 else q for q in nib]
                A[g, 2 * t], A[g, 2 * t + 1] = sv[0], sv[4]
                A[g + 8, 2 * t], A[g + 8, 2 * t + 1] = sv[1], sv[5]
                A[g, 2 * t + 8], A[g, 2 * t + 9] = sv[2], sv[6]
                A[g + 8, 2 * t + 8], A[g + 8, 2 * t + 9] = sv[3], sv[7]
                base = 32 * (j // 2) + 4 * (j % 2) + 8 * t
                for e, kk in ((0, 2 * t), (1, 2 * t + 1), (2, 2 * t + 8), (3, 2 * t + 9)):
                    Bm[kk] = x[base + e]
            out += A @ Bm
        np.testing.assert_allclose(out, v[:, 16 * c:16 * c + 16].T.astype(float) @ x, atol=1e-9)


def test_tiled_rejects_n_not_multiple_of_16():
    with pytest.raises(ValueError):
        oracle.pack_int4_tiled(np.zeros((64, 24), np.int32))


def _read_dq_literals():
    rows = []
    with open(os.path.join(GOLDEN, "dynamic_quant_literals.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, xs, qs, frac = (part.strip() for part in line.split("|"))
            num, den = frac.split("/")
            rows.append((int(bits), [float(v) for v in xs.split()], [int(v) for v in qs.split()],
                         float(np.float32(float(num)) / np.float32(float(den)))))
    return rows


@pytest.mark.parametrize("bits,xs,qs,scale", _read_dq_literals())
def test_dynamic_quant_literals(bits, xs, qs, scale):
    q, s = oracle.dynamic_quant(np.array([xs], np.float32), bits=bits)
    assert q[0].tolist() == qs
    assert s[0] == np.float32(scale)


@pytest.mark.parametrize("bits", [8, 4])
def test_dynamic_quant_properties(bits):
    """Codes within [-qmax, qmax]; the row maximum maps to +-qmax; every element
    is reconstructed within half a step; scaling a row by 2^k leaves the codes and
    multiplies the scale by 2^k (exact in fp32); smooth scales act per column."""
    qmax = 127 if bits == 8 else 7
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 200)) * rng.uniform(0.01, 100, (64, 1))).astype(np.float16)
    xf = x.astype(np.float32)
    q, s = oracle.dynamic_quant(x, bits=bits)
    assert np.abs(q).max() <= qmax
    amax_idx = np.abs(xf).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(64), amax_idx]) == qmax)
    err = np.abs(q.astype(np.float64) * s[:, None] - xf)
    assert np.all(err <= s[:, None] * (0.5 + 1e-5))
    q2, s2 = oracle.dynamic_quant(xf * 2.0 ** 7, bits=bits)
    assert np.array_equal(q2, q) and np.array_equal(s2, s * np.float32(2.0 ** 7))
    sm = rng.uniform(0.5, 2.0, 200).astype(np.float32)
    q3, s3 = oracle.dynamic_quant(x, smooth=sm, bits=bits)
    q4, s4 = oracle.dynamic_quant(xf * sm[None, :], bits=bits)
    assert np.array_equal(q3, q4) and np.array_equal(s3, s4)


def _read_fp4_literals():
    rows = []
    with open(os.path.join(GOLDEN, "fp4_literals.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            vals, out = line.split("->")
            rows.append(([float(v) for v in vals.split()], int(out, 16)))
    return rows


@pytest.mark.parametrize("vals,byte", _read_fp4_literals())
def test_fp4_pack_literals(vals, byte):
    assert int(oracle.pack_fp4(np.array([vals], np.float32))[0, 0]) == byte


def test_fp4_codes_round_trip_and_midpoints():
    mags = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    for c in range(16):
        v = (-1 if c & 8 else 1) * mags[c & 7]
        if c == 8:
            v = -0.0
        b = oracle.pack_fp4(np.array([[v, 0.0]], np.float32))[0, 0]
        assert b & 15 == c and b >> 4 == 0
    for i in range(7):  # a midpoint goes to the neighbour with the even code
        mid = (mags[i] + mags[i + 1]) / 2
        b = oracle.pack_fp4(np.array([[mid, 0.0]], np.float32))[0, 0]
        assert b & 15 == (i if i % 2 == 0 else i + 1)


def _fp4_decode(b, n):
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    lo, hi = b & 15, b >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(b.shape[0], -1)[:, :n]
    return np.where(codes & 8, -1.0, 1.0) * mags[codes & 7]


def _mx_problem(M, K, N, seed, scale_spread=4):
    rng = np.random.default_rng(seed)
    x1 = oracle.pack_fp4(rng.uniform(-6, 6, (M, K)).astype(np.float32))
    x2 = oracle.pack_fp4(rng.uniform(-6, 6, (K, N)).astype(np.float32))
    J = (K + 31) // 32
    s1 = rng.integers(127 - scale_spread, 128 + scale_spread, (M, J)).astype(np.uint8)
    s2 = rng.integers(127 - scale_spread, 128 + scale_spread, (J, N)).astype(np.uint8)
    y = rng.standard_normal((M, N))
    return x1, s1, x2, s2, y


def test_mx_matmul_unit_scales_is_a_plain_matmul():
    M, K, N = 5, 96, 6
    x1, s1, x2, s2, y = _mx_problem(M, K, N, 1)
    s1[:] = 127
    s2[:] = 127
    out = oracle.mx_matmul_add(x1, s1, x2, s2, y, K)
    ref = _fp4_decode(x1, K) @ _fp4_decode(x2, N) + y
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-9)


def test_mx_matmul_scales_act_per_slice_and_short_last_slice():
    """K = 40: slices [0, 32) and [32, 40). Each slice's contribution is its plain
    product times 2^(s1 - 127) * 2^(s2 - 127); changing one scale changes only its
    slice, by the power of two."""
    M, K, N = 3, 40, 4
    x1, s1, x2, s2, y = _mx_problem(M, K, N, 2)
    a, b = _fp4_decode(x1, K), _fp4_decode(x2, N)
    ref = y.copy()
    for j, (k0, k1) in enumerate(((0, 32), (32, 40))):
        ref += (a[:, k0:k1] @ b[k0:k1, :]) * np.exp2(s1[:, j:j + 1].astype(float) - 127) \
            * np.exp2(s2[j:j + 1, :].astype(float) - 127)
    np.testing.assert_allclose(oracle.mx_matmul_add(x1, s1, x2, s2, y, K), ref, rtol=1e-12, atol=1e-12)


def test_mx_matmul_hand_worked():
    """x1 = [[1, -0.5]], x2 = [[2, 3], [4, -6]], one slice (K = 2), scale1 = 2^1,
    scale2 = [2^0, 2^-1], y = [[10, 20]]: row products (1*2 - 0.5*4, 1*3 + 0.5*6)
    = (0, 6), times 2 * (1, 0.5) = (0, 6), plus y = (10, 26)."""
    x1 = oracle.pack_fp4(np.array([[1, -0.5]], np.float32))
    x2 = oracle.pack_fp4(np.array([[2, 3], [4, -6]], np.float32))
    s1 = np.array([[128]], np.uint8)
    s2 = np.array([[127, 126]], np.uint8)
    out = oracle.mx_matmul_add(x1, s1, x2, s2, np.array([[10.0, 20.0]]), 2)
    assert out.tolist() == [[10.0, 26.0]]


def test_pack_rejects_odd_n():
    with pytest.raises(ValueError):
        oracle.pack_int4(np.zeros((2, 3), np.int32))


# --------------------------------------------------------------------------- helpers

def _rand_problem(rng, M, K, N, mode, g=0, with_offset=True, with_bias=True):
    x = rng.standard_normal((M, K))
    q = rng.integers(-8, 8, size=(K, N)).astype(np.int32)
    if mode == "tensor":
        S = rng.uniform(0.002, 0.01, size=(1,))
    elif mode == "channel":
        S = rng.uniform(0.002, 0.01, size=(N,))
    else:
        S = rng.uniform(0.002, 0.01, size=((K + g - 1) // g, N))
    O = rng.uniform(-0.02, 0.02, size=S.shape) if with_offset else None
    b = rng.normal(0, 0.05, size=(N,)) if with_bias else None
    r = rng.standard_normal((M, N))
    gm = rng.uniform(0.5, 1.5, size=(N,))
    return x, q, S, O, b, r, gm


def _numpy_formula(x, q, S, O, b, r, gm, eps, g):
    """Vectorised restatement with library primitives (np.repeat, matmul, mean)."""
    K, N = q.shape
    S2 = S.reshape(1, -1) if S.ndim == 1 else S
    Sf = np.repeat(S2, g, axis=0)[:K] if g else S2
    Sf = np.broadcast_to(Sf, (K, N))
    if O is not None:
        O2 = O.reshape(1, -1) if O.ndim == 1 else O
        Of = np.broadcast_to(np.repeat(O2, g, axis=0)[:K] if g else O2, (K, N))
    else:
        Of = 0.0
    W = q * Sf + Of
    mm = x @ W + (0.0 if b is None else b)
    y = mm + r
    no = y / np.sqrt(np.mean(y * y, axis=1, keepdims=True) + eps) * gm
    return mm, y, no


# --------------------------------------------------------------------------- matmul core

def test_plain_matmul_special_case_is_exact():
    """S = 1, O = 0, bias = 0, residual = 0 reduces mm to x1 @ q; with integer x1
    every partial sum is an exact fp64 integer, so the match is exact."""
    rng = np.random.default_rng(1)
    M, K, N = 5, 96, 24
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float64)
    q = rng.integers(-8, 8, size=(K, N)).astype(np.int32)
    mm, y, _ = oracle.matmul_add_rmsnorm(x, q, np.ones(1), None, None, np.zeros((M, N)),
                                         np.ones(N), 1e-6)
    np.testing.assert_array_equal(mm, x @ q.astype(np.float64))
    np.testing.assert_array_equal(y, mm)


def test_plain_matmul_float_inputs():
    rng = np.random.default_rng(2)
    M, K, N = 7, 200, 33
    x = rng.standard_normal((M, K))
    q = rng.integers(-128, 128, size=(K, N)).astype(np.int32)
    mm, _, _ = oracle.matmul_add_rmsnorm(x, q, np.ones(1), None, None, np.zeros((M, N)),
                                         np.ones(N), 0.0)
    np.testing.assert_allclose(mm, x @ q, rtol=1e-12, atol=1e-9)


def test_not_transposed():
    """A non-square problem where x1 @ q and x1 @ q.T-like mixups cannot both fit."""
    x = np.zeros((1, 3)); x[0, 2] = 1.0          # picks row k=2 of q
    q = np.arange(3 * 4, dtype=np.int32).reshape(3, 4) - 6
    mm, _, _ = oracle.matmul_add_rmsnorm(x, q, np.ones(1), None, None, np.zeros((1, 4)),
                                         np.ones(4), 0.0)
    np.testing.assert_array_equal(mm[0], q[2].astype(np.float64))


# --------------------------------------------------------------------------- antiquant modes

def test_dequant_group_index_and_offset_order():
    """r(k) = floor(k/g) and W = q*S + O (offset after scaling)."""
    K, N, g = 70, 3, 32                       # 3 groups, the last one short (6 rows)
    q = np.full((K, N), 2, np.int32)
    S = np.array([[1.0, 2.0, 3.0], [10.0, 20.0, 30.0], [100.0, 200.0, 300.0]])
    O = np.array([[0.5, 0.5, 0.5], [0.25, 0.25, 0.25], [0.125, 0.125, 0.125]])
    W = oracle.dequant(q, S, O, group=g)
    for k in range(K):
        r = k // 32
        np.testing.assert_array_equal(W[k], 2 * S[r] + O[r])
    assert W[31, 0] == 2.5 and W[32, 0] == 20.25 and W[64, 0] == 200.125 and W[69, 2] == 600.125


def test_group_equal_k_is_per_channel():
    rng = np.random.default_rng(3)
    x, q, S, O, b, r, gm = _rand_problem(rng, 4, 64, 16, "channel")
    ch = oracle.matmul_add_rmsnorm(x, q, S, O, b, r, gm, 1e-6)
    gr = oracle.matmul_add_rmsnorm(x, q, S.reshape(1, -1), O.reshape(1, -1), b, r, gm, 1e-6,
                                   group=64)
    for a, c in zip(ch, gr):
        np.testing.assert_array_equal(a, c)


def test_group_identical_rows_is_per_channel():
    rng = np.random.default_rng(4)
    x, q, S, O, b, r, gm = _rand_problem(rng, 3, 96, 8, "channel")
    Sg = np.tile(S, (3, 1)); Og = np.tile(O, (3, 1))
    ch = oracle.matmul_add_rmsnorm(x, q, S, O, b, r, gm, 1e-6)
    gr = oracle.matmul_add_rmsnorm(x, q, Sg, Og, b, r, gm, 1e-6, group=32)
    for a, c in zip(ch, gr):
        np.testing.assert_array_equal(a, c)


def test_constant_channel_is_per_tensor():
    rng = np.random.default_rng(5)
    x, q, _, _, b, r, gm = _rand_problem(rng, 3, 40, 12, "tensor")
    ten = oracle.matmul_add_rmsnorm(x, q, np.array([0.0075]), np.array([-0.01]), b, r, gm, 1e-6)
    ch = oracle.matmul_add_rmsnorm(x, q, np.full(12, 0.0075), np.full(12, -0.01), b, r, gm, 1e-6)
    for a, c in zip(ten, ch):
        np.testing.assert_array_equal(a, c)


@pytest.mark.parametrize("mode,g", [("channel", 0), ("group", 32)])
def test_offset_linearity(mode, g):
    """Adding O adds sum over each group of x1 times O to mm."""
    rng = np.random.default_rng(6)
    M, K, N = 4, 96, 10
    x, q, S, O, b, r, gm = _rand_problem(rng, M, K, N, mode, g)
    with_o = oracle.matmul_add_rmsnorm(x, q, S, O, b, r, gm, 1e-6, group=g)[0]
    without = oracle.matmul_add_rmsnorm(x, q, S, None, b, r, gm, 1e-6, group=g)[0]
    if g:
        expect = sum(x[:, j * g:(j + 1) * g].sum(1)[:, None] * O[j][None, :]
                     for j in range(O.shape[0]))
    else:
        expect = x.sum(1)[:, None] * O[None, :]
    np.testing.assert_allclose(with_o - without, expect, rtol=1e-9, atol=1e-12)


def test_bias_is_added_once():
    rng = np.random.default_rng(8)
    x, q, S, O, b, r, gm = _rand_problem(rng, 2, 32, 6, "channel")
    a = oracle.matmul_add_rmsnorm(x, q, S, O, b, r, gm, 1e-6)[0]
    c = oracle.matmul_add_rmsnorm(x, q, S, O, None, r, gm, 1e-6)[0]
    np.testing.assert_allclose(a - c, np.broadcast_to(b, a.shape), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode,g,K", [("tensor", 0, 64), ("channel", 0, 100), ("group", 32, 100),
                                      ("group", 64, 256)])
def test_matches_vectorised_restatement(mode, g, K):
    rng = np.random.default_rng(9 + K)
    x, q, S, O, b, r, gm = _rand_problem(rng, 6, K, 20, mode, g)
    got = oracle.matmul_add_rmsnorm(x, q, S, O, b, r, gm, 1e-5, group=g)
    exp = _numpy_formula(x, q, S, O, b, r, gm, 1e-5, g)
    for a, c in zip(got, exp):
        np.testing.assert_allclose(a, c, rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_row_closed_form():
    """x1 = 0, no bias: y = residual; a constant row c gives c / sqrt(c^2 + eps) * gamma."""
    N, eps = 16, 0.25
    gm = np.linspace(0.5, 1.5, N)
    r = np.stack([np.full(N, 3.0), np.full(N, -0.5)])
    _, y, no = oracle.matmul_add_rmsnorm(np.zeros((2, 32)), np.ones((32, N), np.int32),
                                         np.ones(1), None, None, r, gm, eps)
    np.testing.assert_array_equal(y, r)
    np.testing.assert_allclose(no[0], 3.0 / np.sqrt(9.0 + eps) * gm, rtol=1e-15)
    np.testing.assert_allclose(no[1], -0.5 / np.sqrt(0.25 + eps) * gm, rtol=1e-15)


def test_rmsnorm_unit_rms_as_eps_vanishes():
    rng = np.random.default_rng(10)
    x, q, S, O, b, r, gm = _rand_problem(rng, 5, 64, 40, "group", 32)
    for eps in (1e-2, 1e-6, 0.0):
        _, y, no = oracle.matmul_add_rmsnorm(x, q, S, O, b, r, gm, eps, group=32)
        with np.errstate(over="ignore"):  # a planted mistake may blow y up; the check still fails
            ms = np.mean(y * y, axis=1)
        rms = np.sqrt(np.mean((no / gm) ** 2, axis=1))
        np.testing.assert_allclose(rms, 1.0 / np.sqrt(1.0 + eps / ms), rtol=1e-12)
    np.testing.assert_allclose(rms, 1.0, rtol=1e-12)


def test_rmsnorm_uses_n_not_k():
    """mean(y^2) runs over N (the last dim of y), not K: a row of N ones with eps=0
    normalises to exactly gamma whatever K is."""
    for K in (32, 96):
        N = 8
        _, _, no = oracle.matmul_add_rmsnorm(np.zeros((1, K)), np.ones((K, N), np.int32),
                                             np.ones(1), None, None, np.ones((1, N)),
                                             np.arange(1, N + 1, dtype=np.float64), 0.0)
        np.testing.assert_array_equal(no[0], np.arange(1, N + 1))


def test_row_scaling_invariance():
    rng = np.random.default_rng(11)
    x, q, S, O, _, r, gm = _rand_problem(rng, 3, 64, 24, "channel", with_offset=False,
                                         with_bias=False)
    a = oracle.matmul_add_rmsnorm(x, q, S, None, None, r, gm, 0.0)
    c = oracle.matmul_add_rmsnorm(4.0 * x, q, S, None, None, 4.0 * r, gm, 0.0)
    np.testing.assert_allclose(c[1], 4.0 * a[1], rtol=1e-14)
    np.testing.assert_allclose(c[2], a[2], rtol=1e-13)


def test_row_permutation_equivariance_and_sampling():
    rng = np.random.default_rng(12)
    x, q, S, O, b, r, gm = _rand_problem(rng, 9, 64, 16, "group", 32)
    full = oracle.matmul_add_rmsnorm(x, q, S, O, b, r, gm, 1e-6, group=32)
    perm = rng.permutation(9)
    pm = oracle.matmul_add_rmsnorm(x[perm], q, S, O, b, r[perm], gm, 1e-6, group=32)
    sub = oracle.matmul_add_rmsnorm(x, q, S, O, b, r, gm, 1e-6, group=32, rows=[8, 0, 3])
    for f, p, s in zip(full, pm, sub):
        np.testing.assert_array_equal(p, f[perm])
        np.testing.assert_array_equal(s, f[[8, 0, 3]])


# --------------------------------------------------------------------------- hand-worked case

def _golden_hand():
    vals = {}
    with open(os.path.join(GOLDEN, "hand_2x32x2.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, *nums = line.split()
                vals[key] = [float(v) for v in nums]
    D = np.array(vals["D"]).reshape(2, 2)
    H = np.array(vals["H"]).reshape(2, 2)
    return D, H, np.array(vals["ROWSUM"]), np.array(vals["ROWSUM_HALF"])


def _hand_inputs():
    x = np.ones((2, 32)); x[1, 1::2] = -1.0
    q = np.zeros((32, 2), np.int32); q[:, 0] = 7; q[:, 1] = np.arange(32) % 16 - 8
    return x, q


def _rms_closed(y, gm, eps):
    return y / np.sqrt((y ** 2).sum(1, keepdims=True) / 2 + eps) * gm


@pytest.mark.parametrize("with_offset,with_bias", [(False, False), (True, False), (True, True),
                                                   (False, True)])
def test_hand_worked_per_tensor(with_offset, with_bias):
    D, _, rs, _ = _golden_hand()
    x, q = _hand_inputs()
    s, o = 0.5, (0.25 if with_offset else 0.0)
    b = np.array([1.0, -2.0]) if with_bias else np.zeros(2)
    r = np.array([[0.5, -1.0], [2.0, 0.125]])
    gm = np.array([1.0, 0.5]); eps = 0.0625
    mm, y, no = oracle.matmul_add_rmsnorm(x, q, np.array([s]),
                                          np.array([o]) if with_offset else None,
                                          b if with_bias else None, r, gm, eps)
    exp_mm = s * D + o * rs[:, None] + b[None, :]
    np.testing.assert_array_equal(mm, exp_mm)
    np.testing.assert_array_equal(y, exp_mm + r)
    np.testing.assert_allclose(no, _rms_closed(exp_mm + r, gm, eps), rtol=1e-15)


@pytest.mark.parametrize("with_offset,with_bias", [(False, False), (True, True)])
def test_hand_worked_per_channel(with_offset, with_bias):
    D, _, rs, _ = _golden_hand()
    x, q = _hand_inputs()
    s = np.array([0.5, 0.125]); o = np.array([0.25, -0.75]) if with_offset else np.zeros(2)
    b = np.array([1.0, -2.0]) if with_bias else np.zeros(2)
    r = np.zeros((2, 2)); gm = np.array([2.0, 1.0]); eps = 1.0
    mm, y, no = oracle.matmul_add_rmsnorm(x, q, s, o if with_offset else None,
                                          b if with_bias else None, r, gm, eps)
    exp_mm = s[None, :] * D + rs[:, None] * o[None, :] + b[None, :]
    np.testing.assert_array_equal(mm, exp_mm)
    np.testing.assert_allclose(no, _rms_closed(exp_mm, gm, eps), rtol=1e-15)


def test_hand_worked_per_group_g16():
    """Oracle-only: g = 16 splits K = 32 into two halves with separate scales/offsets."""
    _, H, _, rsh = _golden_hand()
    x, q = _hand_inputs()
    S = np.array([[0.5, 0.25], [2.0, 4.0]]); O = np.array([[0.125, -0.5], [1.0, 0.0625]])
    b = np.array([0.5, 0.5]); r = np.array([[1.0, 1.0], [-1.0, 0.0]]); gm = np.ones(2)
    mm, y, no = oracle.matmul_add_rmsnorm(x, q, S, O, b, r, gm, 0.5, group=16)
    exp_mm = (S[0][None, :] * H + rsh[:, None] * O[0][None, :]
              + S[1][None, :] * H + rsh[:, None] * O[1][None, :] + b[None, :])
    np.testing.assert_array_equal(mm, exp_mm)
    np.testing.assert_allclose(no, _rms_closed(exp_mm + r, gm, 0.5), rtol=1e-15)
