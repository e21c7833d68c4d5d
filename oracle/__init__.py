"""fp64 CPU oracle for the weight-only quantized matmul + AddRmsNorm and the INT4 pack.

TEST INFRASTRUCTURE ONLY. The arithmetic lives in ``wq_oracle.c`` (plain C,
fp64, OpenMP over n-chunks); this module builds it with gcc, loads it with
ctypes and converts torch/numpy inputs to fp64 (an exact upcast for fp16/bf16).
It shares nothing with the CUDA library and the CUDA library never imports it.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may use it.

Pages followed (Ascend CANN operator docs): ``aclnnConvertWeightToINT4Pack``
(function description: sparse INT32 -> dense INT4, and its option of a
matrix-unit tiled output, for which the library defines its own tiled
layout), ``aclnnDynamicQuant``
(constraints: INT4 packs along the last dimension), and
``aclnnWeightQuantMatmulAllReduceAddRmsNorm`` (function description: formula;
constraints: scale/offset shapes, group size). Every function is pinned by
``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``wq_oracle.c`` into ``liboracle.so`` (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load(path=None):
    global _lib
    if _lib is None or path is not None:
        if path is None:
            build()
        lib = ctypes.CDLL(path or _LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int64
        lib.wqo_pack_int4.argtypes = [P, I, I, P]
        lib.wqo_unpack_int4.argtypes = [P, I, I, P]
        lib.wqo_dequant.argtypes = [P, I, I, P, P, I, I, I, P]
        lib.wqo_matmul_add_rmsnorm.argtypes = [P, I, I, P, I, P, P, I, I, I, P, P, P,
                                               ctypes.c_double, P, P, P]
        lib.wqo_pack_fp4.argtypes = [P, I, I, P]
        lib.wqo_pack_fp4.restype = ctypes.c_int
        lib.wqo_mx_matmul_add.argtypes = [P, P, P, P, I, I, I, P]
        lib.wqo_mx_matmul_add.restype = ctypes.c_int
        lib.wqo_dynamic_quant.argtypes = [P, I, I, P, ctypes.c_int, P, P]
        lib.wqo_dynamic_quant.restype = ctypes.c_int
        lib.wqo_tiled_bytes.argtypes = [I, I]
        lib.wqo_tiled_bytes.restype = I
        lib.wqo_pack_int4_tiled.argtypes = [P, I, I, P]
        lib.wqo_unpack_int4_tiled.argtypes = [P, I, I, P]
        for f in (lib.wqo_pack_int4, lib.wqo_unpack_int4, lib.wqo_dequant,
                  lib.wqo_matmul_add_rmsnorm, lib.wqo_pack_int4_tiled, lib.wqo_unpack_int4_tiled):
            f.restype = ctypes.c_int
        if path is not None:
            return lib
        _lib = lib
    return _lib


class use_library:
    """Context manager that points this module at another build of the oracle
    source (used by the mutation tests, which plant mistakes in a copy of
    ``wq_oracle.c`` and check that the pins catch them)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self._saved = _lib
        _lib = _load(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _f64(a):
    """Exact upcast of a torch tensor / numpy array / scalar list to contiguous fp64."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: fp16/bf16 -> fp64 is exact
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def pack_int4(v) -> np.ndarray:
    """(K, N) int32 -> (K, N/2) uint8; column 2j -> bits 3:0, column 2j+1 -> bits 7:4."""
    v = _i32(v)
    K, N = v.shape
    out = np.empty((K, N // 2), dtype=np.uint8)
    rc = _load().wqo_pack_int4(_p(v), K, N, _p(out))
    if rc:
        raise ValueError(f"wqo_pack_int4 rejected shape {v.shape}")
    return out


def unpack_int4(b, N: int) -> np.ndarray:
    """(K, N/2) uint8 -> (K, N) int32 in [-8, 7]."""
    if hasattr(b, "detach"):
        b = b.detach().to("cpu").numpy()
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint8))
    K = b.shape[0]
    out = np.empty((K, N), dtype=np.int32)
    rc = _load().wqo_unpack_int4(_p(b), K, N, _p(out))
    if rc:
        raise ValueError("wqo_unpack_int4 rejected its shape")
    return out


def pack_int4_tiled(v) -> np.ndarray:
    """(K, N) int32 -> the kernel-native tiled INT4 bytes (N % 16 == 0; K padded to 64
    with zero nibbles), as defined in wq_oracle.c."""
    v = _i32(v)
    K, N = v.shape
    out = np.empty(int(_load().wqo_tiled_bytes(K, N)), dtype=np.uint8)
    rc = _load().wqo_pack_int4_tiled(_p(v), K, N, _p(out))
    if rc:
        raise ValueError(f"wqo_pack_int4_tiled rejected shape {v.shape}")
    return out


def unpack_int4_tiled(b, K: int, N: int) -> np.ndarray:
    """Tiled INT4 bytes -> (K, N) int32 in [-8, 7]."""
    if hasattr(b, "detach"):
        b = b.detach().to("cpu").numpy()
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint8).reshape(-1))
    out = np.empty((K, N), dtype=np.int32)
    rc = _load().wqo_unpack_int4_tiled(_p(b), K, N, _p(out))
    if rc:
        raise ValueError("wqo_unpack_int4_tiled rejected its shape")
    return out


def pack_fp4(v) -> np.ndarray:
    """(K, N) float32 -> (K, N/2) bytes of FP4 E2M1 codes (nearest, ties to the even
    code, saturating at 6), even column in bits 3:0."""
    if hasattr(v, "detach"):
        v = v.detach().to("cpu").float().numpy()
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    K, N = v.shape
    out = np.empty((K, N // 2), dtype=np.uint8)
    if _load().wqo_pack_fp4(_p(v), K, N, _p(out)):
        raise ValueError("wqo_pack_fp4 rejected its shape")
    return out


def mx_matmul_add(x1, s1, x2, s2, y, K: int):
    """y (M, N) fp64 plus the mx block-scaled product of the packed FP4 x1 (M, K/2)
    and x2 (K, N/2) with E8M0 scales s1 (M, ceil(K/32)) and s2 (ceil(K/32), N)."""
    def u8(a):
        if hasattr(a, "detach"):
            a = a.detach().to("cpu").numpy()
        return np.ascontiguousarray(np.asarray(a, dtype=np.uint8))
    x1, s1, x2, s2 = u8(x1), u8(s1), u8(x2), u8(s2)
    yy = _f64(y).copy()
    M, N = yy.shape
    if _load().wqo_mx_matmul_add(_p(x1), _p(s1), _p(x2), _p(s2), M, K, N, _p(yy)):
        raise ValueError("wqo_mx_matmul_add rejected its arguments")
    return yy


def dynamic_quant(x, smooth=None, bits: int = 8):
    """Per-token symmetric quantization of x (..., K) in fp32 arithmetic.
    Returns (codes int8 with x's shape, scale float32 with x's leading shape);
    INT4 codes lie in [-7, 7] (pack them with ``pack_int4``)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    lead, K = x.shape[:-1], x.shape[-1]
    M = int(np.prod(lead)) if lead else 1
    sm = None
    if smooth is not None:
        if hasattr(smooth, "detach"):
            smooth = smooth.detach().to("cpu").float().numpy()
        sm = np.ascontiguousarray(np.asarray(smooth, dtype=np.float32))
    q = np.empty((M, K), dtype=np.int8)
    s = np.empty(M, dtype=np.float32)
    rc = _load().wqo_dynamic_quant(_p(x), M, K, _p(sm), 127 if bits == 8 else 7, _p(q), _p(s))
    if rc:
        raise ValueError("wqo_dynamic_quant rejected its arguments")
    return q.reshape(x.shape), s.reshape(lead)


def _so_shape(S, N):
    """(Gs, Ns) view of a scale/offset array: (1) -> (1,1); (N) -> (1,N); (G,N) stays."""
    if S.ndim == 1:
        return S.reshape(1, -1)
    return S


def dequant(q, scale, offset=None, group: int = 0) -> np.ndarray:
    """W = q * S[r(k), c(n)] + O[r(k), c(n)] in fp64 (q is (K, N) int32)."""
    q = _i32(q)
    K, N = q.shape
    S = _so_shape(_f64(scale), N)
    O = None if offset is None else _so_shape(_f64(offset), N)
    W = np.empty((K, N), dtype=np.float64)
    rc = _load().wqo_dequant(_p(q), K, N, _p(np.ascontiguousarray(S)),
                             _p(None if O is None else np.ascontiguousarray(O)),
                             S.shape[0], S.shape[1], int(group), _p(W))
    if rc:
        raise ValueError("wqo_dequant rejected its arguments")
    return W


def matmul_add_rmsnorm(x1, q, scale, offset, bias, residual, gamma, eps: float,
                       group: int = 0, rows=None):
    """The fused operator in fp64. Returns (mm, y, normOut), each (R, N).

    x1 is (M, K) (or (b, s, K)), q the (K, N) integer weights, residual (M, N)
    (or (b, s, N)). ``rows`` selects a subset of the M rows (rows are
    independent); the outputs then hold those rows in that order.
    """
    x = _f64(x1)
    K = x.shape[-1]
    x = x.reshape(-1, K)
    q = _i32(q)
    N = q.shape[1]
    r = _f64(residual).reshape(-1, N)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        x = np.ascontiguousarray(x[rows])
        r = np.ascontiguousarray(r[rows])
    M = x.shape[0]
    S = np.ascontiguousarray(_so_shape(_f64(scale), N))
    O = None if offset is None else np.ascontiguousarray(_so_shape(_f64(offset), N))
    b = _f64(bias)
    gm = _f64(gamma)
    mm = np.empty((M, N)); y = np.empty((M, N)); no = np.empty((M, N))
    rc = _load().wqo_matmul_add_rmsnorm(_p(x), M, K, _p(q), N, _p(S), _p(O),
                                        S.shape[0], S.shape[1], int(group), _p(b), _p(r),
                                        _p(gm), float(eps), _p(mm), _p(y), _p(no))
    if rc:
        raise ValueError(f"wqo_matmul_add_rmsnorm rejected its arguments (rc={rc})")
    return mm, y, no
