"""Host-side checks of the C ABI (CPU only: no compute call reaches a GPU).

The library must load on a machine without a GPU, export every function that
include/wq.h declares, and its first phases (pure host validation) must return
the documented status codes for each rule of the operator pages' constraints.
Descriptors here carry fake, non-overlapping device addresses: validation only
compares addresses, it never dereferences them.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B(wq):
    from weight_only_bit_pack_b300 import binding
    return binding


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(wq_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_function(B):
    names = _declared_functions()
    assert "wq_matmul_add_rmsnorm" in names and "wq_pack_int4" in names
    for n in names:
        assert hasattr(B.lib, n), f"libwq.so does not export {n}"


def test_status_strings(B):
    assert B.lib.wq_status_string(0) == b"WQ_OK"
    assert B.lib.wq_status_string(3) == b"WQ_ERR_SHAPE"
    assert B.lib.wq_status_string(99) == b"WQ_ERR_UNKNOWN"
    assert B.lib.wq_version() >= 100


_next_addr = [0x10_0000_0000]


def D(B, dtype, shape, addr=None):
    d = B.WqTensor()
    if addr is None:
        addr = _next_addr[0]
        _next_addr[0] += 1 << 32
    d.data = addr
    d.dtype = int(dtype)
    d.ndim = len(shape)
    for i, v in enumerate(shape):
        d.shape[i] = v
    return d


def _args(B, M=16, K=256, N=128, dt=None, wdt=None, scale_shape=None, group=32, offset=True,
          bias=True, res_shape=None, x_shape=None):
    dt = dt or B.DType.F16
    wdt = wdt or B.DType.INT4
    G = (K + group - 1) // group if group else 1
    scale_shape = scale_shape if scale_shape is not None else ((G, N) if group else (N,))
    res_shape = res_shape or (M, N)
    x_shape = x_shape or (M, K)
    a = dict(x1=D(B, dt, x_shape), x2=D(B, wdt, (K, N)), scale=D(B, dt, scale_shape),
             offset=D(B, dt, scale_shape) if offset else None,
             bias=D(B, dt, (N,)) if bias else None, residual=D(B, dt, res_shape),
             gamma=D(B, dt, (N,)), eps=1e-6, group=group, y=D(B, dt, res_shape),
             normOut=D(B, dt, res_shape))
    return a


def _ws(B, a, kernel=0):
    r = lambda d: None if d is None else ctypes.byref(d)
    ws = ctypes.c_uint64(12345)
    st = B.lib.wq_matmul_add_rmsnorm_get_workspace_ex(
        r(a["x1"]), r(a["x2"]), r(a["scale"]), r(a["offset"]), r(a["bias"]), r(a["residual"]),
        r(a["gamma"]), a["eps"], a["group"], r(a["y"]), r(a["normOut"]), kernel, ctypes.byref(ws))
    return st, ws.value


def test_valid_configs_accepted(B):
    assert _ws(B, _args(B))[0] == 0                                           # tiny
    assert _ws(B, _args(B, M=8, K=4096, N=4096, dt=B.DType.BF16, group=128, offset=False,
                        x_shape=(1, 8, 4096), res_shape=(1, 8, 4096)))[0] == 0  # decode
    assert _ws(B, _args(B, M=2048, K=4096, N=11008, wdt=B.DType.INT8, group=0,
                        scale_shape=(11008,), bias=False))[0] == 0           # W8A16
    assert _ws(B, _args(B, M=8, K=64, N=32, group=0, scale_shape=(1,)))[0] == 0  # per-tensor
    assert _ws(B, _args(B, M=8, K=64, N=32, group=0, scale_shape=(1, 32)))[0] == 0  # (1, n)


def test_empty_m_and_n_need_no_workspace(B):
    st, ws = _ws(B, _args(B, M=0))
    assert st == 0 and ws == 0
    st, ws = _ws(B, _args(B, N=0, group=0, scale_shape=(1,)))
    assert st == 0 and ws == 0


@pytest.mark.parametrize("case,code", [
    ("k_zero", 3), ("k_too_big", 3), ("n_too_big", 3), ("x2_k_mismatch", 3), ("int4_odd_n", 3),
    ("x1_1d", 3), ("x1_dtype", 2), ("x2_dtype", 2), ("scale_dtype", 2), ("gamma_dtype", 2),
    ("group_not_mult32", 4), ("group_ge_k", 4), ("group_small", 4), ("group_scale_rows", 4),
    ("grouped_scale_without_group", 4), ("offset_shape", 3), ("bias_shape", 3),
    ("gamma_shape", 3), ("residual_rows", 3), ("y_shape", 3), ("eps_negative", 3),
    ("null_x1", 1), ("null_data", 1), ("normOut_alias_x1", 9), ("y_partial_alias", 9),
    ("normOut_alias_y", 9), ("bad_kernel", 6)])
def test_validation_errors(B, case, code):
    a = _args(B)
    kernel = 0
    if case == "k_zero":
        a = _args(B, K=0, group=0)
    elif case == "k_too_big":
        a = _args(B, K=65536, group=0)
    elif case == "n_too_big":
        a = _args(B, N=65536, group=0)
    elif case == "x2_k_mismatch":
        a["x2"] = D(B, B.DType.INT4, (255, 128))
    elif case == "int4_odd_n":
        a = _args(B, N=127, group=0)
    elif case == "x1_1d":
        a["x1"] = D(B, B.DType.F16, (256,))
    elif case == "x1_dtype":
        a["x1"] = D(B, B.DType.INT8, (16, 256))
    elif case == "x2_dtype":
        a["x2"] = D(B, B.DType.F16, (256, 128))
    elif case == "scale_dtype":
        a["scale"] = D(B, B.DType.BF16, (8, 128))
    elif case == "gamma_dtype":
        a["gamma"] = D(B, B.DType.BF16, (128,))
    elif case == "group_not_mult32":
        a = _args(B, group=48)
    elif case == "group_ge_k":
        a = _args(B, group=256)
    elif case == "group_small":
        a = _args(B, group=16)
    elif case == "group_scale_rows":
        a["scale"] = D(B, B.DType.F16, (7, 128))
        a["offset"] = None
    elif case == "grouped_scale_without_group":
        a["group"] = 0
        a["offset"] = None
    elif case == "offset_shape":
        a["offset"] = D(B, B.DType.F16, (8, 64))
    elif case == "bias_shape":
        a["bias"] = D(B, B.DType.F16, (127,))
    elif case == "gamma_shape":
        a["gamma"] = D(B, B.DType.F16, (1, 128))
    elif case == "residual_rows":
        a["residual"] = D(B, B.DType.F16, (2, 7, 128))
    elif case == "y_shape":
        a["y"] = D(B, B.DType.F16, (16, 64))
    elif case == "eps_negative":
        a["eps"] = -1.0
    elif case == "null_x1":
        a["x1"] = None
    elif case == "null_data":
        a["x2"].data = None
    elif case == "normOut_alias_x1":
        a["normOut"] = D(B, B.DType.F16, (16, 128), addr=a["x1"].data + 64)
    elif case == "y_partial_alias":
        a["y"] = D(B, B.DType.F16, (16, 128), addr=a["residual"].data + 2)
    elif case == "normOut_alias_y":
        a["normOut"] = D(B, B.DType.F16, (16, 128), addr=a["y"].data)
    elif case == "bad_kernel":
        kernel = 17
    st, _ = _ws(B, a, kernel)
    assert st == code, (case, st, B.lib.wq_last_error())
    assert B.lib.wq_last_error() != b""


def test_in_place_y_is_residual_accepted(B):
    a = _args(B)
    a["y"] = D(B, B.DType.F16, (16, 128), addr=a["residual"].data)
    assert _ws(B, a)[0] == 0


def test_residual_2d_or_3d(B):
    assert _ws(B, _args(B, res_shape=(2, 8, 128)))[0] == 0
    assert _ws(B, _args(B, x_shape=(2, 8, 256), res_shape=(16, 128)))[0] == 0


def test_second_phase_rejects_small_workspace_without_launch(B):
    a = _args(B)
    st, need = _ws(B, a)
    assert st == 0 and need > 0
    r = lambda d: None if d is None else ctypes.byref(d)
    st = B.lib.wq_matmul_add_rmsnorm(
        r(a["x1"]), r(a["x2"]), r(a["scale"]), r(a["offset"]), r(a["bias"]), r(a["residual"]),
        r(a["gamma"]), a["eps"], a["group"], r(a["y"]), r(a["normOut"]), 0x2000_0000_0000,
        need - 1, None)
    assert st == 5


def test_pack_validation(B):
    r = ctypes.byref
    ws = ctypes.c_uint64(7)
    w = D(B, B.DType.INT32, (64, 32)); o = D(B, B.DType.INT4, (64, 32))
    assert B.lib.wq_pack_int4_get_workspace(r(w), r(o), r(ws)) == 0 and ws.value == 0
    assert B.lib.wq_pack_int4_get_workspace(r(D(B, B.DType.INT32, (64, 31))),
                                            r(D(B, B.DType.INT4, (64, 31))), r(ws)) == 3
    assert B.lib.wq_pack_int4_get_workspace(r(D(B, B.DType.INT8, (64, 32))), r(o), r(ws)) == 2
    assert B.lib.wq_pack_int4_get_workspace(r(w), r(D(B, B.DType.INT4, (32, 32))), r(ws)) == 3
    assert B.lib.wq_pack_int4_get_workspace(None, r(o), r(ws)) == 1
    alias = D(B, B.DType.INT4, (64, 32), addr=w.data + 16)
    assert B.lib.wq_pack_int4_get_workspace(r(w), r(alias), r(ws)) == 9
    # empty weight: valid, nothing to do
    assert B.lib.wq_pack_int4(r(D(B, B.DType.INT32, (0, 32))), r(D(B, B.DType.INT4, (0, 32))),
                              None, 0, None) == 0


def test_fp4_pack_validation(B):
    r = ctypes.byref
    ws = ctypes.c_uint64(7)
    w = D(B, B.DType.F32, (64, 32)); o = D(B, B.DType.FP4_E2M1, (64, 32))
    assert B.lib.wq_pack_int4_get_workspace(r(w), r(o), r(ws)) == 0 and ws.value == 0
    # F32 only with an FP4 output, FP4 only from F32
    assert B.lib.wq_pack_int4_get_workspace(r(w), r(D(B, B.DType.INT4, (64, 32))), r(ws)) == 2
    assert B.lib.wq_pack_int4_get_workspace(r(D(B, B.DType.INT32, (64, 32))), r(o), r(ws)) == 2
    assert B.lib.wq_pack_int4_get_workspace(r(D(B, B.DType.F32, (64, 31))),
                                            r(D(B, B.DType.FP4_E2M1, (64, 31))), r(ws)) == 3
    assert B.lib.wq_pack_int4_get_workspace(r(w), r(D(B, B.DType.FP4_E2M1, (32, 32))), r(ws)) == 3
    alias = D(B, B.DType.FP4_E2M1, (64, 32), addr=w.data + 64)
    assert B.lib.wq_pack_int4_get_workspace(r(w), r(alias), r(ws)) == 9
    assert B.lib.wq_pack_int4(r(D(B, B.DType.F32, (0, 32))), r(D(B, B.DType.FP4_E2M1, (0, 32))),
                              None, 0, None) == 0


def _mx(B, M=16, K=96, N=64, J=None):
    J = (K + 31) // 32 if J is None else J
    return [D(B, B.DType.FP4_E2M1, (M, K)), D(B, B.DType.E8M0, (M, J)),
            D(B, B.DType.FP4_E2M1, (K, N)), D(B, B.DType.E8M0, (J, N)), D(B, B.DType.F32, (M, N))]


def _mx_ws(B, ds):
    ws = ctypes.c_uint64(7)
    st = B.lib.wq_mx_matmul_add_get_workspace(*[ctypes.byref(d) for d in ds], ctypes.byref(ws))
    return st, ws.value


def test_mx_matmul_validation(B):
    assert _mx_ws(B, _mx(B)) == (0, 0)
    assert _mx_ws(B, _mx(B, K=70))[0] == 0             # short last slice: J = 3
    assert _mx_ws(B, _mx(B, M=0))[0] == 0
    assert _mx_ws(B, _mx(B, K=70, J=2))[0] == 3        # scale slices must be ceil(K/32)
    assert _mx_ws(B, _mx(B, K=95))[0] == 3             # K odd
    assert _mx_ws(B, _mx(B, N=63))[0] == 3             # N odd
    assert _mx_ws(B, _mx(B, K=0))[0] == 3
    ds = _mx(B); ds[2] = D(B, B.DType.FP4_E2M1, (64, 64))
    assert _mx_ws(B, ds)[0] == 3                       # x2 rows != K
    ds = _mx(B); ds[4] = D(B, B.DType.F32, (16, 62))
    assert _mx_ws(B, ds)[0] == 3
    ds = _mx(B); ds[0] = D(B, B.DType.INT4, (16, 96))
    assert _mx_ws(B, ds)[0] == 2
    ds = _mx(B); ds[3] = D(B, B.DType.INT8, (3, 64))
    assert _mx_ws(B, ds)[0] == 2
    ds = _mx(B); ds[4] = D(B, B.DType.F16, (16, 64))
    assert _mx_ws(B, ds)[0] == 2
    ds = _mx(B); ds[4] = D(B, B.DType.F32, (16, 64), addr=ds[1].data + 8)
    assert _mx_ws(B, ds)[0] == 9                       # y overlaps scale1
    ds = _mx(B); ds[1] = None
    assert B.lib.wq_mx_matmul_add_get_workspace(*[ctypes.byref(d) if d is not None else None
                                                  for d in ds], ctypes.byref(ctypes.c_uint64())) == 1
    # an empty product is valid and launches nothing
    ds = _mx(B, M=0)
    assert B.lib.wq_mx_matmul_add(*[ctypes.byref(d) for d in ds], None, 0, None) == 0


def test_mx_matmul_transposed_x1_validation(B):
    def ds(M=16, K=96, N=64, sM=None):
        J = (K + 31) // 32
        return [D(B, B.DType.FP4_E2M1_T, (K, M)), D(B, B.DType.E8M0, (J, sM if sM else M)),
                D(B, B.DType.FP4_E2M1, (K, N)), D(B, B.DType.E8M0, (J, N)), D(B, B.DType.F32, (M, N))]
    assert _mx_ws(B, ds()) == (0, 0)
    assert _mx_ws(B, ds(M=15))[0] == 3            # packed along m: m even
    bad = ds(); bad[1] = D(B, B.DType.E8M0, (16, 3))
    assert _mx_ws(B, bad)[0] == 3                 # scale1 follows x1's storage: (J, m)
    bad = ds(); bad[2] = D(B, B.DType.FP4_E2M1_T, (64, 96))
    assert _mx_ws(B, bad)[0] == 2                 # x2 is never the transposed form


def test_mx_kernel_selector(B):
    ds = _mx(B, M=0)
    r = [ctypes.byref(d) for d in ds]
    assert B.lib.wq_mx_matmul_add_ex(*r, 0, None, 0, None) == 0
    assert B.lib.wq_mx_matmul_add_ex(*r, 1, None, 0, None) == 0
    assert B.lib.wq_mx_matmul_add_ex(*r, 7, None, 0, None) == 6
