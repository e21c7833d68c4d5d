"""ctypes binding of ``libwq.so`` (the C ABI declared in ``include/wq.h``).

Argument marshalling only: torch tensors become ``wq_tensor`` descriptors, the
current CUDA stream is passed as ``cudaStream_t``, and every status code other
than ``WQ_OK`` raises :class:`WQError`. No computation happens here and there
is no fallback: if the library cannot be loaded, importing this module raises.

Tensor conventions: fp16/bf16 tensors map to WQ_F16/WQ_BF16, ``torch.int8`` to
WQ_INT8, ``torch.int32`` to WQ_INT32, and a ``torch.uint8`` tensor of shape
(K, N/2) is read as packed WQ_INT4 of logical shape (K, N). A weight in the
kernel-native tiled layout is a :class:`TiledInt4` (its bytes plus the logical
(K, N)), described as WQ_INT4_TILED.
"""
from __future__ import annotations

import ctypes
import enum
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libwq.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libwq.so is missing at {_LIB_PATH}; build it with "
                      "`python -m weight_only_bit_pack_b300.build` (there is no CPU fallback)")
lib = ctypes.CDLL(_LIB_PATH)


class Status(enum.IntEnum):
    OK = 0
    ERR_NULL = 1
    ERR_DTYPE = 2
    ERR_SHAPE = 3
    ERR_GROUP = 4
    ERR_WORKSPACE = 5
    ERR_UNSUPPORTED = 6
    ERR_CUDA = 7
    ERR_DEVICE_TIMEOUT = 8
    ERR_ALIAS = 9


class Kernel(enum.IntEnum):
    AUTO = 0
    GENERIC = 1
    DECODE = 2
    PREFILL = 3


class DType(enum.IntEnum):
    F16 = 1
    BF16 = 2
    INT8 = 3
    INT4 = 4
    INT32 = 5
    INT4_TILED = 6
    F32 = 7
    INT8_T = 8
    INT4_T = 9
    FP4_E2M1 = 10
    E8M0 = 11
    FP4_E2M1_T = 12


class WQError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{lib.wq_status_string(status).decode()}: {detail}")


class WqTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 3)]


class TiledInt4:
    """A (K, N) INT4 weight in the kernel-native tiled layout: ``data`` holds its
    ceil(K/64) * 64 * N / 2 bytes (uint8, 16-byte aligned)."""

    def __init__(self, data: torch.Tensor, K: int, N: int):
        if data.dtype != torch.uint8 or data.numel() != tiled_bytes(K, N):
            raise ValueError(f"a tiled ({K}, {N}) INT4 weight holds {tiled_bytes(K, N)} uint8 bytes")
        self.data, self.K, self.N = data, int(K), int(N)

    @property
    def device(self):
        return self.data.device


class TransposedWeight:
    """A (K, N) weight stored transposed: ``data`` is the (N, K) int8 array
    (``bits=8``) or its INT4 packing along K, an (N, K/2) uint8 array (``bits=4``)."""

    def __init__(self, data: torch.Tensor, bits: int):
        if bits not in (4, 8) or data.dim() != 2:
            raise ValueError("a transposed weight is a 2-D int8 (N, K) or uint8 (N, K/2) array")
        self.data, self.bits = data, bits
        self.N = data.shape[0]
        self.K = data.shape[1] * (2 if bits == 4 else 1)

    @property
    def device(self):
        return self.data.device


def tiled_bytes(K: int, N: int) -> int:
    return (K + 63) // 64 * 64 * N // 2


_P = ctypes.POINTER(WqTensor)
_T = [_P] * 7 + [ctypes.c_double, ctypes.c_int64, _P, _P]
lib.wq_pack_int4_get_workspace.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_uint64)]
lib.wq_pack_int4.argtypes = [_P, _P, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
lib.wq_convert_int4_layout.argtypes = [_P, _P, ctypes.c_void_p]
lib.wq_mx_matmul_add_get_workspace.argtypes = [_P, _P, _P, _P, _P, ctypes.POINTER(ctypes.c_uint64)]
lib.wq_mx_matmul_add.argtypes = [_P, _P, _P, _P, _P, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
lib.wq_mx_matmul_add_ex.argtypes = [_P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_void_p, ctypes.c_uint64,
                                    ctypes.c_void_p]
lib.wq_dynamic_quant_get_workspace.argtypes = [_P, _P, _P, _P, ctypes.POINTER(ctypes.c_uint64)]
lib.wq_dynamic_quant.argtypes = [_P, _P, _P, _P, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
lib.wq_matmul_add_rmsnorm_get_workspace.argtypes = _T + [ctypes.POINTER(ctypes.c_uint64)]
lib.wq_matmul_add_rmsnorm.argtypes = _T + [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
lib.wq_matmul_add_rmsnorm_get_workspace_ex.argtypes = _T + [ctypes.c_int32,
                                                            ctypes.POINTER(ctypes.c_uint64)]
lib.wq_matmul_add_rmsnorm_ex.argtypes = _T + [ctypes.c_int32, ctypes.c_void_p, ctypes.c_uint64,
                                              ctypes.c_void_p]
lib.wq_matmul_add_rmsnorm_select_kernel.argtypes = _T
lib.wq_matmul_add_rmsnorm_noalloc.argtypes = _T + [ctypes.c_void_p]
lib.wq_read_device_status.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                                      ctypes.POINTER(ctypes.c_int32)]
lib.wq_check_device_timeout.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_void_p]
lib.wq_noalloc_read_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
lib.wq_test_set_wait_limits.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
lib.wq_status_string.argtypes = [ctypes.c_int32]
lib.wq_status_string.restype = ctypes.c_char_p
lib.wq_last_error.argtypes = []
lib.wq_last_error.restype = ctypes.c_char_p
for _f in ("wq_pack_int4_get_workspace", "wq_pack_int4", "wq_matmul_add_rmsnorm_get_workspace",
           "wq_matmul_add_rmsnorm", "wq_matmul_add_rmsnorm_get_workspace_ex",
           "wq_matmul_add_rmsnorm_ex", "wq_matmul_add_rmsnorm_select_kernel",
           "wq_read_device_status", "wq_version", "wq_matmul_add_rmsnorm_noalloc",
           "wq_check_device_timeout", "wq_noalloc_read_device_status", "wq_test_set_wait_limits",
           "wq_convert_int4_layout", "wq_dynamic_quant_get_workspace", "wq_dynamic_quant",
           "wq_mx_matmul_add_get_workspace", "wq_mx_matmul_add", "wq_mx_matmul_add_ex"):
    getattr(lib, _f).restype = ctypes.c_int32

_TORCH2WQ = {torch.float16: DType.F16, torch.bfloat16: DType.BF16, torch.int8: DType.INT8,
             torch.uint8: DType.INT4, torch.int32: DType.INT32, torch.float32: DType.F32}


def _check(status: int):
    if status != 0:
        raise WQError(status, lib.wq_last_error().decode())


def describe(t: Optional[torch.Tensor], dtype: Optional[int] = None, shape=None):
    """wq_tensor for a contiguous torch tensor (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, TransposedWeight):
        if not t.data.is_contiguous():
            raise ValueError("wq tensors must be contiguous")
        d = WqTensor()
        d.data = t.data.data_ptr()
        d.dtype = int(DType.INT4_T if t.bits == 4 else DType.INT8_T)
        d.ndim = 2
        d.shape[0], d.shape[1] = t.N, t.K
        return d
    if isinstance(t, TiledInt4):
        d = WqTensor()
        d.data = t.data.data_ptr()
        d.dtype = int(DType.INT4_TILED)
        d.ndim = 2
        d.shape[0], d.shape[1] = t.K, t.N
        return d
    if not t.is_contiguous():
        raise ValueError("wq tensors must be contiguous")
    d = WqTensor()
    d.data = t.data_ptr() if t.numel() > 0 else (t.data_ptr() or None)
    d.dtype = int(dtype if dtype is not None else _TORCH2WQ[t.dtype])
    shp = list(shape if shape is not None else t.shape)
    if d.dtype == DType.INT4 and shape is None:
        shp[-1] = shp[-1] * 2  # logical N of a (K, N/2) byte tensor
    d.ndim = len(shp)
    for i, v in enumerate(shp):
        d.shape[i] = int(v)
    return d


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pack_int4_get_workspace(weight: torch.Tensor, out: torch.Tensor) -> int:
    ws = ctypes.c_uint64(0)
    _check(lib.wq_pack_int4_get_workspace(_ref(describe(weight)), _ref(describe(out)),
                                          ctypes.byref(ws)))
    return ws.value


def pack_int4(weight: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """(K, N) int32 -> (K, N/2) uint8 packed INT4, on the GPU (``wq_pack_int4``)."""
    if out is None:
        out = torch.empty((weight.shape[0], weight.shape[1] // 2), dtype=torch.uint8,
                          device=weight.device)
    wd, od = describe(weight), describe(out)
    ws = ctypes.c_uint64(0)
    _check(lib.wq_pack_int4_get_workspace(_ref(wd), _ref(od), ctypes.byref(ws)))
    _check(lib.wq_pack_int4(_ref(wd), _ref(od), None, 0, _stream(stream)))
    return out


def pack_int4_tiled(weight: torch.Tensor, out: Optional[TiledInt4] = None,
                    stream=None) -> TiledInt4:
    """(K, N) int32 -> the kernel-native tiled INT4 layout, on the GPU (``wq_pack_int4``
    with a WQ_INT4_TILED output; N % 16 == 0)."""
    K, N = weight.shape
    if out is None:
        out = TiledInt4(torch.empty(tiled_bytes(K, N), dtype=torch.uint8, device=weight.device),
                        K, N)
    wd, od = describe(weight), describe(out)
    ws = ctypes.c_uint64(0)
    _check(lib.wq_pack_int4_get_workspace(_ref(wd), _ref(od), ctypes.byref(ws)))
    _check(lib.wq_pack_int4(_ref(wd), _ref(od), None, 0, _stream(stream)))
    return out


def int4_to_tiled(w4: torch.Tensor, stream=None) -> TiledInt4:
    """Dense packed INT4 (K, N/2) uint8 -> tiled layout (``wq_convert_int4_layout``)."""
    K, N = w4.shape[0], w4.shape[1] * 2
    out = TiledInt4(torch.empty(tiled_bytes(K, N), dtype=torch.uint8, device=w4.device), K, N)
    _check(lib.wq_convert_int4_layout(_ref(describe(w4)), _ref(describe(out)), _stream(stream)))
    return out


def convert_int4(src, layout: str, stream=None):
    """Any INT4 layout of a weight into another (``wq_convert_int4_layout``):
    ``src`` is a (K, N/2) uint8 dense tensor, a :class:`TiledInt4` or a 4-bit
    :class:`TransposedWeight`; ``layout`` is "dense", "tiled" or "transposed"."""
    if isinstance(src, TiledInt4):
        K, N = src.K, src.N
    elif isinstance(src, TransposedWeight):
        K, N = src.K, src.N
    else:
        K, N = src.shape[0], src.shape[1] * 2
    dev = src.device
    if layout == "dense":
        out = torch.empty((K, N // 2), dtype=torch.uint8, device=dev)
    elif layout == "tiled":
        out = TiledInt4(torch.empty(tiled_bytes(K, N), dtype=torch.uint8, device=dev), K, N)
    elif layout == "transposed":
        out = TransposedWeight(torch.empty((N, K // 2), dtype=torch.uint8, device=dev), 4)
    else:
        raise ValueError(layout)
    _check(lib.wq_convert_int4_layout(_ref(describe(src)), _ref(describe(out)), _stream(stream)))
    return out


def tiled_to_int4(t: TiledInt4, stream=None) -> torch.Tensor:
    """Tiled layout -> dense packed INT4 (K, N/2) uint8 (``wq_convert_int4_layout``)."""
    out = torch.empty((t.K, t.N // 2), dtype=torch.uint8, device=t.device)
    _check(lib.wq_convert_int4_layout(_ref(describe(t)), _ref(describe(out)), _stream(stream)))
    return out


def dynamic_quant(x: torch.Tensor, smooth_scales: Optional[torch.Tensor] = None, bits: int = 8,
                  y: Optional[torch.Tensor] = None, scale: Optional[torch.Tensor] = None,
                  stream=None):
    """Per-token symmetric quantization (``wq_dynamic_quant``). Returns ``(y, scale)``:
    y int8 with x's shape (bits 8), or uint8 (..., K/2) packed INT4 codes (bits 4);
    scale float32 with x's leading shape."""
    lead = tuple(x.shape[:-1])
    if y is None:
        shp = lead + ((x.shape[-1],) if bits == 8 else (x.shape[-1] // 2,))
        y = torch.empty(shp, dtype=torch.int8 if bits == 8 else torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(lead if lead else (1,), dtype=torch.float32, device=x.device)
    yd = describe(y)
    d = [describe(x), describe(smooth_scales), yd, describe(scale)]
    ws = ctypes.c_uint64(0)
    _check(lib.wq_dynamic_quant_get_workspace(*[_ref(v) for v in d], ctypes.byref(ws)))
    _check(lib.wq_dynamic_quant(*[_ref(v) for v in d], None, 0, _stream(stream)))
    return y, scale


def pack_fp4(weight: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """(K, N) float32 -> (K, N/2) uint8 of FP4 E2M1 codes (``wq_pack_int4`` with an
    FP4_E2M1 output): nearest value, ties to the even code, saturating at +-6."""
    K, N = weight.shape
    if out is None:
        out = torch.empty((K, N // 2), dtype=torch.uint8, device=weight.device)
    wd, od = describe(weight), describe(out, DType.FP4_E2M1, (K, N))
    ws = ctypes.c_uint64(0)
    _check(lib.wq_pack_int4_get_workspace(_ref(wd), _ref(od), ctypes.byref(ws)))
    _check(lib.wq_pack_int4(_ref(wd), _ref(od), None, 0, _stream(stream)))
    return out


def mx_matmul_add(x1: torch.Tensor, scale1: torch.Tensor, x2: torch.Tensor, scale2: torch.Tensor,
                  y: torch.Tensor, x1_transposed: bool = False, kernel: str = "tensor",
                  stream=None) -> torch.Tensor:
    """``y += mx(x1, scale1) @ mx(x2, scale2)`` (``wq_mx_matmul_add``): x1 (M, K/2) and
    x2 (K, N/2) uint8 FP4 E2M1 codes, scale1 (M, ceil(K/32)) and scale2 (ceil(K/32), N)
    uint8 E8M0 exponents, y float32 (M, N) updated in place and returned. With
    ``x1_transposed`` x1 is (K, M/2) (packed along M) and scale1 (ceil(K/32), M).
    ``kernel``: "tensor" (slices on the tensor cores, fp32 sum) or "exact" (fp64 sum)."""
    kid = {"tensor": 0, "exact": 1}[kernel]
    N = x2.shape[1] * 2
    if x1_transposed:
        K, M = x1.shape[0], x1.shape[1] * 2
        dx1 = describe(x1, DType.FP4_E2M1_T, (K, M))
    else:
        M, K = x1.shape[0], x1.shape[1] * 2
        dx1 = describe(x1, DType.FP4_E2M1, (M, K))
    d = [dx1, describe(scale1, DType.E8M0),
         describe(x2, DType.FP4_E2M1, (K, N)), describe(scale2, DType.E8M0), describe(y)]
    ws = ctypes.c_uint64(0)
    _check(lib.wq_mx_matmul_add_get_workspace(*[_ref(v) for v in d], ctypes.byref(ws)))
    _check(lib.wq_mx_matmul_add_ex(*[_ref(v) for v in d], kid, None, 0, _stream(stream)))
    return y


def pack_int4_bytes(n_logical: int, data: torch.Tensor) -> WqTensor:
    """Descriptor of packed INT4 bytes with an explicit logical last dimension."""
    shp = list(data.shape)
    shp[-1] = n_logical
    return describe(data, DType.INT4, shp)


def _descs(x1, x2, scale, offset, bias, residual, gamma, y, normOut):
    return [describe(x1), describe(x2), describe(scale), describe(offset), describe(bias),
            describe(residual), describe(gamma), describe(y), describe(normOut)]


def matmul_add_rmsnorm_get_workspace(x1, x2, scale, offset, bias, residual, gamma, eps, group=0,
                                     y=None, normOut=None, kernel: int = Kernel.AUTO) -> int:
    y = residual if y is None else y
    normOut = torch.empty_like(residual) if normOut is None else normOut
    d = _descs(x1, x2, scale, offset, bias, residual, gamma, y, normOut)
    ws = ctypes.c_uint64(0)
    _check(lib.wq_matmul_add_rmsnorm_get_workspace_ex(*[_ref(v) for v in d[:7]], float(eps),
                                                      int(group), _ref(d[7]), _ref(d[8]),
                                                      int(kernel), ctypes.byref(ws)))
    return ws.value


def select_kernel(x1, x2, scale, offset, bias, residual, gamma, eps, group=0) -> Kernel:
    y = torch.empty_like(residual)
    no = torch.empty_like(residual)
    d = _descs(x1, x2, scale, offset, bias, residual, gamma, y, no)
    r = lib.wq_matmul_add_rmsnorm_select_kernel(*[_ref(v) for v in d[:7]], float(eps), int(group),
                                                _ref(d[7]), _ref(d[8]))
    if r < 0:
        _check(-r)
    return Kernel(r)


def matmul_add_rmsnorm(x1, x2, scale, offset, bias, residual, gamma, eps: float, group: int = 0,
                       y: Optional[torch.Tensor] = None, normOut: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, kernel: int = Kernel.AUTO,
                       stream=None, check_status: bool = False):
    """Fused ``y = x1 @ (x2*scale + offset) + bias + residual``,
    ``normOut = y / sqrt(mean(y^2) + eps) * gamma`` (``wq_matmul_add_rmsnorm``).

    Outputs and workspace are allocated with torch when not given (a given
    workspace must have had its first 2048 bytes zeroed once). Pass
    ``y=residual`` for the in-place variant. Returns ``(y, normOut)``.

    ``check_status=True`` waits for the call and reads the workspace's device
    status word: if a device-side wait gave up, the header is zeroed again (so
    the workspace can serve the next call) and :class:`WQError` with
    ``ERR_DEVICE_TIMEOUT`` is raised, naming the place that gave up.
    """
    if y is None:
        y = torch.empty_like(residual)
    if normOut is None:
        normOut = torch.empty_like(residual)
    d = _descs(x1, x2, scale, offset, bias, residual, gamma, y, normOut)
    refs = [_ref(v) for v in d]
    ws = ctypes.c_uint64(0)
    _check(lib.wq_matmul_add_rmsnorm_get_workspace_ex(*refs[:7], float(eps), int(group), refs[7],
                                                      refs[8], int(kernel), ctypes.byref(ws)))
    if workspace is None:
        # the header must start zeroed (include/wq.h); the library keeps it so
        workspace = torch.zeros(max(ws.value, 2048), dtype=torch.uint8, device=residual.device)
    elif workspace.numel() < ws.value:
        raise WQError(Status.ERR_WORKSPACE, f"need {ws.value} bytes")
    _check(lib.wq_matmul_add_rmsnorm_ex(*refs[:7], float(eps), int(group), refs[7], refs[8],
                                        int(kernel), workspace.data_ptr(), workspace.numel(),
                                        _stream(stream)))
    if check_status:
        st = read_device_status(workspace, stream)
        if st != 0:
            workspace[:HEADER_BYTES].zero_()
            torch.cuda.synchronize(workspace.device)
            raise WQError(st & 0xFF, f"device status word 0x{st:x}: the bounded wait at place "
                                     f"{st >> 8} gave up; y and normOut are incomplete")
    return y, normOut


HEADER_BYTES = 2048  # the workspace header of include/wq.h


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check(lib.wq_read_device_status(workspace.data_ptr(), workspace.numel(), _stream(stream),
                                     ctypes.byref(st)))
    return st.value


WHERE_SELF_CHECK = 31  # WQ_WHERE_SELF_CHECK in include/wq.h


def check_device_timeout(workspace: torch.Tensor, budget_cycles: int, stream=None) -> None:
    """``wq_check_device_timeout``: a bounded device wait that must give up and
    record WQ_ERR_DEVICE_TIMEOUT in the workspace status word."""
    _check(lib.wq_check_device_timeout(workspace.data_ptr(), workspace.numel(),
                                       ctypes.c_uint64(budget_cycles), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 8 << 20  # WQ_NOALLOC_SCRATCH_BYTES in include/wq.h
WHERE_PREFILL_ROW_BLOCK = 5       # WQ_WHERE_PREFILL_ROW_BLOCK
WHERE_DECODE_GRID = 15            # WQ_WHERE_DECODE_GRID


def noalloc_read_device_status(stream=None) -> int:
    """``wq_noalloc_read_device_status``: the no-alloc scratch's status word
    (synchronizes the stream); read it before the next no-alloc call clears it."""
    st = ctypes.c_int32(0)
    _check(lib.wq_noalloc_read_device_status(_stream(stream), ctypes.byref(st)))
    return st.value


def set_wait_limits_for_testing(budget_cycles: int, extra_arrivals: int) -> None:
    """``wq_test_set_wait_limits``: for tests of the device error channel only.
    (0, 0) restores the defaults."""
    _check(lib.wq_test_set_wait_limits(ctypes.c_uint64(budget_cycles),
                                       ctypes.c_uint32(extra_arrivals)))


def matmul_add_rmsnorm_noalloc(x1, x2, scale, offset, bias, residual, gamma, eps: float,
                               group: int = 0, y: Optional[torch.Tensor] = None,
                               normOut: Optional[torch.Tensor] = None, stream=None):
    """``wq_matmul_add_rmsnorm_noalloc``: the fused operator without a workspace.

    The library keeps its scratch in a fixed per-device array, for callers that
    cannot allocate device memory. Outputs are allocated here only when not
    given. Calls sharing a device must not overlap on the GPU.
    """
    if y is None:
        y = torch.empty_like(residual)
    if normOut is None:
        normOut = torch.empty_like(residual)
    d = _descs(x1, x2, scale, offset, bias, residual, gamma, y, normOut)
    refs = [_ref(v) for v in d]
    _check(lib.wq_matmul_add_rmsnorm_noalloc(*refs[:7], float(eps), int(group), refs[7], refs[8],
                                             _stream(stream)))
    return y, normOut
