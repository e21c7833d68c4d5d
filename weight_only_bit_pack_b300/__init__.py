"""B300-native weight-only quantized matmul with fused residual-add + RMSNorm.

The compute lives in ``libwq.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/wq.h``). This package is its thin Python binding:
``pack_int4`` and ``matmul_add_rmsnorm`` (plus their ``*_get_workspace`` first
phases) marshal torch tensors into the C structs and call the library on the
current CUDA stream. There is no CPU fallback: if ``libwq.so`` is missing, the
first use of an op raises.
"""
_API = ("pack_int4", "pack_int4_get_workspace", "matmul_add_rmsnorm",
        "matmul_add_rmsnorm_get_workspace", "WQError", "Status", "Kernel", "lib",
        "read_device_status", "pack_int4_bytes", "select_kernel", "describe", "DType",
        "matmul_add_rmsnorm_noalloc", "NOALLOC_SCRATCH_BYTES", "check_device_timeout",
        "WHERE_SELF_CHECK", "noalloc_read_device_status", "set_wait_limits_for_testing",
        "WHERE_PREFILL_ROW_BLOCK", "WHERE_DECODE_GRID", "HEADER_BYTES", "TiledInt4",
        "tiled_bytes", "pack_int4_tiled", "int4_to_tiled", "tiled_to_int4", "dynamic_quant",
        "TransposedWeight", "convert_int4", "pack_fp4", "mx_matmul_add")


def __getattr__(name):
    if name in _API:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
