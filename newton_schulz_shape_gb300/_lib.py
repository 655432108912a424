"""ctypes binding of libnsgb300.so: argument marshalling only.

Every function keeps its C name. Device buffers are passed as integer device
addresses (e.g. ``tensor.data_ptr()``); streams as integer ``cudaStream_t``
handles (e.g. ``torch.cuda.current_stream().cuda_stream``). A missing library
is an ImportError: there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnsgb300.so")

NS_OK = 0
NS_ERR_ARG = -1
NS_ERR_SHAPE = -2
NS_ERR_NOT_DIVISIBLE = -3
NS_ERR_HOME = -4
NS_ERR_CUDA = -5
NS_ERR_TIMEOUT = -6
NS_ERR_DEVICE_CHECK = -7
NS_ERR_UNSUPPORTED = -8
NS_ERR_WORKSPACE = -9

NS_BF16 = 0
NS_FP32_GRAM = 1
NS_FP32_GRAM_SPACE = 2
NS_FP32_AUTO = 3
NS_LAYOUT_ROW_SHARD = 0
NS_LAYOUT_FLAT = 1
NS_LAYOUT_TWO_STAGE = 2

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_vpp = ctypes.POINTER(ctypes.c_void_p)
_planp = ctypes.c_void_p

_SIGS = {
    "ns_cost": (ctypes.c_int, [_i64p, ctypes.c_int, ctypes.c_int, _i64p]),
    "ns_assign_owner_work": (ctypes.c_int, [ctypes.c_int, _i64p, _i32p, _i32p, ctypes.c_int, _i32p]),
    "ns_plan_create": (ctypes.c_int, [ctypes.c_int, _i32p, _i64p, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                      ctypes.c_int, _i32p, ctypes.POINTER(_planp)]),
    "ns_plan_create_flat": (ctypes.c_int, [ctypes.c_int, _i32p, _i64p, _i64p, ctypes.c_int64, _u8p, ctypes.c_int,
                                           ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_int, ctypes.c_float, ctypes.c_int, _i32p,
                                           ctypes.POINTER(_planp)]),
    "ns_plan_create_two_stage": (ctypes.c_int, [ctypes.c_int, _i32p, _i64p, _i32p, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                ctypes.c_float, ctypes.c_int, ctypes.c_float, _i32p,
                                                ctypes.POINTER(_planp)]),
    "ns_plan_rank_splits": (ctypes.c_int, [_planp, ctypes.c_int, _i64p, _i64p, _i64p, _i64p, _i64p, _i64p]),
    "ns_test_stall_next_gemm": (ctypes.c_int, [ctypes.c_uint64]),
    "ns_test_set_route_home": (ctypes.c_int, [_planp, ctypes.c_int, ctypes.c_int]),
    "ns_plan_destroy": (ctypes.c_int, [_planp]),
    "ns_plan_info": (ctypes.c_int, [_planp, _i64p]),
    "ns_plan_homes": (ctypes.c_int, [_planp, _i32p]),
    "ns_plan_home_layout": (ctypes.c_int, [_planp, _i64p, _i64p, _i64p]),
    "ns_plan_workspace_bytes": (ctypes.c_int, [_planp, _u64p]),
    "ns_owner_gather_meta": (ctypes.c_int, [_planp, ctypes.c_int, _i64p, _i64p, _i64p, _i64p]),
    "ns_owner_scatter_meta": (ctypes.c_int, [_planp, ctypes.c_int, _i64p, _i64p, _i64p]),
    "ns_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ns_orthogonalize_batched": (ctypes.c_int, [_planp, _vpp, _vpp, ctypes.c_int, ctypes.c_void_p,
                                                ctypes.c_uint64, ctypes.c_void_p]),
    "ns_pack_to_home": (ctypes.c_int, [_planp, _vpp, ctypes.c_int, ctypes.c_int, _vpp, ctypes.c_void_p]),
    "ns_unpack_from_home": (ctypes.c_int, [_planp, _vpp, ctypes.c_int, ctypes.c_int, _vpp, ctypes.c_void_p]),
    "ns_check_status": (ctypes.c_int, [_planp, ctypes.c_void_p]),
    "ns_orthogonalize_batched_fixed_ws": (ctypes.c_int, [_planp, _vpp, _vpp, ctypes.c_int, ctypes.c_void_p]),
    "ns_pipeline_create": (ctypes.c_int, [_planp, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)]),
    "ns_pipeline_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), _u64p]),
    "ns_pipeline_run": (ctypes.c_int, [ctypes.c_void_p, _vpp, _vpp, _vpp, _vpp, ctypes.c_void_p, ctypes.c_uint64,
                                       ctypes.c_void_p]),
    "ns_pipeline_destroy": (ctypes.c_int, [ctypes.c_void_p]),
    "ns_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "ns_set_gemm_cluster": (ctypes.c_int, [ctypes.c_int]),
    "ns_set_small_path": (ctypes.c_int, [ctypes.c_int]),
    "ns_set_symmetric_store": (ctypes.c_int, [ctypes.c_int]),
    "ns_profile_read": (ctypes.c_int, [ctypes.c_int, _i64p, ctypes.POINTER(ctypes.c_double)]),
}


def header_symbols() -> list:
    """Function names declared in include/nsgb300.h (parsed from the header)."""
    import re
    hdr = os.path.join(os.path.dirname(_HERE), "include", "nsgb300.h")
    with open(hdr) as f:
        text = f.read()
    return sorted(set(re.findall(r"^(?:int|const char\*)\s+(ns_\w+)\(", text, re.M)))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with newton_schulz_shape_gb300.build.build() "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class NsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lib.ns_status_string(code).decode()} ({code})")


def check(code: int, where: str) -> None:
    if code != NS_OK:
        raise NsError(code, where)


def i32_array(vals):
    vals = list(vals)
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def i64_array(vals):
    vals = list(vals)
    return (ctypes.c_int64 * max(1, len(vals)))(*vals)


def ptr_array(vals):
    vals = [int(v) for v in vals]
    return (ctypes.c_void_p * max(1, len(vals)))(*vals)
