"""ctypes binding of libhmoe (include/hmoe.h). Argument marshalling only.

Every computation runs in the library's CUDA kernels. If the shared
library is missing, importing this module raises. There is no CPU
fallback.
"""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libhmoe.so")

HMOE_OK = 0
STATUS_NAMES = {
    0: "HMOE_OK", -1: "HMOE_ERR_INVALID_ARG", -2: "HMOE_ERR_UNSUPPORTED_SHAPE",
    -3: "HMOE_ERR_WORKSPACE_TOO_SMALL", -4: "HMOE_ERR_BAD_BITMAP", -5: "HMOE_ERR_CUDA",
    -6: "HMOE_ERR_DEVICE_TIMEOUT", -7: "HMOE_ERR_BAD_ROUTE",
}
FMT_NF3, FMT_NVFP4, FMT_MXFP4 = 3, 4, 5
ACT_BF16, ACT_F16 = 0, 1
ACT_QUANT_NONE, ACT_QUANT_NVFP4 = 0, 1
TIERS_ONE_LAUNCH, TIERS_KEPT_FIRST, TIERS_NF3_FIRST = 0, 1, 2
PATH_AUTO, PATH_STREAM, PATH_GROUPED = 0, 1, 2
DEBUG_NO_COPIES = 1
DEBUG_GROUPED_PAIR = 2

# Every symbol include/hmoe.h declares.
EXPORTS = (
    "hmoe_packed_size", "hmoe_workspace_size", "hmoe_workspace_init", "hmoe_pack_weights",
    "hmoe_plan_routes", "hmoe_forward", "hmoe_forward_ex", "hmoe_check_device_status",
    "hmoe_debug_dequant", "hmoe_layer_expert_info", "hmoe_layer_destroy", "hmoe_last_error",
    "hmoe_launch_count", "hmoe_version", "hmoe_forward_static", "hmoe_check_device_status_static",
    "hmoe_auto_path", "hmoe_debug_decode_operand", "hmoe_linear_packed_size", "hmoe_linear_workspace_size",
    "hmoe_linear_pack", "hmoe_linear_forward", "hmoe_linear_forward_ex", "hmoe_linear_destroy",
    "hmoe_quantize_act_nvfp4",
)


class LayerDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int), ("topk", ctypes.c_int),
                ("kept_format", ctypes.c_int), ("act_dtype", ctypes.c_int), ("act_quant", ctypes.c_int),
                ("act_global13", ctypes.c_float), ("act_global2", ctypes.c_float)]


class LinearDesc(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("K", ctypes.c_int), ("fmt", ctypes.c_int), ("act_dtype", ctypes.c_int)]


class ExpertSrc(ctypes.Structure):
    _fields_ = [("w13_codes", ctypes.c_void_p), ("w13_scales", ctypes.c_void_p), ("w13_global", ctypes.c_float),
                ("w2_codes", ctypes.c_void_p), ("w2_scales", ctypes.c_void_p), ("w2_global", ctypes.c_float)]


class ForwardOpts(ctypes.Structure):
    _fields_ = [("tier_order", ctypes.c_int), ("path", ctypes.c_int), ("wait_limit_us", ctypes.c_int),
                ("debug_flags", ctypes.c_int), ("stage_events", ctypes.POINTER(ctypes.c_void_p)),
                ("n_stage_events", ctypes.c_int)]


class HmoeError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def load(path=LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"libhmoe.so is not built ({path}); run nf3_moe_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "hmoe_packed_size": (i, [P(LayerDesc), vp, P(sz), P(sz)]),
        "hmoe_workspace_size": (i, [P(LayerDesc), i, P(sz)]),
        "hmoe_workspace_init": (i, [vp, sz, vp]),
        "hmoe_pack_weights": (i, [P(LayerDesc), vp, P(ExpertSrc), vp, vp, vp, P(vp)]),
        "hmoe_plan_routes": (i, [vp, vp, i, vp, vp, vp, vp, vp, sz, vp]),
        "hmoe_forward": (i, [vp, vp, i, vp, vp, vp, vp, vp, vp, sz, vp]),
        "hmoe_forward_ex": (i, [vp, vp, i, vp, vp, vp, vp, vp, vp, sz, P(ForwardOpts), vp]),
        "hmoe_check_device_status": (i, [vp, sz, vp]),
        "hmoe_debug_dequant": (i, [vp, i, i, vp, vp]),
        "hmoe_debug_decode_operand": (i, [vp, i, i, vp, vp, vp]),
        "hmoe_layer_expert_info": (i, [vp, i, P(i), P(ctypes.c_float), P(ctypes.c_float)]),
        "hmoe_layer_destroy": (None, [vp]),
        "hmoe_last_error": (ctypes.c_char_p, []),
        "hmoe_launch_count": (ctypes.c_uint64, []),
        "hmoe_forward_static": (i, [vp, vp, i, vp, vp, vp, vp, vp, vp]),
        "hmoe_check_device_status_static": (i, [vp]),
        "hmoe_version": (i, []),
        "hmoe_auto_path": (i, [P(LayerDesc), i, P(i)]),
        "hmoe_linear_packed_size": (i, [P(LinearDesc), P(sz)]),
        "hmoe_linear_workspace_size": (i, [P(LinearDesc), i, P(sz)]),
        "hmoe_linear_pack": (i, [P(LinearDesc), vp, vp, ctypes.c_float, vp, vp, P(vp)]),
        "hmoe_linear_forward": (i, [vp, vp, i, vp, vp, sz, vp]),
        "hmoe_linear_forward_ex": (i, [vp, vp, i, vp, vp, sz, P(ForwardOpts), vp]),
        "hmoe_linear_destroy": (None, [vp]),
        "hmoe_quantize_act_nvfp4": (i, [vp, i, i, i, ctypes.c_float, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        _LIB = load()
    return _LIB


def check(status):
    if status != HMOE_OK:
        raise HmoeError(status, lib().hmoe_last_error().decode())
    return status
