"""ctypes view of the C ABI in include/fp8lin.h (argument marshalling only).

The shared library is built in-tree by scaled_quantize_fp8_gb300.build; loading fails loudly
when it is missing. There is no fallback implementation of any entry point.
"""
import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8lin.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fp8lin.h")
HEADER_DIR = os.path.dirname(HEADER_PATH)

FP8_OK = 0
STATUS_NAMES = {0: "FP8_OK", 1: "FP8_ERR_NULL", 2: "FP8_ERR_ALIGN", 3: "FP8_ERR_SHAPE",
                4: "FP8_ERR_UNSUPPORTED", 5: "FP8_ERR_CUDA", 6: "FP8_ERR_TIMEOUT",
                7: "FP8_ERR_WORKSPACE"}

RECIPE_DELAYED, RECIPE_TENSORWISE, RECIPE_MXFP8, RECIPE_BLOCKWISE = 0, 1, 2, 3
FORMAT_E4M3, FORMAT_HYBRID = 0, 1
ROLE_ACTIVATION, ROLE_WEIGHT, ROLE_GRAD = 0, 1, 2


class Recipe(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("format", ctypes.c_int32), ("margin", ctypes.c_int32),
                ("amax_history_len", ctypes.c_int32), ("amax_compute_algo", ctypes.c_int32),
                ("fp8_wgrad", ctypes.c_int32), ("power_2_scales", ctypes.c_int32)]


class Tensor(ctypes.Structure):
    _fields_ = [("row", ctypes.c_void_p), ("col", ctypes.c_void_p),
                ("row_scale", ctypes.c_void_p), ("col_scale", ctypes.c_void_p),
                ("amax", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("scale_inv", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("kind", ctypes.c_int32), ("role", ctypes.c_int32),
                ("col_bf16", ctypes.c_int32)]


QUANTIZE_GROUP_MAX = 4


class QuantizeItem(ctypes.Structure):
    _fields_ = [("x_bf16", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("role", ctypes.c_int32), ("want_row", ctypes.c_int32),
                ("want_col", ctypes.c_int32), ("out", ctypes.POINTER(Tensor))]


class AmaxHistory(ctypes.Structure):
    _fields_ = [("history", ctypes.c_void_p), ("head", ctypes.c_void_p), ("len", ctypes.c_int32)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SIG = {
    "fp8_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Recipe), _I64, _I64]),
    "fp8_quantize": (_I32, [ctypes.POINTER(Recipe), _P, _I64, _I64, _I32, _I32, _I32,
                            ctypes.POINTER(Tensor), _P, ctypes.c_size_t, _P, _P]),
    "fp8_quantize_group": (_I32, [ctypes.POINTER(Recipe), _I32, ctypes.POINTER(QuantizeItem),
                                  _P, _P]),
    "fp8_test_quantize_group_stalled": (_I32, [ctypes.POINTER(Recipe), _I32,
                                               ctypes.POINTER(QuantizeItem), _P, _P]),
    "fp8_quantize_master": (_I32, [ctypes.POINTER(Recipe), _P, _I64, _I64, _I32, _I32,
                                   ctypes.POINTER(Tensor), _P, ctypes.c_size_t, _P, _P]),
    "fp8_amax_update": (_I32, [ctypes.POINTER(Recipe), ctypes.POINTER(AmaxHistory), _I32, _P,
                               _P, _P, _P]),
    "fp8_linear_fwd": (_I32, [ctypes.POINTER(Recipe), ctypes.POINTER(Tensor),
                              ctypes.POINTER(Tensor), _P, _I32, _P, _P]),
    "fp8_test_quantize_stalled": (_I32, [ctypes.POINTER(Recipe), _P, _I64, _I64, _I32, _I32,
                                         _I32, ctypes.POINTER(Tensor), _P, ctypes.c_size_t,
                                         _P, _P]),
    "fp8_test_linear_fwd_stalled": (_I32, [ctypes.POINTER(Recipe), ctypes.POINTER(Tensor),
                                           ctypes.POINTER(Tensor), _P, _P, _P]),
    "fp8_linear_bwd": (_I32, [ctypes.POINTER(Recipe), ctypes.POINTER(Tensor),
                              ctypes.POINTER(Tensor), ctypes.POINTER(Tensor), _P, _P, _I32, _P,
                              _P]),
    "fp8_gelu_quantize": (_I32, [ctypes.POINTER(Recipe), _P, _I64, _I64, _P,
                                 ctypes.POINTER(Tensor), ctypes.POINTER(Tensor), _P, _P]),
    "fp8_dgelu_quantize": (_I32, [ctypes.POINTER(Recipe), _P, ctypes.POINTER(Tensor), _P,
                                  ctypes.POINTER(Tensor), _P, _P]),
    "fp8_linear_fwd_gelu": (_I32, [ctypes.POINTER(Recipe), ctypes.POINTER(Tensor),
                                   ctypes.POINTER(Tensor), ctypes.POINTER(Tensor),
                                   ctypes.POINTER(Tensor), _P, _P]),
    "fp8_linear_dgrad_dgelu": (_I32, [ctypes.POINTER(Recipe), ctypes.POINTER(Tensor),
                                      ctypes.POINTER(Tensor), ctypes.POINTER(Tensor),
                                      ctypes.POINTER(Tensor), _P, _P]),
    "fp8_quantize_static_scratch": (_I32, [ctypes.POINTER(Recipe), _P, _I64, _I64, _I32, _I32,
                                           _I32, ctypes.POINTER(Tensor), _P, _P]),
    "fp8_status_str": (ctypes.c_char_p, [_I32]),
    "fp8_last_cuda_error": (ctypes.c_char_p, []),
}

_lib = None


def header_functions():
    """Names of every function the headers in include/ declare (the public ABI and its test
    hooks)."""
    names = set()
    for h in sorted(os.listdir(HEADER_DIR)):
        if h.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, h)).read()
            names |= set(re.findall(r"^\s*(?:fp8_status|size_t|const char \*)\s*(fp8_\w+)\s*\(",
                                    text, flags=re.M))
    return sorted(names)


def load():
    """Load libfp8lin.so (raises if it has not been built) and bind the prototypes."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "scaled_quantize_fp8_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class Fp8Error(RuntimeError):
    def __init__(self, status, where=""):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)}")


def check(status, where):
    if status != FP8_OK:
        if status == 5 and _lib is not None:
            where = f"{where} ({_lib.fp8_last_cuda_error().decode()})"
        raise Fp8Error(status, where)
