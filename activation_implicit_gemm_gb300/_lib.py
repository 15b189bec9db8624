"""ctypes declarations of the C ABI in include/fconv.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfconv.so")

F32, F16 = 0, 1
AUTO_PAD = {"NOTSET": 0, "SAME_UPPER": 1, "SAME_LOWER": 2, "VALID": 3}
ACTIVATIONS = {None: 0, "Relu": 1, "LeakyRelu": 2, "Sigmoid": 3, "Tanh": 4, "HardSigmoid": 5,
               "HardSwish": 6, "Clip": 7, "QuickGelu": 8, "Elu": 9, "Gelu": 10, "FastGelu": 11,
               "Softplus": 12, "ThresholdedRelu": 13, "Erf": 14}
ROUTES = {"auto": 0, "direct": 1, "igemm_tc": 2, "depthwise": 3, "grouped": 4,
          "transposed": 5}
ROUTE_NAMES = {v: k for k, v in ROUTES.items()}
PRECISIONS = {"default": 0, "half2_rows": 1}
STATUS = {0: "OK", 1: "E_NULL", 2: "E_RANK", 3: "E_ATTR_LENGTH", 4: "E_ATTR_VALUE",
          5: "E_PADS_WITH_AUTOPAD", 6: "E_KERNEL_SHAPE", 7: "E_GROUP", 8: "E_BIAS_SHAPE",
          9: "E_Z_SHAPE", 10: "E_ACT_PARAMS", 11: "E_ACTIVATION", 12: "E_OUTPUT_EMPTY",
          13: "E_WORKSPACE", 14: "E_UNSUPPORTED", 15: "E_CUDA", 16: "E_DEVICE_TIMEOUT",
          17: "E_NOMEM", 18: "E_ALIGNMENT", 19: "E_ALIAS"}

I64 = ctypes.c_int64


class FconvDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("rank", ctypes.c_int),
                ("x_shape", I64 * 5), ("w_shape", I64 * 5),
                ("has_bias", ctypes.c_int), ("bias_len", I64),
                ("has_z", ctypes.c_int), ("z_rank", ctypes.c_int), ("z_shape", I64 * 5),
                ("group", I64), ("auto_pad", ctypes.c_int),
                ("n_kernel_shape", ctypes.c_int), ("n_strides", ctypes.c_int),
                ("n_dilations", ctypes.c_int), ("n_pads", ctypes.c_int),
                ("kernel_shape", I64 * 3), ("strides", I64 * 3), ("dilations", I64 * 3),
                ("pads", I64 * 6),
                ("activation", ctypes.c_int), ("n_act_params", ctypes.c_int),
                ("act_params", ctypes.c_float * 2),
                ("transposed", ctypes.c_int), ("n_output_padding", ctypes.c_int),
                ("output_padding", I64 * 3)]


class FconvOptions(ctypes.Structure):
    _fields_ = [("route", ctypes.c_int), ("split_k", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("a_path", ctypes.c_int), ("max_ctas", ctypes.c_int),
                ("precision", ctypes.c_int)]


EXPORTS = ["fconv_plan_create", "fconv_plan_create_ex", "fconv_plan_output_shape",
           "fconv_plan_pads", "fconv_plan_workspace_size", "fconv_plan_route", "fconv_plan_work",
           "fconv_plan_launches",
           "fconv_run", "fconv_check_device", "fconv_destroy", "fconv_status_string",
           "fconv_version"]

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfconv.so; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(activation_implicit_gemm_gb300._build.build())")
    lib = ctypes.CDLL(path)
    P, vp = ctypes.POINTER, ctypes.c_void_p
    lib.fconv_plan_create.argtypes = [P(FconvDesc), ctypes.c_int, P(vp)]
    lib.fconv_plan_create_ex.argtypes = [P(FconvDesc), ctypes.c_int, P(FconvOptions), P(vp)]
    lib.fconv_plan_output_shape.argtypes = [vp, P(I64), P(ctypes.c_int)]
    lib.fconv_plan_pads.argtypes = [vp, P(I64), P(I64)]
    lib.fconv_plan_workspace_size.argtypes = [vp, P(ctypes.c_size_t)]
    lib.fconv_plan_route.argtypes = [vp, P(ctypes.c_int), P(ctypes.c_int), P(ctypes.c_int)]
    lib.fconv_plan_work.argtypes = [vp, P(ctypes.c_double), P(ctypes.c_double)]
    lib.fconv_plan_launches.argtypes = [vp, P(ctypes.c_int)]
    lib.fconv_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.fconv_check_device.argtypes = [vp]
    lib.fconv_destroy.argtypes = [vp]
    lib.fconv_destroy.restype = None
    lib.fconv_status_string.argtypes = [ctypes.c_int]
    lib.fconv_status_string.restype = ctypes.c_char_p
    for name in EXPORTS:
        f = getattr(lib, name)
        if name not in ("fconv_destroy", "fconv_status_string"):
            f.restype = ctypes.c_int
    _lib = lib
    return lib


def make_desc(dtype: int, x_shape, w_shape, *, has_bias: bool = False, bias_len: int = 0,
              z_shape=None, group: int = 1, strides=None, dilations=None, pads=None,
              auto_pad: str = "NOTSET", kernel_shape=None, activation=None,
              activation_params=None, transposed: bool = False,
              output_padding=None) -> FconvDesc:
    d = FconvDesc()
    d.dtype = dtype
    d.rank = len(x_shape) if len(x_shape) == len(w_shape) else -1
    for i, v in enumerate(list(x_shape)[:5]):
        d.x_shape[i] = int(v)
    for i, v in enumerate(list(w_shape)[:5]):
        d.w_shape[i] = int(v)
    d.has_bias = 1 if has_bias else 0
    d.bias_len = int(bias_len)
    if z_shape is not None:
        d.has_z = 1
        d.z_rank = len(z_shape)
        for i, v in enumerate(list(z_shape)[:5]):
            d.z_shape[i] = int(v)
    d.group = int(group)
    if auto_pad not in AUTO_PAD:
        raise ValueError(f"auto_pad must be one of {list(AUTO_PAD)}")
    d.auto_pad = AUTO_PAD[auto_pad]

    def put(arr, vals, cap):
        if vals is None:
            return 0
        vals = list(vals)
        for i, v in enumerate(vals[:cap]):
            arr[i] = int(v)
        return len(vals) if len(vals) <= cap else cap + 1

    d.n_kernel_shape = put(d.kernel_shape, kernel_shape, 3)
    d.n_strides = put(d.strides, strides, 3)
    d.n_dilations = put(d.dilations, dilations, 3)
    d.n_pads = put(d.pads, pads, 6)
    d.transposed = 1 if transposed else 0
    d.n_output_padding = put(d.output_padding, output_padding, 3)
    if activation not in ACTIVATIONS:
        raise ValueError(f"unknown activation {activation!r}")
    d.activation = ACTIVATIONS[activation]
    if activation_params is None:
        d.n_act_params = -1
    else:
        ap = list(activation_params)
        d.n_act_params = len(ap)
        for i, v in enumerate(ap[:2]):
            d.act_params[i] = float(v)
    return d
