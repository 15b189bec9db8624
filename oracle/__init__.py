"""FusedConv CPU oracle (double precision) -- TEST INFRASTRUCTURE ONLY.

Only the tests, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg import
this package. The product library never does. The arithmetic lives in
`fconv_oracle.c` (plain C, built with gcc); this module marshals numpy arrays.
See that file's header for the passages each part follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fconv_oracle.c")
_LIB = os.path.join(_HERE, "libfconv_oracle.so")

ACTIVATIONS = ["Relu", "LeakyRelu", "Sigmoid", "Tanh", "HardSigmoid", "HardSwish", "Clip",
               "QuickGelu", "Elu", "Gelu", "FastGelu", "Softplus", "ThresholdedRelu", "Erf"]
AUTO_PAD = {"NOTSET": 0, "SAME_UPPER": 1, "SAME_LOWER": 2, "VALID": 3}
STATUS = {0: "OK", 1: "BAD_RANK", 2: "ATTR_LENGTH", 3: "ATTR_VALUE", 4: "PADS_AUTOPAD",
          5: "KERNEL_SHAPE", 6: "GROUP", 7: "ACT_PARAMS", 8: "ACTIVATION",
          9: "EMPTY_OUTPUT", 10: "NULL"}


class _Attrs(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int),
                ("x_shape", ctypes.c_int64 * 5),
                ("w_shape", ctypes.c_int64 * 5),
                ("group", ctypes.c_int64),
                ("auto_pad", ctypes.c_int),
                ("n_kernel_shape", ctypes.c_int),
                ("n_strides", ctypes.c_int),
                ("n_dilations", ctypes.c_int),
                ("n_pads", ctypes.c_int),
                ("kernel_shape", ctypes.c_int64 * 3),
                ("strides", ctypes.c_int64 * 3),
                ("dilations", ctypes.c_int64 * 3),
                ("pads", ctypes.c_int64 * 6),
                ("activation", ctypes.c_int),
                ("n_act_params", ctypes.c_int),
                ("act_params", ctypes.c_double * 2)]


class _TAttrs(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int),
                ("x_shape", ctypes.c_int64 * 5),
                ("w_shape", ctypes.c_int64 * 5),
                ("group", ctypes.c_int64),
                ("n_strides", ctypes.c_int),
                ("n_dilations", ctypes.c_int),
                ("n_pads", ctypes.c_int),
                ("n_output_padding", ctypes.c_int),
                ("strides", ctypes.c_int64 * 3),
                ("dilations", ctypes.c_int64 * 3),
                ("pads", ctypes.c_int64 * 6),
                ("output_padding", ctypes.c_int64 * 3),
                ("activation", ctypes.c_int),
                ("n_act_params", ctypes.c_int),
                ("act_params", ctypes.c_double * 2)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP) unless an up-to-date library exists."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        _lib.oracle_output_shape.argtypes = [P(_Attrs), P(ctypes.c_int64), P(ctypes.c_int64),
                                             P(ctypes.c_int64)]
        _lib.oracle_output_shape.restype = ctypes.c_int
        _lib.oracle_fused_conv.argtypes = [P(_Attrs)] + [ctypes.c_void_p] * 6 + [ctypes.c_int]
        _lib.oracle_fused_conv.restype = ctypes.c_int
        _lib.oracle_activation.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                           ctypes.c_double]
        _lib.oracle_activation.restype = ctypes.c_double
        _lib.oracle_max_threads.restype = ctypes.c_int
        _lib.oracle_transpose_output_shape.argtypes = [P(_TAttrs), P(ctypes.c_int64)]
        _lib.oracle_transpose_output_shape.restype = ctypes.c_int
        _lib.oracle_conv_transpose.argtypes = [P(_TAttrs)] + [ctypes.c_void_p] * 6 + [ctypes.c_int]
        _lib.oracle_conv_transpose.restype = ctypes.c_int
    return _lib


def act_id(name: Optional[str]) -> int:
    if name is None:
        return 0
    return ACTIVATIONS.index(name) + 1


def make_attrs(x_shape: Sequence[int], w_shape: Sequence[int], group: int = 1,
               strides=None, dilations=None, pads=None, auto_pad: str = "NOTSET",
               kernel_shape=None, activation: Optional[str] = None,
               activation_params=None) -> _Attrs:
    a = _Attrs()
    a.rank = len(x_shape)
    if len(w_shape) != len(x_shape) or not 3 <= len(x_shape) <= 5:
        a.rank = 0
    for i, v in enumerate(list(x_shape)[:5]):
        a.x_shape[i] = int(v)
    for i, v in enumerate(list(w_shape)[:5]):
        a.w_shape[i] = int(v)
    a.group = int(group)
    a.auto_pad = AUTO_PAD[auto_pad]

    def put(arr, vals, cap):
        if vals is None:
            return 0
        vals = list(vals)
        for i, v in enumerate(vals[:cap]):
            arr[i] = int(v)
        return len(vals) if len(vals) <= cap else cap + 1

    a.n_kernel_shape = put(a.kernel_shape, kernel_shape, 3)
    a.n_strides = put(a.strides, strides, 3)
    a.n_dilations = put(a.dilations, dilations, 3)
    a.n_pads = put(a.pads, pads, 6)
    a.activation = act_id(activation)
    if activation_params is None:
        a.n_act_params = -1
    else:
        ap = list(activation_params)
        a.n_act_params = len(ap)
        for i, v in enumerate(ap[:2]):
            a.act_params[i] = float(v)
    return a


def resolve(x_shape, w_shape, **attrs):
    """(status name, y_shape, pad_begin[d,h,w], pad_end[d,h,w])."""
    a = make_attrs(x_shape, w_shape, **attrs)
    ys = (ctypes.c_int64 * 5)()
    pb = (ctypes.c_int64 * 3)()
    pe = (ctypes.c_int64 * 3)()
    st = lib().oracle_output_shape(ctypes.byref(a), ys, pb, pe)
    if st != 0:
        return STATUS[st], None, None, None
    return "OK", tuple(ys[i] for i in range(len(x_shape))), tuple(pb), tuple(pe)


def output_shape(x_shape, w_shape, **attrs):
    st, ys, _, _ = resolve(x_shape, w_shape, **attrs)
    if st != "OK":
        raise ValueError(f"oracle rejects the attributes: {st}")
    return ys


def fused_conv(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray] = None,
               z: Optional[np.ndarray] = None, nthreads: int = 0, **attrs):
    """Y (float64, unrounded) and sum |x*w| per output, from dtype-rounded inputs."""
    ys = output_shape(x.shape, w.shape, **attrs)
    a = make_attrs(x.shape, w.shape, **attrs)
    xd = np.ascontiguousarray(x, dtype=np.float64)
    wd = np.ascontiguousarray(w, dtype=np.float64)
    bd = None if b is None else np.ascontiguousarray(b, dtype=np.float64)
    zd = None if z is None else np.ascontiguousarray(z, dtype=np.float64)
    if bd is not None and bd.shape != (w.shape[0],):
        raise ValueError("bias must be rank 1 with length M")
    if zd is not None and zd.shape != tuple(ys):
        raise ValueError("Z must have the shape of Y")
    y = np.empty(ys, dtype=np.float64)
    s = np.empty(ys, dtype=np.float64)

    def ptr(arr):
        return None if arr is None else arr.ctypes.data_as(ctypes.c_void_p)

    st = lib().oracle_fused_conv(ctypes.byref(a), ptr(xd), ptr(wd), ptr(bd), ptr(zd), ptr(y),
                                 ptr(s), int(nthreads))
    if st != 0:
        raise ValueError(f"oracle failed: {STATUS[st]}")
    return y, s


def make_tattrs(x_shape, w_shape, group: int = 1, strides=None, dilations=None, pads=None,
                output_padding=None, activation: Optional[str] = None,
                activation_params=None) -> _TAttrs:
    a = _TAttrs()
    a.rank = len(x_shape)
    if len(w_shape) != len(x_shape) or not 3 <= len(x_shape) <= 5:
        a.rank = 0
    for i, v in enumerate(list(x_shape)[:5]):
        a.x_shape[i] = int(v)
    for i, v in enumerate(list(w_shape)[:5]):
        a.w_shape[i] = int(v)
    a.group = int(group)

    def put(arr, vals, cap):
        if vals is None:
            return 0
        vals = list(vals)
        for i, v in enumerate(vals[:cap]):
            arr[i] = int(v)
        return len(vals) if len(vals) <= cap else cap + 1

    a.n_strides = put(a.strides, strides, 3)
    a.n_dilations = put(a.dilations, dilations, 3)
    a.n_pads = put(a.pads, pads, 6)
    a.n_output_padding = put(a.output_padding, output_padding, 3)
    a.activation = act_id(activation)
    if activation_params is None:
        a.n_act_params = -1
    else:
        ap = list(activation_params)
        a.n_act_params = len(ap)
        for i, v in enumerate(ap[:2]):
            a.act_params[i] = float(v)
    return a


def transpose_resolve(x_shape, w_shape, **attrs):
    """(status name, y_shape) of a transposed convolution."""
    a = make_tattrs(x_shape, w_shape, **attrs)
    ys = (ctypes.c_int64 * 5)()
    st = lib().oracle_transpose_output_shape(ctypes.byref(a), ys)
    if st != 0:
        return STATUS[st], None
    return "OK", tuple(ys[i] for i in range(len(x_shape)))


def transpose_output_shape(x_shape, w_shape, **attrs):
    st, ys = transpose_resolve(x_shape, w_shape, **attrs)
    if st != "OK":
        raise ValueError(f"oracle rejects the attributes: {st}")
    return ys


def conv_transpose(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray] = None,
                   z: Optional[np.ndarray] = None, nthreads: int = 0, **attrs):
    """Transposed convolution with the fused epilogue: Y (float64, unrounded) and
    sum |x*w| per output, from dtype-rounded inputs. W is (C, M/group, kernel...)."""
    ys = transpose_output_shape(x.shape, w.shape, **attrs)
    a = make_tattrs(x.shape, w.shape, **attrs)
    xd = np.ascontiguousarray(x, dtype=np.float64)
    wd = np.ascontiguousarray(w, dtype=np.float64)
    bd = None if b is None else np.ascontiguousarray(b, dtype=np.float64)
    zd = None if z is None else np.ascontiguousarray(z, dtype=np.float64)
    if bd is not None and bd.shape != (ys[1],):
        raise ValueError("bias must be rank 1 with length M")
    if zd is not None and zd.shape != tuple(ys):
        raise ValueError("Z must have the shape of Y")
    y = np.empty(ys, dtype=np.float64)
    s = np.empty(ys, dtype=np.float64)

    def ptr(arr):
        return None if arr is None else arr.ctypes.data_as(ctypes.c_void_p)

    st = lib().oracle_conv_transpose(ctypes.byref(a), ptr(xd), ptr(wd), ptr(bd), ptr(zd),
                                     ptr(y), ptr(s), int(nthreads))
    if st != 0:
        raise ValueError(f"oracle failed: {STATUS[st]}")
    return y, s


def activation(name: Optional[str], v: float, alpha: float = 0.0, beta: float = 0.0) -> float:
    """The oracle's activation of one value (alpha/beta as already resolved)."""
    return lib().oracle_activation(act_id(name), float(v), float(alpha), float(beta))


def max_threads() -> int:
    return lib().oracle_max_threads()
