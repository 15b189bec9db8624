"""FusedConv for GB300: Y = act(conv(X, W) + B + Z), 1-3 spatial dims, fp16/fp32.

A thin Python binding over the C ABI of libfconv.so (include/fconv.h). PyTorch only
provides device memory and streams; every step of the convolution runs in the
library's CUDA kernels. There is no CPU path: without the built library every call
raises.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

from . import _lib
from ._lib import ROUTES, ROUTE_NAMES, STATUS

__all__ = ["FconvError", "FusedConvPlan", "fused_conv", "conv_transpose", "plan_for", "load_library",
           "build"]


class FconvError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        self.code = STATUS.get(status, str(status))
        msg = _lib.load().fconv_status_string(status).decode()
        super().__init__(f"{where}: {self.code} ({msg})" if where else f"{self.code} ({msg})")


def load_library() -> ctypes.CDLL:
    return _lib.load()


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def _check(st: int, where: str):
    if st != 0:
        raise FconvError(st, where)


def _dtype_code(torch_dtype) -> int:
    import torch
    if torch_dtype == torch.float16:
        return _lib.F16
    if torch_dtype == torch.float32:
        return _lib.F32
    raise FconvError(14, f"dtype {torch_dtype}")


class FusedConvPlan:
    """A validated FusedConv request: output shape, applied pads, route and workspace."""

    def __init__(self, dtype: int, x_shape: Sequence[int], w_shape: Sequence[int], *,
                 has_bias: bool = False, has_z: bool = False, group: int = 1, strides=None,
                 dilations=None, pads=None, auto_pad: str = "NOTSET", kernel_shape=None,
                 activation: Optional[str] = None, activation_params=None, device: int = -1,
                 route: str = "auto", split_k: int = 0, tile_n: int = 0, z_shape=None,
                 a_path: str = "auto", max_ctas: int = 0, transposed: bool = False,
                 output_padding=None, precision: str = "default"):
        lib = _lib.load()
        self._lib = lib
        self._ptr = ctypes.c_void_p()
        self.dtype = dtype
        self.x_shape = tuple(int(v) for v in x_shape)
        self.w_shape = tuple(int(v) for v in w_shape)
        self.has_bias = bool(has_bias)
        self.has_z = bool(has_z)
        # B has M entries: W.dim0 for the direct form, W.dim1 * group for the transposed one
        if transposed:
            bias_len = int(w_shape[1]) * int(group) if len(w_shape) > 1 else 0
        else:
            bias_len = int(w_shape[0]) if len(w_shape) else 0
        # Z must match Y; when the caller does not give Z's shape, derive Y's first.
        if has_z and z_shape is None:
            probe = _lib.make_desc(dtype, x_shape, w_shape, has_bias=has_bias,
                                   bias_len=bias_len, group=group,
                                   strides=strides, dilations=dilations, pads=pads,
                                   auto_pad=auto_pad, kernel_shape=kernel_shape,
                                   activation=activation, activation_params=activation_params,
                                   transposed=transposed, output_padding=output_padding)
            tmp = ctypes.c_void_p()
            _check(lib.fconv_plan_create(ctypes.byref(probe), device, ctypes.byref(tmp)),
                   "fconv_plan_create")
            ys = (ctypes.c_int64 * 5)()
            rk = ctypes.c_int()
            lib.fconv_plan_output_shape(tmp, ys, ctypes.byref(rk))
            lib.fconv_destroy(tmp)
            z_shape = tuple(ys[i] for i in range(rk.value))
        desc = _lib.make_desc(dtype, x_shape, w_shape, has_bias=has_bias,
                              bias_len=bias_len,
                              z_shape=z_shape if has_z else None, group=group, strides=strides,
                              dilations=dilations, pads=pads, auto_pad=auto_pad,
                              kernel_shape=kernel_shape, activation=activation,
                              activation_params=activation_params, transposed=transposed,
                              output_padding=output_padding)
        opts = _lib.FconvOptions(ROUTES[route], int(split_k), int(tile_n),
                                 {"auto": 0, "gather": 1, "tma": 2}[a_path], int(max_ctas),
                                 _lib.PRECISIONS[precision])
        self.precision = precision
        _check(lib.fconv_plan_create_ex(ctypes.byref(desc), device, ctypes.byref(opts),
                                        ctypes.byref(self._ptr)), "fconv_plan_create")
        ys = (ctypes.c_int64 * 5)()
        rk = ctypes.c_int()
        _check(lib.fconv_plan_output_shape(self._ptr, ys, ctypes.byref(rk)), "output_shape")
        self.y_shape = tuple(ys[i] for i in range(rk.value))
        ws = ctypes.c_size_t()
        _check(lib.fconv_plan_workspace_size(self._ptr, ctypes.byref(ws)), "workspace_size")
        self.workspace_bytes = ws.value
        r, t, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(lib.fconv_plan_route(self._ptr, ctypes.byref(r), ctypes.byref(t),
                                    ctypes.byref(s)), "route")
        self.route = ROUTE_NAMES[r.value]
        self.tile_n = t.value
        self.split_k = s.value
        fl, by = ctypes.c_double(), ctypes.c_double()
        _check(lib.fconv_plan_work(self._ptr, ctypes.byref(fl), ctypes.byref(by)), "work")
        self.flops = fl.value
        self.bytes = by.value
        nl = ctypes.c_int()
        _check(lib.fconv_plan_launches(self._ptr, ctypes.byref(nl)), "launches")
        self.launches = nl.value
        pb, pe = (ctypes.c_int64 * 3)(), (ctypes.c_int64 * 3)()
        _check(lib.fconv_plan_pads(self._ptr, pb, pe), "pads")
        self.pad_begin = tuple(pb)
        self.pad_end = tuple(pe)

    def run_ptrs(self, x: int, w: int, b: int, z: int, y: int, ws: int, ws_bytes: int,
                 stream: int) -> None:
        """Enqueue on raw device pointers (ints; 0 for absent B, Z or workspace)."""
        _check(self._lib.fconv_run(self._ptr, x or None, w or None, b or None, z or None,
                                   y or None, ws or None, ws_bytes, stream or None), "fconv_run")

    def run(self, x, w, b=None, z=None, y=None, workspace=None, stream=None):
        """Run on torch CUDA tensors; allocates Y and the workspace when not given."""
        import torch
        if y is None:
            y = torch.empty(self.y_shape, dtype=x.dtype, device=x.device)
        if workspace is None and self.workspace_bytes:
            workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=x.device)
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        for t in (x, w, b, z, y):
            if t is not None and not t.is_contiguous():
                raise ValueError("FusedConv tensors must be contiguous")
        self.run_ptrs(x.data_ptr(), w.data_ptr(), 0 if b is None else b.data_ptr(),
                      0 if z is None else z.data_ptr(), y.data_ptr(),
                      0 if workspace is None else workspace.data_ptr(),
                      0 if workspace is None else workspace.numel() * workspace.element_size(),
                      stream.cuda_stream)
        return y

    def __del__(self):
        try:
            if self._ptr:
                self._lib.fconv_destroy(self._ptr)
                self._ptr = ctypes.c_void_p()
        except Exception:
            pass


_plans: dict = {}


def plan_for(x, w, b=None, z=None, **attrs) -> FusedConvPlan:
    """Cached plan for torch tensors x, w (and the presence of b, z)."""
    dtype = _dtype_code(x.dtype)
    key = (dtype, tuple(x.shape), tuple(w.shape), b is not None,
           None if z is None else tuple(z.shape), x.device.index,
           tuple(sorted((k, tuple(v) if isinstance(v, (list, tuple)) else v)
                        for k, v in attrs.items())))
    p = _plans.get(key)
    if p is None:
        m = w.shape[1] * attrs.get("group", 1) if attrs.get("transposed") else w.shape[0]
        if b is not None and (b.dim() != 1 or b.shape[0] != m):
            raise FconvError(8, "bias")
        p = FusedConvPlan(dtype, x.shape, w.shape, has_bias=b is not None,
                          has_z=z is not None,
                          z_shape=None if z is None else tuple(z.shape),
                          device=x.device.index if x.device.index is not None else -1,
                          **attrs)
        _plans[key] = p
    return p


def fused_conv(x, w, b=None, z=None, *, group: int = 1, strides=None, dilations=None,
               pads=None, auto_pad: str = "NOTSET", kernel_shape=None,
               activation: Optional[str] = None, activation_params=None, out=None,
               route: str = "auto", split_k: int = 0, tile_n: int = 0, a_path: str = "auto",
               max_ctas: int = 0):
    """Y = act(conv(X, W) + B + Z) on CUDA tensors (the operator's ONNX-style attributes)."""
    if not x.is_cuda:
        raise ValueError("fused_conv runs on CUDA tensors only")
    p = plan_for(x, w, b, z, group=group, strides=strides, dilations=dilations, pads=pads,
                 auto_pad=auto_pad, kernel_shape=kernel_shape, activation=activation,
                 activation_params=activation_params, route=route, split_k=split_k,
                 tile_n=tile_n, a_path=a_path, max_ctas=max_ctas)
    return p.run(x, w, b, z, y=out)


def conv_transpose(x, w, b=None, z=None, *, group: int = 1, strides=None, dilations=None,
                   pads=None, output_padding=None, activation: Optional[str] = None,
                   activation_params=None, out=None):
    """Y = act(convT(X, W) + B + Z) on CUDA tensors: the transposed convolution in gather
    form, W of shape (C, M/group, kernel...)."""
    if not x.is_cuda:
        raise ValueError("conv_transpose runs on CUDA tensors only")
    p = plan_for(x, w, b, z, group=group, strides=strides, dilations=dilations, pads=pads,
                 activation=activation, activation_params=activation_params, transposed=True,
                 output_padding=output_padding)
    return p.run(x, w, b, z, y=out)
