"""fconv_run_noalloc: the entry point for callers that cannot allocate device memory
(code inside allocator hooks or captures that must not allocate, host callbacks,
plugins whose host application owns every device allocation). Its split-K scratch is a
fixed array inside the library instead of a caller-supplied workspace.

Checked through the C ABI against fconv_run (the caller-workspace entry point) on
the same plan and inputs, on two calls in a row, with another plan run in between so
the shared scratch holds a different call's leftovers. This file is collected last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from activation_implicit_gemm_gb300 import FusedConvPlan, _build, _lib
from parity import tolerance

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 * 1024 * 1024


def noalloc_fn():
    lib = _lib.load()
    f = lib.fconv_run_noalloc
    f.argtypes = [ctypes.c_void_p] * 7
    f.restype = ctypes.c_int
    return f


def seeded(seed, x_shape, w_shape, attrs):
    ys = oracle.output_shape(x_shape, w_shape, **attrs)
    kg = int(np.prod(w_shape[1:]))
    x = workloads.draw(seed, x_shape, "normal", 1.0, "f16")
    w = workloads.draw(seed + 1, w_shape, "normal", 1.0 / math.sqrt(kg), "f16")
    b = workloads.draw(seed + 2, (w_shape[0],), "normal", 1.0, "f16")
    z = workloads.draw(seed + 3, ys, "normal", 1.0, "f16")
    return x, w, b, z


def test_noalloc_matches_fconv_run_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _build.build()
    run_noalloc = noalloc_fn()
    stream = torch.cuda.current_stream().cuda_stream

    attrs = dict(pads=[1, 1, 1, 1], activation="Gelu")
    xs, wsh = (2, 32, 19, 21), (48, 32, 3, 3)
    plan = FusedConvPlan(_lib.F16, xs, wsh, has_bias=True, has_z=True, route="igemm_tc",
                         split_k=3, **attrs)
    assert plan.split_k == 3 and 0 < plan.workspace_bytes <= SCRATCH_BYTES
    x, w, b, z = seeded(31, xs, wsh, attrs)
    xd, wd, bd, zd = (torch.from_numpy(a).cuda() for a in (x, w, b, z))

    # the other plan, run through the no-allocation entry point between the two calls
    attrs2 = dict(strides=[2, 2], pads=[1, 1, 1, 1], activation="Relu")
    xs2, wsh2 = (3, 16, 30, 17), (64, 16, 3, 3)
    plan2 = FusedConvPlan(_lib.F16, xs2, wsh2, has_bias=True, has_z=True, route="igemm_tc",
                          split_k=2, **attrs2)
    x2, w2, b2, z2 = seeded(41, xs2, wsh2, attrs2)
    d2 = [torch.from_numpy(a).cuda() for a in (x2, w2, b2, z2)]

    y_ref = plan.run(xd, wd, bd, zd)  # existing entry point, torch-allocated workspace
    torch.cuda.synchronize()
    _, absacc = oracle.fused_conv(x, w, b, z, **attrs)
    ref = y_ref.double().cpu().numpy()
    tol = tolerance(ref, absacc, "f16", int(np.prod(wsh[1:])))

    for call in range(2):
        y = torch.full(plan.y_shape, float("nan"), dtype=torch.float16, device="cuda")
        st = run_noalloc(plan._ptr, xd.data_ptr(), wd.data_ptr(), bd.data_ptr(),
                         zd.data_ptr(), y.data_ptr(), stream)
        assert _lib.STATUS[st] == "OK", f"call {call}: {_lib.STATUS[st]}"
        torch.cuda.synchronize()
        got = y.double().cpu().numpy()
        err = np.abs(got - ref)
        assert np.all(err <= tol), f"call {call}: max err {err.max():.3e}"
        y2 = torch.empty(plan2.y_shape, dtype=torch.float16, device="cuda")
        st = run_noalloc(plan2._ptr, *(t.data_ptr() for t in d2), y2.data_ptr(), stream)
        assert _lib.STATUS[st] == "OK"
        torch.cuda.synchronize()
        y2_ref = plan2.run(*d2)
        torch.cuda.synchronize()
        assert torch.equal(y2, y2_ref)
    assert _lib.load().fconv_check_device(None) == 0


def test_noalloc_rejects_plans_beyond_the_scratch_size():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _build.build()
    run_noalloc = noalloc_fn()
    # 4 splits x 4 B x 2*64*128*128 outputs = 32 MiB > 16 MiB
    plan = FusedConvPlan(_lib.F16, (2, 64, 128, 128), (64, 64, 3, 3), pads=[1, 1, 1, 1],
                         route="igemm_tc", split_k=4)
    assert plan.workspace_bytes > SCRATCH_BYTES
    y = torch.full(plan.y_shape, 3.0, dtype=torch.float16, device="cuda")
    x = torch.zeros(plan.x_shape, dtype=torch.float16, device="cuda")
    w = torch.zeros(plan.w_shape, dtype=torch.float16, device="cuda")
    st = run_noalloc(plan._ptr, x.data_ptr(), w.data_ptr(), None, None, y.data_ptr(), None)
    assert _lib.STATUS[st] == "E_WORKSPACE"
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())
