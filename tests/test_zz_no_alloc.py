"""fconv_run_noalloc: the entry point for callers that cannot allocate device memory
(code inside allocator hooks or captures that must not allocate, host callbacks,
plugins whose host application owns every device allocation). The workspace a
tensor-core plan needs (the weight copy in GEMM order, X repacked for the A operand and
any split-K partial sums) comes from a fixed array inside the library instead of a
caller-supplied buffer.

Each plan runs through the C ABI on two calls in a row, with another plan run in between
so the shared array holds a different call's leftovers. Every output is compared with
fconv_run (the caller-workspace entry point) on the same plan and inputs, and with the
oracle, within the parity tolerance. This file is collected last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from activation_implicit_gemm_gb300 import FusedConvPlan, _build, _lib
from parity import check, tolerance

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


PLANS = [
    # (x_shape, w_shape, attrs, options): gathered A with split-K partials
    ((2, 32, 19, 21), (48, 32, 3, 3), dict(pads=[1, 1, 1, 1], activation="Gelu"),
     dict(split_k=3)),
    # C/group a multiple of 64: TMA boxes over X repacked in the array, split K
    ((3, 64, 8, 8), (40, 64, 3, 3), dict(pads=[1, 1, 1, 1], activation="QuickGelu"),
     dict(split_k=2, a_path="tma")),
    # the same without split-K
    ((2, 128, 9, 7), (72, 128, 3, 3), dict(pads=[1, 0, 1, 1]), dict(a_path="tma")),
]


@pytest.mark.parametrize("idx", range(len(PLANS)))
def test_noalloc_matches_fconv_run_and_oracle_on_two_calls(idx):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _build.build()
    run_noalloc = noalloc_fn()
    stream = torch.cuda.current_stream().cuda_stream

    xs, wsh, attrs, opts = PLANS[idx]
    plan = FusedConvPlan(_lib.F16, xs, wsh, has_bias=True, has_z=True, route="igemm_tc",
                         **opts, **attrs)
    assert 0 < plan.workspace_bytes <= SCRATCH_BYTES
    x, w, b, z = seeded(31 + 10 * idx, xs, wsh, attrs)
    xd, wd, bd, zd = (torch.from_numpy(a).cuda() for a in (x, w, b, z))

    # another plan, run through the no-allocation entry point between the two calls
    attrs2 = dict(strides=[2, 2], pads=[1, 1, 1, 1], activation="Relu")
    xs2, wsh2 = (3, 16, 30, 17), (64, 16, 3, 3)
    plan2 = FusedConvPlan(_lib.F16, xs2, wsh2, has_bias=True, has_z=True, route="igemm_tc",
                          split_k=2, **attrs2)
    x2, w2, b2, z2 = seeded(41, xs2, wsh2, attrs2)
    d2 = [torch.from_numpy(a).cuda() for a in (x2, w2, b2, z2)]

    y_run = plan.run(xd, wd, bd, zd)  # the caller-workspace entry point
    torch.cuda.synchronize()
    ref_run = y_run.double().cpu().numpy()
    ref, absacc = oracle.fused_conv(x, w, b, z, **attrs)
    kg = int(np.prod(wsh[1:]))
    tol = tolerance(ref, absacc, "f16", kg)

    for call in range(2):
        y = torch.full(plan.y_shape, float("nan"), dtype=torch.float16, device="cuda")
        st = run_noalloc(plan._ptr, xd.data_ptr(), wd.data_ptr(), bd.data_ptr(),
                         zd.data_ptr(), y.data_ptr(), stream)
        assert _lib.STATUS[st] == "OK", f"call {call}: {_lib.STATUS[st]}"
        torch.cuda.synchronize()
        got = y.double().cpu().numpy()
        err = np.abs(got - ref_run)
        assert np.all(err <= tol), f"call {call} vs fconv_run: max err {err.max():.3e}"
        check(got, ref, absacc, "f16", kg, activation=attrs.get("activation"),
              what=f"noalloc plan {idx} call {call} vs oracle")
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


def test_noalloc_runs_workspace_free_routes():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _build.build()
    run_noalloc = noalloc_fn()
    attrs = dict(group=8, pads=[1, 1, 1, 1], activation="Clip", activation_params=[-1.0, 1.0])
    xs, wsh = (2, 8, 12, 12), (8, 1, 3, 3)
    plan = FusedConvPlan(_lib.F16, xs, wsh, has_bias=True, has_z=True, route="depthwise",
                         **attrs)
    assert plan.workspace_bytes == 0
    x, w, b, z = seeded(61, xs, wsh, attrs)
    d = [torch.from_numpy(a).cuda() for a in (x, w, b, z)]
    y = torch.empty(plan.y_shape, dtype=torch.float16, device="cuda")
    st = run_noalloc(plan._ptr, *(t.data_ptr() for t in d), y.data_ptr(),
                     torch.cuda.current_stream().cuda_stream)
    assert _lib.STATUS[st] == "OK"
    torch.cuda.synchronize()
    ref, absacc = oracle.fused_conv(x, w, b, z, **attrs)
    check(y.double().cpu().numpy(), ref, absacc, "f16", 9, activation="Clip",
          what="noalloc depthwise")


def test_noalloc_runs_the_fp32_tensor_core_path():
    # the 3xTF32 plan's workspace holds W hi/lo, X hi/lo and the raw sums: all in the array
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _build.build()
    run_noalloc = noalloc_fn()
    xs, wsh = (2, 32, 9, 9), (40, 32, 3, 3)
    attrs = dict(pads=[1, 1, 1, 1], activation="Relu")
    plan = FusedConvPlan(_lib.F32, xs, wsh, has_bias=True, has_z=True, **attrs)
    assert plan.route == "igemm_tc" and 0 < plan.workspace_bytes <= SCRATCH_BYTES
    ys = oracle.output_shape(xs, wsh, **attrs)
    x = workloads.draw(71, xs, "normal", 1.0, "f32")
    w = workloads.draw(72, wsh, "normal", 1.0 / math.sqrt(32 * 9), "f32")
    b = workloads.draw(73, (40,), "normal", 1.0, "f32")
    z = workloads.draw(74, ys, "normal", 1.0, "f32")
    d = [torch.from_numpy(a).cuda() for a in (x, w, b, z)]
    y_run = plan.run(*d)
    torch.cuda.synchronize()
    ref, absacc = oracle.fused_conv(x, w, b, z, **attrs)
    for call in range(2):
        y = torch.full(plan.y_shape, float("nan"), dtype=torch.float32, device="cuda")
        st = run_noalloc(plan._ptr, *(t.data_ptr() for t in d), y.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
        assert _lib.STATUS[st] == "OK", f"call {call}: {_lib.STATUS[st]}"
        torch.cuda.synchronize()
        assert torch.equal(y, y_run)
        check(y.double().cpu().numpy(), ref, absacc, "f32", 32 * 9, activation="Relu",
              what=f"noalloc tf32 call {call}")
