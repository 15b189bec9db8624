"""GPU parity of the transposed FusedConv (gather form, ExecuTorch WebGPU PR #20849) against
the oracle's scatter-form definition, element by element, through the C ABI.

Cases span 1-3 spatial dims, groups, strides 1-3, dilation, asymmetric pads, output_padding,
several output tiles along each axis with ragged tails, more input channels than one
shared-memory chunk holds and more output channels than one channel block, fp16 and fp32,
B, Z and activations; an integer-valued case must match bit for bit. Y sits between NaN-free
guard bands pre-filled with 7 and is itself pre-filled with NaN.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from activation_implicit_gemm_gb300 import FusedConvPlan, _build, _lib
from parity import check

pytestmark = pytest.mark.gpu

GUARD = 64


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _build.build()
    _lib.load()
    yield
    assert _lib.load().fconv_check_device(None) == 0


def to_dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_plan(plan, x, w, b, z, dtype):
    tdt = torch.float16 if dtype == "f16" else torch.float32
    ny = int(np.prod(plan.y_shape))
    buf = torch.full((ny + 2 * GUARD,), float("nan"), dtype=tdt, device="cuda")
    buf[:GUARD] = 7.0
    buf[-GUARD:] = 7.0
    y = buf[GUARD:GUARD + ny].view(plan.y_shape)
    plan.run(to_dev(x), to_dev(w), to_dev(b), to_dev(z), y=y)
    torch.cuda.synchronize()
    assert np.all(buf[:GUARD].float().cpu().numpy() == 7.0), "write before Y"
    assert np.all(buf[-GUARD:].float().cpu().numpy() == 7.0), "write after Y"
    return y.double().cpu().numpy()


def inputs(seed, dtype, xs, ws, attrs, bias=True, zres=True):
    ys = oracle.transpose_output_shape(xs, ws, **attrs)
    kg = int(ws[0] // attrs.get("group", 1)) * int(np.prod(ws[2:]))
    x = workloads.draw(seed, xs, "normal", 1.0, dtype)
    w = workloads.draw(seed + 1, ws, "normal", 1.0 / math.sqrt(kg), dtype)
    b = workloads.draw(seed + 2, (ys[1],), "normal", 1.0, dtype) if bias else None
    z = workloads.draw(seed + 3, ys, "normal", 1.0, dtype) if zres else None
    return x, w, b, z


def compare(dtype, x, w, b, z, attrs, what=""):
    dt = _lib.F16 if dtype == "f16" else _lib.F32
    plan = FusedConvPlan(dt, x.shape, w.shape, has_bias=b is not None, has_z=z is not None,
                         transposed=True, **attrs)
    assert plan.route == "transposed"
    y = run_plan(plan, x, w, b, z, dtype)
    ref, absacc = oracle.conv_transpose(x, w, b, z, **attrs)
    kg = int(w.shape[0] // attrs.get("group", 1)) * int(np.prod(w.shape[2:]))
    check(y, ref, absacc, dtype, kg, activation=attrs.get("activation"), what=what)


CASES = [
    # (x_shape, w_shape (C, M/group, k...), attrs)
    ((2, 6, 17), (6, 5, 4), dict(strides=[2], pads=[1, 2], output_padding=[1])),
    ((3, 4, 40), (4, 3, 3), dict(group=2, strides=[3], dilations=[2], pads=[0, 1],
                                 output_padding=[2], activation="Relu")),
    ((2, 8, 9, 11), (8, 4, 4, 4), dict(strides=[2, 2], pads=[1, 1, 1, 1],
                                       activation="LeakyRelu", activation_params=[0.1])),
    ((1, 12, 7, 9), (12, 3, 3, 3), dict(group=3, strides=[1, 2], dilations=[2, 1],
                                        pads=[2, 0, 1, 1], output_padding=[0, 1])),
    ((2, 16, 6, 6), (16, 1, 4, 4), dict(group=16, strides=[2, 2], pads=[1, 1, 1, 1],
                                        activation="Clip", activation_params=[-1.0, 1.0])),
    # 40 input channels: two shared-memory chunks; 20 output channels: two channel blocks
    ((2, 40, 10, 12), (40, 20, 2, 2), dict(strides=[2, 2], activation="HardSwish")),
    # several output tiles in h and w with ragged tails (32 * sW columns per tile)
    ((1, 3, 45, 70), (3, 2, 3, 3), dict(strides=[1, 1], pads=[1, 1, 1, 1])),
    ((1, 2, 20, 41), (2, 3, 5, 3), dict(strides=[3, 2], dilations=[1, 2],
                                        pads=[2, 1, 0, 3], output_padding=[1, 1])),
    ((2, 4, 3, 5, 6), (4, 2, 3, 2, 3), dict(strides=[2, 1, 2], pads=[1, 0, 1, 1, 0, 1],
                                            output_padding=[1, 0, 1], activation="Tanh")),
    ((1, 6, 4, 4, 4), (6, 2, 2, 2, 2), dict(group=3, strides=[2, 2, 2], activation="Sigmoid")),
]


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("idx", range(len(CASES)))
def test_transposed_parity(idx, dtype):
    xs, ws, attrs = CASES[idx]
    x, w, b, z = inputs(900 + 10 * idx, dtype, xs, ws, attrs)
    compare(dtype, x, w, b, z, attrs, what=f"convT {idx} {dtype}")


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_transposed_without_bias_and_z(dtype):
    xs, ws, attrs = (2, 5, 8, 9), (5, 7, 3, 3), dict(strides=[2, 2], pads=[0, 1, 1, 0])
    x, w, _, _ = inputs(990, dtype, xs, ws, attrs, bias=False, zres=False)
    compare(dtype, x, w, None, None, attrs, what="convT plain")


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_transposed_exact_integers(dtype):
    # small integers: every sum is exact in f32 (and fits f16), so Y must equal the oracle
    xs, ws = (2, 6, 7, 9), (6, 4, 3, 3)
    attrs = dict(group=2, strides=[2, 2], pads=[1, 0, 0, 1], output_padding=[1, 1])
    ys = oracle.transpose_output_shape(xs, ws, **attrs)
    x = workloads.draw_int(1000, xs, -3, 3, dtype)
    w = workloads.draw_int(1001, ws, -2, 2, dtype)
    b = workloads.draw_int(1002, (ys[1],), -4, 4, dtype)
    z = workloads.draw_int(1003, ys, -4, 4, dtype)
    dt = _lib.F16 if dtype == "f16" else _lib.F32
    plan = FusedConvPlan(dt, xs, ws, has_bias=True, has_z=True, transposed=True, **attrs)
    y = run_plan(plan, x, w, b, z, dtype)
    ref, _ = oracle.conv_transpose(x, w, b, z, **attrs)
    assert np.array_equal(y, ref)


def test_transposed_decoder_size():
    # an upsampling stage at benchmark size: X[8,256,32,32] W[256,128,4,4] s2 p1; every
    # output is compared on a sample of (image, channel) planes the oracle computes
    xs, ws = (8, 256, 32, 32), (256, 128, 4, 4)
    attrs = dict(strides=[2, 2], pads=[1, 1, 1, 1], activation="Relu")
    x, w, b, z = inputs(1100, "f16", xs, ws, attrs)
    plan = FusedConvPlan(_lib.F16, xs, ws, has_bias=True, has_z=True, transposed=True, **attrs)
    y = run_plan(plan, x, w, b, z, "f16")
    for n in (0, 7):
        sub_w = w[:, [0, 77, 127]]
        sub_b = b[[0, 77, 127]]
        sub_z = z[n:n + 1, [0, 77, 127]]
        ref, absacc = oracle.conv_transpose(x[n:n + 1], sub_w, sub_b, sub_z, **attrs)
        check(y[n:n + 1, [0, 77, 127]], ref, absacc, "f16", 256 * 16, activation="Relu",
              what=f"decoder image {n}")
