"""GPU parity of the fp32 tensor-core path (3xTF32 split on tcgen05, C/group a multiple of 32)
against the oracle, within the fp32 tolerance |y - ref| <= 1e-5 * sum|x*w| + 1e-6.

Cases span 1-3 spatial dims, groups, stride, dilation, pads, several pixel tiles with ragged
tails, more than one 128-channel tile, forced split-K (the reduce adds the splits in order),
both pixel-tile instantiations and capped grids (many work units per persistent CTA).
Integer-valued inputs are exact in TF32 (their lo halves are zero), so that case must match
the oracle bit for bit.
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


def run(plan, x, w, b, z):
    ny = int(np.prod(plan.y_shape))
    buf = torch.full((ny + 2 * GUARD,), float("nan"), dtype=torch.float32, device="cuda")
    buf[:GUARD] = 7.0
    buf[-GUARD:] = 7.0
    y = buf[GUARD:GUARD + ny].view(plan.y_shape)
    ws = None
    if plan.workspace_bytes:
        ws = torch.full((plan.workspace_bytes // 4,), float("nan"), dtype=torch.float32,
                        device="cuda")
    plan.run(to_dev(x), to_dev(w), to_dev(b), to_dev(z), y=y, workspace=ws)
    torch.cuda.synchronize()
    assert np.all(buf[:GUARD].cpu().numpy() == 7.0) and np.all(buf[-GUARD:].cpu().numpy() == 7.0)
    return y.double().cpu().numpy()


def inputs(seed, xs, ws, attrs):
    ys = oracle.output_shape(xs, ws, **attrs)
    kg = int(np.prod(ws[1:]))
    x = workloads.draw(seed, xs, "normal", 1.0, "f32")
    w = workloads.draw(seed + 1, ws, "normal", 1.0 / math.sqrt(kg), "f32")
    b = workloads.draw(seed + 2, (ws[0],), "normal", 1.0, "f32")
    z = workloads.draw(seed + 3, ys, "normal", 1.0, "f32")
    return x, w, b, z


CASES = [
    # (x_shape, w_shape, attrs, options)
    ((2, 32, 11, 13), (40, 32, 3, 3), dict(pads=[1, 1, 1, 1], activation="Relu"), {}),
    ((3, 64, 9, 7), (130, 64, 3, 3), dict(pads=[1, 0, 1, 2], activation="Gelu"), {}),
    ((2, 64, 12, 12), (48, 32, 3, 3), dict(group=2, strides=[2, 2], pads=[1, 1, 1, 1]),
     dict(tile_n=64)),
    ((2, 32, 40), (24, 32, 5), dict(dilations=[2], auto_pad="SAME_UPPER",
                                    activation="LeakyRelu", activation_params=[0.1]), {}),
    ((1, 32, 5, 9, 8), (16, 32, 3, 3, 3), dict(strides=[1, 2, 1], pads=[1, 1, 1, 1, 1, 1],
                                               activation="Tanh"), {}),
    ((4, 96, 6, 6), (64, 96, 1, 1), dict(activation="Sigmoid"), dict(split_k=3)),
    ((2, 64, 10, 10), (64, 64, 3, 3), dict(pads=[1, 1, 1, 1]), dict(split_k=2)),
    ((5, 32, 8, 8), (32, 32, 3, 3), dict(pads=[1, 1, 1, 1], activation="HardSwish"),
     dict(max_ctas=3)),
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_tf32_parity(idx):
    xs, ws, attrs, opts = CASES[idx]
    x, w, b, z = inputs(1300 + 10 * idx, xs, ws, attrs)
    plan = FusedConvPlan(_lib.F32, xs, ws, has_bias=True, has_z=True, **opts, **attrs)
    assert plan.route == "igemm_tc" and plan.launches == 3
    y = run(plan, x, w, b, z)
    ref, absacc = oracle.fused_conv(x, w, b, z, **attrs)
    check(y, ref, absacc, "f32", int(np.prod(ws[1:])), activation=attrs.get("activation"),
          what=f"tf32 {idx} split={plan.split_k} tile={plan.tile_n}")


def test_tf32_without_bias_and_z():
    xs, ws, attrs = (2, 32, 9, 9), (33, 32, 3, 3), dict(pads=[1, 1, 1, 1])
    x, w, _, _ = inputs(1400, xs, ws, attrs)
    plan = FusedConvPlan(_lib.F32, xs, ws, **attrs)
    y = run(plan, x, w, None, None)
    ref, absacc = oracle.fused_conv(x, w, **attrs)
    check(y, ref, absacc, "f32", int(np.prod(ws[1:])), what="tf32 plain")


def test_tf32_exact_integers():
    xs, ws = (2, 64, 7, 9), (72, 64, 3, 3)
    attrs = dict(pads=[1, 1, 1, 1])
    ys = oracle.output_shape(xs, ws, **attrs)
    x = workloads.draw_int(1500, xs, -3, 3, "f32")
    w = workloads.draw_int(1501, ws, -2, 2, "f32")
    b = workloads.draw_int(1502, (ws[0],), -4, 4, "f32")
    z = workloads.draw_int(1503, ys, -4, 4, "f32")
    plan = FusedConvPlan(_lib.F32, xs, ws, has_bias=True, has_z=True, split_k=2, **attrs)
    y = run(plan, x, w, b, z)
    ref, _ = oracle.fused_conv(x, w, b, z, **attrs)
    assert np.array_equal(y, ref)


def test_tf32_full_size_sample():
    # a ResNet-stage fp32 conv: X[32,64,56,56] W[64,64,3,3]; planes of two images checked
    xs, ws = (32, 64, 56, 56), (64, 64, 3, 3)
    attrs = dict(pads=[1, 1, 1, 1], activation="Relu")
    x, w, b, z = inputs(1600, xs, ws, attrs)
    plan = FusedConvPlan(_lib.F32, xs, ws, has_bias=True, has_z=True, **attrs)
    y = run(plan, x, w, b, z)
    for n in (0, 31):
        ref, absacc = oracle.fused_conv(x[n:n + 1], w, b, z[n:n + 1], **attrs)
        check(y[n:n + 1], ref, absacc, "f32", 576, activation="Relu", what=f"tf32 image {n}")
