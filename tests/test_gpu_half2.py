"""The opt-in half2 row-partial mode of the depthwise kernel (f16 only): each kernel row's
taps are summed for two adjacent outputs with packed f16 FMAs, and the rows are added in
f32. Its error bound is the default f16 tolerance plus K * 2^-11 * sum|x*w| (K FMAs, each
rounded to f16 with unit roundoff 2^-11, per kernel row, none larger than the row's
sum|x*w|). Integer-valued inputs keep every partial exact, so they must match bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from activation_implicit_gemm_gb300 import FusedConvPlan, _build, _lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _build.build()
    _lib.load()
    yield
    assert _lib.load().fconv_check_device(None) == 0


def run(plan, x, w, b, z):
    d = [None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
         for a in (x, w, b, z)]
    y = torch.full(plan.y_shape, float("nan"), dtype=torch.float16, device="cuda")
    plan.run(*d, y=y)
    torch.cuda.synchronize()
    return y.double().cpu().numpy()


CASES = [
    ((2, 16, 24, 32), 3, dict(pads=[1, 1, 1, 1])),
    ((2, 8, 30, 40), 5, dict(pads=[2, 1, 2, 3])),
    ((2, 8, 56, 56), 7, dict(pads=[3, 3, 3, 3])),
    ((1, 4, 70, 72), 7, dict(pads=[3, 0, 3, 2])),
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_half2_rows_within_its_bound(idx):
    xs, k, attrs = CASES[idx]
    C = xs[1]
    attrs = dict(attrs, group=C, activation="Clip", activation_params=[-4.0, 4.0])
    ys = oracle.output_shape(xs, (C, 1, k, k), **attrs)
    x = workloads.draw(1700 + idx, xs, "normal", 1.0, "f16")
    w = workloads.draw(1701 + idx, (C, 1, k, k), "normal", 1.0 / k, "f16")
    b = workloads.draw(1702 + idx, (C,), "normal", 1.0, "f16")
    z = workloads.draw(1703 + idx, ys, "normal", 1.0, "f16")
    plan = FusedConvPlan(_lib.F16, xs, (C, 1, k, k), has_bias=True, has_z=True,
                         precision="half2_rows", **attrs)
    assert plan.route == "depthwise"
    y = run(plan, x, w, b, z)
    ref, absacc = oracle.fused_conv(x, w, b, z, **attrs)
    kg = k * k
    tol = 2e-3 * np.abs(ref) + 1e-3 * absacc / math.sqrt(kg) + k * 2.0 ** -11 * absacc
    err = np.abs(y - ref)
    assert np.all(err <= tol), f"max err {err.max():.3e}"
    # and it is the half2 path: its error differs from the f32-accumulation kernel's
    y32 = run(FusedConvPlan(_lib.F16, xs, (C, 1, k, k), has_bias=True, has_z=True, **attrs),
              x, w, b, z)
    assert np.abs(y32 - ref).max() <= np.abs(y - ref).max()


def test_half2_rows_exact_on_integers():
    xs, k = (2, 8, 20, 24), 7
    attrs = dict(group=8, pads=[3, 3, 3, 3])
    ys = oracle.output_shape(xs, (8, 1, k, k), **attrs)
    x = workloads.draw_int(1800, xs, -3, 3, "f16")
    w = workloads.draw_int(1801, (8, 1, k, k), -2, 2, "f16")
    b = workloads.draw_int(1802, (8,), -4, 4, "f16")
    z = workloads.draw_int(1803, ys, -4, 4, "f16")
    plan = FusedConvPlan(_lib.F16, xs, (8, 1, k, k), has_bias=True, has_z=True,
                         precision="half2_rows", **attrs)
    y = run(plan, x, w, b, z)
    ref, _ = oracle.fused_conv(x, w, b, z, **attrs)
    assert np.array_equal(y, ref)
