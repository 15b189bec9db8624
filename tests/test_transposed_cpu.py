"""Host side of the transposed FusedConv (no GPU): the planner's shapes, statuses, route and
work counts agree with the oracle's resolution of the same requests."""
import itertools
import random

import numpy as np
import pytest

import oracle
from activation_implicit_gemm_gb300 import FconvError, FusedConvPlan, _build, _lib

ORACLE_TO_LIB = {"OK": "OK", "ATTR_VALUE": "E_ATTR_VALUE", "GROUP": "E_GROUP",
                 "EMPTY_OUTPUT": "E_OUTPUT_EMPTY", "ATTR_LENGTH": "E_ATTR_LENGTH"}


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return _lib.load()


def plan_status(xs, ws, **attrs):
    try:
        p = FusedConvPlan(_lib.F16, xs, ws, transposed=True, **attrs)
        return "OK", p
    except FconvError as e:
        return e.code, None


def test_shapes_and_statuses_agree_with_the_oracle():
    rng = random.Random(5)
    seen = set()
    for _ in range(300):
        sr = rng.choice([1, 2, 3])
        g = rng.choice([1, 2, 3])
        C = g * rng.randint(1, 3)
        Mg = rng.randint(1, 4)
        if rng.random() < 0.1:
            C += 1  # a group that does not divide C
        xs = (rng.randint(1, 2), C) + tuple(rng.randint(1, 6) for _ in range(sr))
        ws = (C if rng.random() > 0.05 else C + 1, Mg) + tuple(rng.randint(1, 4) for _ in range(sr))
        st = [rng.randint(1, 3) for _ in range(sr)]
        dl = [rng.randint(1, 2) for _ in range(sr)]
        pads = [rng.randint(0, 3) for _ in range(2 * sr)]
        op = [rng.randint(0, 3) for _ in range(sr)]
        attrs = dict(group=g, strides=st, dilations=dl, pads=pads, output_padding=op)
        ost, oys = oracle.transpose_resolve(xs, ws, **attrs)
        lst, p = plan_status(xs, ws, **attrs)
        assert lst == ORACLE_TO_LIB[ost], (xs, ws, attrs, ost, lst)
        if p is not None:
            assert p.y_shape == oys
            assert p.route == "transposed"
            assert p.workspace_bytes == 0 and p.launches == 1
        seen.add(ost)
    assert {"OK", "ATTR_VALUE", "GROUP", "EMPTY_OUTPUT"} <= seen


def test_flops_count_the_taps_that_land():
    xs, ws = (2, 8, 5, 5), (8, 3, 4, 4)
    attrs = dict(group=2, strides=[2, 2], pads=[1, 1, 1, 1], output_padding=[1, 1])
    p = FusedConvPlan(_lib.F16, xs, ws, transposed=True, **attrs)
    # count, by brute force, the (input, tap) pairs of one axis that reach an output
    out = p.y_shape[2]
    per_axis = sum(1 for i, k in itertools.product(range(5), range(4)) if 0 <= 2 * i - 1 + k < out)
    assert p.flops == 2.0 * 2 * 8 * 3 * per_axis ** 2


def test_rules_specific_to_the_transposed_form():
    # SAME auto_pad is not defined for the transposed form on the pages
    with pytest.raises(FconvError) as e:
        FusedConvPlan(_lib.F16, (1, 4, 5, 5), (4, 2, 3, 3), transposed=True,
                      auto_pad="SAME_UPPER")
    assert e.value.code == "E_UNSUPPORTED"
    # VALID: no pads
    p = FusedConvPlan(_lib.F16, (1, 4, 5, 5), (4, 2, 3, 3), transposed=True, auto_pad="VALID",
                      strides=[2, 2])
    assert p.y_shape == (1, 2, 11, 11)
    # output_padding on a direct convolution
    with pytest.raises(FconvError) as e:
        FusedConvPlan(_lib.F16, (1, 4, 5, 5), (2, 4, 3, 3), output_padding=[1, 0])
    assert e.value.code == "E_ATTR_VALUE"
    # forcing another route on the transposed form, or the transposed route on a direct conv
    with pytest.raises(FconvError) as e:
        FusedConvPlan(_lib.F16, (1, 4, 5, 5), (4, 2, 3, 3), transposed=True, route="direct")
    assert e.value.code == "E_UNSUPPORTED"
    with pytest.raises(FconvError) as e:
        FusedConvPlan(_lib.F16, (1, 4, 5, 5), (2, 4, 3, 3), route="transposed")
    assert e.value.code == "E_UNSUPPORTED"
    # bias length is M = W.dim1 * group
    p = FusedConvPlan(_lib.F32, (1, 4, 5, 5), (4, 3, 3, 3), group=2, transposed=True,
                      has_bias=True)
    assert p.y_shape[1] == 6
