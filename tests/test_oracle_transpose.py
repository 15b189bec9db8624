"""Pins of the oracle's transposed convolution (ExecuTorch WebGPU PR #20849: the transposed
form of aten.convolution.default, gather-form kernel, weight [IC, OC/groups, k...],
output_padding below the stride), each checked against something other than the oracle's
own formula:

* closed forms on tiny inputs worked by hand;
* the adjoint identity <convT(x), dy> = <x, conv(dy)>: the transposed convolution is the
  adjoint of the direct convolution with the same weight tensor read as (C, M/group, k...),
  the same stride, dilation and group, and pads (pad_begin, pad_end - output_padding); the
  direct convolution is the oracle's pinned `fused_conv`;
* PyTorch's float64 conv_transpose1d/2d/3d (a library routine), with asymmetric pads taken
  as a crop of the unpadded result;
* the output-size formula, the validation rules and the fused epilogue.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def rnd(seed, shape):
    return np.random.default_rng(seed).standard_normal(shape)


def test_tiny_closed_forms():
    x = np.array([[[2.0, 3.0]]])
    w = np.array([[[5.0, 7.0]]])
    # stride 2: no overlap, each input writes its own pair
    y, s = oracle.conv_transpose(x, w, strides=[2])
    assert y.tolist() == [[[10.0, 14.0, 15.0, 21.0]]]
    # stride 1: the middle output gets both inputs
    y, s = oracle.conv_transpose(x, w)
    assert y.tolist() == [[[10.0, 29.0, 21.0]]]
    assert s.tolist() == [[[10.0, 29.0, 21.0]]]
    # dilation 2, pad 1 each side, output_padding 0: full = [10, 15, 14, 21] -> crop 1 and 1
    y, _ = oracle.conv_transpose(x, w, dilations=[2], pads=[1, 1])
    assert y.tolist() == [[[15.0, 14.0]]]
    # stride 2, output_padding 1: one more position that nothing reaches
    y, _ = oracle.conv_transpose(x, w, strides=[2], output_padding=[1])
    assert y.tolist() == [[[10.0, 14.0, 15.0, 21.0, 0.0]]]
    # 2 input channels, group 2, one output channel each: channels do not mix
    x2 = np.array([[[1.0, 0.0], [0.0, 1.0]]])
    w2 = np.array([[[1.0, 2.0]], [[3.0, 4.0]]])
    y, _ = oracle.conv_transpose(x2, w2, group=2)
    assert y.tolist() == [[[1.0, 2.0, 0.0], [0.0, 3.0, 4.0]]]
    # same with group 1: both inputs reach both output channels
    w3 = np.array([[[1.0, 2.0], [5.0, 6.0]], [[3.0, 4.0], [7.0, 8.0]]])  # (C=2, M=2, k=2)
    y, _ = oracle.conv_transpose(x2, w3)
    assert y.tolist() == [[[1.0, 2.0 + 3.0, 4.0], [5.0, 6.0 + 7.0, 8.0]]]


ADJ_CASES = [
    # (x_shape, w_shape, attrs)
    ((2, 3, 7), (3, 4, 3), dict(strides=[2], pads=[1, 2], output_padding=[1])),
    ((1, 4, 5, 6), (4, 3, 3, 2), dict(group=2, strides=[2, 3], dilations=[1, 2],
                                      pads=[1, 0, 2, 1], output_padding=[1, 0])),
    ((2, 2, 4, 3, 5), (2, 2, 2, 3, 2), dict(strides=[1, 2, 2], dilations=[2, 1, 1],
                                            pads=[0, 1, 1, 1, 1, 2], output_padding=[0, 1, 1])),
    ((1, 6, 6, 6), (6, 1, 3, 3), dict(group=6, strides=[2, 2], pads=[1, 1, 1, 1],
                                      output_padding=[1, 1])),
]


@pytest.mark.parametrize("idx", range(len(ADJ_CASES)))
def test_adjoint_of_the_direct_convolution(idx):
    xs, ws, attrs = ADJ_CASES[idx]
    x = rnd(10 + idx, xs)
    w = rnd(20 + idx, ws)
    y, _ = oracle.conv_transpose(x, w, **attrs)
    dy = rnd(30 + idx, y.shape)
    sr = len(xs) - 2
    pads = attrs.get("pads", [0] * (2 * sr))
    op = attrs.get("output_padding", [0] * sr)
    conv_pads = list(pads[:sr]) + [pads[sr + i] - op[i] for i in range(sr)]
    assert min(conv_pads) >= 0
    back, _ = oracle.fused_conv(dy, w, group=attrs.get("group", 1),
                                strides=attrs.get("strides"), dilations=attrs.get("dilations"),
                                pads=conv_pads)
    assert back.shape == x.shape
    lhs = float(np.sum(y * dy))
    rhs = float(np.sum(x * back))
    assert math.isclose(lhs, rhs, rel_tol=1e-12, abs_tol=1e-12), (lhs, rhs)


TORCH_CASES = [
    ((2, 3, 9), (3, 5, 4), dict(strides=[3], dilations=[1], pads=[2, 0], output_padding=[2])),
    ((2, 4, 5, 7), (4, 2, 3, 3), dict(group=2, strides=[2, 2], dilations=[2, 1],
                                      pads=[1, 2, 0, 1], output_padding=[1, 1])),
    ((1, 2, 3, 4, 5), (2, 3, 2, 2, 3), dict(strides=[2, 1, 2], pads=[0, 0, 1, 1, 0, 0],
                                            output_padding=[1, 0, 0])),
    ((3, 8, 6, 6), (8, 1, 4, 4), dict(group=8, strides=[2, 2], pads=[1, 1, 1, 1])),
]


@pytest.mark.parametrize("idx", range(len(TORCH_CASES)))
def test_against_torch_float64(idx):
    xs, ws, attrs = TORCH_CASES[idx]
    x = rnd(40 + idx, xs)
    w = rnd(50 + idx, ws)
    b = rnd(60 + idx, (ws[1] * attrs.get("group", 1),))
    y, s = oracle.conv_transpose(x, w, b, **attrs)
    sr = len(xs) - 2
    fn = {1: torch.nn.functional.conv_transpose1d, 2: torch.nn.functional.conv_transpose2d,
          3: torch.nn.functional.conv_transpose3d}[sr]
    full = fn(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b),
              stride=attrs.get("strides", [1] * sr), padding=0,
              output_padding=attrs.get("output_padding", [0] * sr),
              groups=attrs.get("group", 1), dilation=attrs.get("dilations", [1] * sr)).numpy()
    pads = attrs.get("pads", [0] * (2 * sr))
    crop = (slice(None), slice(None)) + tuple(
        slice(pads[i], full.shape[2 + i] - pads[sr + i]) for i in range(sr))
    ref = full[crop]
    assert ref.shape == y.shape
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.all(s >= 0)


def test_output_size_formula():
    # out = (in - 1) * s - pad_begin - pad_end + d * (k - 1) + output_padding + 1
    for (i, k, s, d, pb, pe, op) in [(7, 3, 2, 1, 1, 1, 1), (5, 4, 3, 2, 0, 2, 2),
                                     (1, 1, 1, 1, 0, 0, 0), (10, 5, 1, 3, 4, 4, 0)]:
        ys = oracle.transpose_output_shape((1, 1, i), (1, 1, k), strides=[s], dilations=[d],
                                           pads=[pb, pe], output_padding=[op])
        assert ys == (1, 1, (i - 1) * s - pb - pe + d * (k - 1) + op + 1)


def test_validation():
    ok = dict(strides=[2, 2], output_padding=[1, 1])
    assert oracle.transpose_resolve((1, 4, 3, 3), (4, 2, 3, 3), **ok)[0] == "OK"
    # output_padding must stay below the stride (ExecuTorch rejects output_padding >= stride)
    assert oracle.transpose_resolve((1, 4, 3, 3), (4, 2, 3, 3), strides=[2, 2],
                                    output_padding=[2, 0])[0] == "ATTR_VALUE"
    assert oracle.transpose_resolve((1, 4, 3, 3), (4, 2, 3, 3),
                                    output_padding=[1, 0])[0] == "ATTR_VALUE"
    # W.dim0 must be C; the group must divide C
    assert oracle.transpose_resolve((1, 4, 3, 3), (3, 2, 3, 3))[0] == "GROUP"
    assert oracle.transpose_resolve((1, 4, 3, 3), (4, 2, 3, 3), group=3)[0] == "GROUP"
    # pads that eat the whole output
    assert oracle.transpose_resolve((1, 1, 2), (1, 1, 2), pads=[2, 1])[0] == "EMPTY_OUTPUT"
    assert oracle.transpose_resolve((1, 1, 2), (1, 1, 2), pads=[1, 1])[0] == "OK"
    # attribute lengths follow the spatial rank
    assert oracle.transpose_resolve((1, 1, 4, 4), (1, 1, 2, 2),
                                    output_padding=[0])[0] == "ATTR_LENGTH"


def test_fused_epilogue():
    xs, ws = (2, 4, 5, 5), (4, 3, 3, 3)
    attrs = dict(group=1, strides=[2, 2], pads=[1, 1, 1, 1], output_padding=[1, 1])
    x, w = rnd(70, xs), rnd(71, ws)
    y0, s0 = oracle.conv_transpose(x, w, **attrs)
    b = rnd(72, (y0.shape[1],))
    z = rnd(73, y0.shape)
    y, s = oracle.conv_transpose(x, w, b, z, activation="Clip", activation_params=[-0.5, 1.0],
                                 **attrs)
    ref = np.clip(y0 + b[None, :, None, None] + z, -0.5, 1.0)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(s, s0)
    y, _ = oracle.conv_transpose(x, w, b, z, activation="LeakyRelu", activation_params=[0.1],
                                 **attrs)
    v = y0 + b[None, :, None, None] + z
    np.testing.assert_allclose(y, np.where(v < 0, 0.1 * v, v), rtol=0, atol=1e-12)
