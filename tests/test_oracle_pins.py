"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against a library routine (PyTorch CPU float64
convolutions and activations), a brute-force scatter formulation, a closed form or a
value printed on the pages, chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def torch_reference(x, w, b, z, group, strides, dilations, pad_begin, pad_end):
    """PyTorch CPU float64 conv with explicit (possibly asymmetric) zero padding."""
    sr = x.ndim - 2
    xt = torch.from_numpy(np.asarray(x, dtype=np.float64))
    wt = torch.from_numpy(np.asarray(w, dtype=np.float64))
    # F.pad takes (last axis begin, last axis end, previous axis begin, ...)
    padspec = []
    for ax in reversed(range(sr)):
        padspec += [int(pad_begin[ax]), int(pad_end[ax])]
    xt = F.pad(xt, padspec)
    conv = {1: F.conv1d, 2: F.conv2d, 3: F.conv3d}[sr]
    y = conv(xt, wt, None if b is None else torch.from_numpy(np.asarray(b, np.float64)),
             stride=tuple(strides), dilation=tuple(dilations), groups=group)
    y = y.numpy()
    if z is not None:
        y = y + z
    return y


def random_case(rng, sr):
    """Random small conv geometry of spatial rank sr with groups, strides, dilations, pads."""
    G = int(rng.choice([1, 1, 2, 3]))
    Cg = int(rng.integers(1, 4))
    Mg = int(rng.integers(1, 4))
    N = int(rng.integers(1, 3))
    ins = [int(rng.integers(3, 9)) for _ in range(sr)]
    ks = [int(rng.integers(1, 4)) for _ in range(sr)]
    ss = [int(rng.integers(1, 3)) for _ in range(sr)]
    ds = [int(rng.integers(1, 3)) for _ in range(sr)]
    mode = rng.choice(["NOTSET", "NOTSET", "SAME_UPPER", "SAME_LOWER", "VALID"])
    pads = None
    if mode == "NOTSET":
        pads = [int(rng.integers(0, 3)) for _ in range(2 * sr)]
    for j in range(sr):  # keep every output extent >= 1
        ext = (ks[j] - 1) * ds[j] + 1
        lo = 0 if pads is None else pads[j] + pads[sr + j]
        if ins[j] + (lo if mode == "NOTSET" else 0) < ext:
            ins[j] = ext
    x_shape = (N, G * Cg) + tuple(ins)
    w_shape = (G * Mg, Cg) + tuple(ks)
    return dict(x_shape=x_shape, w_shape=w_shape, group=G, strides=ss, dilations=ds,
                pads=pads, auto_pad=str(mode))


# ----------------------------------------------------------------------------- shapes

def test_config_shapes_golden():
    """Output sizes and pads of every benchmark conv equal the hand-worked values."""
    gold = json.load(open(os.path.join(GOLDEN, "config_shapes.json")))["cases"]
    for c in workloads.ALL_CASES:
        st, ys, pb, pe = oracle.resolve(c.x_shape, c.w_shape, **c.attrs())
        assert st == "OK", c.name
        g = gold[c.name]
        assert list(ys) == g["y"], c.name
        assert list(pb) == g["pad_begin"], c.name
        assert list(pe) == g["pad_end"], c.name


def test_same_output_is_ceil_in_over_stride():
    for inn, s, k, d, mode in itertools.product(range(1, 14), range(1, 5), range(1, 6),
                                               range(1, 4), ["SAME_UPPER", "SAME_LOWER"]):
        st, ys, pb, pe = oracle.resolve((1, 1, inn), (1, 1, k), strides=[s], dilations=[d],
                                        auto_pad=mode)
        assert st == "OK"
        assert ys[2] == -(-inn // s)
        total = max(0, (ys[2] - 1) * s + (k - 1) * d + 1 - inn)
        assert pb[2] + pe[2] == total
        if mode == "SAME_UPPER":
            assert pe[2] >= pb[2] and pe[2] - pb[2] <= 1
        else:
            assert pb[2] >= pe[2] and pb[2] - pe[2] <= 1
        # the applied pads reproduce the same size through the NOTSET formula
        st2, ys2, _, _ = oracle.resolve((1, 1, inn), (1, 1, k), strides=[s], dilations=[d],
                                        pads=[pb[2], pe[2]])
        assert ys2 == ys


def test_notset_and_valid_sizes_match_torch():
    rng = _rng(1)
    for sr in (1, 2, 3):
        for _ in range(20):
            c = random_case(rng, sr)
            st, ys, pb, pe = oracle.resolve(c["x_shape"], c["w_shape"], group=c["group"],
                                            strides=c["strides"], dilations=c["dilations"],
                                            pads=c["pads"], auto_pad=c["auto_pad"])
            assert st == "OK"
            if c["auto_pad"] in ("NOTSET", "VALID"):
                x = np.zeros(c["x_shape"])
                w = np.zeros(c["w_shape"])
                y = torch_reference(x, w, None, None, c["group"], c["strides"], c["dilations"],
                                    pb[3 - sr:], pe[3 - sr:])
                assert tuple(y.shape) == tuple(ys)


# ----------------------------------------------------------------------------- conv sums

@pytest.mark.parametrize("sr", [1, 2, 3])
def test_conv_matches_torch_float64(sr):
    """Random geometry (groups, strides, dilations, asymmetric pads, auto_pad, B, Z)."""
    rng = _rng(100 + sr)
    for it in range(12):
        c = random_case(rng, sr)
        ys = oracle.output_shape(c["x_shape"], c["w_shape"], group=c["group"],
                                 strides=c["strides"], dilations=c["dilations"], pads=c["pads"],
                                 auto_pad=c["auto_pad"])
        _, _, pb, pe = oracle.resolve(c["x_shape"], c["w_shape"], group=c["group"],
                                      strides=c["strides"], dilations=c["dilations"],
                                      pads=c["pads"], auto_pad=c["auto_pad"])
        x = rng.standard_normal(c["x_shape"])
        w = rng.standard_normal(c["w_shape"])
        b = rng.standard_normal(c["w_shape"][0]) if it % 2 == 0 else None
        z = rng.standard_normal(ys) if it % 3 != 2 else None
        y, s = oracle.fused_conv(x, w, b, z, group=c["group"], strides=c["strides"],
                                 dilations=c["dilations"], pads=c["pads"],
                                 auto_pad=c["auto_pad"])
        ref = torch_reference(x, w, b, z, c["group"], c["strides"], c["dilations"],
                              pb[3 - sr:], pe[3 - sr:])
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
        # sum |x*w| over the taps is the convolution of |x| with |w|
        sref = torch_reference(np.abs(x), np.abs(w), None, None, c["group"], c["strides"],
                               c["dilations"], pb[3 - sr:], pe[3 - sr:])
        np.testing.assert_allclose(s, sref, rtol=1e-12, atol=1e-12)


def _scatter_conv(x, w, group, strides, dilations, pad_begin, out_shape):
    """Brute force by scattering: every (input element, tap) pair adds into the output
    position that reads it, if that position exists. Independent of the oracle's
    gather loop order and index formula."""
    N, C = x.shape[:2]
    M, Cg = w.shape[:2]
    sr = x.ndim - 2
    Mg = M // group
    y = np.zeros(out_shape)
    for n, c in itertools.product(range(N), range(C)):
        g, ci = divmod(c, Cg)
        for ipos in itertools.product(*[range(e) for e in x.shape[2:]]):
            for tap in itertools.product(*[range(e) for e in w.shape[2:]]):
                opos = []
                for j in range(sr):
                    num = ipos[j] + pad_begin[j] - tap[j] * dilations[j]
                    if num % strides[j] != 0:
                        break
                    o = num // strides[j]
                    if o < 0 or o >= out_shape[2 + j]:
                        break
                    opos.append(o)
                else:
                    for m in range(g * Mg, (g + 1) * Mg):
                        y[(n, m) + tuple(opos)] += x[(n, c) + ipos] * w[(m, ci) + tap]
    return y


def test_brute_force_scatter_tiny():
    rng = _rng(7)
    for sr in (1, 2, 3):
        for _ in range(4):
            c = random_case(rng, sr)
            st, ys, pb, pe = oracle.resolve(c["x_shape"], c["w_shape"], group=c["group"],
                                            strides=c["strides"], dilations=c["dilations"],
                                            pads=c["pads"], auto_pad=c["auto_pad"])
            x = rng.standard_normal(c["x_shape"])
            w = rng.standard_normal(c["w_shape"])
            y, _ = oracle.fused_conv(x, w, group=c["group"], strides=c["strides"],
                                     dilations=c["dilations"], pads=c["pads"],
                                     auto_pad=c["auto_pad"])
            ref = _scatter_conv(x, w, c["group"], c["strides"], c["dilations"], pb[3 - sr:], ys)
            np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_1x1_is_matmul_readme_shape():
    """The README usage example, x[1,32,8,8] with w[32,32,1,1]: Y[0] = W x X[0]."""
    rng = _rng(3)
    x = rng.standard_normal((1, 32, 8, 8))
    w = rng.standard_normal((32, 32, 1, 1))
    y, _ = oracle.fused_conv(x, w)
    ref = (w[:, :, 0, 0] @ x[0].reshape(32, 64)).reshape(1, 32, 8, 8)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_delta_kernel_is_identity():
    rng = _rng(4)
    for k in (1, 3, 5):
        C = 6
        x = rng.standard_normal((2, C, 7, 9))
        w = np.zeros((C, 1, k, k))
        w[:, 0, k // 2, k // 2] = 1.0
        y, _ = oracle.fused_conv(x, w, group=C, pads=[k // 2] * 4)
        np.testing.assert_array_equal(y, x)


def test_rank_embedding():
    """1-D == 2-D with H = kh = 1 == 3-D with D = kd = 1."""
    rng = _rng(5)
    x = rng.standard_normal((2, 4, 11))
    w = rng.standard_normal((6, 2, 3))
    kw = dict(group=2, strides=[2], dilations=[2], pads=[1, 2])
    y1, _ = oracle.fused_conv(x, w, **kw)
    y2, _ = oracle.fused_conv(x[:, :, None, :], w[:, :, None, :], group=2, strides=[1, 2],
                              dilations=[1, 2], pads=[0, 1, 0, 2])
    y3, _ = oracle.fused_conv(x[:, :, None, None, :], w[:, :, None, None, :], group=2,
                              strides=[1, 1, 2], dilations=[1, 1, 2], pads=[0, 0, 1, 0, 0, 2])
    np.testing.assert_array_equal(y1, y2[:, :, 0, :])
    np.testing.assert_array_equal(y1, y3[:, :, 0, 0, :])


def test_group_is_concatenation_of_dense_convs():
    rng = _rng(6)
    G, Cg, Mg = 3, 2, 4
    x = rng.standard_normal((2, G * Cg, 6, 5))
    w = rng.standard_normal((G * Mg, Cg, 3, 2))
    y, _ = oracle.fused_conv(x, w, group=G, pads=[1, 0, 1, 1])
    parts = [oracle.fused_conv(x[:, g * Cg:(g + 1) * Cg], w[g * Mg:(g + 1) * Mg],
                               pads=[1, 0, 1, 1])[0] for g in range(G)]
    np.testing.assert_array_equal(y, np.concatenate(parts, axis=1))


def test_dilation_equals_zero_inserted_kernel():
    rng = _rng(8)
    x = rng.standard_normal((1, 3, 12, 12))
    w = rng.standard_normal((2, 3, 3, 3))
    y, _ = oracle.fused_conv(x, w, dilations=[2, 3], pads=[2, 3, 2, 3])
    wz = np.zeros((2, 3, 5, 7))
    wz[:, :, ::2, ::3] = w
    y2, _ = oracle.fused_conv(x, wz, pads=[2, 3, 2, 3])
    np.testing.assert_allclose(y, y2, rtol=1e-13, atol=1e-13)


def test_stride_equals_subsampled_stride_one():
    rng = _rng(9)
    x = rng.standard_normal((1, 2, 9, 10))
    w = rng.standard_normal((3, 2, 3, 3))
    y, _ = oracle.fused_conv(x, w, strides=[2, 3], pads=[1, 1, 1, 1])
    y1, _ = oracle.fused_conv(x, w, pads=[1, 1, 1, 1])
    np.testing.assert_array_equal(y, y1[:, :, ::2, ::3][:, :, :y.shape[2], :y.shape[3]])


def test_bias_and_residual_enter_before_activation():
    """With W = 0 the output is act(B + Z); Relu of a negative B + Z is 0."""
    rng = _rng(10)
    x = rng.standard_normal((2, 3, 5, 5))
    w = np.zeros((4, 3, 3, 3))
    b = rng.standard_normal(4)
    ys = oracle.output_shape(x.shape, w.shape, pads=[1, 1, 1, 1])
    z = rng.standard_normal(ys)
    y, _ = oracle.fused_conv(x, w, b, z, pads=[1, 1, 1, 1], activation="Relu")
    np.testing.assert_array_equal(y, np.maximum(b[None, :, None, None] + z, 0.0))


def test_integer_inputs_are_exact():
    rng = _rng(11)
    x = rng.integers(-2, 3, (2, 4, 6, 6)).astype(np.float64)
    w = rng.integers(-2, 3, (5, 4, 3, 3)).astype(np.float64)
    y, _ = oracle.fused_conv(x, w, pads=[1, 1, 1, 1])
    ref = torch_reference(x, w, None, None, 1, [1, 1], [1, 1], [1, 1], [1, 1])
    np.testing.assert_array_equal(y, ref)


# ----------------------------------------------------------------------------- activations

def test_activation_golden_points():
    gold = json.load(open(os.path.join(GOLDEN, "activation_points.json")))
    for p in gold["points"]:
        got = oracle.activation(p["act"], p["v"], p.get("alpha", 0.0), p.get("beta", 0.0))
        assert got == pytest.approx(p["y"], rel=1e-15, abs=1e-15), p


def test_quickgelu_matches_pages_exp2_form():
    c = json.load(open(os.path.join(GOLDEN, "activation_points.json")))["quickgelu_exp2_constant"]
    assert c == pytest.approx(1.702 / math.log(2.0), rel=1e-15)
    for v in np.linspace(-8, 8, 161):
        ref = v / (1.0 + 2.0 ** (v * -c))
        assert oracle.activation("QuickGelu", v, 1.702) == pytest.approx(ref, rel=1e-13, abs=1e-15)


def test_activations_match_torch_library():
    v = torch.linspace(-9.0, 9.0, 721, dtype=torch.float64)
    refs = {
        ("Relu", 0.0, 0.0): F.relu(v),
        ("LeakyRelu", 0.01, 0.0): F.leaky_relu(v, 0.01),
        ("LeakyRelu", 0.3, 0.0): F.leaky_relu(v, 0.3),
        ("Sigmoid", 0.0, 0.0): torch.sigmoid(v),
        ("Tanh", 0.0, 0.0): torch.tanh(v),
        ("HardSigmoid", 1.0 / 6.0, 0.5): F.hardsigmoid(v),
        ("HardSwish", 0.0, 0.0): F.hardswish(v),
        ("Clip", -1.5, 2.0): torch.clamp(v, -1.5, 2.0),
        ("QuickGelu", 1.0, 0.0): F.silu(v),
        ("QuickGelu", 1.702, 0.0): v * torch.sigmoid(1.702 * v),
        ("Elu", 1.0, 0.0): F.elu(v, 1.0),
        ("Elu", 0.5, 0.0): F.elu(v, 0.5),
        ("Gelu", 0.0, 0.0): F.gelu(v, approximate="none"),
        ("Gelu", 1.0, 0.0): F.gelu(v, approximate="tanh"),
        ("FastGelu", 0.0, 0.0): F.gelu(v, approximate="tanh"),
        ("Softplus", 0.0, 0.0): F.softplus(v, beta=1.0, threshold=1e9),
        ("ThresholdedRelu", 1.0, 0.0): F.threshold(v, 1.0, 0.0),
        ("ThresholdedRelu", -0.5, 0.0): F.threshold(v, -0.5, 0.0),
        ("Erf", 0.0, 0.0): torch.erf(v),
    }
    for (name, a, b), ref in refs.items():
        got = np.array([oracle.activation(name, float(t), a, b) for t in v])
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-13, atol=1e-14, err_msg=name)


# ----------------------------------------------------------------------------- validation

@pytest.mark.parametrize("kw,status", [
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), strides=[1]), "ATTR_LENGTH"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), pads=[1, 1]), "ATTR_LENGTH"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), dilations=[1, 1, 1]), "ATTR_LENGTH"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), kernel_shape=[3]), "ATTR_LENGTH"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), strides=[0, 1]), "ATTR_VALUE"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), dilations=[1, 0]), "ATTR_VALUE"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), pads=[1, -1, 1, 1]), "ATTR_VALUE"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), pads=[1, 1, 1, 1],
          auto_pad="SAME_UPPER"), "PADS_AUTOPAD"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), kernel_shape=[3, 2]), "KERNEL_SHAPE"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 2, 3, 3), group=1), "GROUP"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(3, 2, 3, 3), group=2), "GROUP"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), group=0), "GROUP"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), activation="LeakyRelu"), "ACT_PARAMS"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), activation="Clip",
          activation_params=[0.0]), "ACT_PARAMS"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), activation="HardSigmoid"), "ACT_PARAMS"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3, 3), activation="Elu",
          activation_params=[1.0, 2.0]), "ACT_PARAMS"),
    (dict(x_shape=(1, 4, 2, 2), w_shape=(4, 4, 3, 3)), "EMPTY_OUTPUT"),
    (dict(x_shape=(1, 4, 8, 8, 8, 8), w_shape=(4, 4, 3, 3, 3, 3)), "BAD_RANK"),
    (dict(x_shape=(1, 4, 8, 8), w_shape=(4, 4, 3)), "BAD_RANK"),
])
def test_validation_rejects(kw, status):
    x_shape = kw.pop("x_shape")
    w_shape = kw.pop("w_shape")
    st, _, _, _ = oracle.resolve(x_shape, w_shape, **kw)
    assert st == status


def test_activation_param_defaults():
    """Defaults from the manifest's actAlpha/actBeta: optional-parameter activations."""
    v = -0.7
    x = np.full((1, 1, 1), v)
    w = np.ones((1, 1, 1))
    for name, alpha in [("QuickGelu", 1.702), ("Elu", 1.0), ("ThresholdedRelu", 1.0),
                        ("Gelu", 0.0)]:
        y, _ = oracle.fused_conv(x, w, activation=name)
        assert y[0, 0, 0] == oracle.activation(name, v, alpha)
    # parameter-free activations ignore the attribute
    y, _ = oracle.fused_conv(x, w, activation="Sigmoid", activation_params=[5.0, 6.0])
    assert y[0, 0, 0] == pytest.approx(1.0 / (1.0 + math.exp(0.7)), rel=1e-15)


def test_generator_matches_published_splitmix64():
    """splitmix64 from seed 0 starts with 0xE220A8397B1DCDAF (the published reference
    implementation's first output)."""
    assert int(workloads.splitmix64(0, 1)[0]) == 0xE220A8397B1DCDAF
