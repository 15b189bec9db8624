"""GPU parity: the CUDA kernels (through the C ABI) against the CPU oracle, element by
element, on identical seeded inputs.

* small cases that span several tiles and ragged tails, for every route, tile width,
  split-K factor, rank, stride/dilation/padding mode, group and activation;
* the benchmark convolutions at full size, in the launch configuration the benchmark
  times, every output of every image compared;
* the persistent kernels with their grid capped at 1-3 CTAs, so that each CTA walks many
  work units (every TMEM accumulator, every epilogue set, the operand ring's and the
  accumulators' phase wraps, the depthwise kernel's double buffer);
* exact results: integer-valued X, W, B, Z give exact sums, so the GPU output must equal
  the oracle bit for bit on every route;
* Y guard bands and NaN pre-fill catch out-of-bounds and missing writes.
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
    lib = _lib.load()
    assert lib.fconv_check_device(None) == 0, "a kernel reported a bounded-wait timeout"


def to_dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_run(plan: FusedConvPlan, xd, wd, bd, zd, dtype) -> np.ndarray:
    tdt = torch.float16 if dtype == "f16" else torch.float32
    ny = int(np.prod(plan.y_shape))
    buf = torch.full((ny + 2 * GUARD,), float("nan"), dtype=tdt, device="cuda")
    buf[:GUARD] = 7.0
    buf[-GUARD:] = 7.0
    y = buf[GUARD:GUARD + ny].view(plan.y_shape)
    ws = None
    if plan.workspace_bytes:
        ws = torch.full((plan.workspace_bytes // 4,), float("nan"), dtype=torch.float32,
                        device="cuda")
    plan.run(xd, wd, bd, zd, y=y, workspace=ws)
    torch.cuda.synchronize()
    head = buf[:GUARD].float().cpu().numpy()
    tail = buf[-GUARD:].float().cpu().numpy()
    assert np.all(head == 7.0) and np.all(tail == 7.0), "write outside Y"
    return y.double().cpu().numpy()


def compare(dtype, x, w, b, z, attrs, route="auto", split_k=0, tile_n=0, what="",
            a_path="auto", max_ctas=0):
    dt = _lib.F16 if dtype == "f16" else _lib.F32
    plan = FusedConvPlan(dt, x.shape, w.shape, has_bias=b is not None, has_z=z is not None,
                         route=route, split_k=split_k, tile_n=tile_n, a_path=a_path,
                         max_ctas=max_ctas, **attrs)
    y = gpu_run(plan, to_dev(x), to_dev(w), to_dev(b), to_dev(z), dtype)
    ref, absacc = oracle.fused_conv(x, w, b, z, **attrs)
    pre = None
    if attrs.get("activation") == "ThresholdedRelu":
        pre, _ = oracle.fused_conv(x, w, b, z, **{**attrs, "activation": None,
                                                  "activation_params": None})
    alpha = (attrs.get("activation_params") or [1.0])[0]
    kg = int(np.prod(w.shape[1:]))
    check(y, ref, absacc, dtype, kg, activation=attrs.get("activation"), alpha=alpha,
          pre_act=pre, what=f"{what} route={plan.route} tile={plan.tile_n} split={plan.split_k}")
    return plan


def inputs(seed, dtype, x_shape, w_shape, bias, zres, attrs, wscale=None):
    ys = oracle.output_shape(x_shape, w_shape, **attrs)
    kg = int(np.prod(w_shape[1:]))
    x = workloads.draw(seed, x_shape, "normal", 1.0, dtype)
    w = workloads.draw(seed + 1, w_shape, "normal", wscale or 1.0 / math.sqrt(kg), dtype)
    b = workloads.draw(seed + 2, (w_shape[0],), "normal", 1.0, dtype) if bias else None
    z = workloads.draw(seed + 3, ys, "normal", 1.0, dtype) if zres else None
    return x, w, b, z


# ----------------------------------------------------------------------------- tcgen05 path

@pytest.mark.parametrize("tile_n", [64, 128, 256])
@pytest.mark.parametrize("split_k", [1, 2, 3])
def test_tc_tiles_and_splits(tile_n, split_k):
    # 2*11*13 = 286 pixels: several pixel tiles with a ragged tail (tile_n caps the pixel
    # tile); Mg = 40 of a 128-channel tile; Kg = 216: 4 chunks, the last one partial
    attrs = dict(pads=[1, 1, 1, 1], activation="LeakyRelu", activation_params=[0.1])
    x, w, b, z = inputs(11, "f16", (2, 24, 11, 13), (40, 24, 3, 3), True, True, attrs)
    compare("f16", x, w, b, z, attrs, route="igemm_tc", tile_n=tile_n, split_k=split_k,
            what="tiles")


@pytest.mark.parametrize("tile_n", [64, 128, 256])
@pytest.mark.parametrize("split_k", [1, 2])
def test_tc_vector_epilogue_ragged(tile_n, split_k):
    # P = 64 (a multiple of 8: 16-byte Y/Z path); 3*64 = 192 pixels: whole-image boxes with
    # a partly filled last one; Mg = 40 of a 128-channel tile
    attrs = dict(pads=[1, 1, 1, 1], activation="QuickGelu")
    x, w, b, z = inputs(13, "f16", (3, 16, 8, 8), (40, 16, 3, 3), True, True, attrs)
    compare("f16", x, w, b, z, attrs, route="igemm_tc", tile_n=tile_n, split_k=split_k,
            what="vector epilogue")


TMA_CASES = [
    # (x_shape, w_shape, attrs, bias, z, tile_n, split_k): C/group % 64 == 0, so X is
    # repacked in 64-channel blocks and A arrives by TMA boxes
    ((3, 64, 8, 8), (40, 64, 3, 3), dict(pads=[1, 1, 1, 1]), True, True, 0, 0),        # whole images
    ((2, 64, 13, 11), (72, 64, 3, 3), dict(pads=[1, 0, 2, 1]), True, True, 0, 0),      # ragged box
    ((2, 128, 16, 16), (48, 128, 3, 3), dict(pads=[1, 1, 1, 1], activation="Gelu"), False, True, 64, 2),
    ((2, 64, 20, 20), (64, 64, 2, 2), dict(strides=[2, 2]), True, False, 0, 0),        # stride 2
    ((1, 64, 17, 19), (32, 64, 3, 3), dict(dilations=[2, 3], pads=[2, 3, 2, 3]), True, True, 128, 1),
    ((2, 64, 300), (64, 64, 5), dict(dilations=[2], auto_pad="SAME_UPPER"), True, True, 0, 0),
    ((1, 64, 6, 9, 10), (16, 64, 3, 3, 3), dict(strides=[2, 2, 2], auto_pad="SAME_LOWER"), True, True, 0, 0),
    ((2, 128, 7, 9), (96, 64, 3, 3), dict(group=2, pads=[1, 1, 1, 1]), True, True, 0, 0),  # grouped
    ((9, 256, 4, 4), (320, 256, 3, 3), dict(pads=[1, 1, 1, 1], activation="HardSwish"), False, True, 256, 0),
    ((2, 64, 9, 9), (24, 64, 1, 1), dict(), True, False, 0, 0),                        # 1x1
    ((2, 64, 12, 12), (16, 64, 3, 3), dict(strides=[3, 3], pads=[1, 1, 1, 1]), True, True, 64, 3),
    ((2, 384, 6, 6), (300, 384, 3, 3), dict(pads=[1, 1, 1, 1], activation="Relu"), True, True, 0, 0),  # 3 channel tiles
]


@pytest.mark.parametrize("idx", range(len(TMA_CASES)))
def test_tc_tma_path(idx):
    xs, ws, attrs, bias, zres, tile_n, split_k = TMA_CASES[idx]
    x, w, b, z = inputs(300 + 10 * idx, "f16", xs, ws, bias, zres, attrs)
    dt = _lib.F16
    plan = FusedConvPlan(dt, x.shape, w.shape, has_bias=b is not None, has_z=z is not None,
                         route="igemm_tc", a_path="tma", split_k=split_k, tile_n=tile_n, **attrs)
    y = gpu_run(plan, to_dev(x), to_dev(w), to_dev(b), to_dev(z), "f16")
    ref, absacc = oracle.fused_conv(x, w, b, z, **attrs)
    check(y, ref, absacc, "f16", int(np.prod(w.shape[1:])), activation=attrs.get("activation"),
          what=f"tma case {idx} tile={plan.tile_n} split={plan.split_k}")
    # the same request through the in-kernel gather agrees too
    compare("f16", x, w, b, z, attrs, route="igemm_tc", a_path="gather", what=f"gather case {idx}")


TC_CASES = [
    # (x_shape, w_shape, attrs, bias, z)
    ((3, 5, 17, 9), (7, 5, 3, 3), dict(pads=[1, 0, 2, 1]), True, False),          # Kg=45: scalar B
    ((2, 16, 300), (32, 16, 5), dict(dilations=[2], auto_pad="SAME_UPPER"), True, True),
    ((1, 8, 257), (24, 8, 3), dict(strides=[2], auto_pad="SAME_LOWER"), False, True),
    ((2, 12, 9, 10, 11), (16, 12, 3, 3, 3), dict(strides=[2, 2, 2], auto_pad="SAME_LOWER"),
     True, True),
    ((2, 12, 6, 7, 8), (24, 4, 3, 2, 3), dict(group=3, pads=[1, 0, 1, 1, 1, 0]), True, True),
    ((2, 6, 14, 15), (9, 2, 3, 3), dict(group=3, strides=[2, 1], dilations=[1, 2],
                                        pads=[1, 2, 0, 2]), True, False),
    ((1, 32, 8, 8), (32, 32, 1, 1), dict(), False, False),                       # README shape
    ((2, 3, 3, 3), (5, 3, 5, 5), dict(pads=[2, 2, 2, 2]), True, True),           # kernel > input
    ((1, 4, 5, 5), (3, 4, 5, 5), dict(), True, False),                           # 1x1 output
    ((4, 64, 7, 7), (200, 64, 3, 3), dict(pads=[1, 1, 1, 1], activation="Relu"), False, True),
    ((2, 3, 30, 30), (16, 3, 7, 7), dict(strides=[4, 4], pads=[3, 3, 3, 3],
                                         activation="Gelu"), True, False),
    ((2, 16, 12, 12), (32, 16, 2, 2), dict(strides=[2, 2]), False, False),
    ((2, 4, 9, 9), (4, 2, 3, 3), dict(group=2, auto_pad="VALID"), True, True),
    # K in one chunk with 4-channel copy units (padding units zeroed once), ragged rows
    ((3, 3, 11, 13), (10, 3, 3, 3), dict(pads=[1, 1, 1, 1], activation="QuickGelu"), False,
     True),
    # 4x4 images: one repack block spans five images (64-channel blocks, TMA-fed A)
    ((5, 64, 4, 4), (48, 64, 3, 3), dict(pads=[1, 1, 1, 1]), True, True),
]


@pytest.mark.parametrize("idx", range(len(TC_CASES)))
def test_tc_geometries(idx):
    xs, ws, attrs, bias, zres = TC_CASES[idx]
    x, w, b, z = inputs(100 + 10 * idx, "f16", xs, ws, bias, zres, attrs)
    compare("f16", x, w, b, z, attrs, route="igemm_tc", what=f"tc case {idx}")
    compare("f16", x, w, b, z, attrs, route="direct", what=f"direct case {idx}")


ACTS = [(None, None), ("Relu", None), ("LeakyRelu", [0.01]), ("Sigmoid", None),
        ("Tanh", None), ("HardSigmoid", [0.2, 0.5]), ("HardSwish", None), ("Clip", [-0.5, 0.75]),
        ("QuickGelu", None), ("QuickGelu", [1.0]), ("Elu", [0.7]), ("Gelu", None), ("Gelu", [1.0]),
        ("FastGelu", None), ("Softplus", None), ("ThresholdedRelu", [0.3]), ("Erf", None)]


@pytest.mark.parametrize("act,params", ACTS)
@pytest.mark.parametrize("route", ["igemm_tc", "direct", "depthwise", "grouped"])
def test_activations(act, params, route):
    if route == "depthwise":
        xs, ws, extra = (2, 8, 13, 14), (8, 1, 3, 3), dict(group=8)
    elif route == "grouped":
        xs, ws, extra = (2, 16, 8, 10), (32, 4, 3, 3), dict(group=4)
    else:
        # 8x10 output: P % 8 == 0 takes the 16-byte Y/Z epilogue on the tensor-core route
        xs, ws, extra = (2, 16, 8, 10), (24, 16, 3, 3), dict()
    attrs = dict(pads=[1, 1, 1, 1], activation=act, activation_params=params, **extra)
    x, w, b, z = inputs(500, "f16", xs, ws, True, True, attrs, wscale=0.8 / math.sqrt(9))
    compare("f16", x, w, b, z, attrs, route=route, what=f"act {act}")


@pytest.mark.parametrize("act,params", ACTS)
def test_activations_dw_stream(act, params):
    """Every activation through the column-streaming depthwise kernel (rows of X and Y in
    whole 4-element vectors, stride 1, the same-size left pad)."""
    xs, ws = (2, 8, 12, 16), (8, 1, 3, 3)
    attrs = dict(pads=[1, 1, 1, 1], group=8, activation=act, activation_params=params)
    x, w, b, z = inputs(520, "f16", xs, ws, True, True, attrs, wscale=0.8 / math.sqrt(9))
    compare("f16", x, w, b, z, attrs, route="depthwise", what=f"dw stream act {act}")


# ----------------------------------------------------------------------------- depthwise

DW_CASES = [
    ((2, 16, 20, 21), 3, dict(pads=[1, 1, 1, 1])),
    ((1, 8, 15, 16), 5, dict(auto_pad="SAME_UPPER")),
    ((2, 4, 30, 29), 7, dict(pads=[3, 3, 3, 3])),
    ((2, 8, 17, 17), 3, dict(strides=[2, 2], pads=[1, 1, 1, 1])),
    ((1, 8, 16, 19), 3, dict(dilations=[2, 3], pads=[2, 0, 1, 3])),
    ((1, 4, 9, 9), 4, dict(pads=[1, 2, 2, 1])),
    ((2, 3, 200, 220), 3, dict(pads=[1, 1, 1, 1])),  # several row bands per plane
    ((3, 16, 24, 32), 3, dict(pads=[1, 1, 1, 1])),    # persistent: one tile per plane
    ((2, 8, 56, 56), 7, dict(pads=[3, 3, 3, 3])),     # persistent, the stem's geometry
    ((2, 4, 8, 8), 5, dict(pads=[2, 2, 2, 2])),
    # tiled path: several tiles per plane in both directions, each left pad (it sets where
    # a thread's 16-value read starts), widths that are not multiples of 4 or 8
    ((2, 6, 70, 72), 5, dict(pads=[2, 1, 2, 3])),
    ((3, 5, 33, 40), 3, dict(pads=[0, 2, 1, 0])),
    ((2, 4, 19, 24), 7, dict(pads=[3, 0, 3, 0])),
    ((1, 3, 64, 136), 7, dict(auto_pad="SAME_UPPER")),
    ((2, 3, 12, 16), 3, dict(pads=[1, 3, 0, 3])),
    # column streaming (widths in whole 4-element vectors, the same-size left pad): bottom
    # and right pads other than the left and top ones, one column group, tall planes, pads
    # wider than the kernel's half
    ((2, 5, 21, 20), 5, dict(pads=[2, 2, 1, 2])),
    ((1, 6, 9, 4), 3, dict(pads=[1, 1, 1, 1])),
    ((1, 4, 130, 12), 7, dict(pads=[3, 3, 0, 3])),
    ((2, 3, 16, 24), 7, dict(pads=[7, 7, 7, 7])),
]


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("k", [3, 5, 7])
def test_depthwise_stream_without_b_z(k, dtype):
    """The column-streaming kernel with neither bias nor residual."""
    xs = (2, 6, 18, 20)
    attrs = dict(group=6, pads=[(k - 1) // 2] * 4, activation="Relu")
    x, w, b, z = inputs(760 + k, dtype, xs, (6, 1, k, k), False, False, attrs)
    compare(dtype, x, w, b, z, attrs, route="depthwise", what=f"dw stream no b/z k={k}")


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("idx", range(len(DW_CASES)))
def test_depthwise(idx, dtype):
    xs, k, attrs = DW_CASES[idx]
    C = xs[1]
    attrs = dict(attrs, group=C, activation="Clip", activation_params=[-1.0, 1.5])
    x, w, b, z = inputs(700 + idx, dtype, xs, (C, 1, k, k), True, True, attrs)
    compare(dtype, x, w, b, z, attrs, route="depthwise", what=f"dw {idx}")


# ----------------------------------------------------------------------------- grouped (small groups)

GROUPED_CASES = [
    # (x_shape, w_shape, attrs): C/group <= 16, M/group in 1..32, every rank
    ((2, 32, 16, 64, 64), (64, 8, 3, 3, 3), dict(group=4, strides=[2, 2, 2], auto_pad="SAME_LOWER")),
    ((2, 12, 9, 10, 11), (24, 3, 3, 3, 3), dict(group=4, pads=[1, 1, 1, 1, 1, 1])),
    ((2, 8, 7, 9, 8), (8, 1, 3, 3, 3), dict(group=8, pads=[1, 0, 1, 1, 2, 1])),       # 3-D depthwise
    ((3, 16, 300), (16, 1, 7), dict(group=16, auto_pad="SAME_UPPER")),                  # 1-D depthwise
    ((2, 32, 257), (64, 4, 5), dict(group=8, dilations=[2], pads=[4, 4])),
    ((2, 6, 14, 15), (9, 2, 3, 3), dict(group=3, strides=[2, 1], dilations=[1, 2], pads=[1, 2, 0, 2])),
    ((2, 64, 20, 19), (128, 16, 3, 3), dict(group=4, pads=[1, 1, 1, 1])),               # 16 -> 32
    ((1, 10, 70, 90), (20, 5, 5, 5), dict(group=2, strides=[3, 2], pads=[2, 2, 2, 2])),  # several boxes
    ((2, 8, 9, 9), (16, 1, 3, 3), dict(group=8, auto_pad="VALID")),                      # multiplier 2
]


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("idx", range(len(GROUPED_CASES)))
def test_grouped(idx, dtype):
    xs, ws, attrs = GROUPED_CASES[idx]
    attrs = dict(attrs, activation="HardSwish")
    x, w, b, z = inputs(1600 + 10 * idx, dtype, xs, ws, True, idx % 2 == 0, attrs)
    compare(dtype, x, w, b, z, attrs, route="grouped", what=f"grouped {idx}")


# ----------------------------------------------------------------------------- direct fp32

@pytest.mark.parametrize("sr", [1, 2, 3])
def test_direct_f32_random(sr):
    rng = np.random.default_rng(40 + sr)
    for it in range(4):
        G = int(rng.choice([1, 2]))
        Cg, Mg = int(rng.integers(1, 5)), int(rng.integers(1, 6))
        ins = [int(rng.integers(4, 12)) for _ in range(sr)]
        ks = [int(rng.integers(1, 4)) for _ in range(sr)]
        attrs = dict(group=G, strides=[int(rng.integers(1, 3)) for _ in range(sr)],
                     dilations=[int(rng.integers(1, 3)) for _ in range(sr)],
                     auto_pad="SAME_UPPER" if it % 2 else "SAME_LOWER", activation="Elu")
        x, w, b, z = inputs(900 + 10 * it + sr, "f32", (2, G * Cg) + tuple(ins),
                            (G * Mg, Cg) + tuple(ks), it % 2 == 0, it % 3 == 0, attrs)
        compare("f32", x, w, b, z, attrs, route="direct", what=f"direct f32 {sr}/{it}")


# ----------------------------------------------------------------------------- persistent loops

PERSISTENT_CASES = [
    # (x_shape, w_shape, attrs, route, a_path, tile_n, split_k): enough work units that a
    # capped grid walks every accumulator buffer and epilogue set several times
    ((4, 16, 20, 20), (40, 16, 3, 3), dict(pads=[1, 1, 1, 1], activation="QuickGelu"),
     "igemm_tc", "gather", 64, 1),
    ((4, 16, 24, 24), (40, 16, 3, 3), dict(pads=[1, 1, 1, 1]), "igemm_tc", "gather", 64, 2),
    ((3, 5, 23, 21), (130, 5, 3, 3), dict(pads=[1, 1, 1, 1], activation="HardSwish"),
     "igemm_tc", "gather", 128, 1),
    ((2, 8, 30, 32), (200, 8, 3, 3), dict(pads=[0, 1, 2, 1]), "igemm_tc", "gather", 256, 1),
    ((6, 64, 12, 12), (48, 64, 3, 3), dict(pads=[1, 1, 1, 1], activation="Gelu"),
     "igemm_tc", "tma", 64, 1),
    ((6, 64, 12, 12), (80, 64, 3, 3), dict(pads=[1, 1, 1, 1]), "igemm_tc", "tma", 128, 3),
    ((5, 128, 6, 6), (256, 128, 3, 3), dict(pads=[1, 1, 1, 1]), "igemm_tc", "tma", 256, 1),
    ((6, 16, 24, 24), (16, 1, 3, 3), dict(group=16, pads=[1, 1, 1, 1], activation="Relu"),
     "depthwise", "auto", 0, 0),
    ((3, 8, 40, 36), (8, 1, 7, 7), dict(group=8, pads=[3, 3, 3, 3]), "depthwise", "auto", 0, 0),
]


@pytest.mark.parametrize("max_ctas", [1, 2, 3])
@pytest.mark.parametrize("idx", range(len(PERSISTENT_CASES)))
def test_persistent_loop(idx, max_ctas):
    xs, ws, attrs, route, a_path, tile_n, split_k = PERSISTENT_CASES[idx]
    x, w, b, z = inputs(1200 + 10 * idx + max_ctas, "f16", xs, ws, True, True, attrs)
    compare("f16", x, w, b, z, attrs, route=route, a_path=a_path, tile_n=tile_n,
            split_k=split_k, max_ctas=max_ctas, what=f"persistent {idx} ctas={max_ctas}")


# ----------------------------------------------------------------------------- exact results

EXACT_CASES = [
    # (dtype, x_shape, w_shape, attrs, route, options, w range): integer X in [-2, 2],
    # B and Z in [-2, 2]; every |sum| stays below 2048, so f16 holds it exactly
    ("f16", (2, 12, 10, 9), (20, 12, 3, 3), dict(pads=[1, 1, 1, 1]), "igemm_tc",
     dict(a_path="gather"), 2),
    ("f16", (2, 12, 10, 9), (20, 12, 3, 3), dict(pads=[1, 1, 1, 1]), "igemm_tc",
     dict(a_path="gather", split_k=3), 2),
    ("f16", (3, 3, 17, 15), (16, 3, 5, 5), dict(strides=[2, 2], pads=[2, 2, 2, 2]), "igemm_tc",
     dict(a_path="gather"), 2),
    ("f16", (2, 64, 6, 7), (32, 64, 3, 3), dict(pads=[1, 1, 1, 1]), "igemm_tc",
     dict(a_path="tma"), 1),
    ("f16", (2, 64, 6, 7), (32, 64, 3, 3), dict(pads=[1, 1, 1, 1]), "igemm_tc",
     dict(a_path="tma", split_k=2), 1),
    ("f16", (2, 8, 14, 14), (8, 1, 7, 7), dict(group=8, pads=[3, 3, 3, 3]), "depthwise", {}, 2),
    ("f16", (2, 6, 9, 8), (9, 2, 3, 3), dict(group=3, pads=[1, 1, 1, 1]), "direct", {}, 2),
    ("f32", (2, 6, 9, 8), (9, 2, 3, 3), dict(group=3, pads=[1, 1, 1, 1]), "direct", {}, 2),
    ("f32", (2, 3, 5, 9, 8), (4, 3, 3, 3, 3), dict(strides=[1, 2, 1], auto_pad="SAME_UPPER"),
     "direct", {}, 2),
    ("f32", (2, 8, 14, 14), (8, 1, 3, 3), dict(group=8, pads=[1, 1, 1, 1]), "depthwise", {}, 2),
    ("f16", (2, 8, 14, 16), (8, 1, 7, 7), dict(group=8, pads=[3, 3, 3, 3]), "depthwise", {}, 2),
    ("f32", (2, 8, 12, 16), (8, 1, 5, 5), dict(group=8, pads=[2, 2, 2, 2]), "depthwise", {}, 2),
    ("f16", (2, 12, 5, 9, 8), (24, 3, 3, 3, 3), dict(group=4, pads=[1, 1, 1, 1, 1, 1]), "grouped",
     {}, 2),
    ("f32", (2, 16, 40), (32, 4, 5), dict(group=4, strides=[2], auto_pad="SAME_LOWER"), "grouped",
     {}, 2),
]


@pytest.mark.parametrize("idx", range(len(EXACT_CASES)))
def test_exact_integer_results(idx):
    """Integer-valued inputs: the convolution's sums are exact in f32 accumulation and in
    the oracle's fp64, so every output must be identical (no activation applied)."""
    dtype, xs, wsh, attrs, route, opts, wr = EXACT_CASES[idx]
    ys = oracle.output_shape(xs, wsh, **attrs)
    x = workloads.draw_int(1400 + 4 * idx, xs, -2, 2, dtype)
    w = workloads.draw_int(1401 + 4 * idx, wsh, -wr, wr, dtype)
    b = workloads.draw_int(1402 + 4 * idx, (wsh[0],), -2, 2, dtype)
    z = workloads.draw_int(1403 + 4 * idx, ys, -2, 2, dtype)
    dt = _lib.F16 if dtype == "f16" else _lib.F32
    plan = FusedConvPlan(dt, xs, wsh, has_bias=True, has_z=True, route=route, **opts, **attrs)
    y = gpu_run(plan, to_dev(x), to_dev(w), to_dev(b), to_dev(z), dtype)
    ref, absacc = oracle.fused_conv(x, w, b, z, **attrs)
    assert float(np.abs(ref).max()) < 2048.0
    assert np.array_equal(ref, np.round(ref)), "the oracle's sums of integers are integers"
    bad = y != ref
    assert not bad.any(), (f"exact case {idx} ({plan.route}): {int(bad.sum())} of {bad.size} "
                           f"outputs differ, first at {tuple(np.argwhere(bad)[0])}")


# ----------------------------------------------------------------------------- full-size configs

@pytest.mark.parametrize("name", [c.name for c in workloads.ALL_CASES])
def test_config_full_size(name):
    """Auto-planned run at full size, in the launch configuration the benchmark times;
    every output of every image compared with the oracle."""
    c = workloads.case_by_name(name)
    attrs = c.attrs()
    dt = _lib.F16 if c.dtype == "f16" else _lib.F32
    plan = FusedConvPlan(dt, c.x_shape, c.w_shape, has_bias=c.has_bias, has_z=c.has_z, **attrs)
    t = workloads.make_inputs(c, plan.y_shape)
    y = gpu_run(plan, to_dev(t["x"]), to_dev(t["w"]), to_dev(t["b"]), to_dev(t["z"]), c.dtype)
    ref, absacc = oracle.fused_conv(t["x"], t["w"], t["b"], t["z"], **attrs)
    kg = int(np.prod(c.w_shape[1:]))
    alpha = (attrs.get("activation_params") or [1.0])[0]
    check(y, ref, absacc, c.dtype, kg, activation=attrs.get("activation"), alpha=alpha,
          what=f"{name} route={plan.route} split={plan.split_k}")


# ----------------------------------------------------------------------------- stride == kernel
# Even stride and even kernel width along x, dilation 1, even left pad: the patch-fed kernel's
# builders read the taps (kx, kx + 1) of a pixel as one 32-bit load. An odd left pad keeps the
# 2-byte gathers.
PATCHIFY_CASES = [
    ((2, 24, 16, 20), (40, 24, 2, 2), dict(strides=[2, 2]), {}),
    ((1, 3, 64, 64), (32, 3, 4, 4), dict(strides=[4, 4], activation="Gelu"), {}),
    ((2, 16, 40), (24, 16, 2), dict(strides=[2]), {}),
    ((1, 8, 4, 8, 8), (16, 8, 2, 2, 2), dict(strides=[2, 2, 2]), {}),
    ((2, 128, 14, 14), (256, 128, 2, 2), dict(strides=[2, 2]), dict(a_path="gather")),
    ((2, 32, 12, 16), (48, 32, 2, 2), dict(strides=[2, 2], pads=[0, 2, 0, 2]), dict(split_k=2)),
    ((2, 32, 12, 16), (48, 32, 2, 2), dict(strides=[2, 2], pads=[1, 1, 1, 1]), {}),  # odd pad
    # patch embeddings of RGB images: one channel per patch block (its K stays a multiple of 8)
    ((2, 3, 64, 64), (96, 3, 8, 8), dict(strides=[8, 8]), {}),
    ((2, 3, 224, 224), (768, 3, 16, 16), dict(strides=[16, 16], activation="Gelu"), {}),
]


@pytest.mark.parametrize("idx", range(len(PATCHIFY_CASES)))
def test_stride_equals_kernel(idx):
    xs, ws, attrs, opts = PATCHIFY_CASES[idx]
    x, w, b, z = inputs(1900 + 10 * idx, "f16", xs, ws, True, True, attrs)
    compare("f16", x, w, b, z, attrs, route="igemm_tc", what=f"patchify {idx}", **opts)
