"""Seeded synthetic inputs and the benchmark convolution shapes for FusedConv.

This module holds no convolution arithmetic. It only defines shapes and attributes
and draws the input tensors, so that the CPU oracle and the CUDA path are fed
bit-identical data.

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) -> uniform doubles in (0, 1] -> Box-Muller for normals ->
round-to-nearest-even to the tensor dtype.
Seed of tensor t (X=0, W=1, B=2, Z=3) of conv j in workload c: 0xF0C0 + 16*c + 4*j + t.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int) -> np.ndarray:
    """The first n outputs of splitmix64 started from `seed` (uint64 array)."""
    with np.errstate(over="ignore"):
        i = np.arange(1, n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform01(seed: int, n: int) -> np.ndarray:
    """Doubles in (0, 1]: the top 53 bits of each draw, plus one, times 2^-53."""
    z = splitmix64(seed, n)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(seed: int, n: int) -> np.ndarray:
    """Standard normals by Box-Muller over consecutive pairs of uniforms."""
    m = (n + 1) // 2
    u = uniform01(seed, 2 * m)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    th = 2.0 * math.pi * u[1::2]
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    return out[:n]


def draw(seed: int, shape: Sequence[int], dist: str, scale: float, dtype: str) -> np.ndarray:
    """A seeded tensor of `shape`, rounded (RNE) to `dtype` ('f16' or 'f32')."""
    n = int(np.prod(shape)) if len(shape) else 1
    if dist == "normal":
        v = normal(seed, n) * scale
    elif dist == "uniform":  # U[-1, 1) scaled
        v = (uniform01(seed, n) * 2.0 - 1.0) * scale
    else:
        raise ValueError(dist)
    np_dt = np.float16 if dtype == "f16" else np.float32
    return v.astype(np_dt).reshape(shape)


def draw_int(seed: int, shape: Sequence[int], lo: int, hi: int, dtype: str) -> np.ndarray:
    """A seeded tensor of integers uniform in [lo, hi], stored as `dtype` ('f16' or 'f32')."""
    n = int(np.prod(shape)) if len(shape) else 1
    span = hi - lo + 1
    v = np.minimum(np.floor(uniform01(seed, n) * span), span - 1) + lo
    np_dt = np.float16 if dtype == "f16" else np.float32
    return v.astype(np_dt).reshape(shape)


@dataclasses.dataclass(frozen=True)
class ConvCase:
    """One FusedConv call: shapes, attributes and the value distributions of its inputs."""

    name: str
    dtype: str                        # 'f16' or 'f32'
    x_shape: tuple
    w_shape: tuple
    has_bias: bool = False
    has_z: bool = False
    group: int = 1
    strides: Optional[tuple] = None
    dilations: Optional[tuple] = None
    pads: Optional[tuple] = None
    auto_pad: str = "NOTSET"
    activation: Optional[str] = None
    activation_params: Optional[tuple] = None
    x_dist: tuple = ("normal", 1.0)
    w_dist: tuple = ("normal", 1.0)
    b_dist: tuple = ("normal", 1.0)
    z_dist: tuple = ("normal", 1.0)
    workload: int = 0                 # workload index used in the seed
    conv_index: int = 0               # conv index within the workload, used in the seed

    def seed(self, tensor_index: int) -> int:
        return 0xF0C0 + 16 * self.workload + 4 * self.conv_index + tensor_index

    def attrs(self) -> dict:
        return dict(group=self.group, strides=self.strides, dilations=self.dilations,
                    pads=self.pads, auto_pad=self.auto_pad, activation=self.activation,
                    activation_params=self.activation_params)


def make_inputs(case: ConvCase, y_shape: Optional[Sequence[int]] = None,
                batch: Optional[int] = None) -> dict:
    """Draw X, W, B and Z for `case` as numpy arrays of its dtype.

    Z needs the output shape, which the caller derives (oracle or library) and passes in.
    `batch` keeps only the first `batch` images of X and Z (a bounded sample).
    """
    out = {}
    x = draw(case.seed(0), case.x_shape, case.x_dist[0], case.x_dist[1], case.dtype)
    out["x"] = x if batch is None else x[:batch].copy()
    out["w"] = draw(case.seed(1), case.w_shape, case.w_dist[0], case.w_dist[1], case.dtype)
    out["b"] = (draw(case.seed(2), (case.w_shape[0],), case.b_dist[0], case.b_dist[1], case.dtype)
                if case.has_bias else None)
    if case.has_z:
        if y_shape is None:
            raise ValueError("Z needs the output shape")
        z = draw(case.seed(3), tuple(y_shape), case.z_dist[0], case.z_dist[1], case.dtype)
        out["z"] = z if batch is None else z[:batch].copy()
    else:
        out["z"] = None
    return out


def _kaiming(cin: int, k: int) -> float:
    return math.sqrt(2.0 / (cin * k))


# The five benchmark workloads. Shapes follow the operator's input rules (X is
# (N, C, D1..Dn), W is (M, C/group, k1..kn)); the workloads themselves are synthetic.
W1 = [
    ConvCase("2d_f32_3to8_k3_relu", "f32", (2, 3, 16, 16), (8, 3, 3, 3), has_bias=True,
             pads=(1, 1, 1, 1), activation="Relu", x_dist=("uniform", 1.0),
             w_dist=("uniform", 1.0), b_dist=("uniform", 1.0), workload=1, conv_index=0),
]
W2 = [
    ConvCase("1d_f16_64to64_k5_d2_same_upper_leakyrelu", "f16", (4, 64, 1024), (64, 64, 5),
             has_bias=True, has_z=True, dilations=(2,), auto_pad="SAME_UPPER",
             activation="LeakyRelu", activation_params=(0.01,),
             w_dist=("normal", 1.0 / math.sqrt(64 * 5)), workload=2, conv_index=0),
]
W3 = [
    ConvCase("cnn_a_3to64_32x32", "f16", (512, 3, 32, 32), (64, 3, 3, 3), pads=(1, 1, 1, 1),
             activation="QuickGelu", activation_params=(1.702,),
             w_dist=("normal", _kaiming(3, 9)), workload=3, conv_index=0),
    ConvCase("cnn_b_64to128_16x16_z", "f16", (512, 64, 16, 16), (128, 64, 3, 3), has_z=True,
             pads=(1, 1, 1, 1), activation="QuickGelu", activation_params=(1.702,),
             w_dist=("normal", _kaiming(64, 9)), workload=3, conv_index=1),
    ConvCase("cnn_c_128to256_8x8", "f16", (512, 128, 8, 8), (256, 128, 3, 3), pads=(1, 1, 1, 1),
             activation="QuickGelu", activation_params=(1.702,),
             w_dist=("normal", _kaiming(128, 9)), workload=3, conv_index=2),
    ConvCase("cnn_d_256to512_4x4_z", "f16", (512, 256, 4, 4), (512, 256, 3, 3), has_z=True,
             pads=(1, 1, 1, 1), activation="QuickGelu", activation_params=(1.702,),
             w_dist=("normal", _kaiming(256, 9)), workload=3, conv_index=3),
]
W4 = [
    ConvCase("stem_patch_3to128_k7_s4", "f16", (32, 3, 224, 224), (128, 3, 7, 7), has_bias=True,
             strides=(4, 4), pads=(3, 3, 3, 3), activation="Gelu", workload=4, conv_index=0),
    ConvCase("stem_dw_128_k7", "f16", (32, 128, 56, 56), (128, 1, 7, 7), has_bias=True,
             has_z=True, group=128, pads=(3, 3, 3, 3), activation="Clip",
             activation_params=(0.0, 6.0), workload=4, conv_index=1),
    ConvCase("stem_down_128to256_k2_s2", "f16", (32, 128, 56, 56), (256, 128, 2, 2),
             strides=(2, 2), workload=4, conv_index=2),
]
W5 = [
    ConvCase("3d_f16_32to64_k3_s2_same_lower", "f16", (2, 32, 16, 64, 64), (64, 32, 3, 3, 3),
             has_bias=True, strides=(2, 2, 2), auto_pad="SAME_LOWER", activation="HardSwish",
             workload=5, conv_index=0),
    ConvCase("3d_f16_grouped4_z", "f16", (2, 32, 16, 64, 64), (64, 8, 3, 3, 3), has_bias=True,
             has_z=True, group=4, strides=(2, 2, 2), auto_pad="SAME_LOWER",
             activation="HardSwish", workload=5, conv_index=1),
]

WORKLOADS = {1: W1, 2: W2, 3: W3, 4: W4, 5: W5}
ALL_CASES = W1 + W2 + W3 + W4 + W5


def case_by_name(name: str) -> ConvCase:
    for c in ALL_CASES:
        if c.name == name:
            return c
    raise KeyError(name)


# Widening beyond the benchmark suite (measured next to it, not part of its value): the
# transposed convolution of an upsampling stage, W of shape (C, M/group, k, k).
TRANSPOSED_CASES = [
    dict(name="convT_up_256to128_k4_s2", dtype="f16", x_shape=(8, 256, 32, 32),
         w_shape=(256, 128, 4, 4), attrs=dict(strides=[2, 2], pads=[1, 1, 1, 1],
                                              activation="Relu"), seed=0xF1C0),
]


def make_transposed_inputs(case: dict, y_shape: Sequence[int]) -> dict:
    """X ~ N(0,1), W ~ N(0,1)/sqrt(C/group * k*k), B, Z ~ N(0,1) for a transposed case."""
    xs, ws = case["x_shape"], case["w_shape"]
    g = case["attrs"].get("group", 1)
    kg = (ws[0] // g) * int(np.prod(ws[2:]))
    s, dt = case["seed"], case["dtype"]
    return {"x": draw(s, xs, "normal", 1.0, dt),
            "w": draw(s + 1, ws, "normal", 1.0 / float(np.sqrt(kg)), dt),
            "b": draw(s + 2, (y_shape[1],), "normal", 1.0, dt),
            "z": draw(s + 3, y_shape, "normal", 1.0, dt)}


# fp32 convolution on the tensor cores (3xTF32): a ResNet-stage 3x3 conv, measured beside the
# suite with the CUDA-core route timed on the same inputs for comparison.
FP32_TC_CASES = [
    ConvCase("f32_tc_128to128_28x28_k3", "f32", (32, 128, 28, 28), (128, 128, 3, 3),
             has_bias=True, has_z=True, pads=(1, 1, 1, 1), activation="Relu",
             w_dist=("normal", 0.03), workload=6, conv_index=0),
]


# stride == kernel (patchify): a ViT patch embedding of RGB images, 16x16 patches, measured
# beside the suite with the CUDA-core route timed on the same inputs for comparison.
PATCHIFY_CASES = [
    ConvCase("vit_patchify_3to768_k16_s16", "f16", (32, 3, 224, 224), (768, 3, 16, 16),
             has_bias=True, strides=(16, 16), w_dist=("normal", 0.036), workload=7,
             conv_index=0),
]

