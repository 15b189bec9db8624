"""Host-side tests of the C ABI (no GPU): exported symbols, validation and shape
derivation against the oracle, route and split-K planning, run-time argument checks.
fconv_run's argument checks happen before any launch, so they run without a GPU."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import workloads
from activation_implicit_gemm_gb300 import FconvError, FusedConvPlan, _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "fconv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fconv_[a-z_]+)\s*\(", src)))


def test_library_exports_every_header_function(lib):
    names = header_functions()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)


def test_desc_struct_layout_matches_header(lib, tmp_path):
    # the ctypes mirror must have the C layout: compile a probe with gcc against the header
    probe = str(tmp_path / "desc_probe.c")
    with open(probe, "w") as f:
        f.write('#include <stdio.h>\n#include <stddef.h>\n#include "fconv.h"\n'
                'int main(void){printf("%zu %zu %zu %zu %zu\\n", sizeof(fconv_desc),'
                ' offsetof(fconv_desc, bias_len), offsetof(fconv_desc, group),'
                ' offsetof(fconv_desc, pads), offsetof(fconv_desc, act_params));'
                'printf("%zu\\n", sizeof(fconv_options)); return 0;}\n')
    exe = probe[:-2]
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), probe, "-o", exe])
    vals = subprocess.check_output([exe], text=True).split()
    D = _lib.FconvDesc
    assert int(vals[0]) == ctypes.sizeof(D)
    assert int(vals[1]) == D.bias_len.offset
    assert int(vals[2]) == D.group.offset
    assert int(vals[3]) == D.pads.offset
    assert int(vals[4]) == D.act_params.offset
    assert int(vals[5]) == ctypes.sizeof(_lib.FconvOptions)


def plan_status(lib, x_shape, w_shape, dtype=_lib.F16, **attrs):
    d = _lib.make_desc(dtype, x_shape, w_shape, **attrs)
    p = ctypes.c_void_p()
    st = lib.fconv_plan_create(ctypes.byref(d), -1, ctypes.byref(p))
    if st == 0:
        lib.fconv_destroy(p)
    return _lib.STATUS[st]


ORACLE_TO_API = {"OK": "OK", "ATTR_LENGTH": "E_ATTR_LENGTH", "ATTR_VALUE": "E_ATTR_VALUE",
                 "PADS_AUTOPAD": "E_PADS_WITH_AUTOPAD", "KERNEL_SHAPE": "E_KERNEL_SHAPE",
                 "GROUP": "E_GROUP", "ACT_PARAMS": "E_ACT_PARAMS", "EMPTY_OUTPUT": "E_OUTPUT_EMPTY",
                 "BAD_RANK": "E_RANK", "ACTIVATION": "E_ACTIVATION"}


def random_request(rng):
    sr = int(rng.integers(1, 4))
    G = int(rng.choice([1, 2, 3]))
    Cg = int(rng.integers(1, 4))
    Mg = int(rng.integers(1, 4))
    x_shape = (int(rng.integers(1, 3)), G * Cg + int(rng.choice([0, 0, 0, 1]))) + tuple(
        int(rng.integers(1, 9)) for _ in range(sr))
    w_shape = (G * Mg + int(rng.choice([0, 0, 0, 1])), Cg) + tuple(
        int(rng.integers(1, 5)) for _ in range(sr))
    attrs = dict(group=G)
    if rng.random() < 0.5:
        attrs["strides"] = [int(rng.integers(0, 4)) for _ in range(sr + int(rng.random() < 0.1))]
    if rng.random() < 0.5:
        attrs["dilations"] = [int(rng.integers(0, 3)) for _ in range(sr)]
    attrs["auto_pad"] = str(rng.choice(["NOTSET", "NOTSET", "SAME_UPPER", "SAME_LOWER", "VALID"]))
    if rng.random() < 0.6:
        attrs["pads"] = [int(rng.integers(-1, 3)) for _ in range(2 * sr)]
    if rng.random() < 0.2:
        attrs["kernel_shape"] = list(w_shape[2:]) if rng.random() < 0.7 else [9] * sr
    act = rng.choice([None] + oracle.ACTIVATIONS)
    attrs["activation"] = None if act is None else str(act)
    if rng.random() < 0.6:
        attrs["activation_params"] = [0.5] * int(rng.integers(0, 3))
    return x_shape, w_shape, attrs


def test_validation_and_shapes_agree_with_oracle(lib):
    """Random valid and invalid requests: same verdict, same output shape and pads."""
    rng = np.random.default_rng(2024)
    seen = set()
    for _ in range(600):
        x_shape, w_shape, attrs = random_request(rng)
        ost, oys, opb, ope = oracle.resolve(x_shape, w_shape, **attrs)
        d = _lib.make_desc(_lib.F16, x_shape, w_shape, **attrs)
        p = ctypes.c_void_p()
        st = lib.fconv_plan_create(ctypes.byref(d), -1, ctypes.byref(p))
        api = _lib.STATUS[st]
        seen.add(api)
        assert api == ORACLE_TO_API[ost], (x_shape, w_shape, attrs, api, ost)
        if st == 0:
            ys = (ctypes.c_int64 * 5)()
            rk = ctypes.c_int()
            assert lib.fconv_plan_output_shape(p, ys, ctypes.byref(rk)) == 0
            assert tuple(ys[i] for i in range(rk.value)) == oys
            pb, pe = (ctypes.c_int64 * 3)(), (ctypes.c_int64 * 3)()
            assert lib.fconv_plan_pads(p, pb, pe) == 0
            assert tuple(pb) == opb and tuple(pe) == ope
            lib.fconv_destroy(p)
        else:
            assert not p.value
    assert {"OK", "E_GROUP", "E_ATTR_VALUE", "E_ACT_PARAMS"} <= seen


def test_config_shapes_and_routes(lib):
    for c in workloads.ALL_CASES:
        dt = _lib.F16 if c.dtype == "f16" else _lib.F32
        p = FusedConvPlan(dt, c.x_shape, c.w_shape, has_bias=c.has_bias, has_z=c.has_z,
                          **c.attrs())
        assert p.y_shape == oracle.output_shape(c.x_shape, c.w_shape, **c.attrs())
        if c.dtype == "f32":
            assert p.route == "direct"
        elif c.group == c.x_shape[1] and c.w_shape[1] == 1:
            assert p.route == "depthwise"
        elif c.group > 1 and np.prod(c.w_shape[1:]) <= 64:
            # small groups with short reductions: CUDA cores, shared-memory halo box
            assert p.route == "grouped"
        else:
            assert p.route == "igemm_tc"
            assert p.tile_n in (64, 128, 256)  # the pixel tile (MMA N) cap
        expected_flops = 2.0 * np.prod(p.y_shape) * np.prod(c.w_shape[1:])
        assert p.flops == expected_flops


def test_split_k_planned_for_small_grids(lib):
    # one row tile << 152 SMs and a long K (2304 = 36 chunks of 64): K is split
    p = FusedConvPlan(_lib.F16, (1, 256, 8, 8), (128, 256, 3, 3), has_bias=True, has_z=True,
                      pads=[1, 1, 1, 1])
    assert p.split_k > 1
    # f32 partials per split, plus the weights copied into the GEMM's K order
    y_elems = np.prod(p.y_shape)
    assert p.workspace_bytes >= p.split_k * 4 * y_elems + 2 * 128 * 256 * 9
    # the 1-D config has 32 row tiles but only 5 chunks of K: too short to split
    c2 = workloads.case_by_name("1d_f16_64to64_k5_d2_same_upper_leakyrelu")
    p = FusedConvPlan(_lib.F16, c2.x_shape, c2.w_shape, has_bias=True, has_z=True, **c2.attrs())
    assert p.split_k == 1
    cb = workloads.case_by_name("cnn_b_64to128_16x16_z")
    p = FusedConvPlan(_lib.F16, cb.x_shape, cb.w_shape, has_z=True, **cb.attrs())
    # no split: the workspace holds the reordered weights and X repacked in 64-channel
    # blocks for the TMA-fed A operand
    wb = (2 * np.prod(cb.w_shape) + 1023) // 1024 * 1024
    xb = (2 * np.prod(cb.x_shape) + 1023) // 1024 * 1024
    assert p.split_k == 1 and p.workspace_bytes == wb + xb


def test_forced_routes(lib):
    p = FusedConvPlan(_lib.F16, (1, 8, 9, 9), (16, 8, 3, 3), route="igemm_tc", tile_n=128,
                      split_k=2)
    assert (p.route, p.tile_n, p.split_k) == ("igemm_tc", 128, 2)
    with pytest.raises(FconvError) as e:
        FusedConvPlan(_lib.F32, (1, 8, 9, 9), (16, 8, 3, 3), route="igemm_tc")
    assert e.value.code == "E_UNSUPPORTED"
    with pytest.raises(FconvError) as e:
        FusedConvPlan(_lib.F16, (1, 8, 9, 9), (16, 8, 3, 3), route="depthwise")
    assert e.value.code == "E_UNSUPPORTED"
    with pytest.raises(FconvError) as e:
        FusedConvPlan(_lib.F16, (1, 8, 9, 9), (16, 8, 3, 3), route="igemm_tc", tile_n=48)
    assert e.value.code == "E_UNSUPPORTED"
    with pytest.raises(FconvError) as e:  # pixel tiles are 64, 128 or 256
        FusedConvPlan(_lib.F16, (1, 8, 9, 9), (16, 8, 3, 3), route="igemm_tc", tile_n=32)
    assert e.value.code == "E_UNSUPPORTED"


def test_bias_and_z_shape_rules(lib):
    assert plan_status(lib, (1, 4, 8, 8), (6, 4, 3, 3), has_bias=True, bias_len=5) == "E_BIAS_SHAPE"
    assert plan_status(lib, (1, 4, 8, 8), (6, 4, 3, 3), has_bias=True, bias_len=6) == "OK"
    assert plan_status(lib, (1, 4, 8, 8), (6, 4, 3, 3), z_shape=(1, 6, 6, 6)) == "OK"
    assert plan_status(lib, (1, 4, 8, 8), (6, 4, 3, 3), z_shape=(1, 6, 8, 8)) == "E_Z_SHAPE"
    assert plan_status(lib, (1, 4, 8, 8), (6, 4, 3, 3), z_shape=(1, 6, 36)) == "E_Z_SHAPE"
    assert plan_status(lib, (1, 4, 8, 8), (6, 4, 3, 3), dtype=7) == "E_UNSUPPORTED"
    assert plan_status(lib, (1, 0, 8, 8), (6, 0, 3, 3)) == "E_RANK"


def test_run_argument_checks_launch_nothing(lib):
    """Every host-detected error returns before any CUDA call (runs without a GPU)."""
    p = FusedConvPlan(_lib.F16, (1, 8, 33, 20), (16, 8, 3, 3), has_bias=True, has_z=True,
                      pads=[1, 1, 1, 1], route="igemm_tc", split_k=2)
    ws = p.workspace_bytes
    assert ws > 0
    A = 0x10000  # fake, aligned device addresses: never dereferenced on these paths
    codes = {}

    def run(**kw):
        args = dict(x=A, w=2 * A, b=3 * A, z=4 * A, y=5 * A, ws=6 * A, n=ws)
        args.update(kw)
        st = lib.fconv_run(p._ptr, args["x"], args["w"], args["b"], args["z"], args["y"],
                           args["ws"], args["n"], None)
        return _lib.STATUS[st]

    codes["null x"] = run(x=None)
    codes["null b"] = run(b=None)
    codes["null z"] = run(z=None)
    codes["misaligned"] = run(x=A + 2)
    codes["alias"] = run(y=A)
    codes["small ws"] = run(n=ws - 1)
    codes["null ws"] = run(ws=None)
    assert codes == {"null x": "E_NULL", "null b": "E_NULL", "null z": "E_NULL",
                     "misaligned": "E_ALIGNMENT", "alias": "E_ALIAS", "small ws": "E_WORKSPACE",
                     "null ws": "E_WORKSPACE"}
    q = FusedConvPlan(_lib.F16, (1, 8, 9, 9), (16, 8, 3, 3))
    assert _lib.STATUS[lib.fconv_run(q._ptr, A, 2 * A, 3 * A, None, 5 * A, None, 0, None)] == \
        "E_BIAS_SHAPE"
    assert _lib.STATUS[lib.fconv_run(None, A, 2 * A, None, None, 5 * A, None, 0, None)] == "E_NULL"


def test_status_strings(lib):
    for code in _lib.STATUS:
        assert lib.fconv_status_string(code)
    assert lib.fconv_version() >= 100


def test_invariant_divisor_arithmetic(lib):
    """The multiply-shift division the kernels use for index decoding agrees with
    ordinary integer division (checked by the library's host code)."""
    assert lib.fconv_selftest_fastdiv() == 0


def test_launch_counts_and_workspace_regions(lib):
    # patch-fed tensor-core kernel: one launch, no workspace (X is read as it is, the
    # weights are resident or read as they are)
    ca = workloads.case_by_name("cnn_a_3to64_32x32")
    p = FusedConvPlan(_lib.F16, ca.x_shape, ca.w_shape, **ca.attrs())
    assert p.route == "igemm_tc" and p.split_k == 1 and p.launches == 1
    assert p.workspace_bytes == 0
    # a split plan adds the f32 partial sums and the reduction launch
    pk = FusedConvPlan(_lib.F16, (2, 16, 9, 9), (24, 16, 3, 3), pads=[1, 1, 1, 1],
                       route="igemm_tc", a_path="gather", split_k=3)
    assert pk.split_k == 3 and pk.launches == 2
    assert pk.workspace_bytes == 3 * 4 * 2 * 24 * 81
    # weights too large to keep resident with a row length that is not a multiple of 8
    # elements: a padded copy for the TMA boxes, written by its own launch
    pw = FusedConvPlan(_lib.F16, (1, 5, 9, 9), (1024, 5, 3, 3), pads=[1, 1, 1, 1],
                       route="igemm_tc", a_path="gather")
    assert pw.launches == 2 and pw.workspace_bytes == (1024 * 48 * 2 + 1023) // 1024 * 1024
    # TMA-fed kernel (C/group a multiple of 64): a prologue launch (weight copy in the
    # 64-channel block order + X repacked into 64-channel blocks) and the implicit GEMM,
    # plus the reduction when K is split; the workspace holds exactly those buffers
    cb = workloads.case_by_name("cnn_b_64to128_16x16_z")
    pt = FusedConvPlan(_lib.F16, cb.x_shape, cb.w_shape, has_z=True, route="igemm_tc",
                       a_path="tma", **cb.attrs())
    assert pt.launches == 2
    wcopy = (2 * 128 * 576 + 1023) // 1024 * 1024
    xcopy = (2 * 512 * 64 * 16 * 16 + 1023) // 1024 * 1024
    assert pt.workspace_bytes == wcopy + xcopy
    ps = FusedConvPlan(_lib.F16, (1, 256, 8, 8), (128, 256, 3, 3), pads=[1, 1, 1, 1],
                       a_path="tma")
    assert ps.split_k > 1 and ps.launches == 3
    # one kernel and no workspace on the depthwise and direct routes
    cd = workloads.case_by_name("stem_dw_128_k7")
    pd = FusedConvPlan(_lib.F16, cd.x_shape, cd.w_shape, has_bias=True, has_z=True,
                       **cd.attrs())
    assert pd.route == "depthwise" and pd.launches == 1 and pd.workspace_bytes == 0
    c1 = workloads.case_by_name("2d_f32_3to8_k3_relu")
    p1 = FusedConvPlan(_lib.F32, c1.x_shape, c1.w_shape, has_bias=True, **c1.attrs())
    assert p1.route == "direct" and p1.launches == 1 and p1.workspace_bytes == 0


def test_fp32_tensor_core_plans(lib):
    # C/group a multiple of 32: the 3xTF32 tensor-core path (prologue, GEMM, reduce)
    p = FusedConvPlan(_lib.F32, (2, 64, 10, 10), (48, 64, 3, 3), pads=[1, 1, 1, 1])
    assert p.route == "igemm_tc" and p.launches == 3
    kg, xs = 64 * 9, 2 * 64 * 100
    r = lambda v: (v + 1023) // 1024 * 1024
    assert p.workspace_bytes == 2 * r(48 * kg * 4) + 2 * r(xs * 4) + p.split_k * 2 * 48 * 100 * 4
    # forced split and pixel tile
    p = FusedConvPlan(_lib.F32, (2, 64, 10, 10), (48, 64, 3, 3), pads=[1, 1, 1, 1],
                      split_k=3, tile_n=64)
    assert (p.split_k, p.tile_n) == (3, 64)
    # C/group not a multiple of 32 stays on CUDA cores; the patch-fed A path is f16 only
    assert FusedConvPlan(_lib.F32, (2, 48, 10, 10), (16, 48, 3, 3)).route == "direct"
    with pytest.raises(FconvError):
        FusedConvPlan(_lib.F32, (2, 64, 10, 10), (48, 64, 3, 3), route="igemm_tc",
                      a_path="gather")



def test_half2_precision_is_depthwise_f16_only(lib):
    dw = dict(group=8, pads=[3, 3, 3, 3])
    p = FusedConvPlan(_lib.F16, (2, 8, 24, 24), (8, 1, 7, 7), precision="half2_rows", **dw)
    assert p.route == "depthwise"
    bad = [
        ((_lib.F32, (2, 8, 24, 24), (8, 1, 7, 7)), dw),                   # f32
        ((_lib.F16, (2, 8, 24, 24), (16, 8, 3, 3)), dict(pads=[1, 1, 1, 1])),  # not depthwise
        ((_lib.F16, (2, 8, 24, 21), (8, 1, 7, 7)), dw),                   # rows not 16-byte
        ((_lib.F16, (2, 8, 24, 24), (8, 1, 7, 7)), dict(dw, route="direct")),
    ]
    for (dt, xs, ws), attrs in bad:
        with pytest.raises(FconvError) as e:
            FusedConvPlan(dt, xs, ws, precision="half2_rows", **attrs)
        assert e.value.code == "E_UNSUPPORTED"


def test_bench_names_the_depthwise_kernel(lib):
    """The bench report names the streaming depthwise kernel exactly for the shapes the
    library streams (stride 1, K in 3/5/7, the same-size left pad modulo 4, X and Y rows in
    whole 4-element vectors), in either precision, and the tiled kernel otherwise."""
    import importlib.util
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_names", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)

    def name(xs, k, precision="default", **attrs):
        case = workloads.ConvCase("t", "f16", xs, (xs[1], 1, k, k), group=xs[1], **attrs)
        p = FusedConvPlan(_lib.F16, xs, case.w_shape, precision=precision, **case.attrs())
        return bench.main_kernel_name(case, p.route, p)

    stem = workloads.case_by_name("stem_dw_128_k7")
    assert name(stem.x_shape, 7, pads=(3, 3, 3, 3)) == "dw_stream_kernel"
    assert name(stem.x_shape, 7, precision="half2_rows", pads=(3, 3, 3, 3)) == "dw_stream_kernel"
    assert name((2, 8, 16, 16), 3, pads=(1, 1, 1, 1)) == "dw_stream_kernel"
    assert name((2, 8, 16, 16), 7, pads=(7, 7, 7, 7)) == "dw_stream_kernel"   # 7 = 3 mod 4
    assert name((2, 8, 16, 24), 5, auto_pad="SAME_UPPER") == "dw_stream_kernel"
    assert name((2, 8, 16, 21), 3, pads=(1, 1, 1, 1)) == "dw_tile_kernel"     # X rows ragged
    assert name((2, 8, 16, 24), 7, pads=(3, 0, 3, 0)) == "dw_tile_kernel"     # left pad 0
    assert name((2, 8, 16, 16), 3, pads=(1, 1, 1, 2)) == "dw_tile_kernel"     # Y rows ragged
