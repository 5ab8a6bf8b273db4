"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs, element by element, for every kernel family and
dtype, at sizes spanning several tiles with ragged tails; then the five layer
sets at full size, every output element compared; then the boundary's
run-time checks."""
import zlib

import numpy as np
import pytest
import torch

from conv_workloads import CONFIGS, LayerSpec, generate, make_layer, output_hw
from parity_util import (assert_close, make_plan, run_gpu, run_oracle, run_oracle_points,
                         sample_points)

pytestmark = pytest.mark.gpu

_I8 = dict(dtype="i8", act="none", x_dist=("int", -128, 127), w_dist=("int", -127, 127),
           b_dist=("int", -1000, 1000))


def L(name, n, h, w, cin, cout, kh, kw, s=1, ph=0, pw=0, groups=1, dtype="bf16", act=None, **extra):
    if act is None:
        act = "none" if dtype == "i8" else "mish"
    base = dict(x_dist=("uniform", -1.0, 1.0), w_dist=("he",), b_dist=("normal", 0.5))
    if dtype == "i8":
        base = dict(x_dist=_I8["x_dist"], w_dist=_I8["w_dist"], b_dist=_I8["b_dist"])
    base.update(extra)
    return LayerSpec(name, n, h, w, cin, cout, kh, kw, s, ph, pw, groups, dtype, act, **base)


def check(spec, algo="auto", expect_algo=None, seed=0):
    g = torch.Generator("cpu").manual_seed(seed)
    d = make_layer(spec, g)
    y, plan = run_gpu(spec, d, algo)
    if expect_algo:
        assert plan.algo == expect_algo, plan.describe()
    ref = run_oracle(spec, d)
    assert_close(spec, y, ref, f"{spec.name} [{plan.describe()}]")
    return plan


# ------------------------------------------------ tcgen05 implicit GEMM (bf16)

IGEMM = [
    L("3x3_s1_ragged", 2, 19, 21, 64, 80, 3, 3, 1, 1, 1),
    L("3x3_s2_bk32", 1, 23, 17, 32, 64, 3, 3, 2, 1, 1, act="relu"),
    L("3x3_bk16_cout24", 1, 13, 9, 16, 24, 3, 3, 1, 1, 1, act="none"),
    L("5x5_p2", 1, 12, 12, 64, 128, 5, 5, 1, 2, 2),
    L("1x3_asym_pad", 1, 9, 14, 64, 64, 1, 3, 1, 0, 1),
    L("3x3_overpad", 1, 7, 7, 64, 64, 3, 3, 1, 2, 2),
    L("3x3_s3_p0", 1, 20, 20, 64, 64, 3, 3, 3, 0, 0),
    L("3x3_many_kblocks", 1, 10, 10, 256, 256, 3, 3, 1, 1, 1),
    L("3x3_wide_rows", 2, 6, 150, 64, 64, 3, 3, 1, 1, 1),
    L("1x1_flat_ragged", 2, 15, 15, 128, 192, 1, 1),
    L("1x1_flat_bn256", 1, 10, 10, 64, 512, 1, 1, act="relu"),
    L("1x1_stride2", 1, 17, 17, 64, 64, 1, 1, 2, 0, 0),
    L("1x1_cout8", 1, 9, 9, 32, 8, 1, 1, act="none"),
    L("3x3_no_bias", 1, 11, 11, 64, 64, 3, 3, 1, 1, 1, b_dist=None),
    L("7x7_s2_p3", 1, 30, 30, 32, 64, 7, 7, 2, 3, 3),
    L("3x3_single_pixel", 1, 1, 1, 64, 64, 3, 3, 1, 1, 1),
    L("ragged_cout_two_ntiles", 1, 12, 12, 128, 320, 3, 3, 1, 1, 1),
    L("1x1_flat_long_k", 2, 8, 8, 512, 384, 1, 1, act="relu"),
    L("3x3_s2_few_tiles", 1, 20, 20, 256, 512, 3, 3, 2, 1, 1),
]


# Every case runs with the layout the plan picks and with each forced tile
# layout: swapped (c_out <= 128 only), N = 256, 128 and 64, and the CTA pair.
_LAYOUT_DESC = {"igemm_swapped": "swapped", "igemm_n256": "M=128px N=256co", "igemm_n128": "N=128co",
                "igemm_n64": "N=64co", "igemm_pair": "cta-pair M=256px N=256co",
                "igemm_pair128": "cta-pair M=256px N=128co"}


def halo_eligible(spec):
    # halo staging: stride-1 layers with three filter rows
    return spec.stride == 1 and spec.kh == 3


def with_layouts(specs):
    # Layers that can take halo staging run each layout with it and with
    # per-tap boxes forced, as well as with the plan's own choice.
    out = []
    for spec in specs:
        for lay in ["igemm", "igemm_swapped", "igemm_n256", "igemm_n128", "igemm_n64", "igemm_pair",
                    "igemm_pair128"]:
            if lay == "igemm_swapped" and spec.cout > 128:
                continue
            variants = ["", "+halo", "+taps"] if halo_eligible(spec) else [""]
            # the epilogue split, on the layouts that offer both
            if lay in ("igemm", "igemm_n128", "igemm_n64"):
                variants += ["+ept", "+sliced"] + (["+halo+ept"] if halo_eligible(spec) else [])
            for v in variants:
                out.append(pytest.param(spec, lay + v, id=f"{spec.name}-{lay}{v}"))
    return out


def check_layout(spec, layout):
    plan = check(spec, layout, "igemm")
    base, *flags = layout.split("+")
    if base in _LAYOUT_DESC:
        assert _LAYOUT_DESC[base] in plan.describe(), plan.describe()
    if "halo" in flags or "taps" in flags:
        assert (" halo " in plan.describe()) == ("halo" in flags), plan.describe()
    if "ept" in flags or "sliced" in flags:
        assert ("epi=tile" in plan.describe()) == ("ept" in flags), plan.describe()
    return plan


def test_epilogue_per_tile_needs_normal_layout():
    spec = L("ept_cout256", 1, 8, 8, 64, 256, 3, 3, 1, 1, 1)
    d = make_layer(spec, torch.Generator("cpu").manual_seed(0))
    for algo in ("igemm_swapped+ept", "igemm_n256+ept", "igemm_pair+ept", "igemm_pair128+ept"):
        with pytest.raises(RuntimeError, match="UNSUPPORTED"):
            make_plan(spec, d, algo)


def test_halo_staging_needs_stride1_kh3():
    for spec in (L("halo_s2", 1, 12, 12, 64, 64, 3, 3, 2, 1, 1), L("halo_5x5", 1, 12, 12, 64, 64, 5, 5, 1, 2, 2)):
        d = make_layer(spec, torch.Generator("cpu").manual_seed(0))
        with pytest.raises(RuntimeError, match="UNSUPPORTED"):
            make_plan(spec, d, "igemm+halo")


@pytest.mark.parametrize("spec,layout", with_layouts(IGEMM))
def test_igemm_bf16(spec, layout):
    check_layout(spec, layout)


def test_swapped_layout_needs_cout_le_128():
    spec = L("swap_cout256", 1, 8, 8, 64, 256, 3, 3, 1, 1, 1)
    d = make_layer(spec, torch.Generator("cpu").manual_seed(0))
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        make_plan(spec, d, "igemm_swapped")


# int8 on the tensor cores (operands widened to bf16, exact fp32 accumulation):
# results must be bit-identical to the oracle's int64 accumulation.
IGEMM_I8 = [
    L("i8_3x3_64to64_ragged", 1, 21, 19, 64, 64, 3, 3, 1, 1, 1, dtype="i8"),
    L("i8_3x3_relu_sat", 2, 13, 11, 64, 48, 3, 3, 1, 1, 1, dtype="i8", act="relu",
      b_dist=("int", -300000, 300000)),
    L("i8_1x1_32to64", 1, 24, 20, 32, 64, 1, 1, dtype="i8"),
    L("i8_3x3_s2_cin48_pad", 1, 17, 15, 48, 32, 3, 3, 2, 1, 1, dtype="i8"),
    L("i8_cout256_normal_mode", 1, 9, 9, 32, 256, 3, 3, 1, 1, 1, dtype="i8"),
    L("i8_k_1024", 1, 8, 8, 1024, 16, 1, 1, dtype="i8", act="relu"),
    L("i8_cin3_pad", 1, 18, 16, 3, 16, 3, 3, 1, 1, 1, dtype="i8"),
    L("i8_kwfold_s2", 1, 19, 22, 4, 32, 3, 3, 2, 1, 1, dtype="i8", act="relu"),
]


@pytest.mark.parametrize("spec,layout", with_layouts(IGEMM_I8))
def test_igemm_int8_exact(spec, layout):
    plan = check_layout(spec, layout)
    assert "i8-as-bf16" in plan.describe() or "i8-widened-in-kernel" in plan.describe()


# int8 operands widened in the kernel (converter warpgroup) or by the
# pre-pass, forced, on the layers whose rows are whole 16-byte units and
# whose weights stay resident: bit-identical results either way.
I8_WIDEN = [s for s in IGEMM_I8 if s.name in ("i8_3x3_64to64_ragged", "i8_3x3_relu_sat", "i8_1x1_32to64",
                                                "i8_3x3_s2_cin48_pad")]


# (N = 128 keeps nine resident 128-row weight blocks, too many for shared
# memory beside the rings: in the kernel only for the 1x1 layer there)
@pytest.mark.parametrize("spec,layout", [
    pytest.param(spec, f"{lay}+{w}", id=f"{spec.name}-{lay}+{w}")
    for spec in I8_WIDEN for lay in ("igemm", "igemm_n64", "igemm_n128") for w in ("inkernel", "prepass")
    if not (w == "inkernel" and lay == "igemm_n128" and spec.kh > 1)
] + [pytest.param(spec, "igemm_n64+halo+inkernel", id=f"{spec.name}-igemm_n64+halo+inkernel")
     for spec in I8_WIDEN if spec.stride == 1 and spec.kh == 3
] + [pytest.param(spec, f"igemm_n64+{ep}+inkernel", id=f"{spec.name}-igemm_n64+{ep}+inkernel")
     for spec in I8_WIDEN for ep in ("ept", "sliced")])
def test_igemm_int8_widening(spec, layout):
    plan = check(spec, layout, "igemm")
    want = "i8-widened-in-kernel" if "inkernel" in layout else "i8-as-bf16"
    assert want in plan.describe(), plan.describe()
    assert plan.launches == (1 if "inkernel" in layout else 2)


def test_int8_widening_in_kernel_needs_whole_rows():
    spec = L("i8_cin3_no_cvt", 1, 18, 16, 3, 16, 3, 3, 1, 1, 1, dtype="i8")
    d = make_layer(spec, torch.Generator("cpu").manual_seed(0))
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        make_plan(spec, d, "igemm+inkernel")


# bf16 layers with k_w x Cin <= 16 whose image rows are whole 16-byte units:
# the folded operand assembled in the kernel (converter warpgroup) from the
# plain NHWC rows, forced, against the folding pre-pass; both must match the
# oracle.  Ragged heights and widths, stride 2, padding wider than k_w / 2,
# one input channel, k_h = 5 and 10.
FOLD_INKERNEL = [
    L("fold_stem_cin3_ragged_h", 2, 37, 48, 3, 32, 3, 3, 1, 1, 1),
    L("fold_stem_cin3_s2", 1, 41, 64, 3, 32, 3, 3, 2, 1, 1, act="relu"),
    # (128 output columns: the widest tile's raw rows would pass 256 elements)
    L("fold_stem_s2_wide_rows", 1, 21, 256, 3, 32, 3, 3, 2, 1, 1),
    L("fold_cin4_cout48", 1, 23, 20, 4, 48, 3, 3, 1, 1, 1, act="none"),
    L("fold_cin5_s2_overpad_w", 1, 21, 16, 5, 24, 3, 3, 2, 1, 2, act="relu"),
    L("fold_5x2_no_pad", 2, 11, 12, 8, 16, 5, 2, 1, 0, 0),
    L("fold_cin1_10x4", 1, 49, 16, 1, 64, 10, 4, 2, 5, 1, act="none"),
]


@pytest.mark.parametrize("spec,layout", [
    pytest.param(spec, f"{lay}+{w}", id=f"{spec.name}-{lay}+{w}")
    for spec in FOLD_INKERNEL for lay in ("igemm_n64", "igemm_n128") for w in ("inkernel", "prepass")
] + [pytest.param(spec, f"igemm_n64+{st}+{ep}+inkernel", id=f"{spec.name}-igemm_n64+{st}+{ep}+inkernel")
     for spec in FOLD_INKERNEL for st in ("taps", "halo") for ep in ("ept", "sliced")
     if st == "taps" or (spec.stride == 1 and spec.kh == 3)])
def test_kw_fold_in_kernel(spec, layout):
    plan = check(spec, layout, "igemm")
    want = "bf16-kwfold-in-kernel" if "inkernel" in layout else "bf16-cpad-kwfold"
    assert want in plan.describe(), plan.describe()
    assert plan.launches == (1 if "inkernel" in layout else 2)


# The in-kernel fold with tiles of two stacked 128-pixel M blocks (N = 64,
# halo staging, an epilogue per tile; chosen on layers with at least two tiles
# per SM): ragged heights put a tile's bottom block partly or wholly below the
# image (the latter stores nothing), and stride 1 only (halo staging).
FOLD_MB2 = [
    L("fold_mb2_bottom_block_outside", 1, 584, 256, 3, 32, 3, 3, 1, 1, 1),
    L("fold_mb2_b2_half_tile_row", 2, 304, 304, 3, 32, 3, 3, 1, 1, 1, act="relu"),
]


@pytest.mark.parametrize("spec", FOLD_MB2, ids=lambda s: s.name)
def test_kw_fold_two_m_blocks(spec):
    plan = check(spec, "auto", "igemm")
    assert "kwfold-in-kernel" in plan.describe() and "(2 M blocks)" in plan.describe(), plan.describe()


def test_kw_fold_in_kernel_needs_whole_rows():
    # 45 pixels x 3 channels x 2 bytes = 270: not a whole number of 16-byte units
    spec = L("fold_row_270_bytes", 1, 18, 45, 3, 32, 3, 3, 1, 1, 1)
    d = make_layer(spec, torch.Generator("cpu").manual_seed(0))
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        make_plan(spec, d, "igemm+inkernel")


# bf16 layers whose channel rows are too short for TMA: channels padded to 16.
IGEMM_CPAD = [
    L("cpad_stem_cin3", 1, 37, 45, 3, 32, 3, 3, 1, 1, 1),
    L("cpad_cin24_s2", 2, 15, 13, 24, 64, 3, 3, 2, 1, 1, act="relu"),
    L("cpad_cin1_10x4", 1, 49, 10, 1, 64, 10, 4, 2, 5, 1, act="none"),
    # k_w x Cin <= 16: the k_w taps are folded into the padded channels
    L("kwfold_1x3_flat", 1, 9, 40, 4, 32, 1, 3, 1, 0, 1),
    L("kwfold_s2_overpad_w", 1, 21, 23, 5, 24, 3, 3, 2, 1, 2, act="relu"),
    L("kwfold_5x2_no_pad", 2, 11, 12, 8, 16, 5, 2, 1, 0, 0),
]


@pytest.mark.parametrize("spec,layout", with_layouts(IGEMM_CPAD))
def test_igemm_channel_padding(spec, layout):
    plan = check_layout(spec, layout)
    folded = spec.kw > 1 and spec.kw * spec.cin <= 16
    # (a folded layer whose image rows are whole 16-byte units is folded in the kernel)
    assert "cpad" in plan.describe() or (folded and "kwfold-in-kernel" in plan.describe()), plan.describe()
    assert ("kwfold" in plan.describe()) == folded


def test_int8_plan_without_tensor_core_path_falls_to_dp4a():
    # K = 9 * 256 > 1024: the exact-accumulation bound is not met
    spec = L("i8_long_k", 1, 6, 6, 256, 16, 3, 3, 1, 1, 1, dtype="i8")
    plan = check(spec, "auto", "direct")
    assert "dp4a" in plan.describe()


# ------------------------------------------------ depthwise 3x3

DW = []
for dt, C in (("f32", 12), ("bf16", 24), ("i8", 48)):
    for s, p in ((1, 1), (2, 1), (1, 0), (2, 2), (3, 1)):
        act = "relu" if dt != "bf16" else "mish"
        DW.append(L(f"dw_{dt}_s{s}_p{p}", 2, 13, 11, C, C, 3, 3, s, p, p, groups=C, dtype=dt, act=act))
DW.append(L("dw_i8_relu_sat", 1, 9, 9, 32, 32, 3, 3, 1, 1, 1, groups=32, dtype="i8", act="relu",
            b_dist=("int", -200000, 200000)))


@pytest.mark.parametrize("spec", DW, ids=lambda s: s.name)
def test_depthwise(spec):
    check(spec, "depthwise", "depthwise")


# The general depthwise kernel walks 8 output rows a tile on layers with a
# tile per SM or more, and fewer (4, 2, 1) on smaller ones: both regimes, in
# each type (bf16 here at stride 2: stride 1 runs the rolling-row kernel).
DW_TH = [
    (L("dw_i8_160_th8", 1, 160, 160, 64, 64, 3, 3, 1, 1, 1, groups=64, dtype="i8", act="relu"), 8),
    (L("dw_f32_96_th8", 2, 96, 96, 32, 32, 3, 3, 1, 1, 1, groups=32, dtype="f32", act="relu"), 8),
    (L("dw_bf16_s2_192_th8", 1, 192, 192, 64, 64, 3, 3, 2, 1, 1, groups=64, act="mish"), 8),
    (L("dw_i8_24_small", 1, 24, 24, 32, 32, 3, 3, 1, 1, 1, groups=32, dtype="i8"), 1),
]


@pytest.mark.parametrize("spec,th", DW_TH, ids=[s.name for s, _ in DW_TH])
def test_depthwise_tile_rows(spec, th):
    plan = check(spec, "depthwise", "depthwise")
    if th == 8:
        assert "tile=8x" in plan.describe(), plan.describe()
    else:
        assert "tile=8x" not in plan.describe(), plan.describe()


# bf16 stride 1 runs on the rolling-row kernel: ragged row and column tiles,
# each padding and activation, channel counts from one 8-channel block up.
DW_ROWS = [
    L("dwr_c8_p1_mish", 1, 9, 7, 8, 8, 3, 3, 1, 1, 1, groups=8),
    L("dwr_c24_p0_relu", 2, 13, 11, 24, 24, 3, 3, 1, 0, 0, groups=24, act="relu"),
    L("dwr_c40_p2_none", 1, 11, 17, 40, 40, 3, 3, 1, 2, 2, groups=40, act="none"),
    L("dwr_c64_asym_pad", 2, 10, 23, 64, 64, 3, 3, 1, 1, 0, groups=64),
    L("dwr_c136_ragged", 1, 21, 19, 136, 136, 3, 3, 1, 1, 1, groups=136),
    L("dwr_c512_b3", 3, 17, 12, 512, 512, 3, 3, 1, 1, 1, groups=512, b_dist=None),
    L("dwr_single_row", 1, 1, 30, 32, 32, 3, 3, 1, 1, 1, groups=32),
]


@pytest.mark.parametrize("spec", DW_ROWS, ids=lambda s: s.name)
def test_depthwise_rows(spec):
    plan = check(spec, "depthwise", "depthwise")
    assert " rows " in plan.describe(), plan.describe()


# ------------------------------------------------ direct (CUDA cores)

DIRECT = [
    L("f32_3x3", 1, 28, 28, 8, 16, 3, 3, 1, 1, 1, dtype="f32", act="relu"),
    L("f32_stem_10x4", 1, 49, 10, 1, 64, 10, 4, 2, 5, 1, dtype="f32", act="relu"),
    L("f32_grouped", 2, 9, 8, 8, 12, 3, 3, 1, 1, 1, groups=4, dtype="f32", act="mish"),
    L("f32_1x1", 1, 25, 5, 64, 64, 1, 1, dtype="f32", act="relu"),
    L("bf16_stem_cin3", 1, 33, 35, 3, 32, 3, 3, 1, 1, 1),
    L("bf16_grouped", 1, 10, 10, 16, 32, 3, 3, 2, 1, 1, groups=2),
    L("i8_3x3_dp4a", 1, 17, 19, 64, 40, 3, 3, 1, 1, 1, dtype="i8"),
    L("i8_1x1", 1, 12, 12, 32, 64, 1, 1, dtype="i8", act="relu"),
    L("i8_cin3_scalar", 1, 11, 9, 3, 16, 3, 3, 2, 1, 1, dtype="i8"),
    L("i8_grouped", 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, groups=4, dtype="i8"),
]


@pytest.mark.parametrize("spec", DIRECT, ids=lambda s: s.name)
def test_direct(spec):
    check(spec, "direct", "direct")


# Layers with enough pixels that each thread takes two (PT = 2): 16-byte
# channel chunks in flight per batch (a partial last batch: K = 72 is 18
# chunks) and, grouped with 4 channels a group, single values (K = 36).
DIRECT_PT2 = [
    L("direct_pt2_f32_3x3", 1, 640, 640, 8, 16, 3, 3, 1, 1, 1, dtype="f32", act="relu"),
    L("direct_pt2_f32_grouped", 1, 640, 640, 8, 16, 3, 3, 1, 1, 1, groups=2, dtype="f32", act="mish"),
]


@pytest.mark.parametrize("spec", DIRECT_PT2, ids=lambda s: s.name)
def test_direct_two_pixels_a_thread(spec):
    plan = check(spec, "direct", "direct")
    assert "px/thread=2" in plan.describe(), plan.describe()


def test_pointwise_paths_agree():
    """A 1x1 layer through the tcgen05 GEMM and through the direct kernel."""
    spec = L("pw_both", 1, 20, 20, 128, 64, 1, 1)
    g = torch.Generator("cpu").manual_seed(5)
    d = make_layer(spec, g)
    y_ig, p1 = run_gpu(spec, d, "igemm")
    y_di, p2 = run_gpu(spec, d, "direct")
    assert p1.algo == "igemm" and p2.algo == "direct"
    ref = run_oracle(spec, d)
    assert_close(spec, y_ig, ref, "igemm")
    assert_close(spec, y_di, ref, "direct")


def test_int8_depthwise_equals_direct_bitwise():
    spec = L("dw_i8_both", 1, 21, 19, 32, 32, 3, 3, 1, 1, 1, groups=32, dtype="i8")
    g = torch.Generator("cpu").manual_seed(6)
    d = make_layer(spec, g)
    y1, _ = run_gpu(spec, d, "depthwise")
    y2, _ = run_gpu(spec, d, "direct")
    assert torch.equal(y1, y2)


# ------------------------------------------------ the five layer sets, full size

def _check_full(cfg, name, full=True, npoints=3000):
    (d,) = generate(cfg, [name])
    spec = d.spec
    y, plan = run_gpu(spec, d)
    if full:
        ref = run_oracle(spec, d)
        assert_close(spec, y, ref, f"{cfg}/{name} [{plan.describe()}]")
    else:
        pts = sample_points(spec, npoints, seed=zlib.crc32(name.encode()))
        ref = run_oracle_points(spec, d, pts)
        got = y[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
        assert_close(spec, got, ref, f"{cfg}/{name} sampled [{plan.describe()}]")
    return plan


SMALL_CFGS = [(c, s.name) for c in ("mnist_conv3x3_f32", "kws_dscnn_f32", "vww_int8") for s in CONFIGS[c]]


@pytest.mark.parametrize("cfg,name", SMALL_CFGS, ids=[n for _, n in SMALL_CFGS])
def test_layer_sets_small_full_output(cfg, name):
    _check_full(cfg, name, full=True)


BIG_CFGS = [(c, s.name) for c in ("yolov4_m640_bf16", "sweep_b8_bf16") for s in CONFIGS[c]]


@pytest.mark.parametrize("cfg,name", BIG_CFGS, ids=[n for _, n in BIG_CFGS])
def test_layer_sets_large_full_output(cfg, name):
    # every element of the output against the oracle (a few seconds of
    # oracle time per layer on the host's cores)
    plan = _check_full(cfg, name, full=True)
    spec = next(s for s in CONFIGS[cfg] if s.name == name)
    if spec.groups == 1 and spec.cin % 16 == 0:
        assert plan.algo == "igemm"


def test_kws_chain_fp32():
    """Stem -> 4 x (dw, pw), each layer fed the previous GPU output; the
    oracle runs the same chain on its own outputs."""
    layers = generate("kws_dscnn_f32")
    x_gpu = layers[0].x
    x_ref = layers[0].x.double().numpy()
    for d in layers:
        d.x = x_gpu
        y, _ = run_gpu(d.spec, d)
        import oracle
        ref = oracle.conv_f64(x_ref, d.w.double().numpy(), d.b.double().numpy(), d.spec.stride,
                              d.spec.pad_h, d.spec.pad_w, d.spec.groups, d.spec.act)
        assert_close(d.spec, y, ref, f"chain {d.spec.name}")
        x_gpu, x_ref = y, ref


def test_vww_chain_int8_exact():
    layers = generate("vww_int8")
    x = layers[0].x
    for d in layers:
        d.x = x
        y, _ = run_gpu(d.spec, d)
        assert_close(d.spec, y, run_oracle(d.spec, d), f"chain {d.spec.name}")
        x = y


# ------------------------------------------------ boundary checks at run time

def _small_plan():
    spec = L("edge", 1, 8, 8, 64, 64, 3, 3, 1, 1, 1)
    d = make_layer(spec, torch.Generator("cpu").manual_seed(1))
    return spec, d, make_plan(spec, d)


def test_empty_batch_is_a_no_op():
    import convolution_nhwc_implicit_gb300 as cl
    for dtype, cin in (("bf16", 64), ("f32", 8), ("i8", 32)):
        quant = (0.05, 0.05, [0.01] * 16) if dtype == "i8" else None
        p = cl.Plan(0, 8, 8, cin, 16, 3, 3, 1, 1, 1, 1, dtype, "relu" if dtype == "i8" else "mish", quant)
        assert p.output_shape == (0, 8, 8, 16)
        p.run(None, None, None, None)
        p.check_device_status()


def test_misaligned_aliasing_null():
    import convolution_nhwc_implicit_gb300 as cl
    spec, d, plan = _small_plan()
    dev = torch.device("cuda:0")
    x, w, b = d.x.to(dev), d.w.to(dev), d.b.to(dev)
    y = torch.empty(plan.output_shape, dtype=torch.bfloat16, device=dev)
    big = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device=dev)
    xm = big[1:1 + x.numel()].view_as(x)  # 2-byte offset
    with pytest.raises(cl.ConvError) as e:
        plan.run(xm, w, b, y)
    assert e.value.code == -4
    with pytest.raises(cl.ConvError) as e:
        plan.run(x, w, b, x)  # y aliases x
    assert e.value.code == -5
    with pytest.raises(cl.ConvError) as e:
        plan.run(None, w, b, y)
    assert e.value.code == -1
    plan.run(x, w, b, y)
    plan.check_device_status()


def test_bias_optional_everywhere():
    for algo, spec in (("igemm", L("nb_ig", 1, 9, 9, 64, 64, 3, 3, 1, 1, 1, b_dist=None)),
                       ("depthwise", L("nb_dw", 1, 9, 9, 64, 64, 3, 3, 1, 1, 1, groups=64, b_dist=None)),
                       ("direct", L("nb_di", 1, 9, 9, 8, 8, 3, 3, 1, 1, 1, dtype="f32", b_dist=None))):
        check(spec, algo, algo)


def test_repeated_runs_are_deterministic():
    spec = L("det", 2, 16, 16, 64, 128, 3, 3, 1, 1, 1)
    g = torch.Generator("cpu").manual_seed(9)
    d = make_layer(spec, g)
    plan = make_plan(spec, d)
    y1, _ = run_gpu(spec, d, plan=plan)
    y2, _ = run_gpu(spec, d, plan=plan)
    assert torch.equal(y1, y2)


# The swapped layout's two write-outs: TMA tensor stores from swizzled staging
# (plain bf16 layers whose tile width is a multiple of 16, and flat tiles:
# "out_bufs=2") and the staged transpose written by the threads (other
# widths, int8, output options: "out_bufs=1").  Ragged widths and heights put
# part of the last tiles outside the image (clipped stores).
SWAP_WRITE_OUT = [
    (L("swap_tma_ragged", 2, 21, 45, 64, 128, 3, 3, 1, 1, 1), "out_bufs=2"),
    (L("swap_tma_cout64", 1, 17, 33, 32, 64, 3, 3, 1, 1, 1, act="relu"), "out_bufs=2"),
    (L("swap_tma_flat", 2, 15, 17, 64, 96, 1, 1, act="none"), "out_bufs=2"),
    (L("swap_staged_w8", 3, 19, 8, 64, 128, 3, 3, 1, 1, 1), "out_bufs=1"),
    (L("swap_staged_i8", 1, 21, 45, 64, 64, 3, 3, 1, 1, 1, dtype="i8"), "out_bufs=1"),
]


@pytest.mark.parametrize("spec,want", SWAP_WRITE_OUT, ids=[s.name for s, _ in SWAP_WRITE_OUT])
def test_swapped_write_out_paths(spec, want):
    plan = check(spec, "igemm_swapped", "igemm")
    assert "swapped" in plan.describe() and want in plan.describe(), plan.describe()
