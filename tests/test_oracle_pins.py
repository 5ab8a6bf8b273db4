"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-worked cases, closed forms, invariants, and special cases that reduce to
library routines (numpy matmul, torch conv2d / mish in float64).

Each pin is chosen so that a plausible slip in the oracle fails it: a flipped
kernel (correlation vs convolution), swapped pad axes, a dropped bias, a wrong
group offset, a transposed weight, truncation instead of round-half-to-even,
a missing saturation.
"""
import math
import os
import zlib

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _img3x3():
    return np.arange(1, 10, dtype=np.float64).reshape(1, 3, 3, 1)


# ---------------------------------------------------------------- hand cases

def test_hand_case_ones_3x3():
    rows = {r[0]: [float(v) for v in r[1:]] for r in _read_rows("ones3x3_pad1.txt")}
    x = np.array(rows["input"]).reshape(1, 3, 3, 1)
    w = np.ones((1, 3, 3, 1))
    y1 = oracle.conv_f64(x, w, None, stride=1, pad_h=1, pad_w=1)
    assert y1.shape == (1, 3, 3, 1)
    np.testing.assert_array_equal(y1.ravel(), rows["stride1"])
    y2 = oracle.conv_f64(x, w, None, stride=2, pad_h=1, pad_w=1)
    assert y2.shape == (1, 2, 2, 1)
    np.testing.assert_array_equal(y2.ravel(), rows["stride2"])


def test_hand_case_ones_3x3_int8():
    rows = {r[0]: [int(v) for v in r[1:]] for r in _read_rows("ones3x3_pad1.txt")}
    x = np.array(rows["input"], dtype=np.int8).reshape(1, 3, 3, 1)
    w = np.ones((1, 3, 3, 1), dtype=np.int8)
    acc = oracle.conv_i8_acc(x, w, stride=1, pad_h=1, pad_w=1)
    np.testing.assert_array_equal(acc.ravel(), rows["stride1"])
    # s_x = s_y and s_w = 1 give M = 1: requantised output = accumulator.
    M = oracle.requant_multipliers(0.05, 0.05, [1.0])
    assert M[0] == np.float32(1.0)
    y = oracle.conv_i8(x, w, None, M, stride=2, pad_h=1, pad_w=1)
    np.testing.assert_array_equal(y.ravel(), rows["stride2"])


def test_hand_case_asymmetric_kernels_and_pads():
    rows = {r[0]: [float(v) for v in r[1:]] for r in _read_rows("asym_kernels.txt")}
    x = np.array(rows["input"]).reshape(1, 3, 3, 1)
    y = oracle.conv_f64(x, np.ones((1, 3, 1, 1)), None, stride=1, pad_h=1, pad_w=0)
    np.testing.assert_array_equal(y.ravel(), rows["k3x1_pad1_0"])
    y = oracle.conv_f64(x, np.ones((1, 1, 3, 1)), None, stride=1, pad_h=0, pad_w=1)
    np.testing.assert_array_equal(y.ravel(), rows["k1x3_pad0_1"])


def test_correlation_not_convolution():
    # A kernel with a single 1 at its top-left tap picks the pixel up-left of
    # the centre (cross-correlation); a flipped kernel would pick down-right.
    x = _img3x3()
    w = np.zeros((1, 3, 3, 1))
    w[0, 0, 0, 0] = 1.0
    y = oracle.conv_f64(x, w, None, stride=1, pad_h=1, pad_w=1)
    assert y[0, 1, 1, 0] == 1.0 and y[0, 2, 2, 0] == 5.0 and y[0, 0, 0, 0] == 0.0


def test_bias_and_relu_closed_form():
    x = _img3x3()
    w = -np.ones((1, 1, 1, 1))
    y = oracle.conv_f64(x, w, np.array([4.5]), act="relu")
    np.testing.assert_array_equal(y.ravel(), np.maximum(4.5 - np.arange(1, 10), 0.0))
    y = oracle.conv_f64(x, w, np.array([4.5]), act="none")
    np.testing.assert_array_equal(y.ravel(), 4.5 - np.arange(1, 10))


# ---------------------------------------------------------------- shape rule

def test_shape_rule_table():
    for r in _read_rows("shape_rule.txt"):
        H, W, kh, kw, s, ph, pw, OH, OW = map(int, r)
        assert oracle.output_shape(H, W, kh, kw, s, ph, pw) == (OH, OW), r


def test_kws_stem_shape_and_values_against_torch():
    # The keyword-spotting stem: 49x10x1 -> 64, 10x4 kernel, stride 2, pad (5, 1).
    rng = np.random.default_rng(11)
    x = rng.uniform(-1, 1, (1, 49, 10, 1))
    w = rng.normal(0, 0.2, (64, 10, 4, 1))
    b = rng.normal(0, 0.01, 64)
    y = oracle.conv_f64(x, w, b, stride=2, pad_h=5, pad_w=1, act="relu")
    assert y.shape == (1, 25, 5, 64)
    ref = F.relu(F.conv2d(torch.from_numpy(x).permute(0, 3, 1, 2),
                          torch.from_numpy(w).permute(0, 3, 1, 2),
                          torch.from_numpy(b), stride=2, padding=(5, 1)))
    np.testing.assert_allclose(y, ref.permute(0, 2, 3, 1).numpy(), rtol=0, atol=1e-12)
    # Swapping the pad axes (the exporter bug) changes the shape here; with the
    # pads (5, 5) that bug produced, values differ at matching positions.
    bug = oracle.conv_f64(x, w, b, stride=2, pad_h=5, pad_w=5, act="relu")
    assert bug.shape != y.shape or not np.allclose(bug, y)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("k", [1, 3, 5])
@pytest.mark.parametrize("stride", [1, 2])
def test_identity_kernel(k, stride):
    rng = np.random.default_rng(k * 10 + stride)
    C = 5
    x = rng.normal(size=(2, 7, 6, C))
    w = np.zeros((C, k, k, C))
    for c in range(C):
        w[c, k // 2, k // 2, c] = 1.0
    y = oracle.conv_f64(x, w, None, stride=stride, pad_h=k // 2, pad_w=k // 2)
    np.testing.assert_array_equal(y, x[:, ::stride, ::stride, :])
    ym = oracle.conv_f64(x, w, None, stride=stride, pad_h=k // 2, pad_w=k // 2, act="mish")
    expect = np.vectorize(lambda v: v * math.tanh(math.log1p(math.exp(v))))(x[:, ::stride, ::stride, :])
    np.testing.assert_allclose(ym, expect, rtol=1e-14, atol=1e-300)


def test_identity_kernel_depthwise_and_int8():
    rng = np.random.default_rng(3)
    C = 6
    x = rng.integers(-128, 128, size=(1, 5, 4, C)).astype(np.int8)
    w = np.zeros((C, 3, 3, 1), dtype=np.int8)
    w[:, 1, 1, 0] = 1
    acc = oracle.conv_i8_acc(x, w, stride=1, pad_h=1, pad_w=1, groups=C)
    np.testing.assert_array_equal(acc, x.astype(np.int64))
    M = oracle.requant_multipliers(0.05, 0.05, np.ones(C, dtype=np.float32))
    y = oracle.conv_i8(x, w, None, M, stride=1, pad_h=1, pad_w=1, groups=C)
    np.testing.assert_array_equal(y, x)


def test_pointwise_is_gemm():
    # A 1x1, stride-1, unpadded convolution is a GEMM on the input viewed as
    # [N*H*W, Cin] ("nanoinfer", "1x1 convolutions are already a GEMM").
    rng = np.random.default_rng(5)
    x = rng.normal(size=(2, 4, 5, 7))
    w = rng.normal(size=(3, 1, 1, 7))
    b = rng.normal(size=3)
    y = oracle.conv_f64(x, w, b)
    gemm = x.reshape(-1, 7) @ w.reshape(3, 7).T + b
    np.testing.assert_allclose(y.reshape(-1, 3), gemm, rtol=1e-13, atol=1e-13)


def test_pointwise_is_gemm_int8_exact():
    rng = np.random.default_rng(6)
    x = rng.integers(-128, 128, size=(1, 6, 6, 32)).astype(np.int8)
    w = rng.integers(-127, 128, size=(16, 1, 1, 32)).astype(np.int8)
    acc = oracle.conv_i8_acc(x, w)
    gemm = x.reshape(-1, 32).astype(np.int64) @ w.reshape(16, 32).astype(np.int64).T
    np.testing.assert_array_equal(acc.reshape(-1, 16), gemm)


def test_linearity_int8_exact():
    rng = np.random.default_rng(7)
    x = rng.integers(-128, 128, size=(1, 6, 5, 8)).astype(np.int8)
    w1 = rng.integers(-60, 60, size=(4, 3, 3, 8)).astype(np.int8)
    w2 = rng.integers(-60, 60, size=(4, 3, 3, 8)).astype(np.int8)
    a1 = oracle.conv_i8_acc(x, w1, stride=1, pad_h=1, pad_w=1)
    a2 = oracle.conv_i8_acc(x, w2, stride=1, pad_h=1, pad_w=1)
    a12 = oracle.conv_i8_acc(x, (w1.astype(np.int16) + w2).astype(np.int8), stride=1,
                             pad_h=1, pad_w=1)
    np.testing.assert_array_equal(a12, a1 + a2)


def test_translation_equivariance_interior():
    rng = np.random.default_rng(8)
    x = rng.integers(-128, 128, size=(1, 9, 9, 3)).astype(np.int8)
    w = rng.integers(-127, 128, size=(2, 3, 3, 3)).astype(np.int8)
    a = oracle.conv_i8_acc(x, w, pad_h=1, pad_w=1)
    xs = np.roll(x, shift=(2, 1), axis=(1, 2))
    as_ = oracle.conv_i8_acc(xs, w, pad_h=1, pad_w=1)
    # interior outputs (away from the wrapped border) shift with the input
    np.testing.assert_array_equal(as_[:, 3:8, 2:8], a[:, 1:6, 1:7])


# ------------------------------------------------------- library special case

CASES = [
    # (N, H, W, Cin, Cout, kh, kw, stride, pad_h, pad_w, groups)
    (1, 7, 6, 3, 4, 3, 3, 1, 1, 1, 1),
    (2, 9, 8, 4, 6, 3, 3, 2, 1, 1, 1),
    (1, 11, 7, 1, 5, 10, 4, 2, 5, 1, 1),
    (1, 6, 6, 8, 8, 3, 3, 1, 1, 1, 8),     # depthwise
    (1, 7, 5, 6, 6, 3, 3, 2, 0, 2, 6),     # depthwise, stride 2, asymmetric pad
    (2, 5, 5, 4, 6, 3, 3, 1, 1, 1, 2),     # grouped
    (1, 5, 9, 5, 3, 1, 1, 1, 0, 0, 1),     # pointwise
    (1, 8, 8, 2, 3, 2, 5, 3, 0, 2, 1),     # even/asymmetric kernel, stride 3
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("act", ["none", "relu", "mish"])
def test_oracle_vs_torch_conv2d_f64(case, act):
    N, H, W, Cin, Cout, kh, kw, s, ph, pw, g = case
    rng = np.random.default_rng(zlib.crc32(repr((case, act)).encode()))
    x = rng.normal(size=(N, H, W, Cin))
    w = rng.normal(size=(Cout, kh, kw, Cin // g))
    b = rng.normal(size=Cout)
    y = oracle.conv_f64(x, w, b, stride=s, pad_h=ph, pad_w=pw, groups=g, act=act)
    t = F.conv2d(torch.from_numpy(x).permute(0, 3, 1, 2), torch.from_numpy(w).permute(0, 3, 1, 2),
                 torch.from_numpy(b), stride=s, padding=(ph, pw), groups=g)
    if act == "relu":
        t = F.relu(t)
    elif act == "mish":
        t = F.mish(t)
    np.testing.assert_allclose(y, t.permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", CASES)
def test_oracle_int8_acc_vs_torch_conv2d_exact(case):
    N, H, W, Cin, Cout, kh, kw, s, ph, pw, g = case
    rng = np.random.default_rng(1234 + sum(case))
    x = rng.integers(-128, 128, size=(N, H, W, Cin)).astype(np.int8)
    w = rng.integers(-127, 128, size=(Cout, kh, kw, Cin // g)).astype(np.int8)
    acc = oracle.conv_i8_acc(x, w, stride=s, pad_h=ph, pad_w=pw, groups=g)
    t = F.conv2d(torch.from_numpy(x.astype(np.float64)).permute(0, 3, 1, 2),
                 torch.from_numpy(w.astype(np.float64)).permute(0, 3, 1, 2),
                 None, stride=s, padding=(ph, pw), groups=g)
    # |acc| << 2**53: the float64 library result is exact.
    np.testing.assert_array_equal(acc, t.permute(0, 2, 3, 1).numpy().astype(np.int64))


def test_points_match_full():
    rng = np.random.default_rng(9)
    x = rng.normal(size=(2, 8, 7, 6))
    w = rng.normal(size=(4, 3, 3, 3))
    b = rng.normal(size=4)
    y = oracle.conv_f64(x, w, b, stride=2, pad_h=1, pad_w=0, groups=2, act="mish")
    pts = np.array([[n, h, ww, c] for n in range(2) for h in range(y.shape[1])
                    for ww in range(y.shape[2]) for c in range(4)])
    v = oracle.conv_f64_points(x, w, b, pts, stride=2, pad_h=1, pad_w=0, groups=2, act="mish")
    np.testing.assert_array_equal(v, y.reshape(-1))
    xi = rng.integers(-128, 128, size=(1, 6, 6, 4)).astype(np.int8)
    wi = rng.integers(-127, 128, size=(5, 3, 3, 4)).astype(np.int8)
    bi = rng.integers(-1000, 1001, size=5).astype(np.int32)
    M = oracle.requant_multipliers(0.05, 0.05, rng.uniform(0.001, 0.01, 5).astype(np.float32))
    yi = oracle.conv_i8(xi, wi, bi, M, pad_h=1, pad_w=1, relu=True)
    pts = np.array([[0, h, ww, c] for h in range(6) for ww in range(6) for c in range(5)])
    vi = oracle.conv_i8_points(xi, wi, bi, M, pts, pad_h=1, pad_w=1, relu=True)
    np.testing.assert_array_equal(vi, yi.reshape(-1))


# ---------------------------------------------------------------------- Mish

def test_mish_special_values_and_library():
    assert oracle.mish(0.0) == 0.0
    assert oracle.mish(60.0) == 60.0                   # tanh(softplus(60)) == 1 in double
    assert abs(oracle.mish(-60.0)) < 1e-20             # ~ x * e^x
    grid = np.linspace(-30, 30, 2001)
    ours = np.array([oracle.mish(v) for v in grid])
    lib = F.mish(torch.from_numpy(grid)).numpy()
    np.testing.assert_allclose(ours, lib, rtol=1e-14, atol=1e-300)
    # The algebraic form used by the Wormhole kernel: x - 2x / ((1 + e^x)^2 + 1)
    alg = np.array([v - 2 * v / ((1 + math.exp(v)) ** 2 + 1) for v in grid])
    mask = np.abs(grid) < 15   # the algebraic form cancels badly for x << 0
    np.testing.assert_allclose(ours[mask], alg[mask], rtol=1e-12, atol=1e-13)
    # Mish is not HardMish: x * clamp(x + 2, 0, 2) / 2 differs at x = -1.
    hard = -1 * min(max(-1 + 2, 0), 2) / 2
    assert abs(oracle.mish(-1.0) - hard) > 0.1


def test_mish_min_value():
    # Mish has its minimum near x = -1.1924 with value about -0.30884.
    grid = np.linspace(-2, 0, 20001)
    vals = np.array([oracle.mish(v) for v in grid])
    assert abs(grid[vals.argmin()] + 1.1924) < 1e-3
    assert abs(vals.min() + 0.30884) < 1e-4


# ------------------------------------------------------------------ requant

def test_requant_tie_table():
    M = oracle.requant_multipliers(0.05, 0.05, [0.5])
    assert M[0] == np.float32(0.5)
    for v, q, qr in (map(int, r) for r in _read_rows("requant_ties.txt")):
        assert oracle.requant_one(v, M[0], relu=False) == q, v
        assert oracle.requant_one(v, M[0], relu=True) == qr, v


def test_requant_scale_ratio_hand_cases():
    # s_x != s_y: the multiplier is s_x * s_w / s_y, not s_w alone and not its
    # reciprocal ratio; values worked by hand in the golden file.
    rows = _read_rows("requant_scales.txt")
    for _, sx, sy, sw, m in (r for r in rows if r[0] == "mult"):
        M = oracle.requant_multipliers(float(sx), float(sy), [float(sw)])
        assert M[0] == np.float32(float(m)), (sx, sy, sw)
    for _, sx, sy, sw, v, q in (r for r in rows if r[0] == "q"):
        M = oracle.requant_multipliers(float(sx), float(sy), [float(sw)])
        assert oracle.requant_one(int(v), M[0]) == int(q), (sx, sy, sw, v)


def test_requant_scale_ratio_whole_layer():
    rows = {r[0]: [int(v) for v in r[1:]] for r in _read_rows("requant_scales.txt") if r[0].startswith("conv")}
    x = np.arange(1, 10, dtype=np.int8).reshape(1, 3, 3, 1)
    w = np.ones((2, 3, 3, 1), dtype=np.int8)
    M = oracle.requant_multipliers(0.1, 0.05, [0.25, 0.125])
    y = oracle.conv_i8(x, w, np.array([1, 0], dtype=np.int32), M, stride=1, pad_h=1, pad_w=1)
    np.testing.assert_array_equal(y[..., 0].ravel(), rows["conv_ch0"])
    np.testing.assert_array_equal(y[..., 1].ravel(), rows["conv_ch1"])
    pts = np.array([[0, h, w_, c] for h in range(3) for w_ in range(3) for c in range(2)], dtype=np.int32)
    vals = oracle.conv_i8_points(x, w, np.array([1, 0], dtype=np.int32), M, pts, 1, 1, 1)
    np.testing.assert_array_equal(vals, y[0, pts[:, 1], pts[:, 2], pts[:, 3]])


def test_requant_float_rounding_of_accumulator():
    # Above 2**24 the accumulator is first rounded to float (ties to even):
    # 2**24 + 1 -> 2**24, and 2**24 + 3 -> 2**24 + 4.  With M = 2**-17 these
    # give 128 and 128.00003 before saturation; use M = 2**-18 to stay in range.
    M = np.float32(2.0 ** -18)
    assert oracle.requant_one(2**24 + 1, M) == 64          # 2**24 * 2**-18
    assert oracle.requant_one(2**24 + 3, M) == 64          # 64.0000153 -> 64
    # A tie after the multiply rounds to even: 64.5 -> 64 and 65.5 -> 66.
    assert oracle.requant_one(2**25 + 2**18, np.float32(2.0 ** -19)) == 64
    assert oracle.requant_one(2**25 + 3 * 2**18, np.float32(2.0 ** -19)) == 66


def test_requant_against_numpy_float32():
    # numpy float32 arithmetic is IEEE single precision with round-half-even.
    rng = np.random.default_rng(10)
    ws = rng.uniform(0.001, 0.01, 64).astype(np.float32)
    M = oracle.requant_multipliers(0.05, 0.05, ws)
    expect_M = (np.float64(np.float32(0.05)) * ws.astype(np.float64) / np.float64(np.float32(0.05))).astype(np.float32)
    np.testing.assert_array_equal(M, expect_M)
    vs = rng.integers(-3_000_000, 3_000_000, 500)
    for v in vs:
        for co in (0, 17, 63):
            p = np.float32(np.float32(v) * M[co])
            q = int(np.clip(np.rint(p), -128, 127))
            assert oracle.requant_one(int(v), M[co]) == q


def test_requant_is_monotone_so_relu_commutes():
    M = np.float32(0.0371)
    prev = -1000
    for v in range(-5000, 5000, 7):
        q = oracle.requant_one(v, M)
        assert q >= prev
        prev = q
        assert oracle.requant_one(v, M, relu=True) == max(q, 0)


# ------------------------------------------------------------ argument checks

def test_oracle_rejects_bad_shapes():
    x = np.zeros((1, 3, 3, 4))
    with pytest.raises(ValueError):
        oracle.conv_f64(x, np.zeros((4, 3, 3, 3)), None)           # channels/groups mismatch
    with pytest.raises(ValueError):
        oracle.conv_f64(x, np.zeros((4, 5, 5, 4)), None)           # no output fits
    with pytest.raises(ValueError):
        oracle.requant_multipliers(0.05, 0.0, [1.0])


# ---------------------------------------------------------------- K2 / K4 options

def test_residual_is_added_after_the_activation():
    # 1..9 with an all-ones 3x3 kernel, pad 1 (the hand-worked golden case):
    # [[12,21,16],[27,45,33],[24,39,28]]; bias -20, ReLU, residual -1.
    x = np.arange(1, 10, dtype=np.float64).reshape(1, 3, 3, 1)
    w = np.ones((1, 3, 3, 1))
    b = np.array([-20.0])
    r = np.full((1, 3, 3, 1), -1.0)
    y = oracle.conv_residual_f64(x, w, b, r, 1, 1, 1, 1, "relu")
    want = np.array([[-1, 0, -1], [6, 24, 12], [3, 18, 7]], dtype=np.float64)
    assert np.array_equal(y[0, :, :, 0], want)
    # ... which is not relu(conv + b + r): the order of the two steps shows
    assert not np.array_equal(y, oracle.conv_f64(x, w, b - 1.0, 1, 1, 1, 1, "relu"))


def test_residual_with_mish_matches_the_definition():
    rng = np.random.default_rng(7)
    x = rng.uniform(-1, 1, (1, 5, 4, 3))
    w = rng.normal(0, 0.5, (4, 3, 3, 3))
    r = rng.normal(0, 1, (1, 5, 4, 4))
    y = oracle.conv_residual_f64(x, w, None, r, 1, 1, 1, 1, "mish")
    v = oracle.conv_f64(x, w, None, 1, 1, 1, 1, "none")
    ref = v * np.tanh(np.log1p(np.exp(v))) + r
    assert np.allclose(y, ref, rtol=0, atol=1e-13)


def test_place_output_concat_and_upsample():
    y = np.array([[[[1.0], [2.0]]]])  # 1 x 1 x 2 x 1
    out = oracle.place_output(y, y_channels=3, y_channel_offset=1, upsample=2, fill=-9.0)
    assert out.shape == (1, 2, 4, 3)
    assert np.array_equal(out[0, :, :, 1], [[1, 1, 2, 2], [1, 1, 2, 2]])
    assert np.all(out[..., 0] == -9.0) and np.all(out[..., 2] == -9.0)
    # no upsampling, no offset: the output itself
    z = np.arange(24.0).reshape(1, 2, 3, 4)
    assert np.array_equal(oracle.place_output(z, 4), z)


# ---------------------------------------------------------------- SPP max pools (K3)

def _maxpool_numpy(x, k):
    # independent restatement: pad with -inf and take the max of all k*k shifts
    r = k // 2
    N, H, W, C = x.shape
    p = np.full((N, H + 2 * r, W + 2 * r, C), -np.inf)
    p[:, r:r + H, r:r + W] = x
    out = np.full(x.shape, -np.inf)
    for i in range(k):
        for j in range(k):
            out = np.maximum(out, p[:, i:i + H, j:j + W])
    return out


@pytest.mark.parametrize("k", [1, 3, 5, 9, 13])
def test_maxpool_same_matches_shifted_maximum(k):
    rng = np.random.default_rng(k)
    x = rng.normal(0, 1, (2, 7, 11, 3))
    assert np.array_equal(oracle.maxpool_same(x, k), _maxpool_numpy(x, k))


def test_maxpool_same_hand_case_and_negative_edges():
    # 1 x 3 x 3, all values negative: padding must never win the max
    x = -np.arange(1, 10, dtype=np.float64).reshape(1, 3, 3, 1)
    y = oracle.maxpool_same(x, 3)[0, :, :, 0]
    assert np.array_equal(y, [[-1, -1, -2], [-1, -1, -2], [-4, -4, -5]])
    # a window wider than the image covers it all
    assert np.all(oracle.maxpool_same(x, 13) == -1)


def test_spp_cascade_identity_holds_for_the_oracle():
    # mp9 = mp5(mp5), mp13 = mp5(mp5(mp5)): the identity the fast kernel uses
    rng = np.random.default_rng(3)
    x = rng.integers(-128, 128, (1, 12, 9, 4)).astype(np.float64)
    p5, p9, p13 = oracle.spp(x)
    assert np.array_equal(p9, oracle.maxpool_same(p5, 5))
    assert np.array_equal(p13, oracle.maxpool_same(p9, 5))


# ---------------------------------------------------------------- fused dw -> pw pair

def test_dwpw_pair_matches_torch_depthwise_then_pointwise():
    import torch.nn.functional as F
    rng = np.random.default_rng(9)
    x = rng.uniform(-1, 1, (2, 9, 7, 8))
    wd = rng.normal(0, 0.5, (8, 3, 3, 1))
    bd = rng.normal(0, 0.1, 8)
    wp = rng.normal(0, 0.3, (5, 1, 1, 8))
    bp = rng.normal(0, 0.1, 5)
    for stride in (1, 2):
        y = oracle.dwpw_f64(x, wd, bd, wp, bp, stride, 1, "relu", "mish")
        t = torch.from_numpy(x).permute(0, 3, 1, 2)
        z = F.relu(F.conv2d(t, torch.from_numpy(wd).permute(0, 3, 1, 2), torch.from_numpy(bd), stride, 1,
                            groups=8))
        r = F.mish(F.conv2d(z, torch.from_numpy(wp).permute(0, 3, 1, 2), torch.from_numpy(bp)))
        assert np.allclose(y, r.permute(0, 2, 3, 1).numpy(), rtol=0, atol=1e-12)
