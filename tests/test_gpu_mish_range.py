"""GPU parity of Mish far from the origin.

Mish(v) = v * tanh(ln(1 + e^v)) ("YOLOv4, optimized for Wormhole", section 7)
tends to v for large v and to v * e^v (a vanishing negative number) for
v << 0.  The kernels evaluate it through e^v ("YOLOv4, optimized for
Wormhole", section 9, K1: x - 2x / ((1 + e^x)^2 + 1)), whose intermediate
values overflow to +inf above v ~ 44 and underflow to 0 below v ~ -87 in
fp32.  These layers scale the weights so that the pre-activations reach
about +-150, and check every kernel family's Mish against the oracle there
(bf16: |err| <= 1e-2 (1 + |ref|); fp32: 1e-5 (1 + |ref|)).
"""
import numpy as np
import pytest
import torch

import oracle
from conv_workloads import LayerSpec, make_layer
from parity_util import assert_close, run_gpu, run_oracle, to_np64

pytestmark = pytest.mark.gpu


def S(name, n, h, w, cin, cout, k, s=1, p=1, groups=1, dtype="bf16", w_std=3.0, b_std=5.0):
    w_dist = ("he",) if w_std is None else ("normal", w_std)
    return LayerSpec(name, n, h, w, cin, cout, k, k, s, p, p, groups, dtype=dtype, act="mish",
                     x_dist=("uniform", -1.0, 1.0), w_dist=w_dist, b_dist=("normal", b_std))


# fp32 layers reach the far ends through the bias instead of the weights: a
# sum of large products that cancels to a small value carries fp32 rounding
# error beyond 1e-5 (1 + |ref|) in any summation order, which is not what is
# checked here.


CASES = [
    (S("mish_far_3x3_64to64", 1, 21, 19, 64, 64, 3), "igemm"),
    (S("mish_far_3x3_64to64_swapped", 1, 21, 19, 64, 64, 3), "igemm_swapped"),
    (S("mish_far_3x3_64to64_ept", 1, 21, 19, 64, 64, 3), "igemm_n64+ept"),
    (S("mish_far_3x3_64to256_pair", 1, 12, 12, 64, 256, 3), "igemm_pair"),
    (S("mish_far_1x1_128to128", 2, 15, 15, 128, 128, 1, p=0, w_std=6.0), "igemm"),
    (S("mish_far_stem_cin3", 1, 37, 48, 3, 32, 3, w_std=40.0), "igemm"),
    (S("mish_far_dw_rows", 1, 17, 12, 64, 64, 3, groups=64, w_std=50.0), "depthwise"),
    (S("mish_far_dw_s2", 1, 17, 12, 64, 64, 3, s=2, groups=64, w_std=50.0), "depthwise"),
    (S("mish_far_dw_f32", 1, 17, 12, 64, 64, 3, groups=64, dtype="f32", w_std=None, b_std=90.0), "depthwise"),
    (S("mish_far_direct_f32", 1, 28, 28, 8, 32, 3, dtype="f32", w_std=None, b_std=90.0), "direct"),
    (S("mish_far_direct_bf16", 1, 10, 10, 16, 32, 3, groups=2, w_std=25.0), "direct"),
]


@pytest.mark.parametrize("spec,algo", CASES, ids=[s.name for s, _ in CASES])
def test_mish_at_large_magnitudes(spec, algo):
    d = make_layer(spec, torch.Generator("cpu").manual_seed(12))
    pre = oracle.conv_f64(to_np64(d.x), to_np64(d.w), to_np64(d.b), spec.stride, spec.pad_h, spec.pad_w,
                          spec.groups, "none")
    # the layer reaches both the overflow side and the far negative side
    assert (pre > 50).sum() > 0 and (pre < -90).sum() > 0, (pre.min(), pre.max())
    y, plan = run_gpu(spec, d, algo)
    assert plan.algo == algo.split("_")[0].split("+")[0], plan.describe()
    ref = run_oracle(spec, d)
    assert_close(spec, y, ref, f"{spec.name} [{plan.describe()}]")
    assert np.isfinite(y.to(torch.float64).numpy()).all()
