"""GPU parity of the int8 requantisation: an input scale s_x different from
the output scale s_y, and exact round-half-to-even ties.

Symmetric per-output-channel scales with no zero point ("nanoinfer",
post-training quantization) give the multiplier M[co] = s_x * s_w[co] / s_y;
the output is saturate(round_half_to_even(float(acc + b) * M[co])).  Two
families of layers exercise it on every int8 kernel path, each compared bit
for bit with the oracle:

* tie layers: small integer data and power-of-two scales (s_x = 1/8,
  s_y = 1/2, s_w = 2^e for e in [-2, 1], so M in {1/16, 1/8, 1/4, 1/2}),
  which put a large share of the products exactly on .5 -- both the ties
  that round down to even and those that round up -- plus saturated ones;
* ratio layers: the visual-wake-words value ranges with s_x = 0.02 and
  s_y = 0.07, so that a kernel using s_w alone or the inverted ratio would
  differ almost everywhere.

Paths: the tensor-core kernel with operands widened by the pre-pass or in the
kernel, under each tile layout and epilogue split; the depthwise stencil; the
direct kernel with dp4a and with scalar products (input channels not a
multiple of 4).  The allocation-free entry point runs the same families in
tests/test_zz_no_alloc.py.
"""
import numpy as np
import pytest
import torch

import oracle
from conv_workloads import LayerSpec, make_layer
from parity_util import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

TIE = dict(dtype="i8", x_dist=("int", -3, 3), w_dist=("int", -3, 3), b_dist=("int", -40, 40),
           in_scale=0.125, out_scale=0.5, ws_dist=("pow2", -2, 1))
RATIO = dict(dtype="i8", x_dist=("int", -128, 127), w_dist=("int", -127, 127), b_dist=("int", -1000, 1000),
             in_scale=0.02, out_scale=0.07)


def S(name, n, h, w, cin, cout, kh, kw, s=1, ph=0, pw=0, groups=1, act="none", fam=TIE):
    return LayerSpec(name, n, h, w, cin, cout, kh, kw, s, ph, pw, groups, act=act, **fam)


def tie_stats(spec, d):
    """(ties rounded down, ties rounded up, saturated) among the oracle's
    products float(v) * M -- a check that a case really reaches ties."""
    acc = oracle.conv_i8_acc(d.x.numpy(), d.w.numpy(), spec.stride, spec.pad_h, spec.pad_w, spec.groups)
    v = acc + (0 if d.b is None else d.b.numpy().astype(np.int64))
    M = oracle.requant_multipliers(spec.in_scale, spec.out_scale, d.w_scales.numpy())
    p = v.astype(np.float32) * M  # IEEE single multiply, as the definition has it
    frac = p - np.floor(p)
    tie = (frac == 0.5) & (np.abs(p) < 127.5)
    fl = np.floor(p).astype(np.int64)
    down = tie & (fl % 2 == 0)
    up = tie & (fl % 2 != 0)
    sat = np.abs(p) > 127.5
    return int(down.sum()), int(up.sum()), int(sat.sum())


def check(spec, algo, seed=0, want_ties=True):
    d = make_layer(spec, torch.Generator("cpu").manual_seed(seed))
    y, plan = run_gpu(spec, d, algo)
    ref = run_oracle(spec, d)
    assert_close(spec, y, ref, f"{spec.name} [{plan.describe()}]")
    if want_ties:
        down, up, _ = tie_stats(spec, d)
        assert down > 0 and up > 0, (spec.name, down, up)
    return plan


TC_TIE = [
    S("tie_3x3_64to64", 1, 21, 19, 64, 64, 3, 3, 1, 1, 1),
    S("tie_3x3_64to48_relu", 2, 13, 11, 64, 48, 3, 3, 1, 1, 1, act="relu"),
    S("tie_1x1_32to64", 1, 24, 20, 32, 64, 1, 1),
    S("tie_3x3_s2_cin48", 1, 17, 15, 48, 32, 3, 3, 2, 1, 1),
    S("tie_1x1_k1024", 1, 8, 8, 1024, 16, 1, 1, act="relu"),
]
TC_LAYOUTS = ["igemm", "igemm_swapped", "igemm_n256", "igemm_n128", "igemm_n64", "igemm_pair", "igemm_pair128",
              "igemm_n64+halo", "igemm_n64+ept", "igemm_n128+sliced"]


def _tc_cases():
    out = []
    for spec in TC_TIE:
        for lay in TC_LAYOUTS:
            if lay == "igemm_swapped" and spec.cout > 128:
                continue
            if "halo" in lay and not (spec.stride == 1 and spec.kh == 3):
                continue
            out.append(pytest.param(spec, lay, id=f"{spec.name}-{lay}"))
        # the int8 operands widened in the kernel and by the pre-pass, forced
        if spec.cin % 16 == 0 and spec.cin <= 64:
            for w in ("inkernel", "prepass"):
                out.append(pytest.param(spec, f"igemm_n64+{w}", id=f"{spec.name}-igemm_n64+{w}"))
            if spec.stride == 1 and spec.kh == 3:
                out.append(pytest.param(spec, "igemm_n64+halo+ept+inkernel",
                                        id=f"{spec.name}-igemm_n64+halo+ept+inkernel"))
    return out


@pytest.mark.parametrize("spec,algo", _tc_cases())
def test_tensor_core_requant_ties(spec, algo):
    plan = check(spec, algo)
    assert plan.algo == "igemm", plan.describe()
    want = "i8-widened-in-kernel" if "inkernel" in algo else ("i8-as-bf16" if "prepass" in algo else None)
    if want:
        assert want in plan.describe(), plan.describe()


OTHER_TIE = [
    (S("tie_dw_48", 2, 13, 11, 48, 48, 3, 3, 1, 1, 1, groups=48), "depthwise"),
    (S("tie_dw_32_relu_s2", 1, 19, 17, 32, 32, 3, 3, 2, 1, 1, groups=32, act="relu"), "depthwise"),
    (S("tie_dw_48_direct", 2, 13, 11, 48, 48, 3, 3, 1, 1, 1, groups=48), "direct"),
    (S("tie_3x3_64to40_dp4a", 1, 17, 19, 64, 40, 3, 3, 1, 1, 1), "direct"),
    (S("tie_3x3_256to16_long_k", 1, 6, 6, 256, 16, 3, 3, 1, 1, 1), "auto"),
    (S("tie_cin3_scalar", 1, 11, 9, 3, 16, 3, 3, 2, 1, 1), "direct"),
    (S("tie_cin3_tensor_cores", 1, 18, 16, 3, 16, 3, 3, 1, 1, 1), "igemm"),
    (S("tie_grouped", 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, groups=4, act="relu"), "direct"),
]


@pytest.mark.parametrize("spec,algo", OTHER_TIE, ids=[s.name for s, _ in OTHER_TIE])
def test_stencil_and_direct_requant_ties(spec, algo):
    plan = check(spec, algo)
    if algo != "auto":
        assert plan.algo == algo, plan.describe()
    else:
        assert plan.algo == "direct" and "dp4a" in plan.describe(), plan.describe()


RATIO_CASES = [
    (S("ratio_3x3_64to64", 1, 21, 19, 64, 64, 3, 3, 1, 1, 1, fam=RATIO), "igemm+prepass"),
    (S("ratio_3x3_64to64_ik", 1, 21, 19, 64, 64, 3, 3, 1, 1, 1, fam=RATIO), "igemm_n64+inkernel"),
    (S("ratio_3x3_64to64_swapped", 1, 21, 19, 64, 64, 3, 3, 1, 1, 1, fam=RATIO), "igemm_swapped"),
    (S("ratio_1x1_32to64_relu", 1, 24, 20, 32, 64, 1, 1, act="relu", fam=RATIO), "igemm"),
    (S("ratio_dw_32", 1, 20, 18, 32, 32, 3, 3, 1, 1, 1, groups=32, fam=RATIO), "depthwise"),
    (S("ratio_3x3_dp4a", 1, 17, 19, 64, 40, 3, 3, 1, 1, 1, fam=RATIO), "direct"),
    (S("ratio_cin3_scalar", 1, 11, 9, 3, 16, 3, 3, 2, 1, 1, fam=RATIO), "direct"),
]


@pytest.mark.parametrize("spec,algo", RATIO_CASES, ids=[s.name for s, _ in RATIO_CASES])
def test_requant_scale_ratio(spec, algo):
    d = make_layer(spec, torch.Generator("cpu").manual_seed(7))
    y, plan = run_gpu(spec, d, algo)
    ref = run_oracle(spec, d)
    assert_close(spec, y, ref, f"{spec.name} [{plan.describe()}]")
    # the multiplier with s_w alone would give another result: the case
    # discriminates the ratio
    wrong = oracle.conv_i8(d.x.numpy(), d.w.numpy(), d.b.numpy(), d.w_scales.numpy(), spec.stride, spec.pad_h,
                           spec.pad_w, spec.groups, spec.act == "relu")
    assert (wrong != ref).mean() > 0.1
