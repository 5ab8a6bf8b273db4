"""GPU parity of the fused output options (conv_plan_create_fused): the
residual add after the activation ("YOLOv4, optimized for Wormhole",
section 9, K2) and the concatenated / 2x-upsampled output placement (K4),
through every kernel family and tensor-core tile layout that takes them.

Each case runs the layer into a y buffer poisoned with 0x7f bytes, compares
the layer's slice of every upsample replica with the oracle (the residual
added in float64 after the activation), and checks that nothing outside the
slice was written."""
import numpy as np
import pytest
import torch

import oracle
from conv_workloads import LayerSpec, make_layer, output_hw
from parity_util import TORCH_DT, assert_close, make_plan, run_oracle, to_np64

pytestmark = pytest.mark.gpu

GUARD = 4096


def L(name, n, h, w, cin, cout, kh, kw, s=1, ph=0, pw=0, groups=1, dtype="bf16", act="mish", **extra):
    base = dict(x_dist=("uniform", -1.0, 1.0), w_dist=("he",), b_dist=("normal", 0.5))
    if dtype == "i8":
        base = dict(x_dist=("int", -128, 127), w_dist=("int", -127, 127), b_dist=("int", -1000, 1000))
    base.update(extra)
    return LayerSpec(name, n, h, w, cin, cout, kh, kw, s, ph, pw, groups, dtype, act, **base)


def run_fused(spec, out, algo="auto", seed=0):
    import convolution_nhwc_implicit_gb300 as cl
    g = torch.Generator("cpu").manual_seed(seed)
    d = make_layer(spec, g)
    quant = (spec.in_scale, spec.out_scale, d.w_scales.tolist()) if spec.dtype == "i8" else None
    plan = cl.Plan(spec.n, spec.h, spec.w, spec.cin, spec.cout, spec.kh, spec.kw, spec.stride, spec.pad_h,
                   spec.pad_w, spec.groups, spec.dtype, spec.act, quant, algo, out=out)
    oh, ow = output_hw(spec)
    dt = TORCH_DT[spec.dtype]
    r = None
    if out.get("residual"):
        r = torch.empty(spec.n, oh, ow, spec.cout).uniform_(-2, 2, generator=g).to(dt)
    dev = torch.device("cuda:0")
    ys = plan.y_shape
    esz = torch.tensor([], dtype=dt).element_size()
    numel = int(np.prod(ys))
    buf = torch.full((numel * esz + GUARD,), 0x7F, dtype=torch.uint8, device=dev)
    y = buf[: numel * esz].view(dt).view(*ys)
    plan.run(d.x.to(dev), d.w.to(dev), None if d.b is None else d.b.to(dev), y,
             residual=None if r is None else r.to(dev))
    plan.check_device_status()
    torch.cuda.synchronize()
    assert bool((buf[numel * esz:] == 0x7F).all()), "kernel wrote past the end of y"
    # reference: the oracle's layer (+ residual), placed like the plan places it
    if r is not None:
        ref = oracle.conv_residual_f64(to_np64(d.x), to_np64(d.w), None if d.b is None else to_np64(d.b),
                                       to_np64(r), spec.stride, spec.pad_h, spec.pad_w, spec.groups, spec.act)
    else:
        ref = run_oracle(spec, d)
    o = plan.out
    u, off, cy = o["upsample"], o["y_channel_offset"], o["y_channels"]
    got = y.cpu()
    for dy in range(u):
        for dx in range(u):
            sl = got[:, dy::u, dx::u, off:off + spec.cout]
            assert_close(spec, sl if spec.dtype != "i8" else sl.numpy(), ref,
                         f"{spec.name} replica ({dy},{dx}) [{plan.describe()}]")
    # every element outside the slice still holds the poison bytes
    raw = buf[: numel * esz].view(torch.uint8).view(*ys[:3], cy * esz).cpu()
    keep = torch.ones(cy * esz, dtype=torch.bool)
    keep[off * esz:(off + spec.cout) * esz] = False
    assert bool((raw[..., keep] == 0x7F).all()), "the layer wrote outside its channel slice"
    return plan


LAYOUTS = ["igemm", "igemm_swapped", "igemm_n256", "igemm_n128", "igemm_n64", "igemm_pair", "igemm_pair128"]

IGEMM_FUSED = [
    (L("res_3x3_64to64", 1, 13, 11, 64, 64, 3, 3, 1, 1, 1), dict(residual=True)),
    (L("concat_s2_32to48", 1, 15, 17, 32, 48, 3, 3, 2, 1, 1, act="relu"), dict(y_channels=96, y_channel_offset=32)),
    (L("up2_concat_res_1x1", 2, 9, 10, 128, 64, 1, 1, act="mish"),
     dict(y_channels=128, y_channel_offset=64, upsample=2, residual=True)),
    (L("ragged80_res_concat", 1, 11, 12, 64, 80, 3, 3, 1, 1, 1),
     dict(y_channels=112, y_channel_offset=16, residual=True)),
    (L("up2_3x3_cout256", 1, 7, 9, 64, 256, 3, 3, 1, 1, 1, act="none"), dict(upsample=2, residual=True)),
]


@pytest.mark.parametrize("spec,out,layout", [
    pytest.param(s, o, lay, id=f"{s.name}-{lay}") for s, o in IGEMM_FUSED for lay in LAYOUTS
    if not (lay == "igemm_swapped" and s.cout > 128)])
def test_igemm_fused(spec, out, layout):
    plan = run_fused(spec, out, layout)
    assert plan.algo == "igemm"


def test_igemm_int8_concat_upsample_exact():
    spec = L("i8_up2_concat", 1, 10, 9, 32, 32, 3, 3, 1, 1, 1, dtype="i8", act="relu")
    for lay in LAYOUTS:
        plan = run_fused(spec, dict(y_channels=64, y_channel_offset=16, upsample=2), lay)
        assert "i8-as-bf16" in plan.describe()


DIRECT_FUSED = [
    (L("f32_res_relu", 1, 12, 10, 8, 16, 3, 3, 1, 1, 1, dtype="f32", act="relu"), dict(residual=True)),
    (L("f32_up2_concat_mish", 2, 7, 6, 8, 12, 3, 3, 1, 1, 1, dtype="f32"),
     dict(y_channels=20, y_channel_offset=4, upsample=2, residual=True)),
    (L("bf16_dw_res", 1, 9, 11, 32, 32, 3, 3, 1, 1, 1, groups=32), dict(residual=True)),
    (L("bf16_grouped_concat", 1, 8, 8, 16, 32, 3, 3, 2, 1, 1, groups=2), dict(y_channels=48, y_channel_offset=8)),
    (L("i8_dw_up2", 1, 9, 8, 32, 32, 3, 3, 1, 1, 1, groups=32, dtype="i8", act="relu"),
     dict(y_channels=48, y_channel_offset=16, upsample=2)),
]


@pytest.mark.parametrize("spec,out", DIRECT_FUSED, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_direct_fused(spec, out):
    plan = run_fused(spec, out, "auto")
    assert plan.algo == "direct", plan.describe()  # depthwise layers with options run here too


def test_residual_pointer_rules():
    import convolution_nhwc_implicit_gb300 as cl
    spec = L("rules", 1, 8, 8, 16, 16, 3, 3, 1, 1, 1)
    g = torch.Generator("cpu").manual_seed(0)
    d = make_layer(spec, g)
    dev = torch.device("cuda:0")
    x, w = d.x.to(dev), d.w.to(dev)
    y = torch.empty(1, 8, 8, 16, dtype=torch.bfloat16, device=dev)
    p = cl.Plan(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, "bf16", "mish", out=dict(residual=True))
    with pytest.raises(cl.ConvError, match="NULL_ARG"):
        p.run(x, w, None, y)  # the plan needs its residual
    q = cl.Plan(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, "bf16", "mish")
    with pytest.raises(cl.ConvError, match="INVALID_ARG"):
        q.run(x, w, None, y, residual=y.clone())  # a plain plan takes none
    with pytest.raises(cl.ConvError, match="ALIASING"):
        p.run(x, w, None, y, residual=y)  # the residual may not overlap y
