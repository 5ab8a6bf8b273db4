"""GPU parity of the fused depthwise 3x3 -> pointwise pair (conv_run_dwpw)
against the oracle's two layers run one after the other (the intermediate
rounded to the layer type in between)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}
DT = {"f32": torch.float32, "bf16": torch.bfloat16}

CASES = [
    # name, n, h, w, c, cout, stride, pad, dtype, act_dw, act_pw
    ("kws_ds_block_25x5x64", 1, 25, 5, 64, 64, 1, 1, "f32", "relu", "relu"),
    ("f32_s2_ragged", 2, 13, 11, 24, 40, 2, 1, "f32", "none", "mish"),
    ("bf16_mish_mish", 1, 20, 18, 32, 48, 1, 1, "bf16", "mish", "mish"),
    ("bf16_c512_cout64", 1, 10, 10, 512, 64, 1, 1, "bf16", "relu", "none"),
    ("f32_pad0_single_row", 1, 3, 17, 16, 12, 1, 0, "f32", "relu", "relu"),
    ("bf16_cout_not_multiple_of_4", 2, 7, 9, 8, 6, 1, 1, "bf16", "none", "relu"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_dwpw_matches_two_layers(case):
    import convolution_nhwc_implicit_gb300 as cl
    name, n, h, w, c, co, s, p, dt, a1, a2 = case
    g = torch.Generator("cpu").manual_seed(3)
    x = torch.empty(n, h, w, c).uniform_(-1, 1, generator=g).to(DT[dt])
    wd = (torch.randn(c, 3, 3, 1, generator=g) * (2 / 9) ** 0.5).to(DT[dt])
    bd = torch.randn(c, generator=g) * 0.1
    wp = (torch.randn(co, 1, 1, c, generator=g) * (2 / c) ** 0.5).to(DT[dt])
    bp = None if name.startswith("f32_pad0") else torch.randn(co, generator=g) * 0.1
    plan = cl.DwpwPlan(n, h, w, c, co, s, p, dt, a1, a2)
    assert plan.algo == "dwpw", plan.describe()
    dev = torch.device("cuda:0")
    oh, ow = plan.oh, plan.ow
    y = torch.full((n, oh, ow, co), float("nan"), dtype=DT[dt], device=dev)
    plan.run(x.to(dev), wd.to(dev), bd.to(dev), wp.to(dev), None if bp is None else bp.to(dev), y)
    torch.cuda.synchronize()
    rnd = (lambda z: torch.from_numpy(z).to(torch.bfloat16).to(torch.float64).numpy()) if dt == "bf16" else None
    ref = oracle.dwpw_f64(x.double().numpy(), wd.double().numpy(), bd.double().numpy(), wp.double().numpy(),
                          None if bp is None else bp.double().numpy(), s, p, a1, a2, rnd)
    got = y.cpu().double().numpy()
    err = np.abs(got - ref)
    lim = TOL[dt] * (1 + np.abs(ref))
    assert (err <= lim).all(), f"{name} [{plan.describe()}]: max err {err.max():.3e}"


def test_dwpw_plan_runs_only_through_its_entry_point():
    import convolution_nhwc_implicit_gb300 as cl
    plan = cl.DwpwPlan(1, 8, 8, 16, 16)
    dev = torch.device("cuda:0")
    x = torch.zeros(1, 8, 8, 16, device=dev)
    with pytest.raises(cl.ConvError, match="INVALID_ARG"):
        cl.Plan.run(plan, x, x, None, torch.empty_like(x))
