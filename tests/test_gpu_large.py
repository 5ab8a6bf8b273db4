"""GPU parity at sizes past 32-bit offsets: outputs of more than 2^31 bytes
(the tensor-core and int8 cases also more than 2^31 elements), for each
kernel family, through the C ABI.  Inputs are drawn on the GPU by a seeded
generator; outputs are checked on sampled points, among them the last
pixels of the last image, against the oracle evaluated on each point's
receptive field (cut out of x with the zero padding written in)."""
import numpy as np
import pytest
import torch

import oracle
from conv_workloads import LayerSpec, make_layer_device_x, output_hw
from parity_util import TOL, TORCH_DT, assert_close, make_plan, sample_points

pytestmark = pytest.mark.gpu


def _field(spec, x, pts):
    """x cut to each point's k_h x k_w receptive field (zeros outside the image),
    on the host: [len(pts), k_h, k_w, Cin]."""
    oh_, ow_ = pts[:, 1], pts[:, 2]
    out = np.zeros((len(pts), spec.kh, spec.kw, spec.cin),
                   dtype=np.int8 if spec.dtype == "i8" else np.float64)
    for i, (n, oh, ow, _) in enumerate(pts.tolist()):
        h0, w0 = oh * spec.stride - spec.pad_h, ow * spec.stride - spec.pad_w
        hs, he = max(h0, 0), min(h0 + spec.kh, spec.h)
        ws, we = max(w0, 0), min(w0 + spec.kw, spec.w)
        if hs < he and ws < we:
            patch = x[n, hs:he, ws:we, :].cpu()
            patch = patch.numpy() if spec.dtype == "i8" else patch.to(torch.float64).numpy()
            out[i, hs - h0:he - h0, ws - w0:we - w0, :] = patch
    return out


def _oracle_points(spec, d, pts):
    """The oracle on each point's receptive field: a k_h x k_w input with no
    padding and stride 1 gives the point's output at (0, 0)."""
    fields = _field(spec, d.x, pts)
    ref = np.zeros(len(pts), dtype=np.int8 if spec.dtype == "i8" else np.float64)
    b = None if d.b is None else (d.b.numpy() if spec.dtype == "i8" else d.b.double().numpy())
    if spec.dtype == "i8":
        M = oracle.requant_multipliers(spec.in_scale, spec.out_scale, d.w_scales.numpy())
        w = d.w.numpy()
    else:
        w = d.w.double().numpy()
    for i in range(len(pts)):
        f = fields[i:i + 1]
        if spec.dtype == "i8":
            y = oracle.conv_i8(f, w, b, M, 1, 0, 0, spec.groups, spec.act == "relu")
        else:
            y = oracle.conv_f64(f, w, b, 1, 0, 0, spec.groups, spec.act)
        ref[i] = y[0, 0, 0, pts[i, 3]]
    return ref


_I8 = dict(x_dist=("int", -128, 127), w_dist=("int", -127, 127), b_dist=("int", -1000, 1000))

LARGE = [
    # tensor cores, bf16: y 8 x 640 x 640 x 1024 = 3.4e9 elements (6.7 GB)
    (LayerSpec("big_igemm_bf16", 8, 640, 640, 16, 1024, 3, 3, 1, 1, 1, dtype="bf16", act="mish"), "igemm"),
    # tensor cores, exact int8: y 3.4e9 bytes
    (LayerSpec("big_igemm_i8", 8, 640, 640, 16, 1024, 3, 3, 1, 1, 1, dtype="i8", act="relu", **_I8), "igemm"),
    # depthwise stencil, bf16: x and y 8 x 640 x 640 x 512 (3.4 GB each)
    (LayerSpec("big_dw_bf16", 8, 640, 640, 512, 512, 3, 3, 1, 1, 1, groups=512, dtype="bf16", act="mish"),
     "depthwise"),
    # direct FFMA, fp32: y 4 x 1024 x 1024 x 128 x 4 bytes = 2.1 GB
    (LayerSpec("big_direct_f32", 4, 1024, 1024, 16, 128, 1, 1, dtype="f32", act="relu"), "direct"),
]


@pytest.mark.parametrize("spec,algo", LARGE, ids=[s.name for s, _ in LARGE])
def test_outputs_past_32bit_offsets(spec, algo):
    dev = torch.device("cuda:0")
    d = make_layer_device_x(spec, seed=11, device=dev)
    plan = make_plan(spec, d, algo)
    assert plan.algo == algo, plan.describe()
    oh, ow = output_hw(spec)
    y = torch.empty((spec.n, oh, ow, spec.cout), dtype=TORCH_DT[spec.dtype], device=dev)
    b = None if d.b is None else d.b.to(dev)
    plan.run(d.x, d.w.to(dev), b, y)
    plan.check_device_status()
    torch.cuda.synchronize()
    pts = sample_points(spec, 600, seed=7)
    # the last pixels of the last image, every channel class
    last = [(spec.n - 1, oh - 1, ow - 1 - j, c) for j in range(4) for c in (0, spec.cout // 2, spec.cout - 1)]
    pts = np.concatenate([pts, np.array(last, dtype=np.int32)], axis=0)
    pt = torch.from_numpy(pts.astype(np.int64)).to(dev)
    got = y[pt[:, 0], pt[:, 1], pt[:, 2], pt[:, 3]].cpu()
    ref = _oracle_points(spec, d, pts)
    assert_close(spec, got, ref, f"{spec.name} [{plan.describe()}]")
    del y, d
    torch.cuda.empty_cache()
