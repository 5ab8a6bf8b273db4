"""conv_run_i8_noalloc: the int8 layer run that allocates no device memory.

It serves callers that may not call cudaMalloc while running (their device
memory is reserved up front, or an allocation could block or fail where they
call from).  It must compute exactly what the plan path computes.  Two calls
in a row, on different layers, check that each call rewrites the library's
shared requantisation table before using it.  Every result is also compared
bit for bit with the oracle: layers with more output channels than one fill
launch carries (the largest accepted count included), depthwise layers, input
channels not a multiple of 4 (the scalar-product kernel), and the
requantisation families of tests/test_gpu_requant.py (exact ties; an input
scale different from the output scale).

This file is collected last on purpose; it builds the library itself, so it
also passes when run alone in a fresh process.
"""
import ctypes

import pytest
import torch

from conv_workloads import LayerSpec, make_layer
from parity_util import run_oracle

pytestmark = pytest.mark.gpu

_I8 = dict(dtype="i8", x_dist=("int", -128, 127), w_dist=("int", -127, 127),
           b_dist=("int", -1000, 1000), in_scale=0.05, out_scale=0.05)
# power-of-two scales and small data: products land exactly on .5
_TIE = dict(dtype="i8", x_dist=("int", -3, 3), w_dist=("int", -3, 3), b_dist=("int", -40, 40),
            in_scale=0.125, out_scale=0.5, ws_dist=("pow2", -2, 1))
_RATIO = dict(_I8, in_scale=0.02, out_scale=0.07)


@pytest.fixture(scope="module")
def cl():
    from convolution_nhwc_implicit_gb300 import build
    build.build()
    import convolution_nhwc_implicit_gb300 as cl
    cl.load_library()
    return cl


def _plan_path(cl, d):
    s = d.spec
    plan = cl.Plan(s.n, s.h, s.w, s.cin, s.cout, s.kh, s.kw, s.stride, s.pad_h, s.pad_w, s.groups,
                   "i8", s.act, (s.in_scale, s.out_scale, d.w_scales.tolist()))
    dev = torch.device("cuda:0")
    y = torch.empty(plan.output_shape, dtype=torch.int8, device=dev)
    plan.run(d.x.to(dev), d.w.to(dev), d.b.to(dev), y)
    torch.cuda.synchronize()
    return y.cpu(), plan.output_shape


def _noalloc_via_c_abi(cl, d, out_shape):
    """Calls conv_run_i8_noalloc directly through ctypes."""
    s = d.spec
    lib = cl.load_library()
    dev = torch.device("cuda:0")
    x, w, b = d.x.to(dev), d.w.to(dev), d.b.to(dev)
    y = torch.full(out_shape, 0x55, dtype=torch.int8, device=dev)
    ws = (ctypes.c_float * s.cout)(*d.w_scales.tolist())
    q = cl._Quant(s.in_scale, s.out_scale, ctypes.cast(ws, ctypes.POINTER(ctypes.c_float)))
    shape = cl._Shape(s.n, s.h, s.w, s.cin, s.cout, s.kh, s.kw)
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.conv_run_i8_noalloc(ctypes.byref(shape), s.stride, s.pad_h, s.pad_w, s.groups,
                                 cl.ACTS[s.act], ctypes.byref(q), x.data_ptr(), w.data_ptr(),
                                 b.data_ptr(), y.data_ptr(), stream)
    assert rc == 0, cl.status_str(rc)
    return y


def test_noalloc_matches_plan_path_on_consecutive_calls(cl):
    g = torch.Generator("cpu").manual_seed(2024)
    layer_a = make_layer(LayerSpec("na_dense", 1, 96, 96, 64, 64, 3, 3, 1, 1, 1, act="none", **_I8), g)
    layer_b = make_layer(LayerSpec("na_pw", 1, 40, 36, 32, 96, 1, 1, 1, 0, 0, act="relu",
                                   **{**_I8, "out_scale": 0.02}), g)
    ref_a, shape_a = _plan_path(cl, layer_a)
    ref_b, shape_b = _plan_path(cl, layer_b)
    # two calls in a row, different layers and multiplier tables, no sync between
    y_a = _noalloc_via_c_abi(cl, layer_a, shape_a)
    y_b = _noalloc_via_c_abi(cl, layer_b, shape_b)
    torch.cuda.synchronize()
    assert torch.equal(y_a.cpu(), ref_a)  # int8 results are bit-exact
    assert torch.equal(y_b.cpu(), ref_b)
    assert torch.equal(y_a.cpu(), torch.from_numpy(run_oracle(layer_a.spec, layer_a)))
    assert torch.equal(y_b.cpu(), torch.from_numpy(run_oracle(layer_b.spec, layer_b)))
    # and the first layer again, after the table was overwritten
    y_a2 = _noalloc_via_c_abi(cl, layer_a, shape_a)
    torch.cuda.synchronize()
    assert torch.equal(y_a2.cpu(), ref_a)


def test_noalloc_rejects_layers_beyond_its_scratch(cl):
    lib = cl.load_library()
    c_out = cl.NOALLOC_MAX_COUT + 1
    ws = (ctypes.c_float * c_out)(*([0.01] * c_out))
    q = cl._Quant(0.05, 0.05, ctypes.cast(ws, ctypes.POINTER(ctypes.c_float)))
    shape = cl._Shape(1, 4, 4, 16, c_out, 1, 1)
    rc = lib.conv_run_i8_noalloc(ctypes.byref(shape), 1, 0, 0, 1, 0, ctypes.byref(q), None, None,
                                 None, None, None)
    assert rc == -10 and cl.status_str(rc) == "CONV_ERR_SCRATCH_LIMIT"


NOALLOC_CASES = [
    # more output channels than one fill launch carries (1000), and the most accepted
    LayerSpec("na_cout2048", 1, 4, 4, 16, 2048, 1, 1, 1, 0, 0, act="none", **_I8),
    LayerSpec("na_cout_max", 1, 4, 4, 16, 4096, 1, 1, 1, 0, 0, act="relu", **_I8),
    # depthwise (the visual-wake-words layer) and a strided depthwise tie case
    LayerSpec("na_dw_32_96", 1, 96, 96, 32, 32, 3, 3, 1, 1, 1, 32, act="none", **_I8),
    LayerSpec("na_dw_tie_s2", 1, 19, 17, 32, 32, 3, 3, 2, 1, 1, 32, act="relu", **_TIE),
    # input channels not a multiple of 4: scalar products
    LayerSpec("na_cin3", 1, 18, 16, 3, 16, 3, 3, 1, 1, 1, act="none", **_I8),
    LayerSpec("na_cin3_tie", 1, 11, 9, 3, 16, 3, 3, 2, 1, 1, act="none", **_TIE),
    # exact ties and s_x != s_y on the dense kernel
    LayerSpec("na_dense_tie", 1, 21, 19, 64, 64, 3, 3, 1, 1, 1, act="none", **_TIE),
    LayerSpec("na_dense_ratio", 1, 21, 19, 64, 64, 3, 3, 1, 1, 1, act="relu", **_RATIO),
]


@pytest.mark.parametrize("spec", NOALLOC_CASES, ids=lambda s: s.name)
def test_noalloc_matches_oracle(cl, spec):
    d = make_layer(spec, torch.Generator("cpu").manual_seed(31))
    ref = torch.from_numpy(run_oracle(spec, d))
    y1 = _noalloc_via_c_abi(cl, d, tuple(ref.shape))
    y2 = _noalloc_via_c_abi(cl, d, tuple(ref.shape))  # a second call in a row
    torch.cuda.synchronize()
    assert torch.equal(y1.cpu(), ref)
    assert torch.equal(y2.cpu(), ref)
    plan_y, _ = _plan_path(cl, d)
    assert torch.equal(plan_y, ref)
