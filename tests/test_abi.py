"""The C-ABI library: it builds, loads without a GPU, exports every function
include/*.h declares, and rejects invalid layers with the named status codes
(validation runs on the host before any CUDA call, so it is testable here)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from convolution_nhwc_implicit_gb300 import build
    build.build()
    import convolution_nhwc_implicit_gb300 as cl
    return cl.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        for m in re.finditer(r"CONV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for fn in ("conv_plan_create", "conv_run", "conv_plan_destroy", "conv_plan_output_shape",
               "conv_status_str"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert names
    for fn in names:
        assert hasattr(lib, fn), fn
    # and nothing but the C ABI is exported
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert {e for e in exported if e.startswith("conv_")} == names


def test_status_strings(lib):
    import convolution_nhwc_implicit_gb300 as cl
    assert cl.status_str(0) == "CONV_OK"
    codes = {-1: "NULL_ARG", -2: "INVALID_SHAPE", -3: "UNSUPPORTED", -4: "MISALIGNED", -5: "ALIASING",
             -6: "CUDA", -7: "DEVICE_TIMEOUT", -8: "OOM", -9: "INVALID_ARG"}
    for c, name in codes.items():
        assert cl.status_str(c) == "CONV_ERR_" + name
    assert cl.status_str(-1234) == "CONV_ERR_UNKNOWN"
    assert cl.abi_version() == 2


def _create(lib, shape, stride=1, ph=0, pw=0, groups=1, dtype=1, act=0, quant=None, algo=0):
    import convolution_nhwc_implicit_gb300 as cl
    s = cl._Shape(*shape)
    h = ctypes.c_void_p(12345)
    rc = lib.conv_plan_create_ex(ctypes.byref(s), stride, ph, pw, groups, dtype, act, quant, algo,
                                 ctypes.byref(h))
    return rc, h


def _quant(scales, si=0.05, so=0.05):
    import convolution_nhwc_implicit_gb300 as cl
    arr = (ctypes.c_float * len(scales))(*scales)
    q = cl._Quant(si, so, ctypes.cast(arr, ctypes.POINTER(ctypes.c_float)))
    q._keep = arr
    return ctypes.pointer(q)


@pytest.mark.parametrize("shape,kw,expect", [
    ((1, 0, 8, 4, 4, 3, 3), {}, -2),                       # h = 0
    ((1, 8, 8, 0, 4, 3, 3), {}, -2),                       # c_in = 0
    ((-1, 8, 8, 4, 4, 3, 3), {}, -2),                      # n < 0
    ((1, 8, 8, 4, 4, 3, 3), {"stride": 0}, -2),
    ((1, 8, 8, 4, 4, 3, 3), {"ph": -1}, -2),
    ((1, 8, 8, 4, 6, 3, 3), {"groups": 4}, -2),            # groups must divide c_out
    ((1, 8, 8, 6, 4, 3, 3), {"groups": 4}, -2),            # ... and c_in
    ((1, 2, 2, 4, 4, 3, 3), {}, -2),                       # no output position fits
    ((1, 8, 8, 4, 4, 3, 3), {"dtype": 7}, -9),             # bad dtype
    ((1, 8, 8, 4, 4, 3, 3), {"act": 5}, -9),               # bad activation
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 9}, -9),              # bad algo
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 3 | 0x300}, -9),      # both staging flags
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 1 | 0x200}, -9),      # staging flag on the direct family
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 0x100}, -9),          # staging flag with AUTO
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 11 | 0x100}, -9),     # staging flag on a bad algo
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 3 | 0xC00}, -9),      # both epilogue flags
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 2 | 0x800}, -9),      # epilogue flag on the depthwise family
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 3 | 0x4000}, -9),     # an unknown flag bit
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 3 | 0x3000}, -9),     # both widening flags
    ((1, 8, 8, 4, 4, 3, 3), {"algo": 1 | 0x2000}, -9),     # widening flag on the direct family
    ((1, 8, 8, 4, 4, 3, 3), {"dtype": 2}, -1),             # int8 without quant
])
def test_invalid_layers_are_named_failures(lib, shape, kw, expect):
    rc, h = _create(lib, shape, **kw)
    assert rc == expect
    assert h.value is None  # *out_plan is cleared on failure


def test_int8_rules(lib):
    # int8 + Mish is not offered
    rc, _ = _create(lib, (1, 8, 8, 4, 4, 3, 3), dtype=2, act=2, quant=_quant([0.01] * 4))
    assert rc == -3
    # non-positive scales are rejected
    rc, _ = _create(lib, (1, 8, 8, 4, 4, 3, 3), dtype=2, quant=_quant([0.01, 0.0, 0.01, 0.01]))
    assert rc == -9
    rc, _ = _create(lib, (1, 8, 8, 4, 4, 3, 3), dtype=2, quant=_quant([0.01] * 4, so=-1.0))
    assert rc == -9
    # quant given to a float layer
    rc, _ = _create(lib, (1, 8, 8, 4, 4, 3, 3), dtype=1, quant=_quant([0.01] * 4))
    assert rc == -9


def test_null_arguments(lib):
    import convolution_nhwc_implicit_gb300 as cl
    s = cl._Shape(1, 8, 8, 4, 4, 3, 3)
    assert lib.conv_plan_create(ctypes.byref(s), 1, 1, 1, 1, 1, 0, None, None) == -1
    h = ctypes.c_void_p()
    assert lib.conv_plan_create(None, 1, 1, 1, 1, 1, 0, None, ctypes.byref(h)) == -1
    assert lib.conv_run(None, None, None, None, None, None) == -1
    oh = ctypes.c_int()
    assert lib.conv_plan_output_shape(None, ctypes.byref(oh), ctypes.byref(oh)) == -1
    lib.conv_plan_destroy(None)  # NULL-safe


def test_valid_layer_without_gpu_is_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = _create(lib, (1, 8, 8, 64, 64, 3, 3), 1, 1, 1)
    assert rc == -6  # CONV_ERR_CUDA: validation passed, no device to plan for
    assert h.value is None


def test_package_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib
    import convolution_nhwc_implicit_gb300 as cl
    monkeypatch.setattr(cl, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(cl, "_lib", None)
    with pytest.raises(ImportError):
        cl.load_library()


@pytest.mark.parametrize("dtype,out,expect", [
    (1, (0, 0, 3, 0), -9),        # upsample must be 1 or 2
    (1, (0, 0, 1, 2), -9),        # residual is 0 or 1
    (1, (32, 24, 1, 0), -9),      # slice past y's channels (24 + 16 > 32)
    (1, (32, -8, 1, 0), -9),      # negative offset
    (1, (32, 4, 1, 0), -4),       # bf16 offset of 8 bytes: not a 16-byte multiple
    (1, (36, 0, 1, 0), -4),       # bf16 pixel pitch of 72 bytes
    (0, (32, 4, 1, 0), None),     # fp32 offset 4 = 16 bytes: valid, the call goes on to CUDA
    (2, (0, 0, 1, 1), -3),        # int8 with a residual is not offered
])
def test_output_options_are_validated_before_cuda(lib, dtype, out, expect):
    import convolution_nhwc_implicit_gb300 as cl
    s = cl._Shape(1, 8, 8, 16, 16, 3, 3)
    quant = _quant([0.01] * 16) if dtype == 2 else None
    o = cl._Output(*out)
    h = ctypes.c_void_p(12345)
    rc = lib.conv_plan_create_fused(ctypes.byref(s), 1, 1, 1, 1, dtype, 0, quant, ctypes.byref(o), 0,
                                    ctypes.byref(h))
    if expect is None:  # valid options: the CUDA step fails without a GPU (or succeeds with one)
        assert rc in (0, -6, -3)
        if rc == 0:
            lib.conv_plan_destroy(h)
    else:
        assert rc == expect
        assert h.value is None


@pytest.mark.parametrize("args,expect", [
    ((1, 8, 8, 16, 1, 64, 0, 16, 32, 48), 0),     # valid (n = 0 below: no CUDA needed)
    ((1, 8, 8, 16, 1, 64, 0, 8, 32, 48), -9),     # mp5 and mp9 slices overlap
    ((1, 8, 8, 16, 1, 64, 0, 16, 56, -1), -9),    # mp13 slice past y's 64 channels
    ((1, 8, 8, 16, 1, 64, 4, 24, 40, -1), -4),    # offset of 8 bytes
    ((1, 8, 8, 12, 1, 64, 0, 16, 32, -1), -4),    # C of 24 bytes
    ((1, 8, 8, 16, 1, 64, -1, 16, 32, 48), -9),   # the three pools are always written
    ((1, 8, 8, 16, 7, 64, 0, 16, 32, 48), -9),    # bad dtype
])
def test_spp_arguments_are_validated_before_cuda(lib, args, expect):
    n, h, w, c, dt, cy, o5, o9, o13, ox = args
    rc = lib.conv_spp_run(0, h, w, c, dt, None, None, cy, o5, o9, o13, ox, None)
    assert rc == expect


@pytest.mark.parametrize("shape,kw,expect", [
    ((1, 8, 8, 16, 16, 5, 5), {}, -2),            # the depthwise kernel is 3x3
    ((1, 8, 8, 16, 16, 3, 3), {"dtype": 2}, -3),  # int8 pair not offered
    ((1, 8, 8, 16, 16, 3, 3), {"act_pw": 7}, -9), # bad activation
    ((1, 8, 8, 16, 16, 3, 3), {"stride": 0}, -2), # validated like the depthwise layer
])
def test_dwpw_plan_validation_before_cuda(lib, shape, kw, expect):
    import convolution_nhwc_implicit_gb300 as cl
    s = cl._Shape(*shape)
    h = ctypes.c_void_p(12345)
    rc = lib.conv_plan_create_dwpw(ctypes.byref(s), kw.get("stride", 1), 1, kw.get("dtype", 0), 1,
                                   kw.get("act_pw", 1), ctypes.byref(h))
    assert rc == expect
    assert h.value is None
