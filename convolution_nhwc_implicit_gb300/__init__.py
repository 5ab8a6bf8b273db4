"""Python binding of the fused NHWC convolution library (``libconv_nhwc.so``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
fallback: if the compiled library is missing or cannot be loaded, importing
this package raises.

Names follow the C ABI in ``include/conv_nhwc.h``::

    plan = Plan(n, h, w, c_in, c_out, k_h, k_w, stride=1, pad_h=0, pad_w=0,
                groups=1, dtype="bf16", act="mish", quant=None)
    plan.run(x, w, b, y)          # torch CUDA tensors, NHWC / OHWI layouts
    y = conv2d_nhwc(x, w, b, stride=..., pad=(ph, pw), act="mish")
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["Plan", "ConvError", "conv2d_nhwc", "library_path", "load_library", "DTYPES", "ACTS",
           "ALGOS", "status_str", "abi_version", "run_i8_noalloc", "NOALLOC_MAX_COUT", "spp", "DwpwPlan"]

# Largest c_out conv_run_i8_noalloc accepts (its fixed scratch array holds
# that many requantisation multipliers).
NOALLOC_MAX_COUT = 4096

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libconv_nhwc.so")

DTYPES = {"f32": 0, "bf16": 1, "i8": 2}
ACTS = {"none": 0, "relu": 1, "mish": 2}
ALGOS = {"auto": 0, "direct": 1, "depthwise": 2, "igemm": 3, "igemm_swapped": 4, "igemm_n256": 5,
         "igemm_n128": 6, "igemm_n64": 7, "igemm_pair": 8, "dwpw": 9, "igemm_pair128": 10}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}
# Staging, epilogue and int8-widening flags of the tensor-core family
# (CONV_ALGO_STAGE_*, CONV_ALGO_EPI_*, CONV_ALGO_WIDEN_*), written as suffixes
# of the algo name: "igemm+halo", "igemm_n64+taps+ept", "igemm+inkernel".
ALGO_FLAGS = {"taps": 0x100, "halo": 0x200, "sliced": 0x400, "ept": 0x800, "prepass": 0x1000,
              "inkernel": 0x2000}


def _algo_code(algo: str) -> int:
    name, *flags = algo.split("+")
    code = ALGOS[name]
    for f in flags:
        code |= ALGO_FLAGS[f]
    return code


class ConvError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {status_str(code)} ({code})")
        self.code = code


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n", "h", "w", "c_in", "c_out", "k_h", "k_w")]


class _Output(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("y_channels", "y_channel_offset", "upsample", "residual")]


class _Quant(ctypes.Structure):
    _fields_ = [("in_scale", ctypes.c_float), ("out_scale", ctypes.c_float),
                ("w_scales", ctypes.POINTER(ctypes.c_float))]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads libconv_nhwc.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with "
            "`python -m convolution_nhwc_implicit_gb300.build` (or __graft_entry__.build())")
    lib = ctypes.CDLL(_LIB_PATH)
    c_int, c_void_p, pp = ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
    lib.conv_plan_create.argtypes = [ctypes.POINTER(_Shape), c_int, c_int, c_int, c_int, c_int, c_int,
                                     ctypes.POINTER(_Quant), pp]
    lib.conv_plan_create.restype = c_int
    lib.conv_plan_create_ex.argtypes = [ctypes.POINTER(_Shape), c_int, c_int, c_int, c_int, c_int, c_int,
                                        ctypes.POINTER(_Quant), c_int, pp]
    lib.conv_plan_create_ex.restype = c_int
    lib.conv_plan_create_fused.argtypes = [ctypes.POINTER(_Shape), c_int, c_int, c_int, c_int, c_int, c_int,
                                           ctypes.POINTER(_Quant), ctypes.POINTER(_Output), c_int, pp]
    lib.conv_plan_create_fused.restype = c_int
    lib.conv_run.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.conv_run.restype = c_int
    lib.conv_run_fused.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.conv_run_fused.restype = c_int
    lib.conv_plan_destroy.argtypes = [c_void_p]
    lib.conv_plan_destroy.restype = None
    lib.conv_plan_output_shape.argtypes = [c_void_p, ctypes.POINTER(c_int), ctypes.POINTER(c_int)]
    lib.conv_plan_output_shape.restype = c_int
    lib.conv_plan_algo.argtypes = [c_void_p]
    lib.conv_plan_algo.restype = c_int
    lib.conv_plan_launches.argtypes = [c_void_p]
    lib.conv_plan_launches.restype = c_int
    lib.conv_plan_describe.argtypes = [c_void_p]
    lib.conv_plan_describe.restype = ctypes.c_char_p
    lib.conv_plan_check_device_status.argtypes = [c_void_p, c_void_p]
    lib.conv_plan_check_device_status.restype = c_int
    lib.conv_status_str.argtypes = [c_int]
    lib.conv_status_str.restype = ctypes.c_char_p
    lib.conv_abi_version.argtypes = []
    lib.conv_abi_version.restype = c_int
    lib.conv_run_i8_noalloc.argtypes = [ctypes.POINTER(_Shape), c_int, c_int, c_int, c_int, c_int,
                                        ctypes.POINTER(_Quant), c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p]
    lib.conv_run_i8_noalloc.restype = c_int
    lib.conv_plan_create_dwpw.argtypes = [ctypes.POINTER(_Shape), c_int, c_int, c_int, c_int, c_int, pp]
    lib.conv_plan_create_dwpw.restype = c_int
    lib.conv_run_dwpw.argtypes = [c_void_p] * 8
    lib.conv_run_dwpw.restype = c_int
    lib.conv_spp_run.argtypes = [c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                 c_int, c_void_p]
    lib.conv_spp_run.restype = c_int
    _lib = lib
    return lib


def status_str(code: int) -> str:
    return load_library().conv_status_str(int(code)).decode()


def abi_version() -> int:
    return load_library().conv_abi_version()


def _ptr(t):
    """Device pointer of a torch tensor (or None / an int address)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """A validated layer bound to the current CUDA device (see conv_plan_create).

    ``out`` (optional) holds the output options of conv_plan_create_fused:
    dict(y_channels=0, y_channel_offset=0, upsample=1, residual=False)."""

    def __init__(self, n, h, w, c_in, c_out, k_h, k_w, stride=1, pad_h=0, pad_w=0, groups=1,
                 dtype="bf16", act="none", quant=None, algo="auto", out=None):
        lib = load_library()
        self._lib = lib
        self._handle = ctypes.c_void_p()
        self.shape = (n, h, w, c_in, c_out, k_h, k_w)
        self.stride, self.pad_h, self.pad_w, self.groups = stride, pad_h, pad_w, groups
        self.dtype, self.act = dtype, act
        shape = _Shape(n, h, w, c_in, c_out, k_h, k_w)
        qp = None
        if quant is not None:
            in_scale, out_scale, w_scales = quant
            ws = [float(v) for v in w_scales]
            self._ws = (ctypes.c_float * len(ws))(*ws)
            qp = ctypes.pointer(_Quant(float(in_scale), float(out_scale),
                                       ctypes.cast(self._ws, ctypes.POINTER(ctypes.c_float))))
        op = None
        self.out = dict(y_channels=c_out, y_channel_offset=0, upsample=1, residual=False)
        if out is not None:
            o = dict(self.out, **out)
            o["y_channels"] = o["y_channels"] or c_out
            self.out = o
            op = ctypes.pointer(_Output(int(o["y_channels"]), int(o["y_channel_offset"]), int(o["upsample"]),
                                        int(bool(o["residual"]))))
        rc = lib.conv_plan_create_fused(ctypes.byref(shape), stride, pad_h, pad_w, groups, DTYPES[dtype],
                                        ACTS[act], qp, op, _algo_code(algo), ctypes.byref(self._handle))
        if rc != 0:
            raise ConvError("conv_plan_create", rc)
        oh, ow = ctypes.c_int(), ctypes.c_int()
        lib.conv_plan_output_shape(self._handle, ctypes.byref(oh), ctypes.byref(ow))
        self.oh, self.ow = oh.value, ow.value

    @property
    def handle(self) -> int:
        return self._handle.value

    @property
    def output_shape(self):
        """Shape of the layer's own output [N, OH, OW, Cout]."""
        n, _, _, _, c_out, _, _ = self.shape
        return (n, self.oh, self.ow, c_out)

    @property
    def y_shape(self):
        """Shape of the y buffer the plan writes into (with its output options)."""
        u = self.out["upsample"]
        return (self.shape[0], self.oh * u, self.ow * u, self.out["y_channels"])

    @property
    def algo(self) -> str:
        return ALGO_NAMES[self._lib.conv_plan_algo(self._handle)]

    @property
    def launches(self) -> int:
        """Kernels one run() enqueues."""
        return self._lib.conv_plan_launches(self._handle)

    def describe(self) -> str:
        return self._lib.conv_plan_describe(self._handle).decode()

    def run(self, x, w, b, y, stream=None, residual=None) -> None:
        """Enqueue y = act(conv(x, w) + b) [+ residual] on `stream` (default: torch's current stream)."""
        if residual is None:
            rc = self._lib.conv_run(self._handle, _ptr(x), _ptr(w), _ptr(b), _ptr(y), _stream_handle(stream))
        else:
            rc = self._lib.conv_run_fused(self._handle, _ptr(x), _ptr(w), _ptr(b), _ptr(residual), _ptr(y),
                                          _stream_handle(stream))
        if rc != 0:
            raise ConvError("conv_run", rc)

    def check_device_status(self, stream=None) -> None:
        rc = self._lib.conv_plan_check_device_status(self._handle, _stream_handle(stream))
        if rc != 0:
            raise ConvError("conv_plan_check_device_status", rc)

    def close(self) -> None:
        if getattr(self, "_handle", None) is not None and self._handle.value:
            self._lib.conv_plan_destroy(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def conv2d_nhwc(x, w, b=None, stride=1, pad=(0, 0), groups=1, act="none", quant=None, algo="auto",
                plan=None, out=None):
    """One-shot helper on torch CUDA tensors: x NHWC, w OHWI, b [Cout].

    Builds a plan (unless given), allocates y with torch (unless ``out``) and
    runs the layer on the current stream."""
    import torch
    dt = {torch.float32: "f32", torch.bfloat16: "bf16", torch.int8: "i8"}[x.dtype]
    n, h, wd, c_in = x.shape
    c_out, k_h, k_w, _ = w.shape
    if plan is None:
        plan = Plan(n, h, wd, c_in, c_out, k_h, k_w, stride, pad[0], pad[1], groups, dt, act, quant, algo)
    if out is None:
        out = torch.empty(plan.output_shape, dtype=x.dtype, device=x.device)
    plan.run(x, w, b, out)
    return out


def run_i8_noalloc(x, w, b, y, stride=1, pad=(0, 0), groups=1, act="none", quant=None, stream=None):
    """An int8 layer through conv_run_i8_noalloc: no plan and no device
    allocation, for callers that must not allocate device memory at run time
    (their buffers come from a pre-reserved pool).  The library keeps the
    requantisation table in one fixed device array shared by all calls, so
    calls that may overlap on the GPU must be serialised.  x NHWC, w OHWI,
    b int32 [Cout] or None, y preallocated NHWC int8; quant = (s_x, s_y, s_w)."""
    lib = load_library()
    n, h, wd, c_in = x.shape
    c_out, k_h, k_w, _ = w.shape
    in_scale, out_scale, w_scales = quant
    ws = (ctypes.c_float * c_out)(*[float(v) for v in w_scales])
    q = _Quant(float(in_scale), float(out_scale), ctypes.cast(ws, ctypes.POINTER(ctypes.c_float)))
    shape = _Shape(n, h, wd, c_in, c_out, k_h, k_w)
    rc = lib.conv_run_i8_noalloc(ctypes.byref(shape), stride, pad[0], pad[1], groups, ACTS[act],
                                 ctypes.byref(q), _ptr(x), _ptr(w), _ptr(b), _ptr(y), _stream_handle(stream))
    if rc != 0:
        raise ConvError("conv_run_i8_noalloc", rc)
    return y


def spp(x, y, y_channels=None, off5=None, off9=None, off13=None, off_x=-1, stream=None):
    """SPP block (conv_spp_run): the 5x5, 9x9 and 13x13 max pools of x (NHWC,
    torch CUDA tensor) written into channel slices of y.  Defaults: y has
    4*C channels laid out [mp5 | mp9 | mp13 | x]."""
    n, h, w, c = x.shape
    y_channels = y_channels or 4 * c
    off5 = 0 if off5 is None else off5
    off9 = c if off9 is None else off9
    off13 = 2 * c if off13 is None else off13
    if off_x is None:
        off_x = 3 * c
    dt = {"torch.float32": 0, "torch.bfloat16": 1, "torch.int8": 2}[str(x.dtype)]
    rc = load_library().conv_spp_run(n, h, w, c, dt, _ptr(x), _ptr(y), y_channels, off5, off9, off13, off_x,
                                     _stream_handle(stream))
    if rc != 0:
        raise ConvError("conv_spp_run", rc)


class DwpwPlan(Plan):
    """A fused depthwise 3x3 -> pointwise 1x1 pair (conv_plan_create_dwpw):
    y = act_pw(pw(round(act_dw(dw(x) + b_dw))) + b_pw), the intermediate kept
    on chip."""

    def __init__(self, n, h, w, c, c_out, stride=1, pad=1, dtype="f32", act_dw="relu", act_pw="relu"):
        lib = load_library()
        self._lib = lib
        self._handle = ctypes.c_void_p()
        self.shape = (n, h, w, c, c_out, 3, 3)
        self.stride, self.pad_h, self.pad_w, self.groups = stride, pad, pad, 1
        self.dtype, self.act, self.act_pw = dtype, act_dw, act_pw
        self.out = dict(y_channels=c_out, y_channel_offset=0, upsample=1, residual=False)
        shape = _Shape(n, h, w, c, c_out, 3, 3)
        rc = lib.conv_plan_create_dwpw(ctypes.byref(shape), stride, pad, DTYPES[dtype], ACTS[act_dw], ACTS[act_pw],
                                       ctypes.byref(self._handle))
        if rc != 0:
            raise ConvError("conv_plan_create_dwpw", rc)
        oh, ow = ctypes.c_int(), ctypes.c_int()
        lib.conv_plan_output_shape(self._handle, ctypes.byref(oh), ctypes.byref(ow))
        self.oh, self.ow = oh.value, ow.value

    def run(self, x, w_dw, b_dw, w_pw, b_pw, y, stream=None) -> None:  # noqa: D401
        """Enqueue the fused pair on `stream` (default: torch's current stream)."""
        rc = self._lib.conv_run_dwpw(self._handle, _ptr(x), _ptr(w_dw), _ptr(b_dw), _ptr(w_pw), _ptr(b_pw),
                                     _ptr(y), _stream_handle(stream))
        if rc != 0:
            raise ConvError("conv_run_dwpw", rc)
