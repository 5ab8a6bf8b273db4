"""Plain CPU oracle for the fused NHWC convolution layer (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never does, and this package
imports nothing from it: the two share no code.

Every function here is a thin numpy/ctypes wrapper around ``oracle.c``, which
computes the layer by its plain definition in nested loops (double precision
for float layers, exact int64 for int8 layers).  See the header of
``oracle.c`` for the definition and the passages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
# A prebuilt oracle library to load instead (the mutation test points this at
# copies of oracle.c with planted mistakes).
_LIB_OVERRIDE = os.environ.get("ORACLE_LIB")
_lock = threading.Lock()
_lib = None

ACT = {"none": 0, "relu": 1, "mish": 2}


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, OpenMP, no fast-math,
    no FMA contraction so that float rounding is exactly IEEE single/double)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = [
            "gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
            "-fno-fast-math", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if _LIB_OVERRIDE:
                lib = ctypes.CDLL(_LIB_OVERRIDE)
            else:
                build()
                lib = ctypes.CDLL(_LIB_PATH)
            i, d, f, p, l = (ctypes.c_int, ctypes.c_double, ctypes.c_float,
                             ctypes.c_void_p, ctypes.c_long)
            lib.oracle_output_dim.argtypes = [i, i, i, i]
            lib.oracle_output_dim.restype = i
            lib.oracle_mish.argtypes = [d]
            lib.oracle_mish.restype = d
            lib.oracle_conv_f64.argtypes = [p, p, p, p] + [i] * 13
            lib.oracle_conv_f64.restype = i
            lib.oracle_conv_f64_points.argtypes = [p, p, p, p, l, p] + [i] * 13
            lib.oracle_conv_f64_points.restype = i
            lib.oracle_requant_multipliers.argtypes = [f, f, p, i, p]
            lib.oracle_requant_multipliers.restype = i
            lib.oracle_requant_one.argtypes = [ctypes.c_int64, f, i]
            lib.oracle_requant_one.restype = i
            lib.oracle_conv_i8_acc.argtypes = [p, p, p] + [i] * 12
            lib.oracle_conv_i8_acc.restype = i
            lib.oracle_conv_i8.argtypes = [p, p, p, p, p] + [i] * 13
            lib.oracle_conv_i8.restype = i
            lib.oracle_conv_i8_points.argtypes = [p, p, p, p, p, l, p] + [i] * 13
            lib.oracle_conv_i8_points.restype = i
            lib.oracle_max_threads.argtypes = [i]
            lib.oracle_max_threads.restype = i
            lib.oracle_maxpool_same.argtypes = [p, p] + [i] * 6
            lib.oracle_maxpool_same.restype = i
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def output_dim(n_in: int, k: int, pad: int, stride: int) -> int:
    """floor((n_in + 2*pad - k) / stride) + 1, or -1 if nothing fits."""
    return _load().oracle_output_dim(n_in, k, pad, stride)


def output_shape(h, w, kh, kw, stride, pad_h, pad_w):
    return output_dim(h, kh, pad_h, stride), output_dim(w, kw, pad_w, stride)


def mish(v: float) -> float:
    """Mish(v) = v * tanh(ln(1 + e^v)) in double."""
    return _load().oracle_mish(float(v))


def max_threads(nthreads: int = 0) -> int:
    return _load().oracle_max_threads(nthreads)


def _dims(x, w, groups):
    N, H, W, Cin = x.shape
    Cout, KH, KW, cpg = w.shape
    if cpg * groups != Cin:
        raise ValueError(f"weight has {cpg} channels per group, input {Cin}, groups {groups}")
    return N, H, W, Cin, Cout, KH, KW


def conv_f64(x, w, b, stride=1, pad_h=0, pad_w=0, groups=1, act="none", threads=0):
    """y = act(conv(x, w) + b) in double.  x NHWC, w OHWI (channels per group
    innermost), b [Cout] or None.  Returns NHWC float64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    b = None if b is None else np.ascontiguousarray(b, dtype=np.float64)
    N, H, W, Cin, Cout, KH, KW = _dims(x, w, groups)
    OH, OW = output_shape(H, W, KH, KW, stride, pad_h, pad_w)
    if OH < 1 or OW < 1:
        raise ValueError("no output position fits")
    y = np.empty((N, OH, OW, Cout), dtype=np.float64)
    rc = _load().oracle_conv_f64(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, H, W, Cin,
                                 Cout, KH, KW, stride, pad_h, pad_w, groups,
                                 ACT[act], threads)
    if rc:
        raise ValueError("oracle_conv_f64 rejected the arguments")
    return y


def conv_f64_points(x, w, b, points, stride=1, pad_h=0, pad_w=0, groups=1,
                    act="none", threads=0):
    """The float layer at selected outputs; ``points`` is an int array [P, 4]
    of (n, oh, ow, co).  Returns float64 [P]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    b = None if b is None else np.ascontiguousarray(b, dtype=np.float64)
    pts = np.ascontiguousarray(points, dtype=np.int32).reshape(-1, 4)
    N, H, W, Cin, Cout, KH, KW = _dims(x, w, groups)
    vals = np.empty(pts.shape[0], dtype=np.float64)
    rc = _load().oracle_conv_f64_points(_ptr(x), _ptr(w), _ptr(b), _ptr(pts),
                                        pts.shape[0], _ptr(vals), N, H, W, Cin,
                                        Cout, KH, KW, stride, pad_h, pad_w, groups,
                                        ACT[act], threads)
    if rc:
        raise ValueError("oracle_conv_f64_points rejected the arguments")
    return vals


def requant_multipliers(in_scale, out_scale, w_scales):
    """M[co] = float32(s_x * s_w[co] / s_y), formed in double, rounded once."""
    ws = np.ascontiguousarray(w_scales, dtype=np.float32)
    M = np.empty(ws.shape[0], dtype=np.float32)
    rc = _load().oracle_requant_multipliers(float(in_scale), float(out_scale),
                                            _ptr(ws), ws.shape[0], _ptr(M))
    if rc:
        raise ValueError("scales must be positive")
    return M


def requant_one(v: int, M: float, relu: bool = False) -> int:
    """sat_[-128,127](rne(float(v) * M)), then max(q, 0) if relu."""
    return _load().oracle_requant_one(int(v), float(np.float32(M)), int(relu))


def conv_i8_acc(x, w, stride=1, pad_h=0, pad_w=0, groups=1, threads=0):
    """Exact int64 accumulators of an int8 layer (no bias)."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    N, H, W, Cin, Cout, KH, KW = _dims(x, w, groups)
    OH, OW = output_shape(H, W, KH, KW, stride, pad_h, pad_w)
    acc = np.empty((N, OH, OW, Cout), dtype=np.int64)
    rc = _load().oracle_conv_i8_acc(_ptr(x), _ptr(w), _ptr(acc), N, H, W, Cin, Cout,
                                    KH, KW, stride, pad_h, pad_w, groups, threads)
    if rc:
        raise ValueError("oracle_conv_i8_acc rejected the arguments")
    return acc


def conv_i8(x, w, b, M, stride=1, pad_h=0, pad_w=0, groups=1, relu=False, threads=0):
    """int8 layer: requant(conv(x, w) + b) with per-channel multipliers M."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    b = None if b is None else np.ascontiguousarray(b, dtype=np.int32)
    M = np.ascontiguousarray(M, dtype=np.float32)
    N, H, W, Cin, Cout, KH, KW = _dims(x, w, groups)
    OH, OW = output_shape(H, W, KH, KW, stride, pad_h, pad_w)
    y = np.empty((N, OH, OW, Cout), dtype=np.int8)
    rc = _load().oracle_conv_i8(_ptr(x), _ptr(w), _ptr(b), _ptr(M), _ptr(y), N, H, W,
                                Cin, Cout, KH, KW, stride, pad_h, pad_w, groups,
                                int(relu), threads)
    if rc:
        raise ValueError("oracle_conv_i8 rejected the arguments")
    return y


def conv_i8_points(x, w, b, M, points, stride=1, pad_h=0, pad_w=0, groups=1,
                   relu=False, threads=0):
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    b = None if b is None else np.ascontiguousarray(b, dtype=np.int32)
    M = np.ascontiguousarray(M, dtype=np.float32)
    pts = np.ascontiguousarray(points, dtype=np.int32).reshape(-1, 4)
    N, H, W, Cin, Cout, KH, KW = _dims(x, w, groups)
    vals = np.empty(pts.shape[0], dtype=np.int8)
    rc = _load().oracle_conv_i8_points(_ptr(x), _ptr(w), _ptr(b), _ptr(M), _ptr(pts),
                                       pts.shape[0], _ptr(vals), N, H, W, Cin, Cout,
                                       KH, KW, stride, pad_h, pad_w, groups,
                                       int(relu), threads)
    if rc:
        raise ValueError("oracle_conv_i8_points rejected the arguments")
    return vals


def conv_residual_f64(x, w, b, r, stride=1, pad_h=0, pad_w=0, groups=1, act="none", threads=0):
    """Convolution, activation, then a residual (skip) tensor added once:
    y = act(conv(x, w) + b) + r, in double ("YOLOv4, optimized for Wormhole",
    section 9, K2 "Mish + residual add": Mish first, then the add, one
    write).  r is NHWC with the layer's output shape."""
    y = conv_f64(x, w, b, stride, pad_h, pad_w, groups, act, threads)
    r = np.asarray(r, dtype=np.float64)
    if r.shape != y.shape:
        raise ValueError(f"residual shape {r.shape} differs from the output shape {y.shape}")
    return y + r


def place_output(y, y_channels, y_channel_offset=0, upsample=1, fill=np.nan):
    """Where a layer's output lands in the next layer's buffer ("YOLOv4,
    optimized for Wormhole", section 9, K4 "upsample + concat": rows repeated
    for a 2x nearest-neighbour upsample, written into the concatenated
    layout): out[n, u*oh+dy, u*ow+dx, off+co] = y[n, oh, ow, co] for dy, dx
    in [0, u); every other element of out is ``fill``."""
    y = np.asarray(y)
    N, OH, OW, C = y.shape
    if y_channel_offset < 0 or y_channel_offset + C > y_channels or upsample < 1:
        raise ValueError("slice outside the output buffer")
    out = np.full((N, OH * upsample, OW * upsample, y_channels), fill,
                  dtype=np.result_type(y.dtype, np.asarray(fill).dtype))
    rep = np.repeat(np.repeat(y, upsample, axis=1), upsample, axis=2)
    out[..., y_channel_offset:y_channel_offset + C] = rep
    return out


def maxpool_same(x, k, threads=0):
    """k x k max pool, stride 1, output the size of the input, positions
    outside the image left out of the max (the pools of the YOLOv4 SPP block,
    "YOLOv4, optimized for Wormhole", section 9, K3).  Direct evaluation
    over each window in oracle.c.  x NHWC; returns float64 (exact)."""
    xd = np.ascontiguousarray(x, dtype=np.float64)
    N, H, W, C = xd.shape
    y = np.empty_like(xd)
    if _load().oracle_maxpool_same(_ptr(xd), _ptr(y), N, H, W, C, int(k), threads):
        raise ValueError("oracle_maxpool_same rejected the arguments")
    return y


def spp(x, threads=0):
    """The SPP block's three pools of x: (mp5, mp9, mp13)."""
    return tuple(maxpool_same(x, k, threads) for k in (5, 9, 13))


def dwpw_f64(x, w_dw, b_dw, w_pw, b_pw, stride=1, pad=1, act_dw="none", act_pw="none", round_to=None,
             threads=0):
    """The depthwise-separable pair run one layer after the other, in double:
    z = act_dw(depthwise 3x3 (x, w_dw) + b_dw), rounded to the layer type
    (``round_to`` a callable on float64 arrays, e.g. rounding to bf16; None
    for fp32), then y = act_pw(1x1 (z, w_pw) + b_pw).  w_dw [C,3,3,1],
    w_pw [Cout,1,1,C].  (The fused kernel keeps z on chip; the result is the
    same pair of layers.)"""
    C = np.asarray(x).shape[3]
    z = conv_f64(x, w_dw, b_dw, stride, pad, pad, C, act_dw, threads)
    if round_to is not None:
        z = np.asarray(round_to(z), dtype=np.float64)
    return conv_f64(z, w_pw, b_pw, 1, 0, 0, 1, act_pw, threads)
