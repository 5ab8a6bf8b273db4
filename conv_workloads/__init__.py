"""Seeded synthetic workloads for the fused NHWC convolution layer.

This module only draws random tensors: it holds none of the layer's arithmetic,
and both the oracle-side tests and the CUDA-side tests and benchmark take
their inputs from here.

Shapes and value distributions are those of the five layer sets the library
is measured on (edge CNNs from the "nanoinfer" page: an MNIST-sized 3x3 conv,
the keyword-spotting DS-CNN block, the visual-wake-words int8 layers; and
YOLOv4-style bf16 layers from "YOLOv4, optimized for Wormhole": a 4x320
mosaic stem and a batch-8 throughput sweep).  The pages' datasets (MNIST,
Speech Commands, Visual Wake Words, COCO) and trained weights are not used:
seeded synthetic tensors of the same shapes stand in for them.

Draw order: one ``torch.Generator('cpu')`` per layer set, seeded with the
set's seed; layers in listed order; per layer x, then w, then b, then (int8)
the per-channel weight scales.  Layouts: x NHWC, w OHWI (input channels of
the group innermost), b [Cout].  Float values are drawn in fp32 and bf16
tensors are the fp32 draw rounded to nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

__all__ = ["LayerSpec", "LayerData", "CONFIGS", "SEEDS", "generate", "make_layer", "make_layer_device_x",
           "spec_by_name", "macs", "alg_bytes", "output_hw"]


@dataclass(frozen=True)
class LayerSpec:
    name: str
    n: int
    h: int
    w: int
    cin: int
    cout: int
    kh: int
    kw: int
    stride: int = 1
    pad_h: int = 0
    pad_w: int = 0
    groups: int = 1
    dtype: str = "f32"          # "f32" | "bf16" | "i8"
    act: str = "none"           # "none" | "relu" | "mish"
    x_dist: tuple = ("uniform", -1.0, 1.0)
    w_dist: tuple = ("he",)     # ("normal", std) | ("he",) | ("int", lo, hi)
    b_dist: tuple = ("normal", 0.01)  # ("normal", std) | ("int", lo, hi) | None
    in_scale: float = 0.05      # int8 only: activation scale s_x
    out_scale: float = 0.05     # int8 only: output scale s_y
    ws_dist: tuple = ("uniform", 0.001, 0.01)  # int8 only: per-channel s_w, or ("pow2", lo, hi)


@dataclass
class LayerData:
    spec: LayerSpec
    x: torch.Tensor             # CPU, dtype float32 / bfloat16 / int8
    w: torch.Tensor
    b: torch.Tensor | None      # float32 (float layers) or int32 (int8 layers)
    w_scales: torch.Tensor | None = None  # float32 [Cout], int8 layers only
    extra: dict = field(default_factory=dict)


def output_hw(s: LayerSpec):
    oh = (s.h + 2 * s.pad_h - s.kh) // s.stride + 1
    ow = (s.w + 2 * s.pad_w - s.kw) // s.stride + 1
    return oh, ow


def macs(s: LayerSpec) -> int:
    """Multiply-accumulates of the layer (the algorithmic count)."""
    oh, ow = output_hw(s)
    return s.n * oh * ow * s.cout * s.kh * s.kw * (s.cin // s.groups)


def alg_bytes(s: LayerSpec) -> int:
    """Bytes of x, w, b and y, each moved once."""
    es = {"f32": 4, "bf16": 2, "i8": 1}[s.dtype]
    oh, ow = output_hw(s)
    x = s.n * s.h * s.w * s.cin * es
    w = s.cout * s.kh * s.kw * (s.cin // s.groups) * es
    b = s.cout * 4 if s.b_dist is not None else 0
    y = s.n * oh * ow * s.cout * es
    return x + w + b + y


_I8 = dict(dtype="i8", act="none", x_dist=("int", -128, 127), w_dist=("int", -127, 127),
           b_dist=("int", -1000, 1000), in_scale=0.05, out_scale=0.05)
_YOLO = dict(dtype="bf16", act="mish", x_dist=("uniform", 0.0, 1.0), w_dist=("he",),
             b_dist=("normal", 0.01))
_SWEEP = dict(dtype="bf16", act="mish", x_dist=("normal", 1.0), w_dist=("he",),
              b_dist=("normal", 0.01))

CONFIGS: dict[str, list[LayerSpec]] = {
    # Single fp32 3x3 conv, MNIST-sized.
    "mnist_conv3x3_f32": [
        LayerSpec("conv3x3_8to16_28", 1, 28, 28, 8, 16, 3, 3, 1, 1, 1, dtype="f32",
                  act="relu", x_dist=("uniform", -1.0, 1.0), w_dist=("normal", 0.1)),
    ],
    # Keyword-spotting DS-CNN block: 10x4 stem with padding (5, 1), then four
    # depthwise-separable pairs.
    "kws_dscnn_f32": [
        LayerSpec("stem10x4_1to64_49x10", 1, 49, 10, 1, 64, 10, 4, 2, 5, 1, dtype="f32",
                  act="relu"),
    ] + [
        spec for i in range(4) for spec in (
            LayerSpec(f"dw3x3_64_25x5_{i}", 1, 25, 5, 64, 64, 3, 3, 1, 1, 1, groups=64,
                      dtype="f32", act="relu"),
            LayerSpec(f"pw1x1_64to64_25x5_{i}", 1, 25, 5, 64, 64, 1, 1, 1, 0, 0,
                      dtype="f32", act="relu"),
        )
    ],
    # Visual-wake-words-shaped int8 layers.
    "vww_int8": [
        LayerSpec("dw3x3_32_96", 1, 96, 96, 32, 32, 3, 3, 1, 1, 1, groups=32, **_I8),
        LayerSpec("pw1x1_32to64_96", 1, 96, 96, 32, 64, 1, 1, 1, 0, 0, **_I8),
        LayerSpec("conv3x3_64to64_96", 1, 96, 96, 64, 64, 3, 3, 1, 1, 1, **_I8),
    ],
    # YOLOv4-style bf16 layers on a 4x320 mosaic.
    "yolov4_m640_bf16": [
        LayerSpec("stem3x3_3to32_640", 1, 640, 640, 3, 32, 3, 3, 1, 1, 1,
                  **{**_YOLO, "x_dist": ("mosaic", 320)}),
        LayerSpec("conv3x3s2_32to64_640", 1, 640, 640, 32, 64, 3, 3, 2, 1, 1, **_YOLO),
        LayerSpec("pw1x1_128to64_160", 1, 160, 160, 128, 64, 1, 1, 1, 0, 0, **_YOLO),
        LayerSpec("conv3x3s2_256to512_80", 1, 80, 80, 256, 512, 3, 3, 2, 1, 1, **_YOLO),
    ],
    # bf16 throughput sweep at batch 8.
    "sweep_b8_bf16": [
        LayerSpec("conv3x3_64to128_160", 8, 160, 160, 64, 128, 3, 3, 1, 1, 1, **_SWEEP),
        LayerSpec("conv3x3_256to256_80", 8, 80, 80, 256, 256, 3, 3, 1, 1, 1, **_SWEEP),
        LayerSpec("conv3x3_512to1024_40", 8, 40, 40, 512, 1024, 3, 3, 1, 1, 1, **_SWEEP),
        LayerSpec("pw1x1_1024to512_20", 8, 20, 20, 1024, 512, 1, 1, 1, 0, 0, **_SWEEP),
        LayerSpec("dw3x3_512_40", 8, 40, 40, 512, 512, 3, 3, 1, 1, 1, groups=512, **_SWEEP),
    ],
}

SEEDS = {"mnist_conv3x3_f32": 0, "kws_dscnn_f32": 1, "vww_int8": 2,
         "yolov4_m640_bf16": 3, "sweep_b8_bf16": 4}


def spec_by_name(name: str) -> tuple[str, LayerSpec]:
    for cfg, specs in CONFIGS.items():
        for s in specs:
            if s.name == name:
                return cfg, s
    raise KeyError(name)


def _draw(shape, dist, g, fan_in):
    kind = dist[0]
    if kind == "uniform":
        lo, hi = dist[1], dist[2]
        return torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo
    if kind == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32) * dist[1]
    if kind == "he":
        return torch.randn(shape, generator=g, dtype=torch.float32) * math.sqrt(2.0 / fan_in)
    if kind == "int":
        return torch.randint(dist[1], dist[2] + 1, shape, generator=g, dtype=torch.int64)
    raise ValueError(dist)


def _mosaic(s: LayerSpec, g) -> torch.Tensor:
    """Four tiles A, B, C, D of size t x t drawn in that order from U(0, 1)
    and placed top-left, top-right, bottom-left, bottom-right of a 2t x 2t
    canvas ("YOLOv4, optimized for Wormhole", section 4, the 4x320 mosaic)."""
    t = s.x_dist[1]
    assert s.h == 2 * t and s.w == 2 * t
    tiles = [torch.rand((s.n, t, t, s.cin), generator=g, dtype=torch.float32) for _ in range(4)]
    x = torch.empty((s.n, s.h, s.w, s.cin), dtype=torch.float32)
    x[:, :t, :t] = tiles[0]
    x[:, :t, t:] = tiles[1]
    x[:, t:, :t] = tiles[2]
    x[:, t:, t:] = tiles[3]
    return x


def _cast(t: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return t.to(torch.float32)
    if dtype == "bf16":
        return t.to(torch.float32).to(torch.bfloat16)
    if dtype == "i8":
        return t.to(torch.int8)
    raise ValueError(dtype)


def make_layer(s: LayerSpec, g: torch.Generator) -> LayerData:
    """Draw x, w, b (and int8 scales) for one layer from generator ``g``."""
    cpg = s.cin // s.groups
    fan_in = s.kh * s.kw * cpg
    xshape = (s.n, s.h, s.w, s.cin)
    wshape = (s.cout, s.kh, s.kw, cpg)
    if s.x_dist[0] == "mosaic":
        x = _mosaic(s, g)
    else:
        x = _draw(xshape, s.x_dist, g, fan_in)
    w = _draw(wshape, s.w_dist, g, fan_in)
    b = None
    if s.b_dist is not None:
        b = _draw((s.cout,), s.b_dist, g, fan_in)
        b = b.to(torch.int32) if s.dtype == "i8" else b.to(torch.float32)
    ws = None
    if s.dtype == "i8" and s.ws_dist[0] == "pow2":
        # s_w = 2^e with integer e drawn uniformly from [lo, hi]: scales whose
        # multipliers are exact in float, so that requantisation ties occur
        e = torch.randint(s.ws_dist[1], s.ws_dist[2] + 1, (s.cout,), generator=g, dtype=torch.int64)
        ws = torch.pow(2.0, e.to(torch.float64)).to(torch.float32)
    elif s.dtype == "i8":
        lo, hi = s.ws_dist[1], s.ws_dist[2]
        ws = torch.rand((s.cout,), generator=g, dtype=torch.float32) * (hi - lo) + lo
    return LayerData(s, _cast(x, s.dtype), _cast(w, s.dtype), b, ws)


def make_layer_device_x(s: LayerSpec, seed: int, device) -> LayerData:
    """As make_layer, but x is drawn on ``device`` by a generator of that
    device seeded with ``seed`` (for inputs too large to draw on the host):
    uniform x_dist only, or int U[lo, hi] for int8.  w, b (and int8 scales)
    are drawn on the host from a CPU generator seeded with ``seed``."""
    g = torch.Generator("cpu").manual_seed(seed)
    gd = torch.Generator(device=device).manual_seed(seed)
    xshape = (s.n, s.h, s.w, s.cin)
    kind = s.x_dist[0]
    if kind == "uniform":
        lo, hi = s.x_dist[1], s.x_dist[2]
        x = torch.rand(xshape, generator=gd, device=device, dtype=torch.float32).mul_(hi - lo).add_(lo)
    elif kind == "int":
        x = torch.randint(s.x_dist[1], s.x_dist[2] + 1, xshape, generator=gd, device=device, dtype=torch.int16)
    else:
        raise ValueError(f"device draw of {kind!r} inputs is not offered")
    x = _cast(x, s.dtype)
    d = make_layer(replace(s, n=0), g)  # w, b, scales only (x of an empty batch)
    return LayerData(s, x, d.w, d.b, d.w_scales)


def generate(config: str, layers: list[str] | None = None) -> list[LayerData]:
    """All layers of a layer set, drawn in order from the set's seed.  With
    ``layers``, only those are returned (the others are still drawn, so each
    layer's tensors do not depend on which subset was asked for)."""
    g = torch.Generator("cpu").manual_seed(SEEDS[config])
    out = []
    for s in CONFIGS[config]:
        d = make_layer(s, g)
        if layers is None or s.name in layers:
            out.append(d)
    return out


def scaled(s: LayerSpec, **kw) -> LayerSpec:
    """A copy of a layer spec with some fields changed (smaller parity cases)."""
    return replace(s, **kw)
