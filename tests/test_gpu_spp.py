"""GPU parity of the SPP block (conv_spp_run): the cascaded 5/9/13 max pools
against the oracle's direct evaluation of every window, bit-exact in every
dtype, written into channel slices of a wider y whose other channels must
stay untouched."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # (name, n, h, w, c, dtype, y_channels, off5, off9, off13, off_x)
    ("yolov4_m640_20x20x512", 1, 20, 20, 512, "bf16", 2048, 0, 512, 1024, 1536),
    ("yolov4_m640_b8", 8, 20, 20, 512, "bf16", 2048, 0, 512, 1024, 1536),
    ("whole_image_51x51_c8", 1, 51, 51, 8, "bf16", 32, 8, 16, 24, 0),  # ~10 elements a thread
    ("yolov4_320_10x10x512_darknet_order", 1, 10, 10, 512, "bf16", 2048, 1024, 512, 0, 1536),
    ("ragged_f32_b2", 2, 7, 11, 24, "f32", 112, 8, 36, 64, 88),
    ("i8_13x9x48_no_copy", 1, 13, 9, 48, "i8", 192, 16, 80, 144, -1),
    ("single_pixel", 1, 1, 1, 8, "bf16", 32, 0, 8, 16, 24),
    ("wide_image_c8", 2, 3, 40, 8, "bf16", 48, 8, 16, 32, 0),
    # images too large for the whole-image kernel: 8x8 tiles with a 6-pixel halo
    ("tiled_80x80x64", 1, 80, 80, 64, "bf16", 256, 0, 64, 128, 192),
    ("tiled_i8_b2_57x61x32", 2, 57, 61, 32, "i8", 128, 96, 64, 32, 0),
]
DT = {"f32": torch.float32, "bf16": torch.bfloat16, "i8": torch.int8}


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_spp_exact(case):
    import convolution_nhwc_implicit_gb300 as cl
    name, n, h, w, c, dt, cy, o5, o9, o13, ox = case
    g = torch.Generator("cpu").manual_seed(11)
    if dt == "i8":
        x = torch.randint(-128, 128, (n, h, w, c), generator=g, dtype=torch.int8)
    else:
        x = torch.randn(n, h, w, c, generator=g).to(DT[dt])
    dev = torch.device("cuda:0")
    esz = x.element_size()
    buf = torch.full((n * h * w * cy * esz + 4096,), 0x7F, dtype=torch.uint8, device=dev)
    y = buf[: n * h * w * cy * esz].view(DT[dt]).view(n, h, w, cy)
    cl.spp(x.to(dev), y, cy, o5, o9, o13, ox)
    torch.cuda.synchronize()
    assert bool((buf[n * h * w * cy * esz:] == 0x7F).all()), "wrote past the end of y"
    got = y.cpu()
    xd = x.to(torch.float64).numpy() if dt != "i8" else x.numpy().astype(np.float64)
    for off, ref in zip((o5, o9, o13), oracle.spp(xd)):
        sl = got[..., off:off + c]
        sl = sl.to(torch.float64).numpy() if dt != "i8" else sl.numpy().astype(np.float64)
        assert np.array_equal(sl, ref), f"{name}: pooled slice at {off} differs"
    used = np.zeros(cy * esz, dtype=bool)
    for off in (o5, o9, o13) + ((ox,) if ox >= 0 else ()):
        used[off * esz:(off + c) * esz] = True
    if ox >= 0:
        assert torch.equal(got[..., ox:ox + c], x)
    raw = buf[: n * h * w * cy * esz].view(n, h, w, cy * esz).cpu().numpy()
    assert (raw[..., ~used] == 0x7F).all(), "wrote outside the slices"
