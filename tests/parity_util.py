"""Shared helpers of the GPU parity tests: run a layer through the C ABI and
through the oracle on the same seeded inputs, and compare.

Tolerances (elementwise, against the float64 / exact-int oracle):
  fp32 : |y - ref| <= 1e-5 * (1 + |ref|)   (FFMA, never TF32: TF32 would err by ~1e-3)
  bf16 : |y - ref| <= 1e-2 * (1 + |ref|)   (bf16 output rounding is 2^-9 relative)
  int8 : bit-exact
"""
import numpy as np
import torch

import oracle
from conv_workloads import LayerData, LayerSpec, output_hw

TOL = {"f32": 1e-5, "bf16": 1e-2}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "i8": torch.int8}
GUARD = 4096  # bytes of guard band after y


def to_np64(t):
    return t.to(torch.float64).numpy() if t.dtype != torch.int8 else t.numpy()


def make_plan(spec: LayerSpec, d: LayerData, algo="auto"):
    import convolution_nhwc_implicit_gb300 as cl
    quant = None
    if spec.dtype == "i8":
        quant = (spec.in_scale, spec.out_scale, d.w_scales.tolist())
    return cl.Plan(spec.n, spec.h, spec.w, spec.cin, spec.cout, spec.kh, spec.kw, spec.stride,
                   spec.pad_h, spec.pad_w, spec.groups, spec.dtype, spec.act, quant, algo)


def run_gpu(spec: LayerSpec, d: LayerData, algo="auto", plan=None, check_guard=True):
    """Runs the layer on cuda:0 and returns y on the CPU (poisoned output,
    guard band after it checked)."""
    plan = plan or make_plan(spec, d, algo)
    dev = torch.device("cuda:0")
    x = d.x.to(dev)
    w = d.w.to(dev)
    b = None if d.b is None else d.b.to(dev)
    oh, ow = output_hw(spec)
    numel = spec.n * oh * ow * spec.cout
    esz = torch.tensor([], dtype=TORCH_DT[spec.dtype]).element_size()
    # y followed by a guard band, both poisoned with 0x7f bytes (NaN-like for floats)
    buf = torch.full((numel * esz + GUARD,), 0x7F, dtype=torch.uint8, device=dev)
    y = buf[: numel * esz].view(TORCH_DT[spec.dtype]).view(spec.n, oh, ow, spec.cout)
    plan.run(x, w, b, y)
    plan.check_device_status()
    torch.cuda.synchronize()
    if check_guard:
        tail = buf[numel * esz:]
        assert bool((tail == 0x7F).all()), "kernel wrote past the end of y"
    return y.cpu(), plan


def run_oracle(spec: LayerSpec, d: LayerData, threads=0):
    if spec.dtype == "i8":
        M = oracle.requant_multipliers(spec.in_scale, spec.out_scale, d.w_scales.numpy())
        return oracle.conv_i8(d.x.numpy(), d.w.numpy(), None if d.b is None else d.b.numpy(), M,
                              spec.stride, spec.pad_h, spec.pad_w, spec.groups, spec.act == "relu",
                              threads)
    return oracle.conv_f64(to_np64(d.x), to_np64(d.w), None if d.b is None else to_np64(d.b),
                           spec.stride, spec.pad_h, spec.pad_w, spec.groups, spec.act, threads)


def run_oracle_points(spec: LayerSpec, d: LayerData, pts):
    if spec.dtype == "i8":
        M = oracle.requant_multipliers(spec.in_scale, spec.out_scale, d.w_scales.numpy())
        return oracle.conv_i8_points(d.x.numpy(), d.w.numpy(), None if d.b is None else d.b.numpy(), M,
                                     pts, spec.stride, spec.pad_h, spec.pad_w, spec.groups,
                                     spec.act == "relu")
    return oracle.conv_f64_points(to_np64(d.x), to_np64(d.w), None if d.b is None else to_np64(d.b),
                                  pts, spec.stride, spec.pad_h, spec.pad_w, spec.groups, spec.act)


def assert_close(spec: LayerSpec, y, ref, what=""):
    if spec.dtype == "i8":
        got = y.numpy() if isinstance(y, torch.Tensor) else y
        bad = np.argwhere(got != ref)
        assert bad.size == 0, f"{what}: {len(bad)} int8 mismatches, first at {bad[:5].tolist()}"
        return
    got = y.to(torch.float64).numpy() if isinstance(y, torch.Tensor) else np.asarray(y, np.float64)
    tol = TOL[spec.dtype]
    err = np.abs(got - ref)
    lim = tol * (1.0 + np.abs(ref))
    ok = err <= lim
    if not ok.all():
        idx = np.argwhere(~ok)
        i0 = tuple(idx[0])
        raise AssertionError(
            f"{what}: {len(idx)} of {ok.size} outside {tol}*(1+|ref|); first at {list(i0)}: "
            f"got {got[i0]!r} ref {ref[i0]!r}; max err {err.max():.3e}")


def sample_points(spec: LayerSpec, count, seed):
    """Random output points plus every corner / edge class (padding cases)."""
    oh, ow = output_hw(spec)
    rng = np.random.default_rng(seed)
    pts = np.stack([rng.integers(0, spec.n, count), rng.integers(0, oh, count),
                    rng.integers(0, ow, count), rng.integers(0, spec.cout, count)], axis=1)
    edges = []
    for n in {0, spec.n - 1}:
        for h in {0, 1, oh // 2, oh - 2, oh - 1}:
            for w in {0, 1, ow // 2, ow - 2, ow - 1}:
                for c in {0, spec.cout // 2, spec.cout - 1}:
                    if 0 <= h < oh and 0 <= w < ow:
                        edges.append((n, h, w, c))
    return np.concatenate([pts, np.array(edges)], axis=0).astype(np.int32)
