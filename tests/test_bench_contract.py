"""Host-side pieces of bench.py's measurement contract, on the CPU: the
roofline arithmetic (which roof binds a layer, against the ridge of the
measured peaks), the DRAM-traffic records committed under profiles/ (each
entry's algorithmic bytes and read + write sum consistent with the layer
set's definitions), and the rule that a traffic record is reported only
for the exact kernel configuration and sources it was captured on."""
import json
import os

import pytest

import bench
from conv_workloads import CONFIGS, LayerSpec, alg_bytes, macs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PEAKS = {"hbm_gbs": 6796.9, "bf16_tflops": 1903.8, "fp32_ffma_tflops": 80.5}


def test_flops_are_two_per_mac():
    s = LayerSpec("t", 2, 9, 7, 16, 32, 3, 3, 1, 1, 1)
    assert bench.flops_of(s) == 2.0 * macs(s)
    # a 3x3 stride-1 pad-1 layer: every output position sees 9 x Cin MACs per channel
    assert macs(s) == 2 * 9 * 7 * 32 * 9 * 16


@pytest.mark.parametrize("name,bound", [
    ("conv3x3_512to1024_40", "tensor"),   # ~2500 flop/B, far above the ridge (~280)
    ("conv3x3_64to128_160", "tensor"),
    ("dw3x3_512_40", "hbm"),              # 9 MACs per output: memory-bound
    ("pw1x1_1024to512_20", "tensor"),
])
def test_layer_bound_against_the_ridge(name, bound):
    spec = next(s for s in CONFIGS["sweep_b8_bf16"] if s.name == name)
    got, ai = bench.layer_bound(spec, PEAKS)
    assert got == bound
    ridge = PEAKS["bf16_tflops"] * 1e12 / (PEAKS["hbm_gbs"] * 1e9)
    assert (ai >= ridge) == (bound == "tensor")


def test_fp32_layers_take_the_ffma_roof():
    spec = CONFIGS["mnist_conv3x3_f32"][0]
    pk, roof = bench.compute_peak(spec, PEAKS)
    assert (pk, roof) == (PEAKS["fp32_ffma_tflops"], "alu")


def test_job_throughput_counts_every_rank():
    # 1 TFLOP a step on each of 2 ranks, 4 steps in 8 ms: 1000 TFLOP/s for the job
    assert bench.job_tflops(1e12, 2, 4, 8.0) == pytest.approx(1000.0)


def _records():
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        d = json.load(f)
    return {k: v for k, v in d.items() if not k.startswith("_")}


def test_traffic_records_match_the_layer_sets():
    recs = _records()
    assert "sweep_b8_bf16" in recs
    for wl, layers in recs.items():
        specs = {s.name: s for s in CONFIGS[wl]}
        for name, e in layers.items():
            assert name in specs, (wl, name)
            assert e["alg_bytes"] == alg_bytes(specs[name]), (wl, name)
            assert abs(e["bytes_per_launch"] - (e["dram_read"] + e["dram_write"])) <= 1, (wl, name)
            assert e["kernel"] and len(e.get("sources_sha1") or "0" * 40) == 40, (wl, name)
            # compulsory traffic: a launch reads at least its inputs once from
            # DRAM or finds them in L2, never more than a few times over
            assert 0 < e["bytes_per_launch"] < 4 * e["alg_bytes"], (wl, name)


def test_traffic_is_reported_only_for_the_captured_kernel():
    recs = _records()
    wl, layers = "sweep_b8_bf16", recs["sweep_b8_bf16"]
    name, e = next(iter(layers.items()))
    # another configuration of the same layer: no record
    assert bench._traffic_for(wl, name, e["kernel"] + " (another tile)") is None
    # an unknown layer or layer set: no record
    assert bench._traffic_for(wl, "no_such_layer", e["kernel"]) is None
    assert bench._traffic_for("no_such_set", name, e["kernel"]) is None
    # the captured configuration: the record, as long as its sources are unchanged
    got = bench._traffic_for(wl, name, e["kernel"])
    if e["sources_sha1"] == bench.kernel_sources_sha1(e["kernel"]):
        assert got == e["bytes_per_launch"]
    else:
        assert got is None


def test_rate_units_per_roof():
    # int8 layers on the tensor roof are reported in TOPS, bf16 in TFLOP/s,
    # memory-bound layers in GB/s against the HBM peak
    vww = {s.name: s for s in CONFIGS["vww_int8"]}
    ach, pk, unit, bound = bench.rate_of(vww["conv3x3_64to64_96"], 10.0, PEAKS)
    assert (unit, bound, pk) == ("TOPS", "tensor", PEAKS["bf16_tflops"])
    assert ach == pytest.approx(bench.flops_of(vww["conv3x3_64to64_96"]) / 10e-6 / 1e12)
    dw = next(s for s in CONFIGS["sweep_b8_bf16"] if s.name == "dw3x3_512_40")
    ach, pk, unit, bound = bench.rate_of(dw, 8.0, PEAKS)
    assert (unit, bound, pk) == ("GB/s", "hbm", PEAKS["hbm_gbs"])
    assert ach == pytest.approx(alg_bytes(dw) / 8e-6 / 1e9)


def test_layer_row_takes_its_fraction_from_the_time_in_the_step():
    class FakePlan:
        launches = 1

        def describe(self):
            return "fake"
    spec = next(s for s in CONFIGS["sweep_b8_bf16"] if s.name == "conv3x3_512to1024_40")
    meas = {"marginal_us": [70.0], "evented_us": [75.0], "cold_us": [72.0], "warm_us": [69.0]}
    row = bench.layer_row(spec, FakePlan(), meas, 0, PEAKS)
    assert row["us"] == 70.0 and row["us_alone_cold"] == 72.0
    assert row["frac"] == pytest.approx(bench.flops_of(spec) / 70e-6 / 1e12 / PEAKS["bf16_tflops"], rel=1e-3)
    assert row["frac_alone_cold"] < row["frac"]
    assert row["unit"] == "TFLOP/s" and row["bound"] == "tensor"
