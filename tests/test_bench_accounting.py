"""The benchmark's FLOP and byte accounting and its roofline arithmetic (host only).

* The conv_out head's arithmetic intensity is the one the FastVideo head.cu page states in its header
  comment: 256 x 27 MACs per output channel and position over a per-position input window of
  6912 x 2 bytes, 12 FLOP per byte of that window.
* The per-stage FLOP and byte counts the benchmark divides by are the sums over the layers it actually
  runs (``bench.layer_descs()``), counted here from each descriptor: every output position of every
  output channel takes C_in x taps MACs (the zero-padded taps included); a layer reads its input once
  (with its two carried frames when causal) and its weights and bias, and writes its output once.
* ``roof_entry``: t_roof = max(bytes / HBM peak, FLOP / tensor peak) and frac = t_roof / t_measured.
"""
import pytest

import bench


def _out_hw(d):
    s = d.get("stride", 1)
    return (d["H"] - 1) // s + 1, (d["W"] - 1) // s + 1


def _layer_flop(d):
    Ho, Wo = _out_hw(d)
    taps = 27 if d["dims"] == 3 else 9
    frames = d["N"] * (d.get("D", 1) if d["dims"] == 3 else 1)
    return 2.0 * frames * Ho * Wo * d["C_out"] * d["C_in"] * taps


def _layer_bytes(d):
    Ho, Wo = _out_hw(d)
    taps = 27 if d["dims"] == 3 else 9
    in_frames = d["N"] * ((d.get("D", 1) + 2) if d["dims"] == 3 else 1)
    out_frames = d["N"] * (d.get("D", 1) if d["dims"] == 3 else 1)
    return 2.0 * (in_frames * d["H"] * d["W"] * d["C_in"] + out_frames * Ho * Wo * d["C_out"] +
                  d["C_out"] * d["C_in"] * taps + d["C_out"])


def test_head_intensity_is_the_pages():
    flop, _ = bench.stage_cost()
    positions = 4 * 352 * 624
    macs_per_output = flop["head"] / 2 / positions / 12
    assert macs_per_output == 256 * 27
    assert flop["head"] / positions / (6912 * 2) == pytest.approx(12.0)


@pytest.mark.parametrize("stage", bench.STAGES)
def test_stage_costs_are_the_sums_over_the_layers_run(stage):
    flop, nbytes = bench.stage_cost()
    descs = bench.layer_descs()[stage]
    descs = descs if isinstance(descs, list) else [descs]
    assert flop[stage] == pytest.approx(sum(_layer_flop(d) for d in descs), rel=1e-12)
    assert nbytes[stage] == pytest.approx(sum(_layer_bytes(d) for d in descs), rel=1e-12)


def test_roof_entry_arithmetic():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 2000.0}
    # 1 GB at 1000 GB/s = 1 ms; 1 TFLOP at 2000 TFLOP/s = 0.5 ms: bound by HBM; measured 2 ms
    e = bench.roof_entry(2.0, 1e12, 1e9, peaks, "t", frames=4)
    assert e["bound"] == "hbm" and e["t_roof_ms"] == pytest.approx(1.0)
    assert e["frac"] == pytest.approx(0.5) and e["frac_hbm"] == pytest.approx(0.5)
    assert e["frac_tensor"] == pytest.approx(0.25)
    assert e["tflops"] == pytest.approx(500.0) and e["gbs"] == pytest.approx(500.0)
    assert e["ms_per_frame"] == pytest.approx(0.5)
    # 4 TFLOP: 2 ms on the tensor pipe against 1 ms of HBM: tensor-bound, measured at the roof
    e = bench.roof_entry(2.0, 4e12, 1e9, peaks, "t")
    assert e["bound"] == "tensor" and e["frac"] == pytest.approx(1.0) and e["frac_tensor"] == pytest.approx(1.0)
