"""bench.py's host-side post-processing on CPU: the inputs it keeps for the
oracle baselines and the baselines attached to each workload's line (tiny
stand-in shapes, short samples); no GPU involved."""

import json

import numpy as np

import bench
from w4a16_nvfp4_weight_gb300 import synth


def test_host_cases_accept_launches_without_awq_bits():
    r = synth.rng(1)
    decode_like = dict(M=1, K=64, N=256, x_bits=synth.normal_act(r, (1, 64), "bf16"))
    dense_like = dict(M=2, K=64, N=256, x_bits=synth.normal_act(r, (2, 64), "bf16"),
                      pqs_bits=synth.awq_scale_bits(r, 64))
    cases = bench.host_cases([decode_like, dense_like])
    assert cases[0][4] is None and cases[1][4] is dense_like["pqs_bits"]
    assert [c[:3] for c in cases] == [(1, 64, 256), (2, 64, 256)]


def test_attach_cpu_baselines_for_every_workload(monkeypatch):
    monkeypatch.setattr(bench, "DECODE_SHAPES", [(64, 256), (128, 320)])
    monkeypatch.setattr(bench, "DECODE_M", [1, 3])
    out = bench.attach_cpu_baselines({"value": 1.0, "_base": None}, "decode", 1, False, seconds=0.2)
    assert out["cpu_baseline"]["value"] > 0 and out["cpu_baseline"]["cores"] == 1
    assert out["cpu_baseline_all_cores"]["value"] > 0 and out["cpu_baseline_all_cores"]["cores"] >= 1
    json.dumps(out)

    r = synth.rng(2)
    base = {(64, 48): (None,) + tuple(synth.weight_only(64, 48, 3))}
    cases = [(3, 64, 48, synth.normal_act(r, (3, 64), "bf16"), None),
             (5, 64, 48, synth.normal_act(r, (5, 64), "bf16"), synth.awq_scale_bits(r, 64))]
    for wl, unit in (("prefill", "TFLOP/s"), ("lmhead", "GB/s"), ("tails", "GB/s"), ("toy", "GB/s")):
        res = {"value": 1.0, "_base": base, "_cases": cases}
        out = bench.attach_cpu_baselines(res, wl, 1, False, seconds=0.1)
        assert out["cpu_baseline"]["unit"] == unit and out["cpu_baseline"]["value"] > 0
        assert "_base" not in out and "_cases" not in out
        json.dumps(out)

    monkeypatch.setattr(bench, "MOE_TOPK", 2)
    monkeypatch.setattr(bench, "MOE_H", 128)
    monkeypatch.setattr(bench, "MOE_I", 64)
    fc1, fc2 = synth.moe_weights(8, 128, 64, 7)
    case = synth.moe_case(1, 9, E=8, topk=2, H=128, I=64, weights=(fc1, fc2))
    out = bench.attach_cpu_baselines({"value": 1.0, "_base": None, "_moe": (fc1, fc2, case)}, "moe", 1, False,
                                     seconds=0.1)
    assert out["cpu_baseline"]["unit"] == "GB/s" and "_moe" not in out
    json.dumps(out)

    # the dense MLP line has no oracle sample; skipped or multi-rank runs only drop the host data
    out = bench.attach_cpu_baselines({"value": 1.0, "_base": None}, "mlp", 1, False, seconds=0.1)
    assert "cpu_baseline" not in out
    for world, skip in ((2, False), (1, True)):
        res = {"value": 1.0, "_base": base, "_cases": cases}
        out = bench.attach_cpu_baselines(res, "prefill", world, skip)
        assert "cpu_baseline" not in out and "_cases" not in out


def test_traffic_ratio_needs_a_matching_capture(tmp_path, monkeypatch):
    """The roofline's traffic comes from a committed capture record only while
    the kernel's sources still hash to the value the record holds."""
    rec = tmp_path / "rec.json"
    sha = bench.kernel_sources_sha(["common.cuh"])
    rec.write_text(json.dumps({"traffic_ratio": 1.01, "kernel_sources_sha": sha}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "PROFILE_FOR", {"decode": ("rec.json", ["common.cuh"])})
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda srcs: sha)
    assert bench.traffic_ratio("decode") == (1.01, "rec.json")
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda srcs: "different")
    ratio, why = bench.traffic_ratio("decode")
    assert ratio is None and "changed" in why
    monkeypatch.setattr(bench, "PROFILE_FOR", {"decode": ("missing.json", ["common.cuh"])})
    assert bench.traffic_ratio("decode")[0] is None
