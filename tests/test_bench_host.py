"""Host-side pieces of bench.py that its reported numbers rest on: the
algorithmic work per launch (the numerator of every roofline fraction) and
the rule that a captured DRAM traffic figure is reported only while the
kernel sources it was captured from are unchanged."""
import dataclasses
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_moe_ffn_gb300.inputs import CONFIGS  # noqa: E402


def test_decode_gate_up_bytes_match_the_profile():
    """Decode (N=64, H=2048, E=128, top-8, I=768) with 127 experts touched:
    Wg and Wu of the touched experts, x once, and the activation written
    once -- 800,063,488 bytes, the figure the decode profile quotes as
    800.1 MB of algorithmic bytes."""
    b, f, _, _ = bench.algorithmic_work(CONFIGS["decode"], 127)
    assert b["gate_up"] == 127 * (2 * 768 * 2048 * 2) + 64 * 2048 * 2 + 512 * 768 * 2
    assert b["gate_up"] == 800_063_488
    # down: Wd of the touched experts, the activation, the pair outputs at
    # bf16 size and the routing weights
    assert b["down"] == 127 * 2048 * 768 * 2 + 512 * 768 * 2 + 512 * 2048 * 2 + 512 * 4
    assert b["down"] == 402_393_088


def test_prefill_gemm_flops():
    """Prefill: 65,536 pairs; gate/up 4·H·I·P and down 2·H·I·P FLOP, 618.5
    GFLOP for the two grouped GEMMs of a call."""
    _, f, layer, _ = bench.algorithmic_work(CONFIGS["prefill"], 128)
    P = 8192 * 8
    assert f["gate_up"] == 4 * 2048 * 768 * P == 412_316_860_416
    assert f["down"] == 2 * 2048 * 768 * P
    assert f["gate_up"] + f["down"] == 618_475_290_624
    assert layer == 2 * 8192 * 2048 * 128 + 6 * 2048 * 768 * P


def test_shared_expert_work_is_counted_in_the_grouped_gemms():
    """Talker: the shared expert's chunks run inside gate/up and down, so
    their weights and FLOPs are counted there and the shared stage has none."""
    t = CONFIGS["talker"]
    b, f, _, _ = bench.algorithmic_work(t, t.E)
    b0, f0, _, _ = bench.algorithmic_work(dataclasses.replace(t, I_s=0), t.E)
    assert b["shared"] == 0 and f["shared"] == 0
    assert f["gate_up"] - f0["gate_up"] == 4 * t.H * t.I_s * t.N
    assert f["down"] - f0["down"] == 2 * t.H * t.I_s * t.N
    assert b["gate_up"] - b0["gate_up"] == 2 * t.I_s * t.H * 2 + t.N * t.I_s * 2
    # the shared expert's down weights, its activation and its output rows
    assert b["down"] - b0["down"] == t.I_s * t.H * 2 + t.N * t.I_s * 2 + t.N * t.H * 2


def test_captured_traffic_is_reported_only_for_unchanged_sources(monkeypatch):
    """profiles/traffic.json holds one record per stage and workload with the
    hash of the sources it was captured from; a changed source makes the
    bench report null instead of a stale figure."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)
    entry = rec["decode/gate_up"]
    assert entry["bytes_per_launch"] == entry["read"] + entry["write"]
    assert bench.measured_traffic("gate_up", "decode") == entry["bytes_per_launch"]
    monkeypatch.setattr(bench, "source_hash", lambda stage: "not-the-captured-sources")
    assert bench.measured_traffic("gate_up", "decode") is None


def test_max_over_ranks_is_the_identity_on_one_rank():
    assert bench.max_over_ranks(1.25, 1, None) == 1.25
