"""Host-side tests of bench.py (no GPU): the byte model, the traffic records and the
reference arm's JSON line.

The byte model is the roofline numerator, so it is checked against brute-force counts
of the oracle's kept ranges and against the closed forms the definitions give.
"""
import dataclasses
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench
import oracle
import seeded_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _brute_kept(S, L, mask_kind, window):
    """Kept elements of one slice, counted from the oracle's per-row kept ranges."""
    c0, c1 = oracle.kept_ranges(np.array([L], dtype=np.int32), S, mask_kind, window)
    return int(np.maximum(c1 - c0, 0).sum())


@pytest.mark.parametrize("mask_kind,window", [(0, 0), (1, 0), (2, 1), (2, 7), (2, 64), (2, 1000)])
def test_kept_per_slice_matches_brute_force(mask_kind, window):
    S = 97
    w = dataclasses.replace(si.custom("kept", 1, 1, S, "f32", 1.0, seq_lens=(S,)), mask_kind=mask_kind,
                            window=window)
    for L in (-3, 0, 1, 2, 13, 50, 96, 97, 120):
        assert bench.kept_per_slice(w, L) == _brute_kept(S, L, mask_kind, window), (L, mask_kind, window)


def test_required_bytes_closed_forms():
    # the printed worked example: X[3,2,5,5] fp32, seq_lens 3, 4, 5 -> 4 * 2 * (6 + 10 + 15 + 3 * 25) bytes
    w = si.WORKLOADS["worked_example"]
    fwd, bwd = bench.required_bytes(w, si.seq_lens(w))
    assert fwd == 848 and bwd == 0
    # grouped tril, forward e * sum(live + S^2), backward e * sum(2 live + S^2)
    w = si.custom("rb", 2, 3, 10, "bf16", 0.5, seq_lens=(4, 10))
    live = 3 * (4 * 5 // 2 + 10 * 11 // 2)
    assert bench.required_bytes(w, si.seq_lens(w)) == (2 * (live + 6 * 100), 2 * (2 * live + 6 * 100))
    # an explicit mask counts its kept elements and its uint8 [B, S, S] bytes once
    we = si.WORKLOADS["explicit_s2048_bf16"]
    fb, bb = bench.required_bytes(we, si.seq_lens(we), kept_total=1000)
    dense = we.B * we.M * we.S * we.S
    assert fb == 2 * (1000 + dense) + we.B * we.S * we.S
    assert bb == 2 * (2000 + dense) + we.B * we.S * we.S


def test_traffic_records_are_keyed_by_kernel_workload_and_sources():
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    lines = [ln for ln in open(path, encoding="utf-8") if ln.startswith("traffic ")]
    assert lines
    for ln in lines:
        kv = dict(tok.split("=", 1) for tok in ln.split()[1:])
        got = bench.recorded_traffic(kv["kernel"], kv["workload"])
        if kv["source_sha"] == bench.kernel_source_sha(kv["kernel"]):
            assert got == int(kv["dram_bytes_per_launch"])
        else:
            assert got is None
        # a direct capture of the workload itself: read + write, within a few % of the algorithmic bytes
        assert kv["captured_on"] == kv["workload"]
        assert int(kv["dram_read"]) + int(kv["dram_write"]) == int(kv["dram_bytes_per_launch"])
        assert 0.9 < int(kv["dram_bytes_per_launch"]) / int(kv["algorithmic_bytes"]) < 1.1
    assert bench.recorded_traffic("gtms_no_such_kernel", "s1000_b12") is None


def test_kernel_source_families():
    import glob

    csrc = os.path.join(ROOT, "masked_softmax_attention_gb300", "csrc")
    attn = bench.kernel_sources("gtms_attn_dscores_tma_kernel<bf16,d64>")
    assert "gtms_attn_tma.cuh" in attn and "gtms_tcgen05.cuh" in attn and "gtms_stream.cuh" not in attn
    vec = bench.kernel_sources("gtms_bwd_vec_kernel<f32,team32,x8,minb5>")
    assert "gtms_kernels.cuh" in vec and "gtms_stream.cuh" not in vec
    assert "gtms_stream.cuh" in bench.kernel_sources("gtms_fwd_stream_kernel<bf16,team256,x4,minb4>")
    # every listed file exists, so that a rename cannot silently drop it from the hash
    for k in ("gtms_attn_dscores_tma_kernel<bf16,d64>", "gtms_fwd_explicit_kernel<bf16,team64,x4,minb12>",
              "gtms_fwd_stream_kernel<bf16,team256,x4,minb4>", "gtms_fwd_band_kernel<bf16,x2,minb8>",
              "gtms_fwd_vec_kernel<f32,team64,x4,minb0>"):
        for f in bench.kernel_sources(k):
            assert os.path.exists(os.path.join(csrc, f)), f
    assert glob.glob(os.path.join(csrc, "*.cuh"))
    assert bench.kernel_source_sha("gtms_attn_dscores_tma_kernel<bf16,d64>") != bench.kernel_source_sha(
        "gtms_bwd_vec_kernel<f32,team32,x8,minb5>")


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "worked_example", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["config"]["workload"].startswith("worked_example")


def test_fewer_than_three_warmup_steps_are_refused():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "worked_example", "--steps", "1", "--warmup", "2"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0


def test_touched_bytes_count_whole_units_with_a_kept_element():
    """The explicit-mask byte model at 16-byte granularity, against a brute-force count of the units
    that hold a kept element (bf16: 8 elements per unit), the mask and every output."""
    w = dataclasses.replace(si.WORKLOADS["explicit_s2048_bf16"], B=2, M=3, S=64)
    m = si.make_keep_mask(w, "cpu")
    units = sum(int(m[b, r, 8 * j:8 * j + 8].any()) for b in range(w.B) for r in range(w.S) for j in range(w.S // 8))
    dense = w.B * w.M * w.S * w.S * 2
    fwd, bwd = bench.touched_bytes(w, m)
    assert fwd == 16 * w.M * units + w.B * w.S * w.S + dense
    assert bwd == 32 * w.M * units + w.B * w.S * w.S + dense
    # never below the kept-element model: a unit read whole holds at least its kept elements
    kept = int(m.count_nonzero()) * w.M
    rf, rb = bench.required_bytes(w, si.seq_lens(w), kept)
    assert fwd >= rf and bwd >= rb
