"""Host-side logic of bench.py that needs no GPU: the algorithmic-byte model behind
the roofline's numerator, and the clock record that decides whether a run stands.

The per-layer byte counts are written out from the workloads' shapes (batch,
kv heads, stored tokens, head_dim) and the storage formats: 4-bit codes are
D/2 bytes a token, 8-bit codes D bytes, an fp16 scale and zero 4 bytes per
group, a Q4_0 block one fp16 scale per 32 channels, KIVI per-channel keys one
fp16 scale and zero per channel, and Q plus O one row per query head.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402
from oracle import accounting  # noqa: E402


def _io_bytes(w):
    return {"float32": 4, "bfloat16": 2, "float16": 2}[w.io_dtype]


# (workload, stored tokens T, per-layer bytes written out by hand from the shapes)
PER_LAYER = [
    # tinygpt: B1, 8 heads, D32, T = 4 + 256. int8 K and V codes; K per-channel fp16 scale+zero;
    # V per-token fp16 scale+zero; fp32 Q and O.
    ("tinygpt", 260, 8 * 260 * 32 * 2 + 8 * 32 * 4 + 8 * 260 * 4 + 2 * 8 * 32 * 4),
    # mlx g64 4-bit: B1, Hkv 8, Hq 24, D128, T 8192. K and V: 64 code bytes + 2 groups x 4 B a token.
    ("mlx8k", 8192, 2 * 8 * 8192 * (64 + 8) + 2 * 24 * 128 * 2),
    # Q4_0 K + int8 V: B8, Hkv 8, Hq 32, T 32768. K: 64 code bytes + 4 fp16 block scales;
    # V: 128 code bytes + one fp16 scale and zero a token.
    ("q4_0_32k", 32768, 8 * 8 * 32768 * (64 + 8 + 128 + 4) + 2 * 8 * 32 * 128 * 2),
    # KIVI int4 ring 4 + 4096: B64, Hkv 8, Hq 32. K: 64 code bytes a token + per-channel 128 x 4 B;
    # V g32: 64 code bytes + 4 groups x 4 B a token.
    ("ring", 4100, 64 * 8 * (4100 * (64 + 64 + 16) + 128 * 4) + 2 * 64 * 32 * 128 * 2),
]


@pytest.mark.parametrize("name,T,expected", PER_LAYER)
def test_decode_bytes_closed_form(name, T, expected):
    w = synth.get_workload(name)
    assert bench.decode_bytes(w, T) == expected


def test_decode_bytes_per_step_totals():
    """Whole-step figures (every layer) of the 8K, 32K and streaming workloads."""
    totals = {name: synth.get_workload(name).layers * expected for name, _, expected in PER_LAYER}
    assert totals["tinygpt"] == 144_512
    assert totals["mlx8k"] == 264_585_216
    assert totals["q4_0_32k"] == 13_694_402_560
    assert totals["ring"] == 9_715_056_640


@pytest.mark.parametrize("name,T,expected", PER_LAYER)
def test_decode_bytes_agrees_with_oracle_accounting(name, T, expected):
    w = synth.get_workload(name)
    got = accounting.decode_read_bytes(w.batch, w.n_kv_heads, w.n_q_heads, w.head_dim, T,
                                       w.k_format, w.k_bits, w.k_group,
                                       w.v_format, w.v_bits, w.v_group if w.v_group < w.head_dim else w.head_dim,
                                       _io_bytes(w))
    assert got == bench.decode_bytes(w, T) == expected


def test_residual_buffer_bytes():
    """Residual buffer of 128-token K blocks: closed blocks as 4-bit codes plus a per-(block, channel)
    fp16 scale and zero; the T mod 128 tail as fp32 K and V rows; V g32 as in the ring workload."""
    w = synth.get_workload("residual")
    T = 8292                     # 64 closed blocks + a 100-row tail
    closed, tail = 64 * 128, 100
    per_head = closed * (64 + 64 + 16) + 64 * 128 * 4 + tail * 128 * 8
    assert bench.decode_bytes(w, T) == 8 * per_head + 2 * 24 * 128 * 2


def test_stored_after_streaming_cap():
    ring = synth.get_workload("ring")
    for t in (1, 4100, 4101, 40_000 + 4100):
        assert bench.stored_after(ring, t) == min(t, 4100)
    lin = synth.get_workload("mlx8k")
    assert bench.stored_after(lin, 8193) == 8193


FAKE_SMI = """\
2070, 2070, 120.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
1965, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active
1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active
2010, 2070, 1310.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
malformed line
"""


def test_clock_summary_reads_reasons_and_loaded_median():
    s = bench.ClockSampler.summarize(FAKE_SMI)
    assert s["samples"] == 4
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == 1980.0       # median of the three samples drawing > 30% of the peak power
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_flags_thermal_slowdown_and_empty_log():
    hot = "1500, 2070, 1300.0, 0x20, Not Active, Active, Not Active, Not Active\n"
    assert bench.ClockSampler.summarize(hot)["reasons"] == ["hw_thermal_slowdown"]
    assert bench.ClockSampler.summarize("") is None


def test_peaks_come_from_the_measured_file():
    peak, kind = bench.read_peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured" and peak > 1000.0
    else:
        assert (peak, kind) == (6800.0, "fallback")


@pytest.mark.parametrize("S,budget,n_sink", [(200, 24, 4), (64, 64, 4), (64, 100, 0), (300, 17, 0)])
def test_coverage_stats_match_the_oracle(S, budget, n_sink):
    # the bench reports SnapKV coverage with its own torch arithmetic on the
    # device's scores and indices; it must agree with the oracle's definitions
    import numpy as np
    import torch

    from oracle import snapkv as osk

    rng = np.random.default_rng(S + budget)
    sc = rng.random((2, 3, S)) ** 4
    idx = np.stack([np.stack([osk.select_indices(sc[b, h], budget, n_sink) for h in range(3)]) for b in range(2)])
    kept, rnd = bench.coverage_stats(torch.from_numpy(sc).float(), torch.from_numpy(idx), budget, n_sink)
    sc32 = sc.astype(np.float32).astype(np.float64)          # the bench sees fp32 scores
    ref_kept = np.mean([osk.coverage(sc32[b, h], idx[b, h]) for b in range(2) for h in range(3)])
    ref_rnd = np.mean([osk.random_coverage(sc32[b, h], budget, n_sink) for b in range(2) for h in range(3)])
    assert kept == pytest.approx(ref_kept, rel=1e-12) and rnd == pytest.approx(ref_rnd, rel=1e-12)
    if budget >= S:
        assert kept == pytest.approx(1.0) and rnd == 1.0
    else:
        assert kept > rnd


@pytest.mark.parametrize("name", ["tinygpt", "mlx8k", "q4_0_32k", "snapkv", "ring", "residual"])
def test_reference_arm_line(name, capsys):
    # `bench.py --impl reference`: the oracle on a bounded sample of the workload, one JSON line
    import json

    a = bench.parse_args(["--impl", "reference", "--workload", name, "--steps", "1", "--warmup", "1"])
    assert a.warmup == 3                                   # at least three warm-up steps, always
    bench.run_reference(a, 0, 1)
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    w = synth.get_workload(name)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["config"]["workload"] == w.name
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"], d["scaling"], d["data"]) == (1, 1, 3, "weak", "synthetic")
    assert d["vs_baseline"] is None and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["value"] == d["value"] and cb["unit"] == "GB/s" and cb["kind"] == "oracle" and cb["cores"] == 1
    assert cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_cpu_baseline_one_thread_and_all_cores():
    # the oracle timed on one thread and in spawned processes, one per core (two here, to keep the
    # test short), with the core count and the CPU model stated
    w = synth.get_workload("tinygpt")
    cb = bench.cpu_baseline(w, 0.3, nproc=2)
    assert cb["cores"] == 1 and cb["kind"] == "oracle" and cb["value"] > 0 and cb["unit"] == "GB/s"
    assert cb["nproc"] == 2 and isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    ac = cb["all_cores"]
    assert ac["cores"] == 2 and ac["value"] > 0 and ac["unit"] == "GB/s" and "2 processes" in ac["sample"]


def test_every_workload_has_a_traffic_entry_on_the_current_sources():
    # the committed ncu DRAM figures hold for the kernel sources they were taken on:
    # every bench workload has one, and each matches the files as they are now
    kd = os.path.join(ROOT, "bit_kv_cache_quant_gb300")
    for w in synth.WORKLOADS.values():
        t = bench.profile_traffic(w.name, kd)
        assert t is not None and t > 0, f"{w.name}: no DRAM traffic for the current sources"
    assert bench.profile_traffic("no_such_workload", kd) is None


def test_traffic_entry_goes_null_when_a_kernel_source_changes(tmp_path):
    import shutil

    kd = os.path.join(ROOT, "bit_kv_cache_quant_gb300")
    copy = tmp_path / "pkg"
    shutil.copytree(os.path.join(kd, "csrc"), copy / "csrc")
    name = "llama3b_mlx_affine4_g64_ctx8k"
    assert bench.profile_traffic(name, str(copy)) == bench.profile_traffic(name, kd)
    with open(copy / "csrc" / "decode_tc.cuh", "a") as f:
        f.write("\n// edited\n")
    assert bench.profile_traffic(name, str(copy)) is None
    # the SnapKV entry keys a different set of files
    assert bench.profile_traffic("snapkv_s16k_budget512_fp16", str(copy)) is not None
