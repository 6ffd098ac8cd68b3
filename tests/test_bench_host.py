"""The benchmark's host arithmetic on CPU: algorithmic bytes and flops per
workload (the per-unit figures of the kernel table, multiplied out by hand
here), the roofline entry, the arithmetic type it reports, the metric names,
the measured-peak lookup and the rule that a captured DRAM figure is reported
only for the kernel source it was captured on."""
import json
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from kernelized_sequence_mixing_gb300.workloads import WORKLOADS  # noqa: E402


# (workload, bytes, flops), worked out by hand from the per-unit figures:
# forward (2D + 2Dv) es B and 4 D Dv + 3 D + Dv flop per (b, h, token); the
# gated form adds 4D B of fp32 gates and D Dv + D flop; the Performer adds
# its r x D projection matrix once; the backward reads q, k, v, dL/do and
# writes dq, dk, dv, (4D + 3Dv) es B and 12 D Dv + 10 D + 4 Dv flop; decode
# reads and writes the fp32 state, 8 D Dv + 8 D B, plus q, k, v, o, per
# (sequence, head).
HAND = [
    # B2 H16 N16384, D = Dv = 128, bf16: 524,288 units x 1024 B; 66,048 flop
    ("causal_decay_bf16_n16384", 536_870_912, 524_288 * 66_048),
    # B4 H8 N4096, D = Dv = 64, bf16: 131,072 units x 512 B; 16,640 flop
    ("causal_bf16_n4096", 67_108_864, 131_072 * 16_640),
    # B1 H1 N256, D = Dv = 64, fp32: 256 units x 1024 B
    ("causal_f32_n256", 262_144, 256 * 16_640),
    # B8 H16 N65536, D = Dv = 64, bf16: 8,388,608 units x 512 B
    ("noncausal_bf16_n65536", 4_294_967_296, 8_388_608 * 16_640),
    # gated: 1024 + 512 B; 66,048 + 16,384 + 128 flop
    ("gla_bf16_n16384", 805_306_368, 524_288 * 82_560),
    # Performer r = 128: q, k, v, o plus the 128 x 128 bf16 matrix (32 KB);
    # flop 2 (2 D r + 2 D + r) + 4 r Dv + 3 r + Dv = 66,304 + 65,536 + 512
    ("favor_bf16_n16384", 536_903_680, 524_288 * 132_352),
    # backward: (256 + 192) x 2 = 896 B; 49,152 + 640 + 256 = 50,048 flop
    ("backward_bf16_n4096", 117_440_512, 131_072 * 50_048),
    # decode, 256 x 32 units: 131,072 + 1024 + 1024 B; 65,536 + 384 + 128 flop
    ("decode_bf16_h32", 1_090_519_040, 8192 * 66_048),
    # gated decode: + 512 B of gates, + 16,384 + 128 flop per unit
    ("decode_gated_bf16_h32", 1_094_713_344, 8192 * 82_560),
]


@pytest.mark.parametrize("name,byts,flops", HAND)
def test_algorithmic_work_matches_the_hand_count(name, byts, flops):
    w = WORKLOADS[name]
    got = bench.decode_work(w) if w.steps else bench.algorithmic_work(w)
    assert got == (byts, flops)


def test_every_workload_is_counted():
    # the two smaller capture cases are not benchmarked
    assert {n for n, _, _ in HAND} | {"causal_decay_bf16_n8192", "noncausal_bf16_n8192"} == \
        set(WORKLOADS)


def test_hbm_roofline_entry():
    w = WORKLOADS["causal_decay_bf16_n16384"]
    # 1 GB in 1 ms = 1000 GB/s; 2e12 flop in 1 ms = 2000 TFLOP/s
    r = bench.roofline_entry(w, 10**9, 2 * 10**12, 1.0, 2000.0, "measured", 1900.0,
                             None, 1)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(1000.0) and r["frac"] == pytest.approx(0.5)
    assert r["peak"] == 2000.0 and r["tflops"] == pytest.approx(2000.0)
    assert r["traffic"] is None and "measured" in r["peak_source"]


def test_alu_roofline_for_the_cuda_core_paths():
    # 152 SMs x 128 lanes x 2 flop x 2070 MHz = 80.54784 TFLOP/s
    assert bench.ALU_FP32_TFLOPS == pytest.approx(80.54784, rel=1e-12)
    for name, tc in (("backward_bf16_n4096", False), ("gla_bf16_n16384", False)):
        r = bench.roofline_entry(WORKLOADS[name], 10**9, 8 * 10**10, 1.0, 2000.0,
                                 "measured", 1900.0, None, 3, gated_tc=tc)
        assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
        assert r["achieved"] == pytest.approx(80.0)
        assert r["frac"] == pytest.approx(80.0 / 80.54784)
        assert r["hbm_frac"] == pytest.approx(0.5)
    # the tensor-core gated form and the gated decode step are HBM-bound
    for name in ("gla_bf16_n16384", "decode_gated_bf16_h32"):
        r = bench.roofline_entry(WORKLOADS[name], 10**9, 0, 1.0, 2000.0, "fallback",
                                 1900.0, None, 1, gated_tc=True)
        assert r["bound"] == "hbm" and r["peak_source"] == "fallback"
    # so is the tensor-core backward
    r = bench.roofline_entry(WORKLOADS["backward_bf16_n4096"], 10**9, 0, 1.0, 2000.0,
                             "measured", 1900.0, None, 5, bwd_tc=True)
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(0.5)


@pytest.mark.parametrize("name,tc,dtype", [
    ("causal_decay_bf16_n16384", False, "bf16"),
    ("causal_f32_n256", False, "f32"),
    ("noncausal_bf16_n65536", False, "bf16"),
    ("favor_bf16_n16384", False, "bf16"),
    ("gla_bf16_n16384", True, "bf16"),
    ("gla_bf16_n16384", False, "f32"),
    ("backward_bf16_n4096", False, "f32"),
    ("backward_bf16_n4096", True, "bf16"),
    ("decode_bf16_h32", False, "f32"),
    ("decode_gated_bf16_h32", False, "f32"),
])
def test_compute_dtype(name, tc, dtype):
    w = WORKLOADS[name]
    got = bench.compute_dtype(w, bwd_tc=tc) if w.backward else bench.compute_dtype(w, tc)
    assert got == dtype


def test_metric_names():
    names = {n: bench.workload_metric(w) for n, w in WORKLOADS.items()}
    assert names["causal_decay_bf16_n16384"] == bench.METRIC
    assert names["causal_bf16_n4096"] == bench.METRIC
    # every other kind has its own metric
    kinds = ["noncausal_bf16_n65536", "decode_bf16_h32", "decode_gated_bf16_h32",
             "gla_bf16_n16384", "favor_bf16_n16384", "backward_bf16_n4096"]
    assert len({names[k] for k in kinds} | {bench.METRIC}) == len(kinds) + 1


def test_measured_peaks_file_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (bench.FALLBACK_HBM_GBS, bench.FALLBACK_BF16_TFLOPS,
                                      "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6000.5, "bf16_tflops": 1800.25}))
    assert bench.measured_peaks() == (6000.5, 1800.25, "measured")
    (tmp_path / "MEASURED_PEAKS.json").write_text("{}")
    assert bench.measured_peaks()[2] == "fallback"


def test_traffic_only_for_the_captured_source():
    w = WORKLOADS["causal_decay_bf16_n16384"]
    cap = bench.NCU_TRAFFIC[w.name]
    assert bench.ncu_traffic(w, cap["source"]) == cap["bytes"]
    assert bench.ncu_traffic(w, "0" * 16) is None            # source changed
    assert bench.ncu_traffic(w, cap["source"], final_state=True) is None
    assert bench.ncu_traffic(WORKLOADS["causal_bf16_n4096"], cap["source"]) is None


def test_source_hash_follows_the_files(tmp_path, monkeypatch):
    csrc = tmp_path / "kernelized_sequence_mixing_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("x")
    (csrc / "b.cuh").write_text("y")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash(("a.cu", "b.cuh"))
    assert len(h0) == 16 and h0 == bench.kernel_source_hash(("a.cu", "b.cuh"))
    (csrc / "b.cuh").write_text("y2")
    assert bench.kernel_source_hash(("a.cu", "b.cuh")) != h0


def test_each_workload_hashes_the_sources_it_runs():
    src = {n: bench.workload_sources(w)[0] for n, w in WORKLOADS.items()}
    assert src["causal_decay_bf16_n16384"] == "chunk128.cu"
    assert src["causal_bf16_n4096"] == "chunk_tc.cu"
    assert src["causal_f32_n256"] == "causal_simt.cu"
    assert src["noncausal_bf16_n65536"] == "noncausal_tc.cu"
    assert src["decode_bf16_h32"] == src["decode_gated_bf16_h32"] == "decode.cu"
    assert src["gla_bf16_n16384"] == "gla_simt.cu"
    assert src["favor_bf16_n16384"] == "favor.cu"
    assert src["backward_bf16_n4096"] == "backward_tc.cu"
    for w in WORKLOADS.values():
        for f in bench.workload_sources(w):
            assert os.path.exists(os.path.join(ROOT, "kernelized_sequence_mixing_gb300",
                                               "csrc", f))


def test_clock_summary():
    """The clocks object from nvidia-smi lines: median SM clock, the highest
    maximum clock, every throttle reason seen Active, and malformed lines
    skipped."""
    na = "Not Active"
    lines = [
        f"0, 2070, 2070, 900.1, 0x0, {na}, {na}, {na}, {na}",
        f"0, 1980, 2070, 1390.0, 0x4, {na}, {na}, {na}, Active",
        f"0, 2070, 2070, 1100.5, 0x0, {na}, {na}, {na}, {na}",
        "garbage",
        f"0, [N/A], 2070, 1100.5, 0x0, {na}, {na}, {na}, {na}",
        f"0, 1500, 2070, 1200.0, 0x8, Active, {na}, {na}, {na}",
    ]
    c = bench.summarize_clocks(lines)
    assert c["samples"] == 4
    assert c["sm_mhz"] == 2025.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.summarize_clocks([]) == {"sm_mhz": None, "sm_max_mhz": None,
                                          "reasons": [], "samples": 0}


def test_clock_sampler_without_nvidia_smi(monkeypatch):
    """With no nvidia-smi on the machine the sampler reports that instead of
    failing the run."""
    def missing(*a, **kw):
        raise OSError("no nvidia-smi")

    monkeypatch.setattr(bench.subprocess, "Popen", missing)
    s = bench.ClockSampler(0)
    s.start()
    c = s.stop()
    assert c["samples"] == 0 and c["note"] == "nvidia-smi unavailable"


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_config_names_the_workload(name):
    """The config object names the workload and its sizes, and carries no
    model keys (there is no model: the path is one operator)."""
    w = WORKLOADS[name]
    cfg = bench.workload_config(w)
    assert cfg["workload"] == name and "model" not in cfg
    assert (cfg["B"], cfg["H"], cfg["D"], cfg["Dv"]) == (w.B, w.H, w.D, w.Dv)
    assert cfg["global_batch"] == w.B
    # decode steps process one token per sequence after a prefill of N
    assert cfg["seq_len"] == (1 if w.steps else w.N)
    if w.steps:
        assert cfg["prefill_len"] == w.N
    assert ("gamma" in cfg) == w.decayed and ("gates" in cfg) == w.gated
    json.dumps(cfg)   # serialisable into the JSON line


def test_oracle_sample_pairs_units_with_their_decays():
    """The CPU baseline's sample: the first units in (b, h) order, every
    token, each with its own head's decay."""
    import numpy as np
    from kernelized_sequence_mixing_gb300 import workloads as wl
    w = wl.Workload("t", True, 2, 3, 8, 64, 64, torch.float32, 1.0, 0, decayed=True)
    q, k, v = wl.workload_inputs(w)
    qs, ks, vs, gu = bench.oracle_sample(w, 5)
    assert qs.shape == (5, 8, 64) and vs.shape == (5, 8, 64)
    assert np.array_equal(qs[4], q[1, 1].numpy())          # unit 4 = (b 1, h 1)
    g = wl.retnet_gammas(3).numpy()
    assert np.array_equal(gu, np.array([g[0], g[1], g[2], g[0], g[1]]))


def test_oracle_timing_counts_tokens_across_heads():
    """A token is one position of one sequence across all H heads, so a
    sample of u of the H heads of one sequence covers u / H of its N tokens."""
    from kernelized_sequence_mixing_gb300 import workloads as wl
    w = wl.Workload("t", True, 1, 4, 32, 64, 64, torch.float32, 1.0, 0)
    tokens, times, threads = bench.time_oracle(w, 2, 1)
    assert tokens == 2 / 4 * 32 and len(times) == 1 and times[0] > 0 and threads >= 1
    d = wl.Workload("d", True, 4, 8, 4, 64, 64, torch.float32, 1.0, 0, steps=2,
                    step_seed0=1000)
    units_tokens, times, _ = bench.time_oracle_decode(d, 16, 1)
    assert units_tokens == 16 / 8 and len(times) == 1


def test_extra_workloads_cover_every_kind_beside_the_main_line():
    """The configurations timed beside the default line: each a defined
    workload other than the default, with positive algorithmic work, and
    together every kind of step (short causal, fp32, non-causal, decode,
    gated, Performer, backward)."""
    extras = bench.EXTRA_WORKLOADS
    assert len(set(extras)) == len(extras)
    assert bench.DEFAULT_WORKLOAD not in extras
    for name in extras:
        w = WORKLOADS[name]
        byts, flops = bench.decode_work(w) if w.steps else bench.algorithmic_work(w)
        assert byts > 0 and flops > 0, name
    ws = [WORKLOADS[n] for n in extras]
    assert any(w.dtype == torch.float32 for w in ws)
    assert any(not w.causal for w in ws)
    assert any(w.steps for w in ws)
    assert any(w.gated for w in ws)
    assert any(w.favor_r for w in ws)
    assert any(w.backward for w in ws)
