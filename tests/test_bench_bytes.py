"""The bench's algorithmic bytes per step: every target row, the draft rows of
sampling requests only, none with deterministic drafts, and over the full
vocabulary the draw's second read of its rows (two after a rejection, one for
a bonus token)."""
import numpy as np

import bench
import synth


def test_top_k_and_deterministic_rows():
    inp = synth.make_workload("b32_mixed_v248320", V=1000)
    B, gamma, V = inp.shape
    n_samp = int(np.sum(inp.temperature > 0))
    assert n_samp == 21   # temperatures cycle 0 / 0.6 / 1.0 over 32 requests
    assert bench.algorithmic_bytes(inp) == (B * (gamma + 1) + n_samp * gamma) * V * 2
    assert bench.algorithmic_bytes(inp, det=True) == B * (gamma + 1) * V * 2
    # the headline: 403 rows of 248320 bf16 logits
    assert (B * (gamma + 1) + n_samp * gamma) * 248320 * 2 == 200145920


def test_full_vocabulary_draw_reads():
    inp = synth.make_workload("b128_g15_fullvocab_f32", B=4, V=500)
    B, gamma, V = inp.shape
    lens = np.array([1, gamma + 1, 3, gamma + 1])   # two rejections, two bonus draws
    base = (B * (gamma + 1) + B * gamma) * V * 4
    assert bench.algorithmic_bytes(inp, lens) == base + (2 + 1 + 2 + 1) * V * 4


def test_top_p_over_the_vocabulary_counts_the_draw_not_the_cut():
    inp = synth.make_workload("b32_mixed_topp_v248320", B=6, V=700)
    B, gamma, V = inp.shape
    samp = inp.temperature > 0                      # 0 / 0.6 / 1.0: four of six sample
    lens = np.array([1, 2, gamma + 1, 3, 8, gamma + 1])
    base = (B * (gamma + 1) + int(samp.sum()) * gamma) * V * 2
    extra = sum((2 if n <= gamma else 1) for n in lens[samp])
    assert bench.algorithmic_bytes(inp, lens) == base + extra * V * 2


def test_profile_lookup_names():
    assert bench.profile_summary("b32_mixed_v248320") == bench.PROFILE_SUMMARY
    assert bench.profile_summary("b32_mixed_v248320", det=True).endswith("verify_sweep_b32_mixed_v248320_det.md")
    assert bench.profiled_traffic(bench.profile_summary("no_such_workload")) is None


def test_launches_per_step():
    assert bench.launches_per_step(20, 0.95) == 1
    assert bench.launches_per_step(0, 1.0) == 3
    # top-p over the full vocabulary: stream, the rounds' two launches each
    # (the first and up to two refinements for bf16 keys, four for fp32),
    # the two tie launches, accept, the draw's two
    assert bench.launches_per_step(0, 0.95) == 12
    assert bench.launches_per_step(0, 0.95, bf16=False) == 16


def test_profiler_calls_mode_takes_verification_workloads_only():
    """bench.py --calls runs verification calls; the LM head's workload is
    refused on the command line, before anything touches a GPU."""
    import subprocess
    import sys

    r = subprocess.run([sys.executable, bench.__file__, "--workload", bench.LMHEAD_WORKLOAD, "--calls", "1"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "--calls runs a verification workload" in r.stderr
