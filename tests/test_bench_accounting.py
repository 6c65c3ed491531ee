"""Host-side accounting of bench.py (CPU only): the algorithmic bytes and FLOPs of the FFN
stage when the shared expert runs in its own launch add up to those of the single launch,
and the launch count per step follows the library's launch structure."""
import dataclasses
import os

import bench
from expert_routed_ffn_router_gb300 import synth


def test_shared_expert_split_keeps_the_totals():
    for name in ("sweep2", "decode", "prefill"):
        w = synth.workload(name)
        n_act = min(w.E, w.T * w.K)
        b1, f1, lb1, lf1 = bench.algorithmic(w, n_act, 2, side=False)
        b2, f2, lb2, lf2 = bench.algorithmic(w, n_act, 2, side=True)
        assert b2["ffn"] + b2["ffn_shared"] == b1["ffn"]
        assert f2["ffn"] + f2["ffn_shared"] == f1["ffn"]
        assert (lb1, lf1) == (lb2, lf2)
        # the shared expert's weights: 3 H Is bf16 values
        assert b2["ffn_shared"] >= 3 * w.H * w.Is * 2


def test_side_stream_placement_rule():
    assert bench.shared_on_side(synth.workload("decode"))            # T = 128
    assert bench.shared_on_side(synth.workload("sweep2"))
    assert not bench.shared_on_side(synth.workload("prefill"))
    assert not bench.shared_on_side(synth.workload("decode"), fp8=True)


def test_launches_per_step_by_batch_size():
    expect = {2: 5, 8: 5, 16: 6, 128: 6, 200: 5, 512: 8, 3000: 7, 16384: 8}
    for T, n in expect.items():
        assert bench.launches_per_step(synth.workload("decode", T=T), True) == n, T
    # FP8 experts at 128 tokens: router tile + finalise, dispatch, then the quantisation of
    # the permuted rows and of the token rows, up launch, two h quantisations, down launch,
    # and combine (ten launches a step in the ncu launch list of FP8 decode)
    w = synth.workload("decode")
    assert bench.launches_per_step(w, True, fp8=True) == 2 + 1 + 6 + 1
    # without a shared expert: no token-row and no shared-h quantisation
    assert bench.launches_per_step(dataclasses.replace(w, Is=0), True, fp8=True) == 2 + 1 + 4 + 1


def test_targets_by_batch_size():
    assert bench.target_of(synth.workload("sweep2")) == ("hbm_frac_of_8TBs", 0.70)
    assert bench.target_of(synth.workload("sweep64")) == ("hbm_frac_of_8TBs", 0.70)
    assert bench.target_of(synth.workload("decode")) == (None, None)
    assert bench.target_of(synth.workload("skewed")) == ("tensor_frac", 0.60)
    assert bench.target_of(synth.workload("prefill")) == ("tensor_frac", 0.60)


def test_layer_roofline_fractions():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    w = synth.workload("sweep2")
    n_act = 16
    _, _, lb, lf = bench.algorithmic(w, n_act, 2, bench.shared_on_side(w))
    ms = lb / 8e12 * 1e3          # a step moving the algorithmic bytes at exactly 8 TB/s
    r = bench.layer_roofline(w, n_act, ms, peaks)
    assert abs(r["hbm_frac_of_8TBs"] - 1.0) < 1e-3
    assert abs(r["hbm_frac"] - 8000.0 / 6000.0) < 1e-3
    assert abs(r["tensor_frac"] * 2000.0 - r["tensor_frac_sustained"] * 1600.0) < 1e-3 * 2000
    # FP8 experts: the same step measured against the FP8 rate (bf16 x the nominal ratio)
    r8 = bench.layer_roofline(w, n_act, ms, peaks, fp8=True)
    assert r8["tensor_dtype"] == "fp8"
    assert abs(r8["tensor_frac"] * bench.FP8_OVER_BF16 - r["tensor_frac"]) <= 2e-4


def test_fp8_dominant_kernel_takes_the_fp8_peak():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    w = synth.workload("prefill")
    stage_ms = {"router": 1.0, "dispatch": 0.5, "ffn_up": 10.0, "ffn_down": 0.0, "combine": 0.4,
                "ffn": 10.0}
    r16 = bench.dominant_roofline(w, w.E, stage_ms, peaks, "measured", False)
    r8 = bench.dominant_roofline(w, w.E, stage_ms, peaks, "measured", True)
    assert r16["bound"] == r8["bound"] == "tensor"
    assert r16["peak"] == 2000.0 and r8["peak"] == 2000.0 * bench.FP8_OVER_BF16
    assert "ratio" in r8["peak_source"] and "ratio" not in r16["peak_source"]


def test_every_side_workload_exists_and_shares_the_weights():
    base = synth.workload("decode")
    for name in bench.SIDE_WORKLOADS:
        w = synth.workload(name)
        assert (w.H, w.E, w.K, w.I, w.Is, w.seed) == (base.H, base.E, base.K, base.I, base.Is,
                                                      base.seed)


def test_gpus_flag_must_match_world_size(monkeypatch):
    import pytest
    monkeypatch.setattr("sys.argv", ["bench.py", "--gpus", "2"])
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert e.value.code not in (0, None)


def test_cpu_baseline_reports_all_cores_and_one_core():
    # the oracle timed on the tiny workload's CPU-resident weights: the all-core rate and
    # the one-core rate, each with its sample, and the thread count restored afterwards
    import torch

    import oracle
    w = synth.workload("tiny")
    r = synth.routing_inputs(w)
    wt = synth.expert_weights_device(w, torch.device("cpu"))
    before = oracle.num_threads()
    out = bench.cpu_baseline(w, r, wt, budget_s=0.2)
    assert out["kind"] == "oracle" and out["cores"] == before and out["value"] > 0
    assert out["one_core"]["cores"] == 1 and out["one_core"]["value"] > 0
    assert oracle.num_threads() == before


def test_skew_stats_on_a_planted_routing():
    # counts exactly c_r = 1000 r^-1.2 and co-activations only inside clusters of 32: the
    # slope and the within-cluster share come back as planted
    import numpy as np
    E = 64
    c = np.rint(1000.0 * np.arange(1, E + 1) ** -1.2)
    A = np.zeros((E, E), np.int64)
    for k in range(E // 32):
        A[32 * k:32 * k + 32, 32 * k:32 * k + 32] = 3
    np.fill_diagonal(A, 0)
    s = bench.skew_stats(np.random.default_rng(0).permutation(c), A, T=10_000)
    assert abs(s["zipf_slope"] + 1.2) < 0.02
    assert s["within_cluster_coactivation"] == 1.0
    assert s["top_counts"][0] == 1000


def test_ffn_traffic_scales_small_case_ratio_only_for_weight_streaming_batches(tmp_path):
    import hashlib
    import json
    srcs = ["expert_routed_ffn_router_gb300/csrc/ffn_tc.cu",
            "expert_routed_ffn_router_gb300/csrc/common.cuh"]
    h = hashlib.sha256()
    for s in srcs:
        with open(os.path.join(bench.ROOT, s), "rb") as f:
            h.update(f.read())
    rec = {"sources": srcs, "sources_sha256": h.hexdigest(), "ratio": {"bf16": 1.01, "fp8": 1.02}}
    p = tmp_path / "t.json"
    p.write_text(json.dumps(rec))
    dec, pre = synth.workload("decode"), synth.workload("prefill")
    assert bench.ffn_traffic(dec, False, 10**9, str(p)) == 1_010_000_000
    assert bench.ffn_traffic(dec, True, 10**9, str(p)) == 1_020_000_000
    assert bench.ffn_traffic(synth.workload("sweep256"), False, 100, str(p)) == 101
    # larger batches: the small cases do not scale to them
    assert bench.ffn_traffic(pre, False, 10**9, str(p)) is None
    # a record taken on other sources is not reported
    rec["sources_sha256"] = "0" * 64
    p.write_text(json.dumps(rec))
    assert bench.ffn_traffic(dec, False, 10**9, str(p)) is None
