"""Host-side pieces of bench.py, on CPU: algorithmic cost per launch group,
profile aggregation, the source-hash guard on recorded DRAM traffic, peak
loading and the config block of the JSON line."""
import hashlib
import json
import os

import pytest

import bench
import nc_synth

D20 = nc_synth.WORKLOADS["d20_bf16"]


def test_algorithmic_cost_at_d20():
    s, B, T = D20.shape, D20.batch, D20.seq
    M = B * T
    assert bench.algorithmic_cost("fwd.fc_gemm", s, B, T) == ("tensor", 2 * M * 1280 * 5120)
    assert bench.algorithmic_cost("bwd.fc_dw_gemm", s, B, T) == ("tensor", 2 * M * 1280 * 5120)
    assert bench.algorithmic_cost("fwd.qkv_gemm", s, B, T) == ("tensor", 2 * M * 1280 * 1536)
    assert bench.algorithmic_cost("lm.logits_gemm", s, B, T) == ("tensor", 2 * M * 1280 * 65536)
    # causal attention: one causal-half matmul is B H T^2 h FLOPs (2 T^2/2 h per head)
    one = 32 * 10 * 2048 * 2048 * 128
    assert bench.algorithmic_cost("fwd.attention", s, B, T) == ("tensor", 2 * one)
    assert bench.algorithmic_cost("bwd.attention", s, B, T) == ("tensor", 5 * one)
    assert 5 * one == pytest.approx(8.59e11, rel=1e-3)
    assert bench.algorithmic_cost("bwd.qknorm_rope", s, B, T) == ("hbm", M * 11 * 128 * 6)
    assert bench.algorithmic_cost("lm.dlogits", s, B, T) == ("hbm", M * 65536 * 4)
    assert bench.algorithmic_cost("no.such_group", s, B, T) == (None, 0)


def test_aggregate_profile_sums_counts_and_orders():
    rows, total = bench.aggregate_profile([("a", 1.0), ("b", 5.0), ("a", 2.5), ("c", 0.5)])
    assert [r[0] for r in rows] == ["b", "a", "c"]
    assert dict(rows)["a"] == [3.5, 2]
    assert total == pytest.approx(9.0)


def test_measured_traffic_needs_the_captured_source(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "pretraining_step_pretrain_b300", "csrc", "attention_tc.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    f = tmp_path / "traffic.txt"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    f.write_text(f"# comment\nbwd.attention 1.5e9 {h} attention_tc.cu\n")
    assert bench.measured_traffic("bwd.attention") == 1.5e9
    assert bench.measured_traffic("fwd.attention") is None
    f.write_text("bwd.attention 1.5e9 0123456789abcdef attention_tc.cu\n")   # source changed
    assert bench.measured_traffic("bwd.attention") is None
    f.write_text(f"bwd.attention 1.5e9 {h} no_such_file.cu\n")
    assert bench.measured_traffic("bwd.attention") is None


def test_committed_traffic_records_follow_their_sources():
    """Every committed traffic record is reported exactly while its kernel
    source is unchanged since the capture, and as null afterwards."""
    with open(bench.TRAFFIC_FILE) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert rows
    for group, value, sha, *srcs in rows:
        h = hashlib.sha256()
        for src in srcs:
            with open(os.path.join(bench.ROOT, "pretraining_step_pretrain_b300", "csrc", src),
                      "rb") as g:
                h.update(g.read())
        expect = float(value) if h.hexdigest()[:16] == sha else None
        assert bench.measured_traffic(group) == expect, group


def test_load_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6480, "bf16_tflops": 1802, "bf16_tflops_sustained": 1412, "other": 1}))
    peaks, src = bench.load_peaks()
    assert src == "measured"
    assert peaks == {"hbm_gbs": 6480.0, "bf16_tflops": 1802.0, "bf16_tflops_sustained": 1412.0}


def test_config_block_names_the_workload():
    c = bench.config_dict(D20, 4)
    assert c["workload"] == "d20_bf16" and c["global_batch"] == 128 and c["seq_len"] == 2048
    assert c["n_kv_head"] == 1 and "no collective" in c["parallelism"]


def test_host_cpu_names_model_and_cores():
    h = bench.host_cpu()
    assert h["nproc"] >= 1 and isinstance(h["model"], str) and h["model"]
