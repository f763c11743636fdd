"""bench.py's host-side arithmetic, without a GPU: algorithmic bytes and FLOPs per workload
kind against hand-computed values, the metric names and config keys of the JSON line, and the
rule that a committed ncu traffic record is dropped once its kernel's sources change."""
import json
import os
import re

import bench
import workloads as wl


def test_algorithmic_bytes_by_hand():
    W = wl.workloads()
    w = W["prefill_e64"]  # every one of the 64 experts is hit by 16384 uniform entries
    idx = wl.make_idx(w)
    codes_and_groups = 64 * 768 * (2048 // 2 + 4 * (2048 // 64))
    assert bench.algorithmic_bytes(w, idx) == codes_and_groups + 16384 * 2048 * 2 + 16384 * 768 * 2 + 16384 * 4
    g128 = W["prefill_e64_g128"]
    assert bench.algorithmic_bytes(g128, idx) == (64 * 768 * (1024 + 4 * 16) + 16384 * 2048 * 2 + 16384 * 768 * 2
                                                 + 16384 * 4)
    m = W["mlp_e64"]  # gate/up [2I, H] and down [H, I] per hit expert; x in, y (H wide) out
    per_expert = 2 * 768 * (1024 + 4 * 32) + 2048 * (384 + 4 * 12)
    assert bench.algorithmic_bytes(m, wl.make_idx(m)) == 64 * per_expert + 16384 * 2048 * 2 * 2 + 16384 * 4
    nn = W["nn_e4"]  # W[e] = [K = 512, N = 512] quantized along N
    assert bench.algorithmic_bytes(nn, wl.make_idx(nn)) == 4 * 512 * (256 + 4 * 8) + 1024 * 512 * 2 * 2 + 1024 * 4
    xyi = 16384 * 2048 * 2 + 16384 * 768 * 2 + 16384 * 4
    assert bench.algorithmic_bytes(W["prefill_e64_b3"], idx) == 64 * 768 * (768 + 4 * 32) + xyi
    assert bench.algorithmic_bytes(W["prefill_e64_mxfp4"], idx) == 64 * 768 * (1024 + 64) + xyi
    assert bench.algorithmic_bytes(W["prefill_e64_nvfp4"], idx) == 64 * (768 * (1024 + 128) + 4) + xyi
    assert bench.algorithmic_bytes(W["prefill_e64_mxfp8"], idx) == 64 * 768 * (2048 + 64) + xyi
    assert W["prefill_dense"].flops == 2 * 16384 * 2048 * 768
    assert m.flops == 6 * 16384 * 2048 * 768 and nn.flops == 2 * 1024 * 512 * 512


def test_metric_names_and_config_keys():
    W = wl.workloads()
    assert bench.metric_name(W["prefill_e64"]) == "gather_qmm TFLOPs (2*T*A*H*F/time)"
    assert "6*T*A*H*I" in bench.metric_name(W["mlp_e64"])
    assert "2*T*A*K*N" in bench.metric_name(W["nn_e4"])
    c = bench.workload_config(W["prefill_e64_g32"])
    assert c["workload"] == "prefill_e64_g32" and c["group_size"] == 32 and c["F"] == 768
    assert bench.workload_config(W["mlp_e64"])["I"] == 768
    assert bench.workload_config(W["nn_e4"])["K"] == 512 and bench.workload_config(W["nn_e4"])["N"] == 512


def test_traffic_record_is_dropped_when_sources_change(tmp_path, monkeypatch):
    rec = {"kernel": "gemm_tc_kernel", "workload": "toy", "source_sha256": bench.kernel_source_sha("gemm_tc_kernel"),
           "dram_bytes_per_launch": 123}
    (tmp_path / "profiles").mkdir()
    path = tmp_path / "profiles" / "gemm_tc_kernel_toy.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda k: rec["source_sha256"])
    assert bench.measured_traffic("gemm_tc_kernel", "toy") == 123
    monkeypatch.setattr(bench, "kernel_source_sha", lambda k: "0" * 64)  # the sources changed since the capture
    assert bench.measured_traffic("gemm_tc_kernel", "toy") is None
    rec2 = dict(rec, dram_bytes_per_step=456)  # a step with two launches records its total
    path.write_text(json.dumps(rec2))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda k: rec["source_sha256"])
    assert bench.measured_traffic("gemm_tc_kernel", "toy") == 456
    assert bench.measured_traffic("gemm_tc_kernel", "missing") is None


def test_committed_profiles_name_their_kernel_and_workload():
    root = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles")
    for f in os.listdir(root):
        if f.endswith(".json"):
            rec = json.load(open(os.path.join(root, f)))
            base = re.match(r"[A-Za-z_]+", rec["kernel"]).group(0)  # without template arguments or notes
            assert f == f"{base}_{rec['workload']}.json", f
            assert rec["workload"] in wl.workloads()
            assert "dram_bytes_per_launch" in rec or "dram_bytes_per_step" in rec
            assert "--clock-control none" in rec["command"]
