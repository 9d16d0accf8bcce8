"""Host logic of bench.py (no GPU): the roofline arithmetic, the ncu traffic record, the
per-batch rates and the link-aware attainable rate."""
import hashlib
import os

import pytest

import bench
from routed_expert_ffn_gemv_gb300 import synth


def _gv(fused=False):
    return {"gateup_ms_per_launch": 0.010, "gateup_bytes_per_launch": 30e6,
            "down_ms_per_launch": 0.008, "down_bytes_per_launch": 15e6,
            "reduce_ms_per_launch": 0.001, "gemv_ms_per_launch": 0.025, "fused": fused,
            "launches": 72, "steps": 3}


def test_roofline_block_is_the_gate_up_kernel_over_its_own_time():
    cfg = synth.config(1)
    peaks = {"hbm_gbs": 6000.0, "source": "measured"}
    r = bench.gemv_roofline_block(_gv(), cfg, 8, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6000.0
    assert r["achieved"] == pytest.approx(30e6 / 10e-6 / 1e9)   # 3000 GB/s
    assert r["frac"] == pytest.approx(0.5)
    assert r["algorithmic_bytes_per_launch"] == 30e6 and r["ms_per_launch"] == 0.010
    assert r["down_achieved_gbs"] == pytest.approx(15e6 / 8e-6 / 1e9)
    assert r["layer_chain_algorithmic_bytes_per_layer"] == 45e6
    assert r["layer_chain_achieved_gbs"] == pytest.approx(45e6 / 25e-6 / 1e9)
    assert "ks_reduce_kernel" in r["layer_chain_kernels"]
    assert "ffn_fused_kernel" in bench.gemv_roofline_block(_gv(True), cfg, 8, peaks)["layer_chain_kernels"]
    # the driver keeps only flat scalars inside the roofline object
    assert all(not isinstance(v, (dict, list)) for v in r.values())


def test_traffic_record_needs_the_current_kernel_source(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "routed_expert_ffn_gemv_gb300", "csrc", "moe_gemv.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        f"gateup_x {digest} 123 456\ngateup_y 0000000000000000 789 456\n")
    (tmp_path / "routed_expert_ffn_gemv_gb300" / "csrc").mkdir(parents=True)
    (tmp_path / "routed_expert_ffn_gemv_gb300" / "csrc" / "moe_gemv.cu").write_bytes(open(src, "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("gateup_x") == {"bytes_per_launch": 123.0, "algorithmic_bytes_per_launch": 456.0}
    assert bench.traffic_record("gateup_y") is None      # captured from another source
    assert bench.traffic_record("gateup_z") is None      # never captured


def test_committed_traffic_record_is_close_to_the_algorithmic_bytes():
    """Whatever ncu record is committed says DRAM traffic within 1% of the algorithmic bytes."""
    path = os.path.join(bench.ROOT, "profiles", "ncu_traffic.txt")
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4:
            assert abs(float(parts[2]) / float(parts[3]) - 1.0) < 0.01, line


def test_batch_result_counts_every_rank_and_the_link():
    cfg = synth.config(1)
    T, steps, world = 8, 10, 1
    q = 30 * cfg.L * steps                      # 30 distinct experts per layer and step
    st = {"queries": [q], "hits": [q // 2], "h2d_bytes": (q // 2) * cfg.expert_bytes,
          "route_hits": 0, "route_queries": T * cfg.k * cfg.L * steps}
    peaks = {"hbm_gbs": 6784.5}
    r = bench.batch_result(cfg, T, steps, 50.0, st, world, peaks, 211.0)
    assert r["tokens_per_s"] == pytest.approx(T * steps / 0.050)
    assert r["hit_rate"] == pytest.approx(0.5)
    bytes_step = q * cfg.expert_bytes / steps
    assert r["expert_bytes_per_step"] == pytest.approx(bytes_step)
    t_attain = (bytes_step / 2) / 211e9 + (bytes_step / 2) / 6784.5e9
    assert r["link_aware_attainable_tokens_per_s"] == pytest.approx(T / t_attain)
    assert r["frac_of_8tbs_roofline"] == pytest.approx(r["tokens_per_s"] / (T / (bytes_step / 8e12)))
    r2 = bench.batch_result(cfg, T, steps, 50.0, st, 2, peaks, 211.0)
    assert r2["tokens_per_s"] == pytest.approx(2 * r["tokens_per_s"])   # whole job over 2 replicas
    assert r2["frac_of_8tbs_roofline"] == pytest.approx(r["frac_of_8tbs_roofline"])  # per GPU


def test_peaks_fall_back_when_no_measurement(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0 and p["bf16_tflops"] == 1900.0


def test_hit_fields_by_query_route_and_bucket():
    st = {"queries": [10, 30], "hits": [9, 15], "route_queries": 100, "route_hits": 80}
    h = bench.hit_fields(st)
    assert h["hit_rate"] == pytest.approx(24 / 40)
    assert h["route_hit_rate"] == pytest.approx(0.8)
    assert h["hit_rate_le8"] == pytest.approx(0.9) and h["hit_rate_9to32"] == pytest.approx(0.5)
    h0 = bench.hit_fields({"queries": [4, 0], "hits": [1, 0], "route_queries": 0, "route_hits": 0}, "c_")
    assert h0["c_hit_rate"] == 0.25 and h0["c_route_hit_rate"] is None and "c_hit_rate_9to32" not in h0


def test_prefill_block_is_flat_and_summary_prints():
    pf = bench.flat_prefill({"512": {"ffn_ms": 0.3, "ffn_tflops": 120.0, "frac_of_dense_peak": 0.06, "x": "s"},
                             "4096": {"ffn_ms": 0.6, "ffn_tflops": 500.0, "frac_of_dense_peak": 0.27}},
                            {"bf16_tflops": 1854.8})
    assert pf["t512_ffn_ms"] == 0.3 and pf["t4096_frac_of_dense_peak"] == 0.27 and "t512_x" not in pf
    assert all(not isinstance(v, (dict, list)) for v in pf.values())
    line = {"config": {"workload": "w"}, "value": 1.0, "ms_per_step": 2.0, "e2e": {"value": 1.0},
            "roofline": {"achieved": 1.0, "frac": 0.1, "down_frac": 0.2, "layer_chain_frac": 0.3},
            "configs": {"qwen3_b1": {"tokens_per_s": 5.0, "frac_of_8tbs_roofline": 0.1, "hit_rate": 0.5,
                                     "from_cold_hit_rate": 0.4, "resident_tokens_per_s": 9.0,
                                     "resident_frac_of_8tbs_roofline": 0.2}},
            "prefill": pf}
    rows = bench.summary_lines(line)
    assert len(rows) == 5 and rows[2].startswith("qwen3_b1")
