"""Host-side arithmetic of bench.py: the flop count of a step, the whole-job rate, the peaks it
divides by, and the rule that drops the committed DRAM-traffic figure once the GEMM's sources
change.  CPU only."""

import hashlib
import json
import os

import bench


def test_mlp_flops_counts_both_gemms():
    M, H, F = 8192, 4096, 14336
    # GEMM1 [M, H] x [H, 2F] for a gated pair, GEMM2 [M, F] x [F, H]
    assert bench.mlp_flops(M, H, F, True) == 2.0 * M * H * 2 * F + 2.0 * M * F * H
    assert bench.mlp_flops(M, H, F, False) == 2.0 * M * H * F + 2.0 * M * F * H
    # the Llama-shape forward is 2.886 TFLOP (GEMM1 1.924 + GEMM2 0.962)
    assert abs(bench.mlp_flops(M, H, F, True) / 1e12 - 2.886) < 1e-3


def test_whole_job_rate_uses_every_rank_and_the_slowest_time():
    # 3 ranks, 10 units each, slowest step 2 ms: 30 units per 2 ms
    assert bench.whole_job_rate(10, 3, 2.0) == 15000.0
    assert bench.reduce_max(4.5, 1, "cpu") == 4.5


def test_peaks_measured_file_and_fallback(tmp_path, monkeypatch):
    # a peaks file as the pod writes it is read as is
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6671.5, "bf16_tflops": 1941.1, "bf16_tflops_sustained": 1730.3}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p == dict(hbm=6671.5, bf16=1941.1, bf16_sustained=1730.3, source="measured")
    # without one, the fallback figures
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "empty"))
    q = bench.load_peaks()
    assert q["source"] == "fallback" and q["hbm"] == 6800.0 and q["bf16"] == 1900.0


def _profile(tmp_path, sources, digest, traffic=123456):
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"traffic_bytes_per_launch": traffic, "sources": list(sources),
                                "sources_sha256": digest}))
    return str(path)


def _digest(sources):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(bench.ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def test_traffic_kept_only_while_the_gemm_sources_match(tmp_path, monkeypatch):
    src = list(bench.GEMM_SOURCES)
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", _profile(tmp_path, src, _digest(src)))
    assert bench.measured_traffic() == 123456
    # a changed source (another digest) drops the figure
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", _profile(tmp_path, src, "0" * 64))
    assert bench.measured_traffic() is None
    # so does a capture that hashed a different list of files
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", _profile(tmp_path, src[:2], _digest(src[:2])))
    assert bench.measured_traffic() is None
    # and a missing capture
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(tmp_path / "absent.json"))
    assert bench.measured_traffic() is None
