"""The benchmark's host-side bookkeeping, on CPU.

`roofline.traffic` is the DRAM bytes of one launch of the headline kernel from
a committed ncu capture, reported only while the kernel's sources are the ones
the capture was taken of (a SHA-256 over them); a changed kernel reports null.
"""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SOURCES = ["gemm_collective_gb300/csrc/fcc_gemm.cu", "gemm_collective_gb300/csrc/fcc_ptx.cuh",
           "gemm_collective_gb300/csrc/fcc_api.cu"]


def _write_capture(root, sha, total=123456789):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "k.traffic.txt"), "w") as f:
        f.write(f"# a comment = with an equals sign\nsource_sha256 = {sha}\n"
                f"dram_bytes_read = 1\nbytes_per_launch_full = {total}\n")


def _sources(root, texts):
    paths = []
    for i, t in enumerate(texts):
        p = f"src{i}.cu"
        with open(os.path.join(root, p), "w") as f:
            f.write(t)
        paths.append(p)
    return paths


def test_traffic_reported_while_sources_match(tmp_path, monkeypatch):
    root = str(tmp_path)
    paths = _sources(root, ["kernel a", "header b"])
    sha = hashlib.sha256(b"kernel a" + b"header b").hexdigest()
    _write_capture(root, sha)
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.kernel_traffic("k", paths) == 123456789.0


def test_traffic_null_once_a_source_changes(tmp_path, monkeypatch):
    root = str(tmp_path)
    sha = hashlib.sha256(b"kernel a" + b"header b").hexdigest()
    _write_capture(root, sha)
    paths = _sources(root, ["kernel a", "header b, edited"])
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.kernel_traffic("k", paths) is None
    assert bench.kernel_traffic("missing", paths) is None


def test_committed_headline_capture_is_parsed():
    """The committed capture holds a positive per-launch byte count; it is
    reported as long as its hash names the committed kernel sources."""
    got = bench.kernel_traffic("gemm_rs_fused", SOURCES)
    h = hashlib.sha256()
    for s in SOURCES:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    with open(os.path.join(ROOT, "profiles", "gemm_rs_fused.traffic.txt")) as f:
        recorded = [ln.split("=", 1)[1].strip() for ln in f if ln.startswith("source_sha256")]
    assert recorded, "no source_sha256 line"
    if recorded[0] == h.hexdigest():
        assert got is not None and got > 0
    else:
        assert got is None


def _fake_results():
    """Results shaped like the benchmark's legs, with long-digit values."""
    x = 1.23456789012345

    def ms(v):
        return {"ms": v * x, "TFLOP/s": 1876.123456789}

    phases = {"epilogue_busy_frac": 0.4123456, "mma_wait_on_epilogue_frac": 0.0123456}
    check = {"sweep_ms": {str(c): 2.5 * x for c in (1, 2, 4)}, "best_c": 2,
             "model": {"G_ms": 2.1, "X_ms": 0.3, "alpha_ms": 0.01, "c_star": 3,
                       "T_cstar_ms": 2.6, "T_model_ms": 2.5},
             "c_star_within_10pct_of_best": True}
    base = {"unfused": ms(2.4), "interdecom": ms(2.6), "copy_engine": ms(3.3),
            "fused_push": ms(2.5), "cublas_stacked_gemm": ms(1.8), "interdecom_check": check,
            "phases": phases}
    gemm = {"fused": ms(2.1), "unfused": ms(2.4), "interdecom": ms(2.5), "copy_engine": ms(3.4),
            "roofline_frac": 0.98765432, "interdecom_check": check, "phases": phases}
    us = {"us": 81.7654321, "GB/s": 5780.1234}
    ar = {k: v for k, v in gemm.items() if k != "interdecom_check"}
    ops = {"gemm_ar_r8_8192x8192x3584": ar, "ag_gemm_r8_8192x3584x8192": dict(gemm),
           "gemv_ar_r8_8x8192x3584": {"fused": us, "unfused": us, "copy_engine": us,
                                      "roofline_frac": 0.8512345},
           "moe_r8_t4096_h4096_e64_f1408": dict(gemm, combine={
               "us": 56.712345, "roofline_frac": 0.7312345,
               "graph_replay": {"us": 48.512345}}),
           "emb_a2a_r8_t64_v65536_d128_b2048_l32": {"fused": us, "unfused": us,
                                                    "copy_engine": us, "auto": "unfused",
                                                    "roofline_frac": 0.1512345},
           "attn_r8_s4096_h8_d128": {"full": {"ms": 3.81612345, "roofline_frac": 0.6012345},
                                     "causal": {"ms": 2.62312345}},
           "gemm_rs_r2_256x256x128": {"plain_us": 10.2612345, "graph_us": 7.4512345}}
    return base, ops


def test_printed_line_fits_the_kept_tail(capsys, tmp_path):
    """The driver keeps the last 1500 characters of the output: the whole JSON
    line, with every operator's forms and the InterDecom checks, fits."""
    import json
    base, ops = _fake_results()
    line = {"metric": bench.METRIC, "value": 1876.3363284486, "unit": "TFLOP/s", "n_gpus": 8,
            "steps": 400, "warmup": 10, "ms_per_step": 2.0509599685668944,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": bench.WORKLOAD, "l2": "inputs>L2, no flush",
                       "parallelism": "replicas8"},
            "roofline": {"bound": "tensor", "achieved": 1876.3363284, "peak": 1912.2,
                         "unit": "TFLOP/s", "frac": 0.98124481144, "traffic": 4807605760.0},
            "e2e": {"value": 718.2004922511586, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": 939524096, "d2h_bytes_per_step": 134217728},
            "gpu_launches": 400,
            "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0,
                       "reasons": ["hw_slowdown", "sw_power_cap"], "samples": 1234},
            "cpu_baseline": {"value": 0.0546, "unit": "TFLOP/s", "cores": 144, "kind": "oracle",
                             "sample": "1744 rows, 15.0 s"}}
    line["ops_us"], line["interdecom"] = bench.compact_ops(base, ops, 2.0509599685668944)
    line["epilogue"] = bench.compact_phases(base, ops)
    assert set(line["ops_us"]) == {"cols", "rs", "rs_push", "rs_cublas", "ar", "ag", "moe",
                                   "gemv", "combine", "emb", "attn", "rs_r2"}
    assert line["ops_us"]["rs"][0] == 2051 and line["ops_us"]["gemv"][2] is None
    assert set(line["epilogue"]) == {"rs", "ar", "ag", "moe"}
    assert line["interdecom"] == {"rs": [3, 2, 1], "ag": [3, 2, 1], "moe": [3, 2, 1]}
    path = tmp_path / "details.json"
    bench.emit(line, {"ops": ops}, str(path))
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1 and len(out[0]) <= 1500, len(out[0])
    got = json.loads(out[0])
    assert "epilogue" in got and set(got["ops_us"]) == set(line["ops_us"]), "keys dropped"
    assert got["ops_us"]["rs_cublas"] == bench.sig(1.8 * 1.23456789012345 * 1e3)
    assert got["ops_us"]["ag"][2] == bench.sig(2.5 * 1.23456789012345 * 1e3)
    assert "ops" in json.loads(path.read_text())


def test_significant_digits():
    assert bench.sig(2051.2345) == 2051
    assert bench.sig(81.76543) == 81.77
    assert bench.sig(0.0546123) == 0.05461
    assert bench.sig(None) is None and bench.sig(0.0) == 0.0
