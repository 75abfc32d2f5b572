"""CPU checks of the C ABI: the library loads without a GPU, exports every
symbol include/fcc.h declares, rejects bad arguments before touching CUDA,
and the InterDecom chunk model behaves as stated."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fcc.h")


@pytest.fixture(scope="module")
def fcc():
    import __graft_entry__
    __graft_entry__.build()
    import gemm_collective_gb300 as m
    return m


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fcc_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(fcc):
    names = _declared()
    assert "fcc_gemm_rs" in names and "fcc_moe_dispatch_gemm" in names
    lib = ctypes.CDLL(fcc.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_library_needs_no_driver_to_load(fcc):
    # Loaded above in a process that has no GPU: the CUDA runtime is static and
    # the driver is resolved lazily.
    assert fcc.fcc_version().count(".") == 2


def test_status_strings(fcc):
    assert fcc.fcc_status_string(fcc.FCC_OK) == "ok"
    assert "timed out" in fcc.fcc_status_string(fcc.FCC_ERR_TIMEOUT)
    assert fcc.fcc_status_string(99) == "unknown status"


def test_invalid_arguments_rejected_without_cuda(fcc):
    P = ctypes.c_void_p
    two = (P * 2)(16, 32)
    bad = (P * 2)(16, 33)
    null = (P * 2)(16, 0)
    cases = [
        (0, two, two, two, 256, 256, 128, 0, 0),     # R = 0
        (9, two, two, two, 256, 256, 128, 0, 0),     # R > 8
        (2, two, two, two, 255, 256, 128, 0, 0),     # M % R
        (2, two, two, two, 256, 250, 128, 0, 0),     # N % 8
        (2, two, two, two, 256, 256, 100, 0, 0),     # K % 8
        (2, bad, two, two, 256, 256, 128, 0, 0),     # misaligned A
        (2, two, null, two, 256, 256, 128, 0, 0),    # null B
        (2, two, two, bad, 256, 256, 128, 0, 0),     # misaligned output
        (2, two, two, two, 0, 256, 128, 0, 0),       # empty M
        (2, two, two, two, 256, 256, 128, 5, 0),     # bad input dtype
        (2, two, two, two, 256, 256, 128, 0, 7),     # bad output dtype
    ]
    for c in cases:
        st = fcc.raw_status("fcc_gemm_rs", *c, None, None)
        assert st == fcc.FCC_ERR_INVALID, c
    # unsupported input dtype (f16 inputs are not implemented)
    assert fcc.raw_status("fcc_gemm_rs", 2, two, two, two, 256, 256, 128, 1, 0, None,
                          None) == fcc.FCC_ERR_UNSUPPORTED
    # GEMV: more than 16 tokens
    assert fcc.raw_status("fcc_gemv_ar", 2, two, two, two, 17, 256, 128, 0, 2, None,
                          None) == fcc.FCC_ERR_INVALID
    # AG: M % R
    assert fcc.raw_status("fcc_ag_gemm", 2, two, two, two, None, 255, 256, 128, 0, 0, None,
                          None) == fcc.FCC_ERR_INVALID
    # tile shapes other than automatic, one CTA or a CTA pair
    for pair in (3, 4, -1):
        o = ctypes.byref(fcc.make_opts(cta_pair=pair))
        assert fcc.raw_status("fcc_gemm_rs", 2, two, two, two, 256, 256, 128, 0, 0, o,
                              None) == fcc.FCC_ERR_INVALID, pair
        assert fcc.raw_status("fcc_gemm_ar", 2, two, two, two, 256, 256, 128, 0, 0, o,
                              None) == fcc.FCC_ERR_INVALID, pair
        assert fcc.raw_status("fcc_ag_gemm", 2, two, two, two, None, 256, 256, 128, 0, 0, o,
                              None) == fcc.FCC_ERR_INVALID, pair
    # the no-allocation GEMV: an algorithm outside the enum is invalid, the
    # valid unfused forms are unsupported there
    for algo, want in [(99, fcc.FCC_ERR_INVALID), (-1, fcc.FCC_ERR_INVALID),
                       (fcc.FCC_ALGO_UNFUSED, fcc.FCC_ERR_UNSUPPORTED),
                       (fcc.FCC_ALGO_INTERDECOM, fcc.FCC_ERR_UNSUPPORTED),
                       (fcc.FCC_ALGO_CE, fcc.FCC_ERR_UNSUPPORTED)]:
        o = ctypes.byref(fcc.make_opts(algo=algo))
        assert fcc.raw_status("fcc_gemv_ar_static", 2, two, two, two, 8, 256, 128, 0, 2, o,
                              None) == want, algo
    assert fcc.fcc_launch_count() == 0


def test_interdecom_model(fcc):
    # T(c) = max(G,X) + min(G,X)/c + c*alpha, minimised near sqrt(min/alpha)
    G, X, a = 1000.0, 400.0, 4.0
    c = fcc.fcc_interdecom_chunks(G, X, a, 64)
    assert c == 10  # sqrt(400/4) = 10
    t = [fcc.fcc_interdecom_time(G, X, a, k) for k in range(1, 65)]
    assert t.index(min(t)) + 1 == c
    assert math.isclose(fcc.fcc_interdecom_time(G, X, a, 1), G + X + a)
    assert fcc.fcc_interdecom_chunks(G, X, a, 4) == 4      # clamped
    assert fcc.fcc_interdecom_chunks(G, X, 1e9, 64) == 1   # overhead dominates
    assert fcc.fcc_interdecom_chunks(G, X, 0.0, 16) == 16  # free chunks: as many as allowed
    for G, X, a in [(10.0, 90.0, 0.3), (5.0, 5.0, 0.01), (300.0, 1.0, 0.02)]:
        c = fcc.fcc_interdecom_chunks(G, X, a, 128)
        t = [fcc.fcc_interdecom_time(G, X, a, k) for k in range(1, 129)]
        assert math.isclose(t[c - 1], min(t)), (G, X, a, c)


def test_workspace_sizes(fcc):
    o = fcc.make_opts(algo=fcc.FCC_ALGO_UNFUSED)
    assert fcc.fcc_workspace_size(fcc.FCC_OP_GEMM_RS, 8, 8192, 8192, 3584, o) >= 8 * 8192 * 8192 * 4
    # fused, deterministic: the K halves of a short last round (at most half
    # a round of 256 x 256 tiles, f32 partials) and their flags
    fused = fcc.fcc_workspace_size(fcc.FCC_OP_GEMM_RS, 8, 8192, 8192, 3584, None)
    assert 0 < fused <= 128 * 2 * 128 * 256 * 4 + 4096
    o = fcc.make_opts(algo=fcc.FCC_ALGO_CE)
    assert fcc.fcc_workspace_size(fcc.FCC_OP_GEMM_RS, 2, 256, 256, 128, o) >= 2 * 2 * 256 * 256 * 4
    assert fcc.fcc_workspace_size(fcc.FCC_OP_AG_GEMM, 8, 8192, 3584, 8192, None) == 0
    # MoE: room to stage every receive row (recv_x NULL), the receive row of
    # every assignment, and one row counter per (expert, 128-row tile) unit
    R, T, H, F, E, topk, cap = 8, 4096, 4096, 1408, 64, 2, 16384
    need = R * cap * H * 2 + R * T * topk * 4 + (R * T * topk // 128 + E) * 4
    assert fcc.fcc_moe_workspace_size(R, T, H, F, E, topk, cap) >= need
    assert fcc.fcc_moe_workspace_size(0, T, H, F, E, topk, cap) == 0


def test_strategy_selector(fcc):
    """AUTO's choice per operator and shape (host logic only, no device)."""
    F, U = fcc.FCC_ALGO_FUSED, fcc.FCC_ALGO_UNFUSED
    for op in (fcc.FCC_OP_GEMM_RS, fcc.FCC_OP_GEMM_AR, fcc.FCC_OP_AG_GEMM):
        assert fcc.fcc_choose_algo(op, 8, 8192, 8192, 3584, 152) == F
        assert fcc.fcc_choose_algo(op, 2, 256, 256, 128, 152) == F
    gemv = fcc.FCC_OP_GEMV_AR
    # 16 column groups of 512 -> 9 splits on 152 SMs: fused
    assert fcc.fcc_choose_algo(gemv, 8, 8, 8192, 3584, 152) == F
    # 8 groups -> 19 splits: the plain GEMM + reduce
    assert fcc.fcc_choose_algo(gemv, 8, 8, 4096, 3584, 152) == U
    # capped grid: 2 groups on 8 CTAs -> 4 splits: fused again
    assert fcc.fcc_choose_algo(gemv, 8, 8, 1024, 3584, 152, 8) == F
    assert fcc.fcc_choose_algo(gemv, 8, 8, 1024, 3584, 152, 64) == U
    # few K blocks bound the splits: 2 ranks x 1 block of 64 -> 2 splits
    assert fcc.fcc_choose_algo(gemv, 2, 8, 512, 64, 152) == F
    # embedding + all-to-all: the fused pooling + exchange
    assert fcc.fcc_choose_algo(fcc.FCC_OP_EMBEDDING_A2A, 8, 0, 0, 0, 152) == F


def _in_subprocess(env_extra, code):
    """Runs `code` with the library loaded in a fresh process whose environment
    adds env_extra (the environment defaults are read once per process)."""
    import subprocess
    import sys
    env = dict(os.environ)
    env.update(env_extra)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    return r.stdout.strip()


def test_environment_algorithm_default():
    """FCC_ALGO replaces the AUTO rule (here in fcc_choose_algo, which the calls
    use); an unknown value leaves the rule."""
    code = ("import gemm_collective_gb300 as f; "
            "print(f.fcc_choose_algo(f.FCC_OP_GEMM_RS, 8, 8192, 8192, 3584, 152), "
            "f.fcc_choose_algo(f.FCC_OP_EMBEDDING_A2A, 8, 0, 0, 0, 152))")
    import gemm_collective_gb300 as f
    U, C, F = f.FCC_ALGO_UNFUSED, f.FCC_ALGO_CE, f.FCC_ALGO_FUSED
    assert _in_subprocess({"FCC_ALGO": "unfused"}, code) == f"{U} {U}"
    assert _in_subprocess({"FCC_ALGO": "CE"}, code) == f"{C} {C}"
    assert _in_subprocess({"FCC_ALGO": "bogus"}, code) == f"{F} {F}"


def test_environment_deterministic_default_sizes_workspace():
    """FCC_DETERMINISTIC=0 makes calls without opts use the push mode, whose
    bf16 form needs an f32 accumulator: the size query with opts == NULL
    reports it."""
    code = ("import gemm_collective_gb300 as f; "
            "print(f.fcc_workspace_size(f.FCC_OP_GEMM_RS, 8, 8192, 8192, 3584, None))")
    push = int(_in_subprocess({"FCC_DETERMINISTIC": "0"}, code))
    ordered = int(_in_subprocess({"FCC_DETERMINISTIC": "1"}, code))
    assert push >= 8192 * 8192 * 4 > ordered

