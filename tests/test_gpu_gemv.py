"""GPU parity: GEMV + AllReduce (decode shape) against the oracle.

The full decode workload (8 ranks, 8 tokens, K=3584, N=8192) is checked in
full: the oracle computes all 8 x 8192 outputs.  Small cases cover ragged N,
K and token counts 1..16, and every rank's buffer must hold the same bits.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_close, bits, dev_bf16, empty, to_f64

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_collective_gb300 as fcc  # noqa: E402


def _run(R, A, B, M, N, K, out_dtype=fcc.FCC_F32, opts=None):
    """opts None: the fused kernel (asked for explicitly: AUTO may pick the
    plain form for shapes with few column groups)."""
    if opts is None:
        opts = fcc.make_opts(algo=fcc.FCC_ALGO_FUSED)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    tdt = torch.float32 if out_dtype == fcc.FCC_F32 else torch.bfloat16
    outs = [empty((M, N), tdt, fill=float("nan")) for _ in range(R)]
    fcc.fcc_gemv_ar(R, dA, dB, outs, M, N, K, fcc.FCC_BF16, out_dtype, opts)
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    return outs


@pytest.mark.parametrize("R,M,N,K", [(8, 8, 1024, 256), (3, 5, 1000, 200), (1, 1, 128, 64),
                                     (2, 16, 136, 72), (4, 8, 2056, 3584), (8, 13, 384, 8)])
def test_gemv_small(R, M, N, K):
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=R + M + K)
    outs = _run(R, A, B, M, N, K)
    ref = oracle.gemv_ar(A, B)
    assert_close(to_f64(outs[0]), ref)
    for r in range(1, R):
        assert np.array_equal(bits(outs[r]), bits(outs[0])), f"rank {r} buffer differs"


def test_gemv_integer_exact():
    R, M, N, K = 4, 8, 512, 128
    A, B = synth.integer_gemm_inputs(R, M, N, K, -3, 3, seed=9)
    outs = _run(R, A, B, M, N, K)
    assert np.array_equal(to_f64(outs[0]), oracle.gemv_ar(A, B))


def test_gemv_bf16_output_and_repeatable():
    R, M, N, K = 8, 8, 1024, 512
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=3)
    o1 = _run(R, A, B, M, N, K, fcc.FCC_BF16)
    o2 = _run(R, A, B, M, N, K, fcc.FCC_BF16)
    assert_close(to_f64(o1[0]), oracle.gemv_ar(A, B))
    assert np.array_equal(bits(o1[0]), bits(o2[0]))


@pytest.mark.parametrize("ctas", [1, 7, 64])
def test_gemv_grid_sizes(ctas):
    """The stream-K split and the last-arriver sum hold for any grid size."""
    R, M, N, K = 4, 8, 1024, 448
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=5)
    outs = _run(R, A, B, M, N, K, opts=fcc.make_opts(algo=fcc.FCC_ALGO_FUSED, max_ctas=ctas))
    assert_close(to_f64(outs[0]), oracle.gemv_ar(A, B))


@pytest.mark.parametrize("algo", [2, 4])
def test_gemv_unfused_baselines(algo):
    R, M, N, K = 8, 8, 1024, 256
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=6)
    outs = _run(R, A, B, M, N, K, opts=fcc.make_opts(algo=algo))
    ref = oracle.gemv_ar(A, B)
    for r in range(R):
        assert_close(to_f64(outs[r]), ref)


@pytest.mark.parametrize("N,want", [(512, fcc.FCC_ALGO_UNFUSED), (8192, fcc.FCC_ALGO_FUSED)])
def test_gemv_auto_follows_the_selector(N, want):
    """AUTO runs what fcc_choose_algo names (the plain form launches two
    kernels, the fused one), and either is correct."""
    R, M, K = 8, 8, 512
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=N)
    assert fcc.fcc_choose_algo(fcc.FCC_OP_GEMV_AR, R, M, N, K) == want
    l0 = fcc.fcc_launch_count()
    outs = _run(R, A, B, M, N, K, opts=fcc.make_opts())
    assert fcc.fcc_launch_count() - l0 == (2 if want == fcc.FCC_ALGO_UNFUSED else 1)
    assert_close(to_f64(outs[0]), oracle.gemv_ar(A, B))


def test_gemv_full_decode_workload():
    w = synth.WORKLOADS["gemv_ar_r8_8x8192x3584"]
    A, B = synth.gemm_inputs(w.R, w.M, w.N, w.K, w.std_a, w.std_b, seed=0)
    outs = _run(w.R, A, B, w.M, w.N, w.K)
    ref = oracle.gemv_ar(A, B)
    fro, mx = assert_close(to_f64(outs[0]), ref, "decode workload")
    # f32 output: only f32 accumulation rounding over K' = R*K = 28672 terms,
    # typically ~sqrt(K') * 2^-24 = 1e-5 relative; 1e-4 leaves a 10x margin.
    assert fro < 1e-4
    for r in range(1, w.R):
        assert np.array_equal(bits(outs[r]), bits(outs[0]))


@pytest.mark.parametrize("R,M,N,K,ctas", [(8, 8, 8192, 3584, 0), (4, 16, 2048, 1024, 64),
                                          (2, 3, 1032, 512, 24)])
def test_cluster_and_ticket_final_sums_agree_bitwise(R, M, N, K, ctas):
    """Where the splits of a column group fit on the device as one cluster,
    they add their partials through distributed shared memory; the entry point
    that allocates nothing always uses arrival tickets and partials in memory.
    With the same split count both add the same values in the same order, so
    the outputs are bit-identical (and match the oracle)."""
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=N + M)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    o = fcc.make_opts(algo=fcc.FCC_ALGO_FUSED, max_ctas=ctas)
    a = [empty((M, N), torch.float32, fill=float("nan")) for _ in range(R)]
    b = [empty((M, N), torch.float32, fill=float("nan")) for _ in range(R)]
    fcc.fcc_gemv_ar(R, dA, dB, a, M, N, K, fcc.FCC_BF16, fcc.FCC_F32, o)
    fcc.fcc_gemv_ar_static(R, dA, dB, b, M, N, K, fcc.FCC_BF16, fcc.FCC_F32, o)
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    assert_close(to_f64(a[0]), oracle.gemv_ar(A, B))
    for r in range(R):
        assert np.array_equal(bits(a[r]), bits(b[r])), f"rank {r}"
