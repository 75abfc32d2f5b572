"""The GEMV + AllReduce entry point that allocates nothing (fcc_gemv_ar_static).

Some callers cannot call cudaMalloc: a process whose device memory is already
reserved by its own allocator, or a latency-critical path that cannot take the
implicit device synchronisation of cudaMalloc/cudaFree.  For them the library
has a variant of the GEMV + AllReduce kernel whose scratch lives in a static
device array.  This test calls it through the C ABI twice in a row (the second
call reuses the array the first left behind) and checks each result against
the ordinary entry point, fcc_gemv_ar, with the float tolerance of the other
parity tests, and that a size beyond the array's limit is refused.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one.
"""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import assert_close, dev_bf16, empty, to_f64

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_collective_gb300 as fcc  # noqa: E402


@pytest.mark.parametrize("R,M,N,K", [(8, 8, 8192, 3584), (3, 5, 1000, 200)])
def test_static_scratch_matches_allocating_entry_point(R, M, N, K):
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=31 + R)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    ref = [empty((M, N), torch.float32, fill=float("nan")) for _ in range(R)]
    fcc.fcc_gemv_ar(R, dA, dB, ref, M, N, K, fcc.FCC_BF16, fcc.FCC_F32)
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    expect = to_f64(ref[0])
    for call in range(2):
        outs = [empty((M, N), torch.float32, fill=float("nan")) for _ in range(R)]
        fcc.fcc_gemv_ar_static(R, dA, dB, outs, M, N, K, fcc.FCC_BF16, fcc.FCC_F32)
        assert fcc.fcc_stream_status() == fcc.FCC_OK, f"call {call}"
        for r in range(R):
            assert_close(to_f64(outs[r]), expect, f"call {call} rank {r}")


def test_static_scratch_size_limit_is_refused():
    R, M, K = 1, 16, 64
    N = 512 * 128  # 128 column groups x 16 tokens x 2 KiB per CTA: more than the array holds
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=3)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    outs = [empty((M, N), torch.float32) for _ in range(R)]
    before = fcc.fcc_launch_count()
    with pytest.raises(fcc.FccError) as e:
        fcc.fcc_gemv_ar_static(R, dA, dB, outs, M, N, K, fcc.FCC_BF16, fcc.FCC_F32)
    assert e.value.status == fcc.FCC_ERR_WORKSPACE
    assert fcc.fcc_launch_count() == before
    assert np.isfinite(1.0)
