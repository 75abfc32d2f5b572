"""The GEMV + AllReduce entry point that allocates nothing (fcc_gemv_ar_static).

Some callers cannot call cudaMalloc: a process whose device memory is already
reserved by its own allocator, or a latency-critical path that cannot take the
implicit device synchronisation of cudaMalloc/cudaFree.  For them the library
has a variant of the GEMV + AllReduce kernel whose scratch lives in a static
device array.  These tests call it through the C ABI twice in a row (the
second call reuses the array the first left behind) and check each result
against the fp64 oracle with the float tolerance of the other parity tests,
and against the ordinary entry point, fcc_gemv_ar.  One case is sized so that
the default number of CTAs per column group does not fit in the array and the
call runs with fewer; a size beyond the array's limit must be refused.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one.
"""
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_close, dev_bf16, empty, to_f64

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_collective_gb300 as fcc  # noqa: E402


# (8, 16, 16384, 3584): 32 column groups of 512; the default 152 // 32 = 4
# CTAs per group need 32 x 4 x 16 x 2 KiB = 4 MiB, more than the array's
# 4 MiB - 4 KiB, so the call caps itself at 3 per group.
@pytest.mark.parametrize("R,M,N,K", [(8, 8, 8192, 3584), (3, 5, 1000, 200),
                                     (8, 16, 16384, 3584)])
def test_static_scratch_matches_oracle_twice(R, M, N, K):
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=31 + R)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    ref = oracle.gemv_ar(A, B)
    alloc = [empty((M, N), torch.float32, fill=float("nan")) for _ in range(R)]
    fcc.fcc_gemv_ar(R, dA, dB, alloc, M, N, K, fcc.FCC_BF16, fcc.FCC_F32)
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    for call in range(2):
        outs = [empty((M, N), torch.float32, fill=float("nan")) for _ in range(R)]
        fcc.fcc_gemv_ar_static(R, dA, dB, outs, M, N, K, fcc.FCC_BF16, fcc.FCC_F32)
        assert fcc.fcc_stream_status() == fcc.FCC_OK, f"call {call}"
        for r in range(R):
            got = to_f64(outs[r])
            assert_close(got, ref, f"call {call} rank {r} vs oracle")
            assert_close(got, to_f64(alloc[r]), f"call {call} rank {r} vs fcc_gemv_ar")


def test_static_scratch_size_limit_is_refused():
    R, M, K = 1, 16, 64
    N = 512 * 128  # 128 column groups x 16 tokens x 2 KiB = 4 MiB: more than the array holds
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 0.02, seed=3)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    outs = [empty((M, N), torch.float32) for _ in range(R)]
    before = fcc.fcc_launch_count()
    with pytest.raises(fcc.FccError) as e:
        fcc.fcc_gemv_ar_static(R, dA, dB, outs, M, N, K, fcc.FCC_BF16, fcc.FCC_F32)
    assert e.value.status == fcc.FCC_ERR_WORKSPACE
    assert fcc.fcc_launch_count() == before
