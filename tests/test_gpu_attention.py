"""GPU parity: ring attention over R sequence shards against the fp64 oracle.

Each case goes through the C ABI; every output row (or a sample at full size)
is compared with exact softmax attention over all shards' keys and values.
Shapes cover ragged shard lengths (not multiples of the 128-row tiles), one
and several heads, one rank, and the causal mask across shard boundaries.
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


def _run(Q, K, V, causal, out_dtype=fcc.FCC_BF16):
    R = len(Q)
    S, H, d = Q[0].shape
    dq, dk, dv = ([dev_bf16(x) for x in X] for X in (Q, K, V))
    tdt = torch.float32 if out_dtype == fcc.FCC_F32 else torch.bfloat16
    O = [empty((S, H, d), tdt, fill=float("nan")) for _ in range(R)]
    fcc.fcc_ring_attention(R, dq, dk, dv, O, S, H, d, causal, fcc.FCC_BF16, out_dtype)
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    return O


# S = 40 and 64: the second half of every key block is past the shard's end.
@pytest.mark.parametrize("R,S,H", [(2, 128, 1), (2, 200, 2), (3, 256, 2), (1, 300, 1),
                                   (4, 96, 3), (2, 513, 1), (2, 40, 2), (3, 64, 1),
                                   (8, 130, 1), (8, 384, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_attention_small(R, S, H, causal):
    Q, K, V = synth.attention_inputs(R, S, H, 128, seed=R * 1000 + S + H)
    O = _run(Q, K, V, causal)
    ref = oracle.ring_attention(Q, K, V, causal)
    for r in range(R):
        assert_close(to_f64(O[r]).reshape(-1, 128), ref[r].reshape(-1, 128), f"rank {r}")


def test_ring_attention_f32_output_and_repeatable():
    Q, K, V = synth.attention_inputs(2, 256, 2, 128, seed=7)
    a = _run(Q, K, V, True, fcc.FCC_F32)
    b = _run(Q, K, V, True, fcc.FCC_F32)
    ref = oracle.ring_attention(Q, K, V, True)
    for r in range(2):
        assert np.array_equal(bits(a[r]), bits(b[r]))
        assert_close(to_f64(a[r]).reshape(-1, 128), ref[r].reshape(-1, 128), f"rank {r}")


def test_ring_attention_zero_queries_average_the_values():
    """Q = 0: every weight is equal, so each output is the mean of the values
    it may see (all of them, or positions <= its own with the mask)."""
    R, S, H = 2, 160, 1
    Q, K, V = synth.attention_inputs(R, S, H, 128, seed=8)
    Q = [np.zeros_like(q) for q in Q]
    for causal in (False, True):
        O = _run(Q, K, V, causal, fcc.FCC_F32)
        ref = oracle.ring_attention(Q, K, V, causal)
        for r in range(R):
            assert_close(to_f64(O[r]).reshape(-1, 128), ref[r].reshape(-1, 128), f"rank {r}")


def test_ring_attention_invalid_arguments():
    Q, K, V = synth.attention_inputs(2, 16, 1, 64, seed=9)
    dq, dk, dv = ([dev_bf16(x) for x in X] for X in (Q, K, V))
    O = [empty((16, 1, 64), torch.bfloat16) for _ in range(2)]
    with pytest.raises(fcc.FccError) as e:
        fcc.fcc_ring_attention(2, dq, dk, dv, O, 16, 1, 64)          # d = 64
    assert e.value.status == fcc.FCC_ERR_UNSUPPORTED
    with pytest.raises(fcc.FccError) as e:
        fcc.fcc_ring_attention(0, dq, dk, dv, O, 16, 1, 128)
    assert e.value.status == fcc.FCC_ERR_INVALID


@pytest.mark.parametrize("causal", [False, True])
def test_ring_attention_full_workload_sampled(causal):
    """8 ranks x 4096 positions (32768 in all), 8 heads of 128: 32 sampled rows."""
    w = synth.WORKLOADS["attn_r8_s4096_h8_d128"]
    Q, K, V = synth.attention_inputs(w.R, w.M, w.H, w.K, seed=0)
    O = _run(Q, K, V, causal)
    rng = np.random.Generator(np.random.PCG64(2))
    rk = rng.integers(0, w.R, size=32)
    rw = rng.integers(0, w.M, size=32)
    hd = rng.integers(0, w.H, size=32)
    ref = oracle.attention_rows(Q, K, V, causal, rk, rw, hd)
    got = np.stack([to_f64(O[a][b, c]) for a, b, c in zip(rk, rw, hd)])
    assert_close(got, ref, "sampled rows")


@pytest.mark.parametrize("causal", [False, True])
def test_ring_attention_growing_scores_rescale(causal):
    """Scores that grow along the sequence (key row j = 0.002 j in every
    component, query rows of ones): each row's running maximum is raised every
    couple of blocks, so the accumulator rescaling is exercised throughout."""
    R, S, H, d = 2, 512, 1, 128
    _, _, V = synth.attention_inputs(R, S, H, d, seed=12)
    Q = [synth.f32_to_bf16_bits(np.ones((S, H, d), np.float32)) for _ in range(R)]
    K = []
    for r in range(R):
        j = (r * S + np.arange(S, dtype=np.float32))[:, None, None]
        K.append(synth.f32_to_bf16_bits(np.broadcast_to(0.002 * j, (S, H, d)).astype(np.float32)))
    O = _run(Q, K, V, causal, fcc.FCC_F32)
    ref = oracle.ring_attention(Q, K, V, causal)
    for r in range(R):
        assert_close(to_f64(O[r]).reshape(-1, d), ref[r].reshape(-1, d), f"rank {r}")


@pytest.mark.parametrize("causal", [False, True])
def test_ring_attention_mixed_rescale_within_a_warp(causal):
    """The same growing keys, but query row i is (0, 1/2, 1 or 2 by i mod 4)
    times ones: neighbouring rows of one warp raise their maximum every
    block, every second or fourth block, or never, so blocks where only some
    rows of a warp need a raise are redone while the others keep theirs."""
    R, S, H, d = 2, 640, 2, 128
    _, _, V = synth.attention_inputs(R, S, H, d, seed=13)
    gain = np.array([0.0, 0.5, 1.0, 2.0], np.float32)[np.arange(S) % 4]
    Q = [synth.f32_to_bf16_bits(np.broadcast_to(gain[:, None, None], (S, H, d)).astype(np.float32))
         for _ in range(R)]
    K = []
    for r in range(R):
        j = (r * S + np.arange(S, dtype=np.float32))[:, None, None]
        K.append(synth.f32_to_bf16_bits(np.broadcast_to(0.002 * j, (S, H, d)).astype(np.float32)))
    O = _run(Q, K, V, causal, fcc.FCC_F32)
    ref = oracle.ring_attention(Q, K, V, causal)
    for r in range(R):
        assert_close(to_f64(O[r]).reshape(-1, d), ref[r].reshape(-1, d), f"rank {r}")
