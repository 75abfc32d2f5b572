"""GPU parity: embedding + all-to-all (DLRM pooled lookups) against the oracle.

Every case goes through the C ABI and compares with the fp64 oracle on the
same seeded tables and bags: pooled rows within the float tolerance, placed
at (rank g / Bl, sample g % Bl, table t).  Row widths cover 16-byte vector
counts that are not powers of two and widths beyond one warp's step; bags
cover empty ones and ones longer than 32 rows.
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


def _upload(tables, offsets, indices):
    dt = [dev_bf16(t) for t in tables]
    do = [torch.from_numpy(o).cuda() for o in offsets]
    di = [torch.from_numpy(i).cuda() for i in indices]
    return dt, do, di


def _run(R, ntab, V, D, Bl, dt, do, di, out_dtype=fcc.FCC_BF16, algo=fcc.FCC_ALGO_AUTO):
    tdt = torch.float32 if out_dtype == fcc.FCC_F32 else torch.bfloat16
    out = [empty((Bl, ntab, D), tdt, fill=float("nan")) for _ in range(R)]
    fcc.fcc_embedding_a2a(R, ntab, dt, V, D, Bl, do, di, out, fcc.FCC_BF16, out_dtype,
                          fcc.make_opts(algo=algo))
    st = fcc.fcc_stream_status()
    return out, st


CASES = [
    # R, tables, V, D, Bl, L, min_bag
    (2, 4, 100, 128, 16, 8, 1),
    (4, 8, 1000, 64, 33, 5, 0),      # empty bags
    (1, 3, 50, 96, 20, 40, 1),       # 12 vectors a row (not a power of two); bags > 32
    (8, 16, 500, 8, 10, 3, 0),       # one vector a row: 32 rows a step
    (2, 2, 300, 512, 7, 4, 1),       # 64 vectors a row: two passes of 32
    (2, 2, 100, 264, 5, 3, 1),       # 33 vectors a row
]


@pytest.mark.parametrize("R,ntab,V,D,Bl,L,min_bag", CASES)
@pytest.mark.parametrize("algo", [fcc.FCC_ALGO_FUSED, fcc.FCC_ALGO_UNFUSED, fcc.FCC_ALGO_CE])
@pytest.mark.parametrize("out_dtype", [fcc.FCC_BF16, fcc.FCC_F32])
def test_embedding_a2a_small(R, ntab, V, D, Bl, L, min_bag, algo, out_dtype):
    tables, offsets, indices = synth.embedding_inputs(R, ntab, V, D, Bl, L, min_bag=min_bag,
                                                      seed=R * 100 + D)
    ref = oracle.embedding_a2a(tables, offsets, indices, R)
    out, st = _run(R, ntab, V, D, Bl, *_upload(tables, offsets, indices), out_dtype, algo)
    assert st == fcc.FCC_OK
    for r in range(R):
        assert_close(to_f64(out[r]).reshape(-1, D), ref[r].reshape(-1, D), f"rank {r}")


def test_embedding_forms_agree_bitwise_and_repeat():
    """Fused, staged and copy-engine forms pool in the same order: same bits."""
    R, ntab, V, D, Bl, L = 4, 8, 2000, 128, 64, 20
    tables, offsets, indices = synth.embedding_inputs(R, ntab, V, D, Bl, L, seed=5)
    dev = _upload(tables, offsets, indices)
    base, _ = _run(R, ntab, V, D, Bl, *dev, fcc.FCC_F32, fcc.FCC_ALGO_FUSED)
    for algo in (fcc.FCC_ALGO_FUSED, fcc.FCC_ALGO_UNFUSED, fcc.FCC_ALGO_CE):
        again, st = _run(R, ntab, V, D, Bl, *dev, fcc.FCC_F32, algo)
        assert st == fcc.FCC_OK
        for r in range(R):
            assert np.array_equal(bits(again[r]), bits(base[r])), f"algo {algo} rank {r}"


def test_embedding_bad_index_skipped_and_reported():
    """An index outside [0, V) is not read: its bag skips that row, the status
    word says FCC_ERR_INVALID, every other bag is unchanged."""
    R, ntab, V, D, Bl, L = 2, 2, 64, 32, 8, 4
    tables, offsets, indices = synth.embedding_inputs(R, ntab, V, D, Bl, L, seed=9)
    g = 5
    k = int(offsets[1][g])
    good = [i.copy() for i in indices]
    indices[1][k] = V + 1000
    out, st = _run(R, ntab, V, D, Bl, *_upload(tables, offsets, indices), fcc.FCC_F32)
    assert st == fcc.FCC_ERR_INVALID
    assert fcc.fcc_stream_status() == fcc.FCC_OK       # the word was cleared by reading it
    ref = oracle.embedding_a2a(tables, offsets, good, R)
    row = oracle.embedding_bags(tables, offsets, good, [1], [g])[0]
    drop = oracle.embedding_bags([tables[1]], [np.array([0, 1], dtype=np.int32)],
                                 [good[1][k:k + 1]], [0], [0])[0]     # the skipped row
    ref[g // Bl][g % Bl, 1] = row - drop
    for r in range(R):
        assert_close(to_f64(out[r]).reshape(-1, D), ref[r].reshape(-1, D), f"rank {r}")


def test_embedding_invalid_arguments():
    R, ntab, V, D, Bl = 2, 4, 10, 16, 4
    tables, offsets, indices = synth.embedding_inputs(R, ntab, V, D, Bl, 2, seed=3)
    dt, do, di = _upload(tables, offsets, indices)
    out = [empty((Bl, ntab, D), torch.bfloat16) for _ in range(R)]
    for kw in [dict(ntab=3), dict(D=12), dict(R=0)]:
        a = dict(R=R, ntab=ntab, D=D)
        a.update(kw)
        with pytest.raises(fcc.FccError) as e:
            fcc.fcc_embedding_a2a(a["R"], a["ntab"], dt, V, a["D"], Bl, do, di, out)
        assert e.value.status == fcc.FCC_ERR_INVALID
    with pytest.raises(fcc.FccError) as e:
        fcc.fcc_embedding_a2a(R, ntab, dt, V, D, Bl, do, di, out, fcc.FCC_F32)
    assert e.value.status == fcc.FCC_ERR_UNSUPPORTED


def test_embedding_full_workload_sampled():
    """The benchmark's workload (8 ranks, 64 tables of 65536 x 128, 2048 samples
    a rank, bags of 32 on average) on 64 sampled (table, sample) bags."""
    w = synth.WORKLOADS["emb_a2a_r8_t64_v65536_d128_b2048_l32"]
    tables, offsets, indices = synth.embedding_inputs(w.R, w.tables, w.V, w.D, w.B, w.L,
                                                      std=w.std_a, seed=0)
    dev = _upload(tables, offsets, indices)
    rng = np.random.Generator(np.random.PCG64(1))
    g = rng.integers(0, w.R * w.B, size=64)
    t = rng.integers(0, w.tables, size=64)
    ref = oracle.embedding_bags(tables, offsets, indices, t, g)
    for algo in (fcc.FCC_ALGO_AUTO, fcc.FCC_ALGO_FUSED):  # (AUTO is the staged form)
        out, st = _run(w.R, w.tables, w.V, w.D, w.B, *dev, algo=algo)
        assert st == fcc.FCC_OK
        got = np.stack([to_f64(out[gi // w.B][gi % w.B, ti]) for gi, ti in zip(g, t)])
        assert_close(got, ref, f"sampled bags (algo {algo})")
