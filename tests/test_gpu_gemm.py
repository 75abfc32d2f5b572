"""GPU parity: fused GEMM + ReduceScatter / AllReduce / AllGather against the oracle.

Every case calls the library through its C ABI (the ctypes binding) and
compares element by element with the fp64 CPU oracle on the same seeded
inputs.  Small shapes cover several tiles and ragged tails in M, N and K;
the full-size row-parallel MLP shape (8 ranks, 8192 x 8192 x 3584) is checked
on sampled rows the oracle computes one by one.
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


def _upload(A, B):
    return [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]


def _rs(R, dA, dB, M, N, K, out_dtype, opts=None):
    tdt = torch.float32 if out_dtype == fcc.FCC_F32 else torch.bfloat16
    outs = [empty((M // R, N), tdt, fill=float("nan")) for _ in range(R)]
    fcc.fcc_gemm_rs(R, dA, dB, outs, M, N, K, fcc.FCC_BF16, out_dtype, opts)
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    return outs


def _ar(R, dA, dB, M, N, K, out_dtype, opts=None):
    tdt = torch.float32 if out_dtype == fcc.FCC_F32 else torch.bfloat16
    outs = [empty((M, N), tdt, fill=float("nan")) for _ in range(R)]
    fcc.fcc_gemm_ar(R, dA, dB, outs, M, N, K, fcc.FCC_BF16, out_dtype, opts)
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    return outs


# ------------------------------------------------------------ exactness first

@pytest.mark.parametrize("pair", [1, 2])
def test_rs_integer_inputs_bit_exact(pair):
    """Small integers: every f32 partial sum is exact, so GPU == oracle exactly."""
    R, M, N, K = 2, 512, 512, 128
    A, B = synth.integer_gemm_inputs(R, M, N, K, -4, 4, seed=1)
    dA, dB = _upload(A, B)
    outs = _rs(R, dA, dB, M, N, K, fcc.FCC_F32, fcc.make_opts(cta_pair=pair))
    for j in range(R):
        assert np.array_equal(to_f64(outs[j]), oracle.gemm_rs(A, B, j)), f"shard {j}"


def test_rs_one_hot_selects_b_rows():
    """A_r one-hot: the output is a sum of exact B rows (catches layout/descriptor errors)."""
    R, M, N, K = 2, 128, 512, 256
    rng = np.random.Generator(np.random.PCG64(2))
    A, B = [], []
    for r in range(R):
        a = np.zeros((M, K), np.float32)
        a[np.arange(M), rng.integers(0, K, M)] = 1.0
        A.append(synth.f32_to_bf16_bits(a))
        B.append(synth.integer_bf16(rng, (K, N), -8, 8))
    dA, dB = _upload(A, B)
    outs = _rs(R, dA, dB, M, N, K, fcc.FCC_F32)
    for j in range(R):
        assert np.array_equal(to_f64(outs[j]), oracle.gemm_rs(A, B, j))


# ------------------------------------------------------ the 2-rank workload

def test_rs_two_rank_workload_f32():
    w = synth.WORKLOADS["gemm_rs_r2_256x256x128"]
    A, B = synth.gemm_inputs(w.R, w.M, w.N, w.K, w.std_a, w.std_b, seed=0)
    dA, dB = _upload(A, B)
    outs = _rs(w.R, dA, dB, w.M, w.N, w.K, fcc.FCC_F32)
    for j in range(w.R):
        fro, mx = assert_close(to_f64(outs[j]), oracle.gemm_rs(A, B, j), f"shard {j}")
        assert fro < 1e-5  # f32 output: only f32 accumulation rounding
    again = _rs(w.R, dA, dB, w.M, w.N, w.K, fcc.FCC_F32)
    for j in range(w.R):
        assert np.array_equal(bits(outs[j]), bits(again[j])), "not bitwise repeatable"


# ------------------------------------------------------------ ragged shapes

RAGGED = [
    (3, 360, 200, 72),     # shard rows 120, N and K not tile multiples
    (1, 136, 264, 8),      # one rank, K = 8
    (4, 512, 1032, 200),   # several tiles in M and N, ragged N
    (8, 1024, 520, 136),
]


@pytest.mark.parametrize("R,M,N,K", RAGGED)
@pytest.mark.parametrize("out_dtype", [0, 2])
@pytest.mark.parametrize("pair", [1, 2])
def test_rs_ragged(R, M, N, K, out_dtype, pair):
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=R * 7 + K)
    dA, dB = _upload(A, B)
    outs = _rs(R, dA, dB, M, N, K, out_dtype, fcc.make_opts(cta_pair=pair))
    for j in range(R):
        assert_close(to_f64(outs[j]), oracle.gemm_rs(A, B, j), f"shard {j}")


@pytest.mark.parametrize("R,M,N,K", [(4, 200, 264, 136), (2, 130, 16, 64), (8, 256, 256, 64),
                                     (4, 1032, 264, 128)])
@pytest.mark.parametrize("pair", [0, 1, 2])
def test_ar_all_buffers_identical_and_equal_rs(R, M, N, K, pair):
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=3)
    dA, dB = _upload(A, B)
    o = fcc.make_opts(cta_pair=pair)
    outs = _ar(R, dA, dB, M, N, K, fcc.FCC_BF16, o)
    ref = oracle.gemm_ar(A, B)
    assert_close(to_f64(outs[0]), ref, "ar")
    for r in range(1, R):
        assert np.array_equal(bits(outs[r]), bits(outs[0])), f"rank {r} differs"
    if M % R == 0:
        shards = _rs(R, dA, dB, M, N, K, fcc.FCC_BF16, o)
        cat = np.concatenate([bits(s) for s in shards])
        assert np.array_equal(cat, bits(outs[0])), "RS shards != AR rows (deterministic mode)"


# (pair, N, max_ctas that leave a short last round, max_ctas that leave none):
# 32 single-CTA tiles on 10 / 8 CTAs; 16 pair tiles on 5 / 4 pairs.
HALF_CASES = [(1, 1024, 10, 8), (2, 1024, 10, 8)]


@pytest.mark.parametrize("pair,N,split_ctas,whole_ctas", HALF_CASES)
@pytest.mark.parametrize("op", ["rs", "ar"])
def test_last_round_half_tiles_bit_identical(op, pair, N, split_ctas, whole_ctas):
    """The last round's tiles run as two 128-column halves when they fill at most
    half the grid.  Integer inputs keep every partial sum exact: the split and
    the unsplit launch both equal the oracle bit for bit."""
    R, M, K = 2, 1024, 128
    A, B = synth.integer_gemm_inputs(R, M, N, K, -4, 4, seed=11)
    dA, dB = _upload(A, B)
    run = _rs if op == "rs" else _ar
    split = run(R, dA, dB, M, N, K, fcc.FCC_F32,
                fcc.make_opts(cta_pair=pair, max_ctas=split_ctas))
    whole = run(R, dA, dB, M, N, K, fcc.FCC_F32,
                fcc.make_opts(cta_pair=pair, max_ctas=whole_ctas))
    for j in range(R):
        assert np.array_equal(bits(split[j]), bits(whole[j])), f"buffer {j}"
        ref = oracle.gemm_rs(A, B, j) if op == "rs" else oracle.gemm_ar(A, B)
        assert np.array_equal(to_f64(split[j]), ref), f"buffer {j} vs oracle"


# (pair, max_ctas, N): launches of more than one round whose last round holds
# at most half a round of tiles, which then run as two K halves each:
# 16 pair tiles on 5 pairs (one split tile), 32 single-CTA tiles on 10 CTAs
# (two), a narrow last column tile (N % 256 = 128) and a ragged one (136).
KSPLIT_CASES = [(2, 10, 1024), (1, 10, 1024), (1, 10, 896), (2, 10, 904)]


@pytest.mark.parametrize("pair,ctas,N", KSPLIT_CASES)
@pytest.mark.parametrize("out_dtype", [fcc.FCC_BF16, fcc.FCC_F32])
def test_last_round_k_halves(pair, ctas, N, out_dtype):
    """Float inputs: the K-split last round matches the oracle within the
    tolerance, repeats bit for bit, gives the AllReduce the reduce-scatter's
    rows bit for bit, and agrees with the column-halves form (a caller
    workspace too small for the partial sums) within the tolerance."""
    R, M, K = 4, 1024, 256
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=N + pair)
    dA, dB = _upload(A, B)
    o = fcc.make_opts(cta_pair=pair, max_ctas=ctas)
    rs = _rs(R, dA, dB, M, N, K, out_dtype, o)
    again = _rs(R, dA, dB, M, N, K, out_dtype, o)
    ar = _ar(R, dA, dB, M, N, K, out_dtype, o)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    halves = _rs(R, dA, dB, M, N, K, out_dtype,
                 fcc.make_opts(cta_pair=pair, max_ctas=ctas, workspace=ws, workspace_bytes=256))
    Ms = M // R
    for j in range(R):
        ref = oracle.gemm_rs(A, B, j)
        assert_close(to_f64(rs[j]), ref, f"shard {j}")
        assert_close(to_f64(halves[j]), ref, f"column halves, shard {j}")
        assert np.array_equal(bits(rs[j]), bits(again[j])), "not bitwise repeatable"
        assert np.array_equal(bits(rs[j]), bits(ar[0])[j * Ms:(j + 1) * Ms]), "RS != AR rows"
    for r in range(1, R):
        assert np.array_equal(bits(ar[r]), bits(ar[0]))


def test_last_round_k_halves_caller_workspace():
    """The size query covers the K halves' partial sums: a caller workspace of
    that size gives the same bits as the library's own pool."""
    R, M, N, K = 2, 1024, 1024, 128
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=77)
    dA, dB = _upload(A, B)
    o = fcc.make_opts(cta_pair=2, max_ctas=10)
    need = fcc.fcc_workspace_size(fcc.FCC_OP_GEMM_RS, R, M, N, K, o)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    own = _rs(R, dA, dB, M, N, K, fcc.FCC_F32, o)
    given = _rs(R, dA, dB, M, N, K, fcc.FCC_F32,
                fcc.make_opts(cta_pair=2, max_ctas=10, workspace=ws, workspace_bytes=need))
    for j in range(R):
        assert np.array_equal(bits(own[j]), bits(given[j]))
        assert_close(to_f64(given[j]), oracle.gemm_rs(A, B, j))


@pytest.mark.parametrize("R,M,N,K", [(2, 1024, 136, 64), (4, 512, 128, 192), (2, 2048, 264, 64)])
def test_single_ctas_match_pairs_bitwise(R, M, N, K):
    """One CTA per 128-row tile against a CTA pair per 256-row tile: the same K
    order per element, so bit-identical outputs; narrow last column tiles
    (N % 256 <= 128) included."""
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=R + N)
    dA, dB = _upload(A, B)
    one = _rs(R, dA, dB, M, N, K, fcc.FCC_F32, fcc.make_opts(cta_pair=1))
    two = _rs(R, dA, dB, M, N, K, fcc.FCC_F32, fcc.make_opts(cta_pair=2))
    for j in range(R):
        assert np.array_equal(bits(one[j]), bits(two[j])), f"shard {j}"
        assert_close(to_f64(two[j]), oracle.gemm_rs(A, B, j), f"shard {j}")


@pytest.mark.parametrize("pair,ctas", [(1, 8), (2, 8)])
def test_phase_timing_stamps(pair, ctas):
    """opts.phase_ns: every CTA records its span, its epilogue's busy time (at
    most the span), its MMA warp's wait for the epilogue and its tiles; the
    tiles add up to the launch's work items (a pair's two CTAs each store half
    of every tile), and the results are unchanged."""
    R, M, N, K = 2, 1024, 1024, 128
    A, B = synth.integer_gemm_inputs(R, M, N, K, -4, 4, seed=41)
    dA, dB = _upload(A, B)
    buf = torch.zeros(4 * 64, dtype=torch.int64, device="cuda")
    outs = _rs(R, dA, dB, M, N, K, fcc.FCC_F32,
               fcc.make_opts(cta_pair=pair, max_ctas=ctas, phase_ns=buf))
    for j in range(R):
        assert np.array_equal(to_f64(outs[j]), oracle.gemm_rs(A, B, j))
    t = buf.view(-1, 4).cpu().numpy()
    used = t[:ctas]
    assert np.all(t[ctas:] == 0), "stamps beyond the grid"
    assert np.all(used[:, 0] > 0)
    assert np.all(used[:, 1] <= used[:, 0]) and np.all(used[:, 2] <= used[:, 0])
    tiles = (M // (128 * pair)) * (N // 256)
    assert used[:, 3].sum() == tiles * pair


def test_rank_permutation_within_tolerance():
    R, M, N, K = 4, 256, 512, 128
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=5)
    perm = [2, 0, 3, 1]
    dA, dB = _upload(A, B)
    a = _ar(R, dA, dB, M, N, K, fcc.FCC_F32)[0]
    b = _ar(R, [dA[p] for p in perm], [dB[p] for p in perm], M, N, K, fcc.FCC_F32)[0]
    assert_close(to_f64(b), to_f64(a), "permuted")


# ------------------------------------------------------- other algorithms

ALGOS = [
    ("push", dict(algo=1, deterministic=0)),
    ("unfused", dict(algo=2)),
    ("interdecom4", dict(algo=3, chunks=4)),
    ("interdecom_model", dict(algo=3, chunks=0)),
    ("ce", dict(algo=4)),
]


@pytest.mark.parametrize("name,kw", ALGOS)
@pytest.mark.parametrize("out_dtype", [0, 2])
@pytest.mark.parametrize("pair", [1, 2])
def test_rs_algorithms(name, kw, out_dtype, pair):
    R, M, N, K = 4, 640, 520, 192
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=11)
    dA, dB = _upload(A, B)
    outs = _rs(R, dA, dB, M, N, K, out_dtype, fcc.make_opts(cta_pair=pair, **kw))
    for j in range(R):
        assert_close(to_f64(outs[j]), oracle.gemm_rs(A, B, j), f"{name} shard {j}")


@pytest.mark.parametrize("name,kw", ALGOS)
def test_ar_algorithms(name, kw):
    R, M, N, K = 3, 264, 256, 128
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=12)
    dA, dB = _upload(A, B)
    ref = oracle.gemm_ar(A, B)
    for out_dtype in (0, 2):
        outs = _ar(R, dA, dB, M, N, K, out_dtype, fcc.make_opts(**kw))
        for r in range(R):
            assert_close(to_f64(outs[r]), ref, f"{name} rank {r}")


def test_caller_workspace_and_too_small():
    R, M, N, K = 2, 256, 256, 64
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=13)
    dA, dB = _upload(A, B)
    o = fcc.make_opts(algo=fcc.FCC_ALGO_UNFUSED)
    need = fcc.fcc_workspace_size(fcc.FCC_OP_GEMM_RS, R, M, N, K, o)
    assert need >= R * M * N * 4
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = fcc.make_opts(algo=fcc.FCC_ALGO_UNFUSED, workspace=ws, workspace_bytes=need)
    outs = _rs(R, dA, dB, M, N, K, fcc.FCC_F32, o)
    for j in range(R):
        assert_close(to_f64(outs[j]), oracle.gemm_rs(A, B, j))
    small = fcc.make_opts(algo=fcc.FCC_ALGO_UNFUSED, workspace=ws, workspace_bytes=need - 256)
    with pytest.raises(fcc.FccError) as e:
        _rs(R, dA, dB, M, N, K, fcc.FCC_F32, small)
    assert e.value.status == fcc.FCC_ERR_WORKSPACE


# ----------------------------------------------------------------- AG + GEMM

@pytest.mark.parametrize("R,Ms,N,K", [(4, 136, 200, 96), (2, 128, 512, 64), (8, 64, 264, 136),
                                      (2, 520, 264, 64)])
@pytest.mark.parametrize("algo,pair", [(1, 0), (1, 1), (2, 0), (3, 0), (4, 0)])
def test_ag_gemm(R, Ms, N, K, algo, pair):
    """A 256-row pair tile may span two shards (Ms = 136 with 4 ranks, Ms = 520
    with 2); pair = 1 runs one CTA per 128-row tile."""
    X, B = synth.gemm_inputs(R, Ms, N, K, 1.0, 1.0, seed=17 + R)
    dX, dB = _upload(X, B)
    M = R * Ms
    outs = [empty((M, N), torch.bfloat16, fill=float("nan")) for _ in range(R)]
    gath = [empty((M, K), torch.bfloat16, fill=0.0) for _ in range(R)]
    fcc.fcc_ag_gemm(R, dX, dB, outs, gath, M, N, K, fcc.FCC_BF16, fcc.FCC_BF16,
                    fcc.make_opts(algo=algo, cta_pair=pair))
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    full = np.concatenate(X)
    for r in range(R):
        assert_close(to_f64(outs[r]), oracle.ag_gemm(X, B, r), f"rank {r}")
        assert np.array_equal(bits(gath[r]).view(np.uint16), full), f"gathered copy {r}"


@pytest.mark.parametrize("chunks", [1, 2, 3, 64])
@pytest.mark.parametrize("gathered", [False, True])
def test_ag_gemm_interdecom_chunks(chunks, gathered):
    """InterDecom: the gather of each 256-row chunk runs on a side stream ahead
    of that chunk's GEMM; any chunk count (ragged last chunk, more chunks than
    tiles) gives the oracle's result, with or without the gathered copies."""
    R, Ms, N, K = 4, 200, 264, 136
    X, B = synth.gemm_inputs(R, Ms, N, K, 1.0, 1.0, seed=29)
    dX, dB = _upload(X, B)
    M = R * Ms
    outs = [empty((M, N), torch.float32, fill=float("nan")) for _ in range(R)]
    gath = [empty((M, K), torch.bfloat16, fill=0.0) for _ in range(R)] if gathered else None
    fcc.fcc_ag_gemm(R, dX, dB, outs, gath, M, N, K, fcc.FCC_BF16, fcc.FCC_F32,
                    fcc.make_opts(algo=fcc.FCC_ALGO_INTERDECOM, chunks=chunks))
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    full = np.concatenate(X)
    for r in range(R):
        fro, _ = assert_close(to_f64(outs[r]), oracle.ag_gemm(X, B, r), f"rank {r}")
        assert fro < 1e-5  # f32 output
        if gathered:
            assert np.array_equal(bits(gath[r]).view(np.uint16), full), f"gathered copy {r}"


def test_ag_gemm_without_gathered_output():
    R, Ms, N, K = 2, 200, 256, 128
    X, B = synth.gemm_inputs(R, Ms, N, K, 1.0, 1.0, seed=23)
    dX, dB = _upload(X, B)
    M = R * Ms
    outs = [empty((M, N), torch.float32) for _ in range(R)]
    fcc.fcc_ag_gemm(R, dX, dB, outs, None, M, N, K, fcc.FCC_BF16, fcc.FCC_F32)
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    for r in range(R):
        assert_close(to_f64(outs[r]), oracle.ag_gemm(X, B, r))


# ------------------------------------------------------------- full sizes

def _sample_rows(n, k, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = set(rng.choice(n, size=k - 3, replace=False).tolist())
    rows |= {0, n - 1, n // 2}
    return np.array(sorted(rows), dtype=np.int64)


def test_rs_full_size_sampled_rows():
    """The 8-rank 8192x8192x3584 workload, bf16 shards, in the benchmark's launch shape."""
    w = synth.WORKLOADS["gemm_rs_r8_8192x8192x3584"]
    A, B = synth.gemm_inputs(w.R, w.M, w.N, w.K, w.std_a, w.std_b, seed=0)
    dA, dB = _upload(A, B)
    outs = _rs(w.R, dA, dB, w.M, w.N, w.K, fcc.FCC_BF16)
    Ms = w.M // w.R
    for j in range(w.R):
        rows = _sample_rows(Ms, 8, seed=j)
        got = to_f64(outs[j][torch.from_numpy(rows).cuda()])
        assert_close(got, oracle.gemm_rs(A, B, j, rows), f"shard {j}")
    # every element finite and the shards bitwise repeatable
    again = _rs(w.R, dA, dB, w.M, w.N, w.K, fcc.FCC_BF16)
    for j in range(w.R):
        assert torch.isfinite(outs[j].float()).all()
        assert torch.equal(outs[j].view(torch.int16), again[j].view(torch.int16))


def test_ar_full_size_sampled_rows_all_buffers():
    """The all-reduce on the 8-rank 8192x8192x3584 inputs, bf16 outputs, in the
    benchmark's launch shape: sampled rows of every rank's buffer against the
    oracle, every buffer bitwise equal to rank 0's, all of them finite."""
    w = synth.WORKLOADS["gemm_ar_r8_8192x8192x3584"]
    A, B = synth.gemm_inputs(w.R, w.M, w.N, w.K, w.std_a, w.std_b, seed=0)
    dA, dB = _upload(A, B)
    outs = _ar(w.R, dA, dB, w.M, w.N, w.K, fcc.FCC_BF16)
    for r in range(w.R):
        rows = _sample_rows(w.M, 8, seed=200 + r)
        got = to_f64(outs[r][torch.from_numpy(rows).cuda()])
        assert_close(got, oracle.gemm_ar(A, B, rows), f"rank {r}")
        assert torch.isfinite(outs[r].float()).all()
        assert torch.equal(outs[r].view(torch.int16), outs[0].view(torch.int16)), f"rank {r}"


@pytest.mark.parametrize("algo", [fcc.FCC_ALGO_AUTO, fcc.FCC_ALGO_INTERDECOM])
def test_ag_full_size_sampled_rows(algo):
    """The 8-rank 8192x3584x8192 workload in the benchmark's launch shapes: the
    fused kernel and the InterDecom baseline (chunk count from the model)."""
    w = synth.WORKLOADS["ag_gemm_r8_8192x3584x8192"]
    Ms = w.M // w.R
    X, B = synth.gemm_inputs(w.R, Ms, w.N, w.K, w.std_a, w.std_b, seed=0)
    dX, dB = _upload(X, B)
    outs = [empty((w.M, w.N), torch.bfloat16, fill=float("nan")) for _ in range(w.R)]
    fcc.fcc_ag_gemm(w.R, dX, dB, outs, None, w.M, w.N, w.K, fcc.FCC_BF16, fcc.FCC_BF16,
                    fcc.make_opts(algo=algo))
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    for r in range(w.R):
        rows = _sample_rows(w.M, 12, seed=100 + r)
        got = to_f64(outs[r][torch.from_numpy(rows).cuda()])
        assert_close(got, oracle.ag_gemm(X, B, r, rows), f"rank {r}")
        assert torch.isfinite(outs[r].float()).all()


# --------------------------------------------------------- error reporting

def test_bounded_wait_reports_timeout_and_context_survives():
    fcc.fcc_test_wait_timeout(2_000_000)  # 2 ms on a barrier nothing completes
    assert fcc.fcc_stream_status() == fcc.FCC_ERR_TIMEOUT
    assert fcc.fcc_stream_status() == fcc.FCC_OK  # cleared
    R, M, N, K = 2, 256, 256, 128
    A, B = synth.integer_gemm_inputs(R, M, N, K, -2, 2, seed=4)
    dA, dB = _upload(A, B)
    outs = _rs(R, dA, dB, M, N, K, fcc.FCC_F32)
    assert np.array_equal(to_f64(outs[1]), oracle.gemm_rs(A, B, 1))


def test_k_half_wait_reports_timeout_and_context_survives():
    """The second K half of a short last round waits (bounded) for the first
    half's partial: with the flag value it waits for never written, the wait
    runs out, the status word says so and clears, and the same split launch
    afterwards is exact."""
    fcc.fcc_test_ksplit_wait_timeout(2_000_000)  # 2 ms
    assert fcc.fcc_stream_status() == fcc.FCC_ERR_TIMEOUT
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    R, M, N, K = 1, 384, 256, 128  # three 128-row tiles on two CTAs: the last in K halves
    A, B = synth.integer_gemm_inputs(R, M, N, K, -3, 3, seed=8)
    dA, dB = _upload(A, B)
    outs = _rs(R, dA, dB, M, N, K, fcc.FCC_F32, fcc.make_opts(cta_pair=1, max_ctas=2))
    assert np.array_equal(to_f64(outs[0]), oracle.gemm_rs(A, B, 0))


def test_invalid_arguments_rejected_before_launch():
    R, M, N, K = 2, 256, 256, 128
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0)
    dA, dB = _upload(A, B)
    outs = [empty((M // R, N)) for _ in range(R)]
    before = fcc.fcc_launch_count()
    for args in [(0, dA, dB, outs, M, N, K), (2, dA, dB, outs, 255, N, K),
                 (2, dA, dB, outs, M, N, 100), (2, dA, dB, outs, M, 250, K)]:
        with pytest.raises(fcc.FccError) as e:
            fcc.fcc_gemm_rs(*args)
        assert e.value.status == fcc.FCC_ERR_INVALID
    with pytest.raises(fcc.FccError) as e:
        fcc.fcc_gemm_rs(R, [dA[0], dA[1].data_ptr() + 2], dB, outs, M, N, K)
    assert e.value.status == fcc.FCC_ERR_INVALID
    assert fcc.fcc_launch_count() == before
