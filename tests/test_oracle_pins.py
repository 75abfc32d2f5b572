"""Pins for the CPU oracle: checks against values and facts fixed outside it.

Each test pins the oracle to something other than itself: hand-worked values
(tests/golden/hand_examples.txt), exact rational brute force on tiny inputs,
special cases that reduce to a library routine (numpy float64 matmul, argmax,
stable argsort, scipy softmax), closed forms, and invariants of the
definitions (shard concatenation, rank permutation, linearity, gather block
decomposition).  A dropped rank or k term, a transposed operand, a wrong
shard offset or a wrong sort key fails at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split("=", 1)
            vals[k.strip()] = [float(x) for x in v.split()]
    return vals


def _bf16(vals, shape):
    return synth.f32_to_bf16_bits(np.array(vals, dtype=np.float32).reshape(shape))


# ---------------------------------------------------------------- bf16 inputs

def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.Generator(np.random.PCG64(5))
    x = rng.standard_normal(100000, dtype=np.float32) * np.float32(3.0)
    special = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 1e-40, -1e-40, 3.4e38,
                        -3.4e38, 1.00390625, 1.01171875, 1.005859375, 65504.0, 1e-8],
                       dtype=np.float32)
    # exact ties between two bf16 neighbours (round to even both ways)
    ties = (np.arange(1, 2000, dtype=np.uint32) << np.uint32(16)
            | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, special, ties, -ties])
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = synth.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
                          .float().numpy())


def test_generator_is_seeded_and_ordered():
    A1, B1 = synth.gemm_inputs(2, 8, 16, 8, 1.0, 0.5, seed=3)
    A2, B2 = synth.gemm_inputs(2, 8, 16, 8, 1.0, 0.5, seed=3)
    A3, _ = synth.gemm_inputs(2, 8, 16, 8, 1.0, 0.5, seed=4)
    assert all(np.array_equal(a, b) for a, b in zip(A1 + B1, A2 + B2))
    assert not np.array_equal(A1[0], A3[0])
    # A's are drawn before B's: the first A equals a fresh single draw
    rng = np.random.Generator(np.random.PCG64(3))
    assert np.array_equal(A1[0], synth.normal_bf16(rng, (8, 8), 1.0))


# --------------------------------------------------------- hand-worked values

def test_gemm_rs_ar_hand_example():
    g = _golden()
    A = [_bf16(g["gemm.A0"], (2, 2)), _bf16(g["gemm.A1"], (2, 2))]
    B = [_bf16(g["gemm.B0"], (2, 2)), _bf16(g["gemm.B1"], (2, 2))]
    assert np.array_equal(oracle.gemm_ar(A, B), np.array(g["gemm.S"]).reshape(2, 2))
    assert np.array_equal(oracle.gemm_rs(A, B, 0), np.array(g["gemm.shard0"]).reshape(1, 2))
    assert np.array_equal(oracle.gemm_rs(A, B, 1), np.array(g["gemm.shard1"]).reshape(1, 2))


def test_ag_gemm_hand_example():
    g = _golden()
    X = [_bf16(g["ag.X0"], (1, 2)), _bf16(g["ag.X1"], (1, 2))]
    B = [_bf16(g["ag.B0"], (2, 2)), _bf16(g["ag.B1"], (2, 2))]
    assert np.array_equal(oracle.ag_gemm(X, B, 0), np.array(g["ag.out0"]).reshape(2, 2))
    assert np.array_equal(oracle.ag_gemm(X, B, 1), np.array(g["ag.out1"]).reshape(2, 2))


def test_moe_hand_example():
    g = _golden()
    logits = np.array(g["moe.logits"], dtype=np.float32).reshape(2, 2, 4)
    idx, gate = oracle.moe_route(logits, 2)
    assert np.array_equal(idx.reshape(-1), np.array(g["moe.idx"], dtype=np.int32))
    d = oracle.moe_dispatch(idx, R=2, E=4, cap=8)
    assert np.array_equal(d.counts, np.array(g["moe.counts"], dtype=np.int32))
    assert np.array_equal(d.recv_row.reshape(-1), np.array(g["moe.recv_row"], dtype=np.int32))
    assert np.array_equal(d.recv_counts, np.array(g["moe.recv_counts"], dtype=np.int32))
    assert np.array_equal(d.recv_src[0, :5], np.array(g["moe.recv_src0"], dtype=np.int32))
    assert np.array_equal(d.recv_src[1, :3], np.array(g["moe.recv_src1"], dtype=np.int32))
    assert np.all(d.recv_src[0, 5:] == -1) and np.all(d.recv_src[1, 3:] == -1)
    assert np.array_equal(d.send_counts.reshape(-1),
                          np.array(g["moe.send_counts"], dtype=np.int32))
    # gates: closed-form softmax of the all-tied token is 1/E for both slots
    assert np.allclose(gate[1, 1], [0.25, 0.25], rtol=0, atol=1e-15)
    # rank 0 token 0: exp(0)/(exp(-1.5)+1+exp(-3)+exp(-1)) for expert 1
    den = np.exp(-1.5) + 1.0 + np.exp(-3.0) + np.exp(-1.0)
    assert abs(gate[0, 0, 0] - 1.0 / den) < 1e-15
    assert abs(gate[0, 0, 1] - np.exp(-1.0) / den) < 1e-15


# ----------------------------------------------------- brute force, exact math

def _exact_rank_sum(A, B):
    R = len(A)
    M, K = A[0].shape
    N = B[0].shape[1]
    Af = [[[Fraction(float(v)) for v in row] for row in synth.bf16_bits_to_f32(a)] for a in A]
    Bf = [[[Fraction(float(v)) for v in row] for row in synth.bf16_bits_to_f32(b)] for b in B]
    S = [[Fraction(0)] * N for _ in range(M)]
    for r in range(R):
        for i in range(M):
            for n in range(N):
                S[i][n] += sum(Af[r][i][k] * Bf[r][k][n] for k in range(K))
    return S


@pytest.mark.parametrize("R,M,N,K,seed", [(1, 3, 5, 7, 0), (2, 4, 6, 5, 1), (3, 6, 4, 9, 2),
                                          (4, 8, 3, 2, 3)])
def test_rank_sum_brute_force(R, M, N, K, seed):
    A, B = synth.gemm_inputs(R, M, N, K, 1.0, 1.0, seed=seed)
    S = _exact_rank_sum(A, B)
    got = oracle.gemm_ar(A, B)
    for i in range(M):
        for n in range(N):
            exact = S[i][n]
            assert abs(Fraction(got[i, n]) - exact) <= abs(exact) * Fraction(1, 10**14) + \
                Fraction(1, 10**300)
    Ms = M // R
    for j in range(R):
        shard = oracle.gemm_rs(A, B, j)
        for i in range(Ms):
            for n in range(N):
                exact = S[j * Ms + i][n]
                assert abs(Fraction(shard[i, n]) - exact) <= abs(exact) * Fraction(1, 10**14) + \
                    Fraction(1, 10**300)


def test_integer_inputs_exact():
    A, B = synth.integer_gemm_inputs(3, 6, 10, 12, seed=7)
    S = _exact_rank_sum(A, B)
    got = oracle.gemm_ar(A, B)
    assert all(got[i, n] == S[i][n] for i in range(6) for n in range(10))


def test_ag_gemm_brute_force():
    R, Ms, N, K = 3, 2, 5, 4
    X, B = synth.gemm_inputs(R, Ms, N, K, 1.0, 1.0, seed=11)
    Xf = np.concatenate([synth.bf16_bits_to_f32(x) for x in X]).astype(object)
    for r in range(R):
        Bf = synth.bf16_bits_to_f32(B[r])
        got = oracle.ag_gemm(X, B, r)
        for i in range(R * Ms):
            for n in range(N):
                exact = sum(Fraction(float(Xf[i, k])) * Fraction(float(Bf[k, n]))
                            for k in range(K))
                assert abs(Fraction(got[i, n]) - exact) <= abs(exact) * Fraction(1, 10**14) + \
                    Fraction(1, 10**300)


# ------------------------------------------- special cases: library routines

def _f64(a):
    return synth.bf16_bits_to_f32(a).astype(np.float64)


def test_single_rank_is_plain_gemm():
    A, B = synth.gemm_inputs(1, 37, 53, 29, 1.0, 1.0, seed=2)
    ref = _f64(A[0]) @ _f64(B[0])
    assert np.allclose(oracle.gemm_rs(A, B, 0), ref, rtol=1e-12, atol=1e-12)
    X, Bx = synth.gemm_inputs(1, 19, 23, 31, 1.0, 1.0, seed=3)
    assert np.allclose(oracle.ag_gemm(X, Bx, 0), _f64(X[0]) @ _f64(Bx[0]), rtol=1e-12,
                       atol=1e-12)


def test_rank_sum_equals_stacked_gemm():
    """sum_r A_r B_r == [A_0 ... A_{R-1}] @ [B_0; ...; B_{R-1}] (one library GEMM)."""
    A, B = synth.gemm_inputs(4, 24, 40, 16, 1.0, 1.0, seed=9)
    ref = np.concatenate([_f64(a) for a in A], axis=1) @ np.concatenate([_f64(b) for b in B])
    assert np.allclose(oracle.gemm_ar(A, B), ref, rtol=1e-12, atol=1e-12)
    # a non-square case catches a transposed operand
    A, B = synth.gemm_inputs(2, 6, 14, 10, 1.0, 1.0, seed=10)
    ref = _f64(A[0]) @ _f64(B[0]) + _f64(A[1]) @ _f64(B[1])
    assert np.allclose(oracle.gemm_ar(A, B), ref, rtol=1e-12, atol=1e-12)


def test_ag_block_decomposition():
    R, Ms, N, K = 4, 6, 10, 12
    X, B = synth.gemm_inputs(R, Ms, N, K, 1.0, 1.0, seed=4)
    for r in range(R):
        out = oracle.ag_gemm(X, B, r)
        for i in range(R):
            assert np.allclose(out[i * Ms:(i + 1) * Ms], _f64(X[i]) @ _f64(B[r]),
                               rtol=1e-12, atol=1e-12)


# ------------------------------------------------------ closed forms, invariants

def test_ones_closed_form():
    R, M, N, K = 3, 6, 5, 7
    one = synth.f32_to_bf16_bits(np.ones((M, K), np.float32))
    oneb = synth.f32_to_bf16_bits(np.ones((K, N), np.float32))
    assert np.all(oracle.gemm_ar([one] * R, [oneb] * R) == R * K)
    for j in range(R):
        assert np.all(oracle.gemm_rs([one] * R, [oneb] * R, j) == R * K)


def test_one_hot_selects_rows():
    """A_r = e_{row -> p_r(row)} one-hot picks rows of B_r: exact selection."""
    R, M, N, K = 2, 4, 6, 4
    rng = np.random.Generator(np.random.PCG64(1))
    A, B = [], []
    expect = np.zeros((M, N))
    for r in range(R):
        p = rng.permutation(K)[:M]
        a = np.zeros((M, K), np.float32)
        a[np.arange(M), p] = 1.0
        b = rng.integers(-8, 9, size=(K, N)).astype(np.float32)
        A.append(synth.f32_to_bf16_bits(a))
        B.append(synth.f32_to_bf16_bits(b))
        expect += b[p]
    assert np.array_equal(oracle.gemm_ar(A, B), expect)


def test_shard_concat_is_allreduce():
    A, B = synth.gemm_inputs(4, 32, 24, 16, 1.0, 1.0, seed=6)
    full = oracle.gemm_ar(A, B)
    shards = np.concatenate([oracle.gemm_rs(A, B, j) for j in range(4)])
    assert np.array_equal(full, shards)


def test_rank_permutation_invariance():
    A, B = synth.gemm_inputs(5, 10, 12, 8, 1.0, 1.0, seed=8)
    perm = [3, 0, 4, 1, 2]
    a = oracle.gemm_ar(A, B)
    b = oracle.gemm_ar([A[p] for p in perm], [B[p] for p in perm])
    assert np.allclose(a, b, rtol=1e-12, atol=1e-13)
    assert not np.allclose(a, oracle.gemm_ar(A[:4], B[:4]), rtol=1e-6)


def test_linearity_in_one_rank():
    A, B = synth.gemm_inputs(3, 8, 9, 10, 1.0, 1.0, seed=12)
    doubled = synth.f32_to_bf16_bits(2.0 * synth.bf16_bits_to_f32(A[0]))  # exact in bf16
    base = oracle.gemm_ar(A, B)
    twice = oracle.gemm_ar([doubled] + A[1:], B)
    term0 = _f64(A[0]) @ _f64(B[0])
    assert np.allclose(twice - base, term0, rtol=1e-12, atol=1e-12)


def test_selected_rows_match_full():
    A, B = synth.gemm_inputs(2, 40, 16, 8, 1.0, 1.0, seed=13)
    full = oracle.gemm_ar(A, B)
    rows = np.array([39, 0, 17, 17, 5])
    assert np.array_equal(oracle.gemm_ar(A, B, rows), full[rows])
    assert np.array_equal(oracle.gemm_rs(A, B, 1, [3, 0]), full[[23, 20]])


def test_bad_arguments_raise():
    A, B = synth.gemm_inputs(3, 4, 4, 4, 1.0, 1.0)
    with pytest.raises(ValueError):
        oracle.gemm_rs(A, B, 0)          # M % R != 0
    with pytest.raises(ValueError):
        oracle.gemm_ar(A, B, [4])        # row out of range


# ------------------------------------------------------------------- MoE pins

def test_route_vs_sorting_brute_force():
    rng = np.random.Generator(np.random.PCG64(21))
    logits = rng.standard_normal((3, 50, 16), dtype=np.float32)
    # plant exact ties
    logits[0, 0, :] = 1.0
    logits[1, 3, [2, 9]] = 5.0
    idx, gate = oracle.moe_route(logits, 3)
    for s in range(3):
        for t in range(50):
            order = sorted(range(16), key=lambda e: (-float(logits[s, t, e]), e))
            assert list(idx[s, t]) == order[:3]


def test_route_top1_is_argmax_and_gates_are_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.Generator(np.random.PCG64(22))
    logits = rng.standard_normal((200, 64), dtype=np.float32)
    logits[7, [3, 40]] = 9.0  # tie: argmax keeps the first
    idx1, _ = oracle.moe_route(logits, 1)
    assert np.array_equal(idx1[:, 0], np.argmax(logits, axis=1))
    idx2, gate2 = oracle.moe_route(logits, 2)
    p = scipy_special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(gate2, np.take_along_axis(p, idx2.astype(np.int64), 1), rtol=1e-13,
                       atol=0)
    assert np.all(gate2.sum(1) <= 1.0 + 1e-15)
    assert np.all(gate2[:, 0] >= gate2[:, 1])


def _dispatch_case(R=4, T=300, E=16, topk=2, seed=23):
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = rng.standard_normal((R, T, E), dtype=np.float32)
    idx, _ = oracle.moe_route(logits, topk)
    return idx, R, T, E, topk


def test_dispatch_vs_stable_argsort():
    idx, R, T, E, topk = _dispatch_case()
    cap = R * T * topk
    d = oracle.moe_dispatch(idx, R, E, cap)
    flat = idx.reshape(-1)
    assert np.array_equal(d.counts, np.bincount(flat, minlength=E))
    assert d.counts.sum() == R * T * topk
    Eloc = E // R
    order = np.argsort(flat, kind="stable")           # library stable sort by expert
    start = np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))])
    for dst in range(R):
        rows = order[start[dst * Eloc]:start[(dst + 1) * Eloc]]
        n = rows.size
        assert d.recv_counts[dst] == n
        assert np.array_equal(d.recv_src[dst, :n], rows // topk)
        assert np.array_equal(d.recv_expert[dst, :n], flat[rows])
        assert np.all(d.recv_src[dst, n:] == -1)
    # each (token) appears exactly topk times with distinct experts
    seen = {}
    for dst in range(R):
        for row in range(d.recv_counts[dst]):
            seen.setdefault(int(d.recv_src[dst, row]), []).append(int(d.recv_expert[dst, row]))
    assert len(seen) == R * T
    assert all(len(v) == topk and len(set(v)) == topk for v in seen.values())
    # send counts: row sums are what each rank sends, column sums what each receives
    assert np.all(d.send_counts.sum(1) == T * topk)
    assert np.array_equal(d.send_counts.sum(0), d.recv_counts)
    # recv_row agrees with recv_src
    for s in range(R):
        for t in range(0, T, 37):
            for k in range(topk):
                e = idx[s, t, k]
                assert d.recv_src[e // Eloc, d.recv_row[s, t, k]] == s * T + t


def test_dispatch_one_expert_per_rank_is_plain_all_to_all():
    """E == R, top-1: rank d receives, in (source, token) order, the tokens sent to it."""
    R, T = 4, 64
    rng = np.random.Generator(np.random.PCG64(24))
    dest = rng.integers(0, R, size=(R, T, 1)).astype(np.int32)
    d = oracle.moe_dispatch(dest, R, R, R * T)
    for dst in range(R):
        expect = [s * T + t for s in range(R) for t in range(T) if dest[s, t, 0] == dst]
        assert list(d.recv_src[dst, :len(expect)]) == expect
        for s in range(R):
            assert d.send_counts[s, dst] == int(np.sum(dest[s, :, 0] == dst))


def test_dispatch_capacity_overflow():
    idx, R, T, E, topk = _dispatch_case(T=40)
    with pytest.raises(OverflowError):
        oracle.moe_dispatch(idx, R, E, cap=10)


def test_expert_rows_vs_library_matmul():
    X, logits, W = synth.moe_inputs(R=2, T=12, H=24, E=4, F=20, seed=25)
    src_rank = np.array([0, 1, 1, 0])
    src_tok = np.array([3, 0, 11, 3])
    expert = np.array([2, 0, 3, 1])
    got = oracle.moe_expert_rows(X, W, src_rank, src_tok, expert)
    for i in range(4):
        ref = _f64(X[src_rank[i]])[src_tok[i]] @ _f64(W[expert[i]])
        assert np.allclose(got[i], ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- MoE combine

def _combine_case(R=2, T=6, H=16, E=4, F=12, seed=31):
    X, logits, W = synth.moe_inputs(R=R, T=T, H=H, E=E, F=F, seed=seed)
    sr = np.repeat(np.arange(R), T)
    st = np.tile(np.arange(T), R)
    return X, logits, W, sr, st


def test_combine_brute_force_exact():
    """Exact rational sum of gate * (x . w) per token and slot (Fraction)."""
    X, logits, W, sr, st = _combine_case(T=3, H=5, F=4)
    idx = np.array([[2, 0], [1, 3], [3, 2], [0, 1], [2, 1], [3, 0]], dtype=np.int32)
    gate = np.array([[0.5, 0.25], [0.375, 0.125], [0.75, 0.0625],
                     [0.1, 0.3], [0.6, 0.2], [0.05, 0.45]])
    got = oracle.moe_combine(X, W, sr, st, idx, gate)
    xs = [_f64(x) for x in X]
    ws = [_f64(w) for w in W]
    for i in range(len(sr)):
        for f in range(4):
            tot = Fraction(0)
            for j in range(2):
                dot = sum(Fraction(xs[sr[i]][st[i], h]) * Fraction(ws[idx[i, j]][h, f])
                          for h in range(5))
                tot += Fraction(gate[i, j]) * dot
            assert abs(got[i, f] - float(tot)) <= 1e-15 * max(1.0, abs(float(tot)))


def test_combine_top1_is_gate_times_library_matmul():
    X, logits, W, sr, st = _combine_case()
    idx, gate = oracle.moe_route(np.stack(logits), 1)
    got = oracle.moe_combine(X, W, sr, st, idx.reshape(-1, 1), gate.reshape(-1, 1))
    for i in range(len(sr)):
        e = idx.reshape(-1)[i]
        ref = gate.reshape(-1)[i] * (_f64(X[sr[i]])[st[i]] @ _f64(W[e]))
        assert np.allclose(got[i], ref, rtol=1e-12, atol=1e-14)


def test_combine_identical_experts_sum_the_gates():
    """All W_e equal: y = (sum of the token's gates) * x . W (no slot dropped or doubled)."""
    X, logits, W, sr, st = _combine_case()
    W = [W[0]] * len(W)
    idx, gate = oracle.moe_route(np.stack(logits), 2)
    got = oracle.moe_combine(X, W, sr, st, idx.reshape(-1, 2), gate.reshape(-1, 2))
    gsum = gate.reshape(-1, 2).sum(axis=1)
    for i in range(len(sr)):
        ref = gsum[i] * (_f64(X[sr[i]])[st[i]] @ _f64(W[0]))
        assert np.allclose(got[i], ref, rtol=1e-12, atol=1e-14)


def test_combine_linear_in_gates_and_slot_order_free():
    X, logits, W, sr, st = _combine_case()
    idx, gate = oracle.moe_route(np.stack(logits), 2)
    idx, gate = idx.reshape(-1, 2), gate.reshape(-1, 2)
    y1 = oracle.moe_combine(X, W, sr, st, idx, gate)
    y2 = oracle.moe_combine(X, W, sr, st, idx, 3.0 * gate)
    assert np.allclose(y2, 3.0 * y1, rtol=1e-13, atol=1e-15)
    ysw = oracle.moe_combine(X, W, sr, st, idx[:, ::-1], gate[:, ::-1])
    assert np.allclose(ysw, y1, rtol=1e-13, atol=1e-15)


def test_combine_dropped_slot_adds_nothing():
    X, logits, W, sr, st = _combine_case()
    idx, gate = oracle.moe_route(np.stack(logits), 2)
    idx, gate = idx.reshape(-1, 2).copy(), gate.reshape(-1, 2)
    only0 = oracle.moe_combine(X, W, sr, st, idx[:, :1], gate[:, :1])
    idx[:, 1] = -1
    got = oracle.moe_combine(X, W, sr, st, idx, gate)
    assert np.array_equal(got, only0)


# ------------------------------------------------------- embedding + all-to-all

def test_embedding_bag_of_one_is_the_row():
    """Bags of exactly one row: the pooled vector is that table row (numpy indexing)."""
    R, ntab, V, D, Bl = 2, 4, 50, 8, 6
    tables, offsets, indices = synth.embedding_inputs(R, ntab, V, D, Bl, L=1, seed=41)
    out = oracle.embedding_a2a(tables, offsets, indices, R)
    for r in range(R):
        for b in range(Bl):
            for t in range(ntab):
                g = r * Bl + b
                row = _f64(tables[t])[indices[t][offsets[t][g]]]
                assert np.array_equal(out[r][b, t], row)


def test_embedding_single_rank_is_reduceat():
    """R = 1: each table's bags are numpy add.reduceat over the gathered rows."""
    tables, offsets, indices = synth.embedding_inputs(1, 3, 40, 16, 10, L=4, seed=42)
    out = oracle.embedding_a2a(tables, offsets, indices, 1)[0]
    for t in range(3):
        rows = _f64(tables[t])[indices[t]]
        ref = np.add.reduceat(rows, offsets[t][:-1], axis=0)
        assert np.allclose(out[:, t], ref, rtol=1e-14, atol=1e-14)


def test_embedding_closed_form_places_bags():
    """Row v of table t holds t + v + d (exact in bf16): bag (t, g) pools to
    n*(t + d) + sum of its indices, and lands at rank g // Bl, sample g % Bl."""
    R, ntab, V, D, Bl = 4, 3, 16, 6, 5
    _, offsets, indices = synth.embedding_inputs(R, ntab, V, D, Bl, L=3, seed=43)
    tables = [_bf16([t + v + d for v in range(V) for d in range(D)], (V, D))
              for t in range(ntab)]
    out = oracle.embedding_a2a(tables, offsets, indices, R)
    for g in range(R * Bl):
        for t in range(ntab):
            ix = indices[t][offsets[t][g]:offsets[t][g + 1]]
            want = len(ix) * (t + np.arange(D)) + ix.sum()
            assert np.array_equal(out[g // Bl][g % Bl, t], want.astype(np.float64))


def test_embedding_brute_force_and_empty_bags():
    R, ntab, V, D, Bl = 2, 2, 9, 4, 4
    tables, offsets, indices = synth.embedding_inputs(R, ntab, V, D, Bl, L=2, min_bag=0,
                                                      seed=44)
    assert any(offsets[t][g] == offsets[t][g + 1] for t in range(ntab) for g in range(R * Bl))
    out = oracle.embedding_a2a(tables, offsets, indices, R)
    for r in range(R):
        for b in range(Bl):
            for t in range(ntab):
                g = r * Bl + b
                acc = [0.0] * D
                for k in range(offsets[t][g], offsets[t][g + 1]):
                    for d in range(D):
                        acc[d] += float(_f64(tables[t])[indices[t][k], d])
                assert np.allclose(out[r][b, t], acc, rtol=1e-15, atol=0)


# -------------------------------------------------------------- ring attention

def _att(Q):
    return [_f64(q.reshape(-1)).reshape(q.shape) for q in Q]


def test_attention_one_rank_vs_library_softmax():
    from scipy.special import softmax
    Q, K, V = synth.attention_inputs(1, 12, 2, 16, seed=51)
    got = oracle.ring_attention(Q, K, V)[0]
    q, k, v = _att(Q)[0], _att(K)[0], _att(V)[0]
    for h in range(2):
        p = softmax(q[:, h] @ k[:, h].T / np.sqrt(16.0), axis=1)
        assert np.allclose(got[:, h], p @ v[:, h], rtol=1e-12, atol=1e-13)


def test_attention_shard_permutation_invariant():
    """Non-causal: every query sees all (key, value) pairs; swapping two
    ranks' K and V shards together changes nothing."""
    Q, K, V = synth.attention_inputs(3, 7, 2, 8, seed=52)
    a = oracle.ring_attention(Q, K, V)
    perm = [2, 0, 1]
    b = oracle.ring_attention(Q, [K[i] for i in perm], [V[i] for i in perm])
    for r in range(3):
        assert np.allclose(a[r], b[r], rtol=1e-12, atol=1e-14)


def test_attention_zero_queries_average_the_values():
    R, S, H, d = 2, 5, 3, 8
    Q, K, V = synth.attention_inputs(R, S, H, d, seed=53)
    Q = [np.zeros_like(q) for q in Q]
    vall = np.concatenate(_att(V))                           # [R*S, H, d]
    full = oracle.ring_attention(Q, K, V, causal=False)
    caus = oracle.ring_attention(Q, K, V, causal=True)
    for r in range(R):
        assert np.allclose(full[r], vall.mean(axis=0)[None], rtol=1e-13, atol=1e-14)
        for t in range(S):
            p = r * S + t
            assert np.allclose(caus[r][t], vall[:p + 1].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_attention_dominant_key_selects_its_value():
    R, S, H, d = 2, 4, 1, 8
    Q, K, V = synth.attention_inputs(R, S, H, d, seed=54)
    q = np.full((S, H, d), 2.0, dtype=np.float32)
    Q = [synth.f32_to_bf16_bits(q)] * R
    k = synth.bf16_bits_to_f32(K[1]).copy()
    k[2, 0, :] = 8.0                                         # score 2*8*8/sqrt(8) = 45 above the rest
    K = [K[0], synth.f32_to_bf16_bits(k)]
    got = oracle.ring_attention(Q, K, V)
    want = _f64(V[1][2, 0])
    for r in range(R):
        assert np.allclose(got[r][:, 0], want[None], rtol=0, atol=1e-12)


def test_attention_causal_brute_force():
    import math
    R, S, H, d = 2, 3, 1, 4
    Q, K, V = synth.attention_inputs(R, S, H, d, seed=55)
    q, k, v = (np.concatenate(_att(x)) for x in (Q, K, V))   # global positions
    got = np.concatenate(oracle.ring_attention(Q, K, V, causal=True))
    for p in range(R * S):
        sc = [sum(q[p, 0, c] * k[j, 0, c] for c in range(d)) / math.sqrt(d) for j in range(p + 1)]
        m = max(sc)
        w = [math.exp(x - m) for x in sc]
        o = [sum(w[j] * v[j, 0, c] for j in range(p + 1)) / sum(w) for c in range(d)]
        assert np.allclose(got[p, 0], o, rtol=1e-13, atol=1e-15)


def test_oracle_threads_reported():
    assert oracle.num_threads() >= 1
