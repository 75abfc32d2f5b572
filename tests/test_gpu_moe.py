"""GPU parity: MoE route + dispatch (all-to-all) + grouped expert GEMM.

Indices, counts and receive positions must equal the oracle bit for bit; the
staged rows must be the source rows bit for bit; gates match the fp64 softmax
to f32 rounding; expert outputs match the oracle within the float tolerance.
The full workload (8 ranks x 4096 tokens, hidden 4096, 64 experts, top-2,
F = 1408) is checked on all index outputs and on sampled output rows.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_close, dev_bf16, dev_f32, empty, to_f64

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_collective_gb300 as fcc  # noqa: E402

# f32 softmax: E exp() values (a few ulp each) summed in f32 and one division;
# |rel err| <= (E + 3) * 2^-24 ~ 4e-6 for E = 64.
GATE_RTOL = 5e-6


def _run(X, logits, W, R, T, H, F, E, topk, cap, out_dtype=fcc.FCC_BF16, opts=None,
         staged=True, contiguous=False):
    """staged: rows into caller buffers, else recv_x NULL.  contiguous: the
    sources are views of one [R*T, H] tensor, so the expert GEMM gathers its
    rows from them (unless opts asks for FCC_ALGO_UNFUSED); otherwise they are
    separate tensors and the rows are staged (recv_x, or library workspace)."""
    if contiguous:
        whole = dev_bf16(np.concatenate(X))
        dX = [whole[s * T:(s + 1) * T] for s in range(R)]
    else:
        dX = [dev_bf16(x) for x in X]
    dL = [dev_f32(l) for l in logits]
    dW = [dev_bf16(w) for w in W]
    tdt = torch.float32 if out_dtype == fcc.FCC_F32 else torch.bfloat16
    recv_x = [empty((cap, H), torch.bfloat16, fill=0.0) for _ in range(R)] if staged else None
    recv_y = [empty((cap, F), tdt, fill=float("nan")) for _ in range(R)]
    idx = [torch.full((T, topk), -7, dtype=torch.int32, device="cuda") for _ in range(R)]
    gate = [empty((T, topk), torch.float32) for _ in range(R)]
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    send = torch.full((R * R,), -7, dtype=torch.int32, device="cuda")
    src = [torch.full((cap,), -1, dtype=torch.int32, device="cuda") for _ in range(R)]
    fcc.fcc_moe_dispatch_gemm(R, dX, dL, dW, T, H, F, E, topk, recv_x, recv_y, cap, idx, gate,
                              counts, send, src, fcc.FCC_BF16, out_dtype, opts)
    st = fcc.fcc_stream_status()
    return dict(recv_x=recv_x, recv_y=recv_y, idx=idx, gate=gate, counts=counts, send=send,
                src=src, status=st)


def _check(X, logits, W, R, T, H, F, E, topk, cap, out, sample=None, seed=0):
    assert out["status"] == fcc.FCC_OK
    lg = np.stack(logits)
    ref_idx, ref_gate = oracle.moe_route(lg, topk)
    got_idx = np.stack([i.cpu().numpy() for i in out["idx"]])
    assert np.array_equal(got_idx, ref_idx), "top-k indices differ"
    got_gate = np.stack([g.cpu().numpy() for g in out["gate"]]).astype(np.float64)
    assert np.allclose(got_gate, ref_gate, rtol=GATE_RTOL, atol=0), \
        f"gates: max rel {np.max(np.abs(got_gate / ref_gate - 1)):.2e}"
    d = oracle.moe_dispatch(ref_idx, R, E, cap)
    assert np.array_equal(out["counts"].cpu().numpy(), d.counts)
    assert np.array_equal(out["send"].cpu().numpy().reshape(R, R), d.send_counts)
    rng = np.random.Generator(np.random.PCG64(seed))
    for dst in range(R):
        n = int(d.recv_counts[dst])
        src = out["src"][dst].cpu().numpy()
        assert np.array_equal(src[:n], d.recv_src[dst, :n]), f"recv_src of rank {dst}"
        assert np.all(src[n:] == -1), "rows past the count were written"
        rows = np.arange(n) if sample is None else np.sort(
            rng.choice(n, size=min(n, sample), replace=False))
        s_rank = d.recv_src[dst, rows] // T
        s_tok = d.recv_src[dst, rows] % T
        if out["recv_x"] is not None:
            # staged rows are the source rows, bit for bit
            rx = out["recv_x"][dst][torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy()
            want = np.stack([X[s][t] for s, t in zip(s_rank, s_tok)]).view(np.int16)
            assert np.array_equal(rx, want), f"recv_x of rank {dst}"
        ref = oracle.moe_expert_rows(X, W, s_rank, s_tok, d.recv_expert[dst, rows])
        got = to_f64(out["recv_y"][dst][torch.from_numpy(rows).cuda()])
        assert_close(got, ref, f"recv_y of rank {dst}")


# (recv_x given, sources one array, algo) of each launch path:
#   staged         the GEMM's copy warps stage the rows into recv_x, its
#                  tensor cores consume them unit by unit (sources separate)
#   workspace      the same into library workspace (the default)
#   gather         GEMM gathers from the sources with TMA gather4, no copy
#   gather_recv_x  GEMM gathers; recv_x written beside it on a side stream
#   fused_separate FCC_ALGO_FUSED with separate sources: staged as by default
#   unfused        a separate copy kernel into recv_x, then the GEMM
#   unfused_workspace  the same into library workspace
#   interdecom     expert-range chunks: each range's rows copied on a side
#                  stream ahead of that range's GEMM (chunk model), into recv_x
#   interdecom_workspace  the same into library workspace
#   ce             each source packs its rows, the copy engines move the
#                  (source, expert) runs into recv_x, then the GEMM
#   ce_workspace   the same into library workspace
PATHS = {"staged": (True, False, fcc.FCC_ALGO_AUTO),
         "workspace": (False, True, fcc.FCC_ALGO_AUTO),
         "gather": (False, True, fcc.FCC_ALGO_FUSED),
         "gather_recv_x": (True, True, fcc.FCC_ALGO_FUSED),
         "fused_separate": (False, False, fcc.FCC_ALGO_FUSED),
         "unfused": (True, False, fcc.FCC_ALGO_UNFUSED),
         "unfused_workspace": (False, True, fcc.FCC_ALGO_UNFUSED),
         "interdecom": (True, False, fcc.FCC_ALGO_INTERDECOM),
         "interdecom_workspace": (False, True, fcc.FCC_ALGO_INTERDECOM),
         "ce": (True, False, fcc.FCC_ALGO_CE),
         "ce_workspace": (False, True, fcc.FCC_ALGO_CE)}


@pytest.mark.parametrize("R,T,H,F,E,topk", [
    (2, 300, 128, 136, 8, 2),     # ragged chunk, ragged F tile
    (4, 257, 256, 264, 16, 2),
    (8, 64, 64, 64, 64, 2),       # more experts than tokens per expert
    (2, 200, 192, 128, 4, 1),     # top-1
    (4, 130, 128, 72, 4, 2),      # one expert per rank: plain all-to-all
    (1, 500, 128, 256, 8, 2),     # one rank
])
@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("path", list(PATHS))
def test_moe_small(R, T, H, F, E, topk, pair, path):
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=R * 100 + T)
    cap = R * T * topk
    staged, contiguous, algo = PATHS[path]
    out = _run(X, logits, W, R, T, H, F, E, topk, cap,
               opts=fcc.make_opts(cta_pair=pair, algo=algo), staged=staged,
               contiguous=contiguous)
    _check(X, logits, W, R, T, H, F, E, topk, cap, out)


@pytest.mark.parametrize("T", [8192, 8193])
def test_moe_placement_either_side_of_the_one_kernel_limit(T):
    """Up to 512 chunks of 128 tokens the offsets and the ranks are one kernel
    (every CTA sums the whole chunk histogram itself); past that, a scan
    kernel and a rank kernel.  8 x 8192 tokens are 512 chunks, 8 x 8193 are
    520: both give the oracle's integers and rows."""
    R, H, F, E, topk = 8, 64, 64, 64, 2
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=23)
    cap = 2 * T * topk
    for algo in (fcc.FCC_ALGO_AUTO, fcc.FCC_ALGO_CE):
        out = _run(X, logits, W, R, T, H, F, E, topk, cap, opts=fcc.make_opts(algo=algo))
        _check(X, logits, W, R, T, H, F, E, topk, cap, out, sample=384)


# Rows per expert chosen so that an expert's last unit of at most 128 rows
# (an M = 128 pair tile: 64 rows from each CTA of the pair) holds rows on one
# CTA only, on both, or fills it, next to full units, units of 129-255 rows
# and an expert with no rows.
SHORT_UNIT_COUNTS = [1, 2, 17, 31, 32, 33, 34, 63, 64, 65, 66, 127, 128, 129, 257, 289, 321,
                     384, 0, 200]


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("path", ["workspace", "gather", "unfused_workspace"])
def test_moe_short_last_units(pair, path):
    R, H, F, E, topk = 2, 192, 320, len(SHORT_UNIT_COUNTS), 1
    total = sum(SHORT_UNIT_COUNTS)
    T = (total + R - 1) // R
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=41)
    # token i (in (rank, token) order) goes to the expert of its position in
    # the count list; the padding token, if any, to the last expert
    owner = np.repeat(np.arange(E), SHORT_UNIT_COUNTS)
    owner = np.concatenate([owner, np.full(R * T - total, E - 1)])
    rng = np.random.Generator(np.random.PCG64(43))
    rng.shuffle(owner)  # interleave the experts over the chunks
    for s in range(R):
        logits[s][np.arange(T), owner[s * T:(s + 1) * T]] += 50.0
    cap = R * T * topk
    staged, contiguous, algo = PATHS[path]
    out = _run(X, logits, W, R, T, H, F, E, topk, cap,
               opts=fcc.make_opts(cta_pair=pair, algo=algo), staged=staged,
               contiguous=contiguous)
    counts = out["counts"].cpu().numpy()
    want = np.bincount(owner, minlength=E)
    assert np.array_equal(counts, want)
    _check(X, logits, W, R, T, H, F, E, topk, cap, out)


def test_moe_ties_and_f32_output():
    R, T, H, F, E, topk = 2, 128, 64, 64, 8, 2
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=5)
    logits[0][0, :] = 1.0                  # all tied: experts 0, 1
    logits[0][1, [2, 6]] = 9.0             # tie for first: 2 then 6
    logits[1][5, [7, 3, 5]] = [4.0, 4.0, 4.0]
    cap = R * T * topk
    out = _run(X, logits, W, R, T, H, F, E, topk, cap, fcc.FCC_F32, staged=False,
               contiguous=True, opts=fcc.make_opts(algo=fcc.FCC_ALGO_FUSED))
    _check(X, logits, W, R, T, H, F, E, topk, cap, out)
    idx0 = out["idx"][0].cpu().numpy()
    assert list(idx0[0]) == [0, 1] and list(idx0[1]) == [2, 6]


def test_moe_repeatable():
    R, T, H, F, E, topk = 4, 256, 128, 128, 16, 2
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=6)
    cap = R * T * topk
    for path in ("workspace", "gather"):
        staged, contiguous, algo = PATHS[path]
        o = fcc.make_opts(algo=algo)
        a = _run(X, logits, W, R, T, H, F, E, topk, cap, staged=staged, contiguous=contiguous,
                 opts=o)
        b = _run(X, logits, W, R, T, H, F, E, topk, cap, staged=staged, contiguous=contiguous,
                 opts=o)
        for d in range(R):
            assert torch.equal(a["src"][d], b["src"][d])
            assert torch.equal(a["recv_y"][d].view(torch.int16),
                               b["recv_y"][d].view(torch.int16))


@pytest.mark.parametrize("pair", [1, 2])
def test_moe_in_kernel_staging_equals_copy_kernel(pair):
    """The rows the GEMM's copy warps stage, and the products of those rows,
    are bit for bit those of the separate copy kernel (same rows, same MMAs);
    a second call, whose unit counters restart from zero, repeats them."""
    R, T, H, F, E, topk = 4, 700, 320, 264, 8, 2   # 350 rows an expert: a ragged unit
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=9)
    cap = R * T * topk
    o_in = fcc.make_opts(cta_pair=pair, algo=fcc.FCC_ALGO_AUTO)
    o_sep = fcc.make_opts(cta_pair=pair, algo=fcc.FCC_ALGO_UNFUSED)
    a = _run(X, logits, W, R, T, H, F, E, topk, cap, opts=o_in)
    b = _run(X, logits, W, R, T, H, F, E, topk, cap, opts=o_sep)
    c = _run(X, logits, W, R, T, H, F, E, topk, cap, opts=o_in)
    _check(X, logits, W, R, T, H, F, E, topk, cap, a)
    for d in range(R):
        n = int((a["src"][d] >= 0).sum())
        for other in (b, c):
            assert torch.equal(a["src"][d], other["src"][d])
            assert torch.equal(a["recv_x"][d][:n].view(torch.int16),
                               other["recv_x"][d][:n].view(torch.int16))
            assert torch.equal(a["recv_y"][d][:n].view(torch.int16),
                               other["recv_y"][d][:n].view(torch.int16))


@pytest.mark.parametrize("algo", [fcc.FCC_ALGO_AUTO, fcc.FCC_ALGO_UNFUSED,
                                  fcc.FCC_ALGO_INTERDECOM, fcc.FCC_ALGO_CE])
def test_moe_capacity_overflow_reported(algo):
    R, T, H, F, E, topk = 2, 256, 64, 64, 4, 2
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=7)
    cap = 100
    out = _run(X, logits, W, R, T, H, F, E, topk, cap, opts=fcc.make_opts(algo=algo))
    assert out["status"] == fcc.FCC_ERR_CAPACITY
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    # the kept rows are the first cap rows of the full dispatch: their sources,
    # their staged copies and their products
    d = oracle.moe_dispatch(oracle.moe_route(np.stack(logits), topk)[0], R, E, R * T * topk)
    for dst in range(R):
        n = min(cap, int(d.recv_counts[dst]))
        assert np.array_equal(out["src"][dst].cpu().numpy()[:n], d.recv_src[dst, :n])
        s_rank, s_tok = d.recv_src[dst, :n] // T, d.recv_src[dst, :n] % T
        rx = out["recv_x"][dst][:n].view(torch.int16).cpu().numpy()
        want = np.stack([X[s][t] for s, t in zip(s_rank, s_tok)]).view(np.int16)
        assert np.array_equal(rx, want), f"recv_x of rank {dst}"
        ref = oracle.moe_expert_rows(X, W, s_rank, s_tok, d.recv_expert[dst, :n])
        assert_close(to_f64(out["recv_y"][dst][:n]), ref, f"recv_y of rank {dst}")


@pytest.mark.parametrize("chunks", [1, 3, 5, 64])
def test_moe_interdecom_chunk_counts(chunks):
    """Expert ranges of any size (E = 16 over 1, 3, 5 or, clamped, 16 chunks,
    uneven ranges included) give the same rows and products, bit for bit, as
    the separate copy kernel: the same rows and the same MMAs per tile."""
    R, T, H, F, E, topk = 4, 257, 192, 264, 16, 2
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=19)
    cap = R * T * topk
    a = _run(X, logits, W, R, T, H, F, E, topk, cap,
             opts=fcc.make_opts(algo=fcc.FCC_ALGO_INTERDECOM, chunks=chunks))
    _check(X, logits, W, R, T, H, F, E, topk, cap, a)
    b = _run(X, logits, W, R, T, H, F, E, topk, cap,
             opts=fcc.make_opts(algo=fcc.FCC_ALGO_UNFUSED))
    for d in range(R):
        n = int((a["src"][d] >= 0).sum())
        assert torch.equal(a["recv_x"][d][:n].view(torch.int16),
                           b["recv_x"][d][:n].view(torch.int16))
        assert torch.equal(a["recv_y"][d][:n].view(torch.int16),
                           b["recv_y"][d][:n].view(torch.int16))


def test_moe_invalid_arguments():
    R, T, H, F, E, topk = 2, 16, 64, 64, 4, 2
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=8)
    with pytest.raises(fcc.FccError) as e:
        _run(X, logits, W, R, T, H, F, 3, topk, 64)        # E % R != 0
    assert e.value.status == fcc.FCC_ERR_INVALID
    with pytest.raises(fcc.FccError) as e:
        _run(X, logits, W, R, T, H, F, E, 3, 64)           # topk = 3
    assert e.value.status == fcc.FCC_ERR_INVALID


@pytest.mark.parametrize("path", ["workspace", "staged", "unfused_workspace", "gather",
                                  "gather_recv_x", "interdecom_workspace", "ce_workspace"])
def test_moe_full_workload_sampled(path):
    """The benchmark's launches: rows staged in library workspace (or recv_x)
    by the GEMM's copy warps or by a separate copy kernel, gathered by the
    GEMM, gathered with recv_x written beside the GEMM, moved range by range
    ahead of each range's GEMM (InterDecom), or by the copy engines."""
    w = synth.WORKLOADS["moe_r8_t4096_h4096_e64_f1408"]
    X, logits, W = synth.moe_inputs(w.R, w.T, w.H, w.E, w.F, std_x=w.std_a, std_w=w.std_b,
                                    seed=0)
    cap = 2 * w.T * w.topk  # twice the mean load per rank
    staged, contiguous, algo = PATHS[path]
    out = _run(X, logits, W, w.R, w.T, w.H, w.F, w.E, w.topk, cap, staged=staged,
               contiguous=contiguous, opts=fcc.make_opts(algo=algo))
    _check(X, logits, W, w.R, w.T, w.H, w.F, w.E, w.topk, cap, out, sample=48)


# ------------------------------------------------------------------ MoE combine

def _combine(out, R, T, F, E, topk, cap, in_dtype, out_dtype=fcc.FCC_BF16):
    tdt = torch.float32 if out_dtype == fcc.FCC_F32 else torch.bfloat16
    y = [empty((T, F), tdt, fill=float("nan")) for _ in range(R)]
    fcc.fcc_moe_combine(R, out["recv_y"], cap, T, F, E, topk, out["idx"], out["gate"],
                        out["src"], out["counts"], y, in_dtype, out_dtype)
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    return y


def _combine_ref(X, W, logits, R, T, E, topk, cap, tokens=None):
    """Oracle combine from the oracle's own routing; slots whose row falls past
    cap in the full dispatch were dropped (they add nothing)."""
    idx, gate = oracle.moe_route(np.stack(logits), topk)
    d = oracle.moe_dispatch(idx, R, E, R * T * topk)
    ix = idx.reshape(R * T, topk).copy()
    ix[d.recv_row.reshape(R * T, topk) >= cap] = -1
    g = gate.reshape(R * T, topk)
    tok = np.arange(R * T) if tokens is None else np.asarray(tokens)
    return oracle.moe_combine(X, W, tok // T, tok % T, ix[tok], g[tok]), tok


@pytest.mark.parametrize("R,T,H,F,E,topk", [
    (2, 300, 128, 136, 8, 2),
    (4, 257, 256, 264, 16, 2),
    (8, 64, 64, 64, 64, 2),
    (2, 200, 192, 128, 4, 1),
    (1, 500, 128, 256, 8, 2),
])
@pytest.mark.parametrize("dtypes", [(fcc.FCC_BF16, fcc.FCC_BF16), (fcc.FCC_F32, fcc.FCC_F32)])
def test_moe_combine_small(R, T, H, F, E, topk, dtypes):
    """The return all-to-all + gate-weighted sum against the oracle's combine."""
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=R * 10 + T)
    cap = R * T * topk
    mid, out_dtype = dtypes
    out = _run(X, logits, W, R, T, H, F, E, topk, cap, mid, staged=False)
    y = _combine(out, R, T, F, E, topk, cap, mid, out_dtype)
    ref, _ = _combine_ref(X, W, logits, R, T, E, topk, cap)
    got = np.concatenate([to_f64(v) for v in y])
    assert_close(got, ref, "combined rows")


def test_moe_combine_capacity_drops_and_repeatable():
    """Rows dropped for capacity add nothing; two calls agree bit for bit."""
    R, T, H, F, E, topk = 2, 256, 64, 64, 4, 2
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=7)
    cap = 100
    out = _run(X, logits, W, R, T, H, F, E, topk, cap)
    assert out["status"] == fcc.FCC_ERR_CAPACITY
    y1 = _combine(out, R, T, F, E, topk, cap, fcc.FCC_BF16, fcc.FCC_F32)
    y2 = _combine(out, R, T, F, E, topk, cap, fcc.FCC_BF16, fcc.FCC_F32)
    for a, b in zip(y1, y2):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    ref, _ = _combine_ref(X, W, logits, R, T, E, topk, cap)
    assert_close(np.concatenate([to_f64(v) for v in y1]), ref, "combined rows with drops")


def test_moe_combine_invalid_arguments():
    R, T, F, E, topk, cap = 2, 16, 64, 4, 2, 64
    dummy = [empty((cap, F), torch.bfloat16) for _ in range(R)]
    ints = [torch.zeros((T, topk), dtype=torch.int32, device="cuda") for _ in range(R)]
    flts = [torch.zeros((T, topk), dtype=torch.float32, device="cuda") for _ in range(R)]
    src = [torch.zeros((cap,), dtype=torch.int32, device="cuda") for _ in range(R)]
    counts = torch.zeros((E,), dtype=torch.int32, device="cuda")
    y = [empty((T, F), torch.bfloat16) for _ in range(R)]
    for bad in [dict(E=3), dict(topk=3), dict(F=60)]:
        kw = dict(E=E, topk=topk, F=F)
        kw.update(bad)
        with pytest.raises(fcc.FccError) as e:
            fcc.fcc_moe_combine(R, dummy, cap, T, kw["F"], kw["E"], kw["topk"], ints, flts, src,
                                counts, y)
        assert e.value.status == fcc.FCC_ERR_INVALID
    with pytest.raises(fcc.FccError) as e:
        fcc.fcc_moe_combine(R, dummy, cap, T, F, E, topk, ints, flts, src, counts, y,
                            fcc.FCC_F16, fcc.FCC_BF16)
    assert e.value.status == fcc.FCC_ERR_UNSUPPORTED


def test_moe_combine_full_workload_sampled():
    """The benchmark's shapes: dispatch + expert GEMM, then the combine, on 48
    sampled tokens of the 32768."""
    w = synth.WORKLOADS["moe_r8_t4096_h4096_e64_f1408"]
    X, logits, W = synth.moe_inputs(w.R, w.T, w.H, w.E, w.F, std_x=w.std_a, std_w=w.std_b,
                                    seed=0)
    cap = 2 * w.T * w.topk
    out = _run(X, logits, W, w.R, w.T, w.H, w.F, w.E, w.topk, cap, staged=False)
    y = _combine(out, w.R, w.T, w.F, w.E, w.topk, cap, fcc.FCC_BF16)
    rng = np.random.Generator(np.random.PCG64(3))
    tok = np.sort(rng.choice(w.R * w.T, size=48, replace=False))
    ref, tok = _combine_ref(X, W, logits, w.R, w.T, w.E, w.topk, cap, tok)
    got = np.stack([to_f64(y[t // w.T][int(t % w.T)]) for t in tok])
    assert_close(got, ref, "combined rows (sampled)")


def test_grouped_gemm_unit_wait_reports_timeout_and_context_survives():
    """The expert GEMM's TMA producer waits (bounded) for the copy warps to
    publish a unit's rows.  With a unit whose counter nothing raises, the wait
    runs out: the status word reports FCC_ERR_TIMEOUT, reading it clears it,
    and the next dispatch + GEMM on the same context is still correct."""
    fcc.fcc_test_grouped_wait_timeout(2_000_000)  # 2 ms
    assert fcc.fcc_stream_status() == fcc.FCC_ERR_TIMEOUT
    assert fcc.fcc_stream_status() == fcc.FCC_OK
    R, T, H, F, E, topk = 2, 300, 128, 136, 8, 2
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=21)
    cap = R * T * topk
    out = _run(X, logits, W, R, T, H, F, E, topk, cap)
    _check(X, logits, W, R, T, H, F, E, topk, cap, out)


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("H", [320, 200])
def test_moe_workspace_staging_equals_copy_kernel(pair, H):
    """The default with no recv_x: the GEMM's copy warps stage the rows in
    library workspace, so the products are bit for bit those of the rows
    staged by the copy kernel (the same MMAs); H = 200 ends in a partial
    64-wide k block.  A second call repeats them."""
    R, T, F, E, topk = 4, 700, 264, 8, 2   # 350 rows an expert: a ragged unit
    X, logits, W = synth.moe_inputs(R, T, H, E, F, seed=13 + H)
    cap = R * T * topk
    o_auto = fcc.make_opts(cta_pair=pair, algo=fcc.FCC_ALGO_AUTO)
    o_sep = fcc.make_opts(cta_pair=pair, algo=fcc.FCC_ALGO_UNFUSED)
    a = _run(X, logits, W, R, T, H, F, E, topk, cap, opts=o_auto, staged=False)
    b = _run(X, logits, W, R, T, H, F, E, topk, cap, opts=o_sep)
    c = _run(X, logits, W, R, T, H, F, E, topk, cap, opts=o_auto, staged=False)
    _check(X, logits, W, R, T, H, F, E, topk, cap, a)
    for d in range(R):
        n = int((a["src"][d] >= 0).sum())
        for other in (b, c):
            assert torch.equal(a["src"][d], other["src"][d])
            assert torch.equal(a["recv_y"][d][:n].view(torch.int16),
                               other["recv_y"][d][:n].view(torch.int16))
