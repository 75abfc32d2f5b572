"""CPU fp64 oracle for the fused GEMM + collective operators.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library: the arithmetic lives in ``fcc_oracle.c`` (plain loops,
double precision) and this module only marshals numpy arrays to it.

bfloat16 arrays are ``numpy.uint16`` bit patterns (see the ``synth`` module).
Every routine returns float64 arrays (integers for the MoE index work).

The operator definitions and the passages they follow are stated in the
header of ``fcc_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fcc_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fcc_oracle.c into liboracle.so with gcc (-O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.orc_num_threads.restype = I
        lib.orc_rank_sum_rows.argtypes = [I, P, P, I64, I64, I64, P, I64, P]
        lib.orc_gemm_rs_rows.argtypes = [I, P, P, I64, I64, I64, I, P, I64, P]
        lib.orc_ag_gemm_rows.argtypes = [I, P, P, I64, I64, I64, I, P, I64, P]
        lib.orc_moe_route.argtypes = [I64, I, I, P, P, P]
        lib.orc_moe_dispatch.argtypes = [I, I64, I, I, P, I64, P, P, P, P, P, P]
        lib.orc_moe_expert_rows.argtypes = [I, P, P, I64, I64, I64, I, P, P, P, I64, P]
        lib.orc_moe_combine_rows.argtypes = [I, P, P, I64, I64, I64, I, I, P, P, P, P, I64,
                                             P]
        lib.orc_embedding_bags.argtypes = [I, P, I64, I64, P, P, I64, P, P, I64, P]
        lib.orc_attention_rows.argtypes = [I, P, P, P, I64, I, I64, I, I64, P, P, P, P]
        for f in (lib.orc_rank_sum_rows, lib.orc_gemm_rs_rows, lib.orc_ag_gemm_rows,
                  lib.orc_moe_route, lib.orc_moe_dispatch, lib.orc_moe_expert_rows,
                  lib.orc_moe_combine_rows, lib.orc_embedding_bags, lib.orc_attention_rows):
            f.restype = I
        _lib = lib
        return lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().orc_num_threads())


def _ptr_array(arrs, dtype):
    keep = [np.ascontiguousarray(a, dtype=dtype) for a in arrs]
    ptrs = (ctypes.c_void_p * len(keep))(*[a.ctypes.data for a in keep])
    return keep, ptrs


def _rows_arg(rows, limit):
    if rows is None:
        rows = np.arange(limit, dtype=np.int64)
    return np.ascontiguousarray(rows, dtype=np.int64)


def rank_sum(A, B, rows=None) -> np.ndarray:
    """S[rows] with S = sum_r A_r @ B_r (fp64).  The all-reduce result."""
    R = len(A)
    M, K = A[0].shape
    N = B[0].shape[1]
    rows = _rows_arg(rows, M)
    out = np.empty((rows.size, N), dtype=np.float64)
    ka, pa = _ptr_array(A, np.uint16)
    kb, pb = _ptr_array(B, np.uint16)
    rc = _load().orc_rank_sum_rows(R, pa, pb, M, N, K, rows.ctypes.data, rows.size,
                                   out.ctypes.data)
    if rc:
        raise ValueError(f"orc_rank_sum_rows: bad argument ({rc})")
    return out


def gemm_rs(A, B, j: int, local_rows=None) -> np.ndarray:
    """Shard j of the reduce-scatter: rows [j*M/R, (j+1)*M/R) of sum_r A_r @ B_r."""
    R = len(A)
    M, K = A[0].shape
    N = B[0].shape[1]
    if M % R:
        raise ValueError("M must be divisible by R")
    local_rows = _rows_arg(local_rows, M // R)
    out = np.empty((local_rows.size, N), dtype=np.float64)
    ka, pa = _ptr_array(A, np.uint16)
    kb, pb = _ptr_array(B, np.uint16)
    rc = _load().orc_gemm_rs_rows(R, pa, pb, M, N, K, j, local_rows.ctypes.data,
                                  local_rows.size, out.ctypes.data)
    if rc:
        raise ValueError(f"orc_gemm_rs_rows: bad argument ({rc})")
    return out


def gemm_ar(A, B, rows=None) -> np.ndarray:
    """The all-reduce result every rank's buffer must hold (rows of sum_r A_r @ B_r)."""
    return rank_sum(A, B, rows)


def gemv_ar(A, B) -> np.ndarray:
    """GEMV + all-reduce: the full (M<=16) x N rank sum every rank receives."""
    return rank_sum(A, B)


def ag_gemm(X, B, r: int, rows=None) -> np.ndarray:
    """All-gather + GEMM for rank r: rows of [X_0; ...; X_{R-1}] @ B_r."""
    R = len(X)
    Ms, K = X[0].shape
    M = Ms * R
    N = B[0].shape[1]
    rows = _rows_arg(rows, M)
    out = np.empty((rows.size, N), dtype=np.float64)
    kx, px = _ptr_array(X, np.uint16)
    kb, pb = _ptr_array(B, np.uint16)
    rc = _load().orc_ag_gemm_rows(R, px, pb, M, N, K, r, rows.ctypes.data, rows.size,
                                  out.ctypes.data)
    if rc:
        raise ValueError(f"orc_ag_gemm_rows: bad argument ({rc})")
    return out


def moe_route(logits: np.ndarray, topk: int):
    """Top-k experts per token by logit (ties to the lower index) and softmax gates."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    E = lg.shape[-1]
    ntok = lg.size // E
    idx = np.empty((ntok, topk), dtype=np.int32)
    gate = np.empty((ntok, topk), dtype=np.float64)
    rc = _load().orc_moe_route(ntok, E, topk, lg.ctypes.data, idx.ctypes.data,
                               gate.ctypes.data)
    if rc:
        raise ValueError(f"orc_moe_route: bad argument ({rc})")
    shape = lg.shape[:-1] + (topk,)
    return idx.reshape(shape), gate.reshape(shape)


class Dispatch:
    """Result of the MoE all-to-all dispatch (see orc_moe_dispatch)."""

    def __init__(self, counts, send_counts, recv_counts, recv_row, recv_src, recv_expert):
        self.counts = counts            # [E]
        self.send_counts = send_counts  # [R, R]  (source, destination)
        self.recv_counts = recv_counts  # [R]
        self.recv_row = recv_row        # [R, T, topk]
        self.recv_src = recv_src        # [R, cap]  s*T + t, -1 past recv_counts
        self.recv_expert = recv_expert  # [R, cap]


def moe_dispatch(idx: np.ndarray, R: int, E: int, cap: int) -> Dispatch:
    """Stable counting sort of the (source, token, slot) assignments by expert."""
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    topk = ix.shape[-1]
    T = ix.size // (R * topk)
    counts = np.empty(E, dtype=np.int32)
    send = np.empty((R, R), dtype=np.int32)
    recvc = np.empty(R, dtype=np.int32)
    row = np.empty(ix.size, dtype=np.int32)
    src = np.empty((R, cap), dtype=np.int32)
    exp_ = np.empty((R, cap), dtype=np.int32)
    rc = _load().orc_moe_dispatch(R, T, E, topk, ix.ctypes.data, cap, counts.ctypes.data,
                                  send.ctypes.data, recvc.ctypes.data, row.ctypes.data,
                                  src.ctypes.data, exp_.ctypes.data)
    if rc == 2:
        raise OverflowError("a rank receives more rows than cap")
    if rc:
        raise ValueError(f"orc_moe_dispatch: bad argument ({rc})")
    return Dispatch(counts, send, recvc, row.reshape(R, T, topk), src, exp_)


def moe_expert_rows(X, W, src_rank, src_tok, expert) -> np.ndarray:
    """Rows X_{src_rank}[src_tok] @ W_{expert} (fp64), one per entry."""
    R = len(X)
    T, H = X[0].shape
    E = len(W)
    F = W[0].shape[1]
    sr = np.ascontiguousarray(src_rank, dtype=np.int32)
    st = np.ascontiguousarray(src_tok, dtype=np.int32)
    ex = np.ascontiguousarray(expert, dtype=np.int32)
    out = np.empty((sr.size, F), dtype=np.float64)
    kx, px = _ptr_array(X, np.uint16)
    kw, pw = _ptr_array(W, np.uint16)
    rc = _load().orc_moe_expert_rows(R, px, pw, T, H, F, E, sr.ctypes.data, st.ctypes.data,
                                     ex.ctypes.data, sr.size, out.ctypes.data)
    if rc:
        raise ValueError(f"orc_moe_expert_rows: bad argument ({rc})")
    return out


def moe_combine(X, W, src_rank, src_tok, idx, gate) -> np.ndarray:
    """Per token (src_rank[i], src_tok[i]): sum over its slots j of
    gate[i, j] * (X_s[t] @ W_{idx[i, j]}) in fp64, slots in order; idx < 0 = a
    slot whose row was not received (adds nothing).  [n, F]."""
    R = len(X)
    T, H = X[0].shape
    E = len(W)
    F = W[0].shape[1]
    sr = np.ascontiguousarray(src_rank, dtype=np.int32)
    st = np.ascontiguousarray(src_tok, dtype=np.int32)
    ix = np.ascontiguousarray(idx, dtype=np.int32).reshape(sr.size, -1)
    g = np.ascontiguousarray(gate, dtype=np.float64).reshape(ix.shape)
    topk = ix.shape[1]
    out = np.empty((sr.size, F), dtype=np.float64)
    kx, px = _ptr_array(X, np.uint16)
    kw, pw = _ptr_array(W, np.uint16)
    rc = _load().orc_moe_combine_rows(R, px, pw, T, H, F, E, topk, sr.ctypes.data,
                                      st.ctypes.data, ix.ctypes.data, g.ctypes.data, sr.size,
                                      out.ctypes.data)
    if rc:
        raise ValueError(f"orc_moe_combine_rows: bad argument ({rc})")
    return out


def embedding_bags(tables, offsets, indices, bag_table, bag_sample) -> np.ndarray:
    """Pooled (summed) rows of the bags (bag_table[i], bag_sample[i]) in fp64, [n, D].
    tables: list of [V, D] bf16; offsets[tau]: [nsamples + 1]; indices[tau]: [nnz]."""
    V, D = tables[0].shape
    nsamples = len(offsets[0]) - 1
    kt, pt = _ptr_array(tables, np.uint16)
    ko, po = _ptr_array(offsets, np.int32)
    ki, pi = _ptr_array(indices, np.int32)
    bt = np.ascontiguousarray(bag_table, dtype=np.int32)
    bs = np.ascontiguousarray(bag_sample, dtype=np.int64)
    out = np.empty((bt.size, D), dtype=np.float64)
    rc = _load().orc_embedding_bags(len(tables), pt, V, D, po, pi, nsamples, bt.ctypes.data,
                                    bs.ctypes.data, bt.size, out.ctypes.data)
    if rc:
        raise ValueError(f"orc_embedding_bags: bad argument ({rc})")
    return out


def embedding_a2a(tables, offsets, indices, R: int):
    """The all-to-all result: out[r] is [Bl, ntables, D], row (b, tau) the pooled
    bag (tau, r*Bl + b), where Bl = nsamples / R samples live on each rank."""
    ntab = len(tables)
    nsamples = len(offsets[0]) - 1
    Bl = nsamples // R
    g = np.repeat(np.arange(nsamples, dtype=np.int64), ntab)   # sample-major, table-minor
    tau = np.tile(np.arange(ntab, dtype=np.int32), nsamples)
    rows = embedding_bags(tables, offsets, indices, tau, g)
    D = rows.shape[1]
    return [rows[r * Bl * ntab:(r + 1) * Bl * ntab].reshape(Bl, ntab, D) for r in range(R)]


def attention_rows(Q, K, V, causal, rank, row, head) -> np.ndarray:
    """Exact softmax attention (fp64) of the query rows (rank[i], row[i], head[i])
    over the keys and values of all shards; Q[r], K[r], V[r] are [S, H, d] bf16."""
    R = len(Q)
    S, H, d = Q[0].shape
    kq, pq = _ptr_array([q.reshape(-1) for q in Q], np.uint16)
    kk, pk = _ptr_array([k.reshape(-1) for k in K], np.uint16)
    kv, pv = _ptr_array([v.reshape(-1) for v in V], np.uint16)
    rk = np.ascontiguousarray(rank, dtype=np.int32)
    rw = np.ascontiguousarray(row, dtype=np.int64)
    hd = np.ascontiguousarray(head, dtype=np.int32)
    out = np.empty((rk.size, d), dtype=np.float64)
    rc = _load().orc_attention_rows(R, pq, pk, pv, S, H, d, 1 if causal else 0, rk.size,
                                    rk.ctypes.data, rw.ctypes.data, hd.ctypes.data,
                                    out.ctypes.data)
    if rc:
        raise ValueError(f"orc_attention_rows: bad argument ({rc})")
    return out


def ring_attention(Q, K, V, causal=False):
    """All output rows: a list of [S, H, d] fp64 arrays, one per rank."""
    R = len(Q)
    S, H, d = Q[0].shape
    rank = np.repeat(np.arange(R), S * H)
    row = np.tile(np.repeat(np.arange(S), H), R)
    head = np.tile(np.arange(H), R * S)
    o = attention_rows(Q, K, V, causal, rank, row, head)
    return [o[r * S * H:(r + 1) * S * H].reshape(S, H, d) for r in range(R)]


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (for comparing outputs)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
