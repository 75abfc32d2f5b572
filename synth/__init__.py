"""Seeded synthetic inputs for the fused GEMM + collective operators.

Shared by the tests (both the CPU oracle and the CUDA path consume the very
same arrays) and by the benchmark.  This module holds none of the operators'
arithmetic: it only draws float32 normals from numpy's PCG64 generator,
scales them, and rounds them to bfloat16 bit patterns (round to nearest,
ties to even).  bfloat16 tensors are returned as ``numpy.uint16`` arrays of
raw bits; router logits stay float32.

Draw order is fixed per workload so that a seed fully determines every byte:
GEMM workloads draw A_0..A_{R-1} then B_0..B_{R-1}; the MoE workload draws
X_0..X_{R-1}, then logits_0..logits_{R-1}, then W_0..W_{E-1}; the embedding
workload draws the tables 0..n-1, then per table the bag sizes and indices.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = [
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "normal_bf16",
    "integer_bf16",
    "gemm_inputs",
    "integer_gemm_inputs",
    "moe_inputs",
    "embedding_inputs",
    "attention_inputs",
    "WORKLOADS",
    "Workload",
]


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits.

    NaN inputs map to a quiet NaN with the same sign; +-inf stay infinite and
    finite values that round past the largest bfloat16 become infinite.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    is_nan = (u & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    quiet = (u >> np.uint64(16)) | np.uint64(0x0040)
    return np.where(is_nan, quiet, rounded).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """float32 N(0, std^2) draw, rounded to bfloat16 bits."""
    z = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    return f32_to_bf16_bits(z)


def integer_bf16(rng: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    """Uniform integers in [lo, hi] stored as bfloat16 bits (exactly representable)."""
    v = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return f32_to_bf16_bits(v)


def gemm_inputs(R: int, M: int, N: int, K: int, std_a: float, std_b: float,
                seed: int = 0):
    """A_r [M,K] and B_r [K,N] bf16 bits for r < R (A's drawn first, then B's)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    A = [normal_bf16(rng, (M, K), std_a) for _ in range(R)]
    B = [normal_bf16(rng, (K, N), std_b) for _ in range(R)]
    return A, B


def integer_gemm_inputs(R: int, M: int, N: int, K: int, lo: int = -4, hi: int = 4,
                        seed: int = 0):
    """Integer-valued A_r, B_r (exact in bf16); sums stay exact in fp32 when small."""
    rng = np.random.Generator(np.random.PCG64(seed))
    A = [integer_bf16(rng, (M, K), lo, hi) for _ in range(R)]
    B = [integer_bf16(rng, (K, N), lo, hi) for _ in range(R)]
    return A, B


def moe_inputs(R: int, T: int, H: int, E: int, F: int, std_x: float = 1.0,
               std_logit: float = 1.0, std_w: float = 0.02, seed: int = 0):
    """Per-rank tokens X_s [T,H] bf16, router logits [T,E] float32, experts W_e [H,F] bf16."""
    rng = np.random.Generator(np.random.PCG64(seed))
    X = [normal_bf16(rng, (T, H), std_x) for _ in range(R)]
    logits = []
    for _ in range(R):
        z = rng.standard_normal(size=(T, E), dtype=np.float32)
        if std_logit != 1.0:
            z *= np.float32(std_logit)
        logits.append(z)
    W = [normal_bf16(rng, (H, F), std_w) for _ in range(E)]
    return X, logits, W


def embedding_inputs(R: int, ntables: int, V: int, D: int, Bl: int, L: int,
                     min_bag: int = 1, std: float = 1.0, seed: int = 0):
    """Embedding tables [V, D] bf16 (N(0, std)), and per table the bags of the
    R * Bl samples of the global batch in CSR form: bag sizes uniform in
    [min_bag, 2L - min_bag] (mean L), indices uniform in [0, V).
    Returns (tables, offsets, indices): offsets[t] int32 [R*Bl + 1]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    tables = [normal_bf16(rng, (V, D), std) for _ in range(ntables)]
    n = R * Bl
    offsets, indices = [], []
    for _ in range(ntables):
        sizes = rng.integers(min_bag, 2 * L - min_bag + 1, size=n, dtype=np.int64)
        off = np.zeros(n + 1, dtype=np.int64)
        np.cumsum(sizes, out=off[1:])
        offsets.append(off.astype(np.int32))
        indices.append(rng.integers(0, V, size=int(off[-1]), dtype=np.int32))
    return tables, offsets, indices


def attention_inputs(R: int, S: int, H: int, d: int, std: float = 1.0, seed: int = 0):
    """Per rank Q_r, K_r, V_r [S, H, d] bf16, N(0, std), drawn Q_0..Q_{R-1},
    K_0..K_{R-1}, V_0..V_{R-1}."""
    rng = np.random.Generator(np.random.PCG64(seed))
    Q = [normal_bf16(rng, (S, H, d), std) for _ in range(R)]
    K = [normal_bf16(rng, (S, H, d), std) for _ in range(R)]
    V = [normal_bf16(rng, (S, H, d), std) for _ in range(R)]
    return Q, K, V


@dataclass(frozen=True)
class Workload:
    """One named workload: shapes, value distributions and output dtype."""
    name: str
    op: str            # gemm_rs | gemm_ar | gemv_ar | ag_gemm | moe | emb_a2a | attention
    R: int
    M: int = 0         # GEMM rows (all ranks for AG: R * rows per rank)
    N: int = 0
    K: int = 0
    std_a: float = 1.0
    std_b: float = 1.0
    out: str = "bf16"  # output storage dtype
    T: int = 0         # MoE tokens per rank
    H: int = 0
    E: int = 0
    F: int = 0
    topk: int = 0
    tables: int = 0    # embedding: tables (tables / R owned by each rank)
    B: int = 0         # embedding: samples per rank
    V: int = 0         # embedding: rows per table
    D: int = 0         # embedding: row width
    L: int = 0         # embedding: mean bag size (pooling factor)

    def emb_bytes(self) -> int:
        """Embedding: rows read once per lookup plus the pooled outputs written once
        (bf16), the mean lookup count taken as R * Bl * tables * L."""
        n = self.R * self.B * self.tables
        return n * self.L * self.D * 2 + n * self.D * 2

    def flops(self) -> float:
        """2 * useful multiply-adds of the workload."""
        if self.op == "moe":
            return 2.0 * self.R * self.T * self.topk * self.H * self.F
        if self.op == "attention":
            # Q K^T and P V over every (query, key) pair: 4 * S_q * S_k * d per head
            return 4.0 * (self.R * self.M) * (self.R * self.M) * self.K * self.H
        if self.op == "ag_gemm":
            return 2.0 * self.R * self.M * self.N * self.K
        return 2.0 * self.R * self.M * self.N * self.K


WORKLOADS = {
    # GEMM + reduce-scatter, 2 ranks, fp32 row shards of 128x256.
    "gemm_rs_r2_256x256x128": Workload("gemm_rs_r2_256x256x128", "gemm_rs", R=2, M=256,
                                       N=256, K=128, std_a=1.0 / math.sqrt(128.0),
                                       std_b=1.0 / math.sqrt(128.0), out="f32"),
    # Row-parallel MLP down-projection: 8 ranks, bf16 shards of 1024x8192.
    "gemm_rs_r8_8192x8192x3584": Workload("gemm_rs_r8_8192x8192x3584", "gemm_rs", R=8,
                                          M=8192, N=8192, K=3584, std_a=0.02, std_b=0.02,
                                          out="bf16"),
    # Same shape, all-reduce into every rank's full buffer.
    "gemm_ar_r8_8192x8192x3584": Workload("gemm_ar_r8_8192x8192x3584", "gemm_ar", R=8,
                                          M=8192, N=8192, K=3584, std_a=0.02, std_b=0.02,
                                          out="bf16"),
    # Decode GEMV + all-reduce: 8 tokens, fp32 sum written to all 8 rank buffers.
    "gemv_ar_r8_8x8192x3584": Workload("gemv_ar_r8_8x8192x3584", "gemv_ar", R=8, M=8,
                                       N=8192, K=3584, std_a=1.0, std_b=0.02, out="f32"),
    # All-gather + GEMM, column parallel: 8 x 1024 token rows gathered to 8192 rows.
    "ag_gemm_r8_8192x3584x8192": Workload("ag_gemm_r8_8192x3584x8192", "ag_gemm", R=8,
                                          M=8192, N=3584, K=8192, std_a=1.0, std_b=0.02,
                                          out="bf16"),
    # MoE dispatch + expert GEMM: 8 ranks x 4096 tokens, 64 experts, top-2.
    "moe_r8_t4096_h4096_e64_f1408": Workload("moe_r8_t4096_h4096_e64_f1408", "moe", R=8,
                                             T=4096, H=4096, E=64, F=1408, topk=2,
                                             std_a=1.0, std_b=0.02, out="bf16"),
    # Embedding + all-to-all (DLRM-style): 8 ranks x 8 tables of 65536 x 128
    # rows, 2048 samples per rank, bags of 32 rows on average.
    # Ring attention: 8 ranks x 4096 positions (32768 in all), 8 heads, d = 128
    # (M = positions per rank, K = head dimension).
    "attn_r8_s4096_h8_d128": Workload("attn_r8_s4096_h8_d128", "attention", R=8, M=4096,
                                      K=128, H=8, std_a=1.0, out="bf16"),
    "emb_a2a_r8_t64_v65536_d128_b2048_l32": Workload(
        "emb_a2a_r8_t64_v65536_d128_b2048_l32", "emb_a2a", R=8, tables=64, B=2048,
        V=65536, D=128, L=32, std_a=1.0, out="bf16"),
}
