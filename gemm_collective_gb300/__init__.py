"""Python binding of libfcc (fused GEMM + collective on one GB300).

A thin ctypes layer over the C ABI declared in ``include/fcc.h``: every
function has the C name and argument order, and only marshals arguments
(lists of device pointers or CUDA tensors, a stream, an options struct).
All computation runs in the library's CUDA kernels.  Importing this module
loads ``libfcc.so``; if the library has not been built the import fails
loudly -- there is no fallback path.

Pointer-array arguments accept a sequence of ``int`` device addresses or of
objects with ``data_ptr()`` (torch tensors), or an array made once by
``ptr_array()``.  ``stream`` accepts ``None``
(the legacy default stream), an ``int`` handle or an object with a
``cuda_stream`` attribute (``torch.cuda.Stream``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfcc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libfcc.so is not built ({LIB_PATH}); run gemm_collective_gb300/build.py "
        "or __graft_entry__.build() first")

_lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------- constants
FCC_BF16, FCC_F16, FCC_F32 = 0, 1, 2
(FCC_OK, FCC_ERR_INVALID, FCC_ERR_UNSUPPORTED, FCC_ERR_CUDA, FCC_ERR_CAPACITY,
 FCC_ERR_TIMEOUT, FCC_ERR_WORKSPACE) = range(7)
(FCC_ALGO_AUTO, FCC_ALGO_FUSED, FCC_ALGO_UNFUSED, FCC_ALGO_INTERDECOM,
 FCC_ALGO_CE) = range(5)
FCC_OP_GEMM_RS, FCC_OP_GEMM_AR, FCC_OP_GEMV_AR, FCC_OP_AG_GEMM, FCC_OP_EMBEDDING_A2A = range(5)
FCC_MAX_RANKS = 8
FCC_MAX_EXPERTS = 64


class fcc_opts(ctypes.Structure):
    _fields_ = [
        ("algo", ctypes.c_int),
        ("deterministic", ctypes.c_int),
        ("chunks", ctypes.c_int),
        ("max_ctas", ctypes.c_int),
        ("timeout_ns", ctypes.c_int64),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("cta_pair", ctypes.c_int),
        ("phase_ns", ctypes.c_void_p),
    ]


def make_opts(algo=FCC_ALGO_AUTO, deterministic=1, chunks=0, max_ctas=0, timeout_ns=0,
              workspace=None, workspace_bytes=0, cta_pair=0, phase_ns=None) -> fcc_opts:
    ws = workspace.data_ptr() if hasattr(workspace, "data_ptr") else workspace
    ph = phase_ns.data_ptr() if hasattr(phase_ns, "data_ptr") else phase_ns
    return fcc_opts(algo, deterministic, chunks, max_ctas, timeout_ns, ws, workspace_bytes,
                    cta_pair, ph)


class FccError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fcc_status_string(status)} ({status})")


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_OPTS = ctypes.POINTER(fcc_opts)


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_gemm_rs = _sig("fcc_gemm_rs", _I, [_I, _P, _P, _P, _I64, _I64, _I64, _I, _I, _OPTS, _P])
_gemm_ar = _sig("fcc_gemm_ar", _I, [_I, _P, _P, _P, _I64, _I64, _I64, _I, _I, _OPTS, _P])
_gemv_ar = _sig("fcc_gemv_ar", _I, [_I, _P, _P, _P, _I64, _I64, _I64, _I, _I, _OPTS, _P])
_gemv_ar_static = _sig("fcc_gemv_ar_static", _I,
                       [_I, _P, _P, _P, _I64, _I64, _I64, _I, _I, _OPTS, _P])
_ag_gemm = _sig("fcc_ag_gemm", _I, [_I, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _OPTS, _P])
_moe = _sig("fcc_moe_dispatch_gemm", _I,
            [_I, _P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _I64, _P, _P, _P, _P, _P, _I, _I,
             _OPTS, _P])
_combine = _sig("fcc_moe_combine", _I,
                [_I, _P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _P, _I, _I, _OPTS, _P])
_combine_ws = _sig("fcc_moe_combine_workspace_size", ctypes.c_size_t, [_I, _I64, _I])
_emb = _sig("fcc_embedding_a2a", _I,
            [_I, _I, _P, _I64, _I64, _I64, _P, _P, _P, _I, _I, _OPTS, _P])
_emb_ws = _sig("fcc_embedding_workspace_size", ctypes.c_size_t,
               [_I, _I, _I64, _I64, _I, _OPTS])
_ws = _sig("fcc_workspace_size", ctypes.c_size_t, [_I, _I, _I64, _I64, _I64, _OPTS])
_moe_ws = _sig("fcc_moe_workspace_size", ctypes.c_size_t,
               [_I, _I64, _I64, _I64, _I, _I, _I64, _OPTS])
_stream_status = _sig("fcc_stream_status", _I, [_P])
_status_string = _sig("fcc_status_string", ctypes.c_char_p, [_I])
_chunks = _sig("fcc_interdecom_chunks", _I, [ctypes.c_double, ctypes.c_double,
                                              ctypes.c_double, _I])
_itime = _sig("fcc_interdecom_time", ctypes.c_double, [ctypes.c_double, ctypes.c_double,
                                                       ctypes.c_double, _I])
_choose = _sig("fcc_choose_algo", _I, [_I, _I, _I64, _I64, _I64, _I, _I])
_attn = _sig("fcc_ring_attention", _I,
             [_I, _P, _P, _P, _P, _I64, _I, _I64, _I, _I, _I, _OPTS, _P])
_launches = _sig("fcc_launch_count", ctypes.c_uint64, [])
_version = _sig("fcc_version", ctypes.c_char_p, [])
_wait_timeout = _sig("fcc_test_wait_timeout", _I, [_I64, _P])
_grouped_wait_timeout = _sig("fcc_test_grouped_wait_timeout", _I, [_I64, _P])
_ksplit_wait_timeout = _sig("fcc_test_ksplit_wait_timeout", _I, [_I64, _P])


# ---------------------------------------------------------------- marshalling
def _addr(x) -> int:
    if x is None:
        return 0
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x)


def _ptrs(seq):
    if seq is None:
        return None
    if isinstance(seq, ctypes.Array):  # built once by ptr_array()
        return seq
    vals = [_addr(x) for x in seq]
    return (ctypes.c_void_p * len(vals))(*vals)


def ptr_array(seq):
    """The C array of device pointers for a sequence of tensors (or addresses).

    Every call accepts it wherever it takes a pointer array; a loop that calls
    an operator on the same buffers again and again can build its arrays once
    instead of marshalling the tensors on every call.  It holds addresses
    only: the tensors must stay alive (and in place) while it is in use."""
    return _ptrs(list(seq))


def _stream(s) -> int:
    if s is None:
        return 0
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    return int(s)


def _opts(o):
    return ctypes.byref(o) if o is not None else None


def _check(st: int, where: str):
    if st != FCC_OK:
        raise FccError(st, where)


# ------------------------------------------------------------------ the calls
def fcc_gemm_rs(R, A, B, out_shard, M, N, K, in_dtype=FCC_BF16, out_dtype=FCC_BF16, opts=None,
                stream=None):
    _check(_gemm_rs(R, _ptrs(A), _ptrs(B), _ptrs(out_shard), M, N, K, in_dtype, out_dtype,
                    _opts(opts), _stream(stream)), "fcc_gemm_rs")


def fcc_gemm_ar(R, A, B, out, M, N, K, in_dtype=FCC_BF16, out_dtype=FCC_BF16, opts=None,
                stream=None):
    _check(_gemm_ar(R, _ptrs(A), _ptrs(B), _ptrs(out), M, N, K, in_dtype, out_dtype,
                    _opts(opts), _stream(stream)), "fcc_gemm_ar")


def fcc_gemv_ar(R, A, B, out, M, N, K, in_dtype=FCC_BF16, out_dtype=FCC_F32, opts=None,
                stream=None):
    _check(_gemv_ar(R, _ptrs(A), _ptrs(B), _ptrs(out), M, N, K, in_dtype, out_dtype,
                    _opts(opts), _stream(stream)), "fcc_gemv_ar")


def fcc_gemv_ar_static(R, A, B, out, M, N, K, in_dtype=FCC_BF16, out_dtype=FCC_F32, opts=None,
                       stream=None):
    """fcc_gemv_ar with its scratch in the library's static device array (no allocation)."""
    _check(_gemv_ar_static(R, _ptrs(A), _ptrs(B), _ptrs(out), M, N, K, in_dtype, out_dtype,
                           _opts(opts), _stream(stream)), "fcc_gemv_ar_static")


def fcc_ag_gemm(R, X_shard, B, out, gathered, M, N, K, in_dtype=FCC_BF16, out_dtype=FCC_BF16,
                opts=None, stream=None):
    _check(_ag_gemm(R, _ptrs(X_shard), _ptrs(B), _ptrs(out), _ptrs(gathered), M, N, K,
                    in_dtype, out_dtype, _opts(opts), _stream(stream)), "fcc_ag_gemm")


def fcc_moe_dispatch_gemm(R, X, logits, W, T, H, F, E, topk, recv_x, recv_y, cap, topk_idx,
                          topk_gate, expert_counts, send_counts, recv_src, in_dtype=FCC_BF16,
                          out_dtype=FCC_BF16, opts=None, stream=None):
    _check(_moe(R, _ptrs(X), _ptrs(logits), _ptrs(W), T, H, F, E, topk, _ptrs(recv_x),
                _ptrs(recv_y), cap, _ptrs(topk_idx), _ptrs(topk_gate), _addr(expert_counts),
                _addr(send_counts), _ptrs(recv_src), in_dtype, out_dtype, _opts(opts),
                _stream(stream)), "fcc_moe_dispatch_gemm")


def fcc_moe_combine(R, recv_y, cap, T, F, E, topk, topk_idx, topk_gate, recv_src,
                    expert_counts, y, in_dtype=FCC_BF16, out_dtype=FCC_BF16, opts=None,
                    stream=None):
    _check(_combine(R, _ptrs(recv_y), cap, T, F, E, topk, _ptrs(topk_idx), _ptrs(topk_gate),
                    _ptrs(recv_src), _addr(expert_counts), _ptrs(y), in_dtype, out_dtype,
                    _opts(opts), _stream(stream)), "fcc_moe_combine")


def fcc_moe_combine_workspace_size(R, T, topk) -> int:
    return int(_combine_ws(R, T, topk))


def fcc_embedding_a2a(R, ntables, tables, V, D, Bl, offsets, indices, out,
                      in_dtype=FCC_BF16, out_dtype=FCC_BF16, opts=None, stream=None):
    _check(_emb(R, ntables, _ptrs(tables), V, D, Bl, _ptrs(offsets), _ptrs(indices),
                _ptrs(out), in_dtype, out_dtype, _opts(opts), _stream(stream)),
           "fcc_embedding_a2a")


def fcc_embedding_workspace_size(R, ntables, D, Bl, out_dtype=FCC_BF16, opts=None) -> int:
    return int(_emb_ws(R, ntables, D, Bl, out_dtype, _opts(opts)))


def fcc_ring_attention(R, Q, K, V, O, S, H, d, causal=False, in_dtype=FCC_BF16,
                       out_dtype=FCC_BF16, opts=None, stream=None):
    _check(_attn(R, _ptrs(Q), _ptrs(K), _ptrs(V), _ptrs(O), S, H, d, 1 if causal else 0,
                 in_dtype, out_dtype, _opts(opts), _stream(stream)), "fcc_ring_attention")


def fcc_choose_algo(op, R, M, N, K, sms=0, max_ctas=0) -> int:
    """The algorithm FCC_ALGO_AUTO runs for this operator and shape."""
    return int(_choose(op, R, M, N, K, sms, max_ctas))


def fcc_workspace_size(op, R, M, N, K, opts=None) -> int:
    return int(_ws(op, R, M, N, K, _opts(opts)))


def fcc_moe_workspace_size(R, T, H, F, E, topk, cap, opts=None) -> int:
    return int(_moe_ws(R, T, H, F, E, topk, cap, _opts(opts)))


def fcc_stream_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status word."""
    return int(_stream_status(_stream(stream)))


def fcc_status_string(status: int) -> str:
    return _status_string(status).decode()


def fcc_interdecom_chunks(G: float, X: float, alpha: float, max_chunks: int) -> int:
    return int(_chunks(G, X, alpha, max_chunks))


def fcc_interdecom_time(G: float, X: float, alpha: float, chunks: int) -> float:
    return float(_itime(G, X, alpha, chunks))


def fcc_launch_count() -> int:
    return int(_launches())


def fcc_version() -> str:
    return _version().decode()


def fcc_test_wait_timeout(timeout_ns: int, stream=None):
    _check(_wait_timeout(timeout_ns, _stream(stream)), "fcc_test_wait_timeout")


def fcc_test_grouped_wait_timeout(timeout_ns: int, stream=None):
    _check(_grouped_wait_timeout(timeout_ns, _stream(stream)), "fcc_test_grouped_wait_timeout")


def fcc_test_ksplit_wait_timeout(timeout_ns: int, stream=None):
    _check(_ksplit_wait_timeout(timeout_ns, _stream(stream)), "fcc_test_ksplit_wait_timeout")


def raw_status(fn_name: str, *args) -> int:
    """Call a C entry point with already-marshalled ctypes arguments; return its status."""
    return int(getattr(_lib, fn_name)(*args))
