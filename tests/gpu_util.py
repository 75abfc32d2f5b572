"""Helpers for the GPU parity tests: device buffers and the float tolerance.

Tolerance for float outputs (bf16 inputs, f32 accumulation): relative
Frobenius error <= 5e-3 and max |err| <= 1e-2 * max |ref| against the fp64
oracle.
"""
import numpy as np
import torch

REL_FRO = 5e-3
MAX_REL = 1e-2


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """Upload bf16 bit patterns (uint16) as a CUDA bfloat16 tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.cuda().view(torch.bfloat16)


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def empty(shape, dtype=torch.bfloat16, fill=None) -> torch.Tensor:
    t = torch.empty(shape, dtype=dtype, device="cuda")
    if fill is not None:
        t.fill_(fill)
    return t


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bytes of a tensor as a numpy array (bitwise comparisons)."""
    if t.dtype == torch.bfloat16:
        return t.detach().cpu().view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.detach().cpu().view(torch.int32).numpy()
    return t.detach().cpu().numpy()


def errors(got: np.ndarray, ref: np.ndarray):
    diff = got - ref
    fro = np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300)
    mx = np.max(np.abs(diff)) / max(np.max(np.abs(ref)), 1e-300)
    return fro, mx


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    fro, mx = errors(got, ref)
    assert fro <= REL_FRO and mx <= MAX_REL, f"{what}: rel_fro={fro:.3e} max_rel={mx:.3e}"
    return fro, mx
