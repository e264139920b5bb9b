"""Shared pieces of the GPU parity tests: the library handle, seeded inputs
moved to the device, and element-wise comparison against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

_HANDLE = None


def handle():
    global _HANDLE
    if _HANDLE is None:
        import __graft_entry__

        __graft_entry__.build()
        import mxfp8_block_scaled_06_gb300 as mx

        torch.cuda.set_device(0)
        _HANDLE = mx.mx_create(0)
    return _HANDLE


def dev():
    return torch.device("cuda:0")


def bf16_to_device(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def u8(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.uint8).cpu().numpy() if t.dtype != torch.uint8 else t.cpu().numpy()


def operands(seed: int, tag: int, rows: int, k: int, umin: int = -6, umax: int = 6):
    """bf16 bits of a block-scaled N(0,1) matrix, its exact values, and the
    oracle's MXFP8 (codes, plain scale bytes)."""
    bits = synth.block_scaled_bf16(seed, tag, rows, k, umin, umax)
    vals = synth.bf16_bits_to_f64(bits)
    return bits, vals, oracle.mx_quantize(vals)


def quantize_on_gpu(bits: np.ndarray):
    """The product path: bf16 on the device -> mx_quantize_rows (swizzled)."""
    import mxfp8_block_scaled_06_gb300 as mx

    x = bf16_to_device(bits)
    return mx.mx_quantize_rows(handle(), x)


def assert_gemm_close(got_bf16: torch.Tensor, ref: np.ndarray, what: str = "") -> float:
    """|gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref), element by element."""
    got = got_bf16.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    tol = oracle.gemm_tolerance(ref)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements beyond tolerance; first "
            + ", ".join(f"{tuple(i)} got {got[tuple(i)]:.6g} ref {ref[tuple(i)]:.6g}" for i in idx))
    return float((err / np.maximum(tol, 1e-300)).max())
