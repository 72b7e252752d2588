"""Helpers shared by the GPU parity tests: tolerance checks and conversions.

Tolerances (bf16 outputs against the oracle's fp32 values before rounding):
  normwise  ||gpu - ref||_2 / ||ref||_2 <= 5e-3
  elementwise |gpu - ref| <= 1e-2 + 1e-2 * |ref|
Masks and metadata are compared bit for bit.
"""
import numpy as np
import torch

from tests.conftest import bits_of

NORM_TOL = 5e-3
ABS_TOL = 1e-2
REL_TOL = 1e-2


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_close(gpu: torch.Tensor, ref: np.ndarray, name: str, extra=None):
    """extra: optional per-element addition to the elementwise bound (the propagated
    rounding of a bf16 intermediate, see ulp_bf16 / propagated)."""
    g = f32(gpu).astype(np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    if r.size == 0:
        return
    diff = np.abs(g - r)
    nref = np.linalg.norm(r)
    normwise = np.linalg.norm(g - r) / (nref if nref > 0 else 1.0)
    bound = ABS_TOL + REL_TOL * np.abs(r)
    if extra is not None:
        bound = bound + np.asarray(extra, dtype=np.float64)
    bad = diff > bound
    msg = f"{name}: normwise {normwise:.3e}, elementwise fails {int(bad.sum())}/{r.size}"
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg += "; first " + ", ".join(f"{tuple(i)}: gpu {g[tuple(i)]:.5g} ref {r[tuple(i)]:.5g}" for i in idx)
    assert normwise <= NORM_TOL and not bad.any(), msg


def sparse_bits(s):
    """(vals uint16 [rows, ldv], meta uint8 [rows, ldm]) of a Sparse24 on the host."""
    v = bits_of(s.vals)
    m = s.meta.detach().cpu().numpy()
    return v, m


def assert_bits_equal(gpu: np.ndarray, ref: np.ndarray, name: str):
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    if not np.array_equal(gpu, ref):
        bad = np.argwhere(gpu != ref)
        raise AssertionError(f"{name}: {len(bad)} of {gpu.size} differ; first at {bad[:5].tolist()} "
                             f"gpu {[int(gpu[tuple(b)]) for b in bad[:5]]} ref {[int(ref[tuple(b)]) for b in bad[:5]]}")


def ulp_bf16(bits: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at each value (fp32 array): two round-to-nearest
    results of nearly equal fp32 values differ by at most this much."""
    e = ((np.asarray(bits, np.uint16) >> 7) & 0xFF).astype(np.int32)
    return np.ldexp(np.float32(1.0), np.maximum(e, 1) - 127 - 7).astype(np.float32)


def propagated(a_sq: np.ndarray, b_sq: np.ndarray) -> np.ndarray:
    """4 * sqrt(a_sq @ b_sq): four standard deviations of a sum whose terms each
    carry an independent rounding difference of one bf16 ulp of an intermediate
    (a_sq, b_sq: squared factors, one of them the squared ulps)."""
    return 4.0 * np.sqrt(np.maximum(np.matmul(a_sq.astype(np.float32), b_sq.astype(np.float32)), 0.0))
