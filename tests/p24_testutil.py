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


def assert_close(gpu: torch.Tensor, ref: np.ndarray, name: str):
    g = f32(gpu).astype(np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    if r.size == 0:
        return
    diff = np.abs(g - r)
    nref = np.linalg.norm(r)
    normwise = np.linalg.norm(g - r) / (nref if nref > 0 else 1.0)
    bad = diff > ABS_TOL + REL_TOL * np.abs(r)
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
