"""Helpers shared by the GPU parity tests: tolerance checks and conversions.

Tolerances (bf16 outputs against the oracle's fp32 values before rounding):
  normwise  ||gpu - ref||_2 / ||ref||_2 <= 5e-3
  elementwise |gpu - ref| <= 1e-2 + 1e-2 * |ref|
Masks and metadata are compared bit for bit.

Chained outputs of the training step. A GEMM whose operand is itself a bf16
result of the step (H feeds Y and dW_down; dH feeds dX, dW_up and db_up) gets
that operand from its own side: the GPU's product uses the GPU's bf16 H, the
oracle's uses the oracle's. Where the two bf16 operands differ (a rounding that
fell the other way, or a validated decision on a rounded value), the exact
products differ by at most |delta| @ |B| (triangle inequality), with delta the
difference of the two bf16 operands -- known exactly, since both are bf16. That
term (`chain`, see delta_csr / chained) is added to the elementwise bound, and the
relative part of the tolerance is taken of |ref| + chain, the largest magnitude the
GPU's own product can have (its bf16 rounding scales with that magnitude, not with
the oracle's). The term is zero wherever the two sides' operands agree. The
intermediates themselves (H, dH) are checked against the oracle at the plain
tolerance.
"""
import numpy as np
import torch

from tests.conftest import bits_of

NORM_TOL = 5e-3
ABS_TOL = 1e-2
REL_TOL = 1e-2


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_close(gpu: torch.Tensor, ref: np.ndarray, name: str, chain=None, skip=None, extra=None):
    """chain: the exact propagated difference of a bf16 operand the two sides computed
    separately (see the module docstring), added to the elementwise bound.
    skip: boolean mask of elements whose value follows a validated decision taken on a
    rounded value (checked by that validation instead); left out of the elementwise
    check, kept in the normwise one.
    extra: statistical allowance for an intermediate the test cannot observe (only the
    adapter tests use it: the bf16 rank-r products T and U stay inside the step)."""
    g = f32(gpu).astype(np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    if r.size == 0:
        return
    diff = np.abs(g - r)
    nref = np.linalg.norm(r)
    normwise = np.linalg.norm(g - r) / (nref if nref > 0 else 1.0)
    bound = ABS_TOL + REL_TOL * np.abs(r)
    if chain is not None:
        # the GPU's value is the product of its own operand, |value| <= |ref| + chain: its
        # rounding and summation-order share of the tolerance scales with that magnitude
        c = np.asarray(chain, dtype=np.float64)
        bound = bound + (1.0 + REL_TOL) * c
    if extra is not None:
        bound = bound + np.asarray(extra, dtype=np.float64)
    bad = diff > bound
    if skip is not None:
        bad &= ~np.asarray(skip, dtype=bool)
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


def delta_csr(gpu_bits: np.ndarray, ref_bits: np.ndarray):
    """|gpu - ref| of two bf16 arrays (bit patterns) as a sparse fp64 matrix. Exact:
    the difference of two bf16 values is representable in fp64."""
    from scipy.sparse import csr_matrix

    from oracle.prune24_oracle import bf16_to_f32
    g = np.asarray(gpu_bits, np.uint16)
    r = np.asarray(ref_bits, np.uint16)
    assert g.shape == r.shape
    i, j = np.nonzero(g != r)
    v = np.abs(bf16_to_f32(g[i, j]).astype(np.float64) - bf16_to_f32(r[i, j]).astype(np.float64))
    return csr_matrix((v, (i, j)), shape=g.shape)


def chained(delta, b_abs: np.ndarray) -> np.ndarray:
    """sum_j delta[i, j] * b_abs[j, k] (delta: sparse |difference| [a, b]; b_abs [b, c]
    non-negative): the largest change the operand difference can make in the product,
    by the triangle inequality. Summed in fp64."""
    if delta.nnz == 0:
        return np.zeros((delta.shape[0], b_abs.shape[1]))
    used = np.unique(delta.indices)           # only the rows of b_abs a difference touches
    return np.asarray(delta[:, used] @ np.asarray(b_abs[used], dtype=np.float64))
