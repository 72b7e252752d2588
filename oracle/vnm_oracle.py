"""Reference (oracle) implementation of V:2:M vector-wise sparsity — TEST INFRASTRUCTURE ONLY.

Plain numpy, CPU, slow and direct. Only the test suite uses this module; no
product path imports it.

Sources (web pages on N:M sparse training; cited by title and section):
  [ESPLAG]  inno4scale "Success story ESPLAG", section "Solution": semi-structured
            N:M pruning together with a tailored compressed storage format named
            VENOM (the page's format figure is not part of its text).
  [TO24]    "To 2:4 Sparsity and Beyond: Neuron-level Activation Function to
            Accelerate LLM Pre-Training", abstract: 2:4 sparsity for the weights
            and v:n:m (Venom) sparsity for the activations, on hardware whose
            sparse tensor cores run the 2:4 pattern.

No page gives the V:N:M layout, its parameters or how the columns are chosen.
The readings used here, each the plainest one that fits "N:M on the tensor
core's 2:4 pattern with a vector-wise selection on top":
  * A [R, C] is sparse along C, its contiguous (reduction) axis. C is a multiple
    of M, and M is a multiple of 4 (M = 4 is plain 2:4).
  * Rows are taken in blocks of V (the last block may be shorter). In each block
    and each group of M consecutive columns, the same 4 columns are selected for
    every row of the block.
  * A column's score is its L1 norm within the block: the sum of |a| over the
    block's rows, top to bottom, in fp32 (exact bf16 widening, one
    round-to-nearest fp32 addition per row). Scores are ranked by their fp32 bit
    patterns read as unsigned integers, which is their numeric order for
    non-negative values and puts NaN above inf, as the 2:4 magnitude key does.
    The 4 highest scores win; ties go to the lower column.
  * Each row keeps 2 of its 4 values at the selected columns by the 2:4 rule
    (largest magnitude, ties to the lower position).
  * Storage: colidx uint8 [ceil(R/V), C/M, 4], the selected column offsets within
    each group in ascending order; and the condensed matrix A_c [R, 4C/M]
    (A_c[r, 4g + k] = A[r, gM + colidx[r // V, g, k]]) compressed with the 2:4
    format: values [R, 2C/M] and metadata nibbles over the 4 selected positions.
    Sparsity is 1 - 2/M.

All bf16 tensors are numpy uint16 arrays of bit patterns.
"""
from __future__ import annotations

import numpy as np

from oracle.prune24_oracle import bf16_to_f32, compress24, decompress24, f32_to_bf16, matmul_nt_f32


def _check_shape(C: int, M: int, V: int) -> None:
    if M < 4 or M % 4:
        raise ValueError("M must be a positive multiple of 4")
    if C % M:
        raise ValueError("the sparse axis must be a multiple of M")
    if V < 1:
        raise ValueError("V must be positive")


def column_scores(A: np.ndarray, V: int, M: int) -> np.ndarray:
    """fp32 L1 norm of every column within every row block: [ceil(R/V), C].

    The sum runs over the block's rows in order, one fp32 addition per row.
    """
    A = np.asarray(A, dtype=np.uint16)
    R, C = A.shape
    _check_shape(C, M, V)
    absf = bf16_to_f32(A & np.uint16(0x7FFF))
    nb = (R + V - 1) // V
    scores = np.zeros((nb, C), dtype=np.float32)
    for b in range(nb):
        s = np.zeros(C, dtype=np.float32)
        for r in range(b * V, min(R, (b + 1) * V)):
            s = (s + absf[r]).astype(np.float32)
        scores[b] = s
    return scores


def score_key(scores: np.ndarray) -> np.ndarray:
    """Ranking key of a non-negative fp32 score: its bit pattern as an unsigned integer.

    Every NaN maps to one key (0x7FC00000) above inf: the payload an fp32 addition
    leaves in a NaN differs between processors, so NaN scores tie with each other.
    """
    s = np.ascontiguousarray(scores, dtype=np.float32)
    key = s.view(np.uint32).astype(np.int64)
    return np.where(np.isnan(s), np.int64(0x7FC00000), key)


def select_columns(scores: np.ndarray, M: int) -> np.ndarray:
    """Offsets (ascending) of the 4 best-scoring columns of every group: [nb, C/M, 4] uint8.

    Definition: a stable sort of the M columns by descending key; the first four
    are selected. Stability sends ties to the lower column.
    """
    nb, C = scores.shape
    keys = score_key(scores).reshape(nb, C // M, M)
    order = np.argsort(-keys, axis=-1, kind="stable")
    return np.sort(order[..., :4], axis=-1).astype(np.uint8)


def condense(A: np.ndarray, colidx: np.ndarray, V: int, M: int) -> np.ndarray:
    """A_c [R, 4C/M]: each row's values at its block's selected columns, group by group."""
    A = np.asarray(A, dtype=np.uint16)
    R, C = A.shape
    G = C // M
    blk = np.arange(R) // V
    cols = (np.arange(G)[None, :, None] * M + colidx[blk].astype(np.int64))   # [R, G, 4]
    return np.take_along_axis(A, cols.reshape(R, 4 * G), axis=1)


def vnm_compress(A: np.ndarray, V: int, M: int):
    """Prune A [R, C] to V:2:M along C. Returns (colidx, vals, meta)."""
    A = np.asarray(A, dtype=np.uint16)
    colidx = select_columns(column_scores(A, V, M), M)
    vals, meta = compress24(condense(A, colidx, V, M))
    return colidx, vals, meta


def vnm_decompress(colidx: np.ndarray, vals: np.ndarray, meta: np.ndarray, R: int, C: int, V: int,
                   M: int) -> np.ndarray:
    """Dense [R, C] with the kept values at their columns and +0 elsewhere."""
    _check_shape(C, M, V)
    G = C // M
    Ac = decompress24(vals, meta, 4 * G)                                      # [R, 4G]
    blk = np.arange(R) // V
    cols = (np.arange(G)[None, :, None] * M + colidx[blk].astype(np.int64)).reshape(R, 4 * G)
    dense = np.zeros((R, C), dtype=np.uint16)
    np.put_along_axis(dense, cols, Ac, axis=1)
    return dense


def vnm_spmm(X: np.ndarray, colidx: np.ndarray, vals: np.ndarray, meta: np.ndarray, N: int, K: int,
             V: int, M: int):
    """Y = X . W^T with W [N, K] given in V:2:M form (blocks of V rows of W).

    fp32 accumulation on the decompressed operand, as for the 2:4 GEMMs.
    Returns (Y_ref fp32 before rounding, Y bf16 bits).
    """
    W = vnm_decompress(colidx, vals, meta, N, K, V, M)
    Y = matmul_nt_f32(bf16_to_f32(X), bf16_to_f32(W))
    return Y, f32_to_bf16(Y)


def vnm_spmm_gathered_f64(X: np.ndarray, colidx: np.ndarray, vals: np.ndarray, meta: np.ndarray, N: int,
                          K: int, V: int, M: int) -> np.ndarray:
    """The same product the way a kernel forms it, in fp64: for every block of V
    rows of W, gather the block's selected columns of X and multiply by the
    block's condensed 2:4 rows."""
    G = K // M
    Xf = bf16_to_f32(X).astype(np.float64)
    Wc = bf16_to_f32(decompress24(vals, meta, 4 * G)).astype(np.float64)      # [N, 4G]
    Y = np.zeros((X.shape[0], N), dtype=np.float64)
    for b in range((N + V - 1) // V):
        rows = slice(b * V, min(N, (b + 1) * V))
        cols = (np.arange(G)[:, None] * M + colidx[b].astype(np.int64)).reshape(4 * G)
        Y[:, rows] = Xf[:, cols] @ Wc[rows].T
    return Y


def vnm_linear(colidx: np.ndarray, vals: np.ndarray, meta: np.ndarray, R: int, K: int, V: int, M: int,
               B: np.ndarray, bias: np.ndarray | None = None, relu: bool = False):
    """Y = act(A . B + bias) with A [R, K] given in V:2:M form (blocks of V rows of A)
    and B [K, N] dense, bf16 bits: the V:N:M activation A feeding the next linear
    [TO24 abstract], whose weight W [N, K] is passed transposed as B.

    fp32 accumulation on the decompressed operand; bias and ReLU in fp32 (as for the
    2:4 GEMMs). Returns (Y_ref fp32 before rounding, Y bf16 bits).
    """
    A = vnm_decompress(colidx, vals, meta, R, K, V, M)
    Y = np.matmul(bf16_to_f32(A), bf16_to_f32(B)).astype(np.float32)
    if bias is not None:
        Y = (Y + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
    if relu:
        Y = np.where(Y > 0, Y, np.float32(0)).astype(np.float32)
    return Y, f32_to_bf16(Y)
