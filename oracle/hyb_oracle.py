"""Reference (oracle) implementation of the hybrid ELL + dense-overflow activation
format and its training matmuls -- TEST INFRASTRUCTURE ONLY.

Plain numpy, CPU, slow and direct. Only the test suite and the bench's CPU legs
use this module; no product path imports it.

Source: "Sparser, Faster, Lighter Transformer Language Models", "Methodologie":
for training, the (ReLU) activations are held in a hybrid format that splits the
rows dynamically -- rows with few nonzeros go into a compact ELL matrix, rows with
many ("overflows") into a dense backup matrix -- and custom kernels perform
hybrid-to-dense and dense-to-hybrid matrix multiplications for backpropagation.

The page gives no layout, width, ordering or capacity. Readings, each the plainest
one the page supports:
  * A [R, C] (bf16 bit patterns) is read row by row. A value is nonzero when its
    magnitude bits (bits & 0x7FFF) are not 0: -0 counts as zero, as for the 2:4 key.
  * nnz[r] is the number of nonzeros of row r. Row r is an ELL row when
    nnz[r] <= E (the ELL width), else an overflow row.
  * ELL rows: ell_cols[r, :nnz[r]] are the nonzero columns in ascending order and
    ell_vals[r, :nnz[r]] their values (bits copied); the remaining slots hold column
    0 and value +0.
  * Overflow rows: numbered in ascending row order (slot[r] = 0, 1, ...); the dense
    backup ovf[slot[r]] is row r as it is (bits copied, -0 included); their ELL slots
    hold column 0 and value +0. slot[r] = -1 for ELL rows; ovf_rows[k] lists the
    overflow rows by slot. The backup has a caller-given capacity `cap`; more overflow
    rows than that is an error (ovf_rows and ovf keep the first cap).
  * hybrid -> dense:  Y = A . B with B [C, N] dense (e.g. W_down^T for the down
    projection, W_up for dX), fp32 accumulation, one rounding to bf16.
  * dense -> hybrid:  S = (G . B^T) sampled at A's nonzeros, G [R, N], B [C, N]
    (dH = (dY W_down) * [H != 0] with B = W_down^T): the same hybrid layout as A,
    values at A's nonzero positions, fp32 accumulation, one rounding; zeros
    elsewhere (ELL padding, overflow-row positions where A is zero).
"""
from __future__ import annotations

import numpy as np

from oracle.prune24_oracle import bf16_to_f32, f32_to_bf16


def nonzero_mask(A: np.ndarray) -> np.ndarray:
    return (np.asarray(A, dtype=np.uint16) & np.uint16(0x7FFF)) != 0


def hyb_compress(A: np.ndarray, E: int, cap: int) -> dict:
    """The hybrid form of A [R, C]. Returns dict(nnz int32 [R], ell_cols uint16 [R, E],
    ell_vals uint16 [R, E], slot int32 [R], ovf_rows int32 [cap], n_ovf int,
    ovf uint16 [cap, C])."""
    A = np.asarray(A, dtype=np.uint16)
    R, C = A.shape
    if E < 1 or cap < 0 or C > 65536:
        raise ValueError("E >= 1, cap >= 0 and at most 65536 columns")
    nz = nonzero_mask(A)
    nnz = nz.sum(axis=1).astype(np.int32)
    ell_cols = np.zeros((R, E), dtype=np.uint16)
    ell_vals = np.zeros((R, E), dtype=np.uint16)
    slot = np.full(R, -1, dtype=np.int32)
    ovf_rows = np.full(cap, -1, dtype=np.int32)
    ovf = np.zeros((cap, C), dtype=np.uint16)
    n_ovf = 0
    for r in range(R):
        if nnz[r] <= E:
            cols = np.nonzero(nz[r])[0]                  # ascending
            ell_cols[r, :len(cols)] = cols
            ell_vals[r, :len(cols)] = A[r, cols]
        else:
            slot[r] = n_ovf
            if n_ovf < cap:
                ovf_rows[n_ovf] = r
                ovf[n_ovf] = A[r]
            n_ovf += 1
    return {"nnz": nnz, "ell_cols": ell_cols, "ell_vals": ell_vals, "slot": slot, "ovf_rows": ovf_rows,
            "n_ovf": n_ovf, "ovf": ovf, "E": E, "cap": cap, "shape": (R, C)}


def hyb_decompress(h: dict) -> np.ndarray:
    """Dense [R, C]: ELL entries scattered to their columns, overflow rows copied back."""
    R, C = h["shape"]
    out = np.zeros((R, C), dtype=np.uint16)
    for r in range(R):
        s = h["slot"][r]
        if s < 0:
            k = h["nnz"][r]
            out[r, h["ell_cols"][r, :k].astype(np.int64)] = h["ell_vals"][r, :k]
        else:
            if s >= h["cap"]:
                raise ValueError("overflow row beyond the backup's capacity")
            out[r] = h["ovf"][s]
    return out


def hyb_spmm(h: dict, B: np.ndarray):
    """hybrid -> dense: Y = A . B with A in hybrid form [R, C], B [C, N] bf16 bits.
    fp32 accumulation on the decompressed A. Returns (Y_ref fp32, Y bf16 bits)."""
    A = hyb_decompress(h)
    Y = np.matmul(bf16_to_f32(A), bf16_to_f32(B)).astype(np.float32)
    return Y, f32_to_bf16(Y)


def hyb_sddmm(h: dict, G: np.ndarray, B: np.ndarray) -> dict:
    """dense -> hybrid: S = (G . B^T) at A's nonzero positions, in A's hybrid layout.
    G [R, N], B [C, N] bf16 bits. Returns dict(ell_ref fp32 [R, E], ell_vals bf16 bits
    [R, E], ovf_ref fp32 [cap, C], ovf bf16 bits [cap, C])."""
    R, C = h["shape"]
    E, cap = h["E"], h["cap"]
    full = np.matmul(bf16_to_f32(G), bf16_to_f32(B).T).astype(np.float32)      # [R, C], fp32
    ell = np.zeros((R, E), dtype=np.float32)
    ovf = np.zeros((cap, C), dtype=np.float32)
    for r in range(R):
        s = h["slot"][r]
        if s < 0:
            k = h["nnz"][r]
            ell[r, :k] = full[r, h["ell_cols"][r, :k].astype(np.int64)]
        elif s < cap:
            mask = nonzero_mask(h["ovf"][s])
            ovf[s] = np.where(mask, full[r], np.float32(0))
    return {"ell_ref": ell, "ell_vals": f32_to_bf16(ell), "ovf_ref": ovf, "ovf": f32_to_bf16(ovf)}
