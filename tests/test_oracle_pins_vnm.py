"""Pins of the V:2:M oracle (oracle/vnm_oracle.py) against things other than itself (CPU only).

- A hand-worked fixture (tests/golden/vnm_worked_example_4x16.json).
- The special case M = 4, where V:2:M is plain 2:4: it must equal the (separately
  pinned) 2:4 compressor for every V.
- Independent characterisations of the two decisions by counting:
  - a column is selected iff fewer than 4 columns of its group beat it (higher
    exact score, or equal score and lower column);
  - a value is kept iff fewer than 2 of the 4 selected positions beat it.
- Structural invariants.
- The product computed a second way, the way a kernel forms it (gather then 2:4).
- Planted mistakes in the oracle, each caught by a pin.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import prune24_oracle as O
from oracle import vnm_oracle as VNM
from tests.conftest import bits_of

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "vnm_worked_example_4x16.json")


def bf(x):
    """float -> bf16 bits via torch (inputs for the tests only)."""
    return bits_of(torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def ints(shape, lo, hi, seed):
    return bf(np.random.default_rng(seed).integers(lo, hi + 1, size=shape).astype(np.float32))


@pytest.fixture(scope="module")
def ex():
    with open(GOLDEN) as f:
        return json.load(f)


def test_worked_example(ex):
    V, M = ex["V"], ex["M"]
    A = bf(ex["A"])
    colidx, vals, meta = VNM.vnm_compress(A, V, M)
    assert colidx.tolist() == ex["colidx"]
    assert np.array_equal(vals, bf(ex["vals"]))
    assert meta[:, 0].tolist() == ex["meta"]
    R, C = A.shape
    assert np.array_equal(VNM.vnm_decompress(colidx, vals, meta, R, C, V, M), bf(ex["dense"]))
    Y_ref, _ = VNM.vnm_spmm(bf(ex["X"]), colidx, vals, meta, R, C, V, M)
    assert np.array_equal(Y_ref, np.array(ex["Y"], np.float32))


@pytest.mark.parametrize("V", [1, 3, 16])
def test_m4_is_plain_2to4(V):
    rng = np.random.default_rng(V)
    A = bf(rng.standard_normal((37, 64)).astype(np.float32))
    A[rng.random(A.shape) < 0.1] = 0x8000                       # signed zeros: ties
    A[0, :8] = [0x7F80, 0x7FC0, 0x0001, 0x8001, 0x3F80, 0xBF80, 0x0000, 0x7F80]
    colidx, vals, meta = VNM.vnm_compress(A, V, 4)
    assert np.all(colidx == np.arange(4, dtype=np.uint8))
    rv, rm = O.compress24(A)
    assert np.array_equal(vals, rv) and np.array_equal(meta, rm)
    assert np.array_equal(VNM.vnm_decompress(colidx, vals, meta, 37, 64, V, 4), O.decompress24(rv, rm, 64))


def _selected_by_counting(A, V, M):
    """Independent: exact integer column sums (integer-valued inputs), then
    'selected iff fewer than 4 columns beat it'."""
    Af = O.bf16_to_f32(A).astype(np.int64)
    R, C = A.shape
    out = []
    for b in range((R + V - 1) // V):
        s = np.abs(Af[b * V:(b + 1) * V]).sum(axis=0)
        blk = []
        for g in range(C // M):
            sc = s[g * M:(g + 1) * M]
            sel = [j for j in range(M)
                   if sum(1 for k in range(M) if sc[k] > sc[j] or (sc[k] == sc[j] and k < j)) < 4]
            blk.append(sel)
        out.append(blk)
    return np.array(out, dtype=np.uint8)


@pytest.mark.parametrize("V,M,R", [(1, 8, 5), (3, 8, 10), (8, 16, 20), (4, 12, 9)])
def test_column_selection_by_counting(V, M, R):
    A = ints((R, 3 * M), -2, 2, seed=V * 100 + M)              # many equal scores
    colidx, _, _ = VNM.vnm_compress(A, V, M)
    assert np.array_equal(colidx, _selected_by_counting(A, V, M))


@pytest.mark.parametrize("V,M", [(2, 8), (5, 16)])
def test_row_prune_by_counting_and_invariants(V, M):
    R, C = 13, 4 * M
    rng = np.random.default_rng(M)
    A = ints((R, C), -3, 3, seed=V + M)
    A[rng.random(A.shape) < 0.05] = 0x8000
    colidx, vals, meta = VNM.vnm_compress(A, V, M)
    dense = VNM.vnm_decompress(colidx, vals, meta, R, C, V, M)
    key = O.magnitude_key(A)
    kept = np.zeros((R, C), dtype=bool)
    kept_mask = O.mask_from_meta(meta, 4 * (C // M))                      # positions over the condensed rows
    for r in range(R):
        b = r // V
        for g in range(C // M):
            cols = [g * M + int(j) for j in colidx[b, g]]
            k4 = [key[r, c] for c in cols]
            want = [p for p in range(4) if sum(1 for q in range(4) if k4[q] > k4[p] or (k4[q] == k4[p] and q < p)) < 2]
            got = [p for p in range(4) if kept_mask[r, 4 * g + p]]
            assert got == want, (r, g)
            for p in want:
                kept[r, cols[p]] = True
    # kept values copied bit for bit, +0 everywhere else
    assert np.array_equal(dense[kept], A[kept])
    assert np.all(dense[~kept] == 0)
    # exactly 2 kept per row and group; per block and group at most 4 distinct columns used
    assert np.all(kept.reshape(R, C // M, M).sum(-1) == 2)
    for b in range((R + V - 1) // V):
        used = kept[b * V:(b + 1) * V].reshape(-1, C // M, M).any(axis=0).sum(-1)
        assert np.all(used <= 4)
    assert kept.sum() == R * C * 2 // M                         # sparsity 1 - 2/M


def test_product_equals_gathered_2to4_form():
    V, M, N, K, T = 4, 8, 22, 48, 7
    W = ints((N, K), -3, 3, seed=11)
    X = ints((T, K), -3, 3, seed=12)
    colidx, vals, meta = VNM.vnm_compress(W, V, M)
    Y_ref, _ = VNM.vnm_spmm(X, colidx, vals, meta, N, K, V, M)
    Y64 = VNM.vnm_spmm_gathered_f64(X, colidx, vals, meta, N, K, V, M)
    assert np.array_equal(Y_ref.astype(np.float64), Y64)       # small integers: both exact
    dense = O.bf16_to_f32(VNM.vnm_decompress(colidx, vals, meta, N, K, V, M)).astype(np.int64)
    assert np.array_equal(Y64, (O.bf16_to_f32(X).astype(np.int64) @ dense.T).astype(np.float64))


def test_special_scores_rank_nan_over_inf_over_finite_and_signed_zeros_tie():
    # one block of 2 rows, one group of 8: a NaN column, an inf column, finite columns, zeros
    A = np.zeros((2, 8), dtype=np.uint16)
    A[0, 6] = 0x7FC0                                            # NaN
    A[1, 5] = 0xFF80                                            # -inf
    A[0, 2] = bf([3.0])[0]
    A[1, 1] = 0x8000                                            # -0: ties with +0
    A[0, 7] = bf([1.0])[0]
    colidx, _, _ = VNM.vnm_compress(A, 2, 8)
    # ranks: col 6 (NaN) > col 5 (inf) > col 2 (3) > col 7 (1) > zeros
    assert colidx[0, 0].tolist() == [2, 5, 6, 7]
    A2 = A.copy()
    A2[0, 7] = 0
    colidx2, _, _ = VNM.vnm_compress(A2, 2, 8)
    assert colidx2[0, 0].tolist() == [0, 2, 5, 6]              # zeros tie: the lowest column (0) wins


def test_planted_mistakes_are_caught(ex, monkeypatch):
    V, M = ex["V"], ex["M"]
    A = bf(ex["A"])

    def check():
        colidx, vals, meta = VNM.vnm_compress(A, V, M)
        return colidx.tolist() == ex["colidx"] and np.array_equal(vals, bf(ex["vals"]))

    assert check()
    real = VNM.select_columns

    def ties_to_higher(scores, M_):
        nb, C = scores.shape
        keys = VNM.score_key(scores).reshape(nb, C // M_, M_)[..., ::-1]
        order = np.argsort(-keys, axis=-1, kind="stable")
        return np.sort(M_ - 1 - order[..., :4], axis=-1).astype(np.uint8)

    monkeypatch.setattr(VNM, "select_columns", ties_to_higher)
    assert not check()

    def by_column_max(A_, V_, M_):
        Af = O.bf16_to_f32(np.asarray(A_) & np.uint16(0x7FFF))
        nb = (Af.shape[0] + V_ - 1) // V_
        return np.stack([Af[b * V_:(b + 1) * V_].max(axis=0) for b in range(nb)]).astype(np.float32)

    monkeypatch.setattr(VNM, "select_columns", real)
    monkeypatch.setattr(VNM, "column_scores", by_column_max)
    assert not check()


def test_vnm_linear_on_integers_equals_the_exact_sum():
    """On small-integer inputs every fp32 partial sum is an exact integer, so
    vnm_linear(A, B) must equal the int64 product of the decompressed A with B
    (plus bias, then ReLU), whatever the summation order."""
    R, K, N, V, M = 40, 64, 24, 16, 8
    A = ints((R, K), -3, 3, 21)
    B = ints((K, N), -2, 2, 22)
    bias = np.arange(N, dtype=np.float32) - 10
    ci, v, m = VNM.vnm_compress(A, V, M)
    Ad = O.bf16_to_f32(VNM.vnm_decompress(ci, v, m, R, K, V, M)).astype(np.int64)
    exact = Ad @ O.bf16_to_f32(B).astype(np.int64) + bias.astype(np.int64)[None, :]
    Y, Yb = VNM.vnm_linear(ci, v, m, R, K, V, M, B, bias=bias, relu=True)
    assert np.array_equal(Y, np.maximum(exact, 0).astype(np.float32))
    assert np.array_equal(O.bf16_to_f32(Yb), Y)          # small integers are exact in bf16


def test_vnm_linear_is_the_transposed_gathered_product():
    """A . B against the kernel-style formulation (gather B's rows per block, 2:4 on
    the condensed operand) computed in fp64 with the roles of the operands swapped:
    (A . B)^T = B^T . A^T. Within the fp32 accumulation bound."""
    R, K, N, V, M = 48, 128, 16, 12, 16
    rng = np.random.default_rng(23)
    A = bf(rng.standard_normal((R, K)))
    B = bf(rng.standard_normal((K, N)))
    ci, v, m = VNM.vnm_compress(A, V, M)
    Y, _ = VNM.vnm_linear(ci, v, m, R, K, V, M, B)
    ref = VNM.vnm_spmm_gathered_f64(np.ascontiguousarray(B.T), ci, v, m, R, K, V, M).T
    Ad = O.bf16_to_f32(VNM.vnm_decompress(ci, v, m, R, K, V, M)).astype(np.float64)
    bound = K * 2.0 ** -24 * (np.abs(Ad) @ np.abs(O.bf16_to_f32(B).astype(np.float64)))
    assert np.all(np.abs(Y - ref) <= bound + 1e-30)


def test_vnm_linear_m4_reduces_to_the_2to4_forward():
    """At M = 4 the V:2:M operand is plain 2:4 along K, so A . B equals the pinned
    2:4 forward with the roles swapped: spmm24_fwd(B^T, 2:4 of A)^T, bit for bit
    (both accumulate the same fp32 products with numpy's matmul)."""
    R, K, N = 20, 32, 12
    rng = np.random.default_rng(24)
    A = bf(rng.standard_normal((R, K)))
    B = bf(rng.standard_normal((K, N)))
    ci, v, m = VNM.vnm_compress(A, 4, 4)
    Y, _ = VNM.vnm_linear(ci, v, m, R, K, 4, 4, B)
    v2, m2 = O.compress24(A)
    Yt, _ = O.spmm24_fwd(np.ascontiguousarray(B.T), v2, m2, K)
    np.testing.assert_allclose(Y, Yt.T, rtol=0, atol=K * 2.0 ** -24 * np.abs(Yt).max())


def _step_inputs(M, d, ffn, seed):
    rng = np.random.default_rng(seed)
    X = bf(rng.standard_normal((M, d)))
    Wu = bf(0.1 * rng.standard_normal((ffn, d)))
    Wd = bf(0.1 * rng.standard_normal((d, ffn)))
    dY = bf(rng.standard_normal((M, d)))
    return X, Wu, np.zeros(ffn, np.float32), Wd, np.zeros(d, np.float32), dY


def test_ffn_step_vnm_at_m4_is_the_act24_step():
    """V:2:4 keeps all 4 columns of every group, so the V:N:M step reduces to the 2:4
    activation step (separately pinned) on every output, bit for bit."""
    args = _step_inputs(48, 32, 64, 31)
    a = O.ffn_step(*args, act24=True)
    v = O.ffn_step(*args, act_vnm=(16, 4))
    for k in ("H_used", "Y", "dH", "dX", "dW_up", "dW_down", "db_up", "db_down"):
        assert np.array_equal(a[k], v[k]), k


def test_ffn_step_vnm_activation_structure_and_chain():
    """With V:2:8: every row keeps at most 2 values per group of 8, all inside its
    block's 4 selected columns, each equal to H's value there; the down forward is the
    plain product of that H_used (so it equals vnm_linear on the transposed weight)."""
    M, d, ffn, V, Mg = 40, 32, 64, 16, 8
    X, Wu, bu, Wd, bd, dY = _step_inputs(M, d, ffn, 32)
    r = O.ffn_step(X, Wu, bu, Wd, bd, dY, act_vnm=(V, Mg))
    Hu, H = r["H_used"], r["H"]
    nz = (Hu & np.uint16(0x7FFF)) != 0
    assert np.all(nz.reshape(M, ffn // Mg, Mg).sum(-1) <= 2)
    assert np.all(Hu[nz] == H[nz])
    sel = np.zeros((M, ffn), bool)
    for m in range(M):
        for g in range(ffn // Mg):
            sel[m, g * Mg + r["Hv_colidx"][m // V, g].astype(int)] = True
    assert not np.any(nz & ~sel)
    Wm = O.decompress24(r["down_vals"], r["down_meta"], ffn)           # W_down on its 2:4 mask
    Y, _ = VNM.vnm_linear(r["Hv_colidx"], r["Hv_vals"], r["Hv_meta"], M, ffn, V, Mg, np.ascontiguousarray(Wm.T))
    np.testing.assert_allclose(Y, r["Y_ref"], rtol=0, atol=ffn * 2.0 ** -24 * np.abs(Y).max())
