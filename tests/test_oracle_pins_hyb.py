"""Pins of the hybrid ELL + dense-overflow oracle (oracle/hyb_oracle.py) against
things other than itself (CPU only):
- a hand-worked fixture (tests/golden/hyb_worked_example_4x8.json);
- the round trip: decompressing gives back A, with -0 read as zero in ELL rows;
- the ELL/overflow boundary: nnz == E stays ELL, nnz == E + 1 overflows;
- the hybrid -> dense product on integers equals the exact int64 product;
- the dense -> hybrid product equals per-element fp64 dot products within the fp32 bound;
- planted mistakes (descending ELL order, a strict boundary, slots in the wrong
  order), each caught by a pin."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import hyb_oracle as HY
from oracle import prune24_oracle as O
from tests.conftest import bits_of

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hyb_worked_example_4x8.json")


def bf(x):
    a = np.asarray([[float("-0.0") if v == "-0" else v for v in row] for row in x], dtype=np.float32) \
        if isinstance(x, list) else np.asarray(x, dtype=np.float32)
    return bits_of(torch.tensor(a).to(torch.bfloat16))


@pytest.fixture(scope="module")
def ex():
    with open(GOLDEN) as f:
        return json.load(f)


def check_fixture(ex):
    A = bf(ex["A"])
    h = HY.hyb_compress(A, ex["E"], ex["cap"])
    assert h["nnz"].tolist() == ex["nnz"]
    assert h["slot"].tolist() == ex["slot"]
    assert h["n_ovf"] == ex["n_ovf"]
    assert h["ovf_rows"].tolist() == ex["ovf_rows"]
    assert h["ell_cols"].tolist() == ex["ell_cols"]
    assert np.array_equal(h["ell_vals"], bf(ex["ell_vals"]))
    assert np.array_equal(h["ovf"], bf(ex["ovf"]))
    Y, _ = HY.hyb_spmm(h, bf(ex["B"]))
    assert np.array_equal(Y, np.asarray(ex["Y"], np.float32))
    S = HY.hyb_sddmm(h, bf(ex["G"]), bf(ex["B"]))
    assert np.array_equal(S["ell_ref"], np.asarray(ex["S_ell"], np.float32))
    assert np.array_equal(S["ovf_ref"], np.asarray(ex["S_ovf"], np.float32))


def test_worked_example(ex):
    check_fixture(ex)


def random_sparse(R, C, density, seed, row_boost=None):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, C)).astype(np.float32)
    keep = rng.random((R, C)) < density
    if row_boost is not None:
        keep[row_boost] = rng.random((len(row_boost), C)) < 0.5
    return bf(np.where(keep, x, 0.0))


def test_round_trip_and_boundary():
    A = random_sparse(64, 96, 0.05, 1, row_boost=[3, 17, 40])
    A[5, 7] = 0x8000                                           # -0 in an ELL row reads as +0
    E = int(np.sort(HY.nonzero_mask(A).sum(1))[-4])              # the densest ELL row sits exactly at E
    h = HY.hyb_compress(A, E, cap=8)
    back = HY.hyb_decompress(h)
    expect = np.where(HY.nonzero_mask(A) | (h["slot"][:, None] >= 0), A, 0).astype(np.uint16)
    assert np.array_equal(back, expect)
    assert np.all((h["nnz"] > E) == (h["slot"] >= 0))
    assert np.any(h["nnz"] == E) and np.all(h["slot"][h["nnz"] == E] == -1)
    rows = np.nonzero(h["slot"] >= 0)[0]
    assert h["slot"][rows].tolist() == list(range(len(rows)))    # ascending row order
    assert h["ovf_rows"][:len(rows)].tolist() == rows.tolist()
    with pytest.raises(ValueError):
        HY.hyb_decompress(HY.hyb_compress(A, E, cap=len(rows) - 1))   # beyond the capacity


def test_spmm_on_integers_is_exact():
    rng = np.random.default_rng(2)
    Af = np.where(rng.random((40, 64)) < 0.1, rng.integers(-3, 4, (40, 64)), 0).astype(np.float32)
    Af[[2, 9]] = rng.integers(-3, 4, (2, 64))
    B = rng.integers(-2, 3, (64, 12)).astype(np.float32)
    h = HY.hyb_compress(bf(Af), 8, cap=4)
    Y, Yb = HY.hyb_spmm(h, bf(B))
    exact = Af.astype(np.int64) @ B.astype(np.int64)
    assert np.array_equal(Y, exact.astype(np.float32))


def test_sddmm_equals_elementwise_dots():
    A = random_sparse(32, 48, 0.1, 3, row_boost=[5])
    rng = np.random.default_rng(4)
    G = bf(rng.standard_normal((32, 24)))
    B = bf(rng.standard_normal((48, 24)))
    h = HY.hyb_compress(A, 8, cap=32)
    assert 0 < h["n_ovf"] <= 32
    S = HY.hyb_sddmm(h, G, B)
    Gf, Bf = O.bf16_to_f32(G).astype(np.float64), O.bf16_to_f32(B).astype(np.float64)
    nz = HY.nonzero_mask(A)
    for r in range(32):
        s = h["slot"][r]
        for c in range(48):
            want = Gf[r] @ Bf[c] if nz[r, c] else 0.0
            bound = 24 * 2.0 ** -24 * (np.abs(Gf[r]) @ np.abs(Bf[c]))
            if s < 0:
                pos = np.nonzero(h["ell_cols"][r, :h["nnz"][r]] == c)[0]
                got = S["ell_ref"][r, pos[0]] if (nz[r, c] and len(pos)) else 0.0
                assert nz[r, c] == (len(pos) > 0)
            else:
                got = S["ovf_ref"][s, c]
            assert abs(got - want) <= bound + 1e-30


def test_planted_mistakes_are_caught(ex, monkeypatch):
    real = HY.hyb_compress

    def descending(A, E, cap):
        h = real(A, E, cap)
        for r in range(h["ell_cols"].shape[0]):
            k = h["nnz"][r]
            if h["slot"][r] < 0 and k > 1:
                h["ell_cols"][r, :k] = h["ell_cols"][r, :k][::-1].copy()
                h["ell_vals"][r, :k] = h["ell_vals"][r, :k][::-1].copy()
        return h

    def strict(A, E, cap):
        return real(A, E - 1, cap) | {"E": E}

    for planted in (descending, strict):
        monkeypatch.setattr(HY, "hyb_compress", planted)
        with pytest.raises(AssertionError):
            check_fixture(ex)
        monkeypatch.setattr(HY, "hyb_compress", real)
