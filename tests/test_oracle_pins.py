"""Pins of the CPU oracle against things other than itself (CPU only).

Each check ties an oracle function to something independent of its code:
brute-force enumeration, hand-worked fixtures in tests/golden/, closed forms,
invariants the method guarantees, or an independent library routine (torch's
bf16 conversion). A few tests plant a plausible mistake in the oracle and show
that a pin catches it.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import prune24_oracle as O
from tests.conftest import bits_of


def bf(x):
    """float -> bf16 bits via torch (inputs for the tests only)."""
    return bits_of(torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_widen_then_round_is_identity():
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    back = O.f32_to_bf16(O.bf16_to_f32(allbits))
    nan = (allbits & 0x7FFF) > 0x7F80
    assert np.array_equal(back[~nan], allbits[~nan])
    assert np.all((back[nan] & 0x7FFF) > 0x7F80)


def test_bf16_rounding_matches_torch_conversion():
    rng = np.random.default_rng(1)
    u = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    hi = rng.integers(0, 1 << 16, size=1 << 16, dtype=np.uint64).astype(np.uint32) << 16
    ties = np.concatenate([hi | 0x8000, hi | 0x7FFF, hi | 0x8001, hi])
    u = np.concatenate([u, ties]).view(np.float32)
    ours = O.f32_to_bf16(u)
    ref = bits_of(torch.from_numpy(u.copy()).to(torch.bfloat16))
    nan = np.isnan(u)
    assert np.array_equal(ours[~nan], ref[~nan])


@pytest.mark.parametrize("f32bits,bf16bits", [
    (0x3F808000, 0x3F80),  # halfway above 1.0 -> even (down)
    (0x3F818000, 0x3F82),  # halfway above 1.0078125 -> even (up)
    (0x3F808001, 0x3F81),  # just above halfway -> up
    (0x3F807FFF, 0x3F80),  # just below halfway -> down
    (0x7F7FFFFF, 0x7F80),  # max finite rounds to inf
    (0x80000000, 0x8000),  # -0 kept
    (0x00008000, 0x0000),  # tiny subnormal tie -> even zero
])
def test_bf16_rounding_hand_cases(f32bits, bf16bits):
    x = np.array([f32bits], dtype=np.uint32).view(np.float32)
    assert int(O.f32_to_bf16(x)[0]) == bf16bits


# ---------------------------------------------------------------- the 2:4 pick
def _brute_pick(keys):
    """The unique pair {a<b} such that every kept key beats every dropped one
    (larger, or equal at a lower index). Written independently of pick2."""
    winners = []
    for a in range(4):
        for b in range(a + 1, 4):
            kept, dropped = (a, b), [e for e in range(4) if e not in (a, b)]
            if all(keys[k] > keys[e] or (keys[k] == keys[e] and k < e)
                   for k in kept for e in dropped):
                winners.append((a, b))
    assert len(winners) == 1
    return winners[0]


def test_pick2_matches_brute_force_on_all_small_patterns():
    alphabet = bf([0, 1, -1, 2, -2, 3, -3])
    specials = np.array([0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001], dtype=np.uint16)
    for sym in (alphabet, np.concatenate([alphabet[:3], specials])):
        grid = np.stack(np.meshgrid(*([np.arange(len(sym))] * 4), indexing="ij"), -1).reshape(-1, 4)
        groups = sym[grid]
        keys = O.magnitude_key(groups)
        i0, i1 = O.pick2(keys)
        for n in range(len(groups)):
            assert (int(i0[n]), int(i1[n])) == _brute_pick([int(k) for k in keys[n]])


def _load_groups(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "prune24_groups.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            w = [int(t, 16) for t in lhs.split()]
            i0, i1, nib = rhs.split()
            rows.append((w, int(i0), int(i1), int(nib, 16)))
    return rows


def test_pick_and_nibble_match_hand_worked_groups(golden_dir):
    cases = _load_groups(golden_dir)
    assert len(cases) >= 20
    W = np.array([c[0] for c in cases], dtype=np.uint16)
    vals, meta = O.compress24(W)
    for n, (w, i0, i1, nib) in enumerate(cases):
        assert int(meta[n, 0]) & 0xF == nib
        assert int(meta[n, 0]) >> 4 == O.PAD_NIBBLE
        assert list(vals[n, :2]) == [w[i0], w[i1]]


# ---------------------------------------------------------------- worked example
@pytest.fixture(scope="module")
def ex(golden_dir):
    with open(os.path.join(golden_dir, "worked_example_4x8.json")) as f:
        return json.load(f)


def test_worked_example_compress_and_double_prune(ex):
    W = bf(ex["W"])
    vals, meta = O.compress24(W)
    assert np.array_equal(O.bf16_to_f32(vals), np.array(ex["fwd_vals"], np.float32))
    assert list(meta[:, 0]) == ex["fwd_meta"]
    assert np.array_equal(O.bf16_to_f32(O.decompress24(vals, meta, 8)), np.array(ex["W_fwd"], np.float32))
    tv, tm = O.double_prune(vals, meta, 4, 8)
    assert np.array_equal(O.bf16_to_f32(tv), np.array(ex["bwdT_vals"], np.float32))
    assert list(tm[:, 0]) == ex["bwdT_meta"]
    assert np.array_equal(O.bf16_to_f32(O.decompress24(tv, tm, 4)), np.array(ex["W_bwdT"], np.float32))


def test_worked_example_gemms(ex):
    W, X, dY = bf(ex["W"]), bf(ex["X"]), bf(ex["dY"])
    vals, meta = O.compress24(W)
    tv, tm = O.double_prune(vals, meta, 4, 8)
    Yr, Y = O.spmm24_fwd(X, vals, meta, 8)
    assert np.array_equal(Yr, np.array(ex["Y"], np.float32))
    dXr, _ = O.spmm24_bwd_dx(dY, tv, tm, 4)
    assert np.array_equal(dXr, np.array(ex["dX"], np.float32))
    dWr, _ = O.masked_dw(dY, X, meta)
    assert np.array_equal(dWr, np.array(ex["dW"], np.float32))


# ---------------------------------------------------------------- invariants
def _randw(shape, seed, ints=False):
    rng = np.random.default_rng(seed)
    if ints:
        return bf(rng.integers(-2, 3, size=shape).astype(np.float32))
    return bf(rng.standard_normal(shape).astype(np.float32))


@pytest.mark.parametrize("ints", [False, True])
def test_compress_invariants(ints):
    W = _randw((37, 72), 3, ints)
    vals, meta = O.compress24(W, ldv=40, ldm=16)
    mask = O.mask_from_meta(meta, 72)
    assert np.all(mask.reshape(37, 18, 4).sum(-1) == 2)
    nib = O.nibbles(meta, 72)
    assert set(np.unique(nib).tolist()) <= O.LEGAL_NIBBLES
    assert np.array_equal(O.decompress24(vals, meta, 72), np.where(mask, W, 0).astype(np.uint16))
    assert np.all(vals[:, 36:] == 0)                      # value padding
    pad = np.concatenate([meta[:, 9:] & 0xF, meta[:, 9:] >> 4], axis=1)
    assert np.all(pad == O.PAD_NIBBLE)                    # metadata padding
    # kept magnitudes dominate dropped ones in every group
    k = O.magnitude_key(W).reshape(37, 18, 4)
    m = mask.reshape(37, 18, 4)
    assert np.all(np.where(m, k, 1 << 20).min(-1) >= np.where(~m, k, -1).max(-1))
    if not ints:
        assert np.all((O.decompress24(vals, meta, 72) & 0x7FFF != 0).reshape(37, 18, 4).sum(-1) == 2)


@pytest.mark.parametrize("ints", [False, True])
def test_double_prune_subset_and_two_per_group(ints):
    N, K = 48, 40
    W = _randw((N, K), 5, ints)
    vals, meta = O.compress24(W)
    tv, tm = O.double_prune(vals, meta, N, K)
    Wf = O.decompress24(vals, meta, K)
    WbT = O.decompress24(tv, tm, N)                      # [K, N]
    nz_f = (Wf & 0x7FFF) != 0
    nz_b = (WbT.T & 0x7FFF) != 0
    assert not np.any(nz_b & ~nz_f)                      # supp(W_bwd) within supp(W_fwd)
    assert np.all(nz_b.T.reshape(K, N // 4, 4).sum(-1) <= 2)
    # where the forward column group already has <= 2 nonzeros nothing is lost
    grp_f = nz_f.T.reshape(K, N // 4, 4).sum(-1)
    kept = (nz_b.T.reshape(K, N // 4, 4)).sum(-1)
    assert np.array_equal(np.minimum(grp_f, 2), kept)


# ---------------------------------------------------------------- GEMMs
def _brute_nt(A, B):
    """Exact rational A [M,K] . B [N,K]^T (pure Python loops, tiny sizes)."""
    M, K = A.shape
    N = B.shape[0]
    return [[sum(Fraction(float(A[m, k])) * Fraction(float(B[n, k])) for k in range(K))
             for n in range(N)] for m in range(M)]


def _fp32_bound(A, B):
    K = A.shape[1]
    return K * 2.0 ** -23 * (np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64).T) + 1e-30


def test_spmm_fwd_matches_exact_rational_product():
    X, W = _randw((3, 16), 7), _randw((8, 16), 8)
    vals, meta = O.compress24(W)
    Wd = O.bf16_to_f32(O.decompress24(vals, meta, 16))
    Xf = O.bf16_to_f32(X)
    bias = np.array([0.5, -1, 0, 2, 0.25, -0.5, 1, 3], np.float32)
    Yr, Y = O.spmm24_fwd(X, vals, meta, 16, bias=bias, relu=True)
    exact = _brute_nt(Xf, Wd)
    for m in range(3):
        for n in range(8):
            want = max(float(exact[m][n] + Fraction(float(bias[n]))), 0.0)
            assert abs(float(Yr[m, n]) - want) <= _fp32_bound(Xf, Wd)[m, n] + 2.0 ** -23 * abs(want)
    assert np.array_equal(Y, O.f32_to_bf16(Yr))


def test_bwd_dx_and_masked_dw_match_exact_rational_products():
    N, K, M = 8, 12, 5
    W, dY, X = _randw((N, K), 9), _randw((M, N), 10), _randw((M, K), 11)
    vals, meta = O.compress24(W)
    tv, tm = O.double_prune(vals, meta, N, K)
    WbT = O.bf16_to_f32(O.decompress24(tv, tm, N))          # [K, N]
    dYf, Xf = O.bf16_to_f32(dY), O.bf16_to_f32(X)
    gate = _randw((M, K), 12)
    dXr, _ = O.spmm24_bwd_dx(dY, tv, tm, N, gate=gate)
    exact = _brute_nt(dYf, WbT)
    g = O.bf16_to_f32(gate) > 0
    bnd = _fp32_bound(dYf, WbT)
    for m in range(M):
        for k in range(K):
            want = float(exact[m][k]) if g[m, k] else 0.0
            assert abs(float(dXr[m, k]) - want) <= bnd[m, k]
    dWr, _ = O.masked_dw(dY, X, meta)
    exact = _brute_nt(dYf.T.copy(), Xf.T.copy())           # [N, K]
    mask = O.mask_from_meta(meta, K)
    bnd = _fp32_bound(dYf.T, Xf.T)
    for n in range(N):
        for k in range(K):
            want = float(exact[n][k]) if mask[n, k] else 0.0
            assert abs(float(dWr[n, k]) - want) <= bnd[n, k]


def test_sparse_from_compressed_equals_dense_on_decompressed():
    M, N, K = 33, 20, 136
    X, W = _randw((M, K), 13), _randw((N, K), 14)
    vals, meta = O.compress24(W)
    Y64 = O.spmm24_fwd_from_compressed_f64(X, vals, meta, K)
    Yr, _ = O.spmm24_fwd(X, vals, meta, K)
    Wd = O.bf16_to_f32(O.decompress24(vals, meta, K))
    assert np.all(np.abs(Yr - Y64) <= _fp32_bound(O.bf16_to_f32(X), Wd))


def test_closed_forms():
    K = 64
    ones = bf(np.ones((3, K), np.float32))
    vals, meta = O.compress24(bf(np.ones((5, K), np.float32)))
    Yr, _ = O.spmm24_fwd(ones, vals, meta, K)
    assert np.all(Yr == K / 2)                               # two of every four ones survive
    W = _randw((6, K), 15)
    vals, meta = O.compress24(W)
    onehot = bf(np.eye(K, dtype=np.float32)[:10])
    Yr, _ = O.spmm24_fwd(onehot, vals, meta, K)              # row k picks column k of W_fwd
    Wd = O.bf16_to_f32(O.decompress24(vals, meta, K))
    assert np.array_equal(Yr, Wd[:, :10].T)
    G = bf(np.ones((7, 9), np.float32))
    assert np.all(O.colsum(G) == 7)
    G = _randw((31, 5), 16)
    assert np.allclose(O.colsum(G), [sum(float(v) for v in col) for col in O.bf16_to_f32(G).T], rtol=1e-6)


def test_ffn_step_composition_invariants():
    M, d, ffn = 24, 32, 48
    X, Wu, Wd, dY = _randw((M, d), 20), _randw((ffn, d), 21), _randw((d, ffn), 22), _randw((M, d), 23)
    bu = np.linspace(-0.5, 0.5, ffn).astype(np.float32)
    bd = np.linspace(-0.1, 0.1, d).astype(np.float32)
    for act24 in (False, True):
        r = O.ffn_step(X, Wu, bu, Wd, bd, dY, act24=act24)
        Hu = O.bf16_to_f32(r["H_used"])
        assert np.all(Hu >= 0)
        if act24:
            assert np.all(((r["H_used"] & 0x7FFF) != 0).reshape(M, ffn // 4, 4).sum(-1) <= 2)
        assert np.all(r["dH_ref"][Hu <= 0] == 0)
        assert np.all(r["dW_up_ref"][~O.mask_from_meta(r["up_meta"], d)] == 0)
        assert np.all(r["dW_down_ref"][~O.mask_from_meta(r["down_meta"], ffn)] == 0)
        # Y recomputed from the dense masked operands
        Wdd = O.bf16_to_f32(O.decompress24(r["down_vals"], r["down_meta"], ffn))
        assert np.allclose(r["Y_ref"], Hu @ Wdd.T + bd, rtol=1e-5, atol=1e-5)
        assert np.allclose(r["db_down"], O.bf16_to_f32(dY).sum(0), rtol=1e-5, atol=1e-5)


# ---------------------------------------------------------------- planted mistakes
def test_planted_tie_mistake_is_caught(golden_dir, monkeypatch):
    def pick2_high_ties(keys4):                         # ties to the HIGHER index
        order = np.argsort(-keys4[..., ::-1], axis=-1, kind="stable")
        top2 = np.sort(3 - order[..., :2], axis=-1)
        return top2[..., 0], top2[..., 1]
    monkeypatch.setattr(O, "pick2", pick2_high_ties)
    with pytest.raises(AssertionError):
        test_pick_and_nibble_match_hand_worked_groups(golden_dir)


def test_planted_value_order_mistake_is_caught(ex, monkeypatch):
    real = O.compress24

    def descending(W, ldv=None, ldm=None):              # kept values stored high index first
        v, m = real(W, ldv, ldm)
        v = v.copy()
        v[:, 0::2], v[:, 1::2] = v[:, 1::2].copy(), v[:, 0::2].copy()
        return v, m
    monkeypatch.setattr(O, "compress24", descending)
    with pytest.raises(AssertionError):
        test_worked_example_compress_and_double_prune(ex)


def test_planted_unmasked_dw_mistake_is_caught(ex, monkeypatch):
    monkeypatch.setattr(O, "mask_from_meta", lambda meta, cols: np.ones((meta.shape[0], cols), bool))
    with pytest.raises(AssertionError):
        test_worked_example_gemms(ex)


def test_planted_nibble_order_mistake_is_caught(ex, monkeypatch):
    real = O.compress24

    def swapped(W, ldv=None, ldm=None):                 # odd group in the LOW nibble
        v, m = real(W, ldv, ldm)
        return v, ((m >> 4) | (m << 4)).astype(np.uint8)
    monkeypatch.setattr(O, "compress24", swapped)
    with pytest.raises(AssertionError):
        test_worked_example_compress_and_double_prune(ex)


# ---------------------------------------------------------------- SLOPE adapters
def _adapter_case(seed=21, M=24, d=32, ffn=64, r=16, act24=False):
    """Integer-valued inputs (|x| <= 1 or 2): every sum below is an integer far below
    2**24 and every bf16 intermediate (T, U, H, dH) is an integer below 2**8, so the
    oracle's fp32 results are exact and can be compared with fp64 compositions."""
    ints = lambda shape, s, lo=-1, hi=2: bf(np.random.default_rng(s).integers(lo, hi, size=shape).astype(np.float32))  # noqa: E731
    X, dY = ints((M, d), seed), ints((M, d), seed + 1)
    W_up, W_dn = ints((ffn, d), seed + 2, -2, 3), ints((d, ffn), seed + 3, -2, 3)
    ad = {"L_up": ints((ffn, r), seed + 4), "R_up": ints((r, d), seed + 5),
          "L_down": ints((d, r), seed + 6), "R_down": ints((r, ffn), seed + 7)}
    b_up = np.zeros(ffn, np.float32)
    b_dn = np.zeros(d, np.float32)
    out = O.ffn_step(X, W_up, b_up, W_dn, b_dn, dY, act24=act24, adapters=ad)
    f = lambda a: O.bf16_to_f32(a).astype(np.float64)  # noqa: E731
    return out, ad, f, X, dY, ffn, d


@pytest.mark.parametrize("act24", [False, True])
def test_adapter_forward_is_sparse_plus_low_rank(act24):
    """[SLOPE] each linear is the pruned weight plus the rank-r product L R:
    X W_s^T + (X R^T) L^T == X (W_s + L R)^T, exactly."""
    o, ad, f, X, dY, ffn, d = _adapter_case(act24=act24)
    assert np.abs(f(o["T_up"])).max() < 256 and np.abs(f(o["H"])).max() < 256   # exact in bf16
    Wu = f(O.decompress24(o["up_vals"], o["up_meta"], d)) + f(ad["L_up"]) @ f(ad["R_up"])
    assert np.array_equal(o["H_ref"].astype(np.float64), np.maximum(f(X) @ Wu.T, 0))
    Wd = f(O.decompress24(o["down_vals"], o["down_meta"], ffn)) + f(ad["L_down"]) @ f(ad["R_down"])
    assert np.array_equal(o["Y_ref"].astype(np.float64), f(o["H_used"]) @ Wd.T)


def test_adapter_input_gradients_compose():
    """dH = (dY (W_down_bwd + L_down R_down)) * [H > 0] and dX = dH (W_up_bwd + L_up R_up):
    the double-pruned sparse weight plus the exact adapter, exactly."""
    o, ad, f, X, dY, ffn, d = _adapter_case()
    Wdb = f(O.decompress24(o["downT_vals"], o["downT_meta"], d)).T + f(ad["L_down"]) @ f(ad["R_down"])
    dH = (f(dY) @ Wdb) * (f(o["H_used"]) > 0)
    assert np.array_equal(o["dH_ref"].astype(np.float64), dH)
    Wub = f(O.decompress24(o["upT_vals"], o["upT_meta"], ffn)).T + f(ad["L_up"]) @ f(ad["R_up"])
    assert np.array_equal(o["dX_ref"].astype(np.float64), f(o["dH"]) @ Wub)


def _adjoint_residuals(o, ad, f, X, dY):
    """Each adapter gradient G of a parameter P must satisfy the defining identity of a
    gradient of the bilinear loss sum(G_out * out): sum(G_out * out[P'']) == sum(G * P'')
    for any direction P'' (here a random integer one), with out[P''] the output the
    linear produces when P is replaced by P''."""
    rng = np.random.default_rng(99)
    res = {}
    H, dH = f(o["H_used"]), f(o["dH"])
    # down linear: Y += T_down L_down^T, T_down = H R_down^T; upstream gradient dY
    Lp = rng.integers(-2, 3, size=ad["L_down"].shape).astype(np.float64)
    res["dL_down"] = np.sum(f(dY) * (f(o["T_down"]) @ Lp.T)) - np.sum(o["dL_down_ref"].astype(np.float64) * Lp)
    Rp = rng.integers(-2, 3, size=ad["R_down"].shape).astype(np.float64)
    res["dR_down"] = np.sum(f(dY) * ((H @ Rp.T) @ f(ad["L_down"]).T)) - np.sum(o["dR_down_ref"].astype(np.float64) * Rp)
    # up linear: pre-activation += T_up L_up^T, T_up = X R_up^T; upstream gradient dH
    Lp = rng.integers(-2, 3, size=ad["L_up"].shape).astype(np.float64)
    res["dL_up"] = np.sum(dH * (f(o["T_up"]) @ Lp.T)) - np.sum(o["dL_up_ref"].astype(np.float64) * Lp)
    Rp = rng.integers(-2, 3, size=ad["R_up"].shape).astype(np.float64)
    res["dR_up"] = np.sum(dH * ((f(X) @ Rp.T) @ f(ad["L_up"]).T)) - np.sum(o["dR_up_ref"].astype(np.float64) * Rp)
    return res


def test_adapter_weight_gradients_satisfy_their_adjoint_identities():
    """On the exact fp32 gradients (integers below 2**24; their bf16 rounding is pinned
    with the other roundings); the intermediates they use are exact in bf16."""
    o, ad, f, X, dY, _, _ = _adapter_case()
    for name in ("T_up", "T_down", "U_up", "U_down", "H_used", "dH"):
        assert np.abs(f(o[name])).max() < 256
    res = _adjoint_residuals(o, ad, f, X, dY)
    assert all(v == 0 for v in res.values()), res
    for name in ("dL_down", "dR_down", "dL_up", "dR_up"):
        assert np.array_equal(o[name], O.f32_to_bf16(o[name + "_ref"]))


def test_planted_adapter_gradient_mistake_is_caught(monkeypatch):
    """dR computed with its operands' roles swapped (X^T U instead of U^T X, shaped
    back to [r, K]) must fail the adjoint identity."""
    real = O.dense_tn

    def swapped(A, B):
        C_ref, C = real(A, B)
        if A.shape[1] < B.shape[1]:                          # the dR products: [r, K]
            C_ref2, _ = real(B, A)                           # [K, r]
            C_ref = C_ref2.T.copy()[::-1].copy()             # a plausible but wrong [r, K]
            C = O.f32_to_bf16(C_ref)
        return C_ref, C
    monkeypatch.setattr(O, "dense_tn", swapped)
    o, ad, f, X, dY, _, _ = _adapter_case()
    res = _adjoint_residuals(o, ad, f, X, dY)
    assert res["dR_down"] != 0 or res["dR_up"] != 0
