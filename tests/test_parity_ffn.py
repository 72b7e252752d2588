"""GPU parity of the whole FFN training step (ffn24_step) against the oracle.

The oracle runs independently on the same seeded inputs; it is never fed a
GPU result. Two decisions in the step are taken on rounded values (the ReLU
gate on bf16 H, and with 2:4 activations the activation pick on bf16 H); where
the GPU's and the oracle's fp32 sums differ by rounding (a pre-activation
within rounding of 0, two magnitudes within rounding of each other), either
decision is correct. Every such position is located and validated as a
near-zero / near-tie case; only those elements of H and dH are left out of
their elementwise checks. No token row or hidden unit is dropped: outputs
computed from H or dH (Y, dX, dW_up, dW_down, db_up) are checked everywhere,
with the exact propagated difference of the two sides' bf16 operand added to
the elementwise bound (see tests/p24_testutil.py).
"""
import numpy as np
import pytest
import torch

from oracle import prune24_oracle as O
from synth24 import WORKLOADS, FFNWorkload, ffn_inputs, normal_bf16
from tests.conftest import bits_of
from tests.p24_testutil import (assert_bits_equal, assert_close, chained, delta_csr, propagated, sparse_bits,
                                ulp_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import semi_structured_sparse_prune24_gb300 as P
    return P


def run_gpu(P, inp, act24, adapters=None, vnm=None):
    M, ffn = inp["X"].shape[0], inp["W_up"].shape[0]
    dH = torch.empty((M, ffn), dtype=torch.bfloat16, device="cuda")
    o = P.ffn24_step(inp["X"], inp["W_up"], inp["b_up"], inp["W_down"], inp["b_down"], inp["dY"], act24=act24,
                     adapters=adapters, out={"dH": dH}, vnm=vnm)
    if vnm is not None:
        # the step's H before its V:2:M prune: the same deterministic up-forward kernel
        o["H_pre"] = P.spmm24_fwd(inp["X"], P.prune24_compress(inp["W_up"]), bias=inp["b_up"], relu=True)
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    return o


def act_flip_groups(Hg_bits, ref, ffn, scale, slack=None):
    """[M, ffn/4] bool: activation groups whose GPU 2:4 pick differs from the oracle's.
    Each must be a near-tie: the two picks keep magnitudes equal up to bf16 rounding,
    or differ by a value within rounding of 0 (a ReLU-gate decision on a pre-activation
    near 0, judged like the gate flips below: at most 1e-3 * rms(H))."""
    mg = O.mask_from_meta(O.compress24(Hg_bits)[1], ffn)
    mr = O.mask_from_meta(ref["Hs_meta"], ffn)
    diff = (mg != mr).reshape(mg.shape[0], -1, 4).any(-1)
    for m, g in zip(*np.nonzero(diff)):
        h = np.abs(ref["H_ref"][m, 4 * g:4 * g + 4])
        kept_r = h[mr[m, 4 * g:4 * g + 4]]
        kept_g = h[mg[m, 4 * g:4 * g + 4]]
        extra = 0.0 if slack is None else float(np.max(slack[m, 4 * g:4 * g + 4]))
        assert np.allclose(np.sort(kept_r), np.sort(kept_g), rtol=2 ** -7, atol=1e-3 * scale + extra), (m, g, h)
    return diff


def vnm_flagged(o, ref, V: int, Mg: int, scale: float):
    """V:N:M activations: [M, ffn] bool of the block-groups whose column selection the
    GPU took differently, and the rows x groups whose 2:4 pick among the selected
    columns differs, each validated as a decision on rounded values:
      - selection: a column the GPU kept and the oracle did not, against one the oracle
        kept and the GPU did not, must score equal (the oracle's fp32 L1 norms over the
        block) within the two sides' pre-prune H difference summed over the block (the
        GPU's pre-prune H comes from the same deterministic up-forward kernel) plus the
        fp32 rounding of two sums of V terms;
      - pick: the kept nonzero magnitudes must agree up to bf16 rounding, or differ by a
        value within rounding of 0 (a ReLU-gate decision), as for 2:4 activations.
    Returns (mask, number of flagged block-groups)."""
    from oracle import vnm_oracle as VNM
    Hg = bits_of(o["H"])
    Hpre = bits_of(o["H_pre"])
    Hr = ref["H"]
    M, ffn = Hg.shape
    G, nb = ffn // Mg, (M + V - 1) // V
    scores = VNM.column_scores(Hr, V, Mg).astype(np.float64)                    # [nb, ffn]
    dpre = np.abs(O.bf16_to_f32(Hpre).astype(np.float64) - O.bf16_to_f32(Hr))
    slack = np.add.reduceat(dpre, np.arange(0, M, V), axis=0)                    # [nb, ffn]
    rounding = 2 * V * 2.0 ** -24 * scores.max(axis=1, keepdims=True)
    nzg = (Hg & np.uint16(0x7FFF)) != 0
    nzr = (ref["H_used"] & np.uint16(0x7FFF)) != 0
    sel_r = np.zeros((nb, G, Mg), bool)
    np.put_along_axis(sel_r, ref["Hv_colidx"].astype(np.int64), True, axis=2)
    used_g = np.zeros((nb, ffn), bool)
    for b in range(nb):
        used_g[b] = nzg[b * V:(b + 1) * V].any(axis=0)
    used_g = used_g.reshape(nb, G, Mg)
    flagged = np.zeros((M, ffn), bool)
    n_sel = 0
    for b, g in zip(*np.nonzero((used_g & ~sel_r).any(axis=2))):
        extra = np.nonzero(used_g[b, g] & ~sel_r[b, g])[0] + g * Mg           # GPU-kept, not oracle-selected
        lost = np.nonzero(sel_r[b, g] & ~used_g[b, g])[0] + g * Mg             # oracle-selected, unused by GPU
        for a in extra:
            gap = np.abs(scores[b, a] - scores[b, lost])
            assert np.any(gap <= slack[b, a] + slack[b, lost] + rounding[b, 0]), (b, g, a, lost, gap)
        flagged[b * V:(b + 1) * V, g * Mg:(g + 1) * Mg] = True
        n_sel += 1
    assert n_sel <= 16 + 1e-3 * nb * G, n_sel
    # picks within an agreed selection
    diff = ((nzg != nzr) & ~flagged).reshape(M, G, Mg).any(axis=2)
    for m, g in zip(*np.nonzero(diff)):
        h = np.abs(ref["H_ref"][m, g * Mg:(g + 1) * Mg])
        kept_r = np.sort(np.r_[h[nzr[m, g * Mg:(g + 1) * Mg]], 0.0, 0.0])[-2:]
        kept_g = np.sort(np.r_[h[nzg[m, g * Mg:(g + 1) * Mg]], 0.0, 0.0])[-2:]
        assert np.allclose(kept_r, kept_g, rtol=2 ** -7, atol=1e-3 * scale), (m, g, h)
        flagged[m, g * Mg:(g + 1) * Mg] = True
    return flagged, n_sel


def validated_decisions(o, ref, w: FFNWorkload, act24: bool, slack=None, vnm=None):
    """[M, ffn] bool: elements where the GPU and the oracle legitimately took a decision
    on a rounded value differently, each validated here:
      - ReLU gate [H > 0] where the pre-activation is within rounding of 0 (the
        positive side's value must be tiny), and
      - with 2:4 activations, the 4 elements of each group whose pick is a near-tie.
    slack [M, ffn] (optional): how far the two sides' pre-activations may drift apart
    before the decision (the propagated rounding of an unobserved bf16 intermediate,
    the adapters' T); it widens "within rounding of 0" and "near-tie" by that much.
    Returns (mask, number of flagged elements)."""
    Hg = O.bf16_to_f32(bits_of(o["H"]))
    Hr = O.bf16_to_f32(ref["H_used"])
    flagged = np.zeros(Hg.shape, dtype=bool)
    scale = float(np.sqrt(np.mean(ref["H_ref"].astype(np.float64) ** 2))) or 1.0
    sel_flagged = np.zeros(Hg.shape, dtype=bool)
    if act24:
        groups = act_flip_groups(bits_of(o["H"]), ref, w.ffn, scale, slack)
        flagged |= np.repeat(groups, 4, axis=1)
    if vnm is not None:
        sel_flagged, _ = vnm_flagged(o, ref, vnm[0], vnm[1], scale)
        flagged |= sel_flagged
    gate = ((Hg > 0) != (Hr > 0)) & ~flagged
    near_zero = np.maximum(Hg, Hr)[gate]
    limit = 1e-3 * scale + (0.0 if slack is None else slack[gate])
    assert np.all(near_zero <= limit), (near_zero.max(), scale)
    flagged |= gate
    n = int((flagged & ~sel_flagged).sum())
    assert n <= 16 + 1e-5 * flagged.size, n
    return flagged, int(flagged.sum())


def compare_step(o, ref, w: FFNWorkload, act24: bool, adapters: dict | None = None, vnm=None):
    """Every output, every element, against the oracle's fp32 values: H and dH (the
    step's bf16 intermediates) at the plain tolerance outside the validated decisions;
    Y, dX, dW_up, dW_down and db_up at the plain tolerance plus the exact propagated
    difference of their H / dH operand (chained). With adapters, the unobserved bf16
    products T and U add their statistical allowance (propagated)."""
    sq = lambda a: O.bf16_to_f32(a).astype(np.float32) ** 2  # noqa: E731
    var = lambda bound: (bound / 4.0) ** 2  # noqa: E731  (a propagated 4-sigma bound back to a variance)
    slack = None
    if adapters is not None:   # H's pre-activation carries T_up's rounding through L_up
        slack = propagated(ulp_bf16(ref["T_up"]) ** 2, sq(adapters["L_up"]).T)
    flagged, _ = validated_decisions(o, ref, w, act24, slack, vnm)
    absf = lambda a: np.abs(O.bf16_to_f32(a))  # noqa: E731
    Hd = delta_csr(bits_of(o["H"]), ref["H_used"])                      # [M, ffn]
    dHd = delta_csr(bits_of(o["dH"]), ref["dH"])                        # [M, ffn]
    Wd = absf(O.decompress24(ref["down_vals"], ref["down_meta"], w.ffn))       # [d, ffn]
    WubT = absf(O.decompress24(ref["upT_vals"], ref["upT_meta"], w.ffn))       # [d, ffn]
    cY = chained(Hd, Wd.T)                                              # [M, d]
    cdX = chained(dHd, WubT.T)                                          # [M, d]
    cdWu = chained(dHd.T.tocsr(), absf(ref["X"]))                       # [ffn, d]
    cdbu = np.asarray(dHd.sum(axis=0)).ravel()                          # [ffn]
    cdWd = chained(Hd.T.tocsr(), absf(ref["dY"])).T                     # [d, ffn]
    Hm = O.bf16_to_f32(ref["H_used"]) if (act24 or vnm) else ref["H_ref"]
    eH = edH = eY = edX = None
    if adapters is not None:
        L_up2, R_up2, L_dn2, R_dn2 = (sq(adapters[k]) for k in ("L_up", "R_up", "L_down", "R_down"))
        uTup2 = ulp_bf16(ref["T_up"]) ** 2                               # [M, r]
        eH = propagated(uTup2, L_up2.T)                                  # H = ReLU(... + T_up L_up^T)
        uH2 = ulp_bf16(ref["H_used"]) ** 2 + var(eH)
        uTdn2 = ulp_bf16(ref["T_down"]) ** 2 + var(propagated(uH2, R_dn2.T))   # T_dn = H R_dn^T
        uUdn2 = ulp_bf16(ref["U_down"]) ** 2                             # U_dn = dY L_dn
        edH = propagated(uUdn2, R_dn2)                                   # dH gains U_dn R_dn
        udH2 = ulp_bf16(ref["dH"]) ** 2 + var(edH)
        uUup2 = ulp_bf16(ref["U_up"]) ** 2 + var(propagated(udH2, L_up2))     # U_up = dH L_up
        eY = propagated(uTdn2, L_dn2.T)
        edX = propagated(uUup2, R_up2)
    if adapters is not None:
        # H and dH also reach Y, dX and the adapter gradients through the rank-r
        # products T_dn = H R_dn^T and U_up = dH L_up: chain their differences too
        dTdn = chained(Hd, absf(adapters["R_down"]).T)                  # [M, r], bounds |T_dn gpu - ref|
        dUup = chained(dHd, absf(adapters["L_up"]))                     # [M, r], bounds |U_up gpu - ref|
        cY = cY + dTdn @ absf(adapters["L_down"]).T.astype(np.float64)
        cdX = cdX + dUup @ absf(adapters["R_up"]).astype(np.float64)
    assert_close(o["H"], Hm, "H", skip=flagged, extra=eH)
    assert_close(o["dH"], ref["dH_ref"], "dH", skip=flagged, extra=edH)
    assert_close(o["Y"], ref["Y_ref"], "Y", chain=cY, extra=eY)
    assert_close(o["dX"], ref["dX_ref"], "dX", chain=cdX, extra=edX)
    assert_close(o["dW_up"], ref["dW_up_ref"], "dW_up", chain=cdWu)
    assert_close(o["db_up"], ref["db_up"], "db_up", chain=cdbu)
    assert_close(o["dW_down"], ref["dW_down_ref"], "dW_down", chain=cdWd)
    if adapters is not None:
        Tup2, Udn2 = (sq(ref[k]) for k in ("T_up", "U_down"))
        H2, dH2 = sq(ref["H_used"]), sq(ref["dH"])
        # the adapter gradients: H / dH differences chained exactly, T / U statistically
        assert_close(o["dL_down"], ref["dL_down_ref"], "dL_down", chain=absf(ref["dY"]).T.astype(np.float64) @ dTdn,
                     extra=propagated(sq(ref["dY"]).T, uTdn2))
        assert_close(o["dR_down"], ref["dR_down_ref"], "dR_down",
                     chain=chained(Hd.T.tocsr(), absf(ref["U_down"])).T, extra=propagated(uUdn2.T, H2))
        assert_close(o["dL_up"], ref["dL_up_ref"], "dL_up",
                     chain=chained(dHd.T.tocsr(), absf(ref["T_up"])), extra=propagated(dH2.T, uTup2))
        assert_close(o["dR_up"], ref["dR_up_ref"], "dR_up", chain=dUup.T @ absf(ref["X"]).astype(np.float64),
                     extra=propagated(uUup2.T, sq(ref["X"])))
        del Tup2, Udn2
    assert_close(o["db_down"], ref["db_down"], "db_down")
    # masked gradients are exactly zero off the forward masks
    assert np.all(bits_of(o["dW_up"])[~O.mask_from_meta(ref["up_meta"], w.d)] == 0)
    assert np.all(bits_of(o["dW_down"])[~O.mask_from_meta(ref["down_meta"], w.ffn)] == 0)


def oracle_step(inp, act24, adapters=None, vnm=None):
    r = O.ffn_step(bits_of(inp["X"]), bits_of(inp["W_up"]), inp["b_up"].cpu().numpy(), bits_of(inp["W_down"]),
                   inp["b_down"].cpu().numpy(), bits_of(inp["dY"]), act24=act24,
                   adapters=None if adapters is None else {k: bits_of(v) for k, v in adapters.items()},
                   act_vnm=vnm)
    r["X"], r["dY"] = bits_of(inp["X"]), bits_of(inp["dY"])
    return r


def integer_inputs(w: FFNWorkload, seed: int):
    """Values in {-1, 0, 1} (bias in {-2..2}): every product and partial sum of the
    step is a small integer, exact in fp32 in any order, so GPU and oracle must agree
    bit for bit on every output (bf16 roundings of identical fp32 values included)."""
    from synth24 import small_int_bf16
    dev = "cuda"
    return {
        "X": small_int_bf16((w.M, w.d), -1, 1, seed, 1, dev),
        "W_up": small_int_bf16((w.ffn, w.d), -1, 1, seed, 2, dev),
        "W_down": small_int_bf16((w.d, w.ffn), -1, 1, seed, 3, dev),
        "dY": small_int_bf16((w.M, w.d), -1, 1, seed, 6, dev),
        "b_up": small_int_bf16((w.ffn,), -2, 2, seed, 4, dev).float(),
        "b_down": small_int_bf16((w.d,), -2, 2, seed, 5, dev).float(),
    }


@pytest.mark.parametrize("act24", [False, True])
@pytest.mark.parametrize("shape", [(520, 264, 392), (4096, 768, 3072)])
def test_ffn_step_integer_inputs_bit_exact(P, shape, act24):
    M, d, ffn = shape
    w = FFNWorkload("int", M, d, ffn, 1.0)
    inp = integer_inputs(w, seed=3)
    o = run_gpu(P, inp, act24)
    ref = oracle_step(inp, act24)
    # every fp32 sum stays far below 2**24, so the exact result is order-independent
    assert np.abs(ref["dW_up_ref"]).max() < 2 ** 20 and np.abs(ref["dW_down_ref"]).max() < 2 ** 20

    assert_bits_equal(bits_of(o["H"]), ref["H_used"] if act24 else ref["H"], "H")
    assert_bits_equal(bits_of(o["Y"]), ref["Y"], "Y")
    assert_bits_equal(bits_of(o["dX"]), ref["dX"], "dX")
    assert_bits_equal(bits_of(o["dW_up"]), ref["dW_up"], "dW_up")
    assert_bits_equal(bits_of(o["dW_down"]), ref["dW_down"], "dW_down")
    assert np.array_equal(o["db_up"].cpu().numpy(), ref["db_up"])
    assert np.array_equal(o["db_down"].cpu().numpy(), ref["db_down"])


@pytest.mark.parametrize("act24", [False, True])
@pytest.mark.parametrize("shape", [(128, 512, 256), (200, 264, 392)])
def test_ffn_step_small(P, shape, act24):
    M, d, ffn = shape
    w = FFNWorkload("small", M, d, ffn, 0.05)
    inp = ffn_inputs(w, seed=11, device="cuda", bias=True)
    o = run_gpu(P, inp, act24)
    compare_step(o, oracle_step(inp, act24), w, act24)


@pytest.mark.parametrize("name,act24", [("gpt2", False), ("gpt2", True), ("1p3b", False), ("70b_tail", False)])
def test_ffn_step_workloads(P, name, act24):
    w = WORKLOADS[name]
    inp = ffn_inputs(w, seed=0, device="cuda", bias=False)
    o = run_gpu(P, inp, act24)
    compare_step(o, oracle_step(inp, act24), w, act24)


@pytest.mark.parametrize("name", ["70b_m16384", "70b_m8192", "70b_m2048", "7b_act24"])
def test_ffn_step_large_workloads_sampled(P, name):
    """The large configurations in the bench's launch configuration. Compressed and
    double-pruned weights (and W_down on its mask) are checked bit-exactly in full.
    Outputs are checked on 512 seeded token rows (H, dH, Y, dX), 512 hidden units
    (dH, dW_up, db_up) and 512 model features (dW_down, db_down), recomputed by the
    oracle from the seeded inputs alone; the oracle's full H locates and validates the
    decisions taken on rounded values. No row or unit is left out: the chained outputs
    carry the exact propagated difference of their H / dH operand."""
    w = WORKLOADS[name]
    act24 = w.act24
    inp = ffn_inputs(w, seed=0, device="cuda", bias=False)
    o = run_gpu(P, inp, act24)
    X, Wu, Wd, dY = (bits_of(inp[k]) for k in ("X", "W_up", "W_down", "dY"))
    tm = lambda a: torch.as_tensor(a, device="cuda")  # noqa: E731
    absf = lambda a: np.abs(O.bf16_to_f32(a))  # noqa: E731

    # weights: fresh masks and double prunes, bit for bit in full
    Wm = torch.empty((w.d, w.ffn), dtype=torch.bfloat16, device="cuda")
    gu, guT = P.prune24_compress_both(inp["W_up"])
    gd, gdT = P.prune24_compress_both(inp["W_down"], W_masked=Wm)
    up_v, up_m = O.compress24(Wu, gu.ldv, gu.ldm)
    dn_v, dn_m = O.compress24(Wd, gd.ldv, gd.ldm)
    upT_v, upT_m = O.double_prune(up_v, up_m, w.ffn, w.d, guT.ldv, guT.ldm)
    dnT_v, dnT_m = O.double_prune(dn_v, dn_m, w.d, w.ffn, gdT.ldv, gdT.ldm)
    for g, (rv, rm), nm in ((gu, (up_v, up_m), "W_up fwd"), (guT, (upT_v, upT_m), "W_up bwdT"),
                            (gd, (dn_v, dn_m), "W_down fwd"), (gdT, (dnT_v, dnT_m), "W_down bwdT")):
        gv, gmeta = sparse_bits(g)
        assert_bits_equal(gv, rv, nm + " vals")
        assert_bits_equal(gmeta, rm, nm + " meta")
    assert_bits_equal(bits_of(Wm), O.decompress24(dn_v, dn_m, w.ffn), "W_down on its mask")
    del gu, guT, gd, gdT, Wm

    # the oracle's full H (needed for dW_down anyway) and the validated decisions
    H_r, H_b = O.spmm24_fwd(X, up_v, up_m, w.d, relu=True)
    ref = {"H_ref": H_r, "H": H_b}
    if act24:
        ref["Hs_vals"], ref["Hs_meta"] = O.compress24(H_b)
        ref["H_used"] = O.decompress24(ref["Hs_vals"], ref["Hs_meta"], w.ffn)
    else:
        ref["H_used"] = H_b
    Hu = ref["H_used"]
    flagged, n_flag = validated_decisions(o, ref, w, act24)
    Hg = bits_of(o["H"])
    Hd = delta_csr(Hg, Hu)                                  # [M, ffn], the two sides' bf16 H
    print(f"[{w.name}] validated rounded decisions: {n_flag} elements; H differs at {Hd.nnz} of {Hg.size}; "
          "rows or units left out: 0")
    rng = np.random.default_rng(5)
    ms = np.sort(rng.choice(w.M, 512, replace=False))
    fs = (4 * np.sort(rng.choice(w.ffn // 4, 128, replace=False))[:, None] + np.arange(4)).ravel()
    ns = np.sort(rng.choice(w.d, 512, replace=False))

    # token rows: H, dH, Y, dX
    assert_close(o["H"][tm(ms)], O.bf16_to_f32(Hu[ms]) if act24 else H_r[ms], "H rows", skip=flagged[ms])
    dHr_r, dHr_b = O.spmm24_bwd_dx(dY[ms], dnT_v, dnT_m, w.d, gate=Hu[ms])
    dHg_rows = bits_of(o["dH"][tm(ms)])
    assert_close(o["dH"][tm(ms)], dHr_r, "dH rows", skip=flagged[ms])
    Y_r, _ = O.spmm24_fwd(Hu[ms], dn_v, dn_m, w.ffn)
    Wd_abs = absf(O.decompress24(dn_v, dn_m, w.ffn))                    # [d, ffn]
    assert_close(o["Y"][tm(ms)], Y_r, "Y rows", chain=chained(Hd[ms], Wd_abs.T))
    dX_r, _ = O.spmm24_bwd_dx(dHr_b, upT_v, upT_m, w.ffn)
    WubT_abs = absf(O.decompress24(upT_v, upT_m, w.ffn))                # [d, ffn]
    assert_close(o["dX"][tm(ms)], dX_r, "dX rows", chain=chained(delta_csr(dHg_rows, dHr_b), WubT_abs.T))
    del Wd_abs, WubT_abs, dHr_r, Y_r, dX_r
    # hidden units: dH[:, fs], dW_up[fs, :] and db_up[fs] over all tokens
    dHc_r, dHc_b = O.spmm24_bwd_dx(dY, dnT_v[fs], dnT_m[fs], w.d, gate=Hu[:, fs])
    assert_close(o["dH"][:, tm(fs)], dHc_r, "dH columns", skip=flagged[:, fs])
    dHdc = delta_csr(bits_of(o["dH"][:, tm(fs)]), dHc_b)               # [M, 512]
    dWu_r, _ = O.masked_dw(dHc_b, X, up_m[fs])
    assert_close(o["dW_up"][tm(fs)], dWu_r, "dW_up rows", chain=chained(dHdc.T.tocsr(), absf(X)))
    assert_close(o["db_up"][tm(fs)], O.colsum(dHc_b), "db_up entries", chain=np.asarray(dHdc.sum(axis=0)).ravel())
    del dHc_r, dHc_b, dWu_r
    # model features: dW_down[ns, :] = dY[:, ns]^T H_used on the mask, every hidden unit
    dWd_r, _ = O.masked_dw(dY[:, ns], Hu, dn_m[ns])
    assert_close(o["dW_down"][tm(ns)], dWd_r, "dW_down rows", chain=chained(Hd.T.tocsr(), absf(dY[:, ns])).T)
    assert_close(o["db_down"][tm(ns)], O.colsum(dY[:, ns]), "db_down entries")


def oracle_weights(P, W_up_bits, W_down_bits, ffn, d, device="cuda"):
    """Compressed weights and W_down on its mask, computed by the oracle and uploaded
    into the binding's buffers."""
    from tests.conftest import from_bits
    bufs = {"up_fwd": P.Sparse24.empty(ffn, d, device), "up_bwdT": P.Sparse24.empty(d, ffn, device),
            "down_fwd": P.Sparse24.empty(d, ffn, device), "down_bwdT": P.Sparse24.empty(ffn, d, device)}
    uv, um = O.compress24(W_up_bits, bufs["up_fwd"].ldv, bufs["up_fwd"].ldm)
    dv, dm = O.compress24(W_down_bits, bufs["down_fwd"].ldv, bufs["down_fwd"].ldm)
    ref = {"up_fwd": (uv, um), "down_fwd": (dv, dm),
           "up_bwdT": O.double_prune(uv, um, ffn, d, bufs["up_bwdT"].ldv, bufs["up_bwdT"].ldm),
           "down_bwdT": O.double_prune(dv, dm, d, ffn, bufs["down_bwdT"].ldv, bufs["down_bwdT"].ldm)}
    for k, (v, m) in ref.items():
        bufs[k].vals.copy_(from_bits(v, device))
        bufs[k].meta.copy_(torch.from_numpy(m).to(device))
    bufs["W_down_masked"] = from_bits(O.decompress24(dv, dm, ffn), device)
    return bufs, ref


@pytest.mark.parametrize("act24", [False, True])
def test_ffn_step_writes_fresh_masks_to_caller_buffers(P, act24):
    """Gradual magnitude pruning with caller-owned compressed weights: the step's
    fresh masks land in the caller's buffers bit for bit, and a fixed-mask step
    reading those buffers (W_up / W_down not passed) reproduces the outputs."""
    w = FFNWorkload("small", 200, 264, 392, 0.05)
    inp = ffn_inputs(w, seed=12, device="cuda", bias=True)
    bufs = {"up_fwd": P.Sparse24.empty(w.ffn, w.d), "up_bwdT": P.Sparse24.empty(w.d, w.ffn),
            "down_fwd": P.Sparse24.empty(w.d, w.ffn), "down_bwdT": P.Sparse24.empty(w.ffn, w.d),
            "W_down_masked": torch.empty((w.d, w.ffn), dtype=torch.bfloat16, device="cuda")}
    o1 = P.ffn24_step(inp["X"], inp["W_up"], inp["b_up"], inp["W_down"], inp["b_down"], inp["dY"], act24=act24,
                      weights=bufs)
    torch.cuda.synchronize()
    _, ref = oracle_weights(P, bits_of(inp["W_up"]), bits_of(inp["W_down"]), w.ffn, w.d, device="cpu")
    for k, (rv, rm) in ref.items():
        gv, gm = sparse_bits(bufs[k])
        assert_bits_equal(gv, rv, k + " vals")
        assert_bits_equal(gm, rm, k + " meta")
    assert_bits_equal(bits_of(bufs["W_down_masked"]), O.decompress24(*ref["down_fwd"], w.ffn), "W_down_masked")
    o2 = P.ffn24_step(inp["X"], None, inp["b_up"], None, inp["b_down"], inp["dY"], act24=act24,
                      weights=bufs, keep_masks=True)
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    for k in ("H", "Y", "dX", "dW_up", "dW_down"):
        assert_bits_equal(bits_of(o2[k]), bits_of(o1[k]), k + " (fixed masks vs fresh)")
    assert torch.equal(o2["db_down"], o1["db_down"])
    torch.testing.assert_close(o2["db_up"], o1["db_up"], rtol=1e-5, atol=1e-4)   # fp32 atomics: order may differ


@pytest.mark.parametrize("act24", [False, True])
def test_ffn_step_fixed_masks_against_the_oracle(P, act24):
    """Fixed masks taken from another weight W0 (compressed by the oracle and uploaded):
    the step must compute exactly the oracle's step on W0, whatever W_up / W_down hold."""
    w = FFNWorkload("small", 200, 264, 392, 0.05)
    inp = ffn_inputs(w, seed=13, device="cuda", bias=True)
    inp0 = ffn_inputs(w, seed=14, device="cuda", bias=True)          # W0 = inp0's weights
    bufs, _ = oracle_weights(P, bits_of(inp0["W_up"]), bits_of(inp0["W_down"]), w.ffn, w.d)
    o = P.ffn24_step(inp["X"], None, inp["b_up"], None, inp["b_down"], inp["dY"], act24=act24, weights=bufs,
                     keep_masks=True, out={"dH": torch.empty((w.M, w.ffn), dtype=torch.bfloat16, device="cuda")})
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    ref_inp = dict(inp, W_up=inp0["W_up"], W_down=inp0["W_down"])
    compare_step(o, oracle_step(ref_inp, act24), w, act24)


def adapter_inputs(w: FFNWorkload, r: int, seed: int, ints: bool = False, device="cuda"):
    """SLOPE adapters for a workload: L, R ~ N(0, 0.02^2) (tensor ids 10-13), or
    integers in {-1, 0, 1} for the bit-exact test."""
    from synth24 import small_int_bf16
    shapes = {"L_up": (w.ffn, r), "R_up": (r, w.d), "L_down": (w.d, r), "R_down": (r, w.ffn)}
    out = {}
    for i, (k, shape) in enumerate(shapes.items()):
        out[k] = (small_int_bf16(shape, -1, 1, seed, 10 + i, device) if ints
                  else normal_bf16(shape, 0.02, seed, 10 + i, device))
    return out


@pytest.mark.parametrize("act24", [False, True])
def test_ffn_step_adapters_integer_inputs_bit_exact(P, act24):
    """Integer inputs and adapters: every fp32 sum of the step is an integer below
    2**24, exact in any order, so every output (adapter gradients included) must agree
    with the oracle bit for bit."""
    w = FFNWorkload("int", 256, 264, 392, 1.0)
    inp = integer_inputs(w, seed=5)
    ad = adapter_inputs(w, 64, seed=5, ints=True)
    o = run_gpu(P, inp, act24, ad)
    ref = oracle_step(inp, act24, ad)
    for k in ("H_ref", "Y_ref", "dH_ref", "dX_ref", "dW_up_ref", "dW_down_ref",
              "dL_up_ref", "dR_up_ref", "dL_down_ref", "dR_down_ref"):
        assert np.abs(ref[k]).max() < 2 ** 22, k
    assert_bits_equal(bits_of(o["H"]), ref["H_used"] if act24 else ref["H"], "H")
    for k in ("Y", "dX", "dW_up", "dW_down", "dL_up", "dR_up", "dL_down", "dR_down"):
        assert_bits_equal(bits_of(o[k]), ref[k], k)
    assert np.array_equal(o["db_up"].cpu().numpy(), ref["db_up"])
    assert np.array_equal(o["db_down"].cpu().numpy(), ref["db_down"])


@pytest.mark.parametrize("name,act24,r", [("gpt2", False, 64), ("gpt2", True, 64), ("1p3b", False, 128)])
def test_ffn_step_adapters_workloads(P, name, act24, r):
    w = WORKLOADS[name]
    inp = ffn_inputs(w, seed=0, device="cuda", bias=False)
    ad = adapter_inputs(w, r, seed=0)
    o = run_gpu(P, inp, act24, ad)
    compare_step(o, oracle_step(inp, act24, ad), w, act24, {k: bits_of(v) for k, v in ad.items()})


def test_ffn_step_70b_m2048_adapters_in_full(P):
    """The 70B FFN at M=2048 with rank-64 adapters on both linears, in the bench's
    launch configuration: the oracle runs the whole step, every output is compared."""
    w = WORKLOADS["70b_m2048"]
    inp = ffn_inputs(w, seed=0, device="cuda", bias=False)
    ad = adapter_inputs(w, 64, seed=0)
    o = run_gpu(P, inp, False, ad)
    compare_step(o, oracle_step(inp, False, ad), w, False, {k: bits_of(v) for k, v in ad.items()})


# ---------------------------------------------------------------- V:N:M activations
@pytest.mark.parametrize("shape,Mg", [((512, 256, 1024), 8), ((4096, 768, 3072), 8), ((512, 256, 2048), 16)])
def test_ffn_step_vnm_integer_inputs_bit_exact(P, shape, Mg):
    """V:N:M activations (V = 256) on integer inputs: the column scores are exact integer
    sums on both sides, so every decision and every output must agree bit for bit."""
    M, d, ffn = shape
    w = FFNWorkload("int", M, d, ffn, 1.0)
    inp = integer_inputs(w, seed=7)
    o = run_gpu(P, inp, False, vnm=(256, Mg))
    ref = oracle_step(inp, False, vnm=(256, Mg))
    assert np.abs(ref["dW_up_ref"]).max() < 2 ** 20 and np.abs(ref["dW_down_ref"]).max() < 2 ** 20
    assert_bits_equal(bits_of(o["H"]), ref["H_used"], "H (V:2:M pruned)")
    for k in ("Y", "dX", "dW_up", "dW_down"):
        assert_bits_equal(bits_of(o[k]), ref[k], k)
    assert np.array_equal(o["db_up"].cpu().numpy(), ref["db_up"])
    assert np.array_equal(o["db_down"].cpu().numpy(), ref["db_down"])


@pytest.mark.parametrize("name,Mg", [("gpt2", 8), ("1p3b", 8), ("gpt2", 16)])
def test_ffn_step_vnm_workloads(P, name, Mg):
    w = WORKLOADS[name]
    inp = ffn_inputs(w, seed=0, device="cuda", bias=True)
    o = run_gpu(P, inp, False, vnm=(256, Mg))
    compare_step(o, oracle_step(inp, False, vnm=(256, Mg)), w, False, vnm=(256, Mg))
