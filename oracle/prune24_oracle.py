"""Reference (oracle) implementation of 2:4 sparse FFN training — TEST INFRASTRUCTURE ONLY.

Plain numpy, CPU, slow and direct. Only the test suite, the smoke check and the
bench's CPU-baseline leg use this module; the product path never does.

Sources (web pages on N:M sparse training; cited by title and section):
  [ESPLAG]  inno4scale "Success story ESPLAG", sections "Research Topic" and
            "Solution": semi-structured N:M pruning, a tailored compressed
            storage format, a sparse matrix-matrix multiply (SpMM) on Sparse
            Tensor Cores, gradual magnitude pruning (GMP), and a sparse version
            of the complete training step.
  [SLOPE]   NSF PAR award 2340011 listing, SLOPE abstract: the backward pass is
            "double-pruned" -- the transposed weight matrix is pruned again with
            N:M so that the backward GEMM is sparse too.
  [TO24]    "To 2:4 Sparsity and Beyond: Neuron-level Activation Function to
            Accelerate LLM Pre-Training", abstract: 2:4 sparsity for the weights
            of every FFN matmul, sparse activations on top.
  [SFL]     "Sparser, Faster, Lighter Transformer Language Models", section
            "Trainingsstrategie": ReLU as the FFN activation.

The pages give no formula, tie rule, bit encoding or precision. The readings
used here, each the plainest one the rest of the pages supports:
  * magnitude of a bf16 value = its 15 low bits as an unsigned integer
    (exact order of |w| for finite values and inf; NaN sorts above inf;
    +0 and -0 tie);
  * "top-2 of 4" = first two indices of a stable sort by descending magnitude,
    so ties go to the lower index;
  * metadata nibble of a group = i0 | (i1 << 2), i0 < i1; two nibbles per byte,
    even group in the low nibble; row padding = value 0 and nibble 0x4;
  * GEMMs accumulate in fp32; bias and ReLU are applied in fp32; outputs are
    rounded to bf16 with round-half-to-even;
  * ReLU'(0) = 0;
  * the weight gradient is masked by the positions the forward metadata
    selects, and bias gradients are fp32 column sums of the bf16 gradients;
  * SLOPE's low-rank adapters are read as a dense rank-r term beside each sparse
    weight, X W_s^T + (X R^T) L^T, trained with its exact gradients; the
    intermediate products X R^T and dY L are stored in bf16.

All bf16 tensors are numpy uint16 arrays of bit patterns.
"""
from __future__ import annotations

import numpy as np

# The six legal metadata nibbles: i0 | (i1 << 2) with 0 <= i0 < i1 <= 3.
LEGAL_NIBBLES = frozenset(i0 | (i1 << 2) for i0 in range(4) for i1 in range(i0 + 1, 4))
PAD_NIBBLE = 0x4  # (i0, i1) = (0, 1): the pattern an all-zero group prunes to


# ----------------------------------------------------------------------------
# bf16 <-> fp32 (IEEE 754 binary32 with the low 16 mantissa bits dropped)
# ----------------------------------------------------------------------------
def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening: a bf16 pattern is the top half of the binary32 pattern."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round binary32 to bf16, round-to-nearest, ties to even (IEEE 754 default).

    Written from the definition: keep the top 16 bits, add one unit in the last
    kept place when the dropped 16 bits exceed half, or equal half and the kept
    last bit is odd. A carry out of the mantissa correctly bumps the exponent
    (up to inf). NaN stays NaN (quiet bit set, sign kept).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    upper = u >> np.uint64(16)
    lower = u & np.uint64(0xFFFF)
    half = np.uint64(0x8000)
    round_up = (lower > half) | ((lower == half) & ((upper & np.uint64(1)) == np.uint64(1)))
    out = (upper + round_up.astype(np.uint64)) & np.uint64(0xFFFF)
    is_nan = (u & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    out = np.where(is_nan, upper | np.uint64(0x0040), out)
    return out.astype(np.uint16)


# ----------------------------------------------------------------------------
# 2:4 magnitude pruning and compression  [ESPLAG "Solution"; TO24 abstract]
# ----------------------------------------------------------------------------
def magnitude_key(bits: np.ndarray) -> np.ndarray:
    """|w| as an integer: the sign bit cleared from the bf16 pattern."""
    return (np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF)).astype(np.int32)


def pick2(keys4: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Indices (i0 < i1) of the two largest keys in each trailing group of 4.

    Definition: stable sort of the 4 positions by descending key; the first
    two positions are kept. Stability sends ties to the lower index.
    """
    order = np.argsort(-keys4, axis=-1, kind="stable")
    top2 = np.sort(order[..., :2], axis=-1)
    return top2[..., 0], top2[..., 1]


def default_ld(cols: int) -> tuple[int, int]:
    """Smallest row strides (values, metadata bytes) for a compressed row."""
    groups = cols // 4
    return cols // 2, (groups + 1) // 2


def compress24(W: np.ndarray, ldv: int | None = None, ldm: int | None = None):
    """Prune each row of W [R, C] to 2:4 along C and compress it.

    Returns (vals [R, ldv] uint16, meta [R, ldm] uint8):
      vals[r, 2g + j] = W[r, 4g + i_j]   (bits copied, ascending index order)
      nibble of group g = i0 | (i1 << 2), stored in byte g // 2, low nibble if g is even
    Values past C/2 are 0 and nibbles past C/4 are 0x4.
    """
    W = np.asarray(W, dtype=np.uint16)
    R, C = W.shape
    if C % 4:
        raise ValueError("2:4 pruning needs the pruned axis to be a multiple of 4")
    G = C // 4
    dv, dm = default_ld(C)
    ldv = dv if ldv is None else ldv
    ldm = dm if ldm is None else ldm
    if ldv < dv or ldm < dm:
        raise ValueError("row stride too small for a compressed row")
    groups = W.reshape(R, G, 4)
    i0, i1 = pick2(magnitude_key(groups))
    v0 = np.take_along_axis(groups, i0[..., None], axis=-1)[..., 0]
    v1 = np.take_along_axis(groups, i1[..., None], axis=-1)[..., 0]
    vals = np.zeros((R, ldv), dtype=np.uint16)
    vals[:, 0:2 * G:2] = v0
    vals[:, 1:2 * G:2] = v1
    nib = np.full((R, 2 * ldm), PAD_NIBBLE, dtype=np.uint8)
    nib[:, :G] = (i0 | (i1 << 2)).astype(np.uint8)
    meta = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return vals, meta


def nibbles(meta: np.ndarray, cols: int) -> np.ndarray:
    """Unpack the per-group nibbles [R, C/4] of a metadata array."""
    meta = np.asarray(meta, dtype=np.uint8)
    G = cols // 4
    nib = np.empty((meta.shape[0], 2 * meta.shape[1]), dtype=np.uint8)
    nib[:, 0::2] = meta & 0xF
    nib[:, 1::2] = meta >> 4
    return nib[:, :G]


def mask_from_meta(meta: np.ndarray, cols: int) -> np.ndarray:
    """Boolean [R, C]: True at the two positions each group's nibble selects."""
    nib = nibbles(meta, cols).astype(np.int64)
    R, G = nib.shape
    mask = np.zeros((R, G, 4), dtype=bool)
    rows = np.arange(R)[:, None]
    grp = np.arange(G)[None, :]
    mask[rows, grp, nib & 3] = True
    mask[rows, grp, (nib >> 2) & 3] = True
    return mask.reshape(R, cols)


def decompress24(vals: np.ndarray, meta: np.ndarray, cols: int) -> np.ndarray:
    """Scatter the compressed values back: dense [R, C] with zeros off-mask."""
    vals = np.asarray(vals, dtype=np.uint16)
    nib = nibbles(meta, cols).astype(np.int64)
    R, G = nib.shape
    dense = np.zeros((R, G, 4), dtype=np.uint16)
    rows = np.arange(R)[:, None]
    grp = np.arange(G)[None, :]
    dense[rows, grp, nib & 3] = vals[:, 0:2 * G:2]
    dense[rows, grp, (nib >> 2) & 3] = vals[:, 1:2 * G:2]
    return dense.reshape(R, cols)


def double_prune(vals: np.ndarray, meta: np.ndarray, rows: int, cols: int,
                 ldv: int | None = None, ldm: int | None = None):
    """[SLOPE abstract] prune the transposed, already-pruned weight again with 2:4.

    W_fwd = decompress(vals, meta) is [N=rows, K=cols], 2:4 along K. Its
    transpose [K, N] is pruned 2:4 along N with the same rule and compressed.
    Returns (vals_t [K, ldv] uint16, meta_t [K, ldm] uint8) = W_bwd^T compressed.
    """
    if rows % 4:
        raise ValueError("the double prune needs the row count to be a multiple of 4")
    Wf = decompress24(vals, meta, cols)
    return compress24(np.ascontiguousarray(Wf.T), ldv, ldm)


# ----------------------------------------------------------------------------
# GEMMs on the pruned operands, fp32 accumulation  [ESPLAG "Research Topic"]
# ----------------------------------------------------------------------------
def matmul_nt_f32(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """A [M, K] times B [N, K] transposed, fp32 inputs and fp32 accumulation."""
    return np.matmul(np.asarray(A, np.float32), np.asarray(B, np.float32).T)


def relu_f32(x: np.ndarray) -> np.ndarray:
    """max(x, 0) in fp32; [SFL "Trainingsstrategie"]: ReLU is the FFN activation."""
    return np.where(x > 0, x, np.float32(0)).astype(np.float32)


def spmm24_fwd(X: np.ndarray, vals: np.ndarray, meta: np.ndarray, K: int,
               bias: np.ndarray | None = None, relu: bool = False, adapter=None):
    """Y = act(X . W^T + bias) with W given compressed 2:4 along K.

    X [M, K] bf16 bits; vals/meta the compressed W [N, K]; bias fp32 [N].
    adapter (optional): (T, L), bf16 bits T = X R^T [M, r] and L [N, r]; the
    low-rank term T . L^T joins the sum before bias and activation [SLOPE].
    Returns (Y_ref fp32 before rounding, Y bf16 bits).
    """
    W = decompress24(vals, meta, K)
    Y = matmul_nt_f32(bf16_to_f32(X), bf16_to_f32(W))
    if adapter is not None:
        T, L = adapter
        Y = (Y + matmul_nt_f32(bf16_to_f32(T), bf16_to_f32(L))).astype(np.float32)
    if bias is not None:
        Y = (Y + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
    if relu:
        Y = relu_f32(Y)
    return Y, f32_to_bf16(Y)


def spmm24_bwd_dx(dY: np.ndarray, vals_t: np.ndarray, meta_t: np.ndarray, N: int,
                  gate: np.ndarray | None = None, adapter=None):
    """dX = dY . W_bwd, with W_bwd^T [K, N] given compressed 2:4 along N  [SLOPE].

    gate (optional, bf16 bits [M, K]): the forward ReLU output; dX is zeroed
    where gate <= 0 (ReLU'(0) = 0).
    adapter (optional): (U, R), bf16 bits U = dY L [M, r] and R [r, K]; the
    adapter's input gradient U . R joins the sum before the gate [SLOPE].
    Returns (dX_ref fp32, dX bf16 bits).
    """
    WbT = decompress24(vals_t, meta_t, N)            # [K, N]
    dX = matmul_nt_f32(bf16_to_f32(dY), bf16_to_f32(WbT))
    if adapter is not None:
        U, R = adapter
        dX = (dX + np.matmul(bf16_to_f32(U), bf16_to_f32(R))).astype(np.float32)
    if gate is not None:
        dX = np.where(bf16_to_f32(gate) > 0, dX, np.float32(0)).astype(np.float32)
    return dX, f32_to_bf16(dX)


def masked_dw(dY: np.ndarray, X: np.ndarray, meta_fwd: np.ndarray):
    """dW = (dY^T . X) masked to the forward 2:4 mask of W.

    dY [M, N], X [M, K] bf16 bits; meta_fwd the metadata of W [N, K].
    The contraction runs over M, fp32 accumulation. Off-mask entries are 0.
    Returns (dW_ref fp32 [N, K], dW bf16 bits).
    """
    K = X.shape[1]
    dW = np.matmul(bf16_to_f32(dY).T, bf16_to_f32(X)).astype(np.float32)
    dW = np.where(mask_from_meta(meta_fwd, K), dW, np.float32(0)).astype(np.float32)
    return dW, f32_to_bf16(dW)


def colsum(G: np.ndarray) -> np.ndarray:
    """Bias gradient: column sums of a bf16 matrix [M, N] -> fp32 [N] (fp64 accumulation)."""
    return bf16_to_f32(G).astype(np.float64).sum(axis=0).astype(np.float32)


# ----------------------------------------------------------------------------
# The FFN training step  [ESPLAG "Research Topic"; SLOPE; TO24 abstract]
# ----------------------------------------------------------------------------
def dense_nt(A: np.ndarray, B: np.ndarray):
    """C = A . B^T for bf16 bits A [M, K], B [N, K]; fp32 accumulation.
    Returns (C_ref fp32, C bf16 bits). The low-rank products of SLOPE's
    adapters (T = X R^T, U = dY L with L stored as L^T) are of this form."""
    C = matmul_nt_f32(bf16_to_f32(A), bf16_to_f32(B))
    return C, f32_to_bf16(C)


def dense_tn(A: np.ndarray, B: np.ndarray):
    """C = A^T . B for bf16 bits A [M, N], B [M, K] (a contraction over the tokens
    M, like the weight gradient but unmasked): the adapter gradients dL and dR.
    Returns (C_ref fp32, C bf16 bits)."""
    C = np.matmul(bf16_to_f32(A).T, bf16_to_f32(B)).astype(np.float32)
    return C, f32_to_bf16(C)


def ffn_step(X, W_up, b_up, W_down, b_down, dY, act24: bool = False,
             H_override: np.ndarray | None = None, adapters: dict | None = None,
             act_vnm: tuple | None = None) -> dict:
    """One up -> ReLU -> down FFN layer, forward and backward, all matmuls 2:4.

    X [M, d], W_up [ffn, d], W_down [d, ffn], dY [M, d]: bf16 bits; biases fp32.
    Steps (names are those of the returned dict):
      prune both weights 2:4 along their reduction axis (fresh every step);
      double prune their transposes for the backward pass;
      H  = ReLU(X W_up^T + b_up) rounded to bf16;
      act24: H is pruned 2:4 along ffn -> Hs (compressed) and H_used = its dense form;
      Y  = H_used W_down^T + b_down;
      dH = (dY W_down_bwd) * [H_used > 0];  db_up = colsum(dH);  db_down = colsum(dY);
      dW_down = (dY^T H_used) on mask_down;  dX = dH W_up_bwd;  dW_up = (dH^T X) on mask_up.
    H_override replaces the computed bf16 H (to chain another implementation's H).
    adapters (optional) adds SLOPE's low-rank adapters [SLOPE abstract: "low-rank
    adapters" beside the double-pruned sparse weights], each linear becoming
    X W_s^T + (X R^T) L^T: a dict of bf16 bits L_up [ffn, r], R_up [r, d],
    L_down [d, r], R_down [r, ffn]. Then also
      T_up = X R_up^T,  T_down = H_used R_down^T          (bf16, [M, r]);
      U_down = dY L_down,  U_up = dH L_up                  (bf16, [M, r]);
      dH and dX gain U_down R_down and U_up R_up (before the gate for dH);
      dL_down = dY^T T_down,  dR_down = U_down^T H_used,
      dL_up = dH^T T_up,      dR_up = U_up^T X             (bf16).
    act_vnm (optional, V, M): V:N:M activations [TO24 abstract: v:n:m sparsity for the
    activations]: H is pruned V:2:M along ffn (oracle/vnm_oracle.py) and H_used is its
    dense form; the rest of the step is unchanged (Y = H_used W_down_pruned^T, the
    gate is [H_used > 0]).
    """
    ffn, d = W_up.shape
    out: dict = {}
    up_v, up_m = compress24(W_up)
    dn_v, dn_m = compress24(W_down)
    upT_v, upT_m = double_prune(up_v, up_m, ffn, d)
    dnT_v, dnT_m = double_prune(dn_v, dn_m, d, ffn)
    out.update(up_vals=up_v, up_meta=up_m, down_vals=dn_v, down_meta=dn_m,
               upT_vals=upT_v, upT_meta=upT_m, downT_vals=dnT_v, downT_meta=dnT_m)

    ad = adapters
    if ad is not None:
        _, T_up = dense_nt(X, ad["R_up"])
        out["T_up"] = T_up
    H_ref, H = spmm24_fwd(X, up_v, up_m, d, bias=b_up, relu=True,
                          adapter=None if ad is None else (T_up, ad["L_up"]))
    if H_override is not None:
        H = np.asarray(H_override, dtype=np.uint16)
    out.update(H_ref=H_ref, H=H)
    if act24:
        Hs_v, Hs_m = compress24(H)
        H_used = decompress24(Hs_v, Hs_m, ffn)
        out.update(Hs_vals=Hs_v, Hs_meta=Hs_m)
    elif act_vnm is not None:
        from oracle import vnm_oracle as VNM
        V, Mg = act_vnm
        Hv_c, Hv_v, Hv_m = VNM.vnm_compress(H, V, Mg)
        H_used = VNM.vnm_decompress(Hv_c, Hv_v, Hv_m, H.shape[0], ffn, V, Mg)
        out.update(Hv_colidx=Hv_c, Hv_vals=Hv_v, Hv_meta=Hv_m)
    else:
        H_used = H
    out["H_used"] = H_used

    # Y = H_used . W_down_pruned^T + b_down. With act24 the sparse operand is
    # Hs and the dense one W_down on its mask; the product is the same.
    if ad is not None:
        _, T_dn = dense_nt(H_used, ad["R_down"])
        _, U_dn = dense_nt(dY, ad["L_down"].T)
        out.update(T_down=T_dn, U_down=U_dn)
    Y_ref, Y = spmm24_fwd(H_used, dn_v, dn_m, ffn, bias=b_down, relu=False,
                          adapter=None if ad is None else (T_dn, ad["L_down"]))
    out.update(Y_ref=Y_ref, Y=Y)

    dH_ref, dH = spmm24_bwd_dx(dY, dnT_v, dnT_m, d, gate=H_used,
                               adapter=None if ad is None else (U_dn, ad["R_down"]))
    out.update(dH_ref=dH_ref, dH=dH)
    out["db_up"] = colsum(dH)
    out["db_down"] = colsum(dY)
    dWd_ref, dWd = masked_dw(dY, H_used, dn_m)
    out.update(dW_down_ref=dWd_ref, dW_down=dWd)
    if ad is not None:
        _, U_up = dense_nt(dH, ad["L_up"].T)
        out["U_up"] = U_up
    dX_ref, dX = spmm24_bwd_dx(dH, upT_v, upT_m, ffn, gate=None,
                               adapter=None if ad is None else (U_up, ad["R_up"]))
    out.update(dX_ref=dX_ref, dX=dX)
    dWu_ref, dWu = masked_dw(dH, X, up_m)
    out.update(dW_up_ref=dWu_ref, dW_up=dWu)
    if ad is not None:
        for name, (a, b) in (("dL_down", (dY, T_dn)), ("dR_down", (U_dn, H_used)),
                             ("dL_up", (dH, T_up)), ("dR_up", (U_up, X))):
            ref, bits = dense_tn(a, b)
            out[name + "_ref"], out[name] = ref, bits
    return out


# ----------------------------------------------------------------------------
# Independent formulations used only to pin the ones above
# ----------------------------------------------------------------------------
def spmm24_fwd_from_compressed_f64(X: np.ndarray, vals: np.ndarray, meta: np.ndarray, K: int):
    """Y = X . W^T computed straight from the compressed form, fp64 accumulation.

    For each group g and kept slot j, the product X[:, 4g + i_j] * vals[:, 2g + j]
    is added -- the sparse-times-dense meaning of SpMM, without decompressing.
    """
    Xf = bf16_to_f32(X).astype(np.float64)
    V = bf16_to_f32(vals).astype(np.float64)
    nib = nibbles(meta, K).astype(np.int64)
    M = Xf.shape[0]
    N = V.shape[0]
    Y = np.zeros((M, N), dtype=np.float64)
    for g in range(K // 4):
        for j, idx in enumerate((nib[:, g] & 3, (nib[:, g] >> 2) & 3)):
            cols = 4 * g + idx                       # [N] column of X used by row n
            Y += Xf[:, cols] * V[:, 2 * g + j][None, :]
    return Y
