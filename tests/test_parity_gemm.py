"""GPU parity of the tensor-core GEMMs against the oracle (fp32 reference values,
bf16 outputs within the stated tolerances). Sizes span several tiles in every
dimension and end on ragged tails."""
import numpy as np
import pytest
import torch

from oracle import prune24_oracle as O
from synth24 import normal_bf16, normal_f32
from tests.conftest import bits_of
from tests.p24_testutil import assert_bits_equal, assert_close, sparse_bits, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import semi_structured_sparse_prune24_gb300 as P
    return P


# (M tokens, N out features, K reduction): one tile; several tiles + ragged tails
FWD_SHAPES = [(224, 128, 64), (520, 392, 1032), (1000, 264, 8200)]


@pytest.mark.parametrize("M,N,K", FWD_SHAPES)
@pytest.mark.parametrize("bias,relu", [(False, False), (True, True)])
def test_spmm24_fwd(P, M, N, K, bias, relu):
    X = normal_bf16((M, K), 1.0, 1, 1, "cuda")
    W = normal_bf16((N, K), 0.02, 1, 2, "cuda")
    b = normal_f32((N,), 0.1, 1, 4, "cuda") if bias else None
    Ws = P.prune24_compress(W)
    Y = P.spmm24_fwd(X, Ws, bias=b, relu=relu)
    torch.cuda.synchronize()
    vals, meta = sparse_bits(Ws)
    ref, _ = O.spmm24_fwd(bits_of(X), vals, meta, K, bias=None if b is None else b.cpu().numpy(), relu=relu)
    assert_close(Y, ref, "Y")


@pytest.mark.parametrize("M,N,K", [(224, 128, 64), (520, 392, 1032)])
def test_spmm24_fwd_act24(P, M, N, K):
    X = normal_bf16((M, K), 1.0, 2, 1, "cuda")
    W = normal_bf16((N, K), 0.02, 2, 2, "cuda")
    b = normal_f32((N,), 0.1, 2, 4, "cuda")
    Ws = P.prune24_compress(W)
    Y, Y24 = P.spmm24_fwd(X, Ws, bias=b, relu=True, act24=True)
    torch.cuda.synchronize()
    vals, meta = sparse_bits(Ws)
    ref, _ = O.spmm24_fwd(bits_of(X), vals, meta, K, bias=b.cpu().numpy(), relu=True)
    Yb = bits_of(Y)
    # the compressed activation is exactly the 2:4 prune of the GPU's own bf16 output
    hv, hm = sparse_bits(Y24)
    rv, rm = O.compress24(Yb, Y24.ldv, Y24.ldm)
    assert_bits_equal(hv, rv, "Y24 vals")
    assert_bits_equal(hm, rm, "Y24 meta")
    # Y is dense-masked: equal to the decompressed Y24, and within tolerance of the
    # oracle on the positions the mask keeps (a near-tie may pick differently there)
    assert_bits_equal(Yb, O.decompress24(rv, rm, N), "Y == decompress(Y24)")
    mask = O.mask_from_meta(rm, N)
    assert_close(torch.from_numpy(np.where(mask, O.bf16_to_f32(Yb), 0)),
                 np.where(mask, ref, 0), "Y on its mask")
    flips = int((mask != O.mask_from_meta(O.compress24(O.f32_to_bf16(ref))[1], N)).sum())
    assert flips <= max(4, mask.size // 1000), flips


# (520, 4104, 392): 33 K-blocks along N, so the gated tile drains its accumulator before
# the stores (the shorter cases keep it); ragged in every direction.
@pytest.mark.parametrize("M,N,K", [(224, 128, 128), (520, 392, 1032), (1000, 28672 // 64, 8200), (520, 4104, 392)])
@pytest.mark.parametrize("gated", [False, True])
def test_spmm24_bwd_dx(P, M, N, K, gated):
    """dX [M, K] = dY [M, N] . W_bwd, W_bwd^T [K, N] double-pruned along N."""
    W = normal_bf16((N, K), 0.02, 3, 2, "cuda")
    dY = normal_bf16((M, N), 1.0, 3, 6, "cuda")
    fwd, bwdT = P.prune24_compress_both(W)
    gate = torch.relu(normal_bf16((M, K), 1.0, 3, 7, "cuda")) if gated else None
    dbias = torch.full((K,), 7.0, dtype=torch.float32, device="cuda")   # overwritten, not accumulated into
    dX = P.spmm24_bwd_dx(dY, bwdT, gate=gate, dbias=dbias)
    torch.cuda.synchronize()
    tv, tm = sparse_bits(bwdT)
    ref, ref_b = O.spmm24_bwd_dx(bits_of(dY), tv, tm, N, gate=None if gate is None else bits_of(gate))
    assert_close(dX, ref, "dX")
    # fused bias gradient: the column sums of the stored bf16 dX (fp32 atomics, any order) ...
    g = O.bf16_to_f32(bits_of(dX)).astype(np.float64)
    db = dbias.cpu().numpy().astype(np.float64)
    # recursive fp32 summation: |error| <= (additions on the longest path) * 2^-24 * sum |x|;
    # a lane adds <= 32 values, 8 lanes are combined in 3 steps, then one atomic per tile
    fp32_bound = (32 + 3 + M / 128 + 2) * 2.0 ** -24 * np.abs(g).sum(0) + 1e-30
    assert np.all(np.abs(db - g.sum(0)) <= fp32_bound), np.abs(db - g.sum(0)).max()
    # ... and against the oracle's column sums, within the propagated bf16 rounding of dX
    assert_close(dbias, O.colsum(ref_b), "dbias", 4 * np.sqrt((ulp_bf16(ref_b) ** 2).sum(0)))


def test_spmm24_bwd_dx_empty_tokens_zeroes_dbias(P):
    W = normal_bf16((64, 128), 0.02, 3, 2, "cuda")
    _, bwdT = P.prune24_compress_both(W)
    dbias = torch.full((128,), 3.0, dtype=torch.float32, device="cuda")
    P.spmm24_bwd_dx(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), bwdT, dbias=dbias)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dbias).item() == 0


@pytest.mark.parametrize("M,N,K", [(64, 128, 256), (520, 392, 1032), (1000, 264, 8200)])
def test_masked_dw_gemm(P, M, N, K):
    W = normal_bf16((N, K), 0.02, 4, 2, "cuda")
    dY = normal_bf16((M, N), 1.0, 4, 6, "cuda")
    X = normal_bf16((M, K), 1.0, 4, 1, "cuda")
    Ws = P.prune24_compress(W)
    dW = P.masked_dw_gemm(dY, X, Ws)
    torch.cuda.synchronize()
    _, meta = sparse_bits(Ws)
    ref, _ = O.masked_dw(bits_of(dY), bits_of(X), meta)
    assert_close(dW, ref, "dW")
    off = ~O.mask_from_meta(meta, K)
    assert np.all(bits_of(dW)[off] == 0)


@pytest.mark.parametrize("M,N,K", [(128, 224, 64), (520, 392, 1032)])
def test_spmm24_fwd_sparse_act(P, M, N, K):
    H = torch.relu(normal_bf16((M, K), 1.0, 5, 1, "cuda"))
    W = normal_bf16((N, K), 0.02, 5, 3, "cuda")
    b = normal_f32((N,), 0.1, 5, 5, "cuda")
    Hs = P.prune24_compress(H)
    Ws = P.prune24_compress(W)
    Wm = torch.empty_like(W)
    P.prune24_compress(W, P.Sparse24.empty(N, K), W_masked=Wm)
    Y = P.spmm24_fwd_sparse_act(Hs, Wm, bias=b)
    torch.cuda.synchronize()
    hv, hm = sparse_bits(Hs)
    Hd = O.decompress24(hv, hm, K)
    vals, meta = sparse_bits(Ws)
    ref, _ = O.spmm24_fwd(Hd, vals, meta, K, bias=b.cpu().numpy())
    assert_close(Y, ref, "Y")


@pytest.mark.parametrize("M,N", [(1, 8), (1000, 392), (4096, 3072)])
def test_colsum(P, M, N):
    G = normal_bf16((M, N), 1.0, 6, 6, "cuda")
    out = P.p24_colsum(G)
    again = P.p24_colsum(G)
    torch.cuda.synchronize()
    ref = O.colsum(bits_of(G))
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=1e-4, atol=1e-3 * np.sqrt(M))
    assert torch.equal(out, again)            # fixed summation order


def test_status_word_is_clear(P):
    assert P.p24_query_status() == 0
