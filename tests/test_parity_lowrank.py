"""GPU parity of SLOPE's low-rank adapter pieces against the oracle: the dense
rank-r products (p24_gemm_nt, p24_gemm_tn), the transpose, and the sparse GEMMs
with the adapter term added into their accumulator (forward with bias and ReLU,
backward with the ReLU' gate and the fused bias gradient)."""
import numpy as np
import pytest
import torch

from oracle import prune24_oracle as O
from synth24 import normal_bf16
from tests.conftest import bits_of
from tests.p24_testutil import assert_bits_equal, assert_close, sparse_bits, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import semi_structured_sparse_prune24_gb300 as P
    return P


@pytest.mark.parametrize("M,N,K", [(520, 64, 1032), (1000, 128, 8200), (256, 72, 512), (300, 264, 64)])
def test_gemm_nt(P, M, N, K):
    A = normal_bf16((M, K), 1.0, 4, 1, "cuda")
    B = normal_bf16((N, K), 0.02, 4, 2, "cuda")
    C = P.p24_gemm_nt(A, B)
    torch.cuda.synchronize()
    ref, _ = O.dense_nt(bits_of(A), bits_of(B))
    assert_close(C, ref, "C = A B^T")


@pytest.mark.parametrize("M,N,K", [(1000, 264, 64), (520, 64, 1032), (128, 72, 392)])
def test_gemm_tn(P, M, N, K):
    A = normal_bf16((M, N), 1.0, 5, 1, "cuda")
    B = normal_bf16((M, K), 1.0, 5, 2, "cuda")
    C = P.p24_gemm_tn(A, B)
    torch.cuda.synchronize()
    ref, _ = O.dense_tn(bits_of(A), bits_of(B))
    assert_close(C, ref, "C = A^T B")


@pytest.mark.parametrize("rows,cols", [(72, 264), (1000, 64), (33, 40)])
def test_transpose(P, rows, cols):
    S = normal_bf16((rows, cols), 1.0, 6, 1, "cuda")
    D = P.p24_transpose(S)
    torch.cuda.synchronize()
    assert_bits_equal(bits_of(D), np.ascontiguousarray(bits_of(S).T), "transpose")


@pytest.mark.parametrize("M,N,K,r", [(520, 392, 1032, 64), (1000, 264, 8200, 128), (256, 128, 512, 72)])
def test_spmm24_fwd_lowrank(P, M, N, K, r):
    """Y = ReLU(X W^T + T L^T + b) with W 2:4-compressed: the adapter term shares the
    sparse product's fp32 accumulator."""
    W = normal_bf16((N, K), 0.02, 7, 2, "cuda")
    X = normal_bf16((M, K), 1.0, 7, 1, "cuda")
    T = normal_bf16((M, r), 1.0, 7, 8, "cuda")
    L = normal_bf16((N, r), 0.02, 7, 9, "cuda")
    b = (0.1 * torch.randn(N, generator=torch.Generator().manual_seed(7))).float().cuda()
    Ws = P.prune24_compress(W)
    Y = P.spmm24_fwd_lowrank(X, Ws, T, L, bias=b, relu=True)
    torch.cuda.synchronize()
    vals, meta = O.compress24(bits_of(W), Ws.ldv, Ws.ldm)
    ref, _ = O.spmm24_fwd(bits_of(X), vals, meta, K, bias=b.cpu().numpy(), relu=True,
                          adapter=(bits_of(T), bits_of(L)))
    assert_close(Y, ref, "Y")
    assert P.p24_query_status() == 0


@pytest.mark.parametrize("M,N,K,r", [(520, 392, 1032, 64), (1000, 264, 8200, 128)])
def test_spmm24_bwd_dx_lowrank(P, M, N, K, r):
    """dX = (dY W_bwd + U R) * [gate > 0] with W_bwd double-pruned; fused column sums."""
    W = normal_bf16((N, K), 0.02, 8, 2, "cuda")
    dY = normal_bf16((M, N), 1.0, 8, 6, "cuda")
    U = normal_bf16((M, r), 1.0, 8, 8, "cuda")
    R = normal_bf16((r, K), 0.02, 8, 9, "cuda")
    gate = torch.relu(normal_bf16((M, K), 1.0, 8, 7, "cuda"))
    _, bwdT = P.prune24_compress_both(W)
    Rt = P.p24_transpose(R)
    dbias = torch.empty(K, dtype=torch.float32, device="cuda")
    dX = P.spmm24_bwd_dx_lowrank(dY, bwdT, U, Rt, gate=gate, dbias=dbias)
    torch.cuda.synchronize()
    fv, fm = O.compress24(bits_of(W))
    tv, tm = O.double_prune(fv, fm, N, K, bwdT.ldv, bwdT.ldm)
    assert_bits_equal(sparse_bits(bwdT)[0], tv, "bwdT vals")
    ref, ref_b = O.spmm24_bwd_dx(bits_of(dY), tv, tm, N, gate=bits_of(gate), adapter=(bits_of(U), bits_of(R)))
    assert_close(dX, ref, "dX")
    assert_close(dbias, O.colsum(ref_b), "dbias", 4 * np.sqrt((ulp_bf16(ref_b) ** 2).sum(0)))
    assert P.p24_query_status() == 0


def test_lowrank_rejects_bad_rank(P):
    W = P.prune24_compress(normal_bf16((64, 128), 0.02, 9, 2, "cuda"))
    X = normal_bf16((32, 128), 1.0, 9, 1, "cuda")
    T = normal_bf16((32, 12), 1.0, 9, 8, "cuda")      # r = 12: rows of 24 bytes, not 16-byte multiples
    L = normal_bf16((64, 12), 1.0, 9, 9, "cuda")
    with pytest.raises(P.P24Error):
        P.spmm24_fwd_lowrank(X, W, T, L)
