"""GPU parity of each tensor-core GEMM at the benchmark's sizes: the 70B FFN layer
(d = 8192, ffn = 28672) at M = 16384 and 8192 tokens, and the 70B tail linear
(M = 1000, K = 8200, N = 28672).

Every kernel is fed the same inputs as the oracle: seeded synthetic activations
and gradients, and weights compressed / double-pruned by the oracle and uploaded.
Outputs are compared with the oracle's fp32 values at the stated tolerance
(normwise <= 5e-3, elementwise <= 1e-2 + 1e-2 |ref|), with no widening: on 256
seeded rows of each 70B output, and on the whole output of the tail linear.
"""
import numpy as np
import pytest
import torch

from oracle import prune24_oracle as O
from synth24 import normal_bf16, normal_f32
from tests.conftest import bits_of, from_bits
from tests.p24_testutil import assert_close, delta_csr

pytestmark = pytest.mark.gpu

D, FFN = 8192, 28672
ROWS = 256  # sampled output rows per 70B check


@pytest.fixture(scope="module")
def P():
    import semi_structured_sparse_prune24_gb300 as P
    return P


def upload_sparse(P, vals, meta, rows, cols):
    s = P.Sparse24.empty(rows, cols)
    assert s.ldv == vals.shape[1] and s.ldm == meta.shape[1]
    s.vals.copy_(from_bits(vals, "cuda"))
    s.meta.copy_(torch.from_numpy(meta).to("cuda"))
    return s


@pytest.fixture(scope="module")
def w70(P):
    """W_up [ffn, d] and W_down [d, ffn] ~ N(0, 0.01^2), seed 0: the oracle's forward
    compression and double-pruned transposes, host bits and device descriptors."""
    out = {}
    for name, (rows, cols, tid) in {"up": (FFN, D, 2), "down": (D, FFN, 3)}.items():
        W = bits_of(normal_bf16((rows, cols), 0.01, 0, tid))
        fv, fm = O.compress24(W, P.ld_vals(cols), P.ld_meta(cols))
        tv, tm_ = O.double_prune(fv, fm, rows, cols, P.ld_vals(rows), P.ld_meta(rows))
        out[name] = {"fwd": (fv, fm), "bwdT": (tv, tm_),
                     "fwd_dev": upload_sparse(P, fv, fm, rows, cols),
                     "bwdT_dev": upload_sparse(P, tv, tm_, cols, rows)}
    return out


def relu_normal(shape, seed, tid):
    """A ReLU output: N(0, 1) clipped at 0 (the gated activations of the step)."""
    return torch.relu(normal_bf16(shape, 1.0, seed, tid, "cuda"))


def sample(n, k, seed):
    return np.sort(np.random.default_rng(seed).choice(n, k, replace=False))


@pytest.mark.parametrize("M", [16384, 8192])
@pytest.mark.parametrize("which", ["up", "down"])
def test_spmm24_fwd_70b(P, w70, M, which):
    """Up forward H = ReLU(X W_up^T + b) [M, ffn], or down forward Y = H W_down^T [M, d]."""
    N, K = (FFN, D) if which == "up" else (D, FFN)
    X = normal_bf16((M, K), 1.0, 1, 1, "cuda") if which == "up" else relu_normal((M, K), 1, 7)
    b = normal_f32((N,), 0.1, 1, 4, "cuda") if which == "up" else None
    Y = P.spmm24_fwd(X, w70[which]["fwd_dev"], bias=b, relu=which == "up")
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    ms = sample(M, ROWS, 11)
    fv, fm = w70[which]["fwd"]
    ref, _ = O.spmm24_fwd(bits_of(X[torch.as_tensor(ms, device="cuda")]), fv, fm, K,
                          bias=None if b is None else b.cpu().numpy(), relu=which == "up")
    assert_close(Y[torch.as_tensor(ms, device="cuda")], ref, f"{which} forward rows")


@pytest.mark.parametrize("M", [16384, 8192])
@pytest.mark.parametrize("which", ["down", "up"])
def test_spmm24_bwd_dx_70b(P, w70, M, which):
    """Double-pruned backward: dH = (dY W_down_bwd) * [H > 0] [M, ffn] with the fused
    bias gradient (which = "down"), or dX = dH W_up_bwd [M, d] (which = "up")."""
    N, K = (D, FFN) if which == "down" else (FFN, D)   # dY [M, N] -> dX [M, K]
    dY = normal_bf16((M, N), 1.0, 2, 6, "cuda") if which == "down" else \
        normal_bf16((M, N), 1.0, 2, 6, "cuda") * (relu_normal((M, N), 2, 8) > 0)
    gate = relu_normal((M, K), 2, 7) if which == "down" else None
    dbias = torch.empty(K, dtype=torch.float32, device="cuda") if which == "down" else None
    dX = P.spmm24_bwd_dx(dY, w70[which]["bwdT_dev"], gate=gate, dbias=dbias)
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    tv, tm_ = w70[which]["bwdT"]
    ms = sample(M, ROWS, 12)
    tms = torch.as_tensor(ms, device="cuda")
    ref, _ = O.spmm24_bwd_dx(bits_of(dY[tms]), tv, tm_, N, gate=None if gate is None else bits_of(gate[tms]))
    assert_close(dX[tms], ref, f"{which} dX rows")
    if dbias is not None:
        # the fused bias gradient on 512 seeded features (whole groups of 4), over every
        # token: the oracle's column sums of its own bf16 dH, plus the exact propagated
        # difference of the two sides' bf16 dH
        fs = (4 * sample(K // 4, 128, 13)[:, None] + np.arange(4)).ravel()
        tfs = torch.as_tensor(fs, device="cuda")
        _, ref_b = O.spmm24_bwd_dx(bits_of(dY), tv[fs], tm_[fs], N, gate=bits_of(gate[:, tfs]))
        delta = delta_csr(bits_of(dX[:, tfs]), ref_b)
        assert_close(dbias[tfs], O.colsum(ref_b), "fused dbias", chain=np.asarray(delta.sum(axis=0)).ravel())


@pytest.mark.parametrize("M", [16384, 8192])
@pytest.mark.parametrize("which", ["down", "up"])
def test_masked_dw_70b(P, w70, M, which):
    """dW_down = (dY^T H) on mask(W_down) [d, ffn], or dW_up = (dH^T X) on mask(W_up) [ffn, d]."""
    N, K = (D, FFN) if which == "down" else (FFN, D)   # dW [N, K] = dY [M, N]^T X [M, K]
    dY = normal_bf16((M, N), 1.0, 3, 6, "cuda")
    X = relu_normal((M, K), 3, 7) if which == "down" else normal_bf16((M, K), 1.0, 3, 1, "cuda")
    dW = P.masked_dw_gemm(dY, X, w70[which]["fwd_dev"])
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    ns = sample(N, ROWS, 14)
    tns = torch.as_tensor(ns, device="cuda")
    _, fm = w70[which]["fwd"]
    ref, _ = O.masked_dw(bits_of(dY[:, tns]), bits_of(X), fm[ns])
    got = dW[tns]
    assert_close(got, ref, f"{which} dW rows")
    assert np.all(bits_of(got)[~O.mask_from_meta(fm[ns], K)] == 0)


# ---------------------------------------------------------------- the 70B tail linear
TM, TK, TN = 1000, 8200, 28672


@pytest.fixture(scope="module")
def tail(P):
    W = bits_of(normal_bf16((TN, TK), 0.01, 0, 2))
    fv, fm = O.compress24(W, P.ld_vals(TK), P.ld_meta(TK))
    tv, tm_ = O.double_prune(fv, fm, TN, TK, P.ld_vals(TN), P.ld_meta(TN))
    return {"fwd": (fv, fm), "bwdT": (tv, tm_), "fwd_dev": upload_sparse(P, fv, fm, TN, TK),
            "bwdT_dev": upload_sparse(P, tv, tm_, TK, TN)}


def test_tail_linear_forward_in_full(P, tail):
    X = normal_bf16((TM, TK), 1.0, 4, 1, "cuda")
    b = normal_f32((TN,), 0.1, 4, 4, "cuda")
    Y = P.spmm24_fwd(X, tail["fwd_dev"], bias=b, relu=True)
    torch.cuda.synchronize()
    ref, _ = O.spmm24_fwd(bits_of(X), *tail["fwd"], TK, bias=b.cpu().numpy(), relu=True)
    assert_close(Y, ref, "tail forward")


def test_tail_linear_backward_dx_in_full(P, tail):
    dY = normal_bf16((TM, TN), 1.0, 4, 6, "cuda")
    gate = relu_normal((TM, TK), 4, 7)
    dbias = torch.empty(TK, dtype=torch.float32, device="cuda")
    dX = P.spmm24_bwd_dx(dY, tail["bwdT_dev"], gate=gate, dbias=dbias)
    torch.cuda.synchronize()
    ref, ref_b = O.spmm24_bwd_dx(bits_of(dY), *tail["bwdT"], TN, gate=bits_of(gate))
    assert_close(dX, ref, "tail dX")
    delta = delta_csr(bits_of(dX), ref_b)
    assert_close(dbias, O.colsum(ref_b), "tail fused dbias", chain=np.asarray(delta.sum(axis=0)).ravel())


def test_tail_linear_masked_dw_in_full(P, tail):
    dY = normal_bf16((TM, TN), 1.0, 4, 6, "cuda")
    X = normal_bf16((TM, TK), 1.0, 4, 1, "cuda")
    dW = P.masked_dw_gemm(dY, X, tail["fwd_dev"])
    torch.cuda.synchronize()
    _, fm = tail["fwd"]
    ref, _ = O.masked_dw(bits_of(dY), bits_of(X), fm)
    assert_close(dW, ref, "tail dW")
    assert np.all(bits_of(dW)[~O.mask_from_meta(fm, TK)] == 0)

