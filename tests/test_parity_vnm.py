"""GPU parity of the V:2:M path against the oracle: the prune (vnm24_compress: kept
column offsets, values, metadata, padding and the dense masked form, bit for bit)
and the V:2:M GEMM (vnm24_spmm, within the stated tolerance)."""
import numpy as np
import pytest
import torch

from oracle import prune24_oracle as O
from oracle import vnm_oracle as VNM
from synth24 import normal_bf16, small_int_bf16
from tests.conftest import bits_of, from_bits
from tests.p24_testutil import assert_bits_equal, assert_close, sparse_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import semi_structured_sparse_prune24_gb300 as P
    return P


def make_a(rows, cols, kind, seed):
    """A [rows, cols] bf16 view with a row stride of cols rounded up to 8, plus 8."""
    ld = (cols + 7) // 8 * 8 + 8
    if kind == "normal":
        a = normal_bf16((rows, ld), 1.0, seed, 2, "cuda")
    else:
        b = bits_of(small_int_bf16((rows, ld), -2, 2, seed, 2))
        if kind == "specials":
            rng = np.random.default_rng(seed)
            sp = np.array([0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001], np.uint16)
            pick = rng.random(b.shape) < 0.2
            b[pick] = sp[rng.integers(0, len(sp), pick.sum())]
        a = from_bits(b, "cuda")
    return a[:, :cols]


# ragged last 256-column chunk, odd group counts, V above the row count, M from 4 to 128
CASES = [(7, 64, 3, 8), (20, 96, 8, 16), (5, 300, 2, 4), (9, 384, 4, 128), (3, 40, 5, 8), (33, 512, 16, 32),
         (2, 264, 1, 8), (300, 1024, 64, 8), (45, 224, 7, 32), (130, 136, 128, 4), (520, 328, 256, 8)]


@pytest.mark.parametrize("rows,cols,V,M", CASES)
@pytest.mark.parametrize("kind", ["normal", "ints", "specials"])
def test_vnm_compress_bit_exact(P, rows, cols, V, M, kind):
    A = make_a(rows, cols, kind, seed=rows + cols + V)
    colidx, out = P.vnm24_compress(A, V, M)
    torch.cuda.synchronize()
    Ab = bits_of(A)
    rc, _, _ = VNM.vnm_compress(Ab, V, M)
    rv, rm = O.compress24(VNM.condense(Ab, rc, V, M), out.ldv, out.ldm)
    assert np.array_equal(colidx.cpu().numpy(), rc), "colidx"
    gv, gm = sparse_bits(out)
    assert_bits_equal(gv, rv, "vals")
    assert_bits_equal(gm, rm, "meta")
    assert P.p24_query_status() == 0


def test_vnm_compress_large(P):
    """A 4096 x 8192 weight in the 128:2:8 layout (75% sparse), checked in full."""
    A = normal_bf16((4096, 8192), 0.01, 0, 2, "cuda")
    colidx, out = P.vnm24_compress(A, 128, 8)
    torch.cuda.synchronize()
    Ab = bits_of(A)
    rc, _, _ = VNM.vnm_compress(Ab, 128, 8)
    rv, rm = O.compress24(VNM.condense(Ab, rc, 128, 8), out.ldv, out.ldm)
    assert np.array_equal(colidx.cpu().numpy(), rc)
    gv, gm = sparse_bits(out)
    assert_bits_equal(gv, rv, "vals")
    assert_bits_equal(gm, rm, "meta")


def test_vnm_m4_equals_2to4(P):
    A = make_a(64, 256, "specials", seed=5)
    _, out = P.vnm24_compress(A, 16, 4)
    ref = P.prune24_compress(A)
    torch.cuda.synchronize()
    for x, y, name in zip(sparse_bits(out), sparse_bits(ref), ("vals", "meta")):
        assert_bits_equal(x, y, name)


@pytest.mark.parametrize("rows,cols,V,M", [(300, 1024, 256, 8), (40, 264, 16, 8), (9, 384, 4, 128),
                                           (600, 512, 300, 8), (520, 328, 256, 8), (77, 96, 32, 16),
                                           (45, 224, 7, 32), (130, 136, 128, 4), (3, 64, 256, 16)])
@pytest.mark.parametrize("in_place", [False, True])
def test_vnm_compress_masked_output(P, rows, cols, V, M, in_place):
    """The dense masked form A_masked (A with every pruned entry +0), written beside the
    compressed one or over A itself; bit-exact against the oracle's decompression.
    V above 256 (the unstaged kernel) has no masked output: P24_EUNSUPPORTED."""
    A = make_a(rows, cols, "specials", seed=rows + V)
    Ab = bits_of(A)
    if V > 256:
        with pytest.raises(P.P24Error):
            P.vnm24_compress(A, V, M, A_masked=torch.empty_like(A))
        return
    Am = A if in_place else torch.empty_like(A)
    colidx, out = P.vnm24_compress(A, V, M, A_masked=Am)
    torch.cuda.synchronize()
    rc, rv, rm = VNM.vnm_compress(Ab, V, M)
    assert np.array_equal(colidx.cpu().numpy(), rc), "colidx"
    assert_bits_equal(bits_of(Am), VNM.vnm_decompress(rc, rv, rm, rows, cols, V, M), "A_masked")
    gv, gm = sparse_bits(out)
    rv2, rm2 = O.compress24(VNM.condense(Ab, rc, V, M), out.ldv, out.ldm)
    assert_bits_equal(gv, rv2, "vals")
    assert_bits_equal(gm, rm2, "meta")


def oracle_vnm_operand(P, A_bits, V, M):
    """The oracle's V:2:M form of A (colidx, condensed 2:4), uploaded for the GEMM."""
    rows, cols = A_bits.shape
    ci, _, _ = VNM.vnm_compress(A_bits, V, M)
    s = P.Sparse24.empty(rows, 4 * cols // M)
    v, m = O.compress24(VNM.condense(A_bits, ci, V, M), s.ldv, s.ldm)
    s.vals.copy_(from_bits(v, "cuda"))
    s.meta.copy_(torch.from_numpy(m).to("cuda"))
    return torch.from_numpy(ci).to("cuda"), s, (ci, v, m)


# (R rows of A, K, N, V, M): several tiles each way, a ragged last row block, V above 256, M from 4 to 32
SPMM_CASES = [(512, 1024, 512, 256, 8), (700, 2048, 256, 256, 8), (768, 2048, 768, 512, 16),
              (512, 512, 256, 256, 4), (256, 4096, 512, 256, 32)]


@pytest.mark.parametrize("R,K,N,V,M", SPMM_CASES)
@pytest.mark.parametrize("bias,relu", [(False, False), (True, True)])
def test_vnm24_spmm(P, R, K, N, V, M, bias, relu):
    """Y = act(A . B + bias), A V:2:M (the oracle's compression, uploaded), B [K, N]."""
    from synth24 import normal_f32
    A = bits_of(torch.relu(normal_bf16((R, K), 1.0, 7, 7)))
    B = normal_bf16((K, N), 0.02, 7, 3, "cuda")
    b = normal_f32((N,), 0.1, 7, 5, "cuda") if bias else None
    ci, As, (rc, rv, rm) = oracle_vnm_operand(P, A, V, M)
    Y = P.vnm24_spmm(ci, As, V, M, B, bias=b, relu=relu)
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    ref, _ = VNM.vnm_linear(rc, rv, rm, R, K, V, M, bits_of(B), bias=None if b is None else b.cpu().numpy(),
                            relu=relu)
    assert_close(Y, ref, "Y")


def test_vnm24_spmm_70b_down_shape(P):
    """The down linear of the 70B FFN fed V:N:M activations (256:2:8): A = H [16384,
    28672], B = W_down^T [28672, 8192]. Checked on two whole row blocks (512 rows)."""
    R, K, N, V, M = 16384, 28672, 8192, 256, 8
    A = bits_of(torch.relu(normal_bf16((R, K), 1.0, 8, 7)))
    B = normal_bf16((K, N), 0.01, 8, 3, "cuda")
    ci, As, (rc, rv, rm) = oracle_vnm_operand(P, A, V, M)
    Y = P.vnm24_spmm(ci, As, V, M, B)
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    for blk in (3, 41):
        rows = slice(blk * V, (blk + 1) * V)
        ref, _ = VNM.vnm_linear(rc[blk:blk + 1], rv[rows], rm[rows], V, K, V, M, bits_of(B))
        assert_close(Y[rows], ref, f"Y block {blk}")
