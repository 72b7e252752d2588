"""GPU parity of the V:2:M prune (vnm24_compress) against the oracle: the kept
column offsets, values, metadata and padding, bit for bit."""
import numpy as np
import pytest
import torch

from oracle import prune24_oracle as O
from oracle import vnm_oracle as VNM
from synth24 import normal_bf16, small_int_bf16
from tests.conftest import bits_of, from_bits
from tests.p24_testutil import assert_bits_equal, sparse_bits

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
         (2, 264, 1, 8), (300, 1024, 64, 8)]


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
