"""GPU parity of the pruning kernels against the oracle: bit-exact values,
metadata (padding included) and masked copies."""
import numpy as np
import pytest
import torch

from oracle import prune24_oracle as O
from synth24 import normal_bf16, small_int_bf16
from tests.conftest import bits_of, from_bits
from tests.p24_testutil import assert_bits_equal, sparse_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import semi_structured_sparse_prune24_gb300 as P
    return P


def make_w(rows, cols, kind, seed=0):
    """A [rows, cols] bf16 view whose row stride is cols rounded up to 8 (16 bytes)."""
    ld = (cols + 7) // 8 * 8
    if kind == "normal":
        w = normal_bf16((rows, ld), 1.0, seed, 2, "cuda")
    elif kind == "ints":
        w = small_int_bf16((rows, ld), -2, 2, seed, 2, "cuda")
    else:
        # specials: ints sprinkled with -0, inf, -inf, NaN, subnormals
        b = bits_of(small_int_bf16((rows, ld), -2, 2, seed, 2))
        rng = np.random.default_rng(seed)
        specials = np.array([0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001], np.uint16)
        pick = rng.random(b.shape) < 0.2
        b[pick] = specials[rng.integers(0, len(specials), pick.sum())]
        w = from_bits(b, "cuda")
    return w[:, :cols]


SHAPES = [(1, 4), (3, 12), (37, 72), (130, 1028), (257, 1000), (64, 8200)]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("kind", ["normal", "ints", "specials"])
def test_compress_bit_exact(P, rows, cols, kind):
    W = make_w(rows, cols, kind)
    out = P.Sparse24.empty(rows, cols)
    Wm = torch.empty((rows, (cols + 7) // 8 * 8), dtype=torch.bfloat16, device="cuda")[:, :cols]
    P.prune24_compress(W, out, W_masked=Wm)
    gv, gm = sparse_bits(out)
    rv, rm = O.compress24(bits_of(W), out.ldv, out.ldm)
    assert_bits_equal(gv, rv, "vals")
    assert_bits_equal(gm, rm, "meta")
    assert_bits_equal(bits_of(Wm), O.decompress24(rv, rm, cols), "W_masked")


def test_compress_wider_strides_and_strided_input(P):
    rows, cols = 50, 264
    big = make_w(rows, 400, "ints")
    W = big[:, 8:8 + cols]                       # row stride 400, offset 16 bytes
    out = P.Sparse24.empty(rows, cols, ldv=200, ldm=48)
    P.prune24_compress(W, out)
    gv, gm = sparse_bits(out)
    rv, rm = O.compress24(bits_of(W), 200, 48)
    assert_bits_equal(gv, rv, "vals")
    assert_bits_equal(gm, rm, "meta")


# interior tiles only (256, 384); border row only (260, 256); border column only (128, 1032);
# both (260, 520); narrower than one tile (4, 8), (8, 12), (132, 72)
@pytest.mark.parametrize("rows,cols", [(4, 8), (8, 12), (132, 72), (128, 1032), (260, 520), (260, 256), (256, 384)])
@pytest.mark.parametrize("kind", ["normal", "ints", "specials"])
def test_double_prune_bit_exact(P, rows, cols, kind):
    W = make_w(rows, cols, kind, seed=3)
    fwd = P.prune24_compress(W)
    bwdT = P.prune24_transpose_repack(fwd)
    fv, fm = sparse_bits(fwd)
    rfv, rfm = O.compress24(bits_of(W), fwd.ldv, fwd.ldm)   # the oracle's own forward compress
    assert_bits_equal(fv, rfv, "fwd vals")
    assert_bits_equal(fm, rfm, "fwd meta")
    rv, rm = O.double_prune(rfv, rfm, rows, cols, bwdT.ldv, bwdT.ldm)
    gv, gm = sparse_bits(bwdT)
    assert_bits_equal(gv, rv, "bwdT vals")
    assert_bits_equal(gm, rm, "bwdT meta")
    # fused variant: same bits for both outputs
    Wm = torch.empty((rows, (cols + 7) // 8 * 8), dtype=torch.bfloat16, device="cuda")[:, :cols]
    f2, b2 = P.prune24_compress_both(W, W_masked=Wm)
    for a, b, name in ((sparse_bits(f2), (fv, fm), "fwd"), (sparse_bits(b2), (gv, gm), "bwdT")):
        assert_bits_equal(a[0], b[0], f"{name} vals (fused)")
        assert_bits_equal(a[1], b[1], f"{name} meta (fused)")
    assert_bits_equal(bits_of(Wm), O.decompress24(fv, fm, cols), "W_masked (fused)")


def test_every_group_pattern(P):
    """All 4-tuples over a 7-symbol alphabet (2401 groups) in one matrix."""
    sym = bits_of(torch.tensor([0, 1, -1, 2, -2, 3, -3], dtype=torch.float32).to(torch.bfloat16))
    grid = np.stack(np.meshgrid(*([np.arange(7)] * 4), indexing="ij"), -1).reshape(-1, 4)
    flat = sym[grid].reshape(-1)
    flat = np.concatenate([flat, np.zeros((-len(flat)) % 64, np.uint16)])
    Wb = flat.reshape(-1, 64)
    W = from_bits(Wb, "cuda")
    out = P.prune24_compress(W)
    gv, gm = sparse_bits(out)
    rv, rm = O.compress24(Wb, out.ldv, out.ldm)
    assert_bits_equal(gv, rv, "vals")
    assert_bits_equal(gm, rm, "meta")


def test_empty_inputs(P):
    W = torch.empty((0, 16), dtype=torch.bfloat16, device="cuda")
    out = P.prune24_compress(W)
    assert out.vals.shape[0] == 0
    torch.cuda.synchronize()


def test_full_size_standalone_prune_every_row(P):
    """The 1e9-element standalone prune ([31250, 32000]), in the bench's launch
    configuration: every row bit-exactly against the oracle (in blocks of rows)."""
    rows, cols = 31250, 32000
    W = normal_bf16((rows, cols), 0.01, 0, 2, "cuda")
    out = P.prune24_compress(W)
    torch.cuda.synchronize()
    for r0 in range(0, rows, 2048):
        r1 = min(rows, r0 + 2048)
        rv, rm = O.compress24(bits_of(W[r0:r1]), out.ldv, out.ldm)
        assert_bits_equal(bits_of(out.vals[r0:r1]), rv, f"vals rows {r0}-{r1}")
        assert_bits_equal(out.meta[r0:r1].cpu().numpy(), rm, f"meta rows {r0}-{r1}")
    # every nibble legal, everywhere
    m = out.meta[:, :cols // 8]
    lo, hi = (m & 0xF).to(torch.int32), (m >> 4).to(torch.int32)
    legal = torch.zeros(16, dtype=torch.bool, device="cuda")
    legal[list(O.LEGAL_NIBBLES)] = True
    assert bool(legal[lo].all()) and bool(legal[hi].all())
    del W, out
    torch.cuda.empty_cache()
