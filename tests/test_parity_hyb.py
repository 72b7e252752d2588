"""GPU parity of the hybrid ELL + dense-overflow path against the oracle
(oracle/hyb_oracle.py): the format bit for bit (counts, ELL columns and values,
slots, overflow list and backup rows), the hybrid-to-dense and dense-to-hybrid
products within the stated tolerance, and the capacity error."""
import numpy as np
import pytest
import torch

from oracle import hyb_oracle as HY
from oracle import prune24_oracle as O
from synth24 import normal_bf16
from tests.conftest import bits_of, from_bits
from tests.p24_testutil import assert_bits_equal, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import semi_structured_sparse_prune24_gb300 as P
    return P


def sparse_act(rows, cols, seed, dense_every=0, t=2.326, t_dense=1.28, specials=False):
    """ReLU(z - t) with z ~ N(0, 1): about 1% nonzero at t = 2.326; every dense_every-th
    row uses t_dense (about 10% nonzero), so that it overflows a narrow ELL."""
    z = normal_bf16((rows, cols), 1.0, seed, 7).float()
    thr = torch.full((rows, 1), t)
    if dense_every:
        thr[::dense_every] = t_dense
    a = torch.relu(z - thr).to(torch.bfloat16)
    b = bits_of(a)
    if specials:                      # -0 entries (read as zero) and a few negatives
        rng = np.random.default_rng(seed)
        b[rng.random(b.shape) < 0.01] = 0x8000
        neg = rng.random(b.shape) < 0.002
        b[neg] = 0xBF80                # -1.0
    return b


def check_format(h, ref, name=""):
    n = int(h.n_ovf.item())
    assert n == ref["n_ovf"], (name, n, ref["n_ovf"])
    assert np.array_equal(h.nnz.cpu().numpy(), ref["nnz"]), name
    assert np.array_equal(h.slot.cpu().numpy(), ref["slot"]), name
    assert np.array_equal(h.ell_cols.cpu().numpy().view(np.uint16), ref["ell_cols"]), name
    assert_bits_equal(bits_of(h.ell_vals), ref["ell_vals"], name + " ell_vals")
    k = min(n, h.cap)
    assert np.array_equal(h.ovf_rows.cpu().numpy()[:h.cap], ref["ovf_rows"]), name
    assert_bits_equal(bits_of(h.ovf)[:k], ref["ovf"][:k], name + " backup rows")


SHAPES = [(64, 256, 8, 16), (300, 1032, 16, 75), (1000, 2048, 32, 250), (40, 8, 2, 10)]


@pytest.mark.parametrize("R,C,E,cap", SHAPES)
@pytest.mark.parametrize("specials", [False, True])
def test_hyb_compress_bit_exact(P, R, C, E, cap, specials):
    A = sparse_act(R, C, seed=R + C, dense_every=25, t=1.8 if C < 64 else 2.326, specials=specials)
    ref = HY.hyb_compress(A, E, cap)
    assert ref["n_ovf"] <= cap                      # the capacity case has a test of its own
    h = P.hyb_compress(from_bits(A, "cuda"), E, cap)
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    check_format(h, ref, f"{R}x{C}")


@pytest.mark.parametrize("R,C,E,cap,N", [(64, 256, 8, 16, 64), (300, 1032, 16, 75, 256), (1000, 2048, 32, 250, 2056)])
def test_hyb_spmm_and_sddmm(P, R, C, E, cap, N):
    A = sparse_act(R, C, seed=3 * R, dense_every=25)
    B = normal_bf16((C, N), 0.05, 5, 3, "cuda")
    G = normal_bf16((R, N), 1.0, 5, 6, "cuda")
    h = P.hyb_compress(from_bits(A, "cuda"), E, cap)
    Y = P.hyb_spmm(h, B)
    S_ell, S_ovf = P.hyb_sddmm(h, G, B)
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    ref = HY.hyb_compress(A, E, cap)
    Yr, _ = HY.hyb_spmm(ref, bits_of(B))
    assert_close(Y, Yr, "hybrid -> dense")
    S = HY.hyb_sddmm(ref, bits_of(G), bits_of(B))
    assert_close(S_ell, S["ell_ref"], "dense -> hybrid, ELL slots")
    k = ref["n_ovf"]
    assert_close(S_ovf[:k], S["ovf_ref"][:k], "dense -> hybrid, backup rows")
    # exact zeros off the pattern
    assert np.all(bits_of(S_ell)[np.arange(E)[None, :] >= np.where(ref["slot"] < 0, ref["nnz"], 0)[:, None]] == 0)
    assert np.all(bits_of(S_ovf)[:k][~HY.nonzero_mask(ref["ovf"][:k])] == 0)


def test_hyb_capacity_error_is_reported(P):
    """More overflow rows than the backup holds: the format keeps the first cap, the
    product writes zeros for the rest, and the status word says P24_ECAPACITY once."""
    A = sparse_act(100, 256, seed=9, dense_every=10)
    ref = HY.hyb_compress(A, 4, 3)
    assert ref["n_ovf"] > 3
    h = P.hyb_compress(from_bits(A, "cuda"), 4, 3)
    B = normal_bf16((256, 64), 0.05, 9, 3, "cuda")
    Y = P.hyb_spmm(h, B)
    assert P.p24_query_status() == P.P24_ECAPACITY
    assert P.p24_query_status() == 0
    check_format(h, ref, "capacity")
    lost = np.nonzero(ref["slot"] >= 3)[0]
    assert torch.count_nonzero(Y[torch.as_tensor(lost, device="cuda")]).item() == 0


def test_hyb_bench_workload_shape(P):
    """The bench's hybrid workload (1.3B FFN shape: 8192 tokens x 8192 hidden units, ~1%
    nonzero, every 50th token ~10%): format bit-exact, products on 256 seeded rows."""
    R, C, N, E = 8192, 8192, 2048, 256
    A = sparse_act(R, C, seed=0, dense_every=50)
    h = P.hyb_compress(from_bits(A, "cuda"), E, R // 16)
    B = normal_bf16((C, N), 0.02, 0, 3, "cuda")
    G = normal_bf16((R, N), 1.0, 0, 6, "cuda")
    Y = P.hyb_spmm(h, B)
    S_ell, S_ovf = P.hyb_sddmm(h, G, B)
    torch.cuda.synchronize()
    assert P.p24_query_status() == 0
    ref = HY.hyb_compress(A, E, R // 16)
    check_format(h, ref, "bench shape")
    rows = np.sort(np.random.default_rng(1).choice(R, 256, replace=False))
    sub = HY.hyb_compress(A[rows], E, 256)
    Yr, _ = HY.hyb_spmm(sub, bits_of(B))
    assert_close(Y[torch.as_tensor(rows, device="cuda")], Yr, "hybrid -> dense rows")
    S = HY.hyb_sddmm(sub, bits_of(G[torch.as_tensor(rows, device="cuda")]), bits_of(B))
    ell_rows = rows[ref["slot"][rows] < 0]
    sel = np.nonzero(ref["slot"][rows] < 0)[0]
    assert_close(S_ell[torch.as_tensor(ell_rows, device="cuda")], S["ell_ref"][sel], "dense -> hybrid rows")
