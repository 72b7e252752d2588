"""Programmatic-dependent launches stay ordered in a user's stream.

The library launches its kernels with programmatic stream serialization: a kernel
may start while the stream's previous kernel still runs, and waits on the device
for that kernel's completion before its first global access. These tests chain
library calls with torch kernels that rewrite their inputs and outputs in between,
on one stream and with no host synchronisation, and require the results to be
bit-identical to the same calls with a device synchronize after each one (every
kernel of the chain is deterministic)."""
import pytest
import torch

from synth24 import normal_bf16
from tests.conftest import bits_of
from tests.p24_testutil import assert_bits_equal

pytestmark = pytest.mark.gpu

M, K, N, N2 = 1000, 512, 768, 384   # several 256-row tiles with a ragged tail


def _inputs(seed):
    return {"X": normal_bf16((M, K), 1.0, seed, 0, "cuda"), "W": normal_bf16((N, K), 0.05, seed, 1, "cuda"),
            "b": normal_bf16((N,), 0.1, seed, 2, "cuda").float(), "W2": normal_bf16((N2, N), 0.05, seed, 3, "cuda")}


def _chain(P, inp, sync):
    def step():
        if sync:
            torch.cuda.synchronize()

    X = inp["X"].clone()
    fwd = P.prune24_compress(inp["W"]); step()
    Y = P.spmm24_fwd(X, fwd, bias=inp["b"], relu=True); step()
    X.mul_(-1.0)                        # torch rewrites an input of the previous call
    Y.mul_(0.5)                         # and the output that the next calls read
    cs_y = P.p24_colsum(Y); step()
    fwd2, bwd2 = P.prune24_compress_both(inp["W2"]); step()
    Z = P.spmm24_fwd(Y, fwd2); step()
    Y.zero_()                           # the dW below must see the zeroed Y
    Z.add_(1.0)
    dW2 = P.masked_dw_gemm(Z, Y, fwd2); step()
    dY = P.spmm24_bwd_dx(Z, bwd2); step()
    cs_z = P.p24_colsum_noalloc(Z); step()
    Y2 = P.spmm24_fwd(X, fwd); step()   # X as torch left it
    torch.cuda.synchronize()
    return {"Y": Y2, "Z": Z, "dW2": dW2, "dY": dY, "cs_y": cs_y, "cs_z": cs_z}


@pytest.mark.parametrize("side_stream", [False, True])
def test_chain_without_sync_matches_synchronised_chain(side_stream):
    import semi_structured_sparse_prune24_gb300 as P
    inp = _inputs(41)
    ref = _chain(P, inp, sync=True)
    s = torch.cuda.Stream() if side_stream else torch.cuda.current_stream()
    with torch.cuda.stream(s):
        for _ in range(3):              # back to back, so that launches overlap their predecessors
            got = _chain(P, inp, sync=False)
            for k in ("Y", "Z", "dW2", "dY"):
                assert_bits_equal(bits_of(got[k]), bits_of(ref[k]), k)
            for k in ("cs_y", "cs_z"):
                assert torch.equal(got[k], ref[k]), k
    assert float(ref["dW2"].abs().max()) == 0.0   # Y was zeroed before the dW
    assert P.p24_query_status() == 0


def test_chain_joined_across_streams_by_events():
    """A library call on one stream consumes a torch kernel's output from another
    stream, ordered only by an event; its own output is read back on the first."""
    import semi_structured_sparse_prune24_gb300 as P
    inp = _inputs(42)
    fwd = P.prune24_compress(inp["W"])
    torch.cuda.synchronize()
    ref = P.spmm24_fwd(inp["X"] * 2.0, fwd, bias=inp["b"])
    torch.cuda.synchronize()
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(a):
            X2 = inp["X"] * 2.0
            ev = torch.cuda.Event()
            ev.record(a)
        with torch.cuda.stream(b):
            b.wait_event(ev)
            Y = P.spmm24_fwd(X2, fwd, bias=inp["b"])
            cs = P.p24_colsum(Y)
            ev2 = torch.cuda.Event()
            ev2.record(b)
        a.wait_event(ev2)
        with torch.cuda.stream(a):
            Yc = Y.clone()
        X2.record_stream(b)
        Y.record_stream(a)
        torch.cuda.synchronize()
        assert_bits_equal(bits_of(Yc), bits_of(ref), "Y")
        assert torch.equal(cs, P.p24_colsum(ref))
    assert P.p24_query_status() == 0
