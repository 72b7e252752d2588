"""Failure detection without a GPU fault: every wait in the library's kernels is
bounded, and an expired wait is reported through the device status word.

The GPU test makes a wait run out on purpose (a barrier nothing arrives on, with
a 20 ms limit) and checks that the host reads P24_ETIMEOUT, that reading clears
it, and that the context keeps working. Nothing is trapped, faulted or hung.
"""
import pytest
import torch

P24_ETIMEOUT = -4


@pytest.mark.gpu
def test_expired_wait_is_reported_and_the_context_survives():
    import semi_structured_sparse_prune24_gb300 as P
    from synth24 import normal_bf16
    assert P.p24_query_status() == 0
    P.p24_selftest_timeout(20_000_000)
    assert P.p24_query_status() == P24_ETIMEOUT
    assert P.p24_query_status() == 0          # reading the status clears it
    W = normal_bf16((64, 128), 1.0, 0, 2, "cuda")
    out = P.prune24_compress(W)               # the context is still usable
    torch.cuda.synchronize()
    assert out.meta.shape[0] == 64
    assert P.p24_query_status() == 0


def test_selftest_rejects_bad_limits():
    from semi_structured_sparse_prune24_gb300 import _native as N
    assert N.lib.p24_selftest_timeout(0, None) == N.P24_EINVAL
    assert N.lib.p24_selftest_timeout(-5, None) == N.P24_EINVAL
    assert N.lib.p24_selftest_timeout(10 ** 11, None) == N.P24_EINVAL


@pytest.mark.gpu
def test_sparse_gemm_wait_expires_cleanly_and_reports_where():
    """The real sparse GEMM with one pipeline stage's loads withheld in its first CTA
    pair (test-only flag): that pair's bounded waits expire, it drains and exits; the
    status names the CTA and the barrier; the next call on the same buffers is correct."""
    import numpy as np
    import semi_structured_sparse_prune24_gb300 as P
    from oracle import prune24_oracle as O
    from synth24 import normal_bf16
    from tests.conftest import bits_of
    from tests.p24_testutil import assert_close
    W = normal_bf16((512, 1024), 0.02, 3, 2, "cuda")
    X = normal_bf16((512, 1024), 1.0, 3, 1, "cuda")
    Ws = P.prune24_compress(W)
    assert P.p24_query_status() == 0
    Y = P.spmm24_fwd(X, Ws, test_stall=True)
    code, cta, bar = P.p24_query_timeout()
    assert code == P24_ETIMEOUT
    assert cta in (0, 1)                      # a CTA of the first pair
    # the barrier's shared address as its CTA saw it: the offset in the low 24 bits
    # (a cluster CTA's window carries its rank above them), within the 227 KB window
    assert bar >= 0 and (bar & 0xFFFFFF) < 232448
    assert P.p24_query_timeout() == (0, -1, -1)
    Y = P.spmm24_fwd(X, Ws, Y=Y)
    torch.cuda.synchronize()
    vals, meta = O.compress24(bits_of(W), Ws.ldv, Ws.ldm)
    ref, _ = O.spmm24_fwd(bits_of(X), vals, meta, 1024)
    assert_close(Y, ref, "Y after the stalled call")
    assert P.p24_query_status() == 0
