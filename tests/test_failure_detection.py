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
