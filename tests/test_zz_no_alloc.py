"""p24_colsum_noalloc: bias-gradient column sums for callers that cannot
allocate device memory (no workspace argument; the library keeps a fixed
device scratch array). Checked through the C ABI against the oracle's column
sums and against p24_colsum, the workspace version, on two calls in a row:
bit for bit where the scratch holds every row slab, within the colsum
tolerance where fewer slabs are used.

This file is collected last on purpose: the entry point shares one scratch
array across calls, so it is exercised both in a fresh process and after
every other test has run.
"""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import semi_structured_sparse_prune24_gb300 as P
    return P


def _noalloc(P, G, out):
    lib = P.lib  # the C entry point itself (ctypes), no Python-side workspace
    M, N = G.shape
    code = lib.p24_colsum_noalloc(C.c_void_p(G.data_ptr()), M, N, G.stride(0), C.c_void_p(out.data_ptr()),
                                  C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, P.lib.p24_strerror(code)


def test_noalloc_colsum_matches_workspace_version_twice(P):
    from oracle import prune24_oracle as O
    from synth24 import normal_bf16
    from tests.conftest import bits_of
    cases = [(1000, 392), (4096, 3072), (300, 2 ** 19 + 8)]   # the last forces fewer row slabs
    for i, (M, N) in enumerate(cases):
        G = normal_bf16((M, N), 1.0, 40 + i, 6, "cuda")
        want = P.p24_colsum(G)
        got1 = torch.full((N,), float("nan"), device="cuda")
        got2 = torch.full((N,), float("nan"), device="cuda")
        _noalloc(P, G, got1)
        _noalloc(P, G, got2)                                    # second call in a row
        torch.cuda.synchronize()
        ref = O.colsum(bits_of(G))                              # the oracle's fp32 column sums
        for got in (got1, got2):
            np.testing.assert_allclose(got.cpu().numpy(), ref, rtol=1e-4, atol=1e-3 * np.sqrt(M))
            if P.lib.p24_colsum_workspace_size(M, N) <= 4 * 2 ** 20:
                # the scratch holds every slab: the same kernels in the same order as p24_colsum
                assert torch.equal(got, want)
            else:
                np.testing.assert_allclose(got.cpu().numpy(), want.cpu().numpy(), rtol=1e-4,
                                           atol=1e-3 * np.sqrt(M))
        assert torch.equal(got1, got2)
    assert P.p24_query_status() == 0


def test_noalloc_colsum_rejects_too_wide(P):
    N = (1 << 20) + 8
    G = torch.zeros((2, N), dtype=torch.bfloat16, device="cuda")
    out = torch.empty(N, dtype=torch.float32, device="cuda")
    lib = P.lib
    code = lib.p24_colsum_noalloc(C.c_void_p(G.data_ptr()), 2, N, N, C.c_void_p(out.data_ptr()), None)
    assert code == -6  # P24_ENOSPACE, nothing launched
