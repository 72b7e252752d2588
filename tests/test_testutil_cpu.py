"""CPU checks of the parity helpers themselves (no GPU): the chained bound that
the step tests add for a bf16 operand the two sides computed separately."""
import numpy as np

from tests.p24_testutil import assert_close, chained, delta_csr


def test_chained_bound_is_exact_on_a_known_difference():
    """One operand entry differs by one bf16 ulp: the bound is that ulp times the
    matching row of |B|, and entries the difference does not reach get 0."""
    a = np.array([[0x3F80, 0x4000], [0x4040, 0x0000]], dtype=np.uint16)   # [[1, 2], [3, 0]]
    b = np.array([[0x3F81, 0x4000], [0x4040, 0x0000]], dtype=np.uint16)   # 1 -> 1.0078125
    B = np.array([[3.0, -1.0], [5.0, 7.0]])
    c = chained(delta_csr(a, b), np.abs(B))
    assert np.array_equal(c, [[2 ** -7 * 3.0, 2 ** -7 * 1.0], [0.0, 0.0]])


def test_chained_bound_covers_the_product_difference():
    """|a@B - b@B| <= chained(|a - b|, |B|) for random bf16 operands that differ in a
    few entries (the triangle inequality the step tests rely on)."""
    import torch
    rng = np.random.default_rng(0)
    a = torch.from_numpy(rng.standard_normal((20, 30)).astype(np.float32)).to(torch.bfloat16)
    b = a.clone()
    idx = rng.choice(600, 25, replace=False)
    b.view(-1)[idx] = (b.view(-1)[idx].float() * 1.01).to(torch.bfloat16)
    B = rng.standard_normal((30, 12))
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    diff = np.abs(a.double().numpy() @ B - b.double().numpy() @ B)
    bound = chained(delta_csr(bits(a), bits(b)), np.abs(B))
    assert np.all(diff <= bound + 1e-12)      # fp64 rounding of the two products
    assert bound.max() > 0


def test_assert_close_skip_and_chain():
    """skip leaves elements out of the elementwise check only; chain widens it."""
    import pytest
    import torch
    ref = np.array([1.0, 2.0, 3.0, 4.0] * 100)
    gpu = torch.tensor(ref + np.r_[0.05, np.zeros(399)], dtype=torch.float32)
    with pytest.raises(AssertionError):
        assert_close(gpu, ref, "plain")
    assert_close(gpu, ref, "skip", skip=np.r_[True, np.zeros(399, bool)])
    assert_close(gpu, ref, "chain", chain=np.r_[0.05, np.zeros(399)])
