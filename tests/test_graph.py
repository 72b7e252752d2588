"""StepGraph: a training step captured as a CUDA graph and replayed gives the
eager step's results, and follows new input data copied into its buffers."""
import pytest
import torch

from synth24 import WORKLOADS, ffn_inputs
from tests.conftest import bits_of
from tests.p24_testutil import assert_bits_equal

pytestmark = pytest.mark.gpu


def _eager(P, inp, act24, adapters=None):
    return P.ffn24_step(inp["X"], inp["W_up"], inp["b_up"], inp["W_down"], inp["b_down"], inp["dY"], act24=act24,
                        adapters=adapters)


@pytest.mark.parametrize("act24", [False, True])
def test_graph_replay_matches_eager_and_follows_new_inputs(act24):
    import semi_structured_sparse_prune24_gb300 as P
    from semi_structured_sparse_prune24_gb300.graph import StepGraph
    w = WORKLOADS["gpt2"]
    a, b = ffn_inputs(w, seed=31, device="cuda", bias=True), ffn_inputs(w, seed=32, device="cuda", bias=True)
    bufs = {k: v.clone() for k, v in a.items()}
    g = StepGraph(bufs, act24=act24)
    for inp in (a, b, a):                         # replay on new data copied into the captured buffers
        for k in ("X", "W_up", "W_down", "dY"):
            bufs[k].copy_(inp[k])
        o = g.replay()
        g.synchronize()
        ref = _eager(P, dict(inp, b_up=bufs["b_up"], b_down=bufs["b_down"]), act24)
        torch.cuda.synchronize()
        for k in ("H", "Y", "dX", "dW_up", "dW_down"):
            assert_bits_equal(bits_of(o[k]), bits_of(ref[k]), k)
        assert torch.equal(o["db_down"], ref["db_down"])
        torch.testing.assert_close(o["db_up"], ref["db_up"], rtol=1e-5, atol=1e-4)
    assert P.p24_query_status() == 0


def test_graph_with_adapters():
    import semi_structured_sparse_prune24_gb300 as P
    from semi_structured_sparse_prune24_gb300.graph import StepGraph
    from synth24 import normal_bf16
    w = WORKLOADS["gpt2"]
    inp = ffn_inputs(w, seed=33, device="cuda", bias=False)
    r = 64
    ad = {"L_up": normal_bf16((w.ffn, r), 0.02, 33, 10, "cuda"), "R_up": normal_bf16((r, w.d), 0.02, 33, 11, "cuda"),
          "L_down": normal_bf16((w.d, r), 0.02, 33, 12, "cuda"), "R_down": normal_bf16((r, w.ffn), 0.02, 33, 13, "cuda")}
    g = StepGraph(dict(inp), adapters=ad)
    o = g.replay()
    g.synchronize()
    ref = _eager(P, inp, False, ad)
    torch.cuda.synchronize()
    for k in ("Y", "dX", "dW_up", "dW_down", "dL_up", "dR_up", "dL_down", "dR_down"):
        assert_bits_equal(bits_of(o[k]), bits_of(ref[k]), k)
