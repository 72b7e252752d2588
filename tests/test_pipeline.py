"""StepPipeline: host-fed training steps with the copies overlapped must give the
same results as direct ffn24_step calls on device copies of the same batches."""
import pytest
import torch

from synth24 import WORKLOADS, ffn_inputs
from tests.conftest import bits_of
from tests.p24_testutil import assert_bits_equal

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("act24", [False, True])
def test_pipeline_matches_direct_steps(act24):
    import semi_structured_sparse_prune24_gb300 as P
    from semi_structured_sparse_prune24_gb300.pipeline import OUT_KEYS, StepPipeline
    w = WORKLOADS["gpt2"]
    batches = [ffn_inputs(w, seed=s, device="cuda", bias=True) for s in (21, 22)]
    b_up, b_down = batches[0]["b_up"], batches[0]["b_down"]
    host_in = [{k: b[k].cpu().pin_memory() for k in ("X", "W_up", "W_down", "dY")} for b in batches]
    pipe = StepPipeline(w.M, w.d, w.ffn, act24=act24, b_up=b_up, b_down=b_down)
    outs = []
    for i in range(4):                                   # alternate batches, both slots used twice
        o = {k: torch.empty(pipe.outputs[0][k].shape, dtype=pipe.outputs[0][k].dtype).pin_memory()
             for k in OUT_KEYS}
        pipe.submit(host_in[i % 2], o)
        outs.append(o)
    pipe.synchronize()
    for i, o in enumerate(outs):
        b = batches[i % 2]
        ref = P.ffn24_step(b["X"], b["W_up"], b_up, b["W_down"], b_down, b["dY"], act24=act24)
        torch.cuda.synchronize()
        for k in ("Y", "dX", "dW_up", "dW_down"):
            assert_bits_equal(bits_of(o[k]), bits_of(ref[k]), f"step {i} {k}")
        assert torch.equal(o["db_down"], ref["db_down"].cpu())
        torch.testing.assert_close(o["db_up"], ref["db_up"].cpu(), rtol=1e-5, atol=1e-4)
    assert P.p24_query_status() == 0
