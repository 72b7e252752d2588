"""One training step captured as a CUDA graph and replayed.

ffn24_step enqueues only stream-ordered work (kernels and memsets; tensor maps
are kernel parameters), so a step on fixed device buffers can be captured once
and replayed: the replay skips the per-launch host work (argument validation,
tensor-map encoding, launch calls), which matters when the step is short.
Inputs are read from, and outputs written to, the buffers given at capture time:
copy new data into `inputs` before each replay.
"""
from __future__ import annotations

import torch

from . import _native as N


class StepGraph:
    def __init__(self, inputs: dict, act24: bool = False, adapters: dict | None = None):
        """inputs: device tensors X, W_up, b_up, W_down, b_down, dY (biases may be None)."""
        self.inputs = dict(inputs)
        self.act24 = act24
        self.adapters = adapters
        X, Wu = self.inputs["X"], self.inputs["W_up"]
        M, d, ffn = X.shape[0], X.shape[1], Wu.shape[0]
        r = 0 if adapters is None else adapters["L_up"].shape[1]
        size = N.ffn24_workspace_size_lowrank(M, d, ffn, act24, r) if r else N.ffn24_workspace_size(M, d, ffn, act24)
        self.workspace = torch.empty(size, dtype=torch.uint8, device=X.device)
        self.stream = torch.cuda.Stream(X.device)
        # one eager step on the capture stream allocates the outputs and loads the kernels
        self.stream.wait_stream(torch.cuda.current_stream(X.device))
        with torch.cuda.stream(self.stream):
            self.outputs = self._step(None)
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self._step(self.outputs)

    def _step(self, out):
        i = self.inputs
        return N.ffn24_step(i["X"], i["W_up"], i.get("b_up"), i["W_down"], i.get("b_down"), i["dY"], act24=self.act24,
                            out=out, workspace=self.workspace, adapters=self.adapters, stream=self.stream)

    def replay(self) -> dict:
        """Run the captured step on the current contents of `inputs`, on this object's
        stream after the work already queued on the caller's current stream; returns
        `outputs` (valid once `stream` has caught up, e.g. after synchronize())."""
        self.stream.wait_stream(torch.cuda.current_stream(self.stream.device))
        with torch.cuda.stream(self.stream):
            self.graph.replay()
        return self.outputs

    def synchronize(self) -> None:
        self.stream.synchronize()
