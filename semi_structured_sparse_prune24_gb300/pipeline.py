"""Training steps fed from host memory with the copies overlapped.

StepPipeline runs ffn24_step on a sequence of host batches. Two device slots hold
the inputs (X, W_up, W_down, dY) and outputs (Y, H, dX, dW_up, dW_down, db_up,
db_down) of alternate steps, so that three CUDA streams can work at once:

    copy-in   H2D of step i+1's inputs into the other slot
    compute   ffn24_step of step i
    copy-out  D2H of step i-1's outputs

Events order them: a slot's inputs are overwritten only after the step that read
them has finished, and its outputs only after they have been copied out. The
compute stream runs the steps in order and shares one workspace. Host buffers
must be pinned for the copies to be asynchronous.
"""
from __future__ import annotations

import torch

from . import _native as N

IN_KEYS = ("X", "W_up", "W_down", "dY")
OUT_KEYS = ("Y", "dX", "dW_up", "dW_down", "db_up", "db_down")


class StepPipeline:
    def __init__(self, M: int, d: int, ffn: int, act24: bool = False, b_up: torch.Tensor | None = None,
                 b_down: torch.Tensor | None = None, device="cuda"):
        self.M, self.d, self.ffn, self.act24 = M, d, ffn, act24
        self.device = torch.device(device)
        bf = torch.bfloat16
        shapes_in = {"X": (M, d), "W_up": (ffn, d), "W_down": (d, ffn), "dY": (M, d)}
        self.inputs = [{k: torch.empty(s, dtype=bf, device=self.device) for k, s in shapes_in.items()}
                       for _ in range(2)]
        self.outputs = []
        for _ in range(2):
            o = {"Y": torch.empty((M, d), dtype=bf, device=self.device),
                 "H": torch.empty((M, ffn), dtype=bf, device=self.device),
                 "dX": torch.empty((M, d), dtype=bf, device=self.device),
                 "dW_up": torch.empty((ffn, d), dtype=bf, device=self.device),
                 "dW_down": torch.empty((d, ffn), dtype=bf, device=self.device),
                 "db_up": torch.empty(ffn, dtype=torch.float32, device=self.device),
                 "db_down": torch.empty(d, dtype=torch.float32, device=self.device)}
            self.outputs.append(o)
        self.b_up, self.b_down = b_up, b_down
        self.workspace = torch.empty(N.ffn24_workspace_size(M, d, ffn, act24), dtype=torch.uint8,
                                     device=self.device)
        self.s_in = torch.cuda.Stream(self.device)
        self.s_comp = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        self.computed = [None, None]   # event: the slot's step has finished (its inputs are free)
        self.copied_out = [None, None]  # event: the slot's outputs are on the host (its outputs are free)
        self.steps = 0

    def start_after(self, event: torch.cuda.Event) -> None:
        """Make all three streams wait for `event` (e.g. the start of a timed region)."""
        for s in (self.s_in, self.s_comp, self.s_out):
            s.wait_event(event)

    def submit(self, host_in: dict, host_out: dict) -> None:
        """Queue one step: copy host_in's tensors in, run the step, copy its outputs
        (OUT_KEYS) into host_out. Returns at once; host_out is ready after
        synchronize() or after the event of a later wait."""
        slot = self.steps % 2
        dev_in, dev_out = self.inputs[slot], self.outputs[slot]
        with torch.cuda.stream(self.s_in):
            if self.computed[slot] is not None:
                self.s_in.wait_event(self.computed[slot])
            for k in IN_KEYS:
                dev_in[k].copy_(host_in[k], non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(self.s_in)
        self.s_comp.wait_event(ready)
        if self.copied_out[slot] is not None:
            self.s_comp.wait_event(self.copied_out[slot])
        N.ffn24_step(dev_in["X"], dev_in["W_up"], self.b_up, dev_in["W_down"], self.b_down, dev_in["dY"],
                     act24=self.act24, out=dev_out, workspace=self.workspace, stream=self.s_comp)
        done = torch.cuda.Event()
        done.record(self.s_comp)
        self.computed[slot] = done
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(done)
            for k in OUT_KEYS:
                host_out[k].copy_(dev_out[k], non_blocking=True)
            out_done = torch.cuda.Event()
            out_done.record(self.s_out)
        self.copied_out[slot] = out_done
        self.steps += 1

    def finish_on(self, stream: torch.cuda.Stream) -> None:
        """Make `stream` wait for everything submitted so far."""
        for s in (self.s_in, self.s_comp, self.s_out):
            e = torch.cuda.Event()
            e.record(s)
            stream.wait_event(e)

    def synchronize(self) -> None:
        for s in (self.s_in, self.s_comp, self.s_out):
            s.synchronize()
