"""A reusable MoE layer object over the C ABI: owns the caller-side device
buffers (index structures, saved activations, scratch, outputs) for one shape
and runs dispatch build, forward and backward through libmoeblaze.so on the
current CUDA stream.  PyTorch only provides the memory and the stream."""
from __future__ import annotations

from typing import Dict, Optional

import torch

from . import binding as B


class MoELayer:
    def __init__(self, L: int, d: int, h: int, E: int, K: int, dtype: torch.dtype, act: str, device="cuda",
                 with_dgates: bool = True, recompute_h: bool = False):
        """recompute_h: keep no H / Hg temporaries (MOEBLAZE_RECOMPUTE_H):
        smaller scratch, the down projection and dW3 recompute them."""
        self.shape = B.make_shape(L, d, h, E, K, dtype, act, B.RECOMPUTE_H if recompute_h else 0)
        self.L, self.d, self.h, self.E, self.K = L, d, h, E, K
        self.dtype, self.act, self.device = dtype, act, device
        self.disp = B.alloc_dispatch(self.shape, device)
        self.bufs = B.alloc_layer(self.shape, device)
        self.y = torch.empty((L, d), dtype=dtype, device=device)
        self.dX = torch.empty((L, d), dtype=dtype, device=device)
        # gate gradients (for a router's backward): optional extra output
        self.dgates = torch.empty((L, K), dtype=torch.float32, device=device) if with_dgates else None
        if act == "identity":
            self.dW1 = self.dW2 = self.dW3 = None
        else:
            self.dW1 = torch.empty((E, d, h), dtype=dtype, device=device)
            self.dW2 = torch.empty((E, d, h), dtype=dtype, device=device) if act == "swiglu" else None
            self.dW3 = torch.empty((E, h, d), dtype=dtype, device=device)

    @classmethod
    def for_config(cls, cfg, device="cuda", with_dgates: bool = True, recompute_h: bool = False):
        return cls(cfg.L, cfg.d, cfg.h, cfg.E, cfg.K, cfg.torch_dtype, cfg.act, device, with_dgates, recompute_h)

    def dispatch(self, ids: torch.Tensor, validate: bool = False):
        B.dispatch_build(self.shape, ids, self.disp, validate=validate)
        return B.index_views(self.shape, self.disp)

    def route(self, x: torch.Tensor, Wr: torch.Tensor, bias: Optional[torch.Tensor] = None):
        """The softmax top-K router fused with the dispatch build
        (moeblaze_router_dispatch_build): fills this layer's dispatch and
        returns (topk_ids, gates), which forward and backward then take."""
        if not hasattr(self, "_route_bufs"):
            dev = Wr.device
            self._route_bufs = (torch.empty((self.L, self.K), dtype=torch.int32, device=dev),
                                torch.empty((self.L, self.K), dtype=torch.float32, device=dev),
                                torch.empty(B.moeblaze_router_dispatch_workspace_bytes(self.shape), dtype=torch.uint8,
                                            device=dev))
        ids, gates, ws = self._route_bufs
        B.router_dispatch_build(self.shape, x, Wr, bias, ids, gates, self.disp, ws)
        return ids, gates

    def forward(self, x, gates, W1=None, W2=None, W3=None) -> torch.Tensor:
        B.forward(self.shape, x, gates, self.disp, W1, W2, W3, self.y, self.bufs)
        return self.y

    def backward(self, dY, x, gates, W1=None, W2=None, W3=None):
        B.backward(self.shape, dY, x, gates, self.disp, W1, W2, W3, self.bufs, self.dX, self.dW1, self.dW2, self.dW3,
                   self.dgates)
        return self.dX, self.dW1, self.dW2, self.dW3, self.dgates

    def step(self, inp: Dict[str, torch.Tensor]):
        """dispatch build + forward + backward on one batch of inputs."""
        self.dispatch(inp["ids"])
        self.forward(inp["x"], inp["gates"], inp.get("W1"), inp.get("W2"), inp.get("W3"))
        self.backward(inp["dY"], inp["x"], inp["gates"], inp.get("W1"), inp.get("W2"), inp.get("W3"))

    def saved(self):
        if self.act == "identity":
            return None, None
        return B.saved_views(self.shape, self.bufs, self.dtype)

    def device_error(self) -> int:
        return B.device_error(self.shape, self.disp)

    def meta(self):
        return B.meta_arrays(self.shape, self.disp)


class GraphStep:
    """The layer's whole step (dispatch build, forward, backward) captured
    once as a CUDA graph on fixed device buffers and replayed: one graph
    launch instead of a host call per kernel, which is what bounds the small
    layers.  The graph reads the tensors of `inp` (refill them in place
    between replays) and writes the layer's own outputs."""

    def __init__(self, layer: MoELayer, inp: Dict[str, torch.Tensor]):
        self.layer = layer
        self.inp = inp
        # an eager step first: kernel attributes and the library's cached
        # occupancy queries are settled outside the capture
        layer.step(inp)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            layer.step(inp)

    def replay(self):
        self.graph.replay()


class StepPipeline:
    """Runs layer steps whose inputs live in pinned host memory and whose
    outputs (y, dX) go back to pinned host memory, overlapping the copies
    with the compute of the neighbouring steps:

      copy stream     H2D(inputs i+1) into the other input slot, while step i computes
      compute stream  dispatch, forward, backward of step i
      out stream      D2H(y_i) right after forward i (overlaps backward i),
                      D2H(dX_i) after backward i (overlaps the next dispatch and forward)

    The next forward waits for D2H(y_i) and the next backward for D2H(dX_i)
    before overwriting y and dX; an input slot is reused only after the step
    that read it has finished.  Every step's copies are part of the run."""

    def __init__(self, layer: MoELayer, keys=("x", "ids", "gates", "dY")):
        self.layer = layer
        self.keys = keys
        self.slots = None
        self.copy = torch.cuda.Stream()
        self.out = torch.cuda.Stream()
        self.comp = torch.cuda.current_stream()

    def _ensure_slots(self, batch):
        if self.slots is None:
            self.slots = [{k: torch.empty(batch[k].shape, dtype=batch[k].dtype, device="cuda") for k in self.keys}
                          for _ in range(2)]
            self.in_ready = [torch.cuda.Event() for _ in range(2)]
            self.slot_free = [torch.cuda.Event() for _ in range(2)]
            self.y_done = torch.cuda.Event()
            self.dx_done = torch.cuda.Event()
            self.fwd_done = torch.cuda.Event()
            self.bwd_done = torch.cuda.Event()

    def _h2d(self, i, batch):
        s = i % 2
        with torch.cuda.stream(self.copy):
            if i >= 2:
                self.copy.wait_event(self.slot_free[s])
            for k in self.keys:
                self.slots[s][k].copy_(batch[k], non_blocking=True)
            self.in_ready[s].record(self.copy)

    def run(self, batches, outputs, weights):
        """batches[i]: dict of pinned host tensors (x, ids, gates, dY);
        outputs[i]: (y_host, dX_host) pinned; weights: (W1, W2, W3) on the device."""
        L = self.layer
        n = len(batches)
        if n == 0:
            return
        self._ensure_slots(batches[0])
        self._h2d(0, batches[0])
        for i in range(n):
            s = i % 2
            if i + 1 < n:
                self._h2d(i + 1, batches[i + 1])
            d = self.slots[s]
            self.comp.wait_event(self.in_ready[s])
            L.dispatch(d["ids"])
            if i > 0:
                self.comp.wait_event(self.y_done)
            L.forward(d["x"], d["gates"], *weights)
            self.fwd_done.record(self.comp)
            with torch.cuda.stream(self.out):
                self.out.wait_event(self.fwd_done)
                outputs[i][0].copy_(L.y, non_blocking=True)
                self.y_done.record(self.out)
            if i > 0:
                self.comp.wait_event(self.dx_done)
            L.backward(d["dY"], d["x"], d["gates"], *weights)
            self.bwd_done.record(self.comp)
            self.slot_free[s].record(self.comp)
            with torch.cuda.stream(self.out):
                self.out.wait_event(self.bwd_done)
                outputs[i][1].copy_(L.dX, non_blocking=True)
                self.dx_done.record(self.out)
        self.comp.wait_stream(self.out)
        self.comp.wait_stream(self.copy)
