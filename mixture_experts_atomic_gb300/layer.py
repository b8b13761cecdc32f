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
                 with_dgates: bool = True):
        self.shape = B.make_shape(L, d, h, E, K, dtype, act)
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
    def for_config(cls, cfg, device="cuda", with_dgates: bool = True):
        return cls(cfg.L, cfg.d, cfg.h, cfg.E, cfg.K, cfg.torch_dtype, cfg.act, device, with_dgates)

    def dispatch(self, ids: torch.Tensor, validate: bool = False):
        B.dispatch_build(self.shape, ids, self.disp, validate=validate)
        return B.index_views(self.shape, self.disp)

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
