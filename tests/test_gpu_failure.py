"""The bounded-wait failure path of the expert GEMMs on the GPU, in the form
that faults nothing: a host-set short wait limit, and a stage of the down
projection that is never issued (its barrier is never completed), so the
kernel's own wait runs out.  The kernel must record a timeout in the device
error word, let its copies in flight land, free its tensor memory and
return; the same process then runs a clean step that matches the oracle."""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from mixture_experts_atomic_gb300 import binding as B
from mixture_experts_atomic_gb300 import inputs as I
from mixture_experts_atomic_gb300.layer import MoELayer

pytestmark = pytest.mark.gpu

from gpu_util import TOL, ensure_built  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_withheld_stage_times_out_and_the_context_stays_usable():
    cfg = I.MoEConfig("t_timeout", 1000, 256, 384, 5, 2, "swiglu", "bf16", 41, "softmax")
    inp_cpu = I.make_inputs(cfg, "cpu")
    inp = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
    W = (inp["W1"], inp["W2"], inp["W3"])
    layer = MoELayer.for_config(cfg, "cuda")
    layer.dispatch(inp["ids"])
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    # every CTA of the down projection waits for a stage nobody fills: its
    # wait runs out after 20 ms
    B.moeblaze_set_fault_injection(20_000_000, 1)
    try:
        layer.forward(inp["x"], inp["gates"], *W)
    finally:
        B.moeblaze_set_fault_injection(0, 0)
    torch.cuda.synchronize()
    st, code = B.moeblaze_device_error(layer.shape, layer.disp.struct(), None)
    assert st == B.ERR_TIMEOUT and code & 2, (st, code)
    # the context is usable: a clean step (the dispatch build clears the
    # word) gives the oracle's results
    layer.step(inp)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    y = O.forward(inp_cpu["ids"], inp_cpu["gates"], inp_cpu["x"], *(inp_cpu[k] for k in ("W1", "W2", "W3")),
                  cfg.act, E=cfg.E)
    dX, dW1, dW2, dW3, _ = O.backward(inp_cpu["ids"], inp_cpu["gates"], inp_cpu["x"], inp_cpu["dY"],
                                      *(inp_cpu[k] for k in ("W1", "W2", "W3")), cfg.act, E=cfg.E)
    errs = {"y": O.rel_err(layer.y, y), "dX": O.rel_err(layer.dX, dX), "dW1": O.rel_err(layer.dW1, dW1),
            "dW2": O.rel_err(layer.dW2, dW2), "dW3": O.rel_err(layer.dW3, dW3)}
    assert max(errs.values()) <= TOL["bf16"], errs
