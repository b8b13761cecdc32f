"""Argument checks of the Python binding, on the CPU: every tensor handed to
the C library must have the expected shape, dtype and dense layout, and live
on the current CUDA device, before its pointer is passed on.  These checks
run before any library call, so they need no GPU."""
import pytest
import torch

from mixture_experts_atomic_gb300 import binding as B

L, d, h, E, K = 40, 128, 256, 4, 2
BF = torch.bfloat16


def _fwd(act="swiglu", **over):
    shape = B.make_shape(L, d, h, E, K, BF, act)
    a = dict(x=torch.zeros(L, d, dtype=BF), gates=torch.zeros(L, K), y=torch.zeros(L, d, dtype=BF),
             W1=torch.zeros(E, d, h, dtype=BF), W2=torch.zeros(E, d, h, dtype=BF), W3=torch.zeros(E, h, d, dtype=BF))
    a.update(over)
    return B.forward(shape, a["x"], a["gates"], None, a["W1"], a["W2"], a["W3"], a["y"], None)


@pytest.mark.parametrize("over,msg", [
    (dict(x=torch.zeros(L, d + 1, dtype=BF)), "x: shape"),
    (dict(x=torch.zeros(L, d)), "x: dtype"),
    (dict(x=torch.zeros(d, L, dtype=BF).t()), "x: must be contiguous"),
    (dict(gates=torch.zeros(L, K, dtype=torch.float64)), "gates: dtype"),
    (dict(y=torch.zeros(L * d, dtype=BF)), "y: shape"),
    (dict(W1=torch.zeros(E, h, d, dtype=BF)), "W1: shape"),
    (dict(W2=None), "W2: a tensor is required"),
    (dict(W3=torch.zeros(E, h, d)), "W3: dtype"),
])
def test_forward_rejects_malformed_tensors(over, msg):
    with pytest.raises(ValueError, match=msg):
        _fwd(**over)


def test_forward_requires_cuda_tensors():
    with pytest.raises(ValueError, match="x: must be a CUDA tensor"):
        _fwd()


def test_unused_weights_are_not_checked():
    # SiLU has no W2 and the identity expert no weights: whatever is passed
    # there goes to C as NULL, so only the device check of x remains
    with pytest.raises(ValueError, match="x: must be a CUDA tensor"):
        _fwd("silu", W2=torch.zeros(1))
    with pytest.raises(ValueError, match="x: must be a CUDA tensor"):
        _fwd("identity", W1=None, W2=None, W3=None)


def test_backward_checks_gradients():
    shape = B.make_shape(L, d, h, E, K, BF, "silu")
    t = lambda *s, dt=BF: torch.zeros(*s, dtype=dt)  # noqa: E731
    base = dict(dY=t(L, d), x=t(L, d), gates=t(L, K, dt=torch.float32), dX=t(L, d), dgates=None,
                W1=t(E, d, h), W3=t(E, h, d), dW1=t(E, d, h), dW3=t(E, h, d))

    def call(**over):
        a = dict(base, **over)
        B.backward(shape, a["dY"], a["x"], a["gates"], None, a["W1"], None, a["W3"], None, a["dX"], a["dW1"], None,
                   a["dW3"], a["dgates"])

    with pytest.raises(ValueError, match="dgates: dtype"):
        call(dgates=t(L, K))
    with pytest.raises(ValueError, match="dW3: shape"):
        call(dW3=t(E, d, h))
    with pytest.raises(ValueError, match="dY: must be a CUDA tensor"):
        call()


def test_router_and_dispatch_shapes():
    shape = B.make_shape(L, d, 0, E, K, BF, "silu")
    with pytest.raises(ValueError, match="Wr: shape"):
        B.router_forward(shape, torch.zeros(L, d, dtype=BF), torch.zeros(E, d), None,
                         torch.zeros(L, K, dtype=torch.int32), torch.zeros(L, K))
    with pytest.raises(ValueError, match="topk_ids: dtype"):
        B.router_forward(shape, torch.zeros(L, d, dtype=BF), torch.zeros(d, E), None,
                         torch.zeros(L, K, dtype=torch.int64), torch.zeros(L, K))
    with pytest.raises(ValueError, match="topk_ids: shape"):
        B.dispatch_build(shape, torch.zeros(L * K, dtype=torch.int32))
    with pytest.raises(ValueError, match="topk_ids: must be a CUDA tensor"):
        B.dispatch_build(shape, torch.zeros(L, K, dtype=torch.int32))
