"""The token-choice top-K softmax router (the step before the dispatch) and
its backward on the GPU, through the C ABI, against the CPU oracle.

Forward: the oracle ranks fp64 logits, the kernel fp32 logits.  Where the
oracle's K-th and (K+1)-th logits (or two selected logits) are further apart
than LOGIT_TOL the choice is unique and must match exactly; nearer than that
both choices are correct, and the kernel's is checked for validity.  On
integer-valued inputs the fp32 logits are exact, so ties must be broken like
the oracle's (lower expert index first) and the ids match bit for bit.
Backward: the kernel is fed the oracle's own selection; dWr, dbias and dx
are compared with max|gpu - ref| / max|ref| <= 1e-4 (fp32; 2e-2 for a bf16
dx, which is rounded once)."""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from mixture_experts_atomic_gb300 import binding as B
from mixture_experts_atomic_gb300 import inputs as I

pytestmark = pytest.mark.gpu

from gpu_util import ensure_built  # noqa: E402

LOGIT_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _shape(L, d, E, K, dtype):
    return B.make_shape(L, d, 128, E, K, B.BF16 if dtype == "bf16" else B.F32, "swiglu")


def _problem(L, d, E, K, dtype, seed, bias=True, integer=False):
    g = torch.Generator().manual_seed(seed)
    if integer:
        x = torch.randint(-2, 3, (L, d), generator=g).float()
        Wr = torch.randint(-1, 2, (d, E), generator=g).float()
        b = torch.randint(-2, 3, (E,), generator=g).float() if bias else None
    else:
        x = torch.randn(L, d, generator=g)
        Wr = torch.randn(d, E, generator=g) / d ** 0.5
        b = torch.randn(E, generator=g) if bias else None
    x = x.to(torch.bfloat16) if dtype == "bf16" else x
    return x, Wr, b


def _gpu_router(shape, x, Wr, b):
    L, K = shape.L, shape.K
    ids = torch.full((L, K), -1, dtype=torch.int32, device="cuda")
    gates = torch.full((L, K), float("nan"), dtype=torch.float32, device="cuda")
    B.router_forward(shape, x.cuda(), Wr.cuda(), None if b is None else b.cuda(), ids, gates)
    torch.cuda.synchronize()
    return ids.cpu().numpy().astype(np.int64), gates.cpu().numpy().astype(np.float64)


def _check_forward(gi, gg, x, Wr, b, K, gate_atol=2e-6):
    oi, og, lg = O.router(x, Wr, b, K)
    srt = -np.sort(-lg, axis=1)
    E = lg.shape[1]
    boundary = srt[:, K - 1] - srt[:, K] if K < E else np.full(len(lg), np.inf)
    inner = np.min(np.diff(-srt[:, :K], axis=1), axis=1) if K > 1 else np.full(len(lg), np.inf)
    unique = (boundary > LOGIT_TOL) & (inner > LOGIT_TOL)
    assert np.array_equal(gi[unique], oi[unique]), "ids differ where the choice is unique"
    np.testing.assert_allclose(gg[unique], og[unique], rtol=0, atol=gate_atol)
    # near ties: a valid choice - distinct experts within LOGIT_TOL of the K-th
    # largest logit, in non-increasing logit order, gates summing to 1
    for t in np.nonzero(~unique)[0]:
        sel = gi[t]
        assert len(set(sel.tolist())) == K and sel.min() >= 0 and sel.max() < E
        assert np.all(lg[t, sel] >= srt[t, K - 1] - LOGIT_TOL)
        assert np.all(np.diff(lg[t, sel]) <= LOGIT_TOL)
        assert abs(gg[t].sum() - 1.0) < 1e-5
    return int((~unique).sum())


@pytest.mark.parametrize("L,d,E,K,dtype", [
    (1000, 256, 5, 2, "bf16"),
    (3000, 512, 64, 6, "bf16"),
    (700, 128, 256, 8, "f32"),
    (333, 64, 12, 3, "f32"),
    (4100, 1024, 8, 2, "bf16"),
    (129, 192, 130, 1, "bf16"),
    (64, 64, 3, 3, "f32"),
])
def test_router_forward_matches_oracle(L, d, E, K, dtype):
    x, Wr, b = _problem(L, d, E, K, dtype, seed=L + E)
    gi, gg = _gpu_router(_shape(L, d, E, K, dtype), x, Wr, b)
    near = _check_forward(gi, gg, x, Wr, b, K)
    assert near <= max(2, L // 100)


@pytest.mark.parametrize("E,K", [(6, 2), (40, 5), (256, 8)])
def test_router_integer_inputs_break_ties_like_the_oracle(E, K):
    L, d = 2000, 64
    x, Wr, b = _problem(L, d, E, K, "bf16", seed=E, integer=True)
    gi, gg = _gpu_router(_shape(L, d, E, K, "bf16"), x, Wr, b)
    oi, og, lg = O.router(x, Wr, b, K)
    assert np.array_equal(gi, oi)
    np.testing.assert_allclose(gg, og, rtol=0, atol=2e-6)


@pytest.mark.parametrize("ci", [1, 2])
def test_router_forward_on_the_softmax_workloads(ci):
    cfg = I.CONFIGS[ci]
    x = I.make_x(cfg, "cpu")
    Wr, b = I.router_weights(cfg, "cpu")
    gi, gg = _gpu_router(_shape(cfg.L, cfg.d, cfg.E, cfg.K, cfg.dtype), x, Wr, b)
    near = _check_forward(gi, gg, x, Wr, b, cfg.K)
    assert near <= cfg.L // 100  # near ties are rare; each was checked for validity above


@pytest.mark.parametrize("L,d,E,K,dtype", [
    (1000, 256, 5, 2, "bf16"),
    (3000, 512, 64, 6, "f32"),
    (700, 128, 256, 8, "bf16"),
    (5000, 1024, 8, 2, "bf16"),
    (40, 64, 3, 3, "f32"),
    (2100, 1536, 12, 3, "f32"),   # <= 16 experts, one-pass kernel: fp32 x, 1.5 column blocks of 1024
    (1500, 2560, 16, 4, "bf16"),  # 16 experts, 2.5 column blocks
])
def test_router_backward_matches_oracle(L, d, E, K, dtype):
    x, Wr, b = _problem(L, d, E, K, dtype, seed=7 * L + E)
    oi, og, _ = O.router(x, Wr, b, K)
    dg = np.random.default_rng(L).standard_normal((L, K))
    dWr_r, db_r, dx_r, _ = O.router_backward(x, Wr, oi, og, dg, E)
    shape = _shape(L, d, E, K, dtype)
    dWr = torch.full((d, E), float("nan"), device="cuda")
    db = torch.full((E,), float("nan"), device="cuda")
    dx = torch.empty((L, d), dtype=x.dtype, device="cuda")
    B.router_backward(shape, x.cuda(), Wr.cuda(), torch.from_numpy(oi).int().cuda(),
                      torch.from_numpy(og).float().cuda(), torch.from_numpy(dg).float().cuda(), dWr, db, dx)
    torch.cuda.synchronize()
    assert O.rel_err(dWr, dWr_r) <= 1e-4
    assert O.rel_err(db, db_r) <= 1e-4
    assert O.rel_err(dx, dx_r) <= (2e-2 if dtype == "bf16" else 1e-4)
    # bitwise repeatable
    dWr2 = torch.empty_like(dWr)
    B.router_backward(shape, x.cuda(), Wr.cuda(), torch.from_numpy(oi).int().cuda(),
                      torch.from_numpy(og).float().cuda(), torch.from_numpy(dg).float().cuda(), dWr2, None, None)
    torch.cuda.synchronize()
    assert torch.equal(dWr, dWr2)


def test_router_empty_batch():
    shape = _shape(0, 64, 4, 2, "bf16")
    Wr = torch.randn(64, 4, device="cuda")
    dWr = torch.ones(64, 4, device="cuda")
    db = torch.ones(4, device="cuda")
    B.router_forward(shape, None, Wr, None, None, None)
    B.router_backward(shape, None, Wr, None, None, None, dWr, db, None)
    torch.cuda.synchronize()
    assert float(dWr.abs().sum()) == 0 and float(db.abs().sum()) == 0


@pytest.mark.parametrize("fused", [False, True])
def test_router_then_layer_training_step(fused):
    """router -> dispatch -> layer forward/backward (with gate gradients) ->
    router backward on the GPU, against the same composition of oracle
    functions.  The inputs keep every token's selection unique by a wide
    margin, so both sides route identically.  fused: the router and the
    dispatch in one call (MoELayer.route)."""
    L, d, h, E, K = 768, 256, 384, 8, 2
    cfg = I.MoEConfig("t_router_step", L, d, h, E, K, "swiglu", "bf16", 21, "softmax")
    inp = I.make_inputs(cfg, "cpu")
    Wr = torch.from_numpy(np.random.default_rng(3).standard_normal((d, E)).astype(np.float32) * 0.5)
    b = torch.linspace(-0.3, 0.3, E)
    oi, og, lg = O.router(inp["x"], Wr, b, K)
    srt = -np.sort(-lg, axis=1)
    assert np.min(srt[:, K - 1] - srt[:, K]) > 1e-3 and np.min(srt[:, 0] - srt[:, 1]) > 1e-3
    shape = B.make_shape(L, d, h, E, K, B.BF16, "swiglu")
    ids = torch.empty((L, K), dtype=torch.int32, device="cuda")
    gates = torch.empty((L, K), dtype=torch.float32, device="cuda")
    x = inp["x"].cuda()
    from mixture_experts_atomic_gb300.layer import MoELayer
    layer = MoELayer.for_config(cfg, "cuda")
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    if fused:
        ids, gates = layer.route(x, Wr.cuda(), b.cuda())
        layer.forward(x, gates, dev["W1"], dev["W2"], dev["W3"])
        layer.backward(dev["dY"], x, gates, dev["W1"], dev["W2"], dev["W3"])
    else:
        B.router_forward(shape, x, Wr.cuda(), b.cuda(), ids, gates)
        dev["ids"], dev["gates"] = ids, gates
        layer.step(dev)
    dWr = torch.empty((d, E), device="cuda")
    db = torch.empty((E,), device="cuda")
    dxr = torch.empty((L, d), dtype=torch.bfloat16, device="cuda")
    B.router_backward(shape, x, Wr.cuda(), ids, gates, layer.dgates, dWr, db, dxr)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert np.array_equal(ids.cpu().numpy(), oi)
    a = {k: inp[k] for k in ("x", "W1", "W2", "W3", "dY")}
    y = O.forward(oi, og, a["x"], a["W1"], a["W2"], a["W3"], "swiglu", E=E)
    dX, dW1, dW2, dW3, dg = O.backward(oi, og, a["x"], a["dY"], a["W1"], a["W2"], a["W3"], "swiglu", E=E)
    dWr_r, db_r, dxr_r, _ = O.router_backward(a["x"], Wr, oi, og, dg, E)
    assert O.rel_err(layer.y, y) <= 2e-2 and O.rel_err(layer.dX, dX) <= 2e-2
    assert O.rel_err(layer.dgates, dg) <= 2e-2
    assert O.rel_err(dWr, dWr_r) <= 2e-2 and O.rel_err(db, db_r) <= 2e-2 and O.rel_err(dxr, dxr_r) <= 2e-2
