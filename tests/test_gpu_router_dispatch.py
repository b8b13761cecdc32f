"""moeblaze_router_dispatch_build: the router fused with the dispatch
build's first step, on the GPU through the C ABI.

The ids and gates are checked against the CPU oracle's router as the
stand-alone router's are (ids equal wherever the choice is unique, valid
choices at near ties, bit-exact ids and gates on integer inputs).  The
fused kernel forms the logits on the tensor cores, whose fp32 accumulation
of the d products rounds differently from a chain of fp32 FMAs; a softmax
gate moves by at most half the largest logit error (|dg_k| <= 2 g_k (1 -
g_k) max|dl|), and the gates are held to GATE_ATOL = 1e-5 absolute, ten
times inside the fp32 rule max|got - ref| <= 1e-4 max|ref| (gates <= 1).  The dispatch it
builds is checked bit for bit against moeblaze_dispatch_build run on the
ids it produced: the index structures and every metadata table.  Shapes
cover a partial last chunk, a partial last 128-token tile, K = 1, K = E,
E = 64 (the largest fused case) and the shapes that take the unfused path
(fp32 x, E > 64, fewer than 128 tokens)."""
import numpy as np
import pytest
import torch

from mixture_experts_atomic_gb300 import binding as B
from mixture_experts_atomic_gb300 import inputs as I

pytestmark = pytest.mark.gpu

from gpu_util import ensure_built  # noqa: E402
from test_gpu_router import _check_forward, _problem, _shape  # noqa: E402

GATE_ATOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _fused(shape, x, Wr, b):
    L, K = shape.L, shape.K
    ids = torch.full((L, K), -1, dtype=torch.int32, device="cuda")
    gates = torch.full((L, K), float("nan"), dtype=torch.float32, device="cuda")
    disp = B.router_dispatch_build(shape, x.cuda(), Wr.cuda(), None if b is None else b.cuda(), ids, gates)
    torch.cuda.synchronize()
    return ids, gates, disp


def _same_dispatch(shape, ids, disp):
    ref = B.dispatch_build(shape, ids)
    torch.cuda.synchronize()
    for a, r in zip(B.index_views(shape, disp), B.index_views(shape, ref)):
        assert torch.equal(a, r)
    ma, mr = B.meta_arrays(shape, disp), B.meta_arrays(shape, ref)
    assert ma[0] == mr[0]
    for a, r in zip(ma[1:], mr[1:]):
        assert torch.equal(a, r)
    mt = ma[0]
    E = shape.E
    tiles = lambda d: d.meta.view(torch.int32)[8 + 3 * E + 1:8 + 3 * E + 1 + mt]
    assert torch.equal(tiles(disp), tiles(ref))
    assert B.device_error(shape, disp) == 0


@pytest.mark.parametrize("L,d,E,K,dtype", [
    (1000, 256, 5, 2, "bf16"),     # one partial chunk, partial last tile
    (3000, 512, 64, 6, "bf16"),    # E = 64: the widest fused case
    (4100, 1024, 8, 2, "bf16"),    # 5 chunks, the last with 4 tokens
    (2048, 128, 16, 4, "bf16"),    # whole chunks
    (1537, 128, 3, 3, "bf16"),     # K = E
    (129, 256, 13, 1, "bf16"),     # K = 1, one full tile and one token
    (700, 128, 130, 8, "bf16"),    # E > 64: unfused path
    (333, 64, 12, 3, "f32"),       # fp32 x: unfused path
    (100, 128, 8, 2, "bf16"),      # fewer than 128 tokens: unfused path
])
def test_fused_router_dispatch_matches_router_and_dispatch(L, d, E, K, dtype):
    x, Wr, b = _problem(L, d, E, K, dtype, seed=L + 7 * E)
    shape = _shape(L, d, E, K, dtype)
    ids, gates, disp = _fused(shape, x, Wr, b)
    gi = ids.cpu().numpy().astype(np.int64)
    gg = gates.cpu().numpy().astype(np.float64)
    near = _check_forward(gi, gg, x, Wr, b, K, GATE_ATOL)
    assert near <= max(2, L // 100)
    _same_dispatch(shape, ids, disp)


@pytest.mark.parametrize("E,K", [(6, 2), (40, 5), (64, 8)])
def test_fused_router_integer_inputs_break_ties_like_the_oracle(E, K):
    import oracle.moe_oracle as O
    L, d = 2000, 128
    x, Wr, b = _problem(L, d, E, K, "bf16", seed=100 + E, integer=True)
    shape = _shape(L, d, E, K, "bf16")
    ids, gates, disp = _fused(shape, x, Wr, b)
    oi, og, lg = O.router(x, Wr, b, K)
    assert np.array_equal(ids.cpu().numpy().astype(np.int64), oi)
    np.testing.assert_allclose(gates.cpu().numpy().astype(np.float64), og, rtol=0, atol=2e-6)
    _same_dispatch(shape, ids, disp)


@pytest.mark.parametrize("ci", [1, 2, 3])
def test_fused_router_dispatch_on_the_softmax_workloads(ci):
    cfg = I.CONFIGS[ci]
    x = I.make_x(cfg, "cuda")
    Wr, b = I.router_weights(cfg, "cpu")
    shape = _shape(cfg.L, cfg.d, cfg.E, cfg.K, cfg.dtype)
    ids, gates, disp = _fused(shape, x, Wr, b)
    if cfg.L <= 65536:
        rows = torch.arange(cfg.L)
    else:
        # the oracle's router on a sample of the tokens (every token's ids go
        # through the dispatch comparison below)
        rows = torch.from_numpy(np.sort(np.random.default_rng(1).choice(cfg.L, 4096, replace=False)))
    near = _check_forward(ids.cpu()[rows].numpy().astype(np.int64), gates.cpu()[rows].numpy().astype(np.float64),
                          x[rows.cuda()].cpu(), Wr, b, cfg.K, GATE_ATOL)
    assert near <= len(rows) // 100
    _same_dispatch(shape, ids, disp)
