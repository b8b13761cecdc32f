"""Dispatch build on the GPU vs the oracle: bit-exact index structures on the
five workload shapes and on edge cases; determinism; routing validation."""
import numpy as np
import pytest
import torch

from mixture_experts_atomic_gb300 import binding as B
from mixture_experts_atomic_gb300 import inputs as I
from mixture_experts_atomic_gb300.layer import MoELayer

pytestmark = pytest.mark.gpu

from gpu_util import check_dispatch, ensure_built  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _layer(L, E, K, dtype=torch.bfloat16, d=128, h=128, act="swiglu"):
    return MoELayer(L, d, h, E, K, dtype, act, "cuda")


@pytest.mark.parametrize("L,E,K,seed,one", [
    (1, 1, 1, 0, None), (5, 4, 2, 1, None), (1000, 8, 2, 2, None), (1024, 8, 2, 3, None),
    (1025, 16, 4, 4, None), (3000, 64, 6, 5, 3), (4096, 512, 8, 6, None), (2048, 3, 3, 7, None),
    (777, 256, 4, 8, 200), (70000, 32, 2, 9, 0),
    # chunk counts scanned by their own kernel (chunks x experts > 32768):
    (66000, 512, 4, 10, None),   # 65 chunks per expert, scalar runs
    (921000, 64, 2, 11, 5),      # 900 chunks: 4-wide vector runs, the last threads past the end
])
def test_dispatch_matches_oracle(L, E, K, seed, one):
    ids, _ = I.random_routing(L, E, K, seed, one_expert=one)
    layer = _layer(L, E, K)
    layer.dispatch(ids.cuda())
    torch.cuda.synchronize()
    check_dispatch(layer, ids, E)
    assert layer.device_error() == 0


@pytest.mark.parametrize("L,E,e", [(5000, 6, 4), (1057, 8, 7), (33, 16, 15), (1, 256, 255), (2081, 2, 1)])
def test_dispatch_every_token_on_one_expert(L, E, e):
    """Every token on expert e.  With e = E-1 a power of two minus one, the
    expert id has every low bit set, the same bits as the lanes past the last
    token of a ragged chunk: those lanes must not join the expert's group."""
    ids = torch.full((L, 1), e, dtype=torch.int32)
    layer = _layer(L, E, 1)
    layer.dispatch(ids.cuda())
    D1, D2, _, _ = check_dispatch(layer, ids, E)
    assert np.array_equal(D1, np.arange(L))
    assert D2.tolist() == [0] * (e + 1) + [L] * (E - e)
    assert layer.device_error() == 0


def test_dispatch_empty_input():
    layer = _layer(0, 4, 2)
    layer.dispatch(torch.empty((0, 2), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert layer.disp.expert_token_offsets[:5].tolist() == [0] * 5
    assert layer.meta()[0] == 0


@pytest.mark.parametrize("ci", [0, 1, 2, 3, 4])
def test_dispatch_workload_shapes(ci):
    cfg = I.CONFIGS[ci]
    dev = "cuda"
    if cfg.router == "zipf":
        ids, _ = I.make_routing(cfg, device=dev)
    else:
        x = I.make_x(cfg, dev)
        ids, _ = I.make_routing(cfg, x, device=dev)
        del x
    layer = _layer(cfg.L, cfg.E, cfg.K, cfg.torch_dtype, d=128, h=128, act="swiglu")
    layer.dispatch(ids)
    torch.cuda.synchronize()
    check_dispatch(layer, ids.cpu(), cfg.E)
    # a second build gives bitwise-identical outputs
    first = [t.clone() for t in B.index_views(layer.shape, layer.disp)]
    layer.dispatch(ids)
    for a, b in zip(first, B.index_views(layer.shape, layer.disp)):
        assert torch.equal(a, b)


def test_validation_reports_bad_routing():
    L, E, K = 2000, 8, 2
    ids, _ = I.random_routing(L, E, K, 3)
    bad = ids.clone()
    bad[17, 1] = E            # out of range
    layer = _layer(L, E, K)
    with pytest.raises(B.MoEBlazeError) as ei:
        layer.dispatch(bad.cuda(), validate=True)
    assert ei.value.status == B.ERR_BAD_ROUTING
    dup = ids.clone()
    dup[1500, 1] = dup[1500, 0]  # repeated within a token
    layer.dispatch(dup.cuda(), validate=False)
    assert layer.device_error() & 1
    layer.dispatch(ids.cuda(), validate=True)  # a clean build clears the word
    assert layer.device_error() == 0
    neg = ids.clone()
    neg[0, 0] = -3
    with pytest.raises(B.MoEBlazeError):
        layer.dispatch(neg.cuda(), validate=True)
