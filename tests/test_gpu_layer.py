"""Forward + backward of the layer on the GPU (through the C ABI) vs the CPU
oracle: whole-tensor parity at sizes the oracle finishes in seconds (several
tiles, ragged tails, skew, empty experts, K = 1, K = E), and sampled parity
at the full workload sizes in the launch configuration the bench times.
Tolerance: max|gpu - ref| / max|ref| <= 1e-4 (fp32) and 2e-2 (bf16)."""
import numpy as np
import pytest
import torch

from mixture_experts_atomic_gb300 import inputs as I

pytestmark = pytest.mark.gpu

from gpu_util import ensure_built, full_compare, sampled_compare  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _routed_inputs(cfg, seed, one_expert=None):
    inp = I.make_inputs(cfg, "cpu")
    ids, gates = I.random_routing(cfg.L, cfg.E, cfg.K, seed, one_expert=one_expert)
    inp["ids"], inp["gates"] = ids, gates
    return inp


def test_fp32_layer_full_size():
    cfg = I.CONFIGS[0]
    errs, _ = full_compare(cfg, I.make_inputs(cfg, "cpu"))
    assert errs["y"] <= 1e-4


@pytest.mark.parametrize("L,d,h,E,K,act,one", [
    (1000, 256, 384, 5, 2, "swiglu", None),   # h % 256 == 128: half-width tail tiles
    (1000, 256, 384, 5, 2, "silu", None),
    (2500, 128, 256, 16, 6, "swiglu", 3),     # skewed: expert 3 takes every token
    (700, 384, 128, 3, 3, "swiglu", None),    # K == E
    (130, 128, 128, 8, 2, "silu", None),      # tiny, experts with few or no tokens
    (4096, 512, 512, 4, 1, "swiglu", None),   # K = 1
    (3000, 256, 640, 12, 2, "silu", 0),
])
@pytest.mark.parametrize("recompute_h", [False, True])
def test_bf16_layer_small(L, d, h, E, K, act, one, recompute_h):
    """recompute_h: the layer keeps no H / Hg; the down projection and dW3
    recompute them from the saved A, B (its own GEMM variants)."""
    cfg = I.MoEConfig(f"t_{act}_{L}_{d}_{h}_{E}_{K}", L, d, h, E, K, act, "bf16", 11, "softmax")
    full_compare(cfg, _routed_inputs(cfg, 5, one), recompute_h=recompute_h)


@pytest.mark.parametrize("L,d,h,E,K,act,one", [
    (16384, 256, 256, 2, 2, "swiglu", None),  # dW1 || dW2 and dW3 in 256-row tiles
    (16384, 256, 384, 2, 2, "swiglu", None),  # h % 256 == 128: dW3's last wide tile is half empty
    (16384, 512, 256, 2, 2, "silu", None),    # dW1 alone (SiLU)
    (16384, 384, 256, 2, 1, "swiglu", None),  # d % 256 == 128: dW1 || dW2 keeps 128-row tiles, dW3 wide
    (24577, 256, 512, 3, 2, "swiglu", 1),     # skewed: expert 1 takes every token's first slot
    (6000, 512, 640, 5, 4, "swiglu", None),   # just above 4,096 rows per expert; d 512, h 640 (2.5 wide tiles)
    (4000, 768, 256, 6, 3, "silu", 2),        # 2,000 rows per expert: 128-row tiles still
    (13000, 512, 2048, 6, 3, "silu", None),   # down and dX wide too (32 k-blocks, 608+ tiles)
    (10000, 2048, 512, 4, 2, "swiglu", 1),    # up wide too (32 k-blocks), skewed
    (12000, 512, 2048, 5, 3, "swiglu", 4),    # down (stored H) and dX wide, skewed
])
@pytest.mark.parametrize("recompute_h", [False, True])
def test_bf16_layer_wide_tiles(L, d, h, E, K, act, one, recompute_h):
    """At least 4,096 routed rows per expert on average and output rows in
    multiples of 256 (of 128 for dW3): the weight-gradient stages run
    256-row tiles (two M=128 MMAs that share every B tile, one 512-column
    accumulator), with ragged expert segments; with 32+ k-blocks a tile and
    4+ tiles per SM the row stages (up, stored-H down, dX) do too;
    whole-tensor parity."""
    cfg = I.MoEConfig(f"t_wide_{act}_{L}_{d}_{h}_{E}_{K}", L, d, h, E, K, act, "bf16", 12, "softmax")
    full_compare(cfg, _routed_inputs(cfg, 6, one), recompute_h=recompute_h)


def test_bf16_layer_wide_row_stages_with_empty_experts():
    """13 of 16 experts get no token while the down projection and dX run
    256-row tiles (32 and 64 k-blocks, 640 tiles of 128 rows): the wide row
    tiles of the three used experts' segments, and zero weight gradients
    for the empty experts."""
    cfg = I.MoEConfig("t_wide_sparse_experts", 10000, 1024, 2048, 16, 2, "swiglu", "bf16", 15, "softmax")
    inp = I.make_inputs(cfg, "cpu")
    ids3, gates = I.random_routing(cfg.L, 3, cfg.K, 9, one_expert=2)
    used = torch.tensor([1, 7, 15], dtype=torch.int32)
    inp["ids"], inp["gates"] = used[ids3.long()].contiguous(), gates
    errs, layer = full_compare(cfg, inp)
    empty = [e for e in range(cfg.E) if e not in used.tolist()]
    assert float(layer.dW1[empty].float().abs().max()) == 0.0
    assert float(layer.dW3[empty].float().abs().max()) == 0.0


def test_bf16_layer_wide_row_stages_whole_tensor():
    """d = h = 4096 and enough rows for 16 tiles per SM: the up projection,
    the stored-H down projection and dX run 256-row tiles, dH runs as
    cluster pairs, and the weight gradients run 256-row tiles (6,667 rows
    per expert); every output compared whole with the oracle (about a
    minute of fp64 work on the host)."""
    cfg = I.MoEConfig("t_wide_rows_swiglu", 10000, 4096, 4096, 3, 2, "swiglu", "bf16", 31, "softmax")
    full_compare(cfg, _routed_inputs(cfg, 8))


@pytest.mark.parametrize("recompute_h", [False, True])
def test_bf16_layer_most_experts_empty(recompute_h):
    """60 of 64 experts (the last one among them) get no token: the weight
    gradient stages then run long stretches of tiles with no k-blocks on
    every CTA, which must still come out as zero gradients."""
    cfg = I.MoEConfig("t_swiglu_sparse_experts", 2048, 1024, 768, 64, 2, "swiglu", "bf16", 14, "softmax")
    inp = I.make_inputs(cfg, "cpu")
    ids4, gates = I.random_routing(cfg.L, 4, cfg.K, 7)
    used = torch.tensor([0, 9, 30, 41], dtype=torch.int32)
    inp["ids"], inp["gates"] = used[ids4.long()].contiguous(), gates
    errs, layer = full_compare(cfg, inp, recompute_h=recompute_h)
    empty = [e for e in range(cfg.E) if e not in used.tolist()]
    assert float(layer.dW1[empty].float().abs().max()) == 0.0
    assert float(layer.dW3[empty].float().abs().max()) == 0.0


def test_fp32_layer_other_shapes():
    cfg = I.MoEConfig("t_f32_silu", 333, 32, 48, 5, 3, "silu", "f32", 12, "softmax")
    full_compare(cfg, _routed_inputs(cfg, 6))


@pytest.mark.parametrize("dtype,K", [("bf16", 4), ("f32", 4), ("bf16", 3), ("bf16", 8)])
def test_identity_layer_small(dtype, K):
    cfg = I.MoEConfig("t_identity", 1500, 1024 if dtype == "bf16" else 512, 0, 16, K, "identity", dtype, 13, "zipf")
    inp = I.make_inputs(cfg, "cpu")
    full_compare(cfg, inp)


@pytest.mark.parametrize("L,d,E,K,dtype", [
    (2049, 1000, 64, 8, "bf16"),   # 2000-byte rows in chunks of 1024 + 976 bytes
    (999, 3000, 32, 3, "bf16"),    # 6000-byte rows in chunks of 2720, 2720, 560 bytes
    (777, 6144, 256, 4, "bf16"),   # the stress workload's row width: six 2 KB chunks
    (515, 1500, 8, 1, "f32"),      # K = 1, 6000-byte fp32 rows in one chunk
])
def test_identity_layer_ragged_chunks(L, d, E, K, dtype):
    """The identity gather/combine stages each window's routed rows in
    column chunks sized to the ring stage; rows whose width is not a multiple
    of the chunk end in a partial chunk, and the last window is partial."""
    cfg = I.MoEConfig("t_identity_chunks", L, d, 0, E, K, "identity", dtype, 17, "zipf")
    full_compare(cfg, I.make_inputs(cfg, "cpu"))


def test_empty_layer_zero_grads():
    from mixture_experts_atomic_gb300.layer import MoELayer
    layer = MoELayer(0, 128, 128, 4, 2, torch.bfloat16, "swiglu", "cuda")
    z = lambda *s: torch.randn(*s, device="cuda").to(torch.bfloat16)
    W1, W2, W3 = z(4, 128, 128), z(4, 128, 128), z(4, 128, 128)
    layer.dW1.fill_(1); layer.dW2.fill_(1); layer.dW3.fill_(1)
    ids = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    g = torch.empty((0, 2), dtype=torch.float32, device="cuda")
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    layer.step({"ids": ids, "gates": g, "x": x, "dY": x, "W1": W1, "W2": W2, "W3": W3})
    torch.cuda.synchronize()
    assert float(layer.dW1.float().abs().sum()) == 0 and float(layer.dW3.float().abs().sum()) == 0


@pytest.mark.parametrize("ci,recompute_h", [(1, False), (2, False), (3, False), (1, True), (2, True), (3, True)])
def test_workload_sampled(ci, recompute_h):
    errs, frac = sampled_compare(I.CONFIGS[ci], recompute_h=recompute_h)
    print(I.CONFIGS[ci].name, "recompute_h" if recompute_h else "", errs, frac)


@pytest.mark.parametrize("L,E,K,act", [(10000, 3, 2, "swiglu"), (7000, 6, 3, "silu")])
def test_paired_stages_sampled(L, E, K, act):
    """d = h = 4096 and enough rows for 16 tiles per SM: the dH, dX and
    stored-H down projections (64+ k-blocks) run as clusters of two CTAs that
    share the weight tiles (a shape the small whole-tensor cases do not
    reach); sampled rows, columns and every expert's weight gradients."""
    cfg = I.MoEConfig(f"t_paired_{act}", L, 4096, 4096, E, K, act, "bf16", 23, "softmax")
    errs, frac = sampled_compare(cfg)
    print(cfg.name, errs, frac)


def test_identity_workload_sampled():
    sampled_compare(I.CONFIGS[4], n_tok=64)


def test_step_pipeline_matches_plain_steps():
    """The pipelined runner (host inputs -> device, compute, device -> host,
    copies overlapped across steps) gives, for three different batches, the
    same y and dX bits as plain steps (K = 2: every reduction is
    order-independent)."""
    from mixture_experts_atomic_gb300.layer import MoELayer, StepPipeline
    cfg = I.MoEConfig("t_pipeline", 1000, 256, 384, 5, 2, "swiglu", "bf16", 31, "softmax")
    base = I.make_inputs(cfg, "cpu")
    W = tuple(base[k].cuda() for k in ("W1", "W2", "W3"))
    batches = []
    for i in range(3):
        ids, gates = I.random_routing(cfg.L, cfg.E, cfg.K, 40 + i)
        g = torch.Generator().manual_seed(50 + i)
        x = torch.randn(cfg.L, cfg.d, generator=g).to(torch.bfloat16)
        dY = torch.randn(cfg.L, cfg.d, generator=g).to(torch.bfloat16)
        batches.append({"x": x, "ids": ids, "gates": gates, "dY": dY})
    ref = MoELayer.for_config(cfg, "cuda", with_dgates=False)
    want = []
    for bt in batches:
        dev = {k: v.cuda() for k, v in bt.items()}
        dev.update(dict(zip(("W1", "W2", "W3"), W)))
        ref.step(dev)
        want.append((ref.y.cpu().clone(), ref.dX.cpu().clone()))
    layer = MoELayer.for_config(cfg, "cuda", with_dgates=False)
    host = [{k: v.pin_memory() for k, v in bt.items()} for bt in batches]
    outs = [(torch.empty((cfg.L, cfg.d), dtype=torch.bfloat16).pin_memory(),
             torch.empty((cfg.L, cfg.d), dtype=torch.bfloat16).pin_memory()) for _ in batches]
    StepPipeline(layer).run(host, outs, W)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    for (y, dx), (wy, wdx) in zip(outs, want):
        assert torch.equal(y, wy) and torch.equal(dx, wdx)


def test_malformed_arguments_are_refused_before_launch():
    """A CUDA tensor of the wrong shape, dtype or layout is refused by the
    binding before any kernel runs, and the layer stays usable."""
    from mixture_experts_atomic_gb300 import binding as B
    from mixture_experts_atomic_gb300.layer import MoELayer
    cfg = I.MoEConfig("t_args", 300, 128, 128, 4, 2, "silu", "bf16", 3, "softmax")
    inp = {k: v.cuda() for k, v in I.make_inputs(cfg, "cpu").items() if v is not None}
    layer = MoELayer.for_config(cfg, "cuda")
    layer.dispatch(inp["ids"])
    torch.cuda.synchronize()
    n0 = B.moeblaze_kernel_launches()
    with pytest.raises(ValueError, match="x: shape"):
        layer.forward(inp["x"][:, :64].contiguous(), inp["gates"], inp["W1"], None, inp["W3"])
    with pytest.raises(ValueError, match="gates: dtype"):
        layer.forward(inp["x"], inp["gates"].double(), inp["W1"], None, inp["W3"])
    with pytest.raises(ValueError, match="W3: must be contiguous"):
        layer.forward(inp["x"], inp["gates"], inp["W1"], None, inp["W3"].transpose(1, 2).contiguous().transpose(1, 2))
    with pytest.raises(ValueError, match="topk_ids: dtype"):
        layer.dispatch(inp["ids"].long())
    assert B.moeblaze_kernel_launches() == n0
    layer.step(inp)
    torch.cuda.synchronize()
    assert layer.device_error() == 0


@pytest.mark.parametrize("act,dtype,L,d,h,E", [
    ("swiglu", "bf16", 1000, 256, 384, 5),
    ("silu", "bf16", 1000, 256, 384, 5),
    ("swiglu", "f32", 1000, 256, 384, 5),
    ("identity", "bf16", 1000, 256, 0, 5),
    ("swiglu", "bf16", 10000, 1024, 2048, 4),  # 256-row tiles: down, dX, dW1 || dW2, dW3
])
def test_graph_step_matches_eager_step(act, dtype, L, d, h, E):
    """The whole step captured as one CUDA graph (GraphStep) and replayed on
    refilled inputs gives the same bits as eager steps (K = 2: every
    reduction is order-independent)."""
    from mixture_experts_atomic_gb300.layer import GraphStep, MoELayer
    cfg = I.MoEConfig("t_graph", L, d, h, E, 2, act, dtype, 33, "softmax")
    base = {k: (v.cuda() if v is not None else None) for k, v in I.make_inputs(cfg, "cpu").items()}
    eager = MoELayer.for_config(cfg, "cuda", with_dgates=False)
    layer = MoELayer.for_config(cfg, "cuda", with_dgates=False)
    inp = {k: (v.clone() if v is not None else None) for k, v in base.items()}
    g = GraphStep(layer, inp)
    for i in range(2):
        ids, gates = I.random_routing(cfg.L, cfg.E, cfg.K, 60 + i)
        gen = torch.Generator().manual_seed(70 + i)
        x = torch.randn(cfg.L, cfg.d, generator=gen).to(base["x"].dtype).cuda()
        new = dict(base, ids=ids.cuda(), gates=gates.cuda(), x=x)
        for k in ("ids", "gates", "x"):
            inp[k].copy_(new[k])
        g.replay()
        eager.step(new)
        torch.cuda.synchronize()
        assert layer.device_error() == 0 and eager.device_error() == 0
        assert torch.equal(layer.y, eager.y) and torch.equal(layer.dX, eager.dX)
        if act != "identity":
            assert torch.equal(layer.dW1, eager.dW1) and torch.equal(layer.dW3, eager.dW3)
