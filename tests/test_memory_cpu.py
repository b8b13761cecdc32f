"""Activation-memory accounting of bench.py on the CPU: the materialising
layer's retained bytes and this layer's (saved A/B plus index structures),
from the library's host-side size functions.  No GPU."""
import types

import bench
from mixture_experts_atomic_gb300 import binding as B
from mixture_experts_atomic_gb300 import inputs as I


def _cfg(L, d, h, E, K, act, dtype="bf16"):
    return I.MoEConfig(f"t_{act}_{L}", L, d, h, E, K, act, dtype, 0, "softmax")


def test_materialising_ffn_term_matches_the_pages_estimate():
    # MoEBlaze summary page, "问题与动机": at L = 2M tokens and h = 24576 the
    # first MLP's bf16 output is about 98 GB for one layer.  With K = 1 the
    # SiLU layer keeps a and SiLU(a), two such tensors, beside the routed x.
    L, d, h = 2_000_000, 6144, 24576
    silu = bench.materialising_bytes(_cfg(L, d, h, 8, 1, "silu"))
    ident = bench.materialising_bytes(_cfg(L, d, h, 8, 1, "identity"))
    ffn = (silu - ident) / 2
    assert abs(ffn / 1e9 - 98) < 1
    # the routed buffer is L*K*d elements
    assert ident == L * 1 * d * 2


def test_materialising_counts_per_activation():
    L, d, h, E, K = 1000, 256, 384, 8, 3
    routed = L * K * d * 2
    assert bench.materialising_bytes(_cfg(L, d, h, E, K, "identity")) == routed
    assert bench.materialising_bytes(_cfg(L, d, h, E, K, "silu")) == routed + 2 * L * K * h * 2
    assert bench.materialising_bytes(_cfg(L, d, h, E, K, "swiglu")) == routed + 5 * L * K * h * 2
    # fp32 doubles every term
    assert bench.materialising_bytes(_cfg(L, d, h, E, K, "swiglu", "f32")) == 2 * (routed + 5 * L * K * h * 2)


def _host_layer(cfg):
    """The buffers MoELayer allocates, on the host (only their sizes are read)."""
    sh = B.make_shape(cfg.L, cfg.d, cfg.h, cfg.E, cfg.K, cfg.torch_dtype, cfg.act)
    disp = B.alloc_dispatch(sh, "cpu")
    return types.SimpleNamespace(shape=sh, disp=disp)


def test_memory_report_retained_is_saved_plus_indices():
    # the Mixtral-like SwiGLU layer: A and B saved in bf16, padded to 128 rows
    # per expert, against the materialising layer's routed x and five
    # (L*K, h) tensors
    cfg = I.CONFIGS[3]
    layer = _host_layer(cfg)
    rep = bench.memory_report(cfg, layer, 0)
    LK = cfg.L * cfg.K
    rows = -(-(LK + 255 * cfg.E) // 256) * 256
    assert rep["saved_activation_bytes"] == 2 * rows * cfg.h * 2
    assert rep["index_bytes"] == 3 * LK * 4 + (cfg.E + 4) * 4 + B.moeblaze_dispatch_meta_bytes(layer.shape)
    assert rep["retained_fwd_to_bwd_bytes"] == rep["saved_activation_bytes"] + rep["index_bytes"]
    assert rep["materialising_retained_bytes"] == LK * cfg.d * 2 + 5 * LK * cfg.h * 2
    assert 2.6 < rep["materialising_over_retained"] < 2.7
    sc = rep["scratch_bytes"]
    assert rep["peak_activation_bytes"] == rep["retained_fwd_to_bwd_bytes"] + max(sc["forward"], sc["backward"])


def test_memory_report_identity_keeps_only_indices():
    cfg = I.CONFIGS[4]
    layer = _host_layer(cfg)
    rep = bench.memory_report(cfg, layer, 0)
    assert rep["saved_activation_bytes"] == 0
    assert rep["retained_fwd_to_bwd_bytes"] == rep["index_bytes"] < 0.11e9
    assert rep["materialising_retained_bytes"] == cfg.L * cfg.K * cfg.d * 2
    assert rep["scratch_bytes"]["forward"] == rep["scratch_bytes"]["backward"] == 0
