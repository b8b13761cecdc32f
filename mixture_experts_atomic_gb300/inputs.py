"""Seeded synthetic inputs for the MoE layer: the five workload shapes, the
counter-based random generator and the router that turns random logits into
top-K expert ids and gates.

This module holds none of the layer's own arithmetic (no dispatch, no expert
MLP, no combine, no gradient).  It is the one piece of code that both the
CUDA path's callers (tests, bench) and the CPU oracle's callers use, so that
both sides see the very same tensors.

Generator
---------
Every random number is a pure function of (seed, stream, counter):

* ``key  = mix64((seed << 32 | stream) + GAMMA)``
* ``z(i) = mix64(key + (i + 1) * GAMMA)``  (mod 2**64)

where ``mix64`` is the SplitMix64 output function and ``GAMMA`` its
increment (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the constants are those of Vigna's public
``splitmix64.c``).  ``z(i)`` is the (i+1)-th SplitMix64 output from state
``key``, so any element can be regenerated on its own, on any device.

* uniform in (0,1): ``u = ((z >> 11) + 0.5) * 2**-53``
* normal: Box-Muller on the uniforms at counters 2i and 2i+1,
  ``n = sqrt(-2 ln u1) * cos(2 pi u2)`` (fp64)

Streams: x 1, router weight 2, router bias 3, W1 4, W2 5, W3 6, dY 7,
Zipf draws 8, Dirichlet draws 9.

The same code runs as torch int64 ops on the CPU or on a GPU (int64
multiplication wraps mod 2**64 on both).  Float results agree across devices
up to the last bit of fp64 ``log``/``cos``; ids and gates are computed once
and handed to both sides.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Sequence

import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

STREAM_X, STREAM_WR, STREAM_BIAS, STREAM_W1, STREAM_W2, STREAM_W3, STREAM_DY, \
    STREAM_ZIPF, STREAM_DIRICHLET = range(1, 10)


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit Python int as a signed int64 value."""
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (exact, the definition)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return mix64_int(((seed << 32) | stream) + GAMMA)


def splitmix_int(seed: int, stream: int, i: int) -> int:
    """z(i) as a Python int; the slow exact definition used to pin the
    vectorised versions."""
    return mix64_int(stream_key(seed, stream) + (i + 1) * GAMMA)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64_t(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _s64(MIX1)
    z = (z ^ _lsr(z, 27)) * _s64(MIX2)
    return z ^ _lsr(z, 31)


def splitmix_from_state(state: int, counters: torch.Tensor) -> torch.Tensor:
    """Output number counter+1 of SplitMix64 started from ``state``
    (bit patterns as int64)."""
    z = (counters + 1) * _s64(GAMMA) + _s64(state)
    return _mix64_t(z)


def bits(seed: int, stream: int, counters: torch.Tensor) -> torch.Tensor:
    """z(counter) for an int64 tensor of counters (bit pattern as int64)."""
    return splitmix_from_state(stream_key(seed, stream), counters)


def uniform(seed: int, stream: int, counters: torch.Tensor) -> torch.Tensor:
    """Uniform fp64 in the open interval (0,1) at the given counters."""
    v = _lsr(bits(seed, stream, counters), 11)
    return (v.to(torch.float64) + 0.5) * (2.0 ** -53)


def normal_at(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """Standard normal (fp64) number idx of a stream (Box-Muller)."""
    u1 = uniform(seed, stream, 2 * idx)
    u2 = uniform(seed, stream, 2 * idx + 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normal_block(seed: int, stream: int, start: int, shape: Sequence[int],
                 device, std: float = 1.0, out_dtype=torch.float64,
                 chunk: int = 1 << 24) -> torch.Tensor:
    """Normals number start, start+1, ... laid out row-major in ``shape``,
    times ``std``, rounded to ``out_dtype`` (fp64 -> out_dtype, RNE)."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=out_dtype, device=device)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        idx = torch.arange(start + c0, start + c1, dtype=torch.int64, device=device)
        v = normal_at(seed, stream, idx)
        if std != 1.0:
            v = v * std
        if out_dtype == torch.bfloat16:
            v = v.to(torch.float32)
        out[c0:c1] = v.to(out_dtype)
    return out.view(*shape)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    L: int
    d: int
    h: int
    E: int
    K: int
    act: str          # "swiglu" | "silu" | "identity"
    dtype: str        # "f32" | "bf16"
    seed: int
    router: str       # "softmax" | "softmax_bias" | "zipf"

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def scaled(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = [
    # tiny SwiGLU layer in fp32 (the oracle's exact-check size)
    MoEConfig("swiglu_f32_L512_d64_h128_E8_K2", 512, 64, 128, 8, 2, "swiglu", "f32", 0, "softmax"),
    # SiLU (non-gated) layer, bf16
    MoEConfig("silu_bf16_L16384_d1024_h4096_E8_K2", 16384, 1024, 4096, 8, 2, "silu", "bf16", 1, "softmax"),
    # fine-grained SwiGLU with skewed router bias, bf16
    MoEConfig("swiglu_bf16_L65536_d2048_h1408_E64_K6", 65536, 2048, 1408, 64, 6, "swiglu", "bf16", 2, "softmax_bias"),
    # Mixtral-like large-expert SwiGLU, bf16
    MoEConfig("swiglu_bf16_L262144_d4096_h14336_E8_K2", 262144, 4096, 14336, 8, 2, "swiglu", "bf16", 3, "softmax"),
    # dispatch + gather/combine stress with identity experts, Zipf ids, bf16
    MoEConfig("identity_bf16_L2097152_d6144_E256_K4", 2097152, 6144, 0, 256, 4, "identity", "bf16", 4, "zipf"),
]

ZIPF_S = 1.1
ROUTER_BIAS_VAR = 1.5


def x_rows(cfg: MoEConfig, rows: torch.Tensor, device="cpu") -> torch.Tensor:
    """Rows of x (by token index) in the config's dtype, regenerated on their
    own from the counter-based stream."""
    rows = rows.to(device=device, dtype=torch.int64)
    cols = torch.arange(cfg.d, dtype=torch.int64, device=device)
    idx = rows[:, None] * cfg.d + cols[None, :]
    v = normal_at(cfg.seed, STREAM_X, idx)
    return _round(v, cfg.torch_dtype)


def dy_rows(cfg: MoEConfig, rows: torch.Tensor, device="cpu") -> torch.Tensor:
    rows = rows.to(device=device, dtype=torch.int64)
    cols = torch.arange(cfg.d, dtype=torch.int64, device=device)
    idx = rows[:, None] * cfg.d + cols[None, :]
    v = normal_at(cfg.seed, STREAM_DY, idx)
    return _round(v, cfg.torch_dtype)


def _round(v: torch.Tensor, dt) -> torch.Tensor:
    if dt == torch.bfloat16:
        return v.to(torch.float32).to(torch.bfloat16)
    return v.to(dt)


def make_x(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    return normal_block(cfg.seed, STREAM_X, 0, (cfg.L, cfg.d), device, 1.0, cfg.torch_dtype)


def make_dy(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    return normal_block(cfg.seed, STREAM_DY, 0, (cfg.L, cfg.d), device, 1.0, cfg.torch_dtype)


def make_weights(cfg: MoEConfig, device="cpu") -> Dict[str, Optional[torch.Tensor]]:
    """W1, W2 ~ N(0, 1/d) of shape (E,d,h); W3 ~ N(0, 1/h) of shape (E,h,d).
    W2 is absent for SiLU experts, all three for identity experts."""
    dt = cfg.torch_dtype
    if cfg.act == "identity":
        return {"W1": None, "W2": None, "W3": None}
    sd, sh = 1.0 / math.sqrt(cfg.d), 1.0 / math.sqrt(cfg.h)
    W1 = normal_block(cfg.seed, STREAM_W1, 0, (cfg.E, cfg.d, cfg.h), device, sd, dt)
    W2 = (normal_block(cfg.seed, STREAM_W2, 0, (cfg.E, cfg.d, cfg.h), device, sd, dt)
          if cfg.act == "swiglu" else None)
    W3 = normal_block(cfg.seed, STREAM_W3, 0, (cfg.E, cfg.h, cfg.d), device, sh, dt)
    return {"W1": W1, "W2": W2, "W3": W3}


def softmax_router(cfg: MoEConfig, x: torch.Tensor, chunk: int = 1 << 15):
    """Router of the softmax configs: logits = x.Wr (+ bias), top-K by
    probability (ties to the lower expert index), gates = the top-K
    probabilities renormalised to sum 1.  fp64 arithmetic; ids int32 and
    gates fp32.  Wr ~ N(0, 1/d) rounded to fp32; bias ~ N(0, 1.5) (variance)."""
    dev = x.device
    Wr = normal_block(cfg.seed, STREAM_WR, 0, (cfg.d, cfg.E), dev,
                      1.0 / math.sqrt(cfg.d), torch.float32).to(torch.float64)
    bias = None
    if cfg.router == "softmax_bias":
        bias = normal_block(cfg.seed, STREAM_BIAS, 0, (cfg.E,), dev,
                            math.sqrt(ROUTER_BIAS_VAR), torch.float64)
    ids = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=dev)
    gates = torch.empty((cfg.L, cfg.K), dtype=torch.float32, device=dev)
    for r0 in range(0, cfg.L, chunk):
        r1 = min(cfg.L, r0 + chunk)
        lg = x[r0:r1].to(torch.float64) @ Wr
        if bias is not None:
            lg = lg + bias
        # stable descending sort keeps the lower index first among equal logits
        order = torch.sort(lg, dim=1, descending=True, stable=True).indices[:, :cfg.K]
        top = torch.gather(lg, 1, order)
        w = torch.exp(top - top[:, :1])
        ids[r0:r1] = order.to(torch.int32)
        gates[r0:r1] = (w / w.sum(dim=1, keepdim=True)).to(torch.float32)
    return ids, gates


def router_weights(cfg: MoEConfig, device="cpu"):
    """The router parameters of a softmax workload, as handed to a router
    kernel: Wr (d,E) fp32 ~ N(0, 1/d) (the values softmax_router uses) and,
    for the biased router, the bias (E) ~ N(0, 1.5) (variance) rounded to
    fp32; bias None otherwise."""
    Wr = normal_block(cfg.seed, STREAM_WR, 0, (cfg.d, cfg.E), device, 1.0 / math.sqrt(cfg.d), torch.float32)
    bias = None
    if cfg.router == "softmax_bias":
        bias = normal_block(cfg.seed, STREAM_BIAS, 0, (cfg.E,), device, math.sqrt(ROUTER_BIAS_VAR), torch.float32)
    return Wr, bias


def zipf_router(cfg: MoEConfig, device="cpu", chunk: int = 1 << 16):
    """K distinct ids per token drawn one after another without replacement
    from p_e ~ (e+1)^-s (renormalised over the experts not yet drawn; slot
    order = draw order), and Dirichlet(1) gates g_k = -ln U_k / sum_j -ln U_j."""
    E, K, L = cfg.E, cfg.K, cfg.L
    p = torch.arange(1, E + 1, dtype=torch.float64, device=device) ** (-ZIPF_S)
    p = p / p.sum()
    ids = torch.empty((L, K), dtype=torch.int32, device=device)
    gates = torch.empty((L, K), dtype=torch.float32, device=device)
    ar = torch.arange(E, device=device)
    for r0 in range(0, L, chunk):
        r1 = min(L, r0 + chunk)
        n = r1 - r0
        tok = torch.arange(r0, r1, dtype=torch.int64, device=device)
        chosen = torch.zeros((n, E), dtype=torch.bool, device=device)
        for k in range(K):
            u = uniform(cfg.seed, STREAM_ZIPF, tok * K + k)
            pm = torch.where(chosen, torch.zeros((), dtype=torch.float64, device=device), p)
            cum = torch.cumsum(pm, dim=1)
            target = u * cum[:, -1]
            ok = (cum > target[:, None]) & ~chosen
            # first expert whose cumulative mass passes the target; if rounding
            # left none, the last expert not yet drawn
            first = torch.where(ok.any(dim=1), ok.int().argmax(dim=1),
                                (E - 1) - (~chosen).flip(1).int().argmax(dim=1))
            ids[r0:r1, k] = first.to(torch.int32)
            chosen[torch.arange(n, device=device), first] = True
        uu = uniform(cfg.seed, STREAM_DIRICHLET,
                     tok[:, None] * K + torch.arange(K, device=device)[None, :])
        ex = -torch.log(uu)
        gates[r0:r1] = (ex / ex.sum(dim=1, keepdim=True)).to(torch.float32)
    del ar
    return ids, gates


def make_routing(cfg: MoEConfig, x: Optional[torch.Tensor] = None, device="cpu"):
    if cfg.router == "zipf":
        return zipf_router(cfg, device)
    if x is None:
        x = make_x(cfg, device)
    return softmax_router(cfg, x)


def make_inputs(cfg: MoEConfig, device="cpu", with_dy: bool = True) -> Dict[str, torch.Tensor]:
    """All inputs of one layer step: ids (L,K) int32, gates (L,K) fp32,
    x (L,d), W1/W2 (E,d,h), W3 (E,h,d), dY (L,d) on ``device``."""
    x = make_x(cfg, device)
    ids, gates = make_routing(cfg, x, device)
    out = {"ids": ids, "gates": gates, "x": x}
    out.update(make_weights(cfg, device))
    if with_dy:
        out["dY"] = make_dy(cfg, device)
    return out


def random_routing(L: int, E: int, K: int, seed: int, device="cpu",
                   one_expert: Optional[int] = None):
    """Distinct top-K ids per token drawn uniformly (for edge-case shapes),
    with Dirichlet(1) gates; ``one_expert`` forces every token's first slot
    onto that expert."""
    tok = torch.arange(L, dtype=torch.int64, device=device)
    keys = uniform(seed, STREAM_ZIPF, tok[:, None] * E + torch.arange(E, device=device)[None, :])
    order = torch.argsort(keys, dim=1, stable=True)
    if one_expert is not None:
        # move one_expert to slot 0
        pos = (order == one_expert).int().argmax(dim=1)
        first = order[:, 0].clone()
        order[torch.arange(L, device=device), pos] = first
        order[:, 0] = one_expert
    ids = order[:, :K].to(torch.int32).contiguous()
    uu = uniform(seed, STREAM_DIRICHLET, tok[:, None] * K + torch.arange(K, device=device)[None, :])
    ex = -torch.log(uu)
    gates = (ex / ex.sum(dim=1, keepdim=True)).to(torch.float32)
    return ids, gates
