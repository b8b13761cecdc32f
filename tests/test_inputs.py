"""Pins of the seeded input generator (CPU)."""
import math

import numpy as np
import torch

from mixture_experts_atomic_gb300 import inputs as I


def test_splitmix64_published_sequence():
    # first outputs of SplitMix64 seeded with 1234567 (Vigna's splitmix64.c)
    ref = [6457827717110365317, 3203168211198807973, 9817491932198370423,
           4593380528125082431, 16408922859458223821]
    got = I.splitmix_from_state(1234567, torch.arange(5, dtype=torch.int64))
    assert [int(v) & I.MASK64 for v in got] == ref


def test_vectorised_generator_matches_int_definition():
    ctr = torch.tensor([0, 1, 2, 12345, 2**33 + 7, 2**40 - 1], dtype=torch.int64)
    got = I.bits(4, I.STREAM_X, ctr)
    ref = [I.splitmix_int(4, I.STREAM_X, int(c)) for c in ctr]
    assert [int(v) & I.MASK64 for v in got] == ref
    # numpy uint64 restatement agrees as well
    key = np.uint64(I.stream_key(4, I.STREAM_X))
    with np.errstate(over="ignore"):
        z = (ctr.numpy().astype(np.uint64) + np.uint64(1)) * np.uint64(I.GAMMA) + key
        z = (z ^ (z >> np.uint64(30))) * np.uint64(I.MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(I.MIX2)
        z = z ^ (z >> np.uint64(31))
    assert [int(v) for v in z] == ref


def test_uniform_open_interval_and_normal_moments():
    u = I.uniform(0, 1, torch.arange(1 << 18, dtype=torch.int64))
    assert float(u.min()) > 0.0 and float(u.max()) < 1.0
    assert abs(float(u.mean()) - 0.5) < 3e-3
    n = I.normal_block(0, 1, 0, (1 << 18,), "cpu")
    assert abs(float(n.mean())) < 1e-2 and abs(float(n.std()) - 1.0) < 1e-2


def test_rows_regenerate_block():
    cfg = I.CONFIGS[1].scaled(L=64)
    x = I.make_x(cfg)
    rows = torch.tensor([0, 5, 63])
    assert torch.equal(I.x_rows(cfg, rows), x[rows])
    dy = I.make_dy(cfg)
    assert torch.equal(I.dy_rows(cfg, rows), dy[rows])


def test_softmax_router_definition():
    cfg = I.CONFIGS[0].scaled(L=64)
    x = I.make_x(cfg)
    ids, gates = I.softmax_router(cfg, x)
    Wr = I.normal_block(cfg.seed, I.STREAM_WR, 0, (cfg.d, cfg.E), "cpu", 1 / math.sqrt(cfg.d),
                        torch.float32).double()
    lg = x.double() @ Wr
    p = torch.softmax(lg, 1)
    for t in range(cfg.L):
        order = sorted(range(cfg.E), key=lambda e: (-float(p[t, e]), e))[:cfg.K]
        assert ids[t].tolist() == order
        ref = p[t, order] / p[t, order].sum()
        assert torch.allclose(gates[t].double(), ref, rtol=1e-6)


def test_zipf_router_distinct_and_skewed():
    cfg = I.CONFIGS[4].scaled(L=20000)
    ids, gates = I.zipf_router(cfg)
    s = torch.sort(ids, 1).values
    assert bool((s[:, 1:] != s[:, :-1]).all())
    assert int(ids.min()) >= 0 and int(ids.max()) < cfg.E
    cnt = torch.bincount(ids.reshape(-1).long(), minlength=cfg.E)
    # expert 0 is the most popular and draws well above the mean
    assert int(cnt.argmax()) == 0 and float(cnt[0]) > 10 * float(cnt.float().mean())
    assert torch.allclose(gates.double().sum(1), torch.ones(cfg.L, dtype=torch.float64), atol=1e-6)
    assert float(gates.min()) > 0


def test_bias_router_skews_loads():
    cfg = I.CONFIGS[2].scaled(L=4096)
    ids, gates = I.make_routing(cfg)
    cnt = torch.bincount(ids.reshape(-1).long(), minlength=cfg.E).double()
    assert float(cnt.max() / cnt.mean()) > 3.0
