"""The index sampler behind the full-size parity checks (tests/gpu_util.py):
it must reach the first, a middle and the last output tile of each weight
gradient GEMM, with at least 32 picks on every full-size workload.  CPU only."""
import numpy as np

from gpu_util import spread_indices
from mixture_experts_atomic_gb300 import inputs as I


def test_spread_indices_covers_first_middle_last_tile():
    rng = np.random.default_rng(0)
    for cfg in I.CONFIGS[1:4]:
        for tile in (128, 256):
            idx = spread_indices(cfg.h, tile, 10, rng, extra=4)
            assert len(idx) >= 32 and len(set(idx)) == len(idx)
            assert all(0 <= i < cfg.h for i in idx)
            nt = (cfg.h + tile - 1) // tile
            tiles = {i // tile for i in idx}
            assert {0, nt // 2, nt - 1} <= tiles
            assert 0 in idx and cfg.h - 1 in idx


def test_spread_indices_small_extent():
    rng = np.random.default_rng(1)
    assert spread_indices(5, 128, 10, rng) == [0, 1, 2, 3, 4]
