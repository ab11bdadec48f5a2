"""The guard band that keeps generated thresholds clear of block maxima."""
import math

import numpy as np

from oracle import guard


def test_nearest_clear_value_moves_off_ties():
    vals = np.array([1.0, 1.0005, 1.5, 3.0])
    y = guard.nearest_clear_value(1.0002, vals)
    assert np.min(np.abs(vals - y)) >= 1e-3
    assert abs(y - 0.99) < 1e-12  # below the smallest value is the nearest wide gap
    assert guard.nearest_clear_value(2.0, vals) == 2.0  # already clear


def test_guard_table_leaves_minus_inf_and_clears_band():
    rng = np.random.default_rng(0)
    T = np.array([[-math.inf, 0.5, 1.25]], dtype=np.float32)
    compared = {(0, 0): rng.standard_normal(50), (0, 1): np.array([0.5004, 2.0]),
                (0, 2): np.array([1.0, 1.5])}
    Tg, n, shift = guard.guard_thresholds(T, compared)
    assert Tg[0, 0] == -math.inf
    assert n == 1 and shift > 0
    for (h, t), v in compared.items():
        if math.isfinite(Tg[h, t]):
            assert np.min(np.abs(v - float(Tg[h, t]))) >= 1e-3


def test_guard_log_lambda_iterates_to_clear_value():
    def stats(x):  # statistics that do not depend on x
        return np.array([-2.0, -1.0004, 0.3])
    y, moves = guard.guard_log_lambda(-1.0, stats)
    assert moves >= 1 and np.min(np.abs(stats(y) - y)) >= 1e-3
