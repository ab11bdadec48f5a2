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


def test_compared_maxima_keys_and_gqa_mapping():
    """Each (query head, threshold index) collects the candidate block maxima of
    its own KV head (h // (Hq/Hkv)), with blocks past the table's end pooled
    under the last index; brute-force block maxima on a tiny case."""
    rng = np.random.default_rng(5)
    Hq, Hkv, L, d, B, sigma, nT = 4, 2, 20, 3, 4, 0.7, 3
    q, k = rng.standard_normal((Hq, L, d)), rng.standard_normal((Hkv, L, d))
    blocks = [(h, i) for h in range(Hq) for i in range(L // B)]
    got = guard.compared_maxima(q, k, Bq=B, Bk=B, sigma=sigma, nT=nT, blocks=blocks)
    assert sorted(got) == [(h, t) for h in range(Hq) for t in range(nT)]
    for h in range(Hq):
        kh = h // 2
        s = sigma * q[h] @ k[kh].T
        assert got[(h, 0)].size == 0  # query block 0 has no candidates
        for t in range(1, nT):
            expect = []
            for i in range(L // B):
                if min(i, nT - 1) != t:
                    continue
                for j in range(i):  # candidates of query block i: key blocks 0 .. i-1
                    expect.append(s[i * B:(i + 1) * B, j * B:(j + 1) * B].max())
            assert np.allclose(np.sort(got[(h, t)]), np.sort(expect), rtol=0, atol=1e-12)
