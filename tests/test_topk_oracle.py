"""Pins of the top-k oracle against things other than itself: library routines
on tie-free rows, hand-made tie / NaN / signed-zero cases, the defining
properties of the selection on tie-heavy rows, and a brute-force selection by
repeated first-occurrence arg-max on tiny rows."""
import numpy as np
import pytest

from oracle import topk as T


def _rank_key(v):
    """(class, value) used by the defining properties: NaN above every number, -0 == +0."""
    return (0 if np.isnan(v) else 1, 0.0 if np.isnan(v) else -float(v))


def test_tie_free_rows_match_argpartition_and_sort():
    rng = np.random.default_rng(1)
    for n, k in [(5000, 2048), (2048, 2048), (3000, 17), (100, 1)]:
        x = rng.permutation(np.arange(n, dtype=np.float32) * np.float32(0.37) - 50).astype(np.float32)
        idx, val = T.topk_row(x, k)
        ref_set = set(np.argpartition(-x, k - 1)[:k].tolist()) if k < n else set(range(n))
        assert set(idx.tolist()) == ref_set
        np.testing.assert_array_equal(val, np.sort(x)[::-1][:k])
        idx2, val2 = T.topk_row(x, k, "index")
        np.testing.assert_array_equal(idx2, np.sort(idx))


def test_all_equal_row_takes_the_first_positions():
    x = np.full(5000, 1.25, np.float32)
    for order in ("score", "index"):
        idx, val = T.topk_row(x, 2048, order)
        np.testing.assert_array_equal(idx, np.arange(2048))
        assert np.all(val == 1.25)


def test_ties_at_the_threshold_go_to_lower_positions():
    x = np.array([3, 5, 3, 5, 3, 5, 3, 5, 3, 5, 9], np.float32)
    idx, val = T.topk_row(x, 7)
    # 9, then the five 5s by position, then the first 3
    np.testing.assert_array_equal(idx, [10, 1, 3, 5, 7, 9, 0])
    np.testing.assert_array_equal(val, [9, 5, 5, 5, 5, 5, 3])
    idx, _ = T.topk_row(x, 7, "index")
    np.testing.assert_array_equal(idx, [0, 1, 3, 5, 7, 9, 10])


def test_nan_ranks_above_every_number_and_signed_zeros_tie():
    x = np.array([1.0, np.nan, np.inf, -np.nan, 0.0, -0.0, -np.inf], np.float32)
    idx, val = T.topk_row(x, 5)
    np.testing.assert_array_equal(idx, [1, 3, 2, 0, 4])
    assert np.isnan(val[0]) and np.isnan(val[1]) and val[2] == np.inf
    idx, _ = T.topk_row(np.array([-0.0, 0.0, -0.0], np.float32), 2)
    np.testing.assert_array_equal(idx, [0, 1])


def test_short_rows_are_padded():
    idx, val = T.topk_row(np.array([2.0, 7.0, -1.0], np.float32), 6)
    np.testing.assert_array_equal(idx, [1, 0, 2, -1, -1, -1])
    np.testing.assert_array_equal(val[:3], [7, 2, -1])
    assert np.all(val[3:] == -np.inf)
    idx, val = T.topk_row(np.zeros(0, np.float32), 3)
    assert np.all(idx == -1)


def test_lengths_restrict_each_row():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((4, 300)).astype(np.float32)
    s[:, 250:] = 1e9  # beyond the causal length: must never be picked
    lengths = [250, 10, 1, 0]
    idx, _ = T.topk(s, lengths, 20, "index")
    for q, n in enumerate(lengths):
        sel = idx[q][idx[q] >= 0]
        assert sel.size == min(20, n) and np.all(sel < n)


@pytest.mark.parametrize("seed", range(6))
def test_defining_properties_on_tie_heavy_rows(seed):
    rng = np.random.default_rng(10 + seed)
    n = int(rng.integers(1, 6000))
    k = int(rng.integers(1, 3000))
    # few distinct values: massive ties, plus some NaN and signed zeros
    x = rng.integers(-4, 5, n).astype(np.float32) * np.float32(0.5)
    x[rng.random(n) < 0.01] = np.nan
    x[rng.random(n) < 0.05] = -0.0
    idx, val = T.topk_row(x, k)
    take = min(n, k)
    sel = idx[:take]
    assert len(set(sel.tolist())) == take and np.all(idx[take:] == -1)
    unsel = np.setdiff1d(np.arange(n), sel)
    keys_sel = [_rank_key(x[i]) for i in sel]
    # order="score": non-decreasing key, ties by increasing position
    for a in range(take - 1):
        ka, kb = keys_sel[a], keys_sel[a + 1]
        assert ka < kb or (ka == kb and sel[a] < sel[a + 1])
    if unsel.size and take:
        worst = max(keys_sel)
        for i in unsel:
            ku = _rank_key(x[i])
            # nothing left out ranks above the worst selected; at equal rank the selected positions come first
            assert ku >= worst
            if ku == worst:
                assert i > max(s for s, kk in zip(sel, keys_sel) if kk == worst)
    idx2, _ = T.topk_row(x, k, "index")
    np.testing.assert_array_equal(idx2[:take], np.sort(sel))


def _brute_force(x, k):
    """Repeated arg-max with first occurrence, NaN above every number."""
    left = list(range(x.size))
    out = []
    for _ in range(min(k, x.size)):
        nan_pos = [i for i in left if np.isnan(x[i])]
        if nan_pos:
            best = nan_pos[0]
        else:
            vals = np.array([x[i] for i in left], dtype=np.float64)
            best = left[int(np.argmax(vals))]  # argmax returns the first occurrence; -0 == +0
        out.append(best)
        left.remove(best)
    return out


def test_brute_force_on_tiny_rows():
    rng = np.random.default_rng(3)
    for _ in range(300):
        n = int(rng.integers(0, 9))
        k = int(rng.integers(1, 10))
        x = rng.choice(np.array([0.0, -0.0, 1.0, 2.0, -1.0, np.nan, np.inf], np.float32), n)
        idx, _ = T.topk_row(x, k)
        assert idx[:min(n, k)].tolist() == _brute_force(x, k)
