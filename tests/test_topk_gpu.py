"""Deterministic top-k on the GPU against the oracle: positions and scores must
be identical (integer / bit-exact work, no tolerance), for tie-heavy indexer
scores, adversarial rows (all equal, ascending, descending, NaN / signed zeros /
infinities), ragged and short rows, every k edge, both output orders, the
full-size workload (sampled rows, plus properties of every row) and run-to-run
bit identity."""
import numpy as np
import pytest
import torch

from oracle import topk as otopk
from rl_post_loss_gb300 import build as nvbuild
from rl_post_loss_gb300 import capi, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nvbuild.build()
    capi.load()


def _run_and_check(scores, lengths, k, order, rows_to_check=None):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, val = capi.topk(scores, k, lengths=lengths, order=order, device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    gi, gv = idx.cpu().numpy(), val.cpu().numpy()
    s = scores.cpu().numpy()
    ln = None if lengths is None else lengths.cpu().numpy()
    rows = range(s.shape[0]) if rows_to_check is None else rows_to_check
    for q in rows:
        n = s.shape[1] if ln is None else int(ln[q])
        ri, rv = otopk.topk_row(s[q, :n], k, order)
        np.testing.assert_array_equal(gi[q], ri, err_msg=f"row {q} positions")
        np.testing.assert_array_equal(gv[q].view(np.int32), rv.view(np.int32), err_msg=f"row {q} scores")
    return idx, val


@pytest.mark.parametrize("order", ["score", "index"])
def test_indexer_scores_small(order):
    b = synthetic.make_topk_batch("cuda", **{k: v for k, v in synthetic.TOPK_SMALL.items() if k != "name"})
    _run_and_check(b.scores, b.lengths, b.k, order)


@pytest.mark.parametrize("context", [12000, 40000])
@pytest.mark.parametrize("k", [1, 2, 7, 100, 2047, 2048, 2049, 4096])
def test_every_k(k, context):
    b = synthetic.make_topk_batch("cuda", rows=6, context=context, k=k, seed=3)
    _run_and_check(b.scores, b.lengths, k, "score")


def test_ragged_short_and_empty_rows():
    b = synthetic.make_topk_batch("cuda", rows=12, context=9000, seed=4)
    b.lengths.copy_(torch.tensor([0, 1, 2, 100, 2047, 2048, 2049, 4095, 4096, 4097, 8999, 9000], dtype=torch.int32))
    for order in ("score", "index"):
        _run_and_check(b.scores, b.lengths, 2048, order)


def _adversarial_rows(n):
    rng = np.random.default_rng(5)
    rows = [
        np.full(n, 0.75, np.float32),                                # all equal
        np.arange(n, dtype=np.float32),                               # ascending: the bound rises every tile
        np.arange(n, dtype=np.float32)[::-1].copy(),                 # descending
        rng.integers(0, 3, n).astype(np.float32),                    # three values
        np.where(rng.random(n) < 0.5, np.float32(-0.0), np.float32(0.0)),  # signed zeros only
        rng.standard_normal(n).astype(np.float32),
    ]
    x = rng.standard_normal(n).astype(np.float32)
    x[rng.random(n) < 0.02] = np.nan
    x[rng.random(n) < 0.02] = np.inf
    x[rng.random(n) < 0.02] = -np.inf
    x[rng.random(n) < 0.05] = -0.0
    rows.append(x)
    nan_payloads = np.full(n, 1.0, np.float32)
    nan_payloads.view(np.uint32)[::97] = 0x7fc00001
    nan_payloads.view(np.uint32)[::89] = 0xffc12345
    rows.append(nan_payloads)
    nan_heavy = rng.standard_normal(n).astype(np.float32)  # enough NaN that a sampled bound admits NaN only
    nan_heavy[rng.random(n) < 0.3] = np.nan
    rows.append(nan_heavy)
    return np.stack(rows)


# Rows of 16384 scores or more start from a bound taken from a sample of the row; the ascending and
# descending rows put the sample's best scores where the row has fewer than k at or above them, so
# those rows are scanned a second time.
@pytest.mark.parametrize("n", [12004, 20004, 70004])
@pytest.mark.parametrize("order", ["score", "index"])
@pytest.mark.parametrize("k", [1, 2048, 4096])
def test_adversarial_rows(n, order, k):
    s = torch.from_numpy(_adversarial_rows(n)).cuda()
    _run_and_check(s, None, k, order)


def test_long_ragged_rows():
    b = synthetic.make_topk_batch("cuda", rows=10, context=70000, seed=8)
    b.lengths.copy_(torch.tensor([16383, 16384, 16385, 16387, 32769, 50001, 65537, 69999, 70000, 4097],
                                 dtype=torch.int32))
    for k in (1, 100, 2048, 4096):
        _run_and_check(b.scores, b.lengths, k, "score")


def test_unaligned_length_rejected_and_bad_lengths_flagged():
    with pytest.raises(capi.RlLossError):
        capi.topk(torch.zeros((2, 4095), device="cuda"), 16)  # a row stride of 4095 floats is not 16-byte aligned
    s = torch.zeros((2, 4096), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lengths = torch.tensor([5000, -3], dtype=torch.int32, device="cuda")
    idx, _ = capi.topk(s, 16, lengths=lengths, device_status=st)
    torch.cuda.synchronize()
    assert st.item() & (1 << capi.CODES["RL_ERR_SEQLENS"])
    assert bool((idx[1] == -1).all())


def test_repeated_calls_are_bit_identical():
    b = synthetic.make_topk_batch("cuda", rows=64, context=60000, seed=6)
    first = capi.topk(b.scores, b.k, lengths=b.lengths)
    for _ in range(3):
        again = capi.topk(b.scores, b.k, lengths=b.lengths)
        torch.cuda.synchronize()
        assert torch.equal(again[0], first[0]) and torch.equal(again[1].view(torch.int32), first[1].view(torch.int32))


@pytest.mark.slow
def test_full_size_sampled_rows_and_properties():
    b = synthetic.make_topk_batch("cuda")
    rng = np.random.default_rng(7)
    sample = sorted(set([0, b.rows - 1] + rng.choice(b.rows, 30, replace=False).tolist()))
    idx, val = _run_and_check(b.scores, b.lengths, b.k, "score", rows_to_check=sample)
    # every row: k distinct valid positions whose scores are the returned ones, in non-increasing order
    assert bool((idx >= 0).all()) and bool((idx < b.lengths[:, None]).all())
    srt = torch.sort(idx, dim=1).values
    assert bool((srt[:, 1:] != srt[:, :-1]).all())
    assert torch.equal(torch.gather(b.scores, 1, idx.long()).view(torch.int32), val.view(torch.int32))
    assert bool((val[:, :-1] >= val[:, 1:]).all())
    again = capi.topk(b.scores, b.k, lengths=b.lengths)
    torch.cuda.synchronize()
    assert torch.equal(again[0], idx)


# The final pass ranks the selection within buckets of the key's leading bits when the buckets
# are even enough (sum of squared sizes at most 128 per entry) and falls back to an exact select
# plus a separate sort otherwise. When every bucket holds a single key, the spare digit bits split
# the tied entries by position; rows with few distinct values tie heavily, so they take that split
# in score order and the separate sort in position order.
@pytest.mark.parametrize("distinct", [3, 40, 1000, 5000])
@pytest.mark.parametrize("order", ["score", "index"])
def test_few_distinct_values_long_rows(distinct, order):
    rng = np.random.default_rng(20 + distinct)
    n = 60004
    s = (rng.integers(0, distinct, (4, n)).astype(np.float32) * np.float32(0.25)) - np.float32(100.0)
    _run_and_check(torch.from_numpy(s).cuda(), None, 2048, order)


def _warp_skewed_row(n, nhigh, tiles, seed):
    """Standard normal scores, nhigh of them raised by 6 at positions that the first filter warp
    reads (offsets [0, 128) and [2048, 2176) of each 4096-score tile) within the given tiles."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n).astype(np.float32)
    cand = np.array([t * 4096 + o for t in tiles for o in list(range(128)) + list(range(2048, 2176))
                     if t * 4096 + o < n])
    x[rng.choice(cand, nhigh, replace=False)] += np.float32(6.0)
    return x


# Rows that start from the sampled bound append to warp-private regions of the buffer (320
# entries each). These rows put most of the kept scores on one warp's positions: its fill passes
# 288 at a check with room left, after which the row continues with the shared count (460 raised
# scores); and its region overflows with more than k scores at or above the bound (900 in 4 tiles
# that no sample run touches: the row is scanned again from the same bound), with fewer (1500 in
# the first 7 tiles: scanned again from -inf), and between two checks (250).
@pytest.mark.parametrize("order", ["score", "index"])
def test_rows_skewed_onto_one_warp(order):
    n = 200000
    rows = [_warp_skewed_row(n, 460, range(49), 31), _warp_skewed_row(n, 900, (1, 2, 4, 5), 33),
            _warp_skewed_row(n, 1500, range(7), 31), _warp_skewed_row(n, 250, range(49), 31)]
    _run_and_check(torch.from_numpy(np.stack(rows)).cuda(), None, 2048, order)


# k on both sides of the largest selection the bucket ranking orders (2560) and of the power of
# two the bitonic fallback pads to.
@pytest.mark.parametrize("k", [2559, 2560, 2561, 3000])
@pytest.mark.parametrize("order", ["score", "index"])
def test_k_around_the_bucket_limit(k, order):
    b = synthetic.make_topk_batch("cuda", rows=5, context=50000, k=k, seed=9)
    _run_and_check(b.scores, b.lengths, k, order)


@pytest.mark.slow
def test_full_size_repeated_launches_are_bit_identical():
    """Ten launches on the full workload (2 persistent CTAs per SM, every SM busy): the result must
    not depend on which CTA takes which row or on the timing of the tile copies."""
    b = synthetic.make_topk_batch("cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    i0, v0 = capi.topk(b.scores, b.k, lengths=b.lengths, device_status=st)
    for _ in range(10):
        i1, v1 = capi.topk(b.scores, b.k, lengths=b.lengths, device_status=st)
        torch.cuda.synchronize()
        assert torch.equal(i0, i1) and torch.equal(v0.view(torch.int32), v1.view(torch.int32))
    assert st.item() == 0
