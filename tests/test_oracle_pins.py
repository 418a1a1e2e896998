"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

None of these re-types the oracle's formula: each checks a closed form, an
invariant, a hand-derived worked example, a special case, or the gradient
against finite differences of the loss, chosen so that a dropped term, a wrong
sign, a wrong index or a transposed operand in ``oracle/rl_loss_oracle.c``
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import BF16, F32, F64, LossParams

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _batch(logits, targets, logp_old, logp_infer, mask, cu, rewards):
    return dict(logits=np.ascontiguousarray(logits), targets=np.asarray(targets, np.int32),
                logp_old=np.asarray(logp_old, np.float32), logp_infer=np.asarray(logp_infer, np.float32),
                mask=np.asarray(mask, np.uint8), cu_seqlens=np.asarray(cu, np.int32),
                rewards_or_adv=np.asarray(rewards, np.float32))


def _row_logp(z, dtype=F64):
    """Oracle log-prob of every vocabulary entry of one row (target = v)."""
    V = z.shape[0]
    T = V
    b = _batch(np.tile(z, (T, 1)), np.arange(V), np.zeros(T), np.zeros(T), np.ones(T), [0, T], [1.0])
    p = LossParams(group_size=1, adv_mode=1)
    _, adv, w = oracle.seq_prep(b["cu_seqlens"], b["mask"], b["rewards_or_adv"], p)
    return oracle.rows(np.arange(T), b["logits"], dtype, V, b["targets"], b["logp_old"], b["logp_infer"],
                       b["mask"], b["cu_seqlens"], adv, w, p)


# ----------------------------------------------------------------------------- log-softmax / entropy

@pytest.mark.parametrize("V", [1, 2, 7, 4096])
def test_uniform_row_closed_form(V):
    out = _row_logp(np.zeros(V, np.float64)) if V <= 64 else None
    if out is None:  # large V: one row, one target
        b = _batch(np.zeros((1, V), np.float32), [3], [0], [0], [1], [0, 1], [1.0])
        p = LossParams(group_size=1, adv_mode=1)
        out = oracle.forward_backward(b, F32, V, p)
    np.testing.assert_allclose(out["logp"], -math.log(V), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["entropy"], math.log(V), rtol=0, atol=1e-12)


@pytest.mark.parametrize("a,b", [(0.0, 0.0), (0.3, -1.7), (5.0, -5.0), (-20.0, 3.0)])
def test_two_value_closed_form(a, b):
    out = _row_logp(np.array([a, b]))
    p0 = 1.0 / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(out["logp"][0], -math.log1p(math.exp(b - a)), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(out["logp"][1], -math.log1p(math.exp(a - b)), rtol=1e-13, atol=1e-14)
    h = -(p0 * math.log(p0) + (1 - p0) * math.log(1 - p0))
    np.testing.assert_allclose(out["entropy"][0], h, rtol=1e-12, atol=1e-14)


def test_logprobs_exponentiate_to_one_and_shift_invariance():
    rng = np.random.default_rng(1)
    z = rng.normal(0, 3, 300)
    out = _row_logp(z)
    assert abs(np.exp(out["logp"]).sum() - 1.0) < 1e-12
    out2 = _row_logp(z + 123.25)
    np.testing.assert_allclose(out2["logp"], out["logp"], rtol=0, atol=1e-11)
    np.testing.assert_allclose(out2["entropy"], out["entropy"], rtol=0, atol=1e-11)
    # the log-prob of entry v is attached to entry v (no off-by-one / transposition)
    order = np.argsort(z)
    assert np.all(np.diff(out["logp"][order]) >= 0)


def test_dominant_logit_and_entropy_bounds():
    z = np.zeros(50)
    z[17] = 1e4
    out = _row_logp(z)
    assert abs(out["logp"][17]) < 1e-300 + 1e-12
    assert abs(out["entropy"][0]) < 1e-12
    rng = np.random.default_rng(2)
    for V in (3, 40):
        for _ in range(5):
            o = _row_logp(rng.normal(0, 4, V))
            assert np.all(o["entropy"] >= -1e-15) and np.all(o["entropy"] <= math.log(V) + 1e-12)


def test_minus_infinity_logits_are_absent_entries():
    """A -inf logit has probability 0: the log-probs and the entropy of the other entries
    equal those of the row without it (0 log 0 = 0), and its own log-prob is -inf."""
    z = np.array([1.0, -np.inf, 0.5, -np.inf, 2.0, -3.0])
    keep = np.isfinite(z)
    full = _row_logp(z)
    part = _row_logp(z[keep])
    np.testing.assert_allclose(full["logp"][keep], part["logp"], rtol=0, atol=1e-15)
    assert np.all(full["logp"][~keep] == -np.inf)
    np.testing.assert_allclose(full["entropy"], part["entropy"][0], rtol=0, atol=1e-15)
    one = _row_logp(np.array([-np.inf, 4.0, -np.inf]))
    assert one["logp"][1] == 0.0 and np.all(one["entropy"] == 0.0)


def test_bf16_widening_is_exact():
    # bf16 bit patterns of 1.0, -2.5, 0.15625 and 3.0 (upper halves of binary32 words)
    bits = np.array([[0x3F80, 0xC020, 0x3E20, 0x4040]], np.uint16)
    vals = np.array([1.0, -2.5, 0.15625, 3.0])
    b = _batch(bits, [2], [0], [0], [1], [0, 1], [1.0])
    p = LossParams(group_size=1, adv_mode=1)
    out = oracle.forward_backward(b, BF16, 4, p)
    ref = vals[2] - math.log(np.exp(vals).sum())
    assert abs(out["logp"][0] - ref) < 1e-14


# ----------------------------------------------------------------------------- advantages / weights

@pytest.mark.parametrize("G,k", [(4, 1), (8, 3), (32, 16), (32, 31)])
def test_bernoulli_group_advantage_closed_form(G, k):
    R = np.zeros(G, np.float32)
    R[:k] = 1.0
    cu = np.arange(G + 1, dtype=np.int32)
    for unbiased in (0, 1):
        p = LossParams(group_size=G, adv_eps=0.0, std_unbiased=unbiased)
        _, adv, _ = oracle.seq_prep(cu, np.ones(G), R, p)
        mu = k / G
        sd = math.sqrt(k * (G - k) / (G * (G - 1))) if unbiased else math.sqrt(mu * (1 - mu))
        np.testing.assert_allclose(adv[:k], (1 - mu) / sd, rtol=1e-14)
        np.testing.assert_allclose(adv[k:], -mu / sd, rtol=1e-14)


def test_advantage_invariants():
    rng = np.random.default_rng(3)
    G, P = 8, 5
    R = rng.normal(size=G * P).astype(np.float32)
    cu = np.arange(G * P + 1, dtype=np.int32)
    p = LossParams(group_size=G, adv_eps=0.0)
    _, adv, _ = oracle.seq_prep(cu, np.ones(G * P), R, p)
    grp = adv.reshape(P, G)
    np.testing.assert_allclose(grp.sum(1), 0.0, atol=1e-12)            # centred per group
    np.testing.assert_allclose((grp ** 2).mean(1), 1.0, rtol=1e-12)    # unit population std
    # groups are consecutive responses: group 1's advantages depend on group 1 only
    R2 = R.copy()
    R2[:G] += 10.0
    _, adv2, _ = oracle.seq_prep(cu, np.ones(G * P), R2, p)
    np.testing.assert_array_equal(adv2[G:], adv[G:])
    # all-equal rewards: exactly zero advantage
    _, adv3, _ = oracle.seq_prep(cu[:G + 1], np.ones(G), np.full(G, 0.7, np.float32),
                                 LossParams(group_size=G))
    assert np.all(adv3 == 0.0)
    # adv_eps enters the denominator: (R - mean) / (std + eps)
    _, adv4, _ = oracle.seq_prep(cu[:3], np.ones(2), np.array([1, 0], np.float32),
                                 LossParams(group_size=2, adv_eps=0.5))
    np.testing.assert_allclose(adv4, [0.5, -0.5], rtol=1e-15)


def test_token_counts_and_weights_follow_mask_table():
    spec = json.load(open(os.path.join(GOLDEN, "mask_table.json")))
    seg_masks = [s["loss_mask"] for s in spec["segments"]]
    assert seg_masks == [1, 0, 0, 1]
    # response 0: the four segments of 5, 7, 3, 4 tokens; response 1: one fully masked segment
    mask = np.concatenate([np.full(n, m, np.uint8) for n, m in zip((5, 7, 3, 4), seg_masks)] +
                          [np.zeros(6, np.uint8)])
    cu = np.array([0, 19, 25], np.int32)
    n, _, w = oracle.seq_prep(cu, mask, np.array([0.3, -0.2], np.float32), LossParams(group_size=1, adv_mode=1))
    assert list(n) == [9, 0]
    np.testing.assert_allclose(w, [1.0 / (2 * 9), 0.0], rtol=1e-15)


# ----------------------------------------------------------------------------- the loss

def test_worked_example_golden():
    ex = json.load(open(os.path.join(GOLDEN, "eq1_worked_example.json")))
    ln = math.log
    lo = [ln(3 / 4) - ln(1.5), ln(1 / 4) - ln(0.9)]
    li = [lo[0] - ln(1.25), lo[1] - ln(0.8)]
    b = _batch(np.array([[0.0, ln(3)], [ln(3), 0.0]]), [1, 1], lo, li, [1, 1], [0, 1, 2], [1.0, 0.0])
    p = LossParams(group_size=2, adv_eps=0.0)
    out = oracle.forward_backward(b, F64, 2, p, want_dz=True)
    e = ex["expected"]
    assert abs(out["loss"] - e["loss"]) < 2e-6
    np.testing.assert_allclose(out["logp"], [ln(3 / 4), ln(1 / 4)], rtol=1e-14)
    h = -(0.25 * ln(0.25) + 0.75 * ln(0.75))
    np.testing.assert_allclose(out["entropy"], [h, h], rtol=1e-14)
    assert list(out["flags"] & 1) == e["pop_in_bounds"]
    assert list((out["flags"] >> 1) & 1) == e["clip_active"]
    np.testing.assert_allclose(out["g"], e["dlogp"], rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(out["dz"], e["dlogits"], rtol=1e-6, atol=1e-12)


def _onpolicy_batch(rng, lengths, V, adv, dtype=F64):
    """Random logits; logp_old = the oracle's own log-prob (fl32), logp_infer = logp_old."""
    T = sum(lengths)
    z = rng.normal(0, 2, (T, V))
    tg = rng.integers(0, V, T)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    b = _batch(z, tg, np.zeros(T), np.zeros(T), np.ones(T), cu, adv)
    p = LossParams(group_size=1, adv_mode=1)
    first = oracle.forward_backward(b, dtype, V, p)
    b["logp_old"] = first["logp"].astype(np.float32)
    b["logp_infer"] = b["logp_old"].copy()
    return b


def test_closed_form_on_policy_loss_is_minus_mean_advantage():
    rng = np.random.default_rng(4)
    lengths, A = [3, 7, 1, 5], [0.7, -1.3, 0.25, 2.0]
    b = _onpolicy_batch(rng, lengths, 33, A)
    p = LossParams(group_size=1, adv_mode=1)
    out = oracle.forward_backward(b, F64, 33, p)
    S = len(lengths)
    # r = exp(logp - fl32(logp)) = 1 up to the fp32 rounding of logp_old (|logp| < 8: 4.8e-7)
    assert abs(out["loss"] - (-sum(A) / S)) < 5e-7 * sum(map(abs, A))
    want_g = np.concatenate([np.full(n, -a / (S * n)) for n, a in zip(lengths, A)])
    np.testing.assert_allclose(out["g"], want_g, rtol=5e-7)
    assert np.all(out["flags"] & 1) and not np.any(out["flags"] & 2)


def test_closed_form_constant_rho():
    rng = np.random.default_rng(5)
    lengths, A = [4, 6], [1.5, -0.5]
    b = _onpolicy_batch(rng, lengths, 17, A)
    rho_in = np.array([1.3, 0.6, 1.9, 0.75, 1.1, 0.55, 1.0, 1.99, 0.51, 1.4])
    b["logp_infer"] = (b["logp_old"].astype(np.float64) - np.log(rho_in)).astype(np.float32)
    rho = np.exp(b["logp_old"].astype(np.float64) - b["logp_infer"].astype(np.float64))
    p = LossParams(group_size=1, adv_mode=1)
    out = oracle.forward_backward(b, F64, 17, p)
    want = -(A[0] * rho[:4].mean() + A[1] * rho[4:].mean()) / 2
    assert abs(out["loss"] - want) < 1e-6
    p1 = LossParams(group_size=1, adv_mode=1, pop_indicator=1)
    out1 = oracle.forward_backward(b, F64, 17, p1)
    assert abs(out1["loss"] - (-sum(A) / 2)) < 1e-6


def test_pop_out_of_bounds_contributes_exactly_zero_and_boundary_is_closed():
    rng = np.random.default_rng(6)
    b = _onpolicy_batch(rng, [5], 9, [1.0])
    B = oracle.thresholds_f32(2.0, 0.2, 0.28)[0]
    assert B == np.float32(math.log(2.0))
    d = np.array([1.0, -1.0, 0.0, 0.5, -0.5], np.float32)
    b["logp_infer"] = (b["logp_old"] - d).astype(np.float32)
    p = LossParams(group_size=1, adv_mode=1)
    out = oracle.forward_backward(b, F64, 9, p, want_dz=True)
    assert list(out["flags"] & 1) == [0, 0, 1, 1, 1]
    assert np.all(out["tok_obj"][:2] == 0.0) and np.all(out["g"][:2] == 0.0)
    assert np.all(out["dz"][:2] == 0.0) and np.all(out["dz"][2:].any(axis=1))
    # closed interval in fp32: d == fl32(ln 2) is in bounds, the next float up is out
    lo = np.float32(-1.0)
    for dd, want in ((B, True), (-B, True), (np.nextafter(B, np.float32(9)), False),
                     (np.nextafter(-B, np.float32(-9)), False)):
        li = np.float32(lo - dd)
        if np.float32(lo - li) == dd:
            assert oracle.pop_in_bounds(float(lo), float(li), 2.0) == want


@pytest.mark.parametrize("A,r,clipped,value", [
    (0.8, 1.5, True, 1.28), (-0.8, 1.5, False, 1.5), (0.8, 0.5, False, 0.5), (-0.8, 0.5, True, 0.8),
    (0.8, 1.1, False, 1.1), (-0.8, 0.9, False, 0.9), (0.0, 1.5, False, 0.0)])
def test_clip_sides(A, r, clipped, value):
    rng = np.random.default_rng(7)
    b = _onpolicy_batch(rng, [1], 12, [A])
    b["logp_old"] = (b["logp_old"] - np.float32(math.log(r))).astype(np.float32)
    b["logp_infer"] = b["logp_old"].copy()
    p = LossParams(group_size=1, adv_mode=1)
    out = oracle.forward_backward(b, F64, 12, p, want_dz=True)
    assert bool(out["flags"][0] & 2) == clipped
    np.testing.assert_allclose(out["tok_obj"][0], value * A, rtol=1e-6)
    if clipped or A == 0.0:
        assert out["g"][0] == 0.0 and np.all(out["dz"] == 0.0)
    else:
        np.testing.assert_allclose(out["g"][0], -A * r, rtol=1e-6)


def test_masked_rows_have_zero_gradient_and_do_not_count():
    rng = np.random.default_rng(8)
    V = 11
    b = _onpolicy_batch(rng, [6, 4], V, [1.0, -2.0])
    b["mask"] = np.array([1, 0, 0, 1, 1, 0, 1, 1, 0, 1], np.uint8)
    p = LossParams(group_size=1, adv_mode=1)
    out = oracle.forward_backward(b, F64, V, p, want_dz=True)
    assert list(out["n_tokens"]) == [3, 3]
    m = b["mask"].astype(bool)
    assert np.all(out["dz"][~m] == 0.0) and np.all(out["tok_obj"][~m] == 0.0)
    assert list((out["flags"] >> 2) & 1) == list((~m).astype(int))
    b2 = dict(b)
    z2 = b["logits"].copy()
    z2[~m] = rng.normal(0, 5, (int((~m).sum()), V))
    b2["logits"] = z2
    out2 = oracle.forward_backward(b2, F64, V, p)
    assert out2["loss"] == out["loss"]


def test_row_gradient_sums_to_zero_and_zero_advantage():
    rng = np.random.default_rng(9)
    b = _onpolicy_batch(rng, [5, 3], 21, [0.9, -0.4])
    b["logp_infer"] = (b["logp_old"] + rng.normal(0, 0.3, 8)).astype(np.float32)
    p = LossParams(group_size=1, adv_mode=1)
    out = oracle.forward_backward(b, F64, 21, p, want_dz=True)
    np.testing.assert_allclose(out["dz"].sum(1), 0.0, atol=1e-15)
    b["rewards_or_adv"] = np.zeros(2, np.float32)
    out0 = oracle.forward_backward(b, F64, 21, p, want_dz=True)
    assert out0["loss"] == 0.0 and np.all(out0["dz"] == 0.0)


def test_normalisation_invariants():
    """1/|y_i|: repeating a response's tokens leaves L unchanged; 1/S: repeating
    every group leaves L unchanged; L does not depend on the order of groups."""
    rng = np.random.default_rng(10)
    V, G = 13, 2
    lengths = [3, 5, 2, 4]
    T = sum(lengths)
    z = rng.normal(0, 2, (T, V))
    tg = rng.integers(0, V, T)
    lo = rng.normal(-2.5, 0.5, T).astype(np.float32)
    li = (lo + rng.normal(0, 0.3, T)).astype(np.float32)
    R = np.array([1, 0, 0.3, 0.9], np.float32)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    p = LossParams(group_size=G)
    base = oracle.forward_backward(_batch(z, tg, lo, li, np.ones(T), cu, R), F64, V, p)["loss"]
    # every response's tokens repeated twice
    idx = np.concatenate([np.tile(np.arange(cu[i], cu[i + 1]), 2) for i in range(4)])
    cu2 = np.concatenate([[0], np.cumsum(np.array(lengths) * 2)]).astype(np.int32)
    rep = oracle.forward_backward(_batch(z[idx], tg[idx], lo[idx], li[idx], np.ones(2 * T), cu2, R), F64, V, p)
    assert abs(rep["loss"] - base) < 1e-12
    # every group repeated (S doubles)
    idx2 = np.concatenate([np.arange(T), np.arange(T)])
    cu3 = np.concatenate([[0], np.cumsum(lengths + lengths)]).astype(np.int32)
    dup = oracle.forward_backward(_batch(z[idx2], tg[idx2], lo[idx2], li[idx2], np.ones(2 * T), cu3,
                                         np.concatenate([R, R])), F64, V, p)
    assert abs(dup["loss"] - base) < 1e-12
    # groups swapped
    order = np.concatenate([np.arange(cu[2], cu[4]), np.arange(cu[0], cu[2])])
    cu4 = np.concatenate([[0], np.cumsum(lengths[2:] + lengths[:2])]).astype(np.int32)
    sw = oracle.forward_backward(_batch(z[order], tg[order], lo[order], li[order], np.ones(T), cu4,
                                        np.concatenate([R[2:], R[:2]])), F64, V, p)
    assert abs(sw["loss"] - base) < 1e-12


def test_gradient_matches_finite_differences():
    """dL/dz of every entry against central differences of the oracle's own
    loss (catches sign, index and transposition mistakes in the backward)."""
    rng = np.random.default_rng(11)
    V, G = 7, 2
    lengths = [3, 2, 2, 1]
    T = sum(lengths)
    z = rng.normal(0, 1.5, (T, V))
    tg = rng.integers(0, V, T).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    R = np.array([1.0, 0.0, 0.2, 0.9], np.float32)
    p = LossParams(group_size=G)
    # exact log-probs, then move tokens onto chosen branches, away from every boundary
    b = _batch(z, tg, np.zeros(T), np.zeros(T), np.ones(T), cu, R)
    lp = oracle.forward_backward(b, F64, V, p)["logp"]
    ln_r = np.array([0.05, 0.6, -0.5, 0.1, -0.03, 0.4, -0.6, 0.0])  # r = e^{ln_r}
    lo = (lp - ln_r).astype(np.float32)
    li = (lo.astype(np.float64) - np.array([0.1, -0.2, 0.3, 1.2, 0.0, -0.4, 0.2, 0.05])).astype(np.float32)
    mask = np.array([1, 1, 1, 1, 0, 1, 1, 1], np.uint8)
    b = _batch(z, tg, lo, li, mask, cu, R)
    out = oracle.forward_backward(b, F64, V, p, want_dz=True)
    flags = out["flags"]
    assert (flags & 2).any() and not (flags & 1).all()  # some clipped, some popped
    h = 1e-6
    fd = np.zeros((T, V))
    for t in range(T):
        for v in range(V):
            zp, zm = z.copy(), z.copy()
            zp[t, v] += h
            zm[t, v] -= h
            Lp = oracle.forward_backward(_batch(zp, tg, lo, li, mask, cu, R), F64, V, p)["loss"]
            Lm = oracle.forward_backward(_batch(zm, tg, lo, li, mask, cu, R), F64, V, p)["loss"]
            fd[t, v] = (Lp - Lm) / (2 * h)
    scale = np.abs(out["dz"]).max()
    np.testing.assert_allclose(out["dz"], fd, rtol=1e-6, atol=1e-7 * scale)


def test_bad_target_is_excluded():
    z = np.zeros((2, 4))
    b = _batch(z, [5, 1], [-1.4, -1.4], [-1.4, -1.4], [1, 1], [0, 2], [1.0])
    p = LossParams(group_size=1, adv_mode=1)
    out = oracle.forward_backward(b, F64, 4, p, want_dz=True)
    assert out["flags"][0] & 8 and not out["flags"][1] & 8
    assert math.isnan(out["logp"][0]) and out["tok_obj"][0] == 0.0 and np.all(out["dz"][0] == 0.0)


def test_hyperparameters_match_the_page():
    hp = json.load(open(os.path.join(GOLDEN, "eq1_hyperparams.json")))
    p = LossParams(group_size=hp["group_size"])
    assert (p.beta, p.eps_low, p.eps_high) == (hp["beta"], hp["eps_low"], hp["eps_high"])
    from rl_post_loss_gb300 import synthetic
    for cid in (0, 1, 2):
        assert synthetic.CASES[cid]["beta"] == hp["beta"]
    assert (synthetic.EPS_LOW, synthetic.EPS_HIGH) == (hp["eps_low"], hp["eps_high"])


# ----------------------------------------------------------------------------- fused projection oracle

def test_projection_logits_exact_on_integer_inputs():
    """Small integers are exact in bf16 and their products and sums exact in
    float64: the projection must equal the integer matrix product."""
    rng = np.random.default_rng(12)
    hi = rng.integers(-8, 9, (5, 7))
    wi = rng.integers(-8, 9, (6, 7))
    to_bits = lambda a: (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    z = oracle.projection_logits(to_bits(hi), to_bits(wi))
    want = [[sum(int(hi[i, k]) * int(wi[j, k]) for k in range(7)) for j in range(6)] for i in range(5)]
    assert np.array_equal(z, np.array(want, np.float64))


def test_projection_gradients_match_finite_differences():
    """dL/dh and dL/dW of the fused-path oracle against central differences of
    its loss in every entry of h and W (catches a transposed or swapped operand)."""
    rng = np.random.default_rng(13)
    T, H, V = 6, 5, 7
    h = rng.normal(0, 1, (T, H))
    W = rng.normal(0, 0.5, (V, H))
    cu = np.array([0, 2, 4, 6], np.int32)
    tg = rng.integers(0, V, T).astype(np.int32)
    b = _batch(np.zeros((T, V)), tg, np.zeros(T), np.zeros(T), np.ones(T), cu, [0.7, -0.4, 1.1])
    p = LossParams(group_size=1, adv_mode=1)
    lp = oracle.projection_forward_backward_f64(h, W, b, p)["logp"]
    b["logp_old"] = (lp - np.array([0.05, -0.1, 0.3, 0.0, -0.02, 0.12])).astype(np.float32)
    b["logp_infer"] = (b["logp_old"].astype(np.float64) - rng.normal(0, 0.2, T)).astype(np.float32)
    out = oracle.projection_forward_backward_f64(h, W, b, p)
    hstep = 1e-6
    for name, X, grad in (("h", h, out["dh"]), ("W", W, out["dW"])):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += hstep
            Xm[idx] -= hstep
            args_p = (Xp, W) if name == "h" else (h, Xp)
            args_m = (Xm, W) if name == "h" else (h, Xm)
            fd[idx] = (oracle.projection_forward_backward_f64(*args_p, b, p)["loss"] -
                       oracle.projection_forward_backward_f64(*args_m, b, p)["loss"]) / (2 * hstep)
        np.testing.assert_allclose(grad, fd, rtol=1e-5, atol=1e-8 * np.abs(grad).max(), err_msg=name)


def _bf16_bits(x):
    """Round-to-nearest-even bf16 bit patterns of float values."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _projection_case(seed, T=40, H=24, V=37):
    rng = np.random.default_rng(seed)
    hb = _bf16_bits(rng.normal(0, 1, (T, H)))
    wb = _bf16_bits(rng.normal(0, 0.4, (V, H)))
    cu = np.array([0, 9, 17, 30, 40], np.int32)
    tg = rng.integers(0, V, T).astype(np.int32)
    b = _batch(np.zeros((T, V)), tg, np.zeros(T), np.zeros(T), (rng.random(T) > 0.2).astype(np.uint8), cu,
               [1.0, 0.0, 0.0, 1.0])
    p = LossParams(group_size=2)
    lp = oracle.projection_forward_backward(hb, wb, b, p)["logp"]
    b["logp_old"] = (lp - rng.normal(0, 0.15, T)).astype(np.float32)
    b["logp_infer"] = (b["logp_old"].astype(np.float64) - rng.normal(0, 0.3, T)).astype(np.float32)
    return hb, wb, b, p


def test_projection_rows_equal_the_whole_batch_oracle():
    """The row-subset oracle of the fused path (used at sizes where the whole
    batch cannot be formed) gives, on any subset of rows, the log-prob,
    entropy, flags, dL/dlogp and dL/dh of the whole-batch oracle, whose
    gradients are pinned by finite differences above. H != V, so a transposed
    W or a wrong row gather fails here."""
    hb, wb, b, p = _projection_case(31)
    full = oracle.projection_forward_backward(hb, wb, b, p)
    n, adv, w = oracle.seq_prep(b["cu_seqlens"], b["mask"], b["rewards_or_adv"], p)
    ids = np.array([3, 0, 39, 17, 22, 8, 30])
    sub = oracle.projection_rows(ids, hb, wb, b["targets"], b["logp_old"], b["logp_infer"], b["mask"],
                                 b["cu_seqlens"], adv, w, p, want_dh=True)
    for k in ("logp", "entropy", "g", "tok_obj"):
        np.testing.assert_allclose(sub[k], full[k][ids], rtol=1e-12, atol=1e-14, err_msg=k)
    assert np.array_equal(sub["flags"], full["flags"][ids])
    np.testing.assert_allclose(sub["dh"], full["dh"][ids], rtol=1e-12, atol=1e-14)
    assert np.abs(full["g"][ids]).min() >= 0 and np.count_nonzero(full["g"][ids]) >= 3


def test_projection_streamed_forward_and_dw_rows_equal_the_whole_batch_oracle():
    """The streamed forward (exact loss over every row without a [T, V] array)
    and the sampled dL/dW rows computed from its log-probs and dL/dlogp equal
    the whole-batch oracle, whose dL/dW is pinned by finite differences."""
    hb, wb, b, p = _projection_case(32)
    full = oracle.projection_forward_backward(hb, wb, b, p)
    st = oracle.projection_forward_stats(hb, wb, b, p, row_block=7)
    for k in ("logp", "entropy", "g", "tok_obj"):
        np.testing.assert_allclose(st[k], full[k], rtol=1e-12, atol=1e-14, err_msg=k)
    assert np.array_equal(st["flags"], full["flags"])
    assert abs(st["loss"] - full["loss"]) <= 1e-13 * abs(full["loss"])
    ids = np.array([0, 36, 5, 11, 20])
    h64, W64 = oracle.bf16_bits_to_f64(hb), oracle.bf16_bits_to_f64(wb)
    dw = oracle.projection_dw_rows(ids, h64, W64, b["targets"], st["logp"], st["g"])
    np.testing.assert_allclose(dw, full["dW"][ids], rtol=1e-10, atol=1e-14 * np.abs(full["dW"]).max())


def test_clip_active_vec_matches_the_scalar_rule_at_threshold_neighbours():
    """The vector clip decision (the checker of every clip bit) equals the
    scalar rule token by token, and both follow the strict one-sided
    inequalities at the fp32 thresholds and their fp32 neighbours."""
    eps_low, eps_high = 0.2, 0.28
    _, hi, lo = oracle.thresholds_f32(2.0, eps_low, eps_high)
    hi, lo = np.float32(hi), np.float32(lo)
    cases = []  # (logp, logp_old = 0 so that fl32(logp - logp_old) = logp exactly, adv)
    for thr in (hi, lo):
        for e in (thr, np.nextafter(thr, np.float32(np.inf)), np.nextafter(thr, np.float32(-np.inf))):
            for adv in (0.7, -0.7, 0.0):
                cases.append((np.float32(e), np.float32(0.0), adv))
    rng = np.random.default_rng(40)
    for _ in range(200):
        lo_ = np.float32(rng.normal(-2, 1))
        lp = np.float32(lo_ + np.float32(rng.normal(0, 0.4)))
        cases.append((lp, lo_, float(rng.choice([-1.3, 0.0, 0.4]))))
    lp = np.array([c[0] for c in cases], np.float32)
    lo_ = np.array([c[1] for c in cases], np.float32)
    adv = np.array([c[2] for c in cases], np.float64)
    vec = oracle.clip_active_vec(lp, lo_, adv, eps_low, eps_high)
    for k, (a, o, A) in enumerate(cases):
        assert int(vec[k]) == int(oracle.clip_active(float(a), float(o), A, eps_low, eps_high)), k
    assert vec[:18].reshape(2, 3, 3).tolist() == [
        # ln r at fl32(ln(1 + eps_high)), one ulp above, one ulp below; A = +0.7, -0.7, 0
        [[0, 0, 0], [1, 0, 0], [0, 0, 0]],
        # ln r at fl32(ln(1 - eps_low)), one ulp above, one ulp below
        [[0, 0, 0], [0, 0, 0], [0, 1, 0]]]


# ----------------------------------------------------------------------------- DIS, OPD, per-token advantages

def _tok_batch(rng, lengths, V, token_adv=None):
    b = _onpolicy_batch(rng, lengths, V, [0.0] * len(lengths))
    if token_adv is not None:
        b["token_adv"] = np.asarray(token_adv, np.float32)
    return b


def test_dis_closed_form_at_r_one_and_token_mean():
    rng = np.random.default_rng(20)
    lengths = [3, 5, 2]
    A = rng.normal(0, 1, 10).astype(np.float32)
    b = _tok_batch(rng, lengths, 19, A)
    b["logp_infer"] = b["logp_old"].copy()  # the rollout log-prob: r = 1 up to fp32 rounding
    p = LossParams(group_size=1, adv_mode=2, objective=1, loss_norm=1)
    out = oracle.forward_backward(b, F64, 19, p)
    want = -float(np.mean(A.astype(np.float64) * out["logp"]))
    assert abs(out["loss"] - want) < 1e-6 * np.abs(A).sum()
    np.testing.assert_allclose(out["g"], -A / 10.0, rtol=1e-6)  # stop-gradient reading: -f A / N
    assert np.all(out["flags"] & 1)


def test_dis_gate_is_open_interval_and_sign_free():
    rng = np.random.default_rng(21)
    b = _tok_batch(rng, [6], 11, [0.5, -0.5, 0.5, -0.5, 0.5, -0.5])
    r = np.array([1.5, 1.5, 0.7, 0.7, 1.1, 0.9])
    b["logp_infer"] = (b["logp_old"].astype(np.float64) - np.log(r)).astype(np.float32)
    p = LossParams(group_size=1, adv_mode=2, objective=1, loss_norm=1)
    out = oracle.forward_backward(b, F64, 11, p, want_dz=True)
    assert list(out["flags"] & 1) == [0, 0, 0, 0, 1, 1]  # outside on both sides whatever the sign of A
    assert np.all(out["dz"][:4] == 0.0) and np.all(out["tok_obj"][:4] == 0.0)
    # the interval is open: ln r exactly at fl32(ln 1.28) or fl32(ln 0.8) is outside
    hi, lo = oracle.thresholds_f32(2.0, 0.2, 0.28)[1:]
    b1 = _tok_batch(rng, [1], 4, [1.0])
    b1["logits"] = np.array([[5.0, 0.0, 0.0, 0.0]])
    b1["targets"] = np.array([0], np.int32)
    lp32 = np.float32(oracle.forward_backward(b1, F64, 4, p)["logp"][0])
    checked = 0
    for e, inside in ((hi, False), (lo, False), (np.nextafter(hi, np.float32(0)), True),
                      (np.nextafter(lo, np.float32(0)), True)):
        li = np.float32(lp32 - e)
        if np.float32(lp32 - li) != e:
            continue  # this e is not reachable from lp32 by one fp32 subtraction
        b1["logp_infer"] = np.array([li], np.float32)
        assert bool(oracle.forward_backward(b1, F64, 4, p)["flags"][0] & 1) == inside, (e, inside)
        checked += 1
    assert checked >= 2


def test_dis_full_autodiff_gradient_matches_finite_differences():
    rng = np.random.default_rng(22)
    V, lengths = 6, [3, 2]
    T = sum(lengths)
    z = rng.normal(0, 1.5, (T, V))
    tg = rng.integers(0, V, T).astype(np.int32)
    cu = np.array([0, 3, 5], np.int32)
    A = np.array([0.7, -1.2, 0.4, 1.5, -0.3], np.float32)
    b = _batch(z, tg, np.zeros(T), np.zeros(T), np.ones(T), cu, [0.0, 0.0])
    b["token_adv"] = A
    p = LossParams(group_size=1, adv_mode=2, objective=1, loss_norm=1, dis_stopgrad=0)
    lp = oracle.forward_backward(b, F64, V, p)["logp"]
    b["logp_infer"] = (lp - np.array([0.05, -0.1, 0.15, 0.6, -0.02])).astype(np.float32)  # token 3 outside
    out = oracle.forward_backward(b, F64, V, p, want_dz=True)
    assert not (out["flags"][3] & 1) and (out["flags"][[0, 1, 2, 4]] & 1).all()
    h = 1e-6
    fd = np.zeros((T, V))
    for t in range(T):
        for v in range(V):
            zp, zm = z.copy(), z.copy()
            zp[t, v] += h
            zm[t, v] -= h
            bp, bm = dict(b, logits=zp), dict(b, logits=zm)
            fd[t, v] = (oracle.forward_backward(bp, F64, V, p)["loss"] -
                        oracle.forward_backward(bm, F64, V, p)["loss"]) / (2 * h)
    np.testing.assert_allclose(out["dz"], fd, rtol=1e-5, atol=1e-8 * np.abs(out["dz"]).max())


def test_stop_gradient_readings_equal_frozen_surrogates():
    """DIS with f frozen, and OPD with A frozen: dL/dz is the gradient of
    sum_t c_t logp_t(z) with the per-token coefficients held at their value."""
    rng = np.random.default_rng(23)
    V, T = 7, 4
    z = rng.normal(0, 1.0, (T, V))
    tg = rng.integers(0, V, T).astype(np.int32)
    cu = np.array([0, 4], np.int32)
    base = _batch(z, tg, np.zeros(T), np.zeros(T), np.ones(T), cu, [0.0])
    p0 = LossParams(group_size=1, adv_mode=1)
    lp = oracle.forward_backward(base, F64, V, p0)["logp"]
    cases = []
    bd = dict(base, token_adv=np.array([0.9, -0.6, 1.3, -1.1], np.float32),
              logp_infer=(lp - np.array([0.05, -0.1, 0.12, 0.0])).astype(np.float32))
    cases.append((bd, LossParams(group_size=1, adv_mode=2, objective=1, loss_norm=1, dis_stopgrad=1)))
    bo = dict(base, token_adv=(lp + np.array([0.3, -0.4, 0.2, -0.1])).astype(np.float32),
              logp_old=(lp - np.array([0.05, 0.0, -0.06, 0.02])).astype(np.float32))
    bo["logp_infer"] = bo["logp_old"].copy()
    cases.append((bo, LossParams(group_size=1, adv_mode=3)))
    for b, p in cases:
        out = oracle.forward_backward(b, F64, V, p, want_dz=True)
        c = out["g"]  # dL/dlogp with the stop-gradient factors frozen
        h = 1e-6
        fd = np.zeros((T, V))
        for t in range(T):
            for v in range(V):
                zp, zm = z.copy(), z.copy()
                zp[t, v] += h
                zm[t, v] -= h
                lp_p = oracle.forward_backward(dict(base, logits=zp), F64, V, p0)["logp"]
                lp_m = oracle.forward_backward(dict(base, logits=zm), F64, V, p0)["logp"]
                fd[t, v] = float(np.dot(c, lp_p - lp_m)) / (2 * h)
        np.testing.assert_allclose(out["dz"], fd, rtol=1e-5, atol=1e-9 * np.abs(out["dz"]).max())


def test_opd_teacher_advantage_closed_form_and_clip_side():
    rng = np.random.default_rng(24)
    lengths = [4, 3]
    b = _onpolicy_batch(rng, lengths, 13, [0.0, 0.0])
    lp = oracle.forward_backward(b, F64, 13, LossParams(group_size=1, adv_mode=1))["logp"]
    delta = np.array([0.3, -0.2, 0.5, 0.1, -0.4, 0.25, -0.05])
    b["token_adv"] = (lp + delta).astype(np.float32)  # teacher log-probs
    p = LossParams(group_size=1, adv_mode=3)
    out = oracle.forward_backward(b, F64, 13, p)
    want = -(np.mean(delta[:4]) + np.mean(delta[4:])) / 2  # r = 1, rho = 1: L = -(1/S) sum_i mean_t A_t
    assert abs(out["loss"] - want) < 2e-6
    # the sign of the distillation advantage picks the clipped side
    b2 = dict(b)
    b2["logp_old"] = (b["logp_old"].astype(np.float64) - np.log(1.5)).astype(np.float32)  # r = 1.5
    b2["logp_infer"] = b2["logp_old"].copy()
    out2 = oracle.forward_backward(b2, F64, 13, p)
    assert list((out2["flags"] >> 1) & 1) == [int(d > 0) for d in delta]


def test_per_token_advantages_reduce_to_per_response_and_token_norm_invariance():
    rng = np.random.default_rng(25)
    lengths = [3, 4, 2]
    A = [0.8, -0.3, 1.2]
    b = _onpolicy_batch(rng, lengths, 9, A)
    b["logp_infer"] = (b["logp_old"] + rng.normal(0, 0.2, 9)).astype(np.float32)
    per_seq = oracle.forward_backward(b, F64, 9, LossParams(group_size=1, adv_mode=1), want_dz=True)
    bt = dict(b, token_adv=np.repeat(np.array(A, np.float32), lengths))
    per_tok = oracle.forward_backward(bt, F64, 9, LossParams(group_size=1, adv_mode=2), want_dz=True)
    assert per_tok["loss"] == per_seq["loss"] and np.array_equal(per_tok["dz"], per_seq["dz"])
    # with the token mean, splitting response 1 into two responses changes nothing
    pt = LossParams(group_size=1, adv_mode=2, loss_norm=1)
    L = oracle.forward_backward(bt, F64, 9, pt)["loss"]
    split = dict(bt, cu_seqlens=np.array([0, 3, 5, 7, 9], np.int32))
    assert abs(oracle.forward_backward(split, F64, 9, pt)["loss"] - L) < 1e-15
    ps = LossParams(group_size=1, adv_mode=2, loss_norm=0)
    assert abs(oracle.forward_backward(split, F64, 9, ps)["loss"] - oracle.forward_backward(bt, F64, 9, ps)["loss"]) > 1e-6


# ----------------------------------------------------------------------------- GAE

def _gae_case(rng, lengths, obs_frac=0.3):
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    r = np.where(rng.random(T) < 0.1, rng.normal(0, 1, T), 0.0).astype(np.float32)
    v = rng.normal(0, 1, T).astype(np.float32)
    m = (rng.random(T) >= obs_frac).astype(np.uint8)
    return cu, r, v, m


def test_gae_special_cases():
    rng = np.random.default_rng(30)
    cu, r, v, m = _gae_case(rng, [7, 1, 12], obs_frac=0.0)
    # lambda = 1, gamma = 1: Monte-Carlo return minus value
    a = oracle.gae(cu, r, v, m, 1.0, 1.0)
    for i in range(3):
        for t in range(cu[i], cu[i + 1]):
            assert abs(a[t] - (float(np.sum(r[t:cu[i + 1]], dtype=np.float64)) - float(v[t]))) < 1e-12
    # lambda = 0: the one-step TD error
    a0 = oracle.gae(cu, r, v, m, 0.9, 0.0)
    for i in range(3):
        for t in range(cu[i], cu[i + 1]):
            v_next = float(v[t + 1]) if t + 1 < cu[i + 1] else 0.0
            assert abs(a0[t] - (float(r[t]) + 0.9 * v_next - float(v[t]))) < 1e-12


def test_gae_general_case_is_the_discounted_sum_of_td_errors():
    # the definition written out: over the action tokens t_0 < t_1 < ... of a response,
    # delta_j = r_{t_j} + gamma V_{t_{j+1}} - V_{t_j} (V after the last action token = 0) and
    # A_{t_j} = sum_{l >= 0} (gamma lambda)^l delta_{j+l}; observation tokens get 0
    rng = np.random.default_rng(33)
    cu, r, v, m = _gae_case(rng, [11, 1, 17, 6])
    gamma, lam = 0.93, 0.71
    a = oracle.gae(cu, r, v, m, gamma, lam)
    for i in range(len(cu) - 1):
        acts = [t for t in range(cu[i], cu[i + 1]) if m[t]]
        vals = [float(v[t]) for t in acts] + [0.0]
        delta = [float(r[t]) + gamma * vals[j + 1] - vals[j] for j, t in enumerate(acts)]
        for j, t in enumerate(acts):
            want = sum((gamma * lam) ** l * delta[j + l] for l in range(len(acts) - j))
            assert abs(a[t] - want) < 1e-12
        for t in range(cu[i], cu[i + 1]):
            if not m[t]:
                assert a[t] == 0.0


def test_gae_skip_observations_equals_gae_on_the_action_tokens_alone():
    rng = np.random.default_rng(31)
    cu, r, v, m = _gae_case(rng, [15, 9, 20])
    a = oracle.gae(cu, r, v, m, 0.97, 0.9)
    assert np.all(a[m == 0] == 0.0)
    keep = m.astype(bool)
    lens = [int(m[cu[i]:cu[i + 1]].sum()) for i in range(3)]
    cu2 = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    a2 = oracle.gae(cu2, r[keep], v[keep], np.ones(int(keep.sum()), np.uint8), 0.97, 0.9, skip_observations=False)
    np.testing.assert_allclose(a[keep], a2, rtol=0, atol=1e-13)
    # responses are independent: changing one response leaves the others unchanged
    r3 = r.copy()
    r3[cu[1]:cu[2]] += 5.0
    a3 = oracle.gae(cu, r3, v, m, 0.97, 0.9)
    assert np.array_equal(a3[:cu[1]], a[:cu[1]]) and np.array_equal(a3[cu[2]:], a[cu[2]:])


def test_gae_cross_trajectory_discount():
    rng = np.random.default_rng(32)
    cu, r, v, m = _gae_case(rng, [6, 5, 8, 4])
    ro = np.array([7, 7, 7, 9], np.int32)  # responses 0-2 are segments of one rollout
    gl = 0.95 * 0.9
    loc = oracle.gae(cu, r, v, m, 0.95, 0.9)
    a = oracle.gae(cu, r, v, m, 0.95, 0.9, rollout_ids=ro)
    n = [int(m[cu[i]:cu[i + 1]].sum()) for i in range(4)]
    later = [n[1] + n[2], n[2], 0, 0]
    for i in range(4):
        np.testing.assert_allclose(a[cu[i]:cu[i + 1]], loc[cu[i]:cu[i + 1]] * gl ** later[i], rtol=1e-14)
