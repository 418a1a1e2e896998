"""The loss tolerance of the on-policy distillation advantage, checked on the CPU.

With A_t = sg[log pi_teacher(y_t) - logp_t] ("GLM-5: from Vibe Coding to Agentic
Engineering", section 3.5, Eq. (2)) every token term of Eq. (1) depends on the
log-prob through r and through A, so a log-prob error moves the loss by about the
error itself. parity_helpers.distillation_loss_slack adds twice the first-order
sum to the relative loss tolerance. Here a numpy restatement of the loss from a
log-prob vector must reproduce the oracle's loss, and shifting the log-probs,
uniformly or at random, must move it by no more than the slack."""
import numpy as np
import pytest
import torch

from parity_helpers import OracleRun, distillation_loss_slack, params_for
from rl_post_loss_gb300 import synthetic


def _opd_batch(seed):
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(8, 61, size=16)]
    return synthetic.make_batch(1, "cpu", seed=seed, lengths=lengths, vocab=2048,
                                case_overrides=dict(token_adv="teacher", group=1, prompts=16))


def _loss_from_logp(run, lp):
    """-sum_i w_i sum_t m pop min(r A, clip(r) A) with r and A taken from ``lp``."""
    a = run.np
    lo = a["logp_old"].astype(np.float64)
    r = np.exp(lp - lo)
    A = run.token_adv.astype(np.float64) - lp
    rho = np.exp(lo - a["logp_infer"].astype(np.float64))
    pop = np.where((run.tok["flags"] & 1) != 0, rho, 0.0) * (a["mask"] != 0)
    clipped_r = np.clip(r, 1.0 - run.p.eps_low, 1.0 + run.p.eps_high)
    w = np.repeat(np.asarray(run.w, np.float64), np.diff(a["cu_seqlens"]))
    return -float(np.sum(w * pop * np.minimum(r * A, clipped_r * A)))


@pytest.mark.parametrize("seed", [0, 11])
def test_restatement_matches_the_oracle_loss(seed):
    b = _opd_batch(seed)
    run = OracleRun(b, params_for(b))
    assert np.all(np.isfinite(run.tok["logp"]))
    assert abs(_loss_from_logp(run, run.tok["logp"]) - run.loss) <= 1e-12 * max(1.0, abs(run.loss))


@pytest.mark.parametrize("seed", [0, 11])
@pytest.mark.parametrize("scale", [1e-6, 1e-4])
def test_logprob_errors_stay_inside_the_slack(seed, scale):
    b = _opd_batch(seed)
    run = OracleRun(b, params_for(b))
    lp = run.tok["logp"]
    base = _loss_from_logp(run, lp)
    shifts = [np.full(lp.shape, scale), np.full(lp.shape, -scale)]
    shifts += [np.random.default_rng(s).uniform(-scale, scale, lp.shape) for s in range(8)]
    for d in shifts:
        out = {"logp": torch.from_numpy(lp + d)}  # float64: the slack sees exactly the shift
        slack = distillation_loss_slack(run, out)
        assert slack > 0.0
        # the slack is twice the first-order bound; a uniform shift reaches about a third of it
        assert abs(_loss_from_logp(run, lp + d) - base) <= 0.5 * slack * (1.0 + 10.0 * scale)


def test_slack_is_zero_for_other_advantage_modes():
    b = synthetic.make_batch(1, "cpu", lengths=[20] * 8, vocab=512)
    run = OracleRun(b, params_for(b))
    out = {"logp": torch.from_numpy(run.tok["logp"] + 1e-3)}
    assert distillation_loss_slack(run, out) == 0.0
