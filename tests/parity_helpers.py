"""Comparison of the CUDA path's outputs with the fp64 oracle on the same inputs.

Tolerances (stated for this workload): per-token log-prob and entropy abs 1e-4
with fp32 logits, 2e-3 with bf16 logits; scalar loss rel 1e-4 (plus, for the distillation advantage, the
first-order effect of the log-prob error on the loss: see distillation_loss_slack); dL/dlogits
abs 1e-6 + rel 8e-3; pop flags bit-exact; clip flags bit-exact against the
clip rule applied to the kernel's own fp32 log-prob, and equal to the
oracle's own decision wherever the oracle's log-prob is not within the
log-prob tolerance of a clip threshold. On top of the stated dL/dlogits bound a
tighter one is checked that follows from the arithmetic: one rounding to the
output dtype (2^-9 relative for bf16) plus about 1e-6 relative from the fp32
softmax, i.e. rel 4e-3 (bf16) / 1e-5 (fp32) + 2e-6 |dL/dlogp| + 1e-30; for the
DIS objective without stop-gradient the factor (1 + logp) of dL/dlogp adds
1e-5 / |1 + logp| relative.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import LossParams
from rl_post_loss_gb300 import synthetic

TOL_LOGP = {"f32": 1e-4, "bf16": 2e-3}
TOL_LOSS_REL = 1e-4
DZ_ABS, DZ_REL = 1e-6, 8e-3
DZ_STRICT_REL = {"f32": 1e-5, "bf16": 4e-3}


def params_for(batch, **over) -> LossParams:
    kw = dict(group_size=batch.group, eps_low=batch.eps_low, eps_high=batch.eps_high, beta=batch.beta,
              adv_eps=batch.adv_eps, adv_mode=batch.adv_mode, objective=batch.objective,
              loss_norm=batch.loss_norm)
    kw.update(over)
    return LossParams(**kw)


def odtype(batch) -> int:
    return oracle.BF16 if batch.dtype == "bf16" else oracle.F32


def logits_rows_np(batch, row_ids) -> np.ndarray:
    idx = torch.as_tensor(np.asarray(row_ids, np.int64), device=batch.logits.device)
    lg = batch.logits.index_select(0, idx)[:, :batch.vocab].contiguous().cpu()
    if lg.dtype == torch.bfloat16:
        return lg.view(torch.int16).numpy().view(np.uint16)
    return lg.numpy()


def dz_rows_np(dlogits, row_ids, V) -> np.ndarray:
    idx = torch.as_tensor(np.asarray(row_ids, np.int64), device=dlogits.device)
    return dlogits.index_select(0, idx)[:, :V].float().cpu().numpy().astype(np.float64)


class OracleRun:
    """Oracle results for a batch: the sequence-level part, every row's
    per-token results (streamed, no dL/dlogits), and the loss."""

    def __init__(self, batch, p: LossParams, block: int = 2048):
        self.batch, self.p = batch, p
        self.np = {k: v.cpu().numpy() for k, v in dict(targets=batch.targets, logp_old=batch.logp_old,
                                                       logp_infer=batch.logp_infer, mask=batch.mask,
                                                       cu_seqlens=batch.cu_seqlens,
                                                       rewards_or_adv=batch.rewards_or_adv).items()}
        a = self.np
        self.token_adv = None if batch.token_adv is None else batch.token_adv.cpu().numpy()
        self.n, self.adv, self.w = oracle.seq_prep(a["cu_seqlens"], a["mask"], a["rewards_or_adv"], p)
        T = batch.num_tokens
        parts = []
        for r0 in range(0, T, block):
            ids = np.arange(r0, min(T, r0 + block))
            parts.append(self.rows(ids))
        keys = ("logp", "entropy", "flags", "tok_obj", "g")
        self.tok = {k: (np.concatenate([q[k] for q in parts]) if parts else np.zeros(0)) for k in keys}
        self.loss = oracle.loss(a["cu_seqlens"], self.w, self.tok["tok_obj"]) if T else 0.0

    def rows(self, ids, want_dz=False):
        a = self.np
        return oracle.rows(ids, logits_rows_np(self.batch, ids), odtype(self.batch), self.batch.vocab,
                           a["targets"], a["logp_old"], a["logp_infer"], a["mask"], a["cu_seqlens"], self.adv,
                           self.w, self.p, want_dz=want_dz, token_adv=self.token_adv)

    def adv_per_token(self, logp32=None) -> np.ndarray:
        """Each token's advantage; for the distillation advantage, its fp32
        value from the given fp32 log-probs (the sign decides the clip side)."""
        if self.p.adv_mode == 2:
            return self.token_adv.astype(np.float64)
        if self.p.adv_mode == 3:
            return (self.token_adv.astype(np.float32) - np.asarray(logp32, np.float32)).astype(np.float64)
        cu = self.np["cu_seqlens"]
        return np.repeat(self.adv, np.diff(cu))


def check_tokens(batch, run: OracleRun, out: dict, report: dict | None = None):
    """Per-token log-prob, entropy and flags of every token."""
    tol = TOL_LOGP[batch.dtype]
    logp = out["logp"].cpu().numpy().astype(np.float64)
    ent = out["entropy"].cpu().numpy().astype(np.float64)
    flags = out["flags"].cpu().numpy()
    o = run.tok
    ok_t = (o["flags"] & 8) == 0
    assert np.array_equal(flags & 8, o["flags"] & 8), "bad-target bits differ"
    assert np.array_equal(flags & 4, o["flags"] & 4), "mask bits differ"
    err = np.abs(logp[ok_t] - o["logp"][ok_t])
    assert err.size == 0 or err.max() <= tol, f"logp max err {err.max()}"
    assert np.all(np.isnan(logp[~ok_t]))
    eerr = np.abs(ent - o["entropy"])
    assert eerr.size == 0 or eerr.max() <= tol, f"entropy max err {eerr.max()}"
    lp32 = out["logp"].cpu().numpy()
    hi, lo_thr = oracle.thresholds_f32(run.p.beta, run.p.eps_low, run.p.eps_high)[1:]
    if run.p.objective == 1:
        # the DIS gate: exact against the rule on the kernel's own fp32 log-prob
        li = run.np["logp_infer"]
        e32 = (np.where(ok_t, lp32, 0).astype(np.float32) - li.astype(np.float32)).astype(np.float32)
        rule = (ok_t & (e32 > lo_thr) & (e32 < hi)).astype(np.uint8)
        assert np.array_equal(flags & 1, rule), "DIS gate bits differ from the rule on the kernel's logp"
        assert not np.any(flags & 2)
        e64 = o["logp"] - li.astype(np.float64)
        near = ok_t & ((np.abs(e64 - hi) <= tol) | (np.abs(e64 - lo_thr) <= tol))
        diff = (flags & 1) != (o["flags"] & 1)
        assert not np.any(diff & ~near), "DIS gate bits differ away from a threshold"
    else:
        assert np.array_equal(flags & 1, o["flags"] & 1), "pop bits differ"
        # clip bits: exact against the rule applied to the kernel's own fp32 log-prob
        advt = run.adv_per_token(lp32)
        lo = run.np["logp_old"]
        rule = oracle.clip_active_vec(np.where(ok_t, lp32, 0), lo, np.where(ok_t, advt, 0.0), run.p.eps_low,
                                      run.p.eps_high)
        assert np.array_equal((flags >> 1) & 1, rule), "clip bits differ from the rule on the kernel's logp"
        # and equal to the oracle's own decision away from the thresholds (and, for
        # the distillation advantage, away from a zero advantage)
        e64 = o["logp"] - lo.astype(np.float64)
        near = ok_t & ((np.abs(e64 - hi) <= tol) | (np.abs(e64 - lo_thr) <= tol))
        if run.p.adv_mode == 3:
            near |= ok_t & (np.abs(run.token_adv.astype(np.float64) - o["logp"]) <= tol)
        diff = ((flags >> 1) & 1) != ((o["flags"] >> 1) & 1)
        assert not np.any(diff & ~near), "clip bits differ away from a threshold"
    if report is not None:
        report.update(logp_max_err=float(err.max()) if err.size else 0.0,
                      entropy_max_err=float(eerr.max()) if eerr.size else 0.0,
                      ambiguous_clip=int(near.sum()), clip_diff=int(diff.sum()))
    return near


def distillation_loss_slack(run: OracleRun, out: dict) -> float:
    """With the distillation advantage A_t = teacher_t - logp_t, every token term
    depends on the kernel's fp32 log-prob (through r and through A): a log-prob off by
    d_t moves the term m pop min(r A, clip(r) A) by at most pop max(r, 1 + eps_high)
    (|A_t| + 1) |d_t| to first order. The loss, which is near zero when A is centred,
    therefore carries the log-prob error (its own tolerance is absolute) on top of the
    relative loss tolerance. Returns twice that first-order sum over the tokens, with
    the measured per-token log-prob differences."""
    a = run.np
    T = run.batch.num_tokens
    if run.p.adv_mode != 3 or T == 0:
        return 0.0
    lp = run.tok["logp"]
    ok = np.isfinite(lp)
    d = np.where(ok, np.abs(out["logp"].cpu().numpy().astype(np.float64) - np.where(ok, lp, 0.0)), 0.0)
    lo = a["logp_old"].astype(np.float64)
    rho = np.exp(lo - a["logp_infer"].astype(np.float64))
    pop = np.where((run.tok["flags"] & 1) != 0, 1.0 if run.p.pop_indicator else rho, 0.0) * (a["mask"] != 0)
    r = np.exp(np.where(ok, lp, lo) - lo)
    A = run.token_adv.astype(np.float64) - np.where(ok, lp, 0.0)
    w = np.repeat(np.asarray(run.w, np.float64), np.diff(a["cu_seqlens"]))
    return 2.0 * float(np.sum(w * pop * np.maximum(r, 1.0 + run.p.eps_high) * (np.abs(A) + 1.0) * d))


def check_loss(batch, run: OracleRun, out: dict, report: dict | None = None):
    L = float(out["loss_f64"].cpu()[0])
    L32 = float(out["loss"].cpu()[0])
    ref = run.loss
    tol = TOL_LOSS_REL * abs(ref) + distillation_loss_slack(run, out) + 1e-12
    assert abs(L - ref) <= tol, f"loss {L} vs oracle {ref}"
    assert abs(L32 - ref) <= tol, f"loss f32 {L32} vs oracle {ref}"
    if report is not None:
        report.update(loss=L, loss_oracle=ref, loss_rel_err=abs(L - ref) / max(abs(ref), 1e-300))


def check_seq_outputs(batch, run: OracleRun, out: dict):
    np.testing.assert_allclose(out["seq_adv"].cpu().numpy(), run.adv, rtol=1e-6, atol=1e-7)
    cnt = out["counts"].cpu().numpy()
    o = run.tok["flags"]
    m = run.np["mask"] != 0
    gflags = out["flags"].cpu().numpy()
    assert cnt[0] == int((m & ((gflags & 1) == 0)).sum()), "popped count"
    assert cnt[1] == int((m & ((gflags & 2) != 0)).sum()), "clipped count"
    assert cnt[2] == int((~m).sum()), "masked count"
    assert cnt[3] == int((run.n == 0).sum()), "empty responses"
    if m.any():
        ref = float(run.tok["entropy"][m].mean())
        assert abs(float(out["mean_entropy"].cpu()[0]) - ref) <= TOL_LOGP[batch.dtype]


def check_dz_rows(batch, run: OracleRun, out: dict, row_ids, skip_rows=None, report: dict | None = None):
    row_ids = np.asarray(row_ids, np.int64)
    if skip_rows is not None:
        row_ids = row_ids[~skip_rows[row_ids]]
    if row_ids.size == 0:
        return
    V = batch.vocab
    ref = run.rows(row_ids, want_dz=True)
    got = dz_rows_np(out["dlogits"], row_ids, V)
    dz = ref["dz"]
    err = np.abs(got - dz)
    bound = DZ_ABS + DZ_REL * np.abs(dz)
    assert np.all(err <= bound), f"dlogits stated bound: worst excess {(err - bound).max()}"
    g = np.abs(ref["g"])[:, None]
    rel = np.full((row_ids.size, 1), DZ_STRICT_REL[batch.dtype])
    if run.p.objective == 1 and not run.p.dis_stopgrad:
        # dL/dlogp = -w r A (1 + logp): an fp32 logp (abs error ~1e-6) makes the
        # factor (1 + logp) lose relative accuracy as logp approaches -1
        rel = rel + 1e-5 / np.maximum(np.abs(1.0 + ref["logp"]), 1e-12)[:, None]
    strict = rel * np.abs(dz) + 2e-6 * g + 1e-30
    bad = err > strict
    assert not bad.any(), f"dlogits strict bound violated at {np.argwhere(bad)[:5]} ({err[bad][:5]}, {dz[bad][:5]})"
    zero_rows = ref["g"] == 0.0
    assert np.all(got[zero_rows] == 0.0), "rows with zero dL/dlogp must be exact zeros"
    if report is not None:
        nz = dz != 0
        rel = np.abs(got[nz] - dz[nz]) / np.abs(dz[nz]) if nz.any() else np.zeros(1)
        report.update(dz_rows=int(row_ids.size), dz_max_rel_err=float(rel.max()), dz_max_abs_err=float(err.max()))


def check_all(batch, out, p=None, dz_rows="all", seed=0, report=None):
    p = p or params_for(batch)
    run = OracleRun(batch, p)
    near = check_tokens(batch, run, out, report)
    check_loss(batch, run, out, report)
    check_seq_outputs(batch, run, out)
    T = batch.num_tokens
    if dz_rows == "all":
        ids = np.arange(T)
    else:
        rng = np.random.default_rng(seed)
        ids = np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=min(T, dz_rows), replace=False)]))
    check_dz_rows(batch, run, out, ids, skip_rows=near, report=report)
    return run
