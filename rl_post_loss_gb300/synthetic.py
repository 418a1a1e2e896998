"""Seeded synthetic inputs for the GRPO + IcePop token-level loss.

This module only *shapes inputs*: lengths, logits, sampled target ids,
perturbed old / inference log-probs, rewards and loss masks. Both the CUDA path
and the oracle consume its tensors as given; neither side's arithmetic lives
here. It imports torch only (never the CUDA library, never the oracle).

Workloads (the token counts, vocabularies, noise levels and hyper-parameters of
the five cases the loss is measured on):

====  ===================  ===========  ======  ===============================
case  responses            length       V       notes
====  ===================  ===========  ======  ===============================
0     2 prompts x G=4      U{16..128}   4096    fp32 logits N(0,2)
1     8 prompts x G=8      U{256..2048} 32768   bf16 N(0,3), +8 spike per row
2     4 prompts x G=8      U{512..4096} 151552  bf16 N(0,3) - 1.1 ln(v+1), 25% masked
3     8 responses, G=1     16384        151552  as 2, 30% masked, adv = U - U, beta 1.5
4     64 prompts x G=8     128          151552  hidden [N,6144] x W_lm [V,6144]
====  ===================  ===========  ======  ===============================

Each tensor draws from its own generator, seeded ``base * 100 + stream`` with
``base = 20261202 + case (+ seed offset)``; streams: 0 lengths, 1 logits,
2 targets, 3 old-noise, 4 infer-noise, 5 outliers, 6 rewards, 7 mask spans.
Large tensors are drawn in row chunks on the target device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

CASES = {
    0: dict(name="tiny-fp32 2x4 L16-128 V4096", prompts=2, group=4, len_lo=16, len_hi=128, vocab=4096,
            dtype="f32", z_std=2.0, spike=None, zipf=None, mask_frac=0.0, old_noise=0.05, infer_noise=0.1,
            outlier_frac=0.01, reward_p=0.5, adv_mode=0, beta=2.0, force_equal_group=False),
    1: dict(name="bf16 8x8 L256-2048 V32768", prompts=8, group=8, len_lo=256, len_hi=2048, vocab=32768,
            dtype="bf16", z_std=3.0, spike=8.0, zipf=None, mask_frac=0.0, old_noise=0.05, infer_noise=0.1,
            outlier_frac=0.02, reward_p=0.3, adv_mode=0, beta=2.0, force_equal_group=True),
    2: dict(name="bf16 4x8 L512-4096 V151552 masked25", prompts=4, group=8, len_lo=512, len_hi=4096,
            vocab=151552, dtype="bf16", z_std=3.0, spike=None, zipf=1.1, mask_frac=0.25, old_noise=0.05,
            infer_noise=0.1, outlier_frac=0.01, reward_p=0.5, adv_mode=0, beta=2.0, force_equal_group=False),
    3: dict(name="bf16 G1 8x16384 V151552 masked30", prompts=8, group=1, len_lo=16384, len_hi=16384,
            vocab=151552, dtype="bf16", z_std=3.0, spike=None, zipf=1.1, mask_frac=0.30, old_noise=0.05,
            infer_noise=0.2, outlier_frac=0.03, reward_p=None, adv_mode=1, beta=1.5, force_equal_group=False),
}

EPS_LOW, EPS_HIGH, ADV_EPS = 0.2, 0.28, 1e-6


@dataclass
class Batch:
    """One batch of packed variable-length responses.

    logits      [T, ld]  fp32 or bf16 (ld >= V, rows 16-byte aligned)
    targets     [T]      int32 sampled token ids
    logp_old    [T]      fp32 log pi_old^train of the sampled token
    logp_infer  [T]      fp32 log pi_old^infer of the sampled token
    mask        [T]      uint8 loss mask (1 = generated token)
    cu_seqlens  [S+1]    int32 response offsets; groups are G consecutive responses
    rewards_or_adv [S]   fp32 rewards (adv_mode 0) or advantages (adv_mode 1)
    """
    logits: torch.Tensor
    targets: torch.Tensor
    logp_old: torch.Tensor
    logp_infer: torch.Tensor
    mask: torch.Tensor
    cu_seqlens: torch.Tensor
    rewards_or_adv: torch.Tensor
    vocab: int
    group: int
    dtype: str
    adv_mode: int
    beta: float
    eps_low: float = EPS_LOW
    eps_high: float = EPS_HIGH
    adv_eps: float = ADV_EPS
    meta: dict = field(default_factory=dict)
    token_adv: torch.Tensor | None = None  # [T] advantages (adv_mode 2) or teacher log-probs (adv_mode 3)
    objective: int = 0                     # 0: GRPO + IcePop, 1: direct double-sided importance sampling
    loss_norm: int = 0                     # 0: per response, 1: mean over generated tokens

    @property
    def num_tokens(self) -> int:
        return int(self.targets.shape[0])

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    def to(self, device) -> "Batch":
        kw = {k: getattr(self, k).to(device) for k in
              ("logits", "targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv")}
        return Batch(**kw, vocab=self.vocab, group=self.group, dtype=self.dtype, adv_mode=self.adv_mode,
                     beta=self.beta, eps_low=self.eps_low, eps_high=self.eps_high, adv_eps=self.adv_eps,
                     meta=dict(self.meta), objective=self.objective, loss_norm=self.loss_norm,
                     token_adv=None if self.token_adv is None else self.token_adv.to(device))


def _gen(device, base: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(base * 100 + stream)
    return g


def padded_ld(vocab: int, dtype: str) -> int:
    """Smallest leading dimension >= vocab whose rows start on 16-byte boundaries."""
    per16 = 8 if dtype == "bf16" else 4
    return (vocab + per16 - 1) // per16 * per16


def span_mask(length: int, frac: float, rng: np.random.Generator, span_lo: int = 32, span_hi: int = 256):
    """Loss mask of one response: floor(frac * length) tokens set to 0 in
    non-overlapping spans of length U{span_lo..span_hi} (the last span
    truncated to hit the count), the spans placed at random gaps."""
    m = np.ones(length, np.uint8)
    target = int(math.floor(frac * length))
    if target <= 0:
        return m
    spans = []
    left = target
    while left > 0:
        s = int(rng.integers(span_lo, span_hi + 1))
        spans.append(min(s, left))
        left -= spans[-1]
    free = length - target
    cuts = np.sort(rng.integers(0, free + 1, size=len(spans)))
    gaps = np.diff(np.concatenate([[0], cuts]))
    pos = 0
    for gap, s in zip(gaps, spans):
        pos += int(gap)
        m[pos:pos + s] = 0
        pos += s
    return m


def make_lengths(case: dict, base: int) -> list[int]:
    S = case["prompts"] * case["group"]
    g = _gen("cpu", base, 0)
    return torch.randint(case["len_lo"], case["len_hi"] + 1, (S,), generator=g).tolist()


def make_batch(case_id: int, device="cpu", seed: int = 0, lengths: list[int] | None = None,
               vocab: int | None = None, ld: int | None = None, case_overrides: dict | None = None,
               chunk_rows: int = 2048) -> Batch:
    """Draw one batch of the given case. ``lengths`` / ``vocab`` / overrides
    shrink a case for small tests (same value recipe, smaller shape)."""
    case = dict(CASES[case_id])
    if case_overrides:
        case.update(case_overrides)
    if vocab is not None:
        case["vocab"] = vocab
    V = case["vocab"]
    base = 20261202 + case_id + 1000 * seed
    if lengths is None:
        lengths = make_lengths(case, base)
    S = len(lengths)
    G = case["group"]
    if S % G != 0:
        raise ValueError("number of responses must be a multiple of the group size")
    T = int(sum(lengths))
    cu = torch.zeros(S + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    dt = torch.bfloat16 if case["dtype"] == "bf16" else torch.float32
    ld = ld or padded_ld(V, case["dtype"])
    logits = torch.zeros((T, ld), dtype=dt, device=device)
    targets = torch.empty(T, dtype=torch.int32, device=device)
    logp_true = torch.empty(T, dtype=torch.float32, device=device)

    g_logits = _gen(device, base, 1)
    g_tgt = _gen(device, base, 2)
    offset = None
    if case["zipf"]:
        offset = -case["zipf"] * torch.log(torch.arange(1, V + 1, device=device, dtype=torch.float32))
    for r0 in range(0, T, chunk_rows):
        r1 = min(T, r0 + chunk_rows)
        z = torch.randn((r1 - r0, V), generator=g_logits, device=device, dtype=torch.float32) * case["z_std"]
        if case["spike"] is not None:
            idx = torch.randint(0, V, (r1 - r0,), generator=g_logits, device=device)
            z[torch.arange(r1 - r0, device=device), idx] += case["spike"]
        if offset is not None:
            z += offset
        zq = z.to(dt)
        logits[r0:r1, :V] = zq
        zf = zq.float()
        # target ~ softmax(z) by the Gumbel-max trick, on the logits as stored
        u = torch.rand((r1 - r0, V), generator=g_tgt, device=device, dtype=torch.float32)
        gumbel = -torch.log(-torch.log(u.clamp_min(1e-30)))
        y = torch.argmax(zf + gumbel, dim=1)
        targets[r0:r1] = y.to(torch.int32)
        logp_true[r0:r1] = torch.log_softmax(zf, dim=1).gather(1, y[:, None])[:, 0]
        del z, zq, zf, u, gumbel

    g_old = _gen(device, base, 3)
    g_inf = _gen(device, base, 4)
    g_out = _gen(device, base, 5)
    logp_old = logp_true + case["old_noise"] * torch.randn(T, generator=g_old, device=device)
    logp_infer = logp_old + case["infer_noise"] * torch.randn(T, generator=g_inf, device=device)
    is_out = torch.rand(T, generator=g_out, device=device) < case["outlier_frac"]
    sign = torch.where(torch.rand(T, generator=g_out, device=device) < 0.5, -1.0, 1.0)
    logp_infer = logp_infer + is_out.float() * sign * 2.0

    g_rw = _gen("cpu", base, 6)
    if case["adv_mode"] == 0:
        rewards = (torch.rand(S, generator=g_rw) < case["reward_p"]).float()
        if case["force_equal_group"]:
            grp = rewards.view(-1, G)
            if not bool(((grp == grp[:, :1]).all(dim=1)).any()):
                rewards[:G] = 0.0
        rw = rewards
    else:  # teacher_score - student_score, both U[0,1]
        rw = torch.rand(S, generator=g_rw) - torch.rand(S, generator=g_rw)

    rng = np.random.default_rng(base * 100 + 7)
    mask = np.concatenate([span_mask(L, case["mask_frac"], rng) for L in lengths]) if T else np.zeros(0, np.uint8)

    # optional variants of the objective (overrides): per-token advantages ~ N(0, 1)
    # ("token_adv": "normal", adv_mode 2), teacher log-probs logp_old + N(0, teacher_noise)
    # ("token_adv": "teacher", adv_mode 3), the DIS objective ("objective": 1), the
    # mean over tokens ("loss_norm": 1)
    token_adv, adv_mode = None, case["adv_mode"]
    if case.get("token_adv"):
        g_ta = _gen(device, base, 9)
        if case["token_adv"] == "teacher":
            token_adv = (logp_old + case.get("teacher_noise", 0.3) * torch.randn(T, generator=g_ta, device=device))
            adv_mode = 3
        else:
            token_adv = torch.randn(T, generator=g_ta, device=device)
            adv_mode = 2
        token_adv = token_adv.float().contiguous()
    return Batch(logits=logits, targets=targets, logp_old=logp_old.float().contiguous(),
                 logp_infer=logp_infer.float().contiguous(), mask=torch.from_numpy(mask).to(device),
                 cu_seqlens=cu.to(device), rewards_or_adv=rw.float().to(device), vocab=V, group=G,
                 dtype=case["dtype"], adv_mode=adv_mode, beta=case["beta"],
                 meta=dict(case=case_id, name=case["name"], seed=seed, lengths=list(lengths)),
                 token_adv=token_adv, objective=case.get("objective", 0), loss_norm=case.get("loss_norm", 0))


def to_numpy(batch: Batch) -> dict:
    """Host copies in the oracle's array layout (bf16 logits as uint16 bits)."""
    lg = batch.logits.detach().cpu()
    if lg.dtype == torch.bfloat16:
        lg = lg.view(torch.int16).numpy().view(np.uint16)
    else:
        lg = lg.numpy()
    return dict(logits=np.ascontiguousarray(lg[:, :batch.vocab]), targets=batch.targets.cpu().numpy(),
                logp_old=batch.logp_old.cpu().numpy(), logp_infer=batch.logp_infer.cpu().numpy(),
                mask=batch.mask.cpu().numpy(), cu_seqlens=batch.cu_seqlens.cpu().numpy(),
                rewards_or_adv=batch.rewards_or_adv.cpu().numpy())


# ---------------------------------------------------------------------------- fused projection (case 4)

PROJ_CASE = dict(name="fused projection 64x8 L128 H6144 V151552 chunk4096", prompts=64, group=8, length=128,
                 hidden=6144, vocab=151552, chunk=4096, h_std=1.0, w_std=0.02, old_noise=0.05, infer_noise=0.1,
                 outlier_frac=0.01, reward_p=0.5, mask_frac=0.25, beta=2.0)


@dataclass
class ProjBatch:
    """Hidden states, LM head and the per-token inputs of the fused path.

    hidden [T, ldh] bf16 ~ N(0, h_std); w [V, ldw] bf16 ~ N(0, w_std); targets
    drawn from softmax(hidden @ w^T); the rest as in ``Batch`` (``batch.logits``
    is an empty placeholder: the logits are never materialised).
    """
    hidden: torch.Tensor
    w: torch.Tensor
    batch: Batch
    chunk: int

    @property
    def hidden_dim(self) -> int:
        return int(self.hidden.shape[1])


def make_projection_batch(device="cpu", seed: int = 0, chunk_rows: int = 1024, **over) -> ProjBatch:
    """Case 4 (or a smaller variant of it through keyword overrides of PROJ_CASE)."""
    case = dict(PROJ_CASE)
    case.update(over)
    base = 20261202 + 4 + 1000 * seed
    S = case["prompts"] * case["group"]
    lengths = [case["length"]] * S
    T, H, V = S * case["length"], case["hidden"], case["vocab"]
    if H % 8:
        raise ValueError("hidden size must be a multiple of 8 (16-byte rows)")
    ldh, ldw = padded_ld(H, "bf16"), padded_ld(H, "bf16")
    g_h, g_w = _gen(device, base, 1), _gen(device, base, 8)
    hidden = torch.zeros((T, ldh), dtype=torch.bfloat16, device=device)
    w = torch.zeros((V, ldw), dtype=torch.bfloat16, device=device)
    for r0 in range(0, T, chunk_rows):
        r1 = min(T, r0 + chunk_rows)
        hidden[r0:r1, :H] = (torch.randn((r1 - r0, H), generator=g_h, device=device) * case["h_std"]).to(torch.bfloat16)
    for r0 in range(0, V, 8 * chunk_rows):
        r1 = min(V, r0 + 8 * chunk_rows)
        w[r0:r1, :H] = (torch.randn((r1 - r0, H), generator=g_w, device=device) * case["w_std"]).to(torch.bfloat16)
    targets = torch.empty(T, dtype=torch.int32, device=device)
    logp_true = torch.empty(T, dtype=torch.float32, device=device)
    g_tgt = _gen(device, base, 2)
    for r0 in range(0, T, chunk_rows):
        r1 = min(T, r0 + chunk_rows)
        z = (hidden[r0:r1, :H] @ w[:, :H].T).float()  # input shaping only
        u = torch.rand(z.shape, generator=g_tgt, device=device, dtype=torch.float32)
        y = torch.argmax(z - torch.log(-torch.log(u.clamp_min(1e-30))), dim=1)
        targets[r0:r1] = y.to(torch.int32)
        logp_true[r0:r1] = torch.log_softmax(z, dim=1).gather(1, y[:, None])[:, 0]
        del z, u
    g_old, g_inf, g_out = _gen(device, base, 3), _gen(device, base, 4), _gen(device, base, 5)
    logp_old = logp_true + case["old_noise"] * torch.randn(T, generator=g_old, device=device)
    logp_infer = logp_old + case["infer_noise"] * torch.randn(T, generator=g_inf, device=device)
    is_out = torch.rand(T, generator=g_out, device=device) < case["outlier_frac"]
    sign = torch.where(torch.rand(T, generator=g_out, device=device) < 0.5, -1.0, 1.0)
    logp_infer = logp_infer + is_out.float() * sign * 2.0
    rewards = (torch.rand(S, generator=_gen("cpu", base, 6)) < case["reward_p"]).float()
    rng = np.random.default_rng(base * 100 + 7)
    mask = np.concatenate([span_mask(L, case["mask_frac"], rng) for L in lengths])
    cu = torch.zeros(S + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    b = Batch(logits=torch.empty((T, 0), dtype=torch.bfloat16, device=device), targets=targets,
              logp_old=logp_old.float().contiguous(), logp_infer=logp_infer.float().contiguous(),
              mask=torch.from_numpy(mask).to(device), cu_seqlens=cu.to(device), rewards_or_adv=rewards.to(device),
              vocab=V, group=case["group"], dtype="bf16", adv_mode=0, beta=case["beta"],
              meta=dict(case=4, name=case["name"], seed=seed, lengths=lengths))
    return ProjBatch(hidden=hidden, w=w, batch=b, chunk=case["chunk"])


# ---------------------------------------------------------------------------- GAE inputs

GAE_CASE = dict(name="GAE 128 rollouts x 2 segments x 65536 tokens, 30% observation", rollouts=128, segments=2,
                length=65536, obs_frac=0.30, gamma=1.0, lam=0.95)


@dataclass
class GaeBatch:
    """Per-token rewards (a Bernoulli(0.5) outcome on each rollout's last action
    token, 1% of action tokens with N(0, 0.1) process rewards), critic values
    N(0, 0.5), observation spans (mask 0) covering obs_frac of every segment,
    and rollout ids (consecutive segments of one rollout share an id)."""
    rewards: torch.Tensor
    values: torch.Tensor
    mask: torch.Tensor
    cu_seqlens: torch.Tensor
    rollout_ids: torch.Tensor
    gamma: float
    lam: float

    @property
    def num_tokens(self) -> int:
        return int(self.rewards.shape[0])


def make_gae_batch(device="cpu", seed: int = 0, lengths: list[int] | None = None, **over) -> GaeBatch:
    case = dict(GAE_CASE)
    case.update(over)
    base = 20261202 + 5 + 1000 * seed
    if lengths is None:
        lengths = [case["length"]] * (case["rollouts"] * case["segments"])
    S, T = len(lengths), int(sum(lengths))
    rng = np.random.default_rng(base * 100 + 7)
    mask = np.concatenate([span_mask(L, case["obs_frac"], rng) for L in lengths]) if T else np.zeros(0, np.uint8)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    g = _gen("cpu", base, 6)
    rewards = torch.zeros(T)
    proc = torch.rand(T, generator=g) < 0.01
    rewards[proc] = 0.1 * torch.randn(int(proc.sum()), generator=g)
    seg = case["segments"]
    rollout_ids = np.arange(S, dtype=np.int32) // max(1, seg)
    for i in range(S):  # the outcome reward on the last action token of each rollout's last segment
        if (i + 1) % seg == 0 or i == S - 1:
            act = np.nonzero(mask[cu[i]:cu[i + 1]])[0]
            if act.size:
                rewards[cu[i] + act[-1]] += float(torch.rand(1, generator=g) < 0.5)
    rewards = rewards * torch.from_numpy(mask).float()
    values = 0.5 * torch.randn(T, generator=_gen("cpu", base, 1))
    return GaeBatch(rewards=rewards.to(device), values=values.to(device), mask=torch.from_numpy(mask).to(device),
                    cu_seqlens=torch.from_numpy(cu).to(device), rollout_ids=torch.from_numpy(rollout_ids).to(device),
                    gamma=case["gamma"], lam=case["lam"])


# ------------------------------------------------------------------ DSA indexer scores for top-k

TOPK_CASE = dict(name="DSA indexer top-k: last 4096 query positions of a 202,752-token context, k=2048",
                 rows=4096, context=202752, k=2048)
TOPK_SMALL = dict(name="DSA indexer top-k, small: 48 query positions of a 20,000-token context", rows=48,
                  context=20000, k=2048)
_INDEXER_HEAD_WEIGHTS = (1.0, 0.8, 0.6, 0.4)


@dataclass
class TopkBatch:
    """Indexer-like scores: sum over 4 heads of w_h * relu(N(0,1)), rounded to
    bf16 precision (the indexer runs in low precision, so scores tie often) and
    stored as fp32 [rows, ld]; row q is causal and holds lengths[q] = context -
    rows + 1 + q valid keys (the rest of the row is filled but not part of it)."""
    scores: torch.Tensor
    lengths: torch.Tensor
    k: int

    @property
    def rows(self) -> int:
        return int(self.scores.shape[0])

    @property
    def ld(self) -> int:
        return int(self.scores.shape[1])


def topk_ld(context: int) -> int:
    """Row stride: the context rounded up to a multiple of 32 keys."""
    return (context + 31) // 32 * 32


def make_topk_batch(device="cpu", seed: int = 0, **over) -> TopkBatch:
    case = dict(TOPK_CASE)
    case.update(over)
    rows, context = int(case["rows"]), int(case["context"])
    base = 20261202 + 7 + 1000 * seed
    ld = topk_ld(context)
    g = _gen(device, base, 1)
    scores = torch.empty((rows, ld), dtype=torch.float32, device=device)
    block = max(1, (1 << 26) // max(ld, 1))
    for r0 in range(0, rows, block):
        r1 = min(rows, r0 + block)
        acc = torch.zeros((r1 - r0, ld), dtype=torch.float32, device=device)
        for w in _INDEXER_HEAD_WEIGHTS:
            acc += w * torch.relu(torch.randn((r1 - r0, ld), generator=g, device=device))
        scores[r0:r1] = acc.to(torch.bfloat16).to(torch.float32)
    lengths = torch.arange(rows, dtype=torch.int32, device=device) + (context - rows + 1)
    return TopkBatch(scores=scores, lengths=lengths, k=int(case["k"]))
