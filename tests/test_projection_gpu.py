"""The fused sequence-chunked projection + loss path against the fp64 oracle:
the tcgen05 projection GEMM alone (ragged tiles, full width), the whole fused
forward+backward on small cases spanning several chunks and tiles, its
determinism, and the full-size case on sampled rows plus identities."""
import os

import numpy as np
import pytest
import torch

import oracle
from parity_helpers import params_for
from rl_post_loss_gb300 import build as nvbuild
from rl_post_loss_gb300 import capi, synthetic

pytestmark = pytest.mark.gpu

TOL_LOGP_STATED = 3e-2   # fused-GEMM configuration, as stated for this workload
TOL_LOGP_STRICT = 2e-4   # fp32-accumulated logits: what the arithmetic gives


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nvbuild.build()
    capi.load()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,K,N", [(128, 64, 256), (300, 320, 1000), (257, 6144, 2048), (64, 6144, 151552)])
def test_projection_gemm_matches_fp64(M, K, N):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + K + N)
    h = (torch.randn((M, K), generator=g, device="cuda")).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    rl = capi.RlLoss(N, 1, M, 1, capi.RL_BF16)
    rl.projection_setup(K, M)
    ldz = (N + 3) // 4 * 4
    z = torch.full((M, ldz), float("nan"), dtype=torch.float32, device="cuda")
    rl.projection_logits(h, w, M, z)
    torch.cuda.synchronize()
    got = z[:, :N].double().cpu().numpy()
    ref = oracle.projection_logits(_bits(h), _bits(w))
    scale = oracle.bf16_bits_to_f64(_bits(h)).__abs__() @ oracle.bf16_bits_to_f64(_bits(w)).__abs__().T
    err = np.abs(got - ref)
    assert np.all(err <= 1e-5 * scale + 1e-6), f"max err {err.max()} (scaled {(err / (scale + 1e-30)).max()})"
    assert bool(torch.isnan(z[:, N:]).all()), "padding columns written"


def _small(prompts=2, group=4, length=50, hidden=320, vocab=1000, chunk=160, seed=0, **over):
    return synthetic.make_projection_batch("cuda", seed=seed, prompts=prompts, group=group, length=length,
                                           hidden=hidden, vocab=vocab, chunk=chunk, **over)


def _check_fused(pb, out, report=None):
    b = pb.batch
    p = params_for(b)
    npb = {k: getattr(b, k).cpu().numpy() for k in
           ("targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv")}
    H = pb.hidden_dim
    ref = oracle.projection_forward_backward(_bits(pb.hidden[:, :H]), _bits(pb.w[:, :H]), npb, p)
    L = out["loss_f64"].item()
    assert abs(L - ref["loss"]) <= 1e-4 * abs(ref["loss"]) + 1e-12, (L, ref["loss"])
    lp = out["logp"].cpu().numpy().astype(np.float64)
    assert np.abs(lp - ref["logp"]).max() <= TOL_LOGP_STATED
    assert np.abs(lp - ref["logp"]).max() <= TOL_LOGP_STRICT
    assert np.abs(out["entropy"].cpu().numpy() - ref["entropy"]).max() <= TOL_LOGP_STRICT
    f = out["flags"].cpu().numpy()
    assert np.array_equal(f & 0xD, ref["flags"] & 0xD)
    advt = np.repeat(ref["adv"], np.diff(npb["cu_seqlens"]))
    rule = oracle.clip_active_vec(out["logp"].cpu().numpy(), npb["logp_old"], advt, p.eps_low, p.eps_high)
    assert np.array_equal((f >> 1) & 1, rule)
    near = np.abs(np.abs(ref["logp"] - npb["logp_old"]) - 0.2469) < 1e-3  # none expected at these noise levels
    ok = ~near
    dh = out["dhidden"][:, :H].double().cpu().numpy()
    dw = out["dw_lm"][:, :H].double().cpu().numpy()
    T, V = dh.shape[0], ref["dz"].shape[1]
    hT, W64 = oracle.bf16_bits_to_f64(_bits(pb.hidden[:T, :H])), oracle.bf16_bits_to_f64(_bits(pb.w[:, :H]))
    dz = ref["dz"]
    rep = _grad_close("dhidden", dh[ok], ref["dh"][ok], (np.abs(dz) @ np.abs(W64))[ok],
                      np.sqrt((dz * dz) @ (W64 * W64))[ok], V, True)
    rep.update(_grad_close("dW", dw, ref["dW"], np.abs(dz).T @ np.abs(hT), np.sqrt((dz * dz).T @ (hT * hT)), T, False))
    if report is not None:
        report.update(rep)
        report.update(loss=L, loss_oracle=ref["loss"], logp_max_err=float(np.abs(lp - ref["logp"]).max()))


@pytest.mark.parametrize("kw", [dict(), dict(vocab=4097, hidden=128, chunk=96), dict(prompts=1, length=300, chunk=512)])
def test_fused_projection_small_parity(kw):
    pb = _small(**kw)
    rl = capi.projection_handle(pb)
    out = capi.alloc_projection_outputs(pb)
    capi.run_projection(rl, pb, out)
    torch.cuda.synchronize()
    assert rl.device_status() & ~(1 << capi.CODES["RL_ERR_EMPTY_SEQ"]) == 0
    rep = {}
    _check_fused(pb, out, rep)
    print(rep)


def test_fused_projection_bit_identical_runs():
    pb = _small(prompts=2, group=8, length=64, hidden=512, vocab=3000, chunk=200)
    rl = capi.projection_handle(pb)
    outs = []
    for _ in range(3):
        out = capi.alloc_projection_outputs(pb)
        capi.run_projection(rl, pb, out)
        torch.cuda.synchronize()
        outs.append(out)
    for k in outs[0]:
        for o in outs[1:]:
            assert torch.equal(outs[0][k].view(torch.uint8), o[k].view(torch.uint8)), k


U_BF16 = 2.0 ** -8  # unit roundoff of bf16 (8 significant bits)


def _grad_close(name, got, want, mag, l2, K, bf16_out):
    """A gradient product D = dZ B (dH = dZ W, or dW = dZ^T H) against the fp64
    oracle. dZ carries two bf16 roundings (the stored scaled probability and dZ
    itself), each with relative error <= u = 2^-8, so every term of the sum is
    off by at most (1 + u)^2 - 1; the fp32 accumulation over K terms adds at most
    K 2^-24 of the terms' magnitudes (doubled here), and a bf16 output one more
    rounding of u |D|. With mag = |dZ| |B| and l2 = sqrt(dZ^2 B^2) (element-wise
    squares):
      rigorous:     |err| <= (2u + u^2) mag + K 2^-23 mag (+ u |D|)
      statistical:  |err| <= 6 sqrt(2/3) u l2 + K 2^-23 mag (+ u |D|): a bf16
                    rounding error is uniform with standard deviation u/sqrt(3)
                    of the value at most, independent from term to term, so 6
                    standard deviations of their sum;
    and each nonzero row within relative L2 1e-2; rows whose exact gradient is
    zero are exact zeros."""
    err = np.abs(got - want)
    fp32 = K * 2.0 ** -23 * mag
    out = U_BF16 * np.abs(want) if bf16_out else 0.0
    rigorous = (2 * U_BF16 + U_BF16 ** 2) * mag + fp32 + out
    assert np.all(err <= rigorous), f"{name}: rigorous bound exceeded by {(err / (rigorous + 1e-300)).max()}"
    stat = 6.0 * np.sqrt(2.0 / 3.0) * U_BF16 * l2 + fp32 + out
    assert np.all(err <= stat), f"{name}: statistical bound exceeded by {(err / (stat + 1e-300)).max()}"
    nrm = np.linalg.norm(want, axis=1)
    nz = nrm > 0
    rn = np.linalg.norm(got - want, axis=1)[nz] / nrm[nz]
    assert rn.size == 0 or rn.max() <= 1e-2, f"{name} row relative L2 {rn.max()}"
    assert np.all(got[~nz] == 0.0), f"{name}: rows with zero gradient must be exact zeros"
    return {name + "_row_rel_l2_max": float(rn.max()) if rn.size else 0.0,
            name + "_of_rigorous": float((err / (rigorous + 1e-300)).max()),
            name + "_of_statistical": float((err / (stat + 1e-300)).max())}


def _check_exact_forward_and_sampled_grads(pb, out, n_vocab_rows=256, n_token_rows=64, seed=5):
    """The loss against the exact fp64 loss over every row (streamed forward), every
    row's log-prob / entropy / flags, and sampled rows of dL/dW and dL/dh element by
    element (dL/dW_v = sum_t dL/dz_tv h_t needs the forward of every row)."""
    b = pb.batch
    T, H, V = b.num_tokens, pb.hidden_dim, b.vocab
    p = params_for(b)
    npb = {k: getattr(b, k).cpu().numpy() for k in
           ("targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv")}
    hb, wb = _bits(pb.hidden[:, :H]), _bits(pb.w[:, :H])
    h64, W64 = oracle.bf16_bits_to_f64(hb), oracle.bf16_bits_to_f64(wb)
    ref = oracle.projection_forward_stats(hb, None, npb, p, w64=W64)
    L = out["loss_f64"].item()
    assert abs(L - ref["loss"]) <= 1e-4 * abs(ref["loss"]) + 1e-12, (L, ref["loss"])
    lp = out["logp"].cpu().numpy().astype(np.float64)
    assert np.abs(lp - ref["logp"]).max() <= TOL_LOGP_STATED
    assert np.abs(lp - ref["logp"]).max() <= TOL_LOGP_STRICT
    assert np.abs(out["entropy"].cpu().numpy() - ref["entropy"]).max() <= TOL_LOGP_STRICT
    f = out["flags"].cpu().numpy()
    assert np.array_equal(f & 0xD, ref["flags"] & 0xD)
    advt = np.repeat(ref["adv"], np.diff(npb["cu_seqlens"]))
    rule = oracle.clip_active_vec(out["logp"].cpu().numpy(), npb["logp_old"], advt, p.eps_low, p.eps_high)
    assert np.array_equal((f >> 1) & 1, rule)
    rng = np.random.default_rng(seed)
    # vocabulary rows: both ends, tile edges, the targets of a few tokens, and a random sample
    vids = np.unique(np.concatenate([[0, V - 1, 255, 256, 511, 512], npb["targets"][rng.choice(T, 16)],
                                     rng.choice(V, n_vocab_rows, replace=False)]))[:n_vocab_rows]
    dw_ref, dw_mag, dw_l2 = oracle.projection_dw_rows(vids, h64, W64, npb["targets"], ref["logp"], ref["g"],
                                                      magnitudes=True)
    dw = out["dw_lm"][torch.as_tensor(vids, device="cuda"), :H].double().cpu().numpy()
    rep = _grad_close("dW", dw, dw_ref, dw_mag, dw_l2, T, False)
    tids = np.unique(np.concatenate([[0, T - 1, min(4095, T - 1), min(4096, T - 1)],
                                     rng.choice(T, n_token_rows, replace=False)]))
    n, adv, w = oracle.seq_prep(npb["cu_seqlens"], npb["mask"], npb["rewards_or_adv"], p)
    rows = oracle.projection_rows(tids, hb, None, npb["targets"], npb["logp_old"], npb["logp_infer"], npb["mask"],
                                  npb["cu_seqlens"], adv, w, p, want_dh=True, w64=W64)
    dh = out["dhidden"][torch.as_tensor(tids, device="cuda"), :H].double().cpu().numpy()
    dz = rows["dz"]
    rep.update(_grad_close("dhidden", dh, rows["dh"], np.abs(dz) @ np.abs(W64), np.sqrt((dz * dz) @ (W64 * W64)), V,
                           True))
    rep.update(loss=L, loss_oracle=ref["loss"], logp_max_err=float(np.abs(lp - ref["logp"]).max()))
    return rep


def test_fused_projection_mid_size_exact():
    """8,192 tokens (two 4,096-row chunks) x V = 32,768 x H = 6,144: the exact loss,
    every row's log-prob, and 256 dL/dW rows and 64 dL/dh rows element by element."""
    pb = synthetic.make_projection_batch("cuda", prompts=8, vocab=32768)
    rl = capi.projection_handle(pb)
    out = capi.alloc_projection_outputs(pb)
    capi.run_projection(rl, pb, out)
    torch.cuda.synchronize()
    assert rl.device_status() & ~(1 << capi.CODES["RL_ERR_EMPTY_SEQ"]) == 0
    print(_check_exact_forward_and_sampled_grads(pb, out))


@pytest.mark.slow
@pytest.mark.skipif(os.environ.get("RL_LOSS_FULL_ORACLE") != "1",
                    reason="the exact full-size oracle takes minutes of host time: set RL_LOSS_FULL_ORACLE=1")
def test_fused_projection_full_size_exact_loss_and_dw_rows():
    """The full case (65,536 tokens x V = 151,552 x H = 6,144): the loss against the
    exact fp64 loss streamed over every row, and 256 dL/dW rows element by element."""
    torch.cuda.empty_cache()
    pb = synthetic.make_projection_batch("cuda")
    rl = capi.projection_handle(pb)
    out = capi.alloc_projection_outputs(pb)
    capi.run_projection(rl, pb, out)
    torch.cuda.synchronize()
    assert rl.device_status() & ~(1 << capi.CODES["RL_ERR_EMPTY_SEQ"]) == 0
    print(_check_exact_forward_and_sampled_grads(pb, out))


@pytest.mark.slow
def test_fused_projection_full_size_sampled():
    torch.cuda.empty_cache()
    pb = synthetic.make_projection_batch("cuda")
    b = pb.batch
    rl = capi.projection_handle(pb)
    out = capi.alloc_projection_outputs(pb)
    capi.run_projection(rl, pb, out)
    torch.cuda.synchronize()
    assert rl.device_status() & ~(1 << capi.CODES["RL_ERR_EMPTY_SEQ"]) == 0
    T, H = b.num_tokens, pb.hidden_dim
    p = params_for(b)
    npb = {k: getattr(b, k).cpu().numpy() for k in
           ("targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv")}
    n, adv, w = oracle.seq_prep(npb["cu_seqlens"], npb["mask"], npb["rewards_or_adv"], p)
    rng = np.random.default_rng(4)
    ids = np.unique(np.concatenate([[0, T - 1, 4095, 4096], rng.choice(T, 28, replace=False)]))
    wb = _bits(pb.w[:, :H])
    ref = oracle.projection_rows(ids, _bits(pb.hidden[:, :H]), wb, npb["targets"], npb["logp_old"],
                                 npb["logp_infer"], npb["mask"], npb["cu_seqlens"], adv, w, p, want_dh=True)
    lp = out["logp"].cpu().numpy()[ids].astype(np.float64)
    assert np.abs(lp - ref["logp"]).max() <= TOL_LOGP_STATED
    assert np.abs(lp - ref["logp"]).max() <= TOL_LOGP_STRICT
    assert np.abs(out["entropy"].cpu().numpy()[ids] - ref["entropy"]).max() <= TOL_LOGP_STRICT
    assert np.array_equal(out["flags"].cpu().numpy()[ids] & 0xD, ref["flags"] & 0xD)
    dh = out["dhidden"][torch.as_tensor(ids, device="cuda"), :H].double().cpu().numpy()
    nz = np.linalg.norm(ref["dh"], axis=1) > 0
    rn = np.linalg.norm(dh - ref["dh"], axis=1)[nz] / np.linalg.norm(ref["dh"], axis=1)[nz]
    assert rn.size == 0 or rn.max() <= 1e-2, rn.max()
    # identity at any size: sum_t <dH_t, h_t> = sum_{t,v} dZ_tv z_tv = sum_v <dW_v, W_v>
    lhs = (out["dhidden"][:, :H].double() * pb.hidden[:, :H].double()).sum().item()
    rhs = (out["dw_lm"][:, :H].double() * pb.w[:, :H].double()).sum().item()
    assert abs(lhs - rhs) <= 1e-2 * max(abs(lhs), abs(rhs)) + 1e-9, (lhs, rhs)
    print({"logp_max_err": float(np.abs(lp - ref["logp"]).max()), "dh_row_rel_l2_max": float(rn.max()),
           "trace_dH_h": lhs, "trace_dW_W": rhs, "loss": out["loss_f64"].item()})
