"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on the
seeded workloads at sizes the oracle finishes in seconds, plus edge cases,
error paths and run-to-run determinism."""
import hashlib

import numpy as np
import pytest
import torch

from parity_helpers import OracleRun, check_all, params_for
from rl_post_loss_gb300 import build as nvbuild
from rl_post_loss_gb300 import capi, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nvbuild.build()
    capi.load()


def _run(batch, in_place=False, ld_out=None, **over):
    rl = capi.handle_for_batch(batch, **over)
    out = capi.alloc_outputs(batch, in_place=in_place, ld=ld_out)
    capi.run_batch(rl, batch, out)
    torch.cuda.synchronize()
    bits = rl.device_status()
    return rl, out, bits


def _lengths(case_id, n_prompts, lo, hi, seed=0):
    g = np.random.default_rng(1234 + case_id + seed)
    G = synthetic.CASES[case_id]["group"]
    return [int(x) for x in g.integers(lo, hi + 1, size=n_prompts * G)]


def test_case0_full_size_every_row():
    b = synthetic.make_batch(0, "cuda")
    _, out, bits = _run(b)
    assert bits == 0
    rep = {}
    check_all(b, out, dz_rows="all", report=rep)
    assert rep["ambiguous_clip"] <= 1


@pytest.mark.parametrize("case_id,n_prompts,lo,hi,dz_rows", [
    (1, 2, 8, 64, "all"),
    (2, 1, 40, 160, 96),
    (3, 4, 48, 96, 96),
])
def test_cases_reduced_length_full_vocab(case_id, n_prompts, lo, hi, dz_rows):
    b = synthetic.make_batch(case_id, "cuda", lengths=_lengths(case_id, n_prompts, lo, hi))
    _, out, bits = _run(b)
    assert bits & ~(1 << capi.CODES["RL_ERR_EMPTY_SEQ"]) == 0
    check_all(b, out, dz_rows=dz_rows)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 13, 1001, 4097, 8961, 40000, 70001, 151553, 200003])
def test_ragged_vocab_and_padded_rows(dtype, V):
    # rows up to 128 KB take the 256-thread kernel, longer ones the 1024-thread kernel with a
    # staged shared-memory prefix (fp32 from V = 40000, bf16 from V = 70001); every V leaves a
    # ragged tail for some thread, and the padded strides check that columns >= V stay untouched
    lengths = _lengths(0, 1, 3, 40)
    ld = synthetic.padded_ld(V, dtype) + (64 if V % 2 else 0)
    b = synthetic.make_batch(0, "cuda", lengths=lengths, vocab=V, ld=ld, case_overrides={"dtype": dtype})
    _, out, bits = _run(b, ld_out=synthetic.padded_ld(V, dtype) + 8)
    assert bits == 0
    check_all(b, out, dz_rows="all")


def test_padding_columns_untouched_and_in_place():
    V, dtype = 1001, "bf16"
    b = synthetic.make_batch(0, "cuda", lengths=_lengths(0, 1, 5, 30), vocab=V, case_overrides={"dtype": dtype})
    ld = b.logits.stride(0)
    rl, out, _ = _run(b)
    ref = out["dlogits"][:, :V].clone()
    sentinel = capi.alloc_outputs(b)
    sentinel["dlogits"].fill_(7.0)
    capi.run_batch(rl, b, sentinel)
    torch.cuda.synchronize()
    assert torch.equal(sentinel["dlogits"][:, :V], ref)
    assert bool((sentinel["dlogits"][:, V:ld] == 7.0).all())
    # in place: dlogits aliases logits
    b2 = synthetic.make_batch(0, "cuda", lengths=b.meta["lengths"], vocab=V, case_overrides={"dtype": dtype})
    inp = capi.alloc_outputs(b2, in_place=True)
    capi.run_batch(rl, b2, inp)
    torch.cuda.synchronize()
    assert torch.equal(b2.logits[:, :V], ref)
    assert torch.equal(inp["loss_f64"], out["loss_f64"])


def test_clip_heavy_inputs_and_variants():
    over = {"old_noise": 0.35, "infer_noise": 0.4}
    b = synthetic.make_batch(1, "cuda", lengths=_lengths(1, 2, 8, 40), case_overrides=over)
    _, out, _ = _run(b)
    cnt = out["counts"].cpu().numpy()
    assert cnt[0] > 0 and cnt[1] > 0, cnt  # both popped and clipped tokens occur
    check_all(b, out, dz_rows="all")
    for kw in (dict(pop_indicator=True), dict(std_unbiased=True), dict(beta=1.25, eps_low=0.1, eps_high=0.1)):
        _, out, _ = _run(b, **kw)
        p = params_for(b, **{k: (int(v) if isinstance(v, bool) else v) for k, v in kw.items()})
        check_all(b, out, p=p, dz_rows=64)


def test_single_token_and_empty_batch():
    b = synthetic.make_batch(3, "cuda", lengths=[1], vocab=4096, case_overrides={"prompts": 1})
    _, out, bits = _run(b)
    check_all(b, out, dz_rows="all")
    e = synthetic.make_batch(0, "cuda", lengths=[0, 0, 0, 0])
    assert e.num_tokens == 0
    rl = capi.handle_for_batch(e, max_tokens=16)
    out = capi.alloc_outputs(e)
    capi.run_batch(rl, e, out)
    torch.cuda.synchronize()
    assert float(out["loss"].cpu()[0]) == 0.0
    assert rl.device_status() == 1 << capi.CODES["RL_ERR_EMPTY_SEQ"]
    assert out["counts"].cpu().tolist() == [0, 0, 0, 4]


def test_fully_masked_response_warns_and_adds_zero():
    b = synthetic.make_batch(1, "cuda", lengths=_lengths(1, 1, 8, 30))
    cu = b.cu_seqlens.cpu().numpy()
    b.mask[cu[2]:cu[3]] = 0
    _, out, bits = _run(b)
    assert bits == 1 << capi.CODES["RL_ERR_EMPTY_SEQ"]
    run = check_all(b, out, dz_rows="all")
    assert run.n[2] == 0 and out["counts"].cpu().tolist()[3] == 1


def test_bad_targets_are_flagged_and_excluded():
    b = synthetic.make_batch(0, "cuda", lengths=_lengths(0, 1, 4, 20))
    b.targets[1] = b.vocab
    b.targets[3] = -1
    _, out, bits = _run(b)
    assert bits & (1 << capi.CODES["RL_ERR_TARGET_RANGE"])
    f = out["flags"].cpu().numpy()
    assert f[1] & 8 and f[3] & 8
    assert bool((out["dlogits"][1] == 0).all()) and bool((out["dlogits"][3] == 0).all())
    check_all(b, out, dz_rows="all")


def test_minus_infinity_logits_are_zero_probability():
    """A -inf logit (a masked vocabulary entry) is valid: probability 0, no entropy term
    (0 log 0 = 0), a zero gradient, no status bit; the short-row and the long-row kernel.
    One row keeps only its target finite: log-prob 0 and entropy 0."""
    for dtype, V in (("f32", 4096), ("bf16", 200003)):
        b = synthetic.make_batch(0, "cuda", lengths=_lengths(0, 1, 10, 40), vocab=V,
                                 case_overrides={"dtype": dtype})
        g = torch.Generator(device="cuda").manual_seed(V)
        hole = torch.rand((b.num_tokens, V), generator=g, device="cuda") < 0.1
        hole[torch.arange(b.num_tokens, device="cuda"), b.targets.long()] = False
        hole[3] = True
        hole[3, b.targets[3].long()] = False
        view = b.logits[:, :V]
        view[hole] = float("-inf")
        _, out, bits = _run(b)
        assert bits == 0, capi.status_bits_to_names(bits)
        assert bool(torch.isfinite(out["entropy"]).all()) and bool(torch.isfinite(out["loss_f64"]).all())
        assert abs(out["logp"][3].item()) <= 1e-6 and abs(out["entropy"][3].item()) <= 1e-6
        assert bool((out["dlogits"][:, :V][hole] == 0).all())
        check_all(b, out, dz_rows="all" if dtype == "f32" else 16)


def test_nonfinite_and_malformed_offsets_raise_device_bits():
    for dtype, V in (("f32", 4096), ("bf16", 200003)):  # the short-row and the long-row kernel
        for bad in (float("nan"), float("inf")):
            b = synthetic.make_batch(0, "cuda", lengths=_lengths(0, 1, 4, 20), vocab=V,
                                     case_overrides={"dtype": dtype})
            b.rewards_or_adv.fill_(1.0)  # zero advantages: the row adds nothing to the loss
            b.logits[2, 5] = bad
            _, out, bits = _run(b)
            assert bits & (1 << capi.CODES["RL_ERR_NONFINITE"]), (dtype, bad)
    b = synthetic.make_batch(0, "cuda", lengths=_lengths(0, 1, 4, 20))
    b.cu_seqlens[-1] -= 1  # last response ends before num_tokens
    _, out, bits = _run(b)
    assert bits & (1 << capi.CODES["RL_ERR_SEQLENS"])


def test_host_side_argument_errors_launch_nothing():
    b = synthetic.make_batch(0, "cuda", lengths=_lengths(0, 1, 4, 20))
    rl = capi.handle_for_batch(b, max_tokens=b.num_tokens - 1)
    out = capi.alloc_outputs(b)
    before = rl.launch_count()
    with pytest.raises(capi.RlLossError) as e:
        capi.run_batch(rl, b, out)
    assert e.value.code == capi.CODES["RL_ERR_CAPACITY"]
    rl = capi.handle_for_batch(b)
    bad = b.to("cuda")
    bad.logits = torch.zeros((b.num_tokens, b.vocab + 1), dtype=b.logits.dtype, device="cuda")
    with pytest.raises(capi.RlLossError) as e:
        capi.run_batch(rl, bad, out)
    assert e.value.code == capi.CODES["RL_ERR_ALIGNMENT"]
    bad = b.to("cuda")
    bad.cu_seqlens = b.cu_seqlens[:4]  # 3 responses, G = 4
    with pytest.raises(capi.RlLossError) as e:
        capi.run_batch(rl, bad, out)
    assert e.value.code == capi.CODES["RL_ERR_SHAPE"]
    assert rl.launch_count() == 0 and before == 0


def _digest(out):
    h = hashlib.sha256()
    for k in sorted(out):
        h.update(out[k].contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()


def test_bit_identical_across_runs_and_streams():
    b = synthetic.make_batch(2, "cuda", lengths=_lengths(2, 1, 64, 200))
    rl = capi.handle_for_batch(b)
    digests = set()
    for k in range(5):
        out = capi.alloc_outputs(b)
        s = torch.cuda.Stream() if k % 2 else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            capi.run_batch(rl, b, out)
        torch.cuda.synchronize()
        digests.add(_digest(out))
    assert len(digests) == 1


def test_profile_and_launch_count():
    b = synthetic.make_batch(0, "cuda")
    rl = capi.handle_for_batch(b)
    out = capi.alloc_outputs(b)
    rl.profile_start(3)
    for _ in range(3):
        capi.run_batch(rl, b, out)
    prof = rl.profile_read()
    used = {"seg_prep", "token_prep", "row_loss", "entropy_fix", "seg_reduce", "final_reduce"}
    assert used <= set(prof)
    assert all(prof[k][0] == 3 and prof[k][1] > 0 for k in used)
    assert all(n == 0 for k, (n, _) in prof.items() if k not in used)
    assert rl.launch_count() == 18


def test_alternating_vocab_sizes_on_one_kernel_configuration():
    # the long-row kernel serves V = 151552 and V = 70001 with different dynamic shared-memory
    # sizes (its staged prefix); launching them in turn must keep working
    for V in (151552, 70001, 151552, 70001):
        b = synthetic.make_batch(2, "cuda", lengths=_lengths(2, 1, 8, 24), vocab=V)
        _, out, bits = _run(b)
        assert bits & ~(1 << capi.CODES["RL_ERR_EMPTY_SEQ"]) == 0
        check_all(b, out, dz_rows=16)


@pytest.mark.parametrize("over", [
    dict(objective=1, token_adv="normal", loss_norm=1),                        # DIS, per-token A, token mean
    dict(objective=1, token_adv="normal", loss_norm=1, old_noise=0.2, infer_noise=0.25),
    dict(objective=1, loss_norm=0),                                            # DIS, group-normalised A
    dict(token_adv="teacher", group=1, prompts=16),                           # OPD: A_t = teacher - logp
    dict(token_adv="normal"),                                                  # Eq. (1), per-token A
    dict(loss_norm=1),                                                         # Eq. (1), token mean
])
def test_objective_and_advantage_variants(over):
    G = over.get("group", 8)
    n = over.get("prompts", 2) * G
    rng = np.random.default_rng(99)
    lengths = [int(x) for x in rng.integers(8, 60, size=n)]
    b = synthetic.make_batch(1, "cuda", lengths=lengths, case_overrides=over)
    for stop in ((True, False) if over.get("objective") == 1 else (True,)):
        _, out, bits = _run(b, dis_stopgrad=stop)
        assert bits & ~(1 << capi.CODES["RL_ERR_EMPTY_SEQ"]) == 0
        check_all(b, out, p=params_for(b, dis_stopgrad=int(stop)), dz_rows="all")


def test_dis_variants_in_fused_projection():
    pb = synthetic.make_projection_batch("cuda", prompts=2, group=4, length=40, hidden=128, vocab=900, chunk=100)
    b = pb.batch
    b.objective, b.loss_norm = 1, 1
    rl = capi.projection_handle(pb)
    out = capi.alloc_projection_outputs(pb)
    capi.run_projection(rl, pb, out)
    torch.cuda.synchronize()
    import oracle
    bits = lambda t: t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    npb = {k: getattr(b, k).cpu().numpy() for k in
           ("targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv")}
    ref = oracle.projection_forward_backward(bits(pb.hidden), bits(pb.w), npb, params_for(b))
    assert abs(out["loss_f64"].item() - ref["loss"]) <= 1e-4 * abs(ref["loss"]) + 1e-12
    dh = out["dhidden"].double().cpu().numpy()
    assert np.linalg.norm(dh - ref["dh"]) <= 1e-2 * np.linalg.norm(ref["dh"])
