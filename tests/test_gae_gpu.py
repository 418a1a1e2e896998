"""Skip-observation GAE (segmented reverse scan) on the GPU against the fp64
oracle: several layouts, the cross-trajectory discount, edge cases, full size,
determinism.

Tolerance, derived from the kernel's fp32 arithmetic. Every action token's
advantage is a weighted sum A_t = sum_k x^k delta_{t+k} (x = gamma lambda, k
counting action tokens), evaluated by the kernel through per-thread folds of 32
tokens, a fixed tree over the 256 threads of an 8192-token chunk, a look-back
tree over the chunks to the right, and a per-thread re-walk. A composition adds
at most 3 roundings to a term, so a term passes through at most about 170 fp32
roundings (fold 33, the chunk's tree 24, the look-back tree 15 plus 3 for every
further 32 chunks, the exclusive tree 27, the re-walk 64), and the weight x^k
is a product of k rounded factors, so
  |err_t| <= u (256 S0_t + 2 S1_t) + 2 u |A_t|,
  S0_t = sum_k x^k M_{t+k},  S1_t = sum_k k x^k M_{t+k},
  M_j = |r_j| + |V_j| + gamma |V_next(j)|,  u = 2^-24,
with S1 dropped when fl32(x) is 0 or 1 (the products are then exact). The
cross-trajectory factor (gamma lambda)^N, evaluated as 2^(N log2 x) with a
degree-7 Taylor series for the fractional power, is within 3u of exact: it
scales the bound, adds 4 u |A_t| and one rounding of the product, and 2^-147
absolute for products below the normal range.
"""
import numpy as np
import pytest
import torch
from scipy.signal import lfilter

import oracle
from rl_post_loss_gb300 import build as nvbuild
from rl_post_loss_gb300 import capi, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nvbuild.build()
    capi.load()


def _check(gb, skip=True, cross=False, gamma=None, lam=None):
    gamma = gb.gamma if gamma is None else gamma
    lam = gb.lam if lam is None else lam
    ro = gb.rollout_ids if cross else None
    ret = torch.empty_like(gb.rewards)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    adv = capi.gae(gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gamma, lam, skip, rollout_ids=ro, returns=ret,
                   device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.gae(gb.cu_seqlens.cpu().numpy(), gb.rewards.cpu().numpy(), gb.values.cpu().numpy(),
                     gb.mask.cpu().numpy(), gamma, lam, skip, None if ro is None else ro.cpu().numpy())
    got = adv.double().cpu().numpy()
    act = gb.mask.cpu().numpy().astype(bool) if skip else np.ones(ref.shape, bool)
    bound = gae_error_bound(gb, ref, act, gamma, lam, ro is not None)
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"max excess {(err - bound).max()}, max err {err.max()}"
    r = ret.double().cpu().numpy()
    want_ret = ref + gb.values.double().cpu().numpy()
    rb = bound + U32 * np.abs(want_ret)
    assert np.all(np.abs(r[act] - want_ret[act]) <= rb[act])
    if skip:
        assert np.all(got[~act] == 0.0)
    return adv


U32 = 2.0 ** -24


def _reverse_geometric(x, seq):
    """y_j = sum_{k>=0} x^k seq_{j+k}."""
    return lfilter([1.0], [1.0, -x], seq[::-1])[::-1] if seq.size else seq


def gae_error_bound(gb, ref, act, gamma, lam, cross):
    """The fp32 error bound stated in the module docstring, per token."""
    cu = gb.cu_seqlens.cpu().numpy()
    r = np.abs(gb.rewards.double().cpu().numpy())
    v = np.abs(gb.values.double().cpu().numpy())
    x = gamma * lam
    x32 = float(np.float32(x))
    exact_powers = x32 in (0.0, 1.0)
    scale = np.ones(ref.size)
    if cross:
        mask = gb.mask.cpu().numpy()
        ro = gb.rollout_ids.cpu().numpy()
        for s in range(cu.size - 1):
            later, u = 0, s + 1
            while u < cu.size - 1 and ro[u] == ro[s]:
                later += int(mask[cu[u]:cu[u + 1]].sum())
                u += 1
            scale[cu[s]:cu[s + 1]] = x ** later
    bound = np.zeros(ref.size)
    for s in range(cu.size - 1):
        idx = cu[s] + np.nonzero(act[cu[s]:cu[s + 1]])[0]
        if idx.size == 0:
            continue
        vn = np.append(v[idx[1:]], 0.0)
        M = r[idx] + v[idx] + gamma * vn
        s0 = _reverse_geometric(x, M)
        b = 256.0 * s0
        if not exact_powers:
            z = np.append(x * s0[1:], 0.0)
            b = b + 2.0 * _reverse_geometric(x, z)
        a_unscaled = np.abs(ref[idx]) / np.where(scale[idx] > 0, scale[idx], 1.0)
        extra = 4.0 if cross else 0.0
        bound[idx] = U32 * (b + (2.0 + extra) * a_unscaled) * scale[idx] + U32 * np.abs(ref[idx])
        if cross:
            bound[idx] += 2.0 ** -147
    return bound * 1.0001 + 1e-30


@pytest.mark.parametrize("lengths", [[1], [5, 0, 7], [1000, 1024, 1025, 3000], [40] * 64, [20000, 16384],
                                     [33, 31, 1, 2, 64, 63, 65, 100, 7, 25] * 30])
@pytest.mark.parametrize("skip,cross", [(True, False), (False, False), (True, True)])
def test_gae_layouts(lengths, skip, cross):
    gb = synthetic.make_gae_batch("cuda", lengths=lengths, segments=2)
    _check(gb, skip=skip, cross=cross)


@pytest.mark.parametrize("lengths,segments", [([9000, 8000, 20000, 12000], 2), ([5000, 7000, 300, 9000, 4100, 1], 3),
                                               ([70000, 3000, 40000, 1, 5000], 5)])
def test_gae_cross_trajectory_discount_without_underflow(lengths, segments):
    # gamma lambda close to 1: (gamma lambda)^N stays well inside the fp32 range over whole segments
    gb = synthetic.make_gae_batch("cuda", lengths=lengths, segments=segments)
    adv = _check(gb, cross=True, gamma=1.0, lam=0.9999)
    assert float(adv.abs().min()) >= 0.0 and int((adv != 0).sum()) > 0.5 * int(gb.mask.sum())


@pytest.mark.parametrize("gamma,lam", [(1.0, 1.0), (1.0, 0.0), (0.99, 0.95), (0.0, 0.5)])
def test_gae_parameters(gamma, lam):
    gb = synthetic.make_gae_batch("cuda", lengths=[3000, 257, 4096, 1])
    _check(gb, gamma=gamma, lam=lam, cross=True)


def test_gae_all_observation_response_and_bad_offsets():
    gb = synthetic.make_gae_batch("cuda", lengths=[50, 60])
    gb.mask[50:] = 0
    adv = _check(gb)
    assert bool((adv[50:] == 0).all())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu = gb.cu_seqlens.clone()
    cu[-1] += 5  # runs past num_tokens
    capi.gae(gb.rewards, gb.values, gb.mask, cu, 1.0, 0.9, device_status=st)
    torch.cuda.synchronize()
    assert st.item() & (1 << capi.CODES["RL_ERR_SEQLENS"])


@pytest.mark.slow
def test_gae_full_size_and_bit_identical():
    gb = synthetic.make_gae_batch("cuda")
    a1 = _check(gb, cross=True)
    a2 = capi.gae(gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.gamma, gb.lam, True, rollout_ids=gb.rollout_ids)
    torch.cuda.synchronize()
    assert torch.equal(a1.view(torch.int32), a2.view(torch.int32))


def _workspace_is_clear(T):
    """The ticket and done counters are zero again (a chunk's record counts only under the tag of
    the launch that wrote it, so the records need no clearing), and the launch epoch is set."""
    ws = capi.gae_workspace(T, torch.device("cuda", torch.cuda.current_device()))
    torch.cuda.synchronize()
    assert ws.data_ptr() == capi.gae_workspace(T, "cuda").data_ptr()
    words = ws.view(torch.int32).cpu().numpy()
    return bool(np.all(words[:2] == 0)) and int(words[2]) != 0


def test_gae_long_responses_span_many_chunks():
    # 300000 tokens = 37 chunks of 8192: the look-back composes more than one window of 32 chunks
    gb = synthetic.make_gae_batch("cuda", lengths=[300000, 3, 140000, 70000], segments=2)
    _check(gb, cross=True)
    _check(gb, skip=False)
    assert _workspace_is_clear(gb.num_tokens)


def test_gae_empty_responses_and_rollout_breaks():
    lengths = [0, 500, 0, 0, 4100, 0, 7, 0, 9000, 1]
    gb = synthetic.make_gae_batch("cuda", lengths=lengths, segments=3)
    # an empty response with another rollout id between two segments of rollout 0 ends that rollout
    gb.rollout_ids.copy_(torch.tensor([0, 0, 1, 0, 0, 0, 2, 2, 2, 3], dtype=torch.int32))
    _check(gb, cross=True)
    _check(gb, cross=False)


def test_gae_unaligned_arrays_take_the_scalar_path():
    base = synthetic.make_gae_batch("cuda", lengths=[3000, 5000, 1234, 4096], segments=2)
    T = base.num_tokens

    def shifted(t):
        buf = torch.zeros(T + 1, dtype=t.dtype, device=t.device)
        buf[1:] = t
        return buf[1:]

    gb = synthetic.GaeBatch(rewards=shifted(base.rewards), values=shifted(base.values), mask=shifted(base.mask),
                            cu_seqlens=base.cu_seqlens, rollout_ids=base.rollout_ids, gamma=base.gamma, lam=base.lam)
    assert gb.rewards.data_ptr() % 16 != 0 and gb.mask.data_ptr() % 16 != 0
    a_scalar = _check(gb, cross=True)
    a_vec = _check(base, cross=True)
    assert torch.equal(a_scalar.view(torch.int32), a_vec.view(torch.int32))


def test_gae_tokens_outside_the_responses_are_not_written():
    lengths = [5000, 0, 3100]
    gb = synthetic.make_gae_batch("cuda", lengths=lengths, segments=1)
    pad_l, pad_r = 100, 4200
    T = gb.num_tokens + pad_l + pad_r

    def padded(t):
        buf = torch.zeros(T, dtype=t.dtype, device=t.device)
        buf[pad_l:pad_l + t.numel()] = t
        return buf

    r, v, m = padded(gb.rewards), padded(gb.values), padded(gb.mask)
    m[:pad_l] = 1
    m[pad_l + gb.num_tokens:] = 1
    cu = gb.cu_seqlens + pad_l
    adv = torch.full((T,), 7.0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.gae(r, v, m, cu, gb.gamma, gb.lam, True, advantages=adv, device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = adv.cpu().numpy()
    assert np.all(got[:pad_l] == 7.0) and np.all(got[pad_l + gb.num_tokens:] == 7.0)
    ref = oracle.gae(cu.cpu().numpy(), r.cpu().numpy(), v.cpu().numpy(), m.cpu().numpy(), gb.gamma, gb.lam, True)
    inner = slice(pad_l, pad_l + gb.num_tokens)
    bound = gae_error_bound(gb, ref[inner], gb.mask.cpu().numpy().astype(bool), gb.gamma, gb.lam, False)
    assert np.all(np.abs(got[inner] - ref[inner]) <= bound)


def test_gae_repeated_calls_are_bit_identical_and_leave_the_workspace_clear():
    gb = synthetic.make_gae_batch("cuda", lengths=[20000, 7, 65536, 300, 12000] * 4, segments=2)
    outs = []
    for _ in range(4):
        outs.append(capi.gae(gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.gamma, gb.lam, True,
                             rollout_ids=gb.rollout_ids))
        torch.cuda.synchronize()
        assert _workspace_is_clear(gb.num_tokens)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))


def test_a_withheld_chunk_map_runs_the_bounded_wait_out():
    """Failure detection without a fault: the map of chunk 20 of a 300,000-token response
    (37 chunks) is never published, so the look-back of the chunks to its left waits for it
    until the 20-ms bound runs out. The call must complete with RL_ERR_TIMEOUT raised; the
    withheld chunk and those to its right (which never wait for it) must equal a normal call
    bit for bit while the chunks to its left differ; the workspace must be clear again, and
    the next normal call must repeat the first one bit for bit."""
    import time
    gb = synthetic.make_gae_batch("cuda", lengths=[300000, 3, 140000, 70000], segments=2)
    T, S = gb.num_tokens, gb.cu_seqlens.numel() - 1
    ref = capi.gae(gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.gamma, gb.lam, True, rollout_ids=gb.rollout_ids)
    torch.cuda.synchronize()
    w = 20
    adv = torch.full((T,), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = capi.gae_workspace(T, "cuda")
    cfg = capi.rl_gae_config(gb.gamma, gb.lam, 1, 1)
    p = capi._ptr
    t0 = time.perf_counter()
    rc = capi.rl_gae_advantages_withheld(cfg, T, S, p(gb.rewards), p(gb.values), p(gb.mask), p(gb.cu_seqlens),
                                         p(gb.rollout_ids), p(adv), None, p(ws), ws.numel(), p(st),
                                         torch.cuda.current_stream().cuda_stream, w, 0.02)
    assert rc == 0
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert capi.status_bits_to_names(int(st.item())) == ["RL_ERR_TIMEOUT"]
    lo = w * 8192
    assert torch.equal(adv[lo:].view(torch.int32), ref[lo:].view(torch.int32))
    assert not torch.equal(adv[:lo], ref[:lo])
    assert _workspace_is_clear(T)
    st.zero_()
    again = capi.gae(gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.gamma, gb.lam, True,
                     rollout_ids=gb.rollout_ids, device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(again.view(torch.int32), ref.view(torch.int32))
    # arguments the injection entry point refuses before launching anything
    for bad_w, bad_s in ((-1, 0.02), (w, 0.0), (w, 2.0)):
        assert capi.rl_gae_advantages_withheld(cfg, T, S, p(gb.rewards), p(gb.values), p(gb.mask),
                                               p(gb.cu_seqlens), p(gb.rollout_ids), p(adv), None, p(ws),
                                               ws.numel(), p(st), 0, bad_w, bad_s) == capi.CODES["RL_ERR_INVALID_ARG"]


@pytest.mark.slow
def test_gae_full_size_repeated_launches_are_bit_identical():
    """Ten launches on the full workload (2048 chunks, several waves): the tickets go to whichever
    block asks first and the look-back waits on whatever is published, yet every advantage must
    come out bit-identical and the workspace clear."""
    gb = synthetic.make_gae_batch("cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run = lambda: capi.gae(gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.gamma, gb.lam, True,
                           rollout_ids=gb.rollout_ids, device_status=st)
    a0 = run().clone()
    for _ in range(10):
        a1 = run()
        torch.cuda.synchronize()
        assert torch.equal(a0.view(torch.int32), a1.view(torch.int32))
    assert st.item() == 0
    assert _workspace_is_clear(gb.num_tokens)


def test_records_of_an_earlier_call_are_never_read():
    """A chunk's published map counts only under the tag of the launch that wrote it: a call on a
    workspace that holds another batch's records (same token count) must equal the same call on a
    fresh, zeroed workspace, bit for bit."""
    a = synthetic.make_gae_batch("cuda", seed=0, lengths=[300000, 3, 140000, 70000], segments=2)
    b = synthetic.make_gae_batch("cuda", seed=1, lengths=[300000, 3, 140000, 70000], segments=2)
    T = a.num_tokens
    ws = torch.zeros(capi.rl_gae_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    capi.gae(a.rewards, a.values, a.mask, a.cu_seqlens, a.gamma, a.lam, True, rollout_ids=a.rollout_ids, workspace=ws)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = capi.gae(b.rewards, b.values, b.mask, b.cu_seqlens, b.gamma, b.lam, True, rollout_ids=b.rollout_ids,
                   workspace=ws, device_status=st)
    fresh = torch.zeros_like(ws)
    want = capi.gae(b.rewards, b.values, b.mask, b.cu_seqlens, b.gamma, b.lam, True, rollout_ids=b.rollout_ids,
                    workspace=fresh)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    assert not torch.equal(got, capi.gae(a.rewards, a.values, a.mask, a.cu_seqlens, a.gamma, a.lam, True,
                                          rollout_ids=a.rollout_ids, workspace=fresh))
