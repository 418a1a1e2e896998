"""Skip-observation GAE (segmented reverse scan) on the GPU against the fp64
oracle: several layouts, the cross-trajectory discount, edge cases, full size,
determinism.

Tolerance, derived from the kernel's fp32 arithmetic. Every action token's
advantage is a weighted sum A_t = sum_k x^k delta_{t+k} (x = gamma lambda, k
counting action tokens), evaluated by the kernel through per-thread folds, a
fixed-tree scan and a per-thread re-walk, with the carry between tiles held in
double. Each term passes through at most about 64 fp32 roundings in any one
tile (fewer than 41 more per tile boundary crossed), and the weight x^k is a
product of k rounded factors, so
  |err_t| <= u (128 S0_t + 2 S1_t) + 2 u |A_t|,
  S0_t = sum_k x^k M_{t+k},  S1_t = sum_k k x^k M_{t+k},
  M_j = |r_j| + |V_j| + gamma |V_next(j)|,  u = 2^-24,
with S1 dropped when fl32(x) is 0 or 1 (the products are then exact); the
cross-trajectory factor scales the bound and adds one rounding.
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
        b = 128.0 * s0
        if not exact_powers:
            z = np.append(x * s0[1:], 0.0)
            b = b + 2.0 * _reverse_geometric(x, z)
        a_unscaled = np.abs(ref[idx]) / np.where(scale[idx] > 0, scale[idx], 1.0)
        bound[idx] = U32 * (b + 2.0 * a_unscaled) * scale[idx] + U32 * np.abs(ref[idx])
    return bound * 1.0001 + 1e-30


@pytest.mark.parametrize("lengths", [[1], [5, 0, 7], [1000, 1024, 1025, 3000], [40] * 64, [20000, 16384]])
@pytest.mark.parametrize("skip,cross", [(True, False), (False, False), (True, True)])
def test_gae_layouts(lengths, skip, cross):
    gb = synthetic.make_gae_batch("cuda", lengths=lengths, segments=2)
    _check(gb, skip=skip, cross=cross)


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
