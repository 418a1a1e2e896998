"""The entry points inside CUDA graphs.

rl_loss_forward_backward (with a handle), rl_gae_advantages and rl_topk
allocate nothing, never synchronise and launch only on the given stream, so a
caller can capture them into a CUDA graph once and replay it every step
(which removes the launch cost that dominates small batches). These tests
capture each of them with torch.cuda.CUDAGraph after one warm-up call (the
per-device setup runs outside the capture), replay the graph and require
results bit-identical to an eager call; then change the inputs in place and
require the replay to follow them.
"""
import pytest
import torch

from rl_post_loss_gb300 import build as nvbuild
from rl_post_loss_gb300 import capi, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nvbuild.build()
    capi.load()


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # warm-up: first-use setup (shared-memory opt-ins, device queries) happens here
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def _loss_outputs_equal(b, x, y):
    V = b.vocab
    for key in x:
        if key == "dlogits":
            assert _same(x[key][:, :V], y[key][:, :V]), key
        else:
            assert _same(x[key], y[key]), key


@pytest.mark.parametrize("case_id", [0, 1])
def test_loss_step_in_a_graph(case_id):
    lengths = None if case_id == 0 else [40, 64, 17, 90, 33, 8, 51, 70]
    b = synthetic.make_batch(case_id, "cuda", lengths=lengths)
    rl = capi.handle_for_batch(b)
    out = capi.alloc_outputs(b)
    g = _capture(lambda: capi.run_batch(rl, b, out))
    for t in out.values():
        t.fill_(7)
    g.replay()
    torch.cuda.synchronize()
    eager = capi.alloc_outputs(b)
    capi.run_batch(rl, b, eager)
    torch.cuda.synchronize()
    _loss_outputs_equal(b, out, eager)
    assert rl.device_status() == 0
    # the graph reads the inputs' current contents
    b.logits.mul_(0.5)
    b.rewards_or_adv.copy_(b.rewards_or_adv.flip(0))
    g.replay()
    capi.run_batch(rl, b, eager)
    torch.cuda.synchronize()
    _loss_outputs_equal(b, out, eager)


def test_gae_in_a_graph():
    gb = synthetic.make_gae_batch("cuda", rollouts=4, segments=2, length=20000)
    T = int(gb.rewards.shape[0])
    ws = capi.gae_workspace(T, gb.rewards.device)
    adv = torch.empty(T, dtype=torch.float32, device="cuda")
    ret = torch.empty_like(adv)
    run = lambda a, r: capi.gae(gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.gamma, gb.lam, True,
                                rollout_ids=gb.rollout_ids, returns=r, advantages=a, workspace=ws)
    g = _capture(lambda: run(adv, ret))
    adv.fill_(7)
    ret.fill_(7)
    g.replay()
    e_adv, e_ret = torch.empty_like(adv), torch.empty_like(adv)
    run(e_adv, e_ret)
    torch.cuda.synchronize()
    assert _same(adv, e_adv) and _same(ret, e_ret)
    gb.rewards.mul_(-0.25)
    g.replay()
    run(e_adv, e_ret)
    torch.cuda.synchronize()
    assert _same(adv, e_adv) and _same(ret, e_ret)


@pytest.mark.parametrize("order", ["score", "index"])
def test_topk_in_a_graph(order):
    b = synthetic.make_topk_batch("cuda", rows=40, context=40000, seed=11)
    idx = torch.empty((b.rows, b.k), dtype=torch.int32, device="cuda")
    val = torch.empty((b.rows, b.k), dtype=torch.float32, device="cuda")
    g = _capture(lambda: capi.topk(b.scores, b.k, lengths=b.lengths, order=order, out_idx=idx, out_val=val))
    idx.fill_(7)
    g.replay()
    e_idx, e_val = capi.topk(b.scores, b.k, lengths=b.lengths, order=order)
    torch.cuda.synchronize()
    assert torch.equal(idx, e_idx) and _same(val, e_val)
    b.scores.copy_(b.scores.flip(1))
    g.replay()
    e_idx, e_val = capi.topk(b.scores, b.k, lengths=b.lengths, order=order)
    torch.cuda.synchronize()
    assert torch.equal(idx, e_idx) and _same(val, e_val)
