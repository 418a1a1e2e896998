"""Canary guard regions around every output buffer.

Each output of a call is carved out of a larger device buffer whose bytes
before and after it hold a fixed canary pattern; after the call (and a
synchronize) every canary byte must be unchanged, and every input must be
bit-identical to what it was. This catches writes past the end of an output
(or before its start) that parity checks on the outputs themselves would miss:
the loss path on fp32 and bf16 logits with a ragged vocabulary, the fused
projection, GAE and top-k.
"""
import numpy as np
import pytest
import torch

from parity_helpers import check_all
from rl_post_loss_gb300 import build as nvbuild
from rl_post_loss_gb300 import capi, synthetic

pytestmark = pytest.mark.gpu

GUARD = 4096  # canary bytes on each side
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nvbuild.build()
    capi.load()


class Guarded:
    """Device tensors of the given shapes carved out of canary-filled buffers."""

    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        view = buf[GUARD:GUARD + n].view(dtype).view(*shape)
        if fill is not None:
            view.fill_(fill)
        self.bufs.append(buf)
        return view

    def check(self):
        torch.cuda.synchronize()
        for buf in self.bufs:
            assert bool((buf[:GUARD] == CANARY).all()), "canary before an output overwritten"
            assert bool((buf[-GUARD:] == CANARY).all()), "canary after an output overwritten"


def _snap(tensors):
    return [t.clone() for t in tensors]


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("case_id,vocab", [(0, 4097), (1, 1001), (2, 200003)])
def test_loss_outputs_keep_their_canaries(case_id, vocab):
    b = synthetic.make_batch(case_id, "cuda", lengths=[37, 5, 120, 64] * synthetic.CASES[case_id]["group"],
                             vocab=vocab)
    T, S = b.num_tokens, b.num_seqs
    g = Guarded()
    out = dict(loss=g.empty((1,), torch.float32), loss_f64=g.empty((1,), torch.float64),
               dlogits=g.empty((T, b.logits.stride(0)), b.logits.dtype, fill=7.0),
               logp=g.empty((T,), torch.float32), entropy=g.empty((T,), torch.float32),
               flags=g.empty((T,), torch.uint8), seq_adv=g.empty((S,), torch.float32),
               counts=g.empty((4,), torch.int32), mean_entropy=g.empty((1,), torch.float32))
    ins = capi.batch_inputs(b)
    before = _snap(ins.values())
    rl = capi.handle_for_batch(b)
    capi.run_batch(rl, b, out)
    g.check()
    assert rl.device_status() == 0
    for t0, t1 in zip(before, ins.values()):
        assert _same(t0, t1), "an input changed"
    assert bool((out["dlogits"][:, vocab:] == 7.0).all())  # padding columns are not written
    check_all(b, out, dz_rows=16)


def test_projection_outputs_keep_their_canaries():
    pb = synthetic.make_projection_batch("cuda", prompts=1, group=4, length=70, hidden=256, vocab=3001, chunk=96)
    b = pb.batch
    T, S = b.num_tokens, b.num_seqs
    g = Guarded()
    out = dict(loss=g.empty((1,), torch.float32), loss_f64=g.empty((1,), torch.float64), dlogits=None,
               logp=g.empty((T,), torch.float32), entropy=g.empty((T,), torch.float32),
               flags=g.empty((T,), torch.uint8), seq_adv=g.empty((S,), torch.float32),
               counts=g.empty((4,), torch.int32), mean_entropy=g.empty((1,), torch.float32),
               dhidden=g.empty(tuple(pb.hidden.shape), torch.bfloat16),
               dw_lm=g.empty((pb.w.shape[0], pb.w.shape[1]), torch.float32))
    del out["dlogits"]
    before = _snap([pb.hidden, pb.w, b.targets, b.logp_old, b.logp_infer, b.mask, b.cu_seqlens, b.rewards_or_adv])
    rl = capi.projection_handle(pb)
    capi.run_projection(rl, pb, out)
    g.check()
    assert rl.device_status() & ~(1 << capi.CODES["RL_ERR_EMPTY_SEQ"]) == 0
    for t0, t1 in zip(before, [pb.hidden, pb.w, b.targets, b.logp_old, b.logp_infer, b.mask, b.cu_seqlens,
                               b.rewards_or_adv]):
        assert _same(t0, t1), "an input changed"
    assert bool(torch.isfinite(out["dw_lm"]).all()) and bool(torch.isfinite(out["dhidden"].float()).all())


def test_gae_and_topk_outputs_keep_their_canaries():
    gb = synthetic.make_gae_batch("cuda", lengths=[3000, 0, 9001, 41, 20000], segments=2)
    T = gb.num_tokens
    g = Guarded()
    adv = g.empty((T,), torch.float32)
    ret = g.empty((T,), torch.float32)
    st = g.empty((1,), torch.int32, fill=0)
    before = _snap([gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.rollout_ids])
    capi.gae(gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.gamma, gb.lam, True, rollout_ids=gb.rollout_ids,
             returns=ret, advantages=adv, device_status=st)
    g.check()
    assert st.item() == 0
    for t0, t1 in zip(before, [gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.rollout_ids]):
        assert _same(t0, t1), "an input changed"

    tb = synthetic.make_topk_batch("cuda", rows=5, context=20000, k=2048)
    g = Guarded()
    rows, k = tb.rows, tb.k
    idx = g.empty((rows, k), torch.int32)
    val = g.empty((rows, k), torch.float32)
    st = g.empty((1,), torch.int32, fill=0)
    before = _snap([tb.scores, tb.lengths])
    cfg = capi.rl_topk_config(k, capi.RL_TOPK_BY_SCORE)
    p = capi._ptr
    rc = capi.load().rl_topk(cfg, rows, p(tb.scores), tb.scores.stride(0), p(tb.lengths), p(idx), p(val), k, p(st),
                             torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    g.check()
    assert st.item() == 0
    for t0, t1 in zip(before, [tb.scores, tb.lengths]):
        assert _same(t0, t1), "an input changed"
