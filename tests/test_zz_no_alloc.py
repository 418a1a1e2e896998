"""The allocation-free entry point ``rl_loss_forward_backward_noalloc``.

Callers that cannot allocate device memory when they need the loss (code
inside a framework whose caching allocator owns the device memory, or a
process with a fixed memory budget, where an allocation could fail or
synchronise the device) use this entry point: it takes no handle and keeps its workspace in a static device
array of the library. These tests call it through the C ABI and check that two
calls in a row give the same results as the handle-based entry point, within
the parity tolerances used everywhere else, and that the static workspace does
not carry state from one call into the next. The file is named to be collected
last, so that a run stopping at its first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from rl_post_loss_gb300 import build as nvbuild
from rl_post_loss_gb300 import capi, synthetic

pytestmark = pytest.mark.gpu

TOL_LOGP = {"f32": 1e-4, "bf16": 2e-3}


def _structs(batch, out):
    T, S = batch.num_tokens, batch.num_seqs
    p = capi._ptr
    inp = capi.rl_loss_inputs(T, S, batch.logits.stride(0), p(batch.logits), p(batch.targets), p(batch.logp_old),
                              p(batch.logp_infer), p(batch.mask), p(batch.cu_seqlens), p(batch.rewards_or_adv))
    o = capi.rl_loss_outputs(p(out["loss"]), p(out["loss_f64"]), p(out["dlogits"]), out["dlogits"].stride(0),
                             p(out["logp"]), p(out["entropy"]), p(out["flags"]), p(out["seq_adv"]),
                             p(out["counts"]), p(out["mean_entropy"]))
    return inp, o


def _noalloc(batch, config, out, status):
    inp, o = _structs(batch, out)
    stream = torch.cuda.current_stream().cuda_stream
    return capi.rl_loss_forward_backward_noalloc(config, inp, o, status.data_ptr(), stream)


def _close(batch, ref, got):
    V = batch.vocab
    a = ref["loss_f64"].item()
    assert abs(got["loss_f64"].item() - a) <= 1e-4 * abs(a) + 1e-12
    tol = TOL_LOGP[batch.dtype]
    assert (got["logp"] - ref["logp"]).abs().max().item() <= tol
    assert (got["entropy"] - ref["entropy"]).abs().max().item() <= tol
    assert torch.equal(got["flags"], ref["flags"])
    assert torch.equal(got["counts"], ref["counts"])
    r = ref["dlogits"][:, :V].double()
    g = got["dlogits"][:, :V].double()
    assert bool(((g - r).abs() <= 1e-6 + 8e-3 * r.abs()).all())


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return capi.load()


@pytest.mark.parametrize("case_id,n_prompts,lo,hi", [(0, 2, 16, 128), (1, 1, 32, 200), (2, 1, 16, 64)])
def test_noalloc_matches_handle_path_on_two_calls(lib, case_id, n_prompts, lo, hi):
    rng = np.random.default_rng(77 + case_id)
    G = synthetic.CASES[case_id]["group"]
    lengths = [int(x) for x in rng.integers(lo, hi + 1, size=n_prompts * G)]
    batch = synthetic.make_batch(case_id, "cuda", lengths=lengths)
    rl = capi.handle_for_batch(batch)
    ref = capi.alloc_outputs(batch)
    capi.run_batch(rl, batch, ref)
    torch.cuda.synchronize()
    assert rl.device_status() == 0
    status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    for _ in range(2):
        got = capi.alloc_outputs(batch)
        assert _noalloc(batch, rl.config, got, status) == 0
        torch.cuda.synchronize()
        assert status.item() == 0
        _close(batch, ref, got)


def test_noalloc_static_workspace_carries_no_state(lib):
    batch = synthetic.make_batch(0, "cuda")
    rl = capi.handle_for_batch(batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = synthetic.make_batch(0, "cuda")
    bad.targets[0] = bad.vocab  # raises RL_ERR_TARGET_RANGE on the device
    out = capi.alloc_outputs(bad)
    assert _noalloc(bad, rl.config, out, status) == 0
    torch.cuda.synchronize()
    assert status.item() == 1 << capi.CODES["RL_ERR_TARGET_RANGE"]
    ref = capi.alloc_outputs(batch)
    capi.run_batch(rl, batch, ref)
    got = capi.alloc_outputs(batch)
    assert _noalloc(batch, rl.config, got, status) == 0
    torch.cuda.synchronize()
    assert status.item() == 0  # the previous call's bits were cleared
    _close(batch, ref, got)


def test_noalloc_rejects_sizes_beyond_its_maximum(lib):
    batch = synthetic.make_batch(0, "cuda", lengths=[4, 4, 4, 4])
    cfg = capi.handle_for_batch(batch).config
    out = capi.alloc_outputs(batch)
    inp, o = _structs(batch, out)
    inp.num_tokens = 262145
    rc = lib.rl_loss_forward_backward_noalloc(ctypes.byref(cfg), ctypes.byref(inp), ctypes.byref(o), None,
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == capi.CODES["RL_ERR_CAPACITY"]
    inp.num_tokens = batch.num_tokens
    inp.num_seqs = 8196
    rc = lib.rl_loss_forward_backward_noalloc(ctypes.byref(cfg), ctypes.byref(inp), ctypes.byref(o), None,
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == capi.CODES["RL_ERR_CAPACITY"]
