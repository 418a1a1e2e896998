"""rl_loss_forward_backward_from_host: inputs in pinned host memory, copied in
row blocks on the handle's copy stream with each block computed as soon as it
lands. Every output must be bit-identical to rl_loss_forward_backward on the
same inputs already on the device (same per-row arithmetic, reductions once
over all rows); the oracle parity of that path is covered elsewhere, and one
case here is also checked against the oracle directly."""
import numpy as np
import pytest
import torch

from parity_helpers import check_all, params_for
from rl_post_loss_gb300 import build as nvbuild
from rl_post_loss_gb300 import capi, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nvbuild.build()
    capi.load()


def _lengths(n, lo, hi, seed):
    g = np.random.default_rng(seed)
    return [int(x) for x in g.integers(lo, hi + 1, size=n)]


def _host_copy(d: dict) -> dict:
    return {k: v.cpu().pin_memory() for k, v in d.items()}


def _device_like(d: dict, ld: int | None = None) -> dict:
    out = {}
    for k, v in d.items():
        if k == "logits" and ld is not None:
            t = torch.full((v.shape[0], ld), 7.0, dtype=v.dtype, device="cuda")
            out[k] = t
        else:
            out[k] = torch.full_like(v, 3, device="cuda")
    return out


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def _equal_outputs(b, x, y):
    V = b.vocab
    for key in x:
        if key == "dlogits":
            assert _same(x[key][:, :V], y[key][:, :V]), key
        else:
            assert _same(x[key], y[key]), key


def _both(b, num_chunks, ld_dev=None, **over):
    rl = capi.handle_for_batch(b, **over)
    ref = capi.alloc_outputs(b)
    capi.run_batch(rl, b, ref)
    torch.cuda.synchronize()
    ref_bits = rl.device_status()
    src = capi.batch_inputs(b)
    host = _host_copy(src)
    dev = _device_like(src, ld_dev)
    out = capi.alloc_outputs(b)
    for t in out.values():
        t.fill_(5)
    capi.run_batch_from_host(rl, host, dev, out, num_chunks=num_chunks)
    torch.cuda.synchronize()
    bits = rl.device_status()
    return rl, ref, ref_bits, out, bits, host, dev


@pytest.mark.parametrize("num_chunks", [1, 3, 8, 64])
def test_bit_identical_to_the_device_call(num_chunks):
    b = synthetic.make_batch(1, "cuda", lengths=_lengths(16, 20, 300, 5))
    _, ref, ref_bits, out, bits, host, dev = _both(b, num_chunks)
    assert bits == ref_bits
    _equal_outputs(b, out, ref)
    # the device buffers received the inputs
    for k in ("targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv"):
        assert _same(dev[k], host[k].cuda()), k
    assert _same(dev["logits"], host["logits"].cuda())


def test_long_rows_fp32_and_more_blocks_than_rows():
    b = synthetic.make_batch(2, "cuda", lengths=_lengths(8, 2, 6, 6))  # 151552-wide bf16 rows, T < 64
    assert b.num_tokens < 64
    _, ref, ref_bits, out, bits, _, _ = _both(b, 64)
    assert bits == ref_bits
    _equal_outputs(b, out, ref)
    b0 = synthetic.make_batch(0, "cuda")  # fp32 logits
    _, ref, ref_bits, out, bits, _, _ = _both(b0, 5)
    assert bits == ref_bits
    _equal_outputs(b0, out, ref)
    check_all(b0, out, dz_rows="all")


def test_device_row_stride_differs_from_the_host_one():
    b = synthetic.make_batch(1, "cuda", lengths=_lengths(8, 10, 80, 7), vocab=1001)
    ld = 1024 + 8
    _, ref, ref_bits, out, bits, host, dev = _both(b, 6, ld_dev=ld)
    assert bits == ref_bits
    _equal_outputs(b, out, ref)
    assert dev["logits"].stride(0) == ld
    assert _same(dev["logits"][:, :b.vocab], host["logits"][:, :b.vocab].cuda())
    assert bool((dev["logits"][:, b.vocab:] == 7.0).all())  # columns past V are not written


def test_equal_padded_strides_touch_neither_padding_nor_past_the_last_row():
    """Host and device rows both padded (ld > V, same stride): the padding
    columns of the device buffer keep their sentinels, and a host buffer that
    ends right after the last row's V-th element is enough."""
    b = synthetic.make_batch(1, "cuda", lengths=_lengths(8, 10, 80, 8), vocab=1001)
    T, V, ld = b.num_tokens, b.vocab, 1024 + 8
    rl = capi.handle_for_batch(b)
    ref = capi.alloc_outputs(b)
    capi.run_batch(rl, b, ref)
    torch.cuda.synchronize()
    ref_bits = rl.device_status()
    src = capi.batch_inputs(b)
    host = _host_copy(src)
    flat = torch.empty((T - 1) * ld + V, dtype=src["logits"].dtype).pin_memory()
    hl = flat.as_strided((T, V), (ld, 1))
    hl.copy_(src["logits"][:, :V].cpu())
    host["logits"] = hl
    dev = _device_like(src, ld)
    out = capi.alloc_outputs(b)
    capi.run_batch_from_host(rl, host, dev, out, num_chunks=4)
    torch.cuda.synchronize()
    assert rl.device_status() == ref_bits
    _equal_outputs(b, out, ref)
    assert dev["logits"].stride(0) == ld
    assert _same(dev["logits"][:, :V], src["logits"][:, :V])
    assert bool((dev["logits"][:, V:] == 7.0).all())  # padding columns are not written


@pytest.mark.parametrize("over", [
    dict(token_adv="normal"),
    dict(token_adv="teacher", group=1, prompts=16),
    dict(objective=1, token_adv="normal", loss_norm=1),
])
def test_advantage_modes(over):
    G = over.get("group", 8)
    n = over.get("prompts", 2) * G
    b = synthetic.make_batch(1, "cuda", lengths=_lengths(n, 8, 60, 11), case_overrides=over)
    _, ref, ref_bits, out, bits, _, _ = _both(b, 4)
    assert bits == ref_bits
    _equal_outputs(b, out, ref)
    check_all(b, out, p=params_for(b, dis_stopgrad=1), dz_rows=32)


def test_back_to_back_calls_follow_the_host_buffers():
    b = synthetic.make_batch(1, "cuda", lengths=_lengths(16, 40, 200, 12))
    rl = capi.handle_for_batch(b)
    src = capi.batch_inputs(b)
    host = _host_copy(src)
    dev = _device_like(src)
    outs = []
    stream = torch.cuda.current_stream()
    for step in range(3):
        out = capi.alloc_outputs(b)
        capi.run_batch_from_host(rl, host, dev, out, num_chunks=8)
        outs.append(out)
        # the next step's inputs are written only once this step has consumed them
        stream.synchronize()
        host["logits"].mul_(0.5)
        host["rewards_or_adv"].copy_(host["rewards_or_adv"].flip(0))
    torch.cuda.synchronize()
    assert rl.device_status() == 0
    for step in range(3):
        ref_in = {k: v.clone() for k, v in host.items()}
        for _ in range(3 - step):  # undo the later changes
            ref_in["logits"].mul_(2.0)
            ref_in["rewards_or_adv"].copy_(ref_in["rewards_or_adv"].flip(0))
        bb = synthetic.Batch(**{**b.__dict__, "logits": ref_in["logits"].cuda(),
                                "rewards_or_adv": ref_in["rewards_or_adv"].cuda()})
        ref = capi.alloc_outputs(bb)
        capi.run_batch(rl, bb, ref)
        torch.cuda.synchronize()
        _equal_outputs(bb, outs[step], ref)


def test_argument_errors_leave_nothing_enqueued():
    b = synthetic.make_batch(1, "cuda", lengths=_lengths(8, 10, 40, 13))
    rl = capi.handle_for_batch(b)
    src = capi.batch_inputs(b)
    host = _host_copy(src)
    dev = _device_like(src)
    out = capi.alloc_outputs(b)
    for bad in (0, 65):
        with pytest.raises(capi.RlLossError) as e:
            capi.run_batch_from_host(rl, host, dev, out, num_chunks=bad)
        assert e.value.code == capi.CODES["RL_ERR_INVALID_ARG"]
    misaligned = dict(dev, logits=torch.empty(dev["logits"].numel() + 8, dtype=dev["logits"].dtype,
                                              device="cuda")[1:1 + dev["logits"].numel()].view(dev["logits"].shape))
    with pytest.raises(capi.RlLossError) as e:
        capi.run_batch_from_host(rl, host, misaligned, out, num_chunks=4)
    assert e.value.code == capi.CODES["RL_ERR_ALIGNMENT"]
    torch.cuda.synchronize()
    assert rl.launch_count() == 0
