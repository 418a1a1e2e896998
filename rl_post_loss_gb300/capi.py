"""Thin ctypes binding of ``include/rl_loss.h`` (argument marshalling only).

Every function of the C ABI is exposed under its own name; ``RlLoss`` wraps a
handle and marshals torch tensors (device memory and the current stream come
from PyTorch; every step of the computation runs in the CUDA library). The
binding fails loudly when ``librl_loss.so`` is missing or a call returns an
error: there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librl_loss.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "rl_loss.h")

RL_F32, RL_BF16 = 0, 1
RL_ADV_GROUP_REWARDS, RL_ADV_PER_SEQ, RL_ADV_PER_TOKEN, RL_ADV_TEACHER_LOGP = 0, 1, 2, 3
RL_OBJ_GRPO_ICEPOP, RL_OBJ_DIS = 0, 1
RL_NORM_PER_RESPONSE, RL_NORM_PER_TOKEN = 0, 1
RL_FLAG_POP_IN_BOUNDS, RL_FLAG_CLIP_ACTIVE, RL_FLAG_MASKED, RL_FLAG_BAD_TARGET = 1, 2, 4, 8

STATUS_NAMES = {0: "RL_OK", 1: "RL_ERR_INVALID_ARG", 2: "RL_ERR_SHAPE", 3: "RL_ERR_DTYPE",
                4: "RL_ERR_ALIGNMENT", 5: "RL_ERR_CAPACITY", 6: "RL_ERR_CUDA", 7: "RL_ERR_TARGET_RANGE",
                8: "RL_ERR_NONFINITE", 9: "RL_ERR_EMPTY_SEQ", 10: "RL_ERR_TIMEOUT", 11: "RL_ERR_UNSUPPORTED",
                12: "RL_ERR_SEQLENS", 13: "RL_ERR_DEVICE", 14: "RL_ERR_INTERNAL"}
CODES = {v: k for k, v in STATUS_NAMES.items()}


class RlLossError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")
        self.code = code


class rl_loss_config(ctypes.Structure):
    _fields_ = [("vocab_size", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
                ("eps_low", ctypes.c_float), ("eps_high", ctypes.c_float), ("beta", ctypes.c_float),
                ("adv_eps", ctypes.c_float), ("adv_mode", ctypes.c_int32), ("std_unbiased", ctypes.c_int32),
                ("pop_indicator", ctypes.c_int32), ("logits_dtype", ctypes.c_int32), ("objective", ctypes.c_int32),
                ("loss_norm", ctypes.c_int32), ("dis_stopgrad", ctypes.c_int32)]


class rl_loss_inputs(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_seqs", ctypes.c_int32), ("ld_logits", ctypes.c_int64),
                ("logits", ctypes.c_void_p), ("targets", ctypes.c_void_p), ("logp_old", ctypes.c_void_p),
                ("logp_infer", ctypes.c_void_p), ("mask", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
                ("rewards_or_adv", ctypes.c_void_p)]


class rl_loss_outputs(ctypes.Structure):
    _fields_ = [("loss", ctypes.c_void_p), ("loss_f64", ctypes.c_void_p), ("dlogits", ctypes.c_void_p),
                ("ld_dlogits", ctypes.c_int64), ("logp", ctypes.c_void_p), ("entropy", ctypes.c_void_p),
                ("flags", ctypes.c_void_p), ("seq_adv", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("mean_entropy", ctypes.c_void_p)]


class rl_gae_config(ctypes.Structure):
    _fields_ = [("gamma", ctypes.c_double), ("lambda_", ctypes.c_double), ("skip_observations", ctypes.c_int32),
                ("cross_trajectory", ctypes.c_int32)]


class rl_topk_config(ctypes.Structure):
    _fields_ = [("k", ctypes.c_int32), ("order", ctypes.c_int32)]


RL_TOPK_BY_SCORE, RL_TOPK_BY_POSITION = 0, 1


class rl_loss_profile(ctypes.Structure):
    _fields_ = [("num_kernels", ctypes.c_int32), ("names", (ctypes.c_char * 32) * 12),
                ("launches", ctypes.c_int64 * 12), ("total_ms", ctypes.c_double * 12)]


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built). RL_LOSS_LIB in the
    environment names another build of it, such as the debug build."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("RL_LOSS_LIB") or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing; build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    st = ctypes.c_int
    sig = {
        "rl_loss_create": ([ctypes.POINTER(rl_loss_config), ctypes.POINTER(P)], st),
        "rl_loss_destroy": ([P], st),
        "rl_loss_forward_backward": ([P, ctypes.POINTER(rl_loss_inputs), ctypes.POINTER(rl_loss_outputs), P], st),
        "rl_loss_forward_backward_from_host": ([P, ctypes.POINTER(rl_loss_inputs), ctypes.POINTER(rl_loss_inputs),
                                                ctypes.POINTER(rl_loss_outputs), ctypes.c_int32, P], st),
        "rl_loss_get_device_status": ([P, P, ctypes.POINTER(ctypes.c_uint32)], st),
        "rl_loss_status_string": ([st], ctypes.c_char_p),
        "rl_loss_profile_start": ([P, ctypes.c_int32], st),
        "rl_loss_profile_read": ([P, ctypes.POINTER(rl_loss_profile)], st),
        "rl_loss_launch_count": ([P, ctypes.POINTER(ctypes.c_int64)], st),
        "rl_loss_last_cuda_error": ([P], ctypes.c_char_p),
        "rl_loss_version": ([], ctypes.c_int32),
        "rl_loss_forward_backward_noalloc": ([ctypes.POINTER(rl_loss_config), ctypes.POINTER(rl_loss_inputs),
                                              ctypes.POINTER(rl_loss_outputs), P, P], st),
        "rl_loss_projection_setup": ([P, ctypes.c_int32, ctypes.c_int32], st),
        "rl_gae_advantages": ([ctypes.POINTER(rl_gae_config), ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, P, P, P,
                               ctypes.c_size_t, P, P], st),
        "rl_gae_advantages_withheld": ([ctypes.POINTER(rl_gae_config), ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, P,
                                        P, P, ctypes.c_size_t, P, P, ctypes.c_int32, ctypes.c_double], st),
        "rl_gae_workspace_bytes": ([ctypes.c_int32], ctypes.c_size_t),
        "rl_topk_max_k": ([], ctypes.c_int32),
        "rl_topk": ([ctypes.POINTER(rl_topk_config), ctypes.c_int32, P, ctypes.c_int64, P, P, P, ctypes.c_int64, P, P],
                    st),
        "rl_loss_projection_logits": ([P, P, ctypes.c_int64, P, ctypes.c_int64, ctypes.c_int32, P, ctypes.c_int64,
                                       P], st),
        "rl_loss_fused_projection_forward_backward": ([P, P, ctypes.c_int64, P, ctypes.c_int64,
                                                       ctypes.POINTER(rl_loss_inputs), P, ctypes.c_int64, P,
                                                       ctypes.c_int64, ctypes.POINTER(rl_loss_outputs), P], st),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def header_functions(path: str = HEADER) -> list[str]:
    """Names of every function the C header declares."""
    text = open(path).read()
    return sorted(set(re.findall(r"RL_LOSS_API\s+[\w\s\*]+?\b(rl_(?:loss_|gae_|topk)\w*)\s*\(", text)))


def _check(code: int, what: str):
    if code != 0:
        raise RlLossError(code, what)


# ------------------------------------------------------------------ the C names, one to one

def rl_loss_create(config: rl_loss_config) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(load().rl_loss_create(ctypes.byref(config), ctypes.byref(h)), "rl_loss_create")
    return h


def rl_loss_destroy(handle) -> None:
    _check(load().rl_loss_destroy(handle), "rl_loss_destroy")


def rl_loss_forward_backward(handle, inputs: rl_loss_inputs, outputs: rl_loss_outputs, stream: int) -> int:
    return load().rl_loss_forward_backward(handle, ctypes.byref(inputs), ctypes.byref(outputs),
                                           ctypes.c_void_p(stream))


def rl_loss_forward_backward_from_host(handle, host: rl_loss_inputs, device: rl_loss_inputs,
                                       outputs: rl_loss_outputs, num_chunks: int, stream: int) -> int:
    return load().rl_loss_forward_backward_from_host(handle, ctypes.byref(host), ctypes.byref(device),
                                                     ctypes.byref(outputs), num_chunks, ctypes.c_void_p(stream))


def rl_loss_get_device_status(handle, stream: int) -> int:
    bits = ctypes.c_uint32(0)
    _check(load().rl_loss_get_device_status(handle, ctypes.c_void_p(stream), ctypes.byref(bits)),
           "rl_loss_get_device_status")
    return int(bits.value)


def rl_loss_status_string(code: int) -> str:
    return load().rl_loss_status_string(code).decode()


def rl_loss_profile_start(handle, max_calls: int) -> None:
    _check(load().rl_loss_profile_start(handle, max_calls), "rl_loss_profile_start")


def rl_loss_profile_read(handle) -> dict:
    prof = rl_loss_profile()
    _check(load().rl_loss_profile_read(handle, ctypes.byref(prof)), "rl_loss_profile_read")
    return {prof.names[k].value.decode(): (int(prof.launches[k]), float(prof.total_ms[k]))
            for k in range(prof.num_kernels)}


def rl_loss_launch_count(handle) -> int:
    n = ctypes.c_int64(0)
    _check(load().rl_loss_launch_count(handle, ctypes.byref(n)), "rl_loss_launch_count")
    return int(n.value)


def rl_loss_forward_backward_noalloc(config: rl_loss_config, inputs: rl_loss_inputs, outputs: rl_loss_outputs,
                                     device_status_ptr: int | None, stream: int) -> int:
    """The allocation-free entry point (no handle; static device workspace)."""
    return load().rl_loss_forward_backward_noalloc(ctypes.byref(config), ctypes.byref(inputs),
                                                   ctypes.byref(outputs), ctypes.c_void_p(device_status_ptr),
                                                   ctypes.c_void_p(stream))


def rl_loss_last_cuda_error(handle) -> str:
    return load().rl_loss_last_cuda_error(handle).decode()


def rl_loss_projection_setup(handle, hidden_dim: int, chunk_tokens: int) -> None:
    _check(load().rl_loss_projection_setup(handle, hidden_dim, chunk_tokens), "rl_loss_projection_setup")


def rl_loss_projection_logits(handle, hidden, ld_hidden, w_lm, ld_w, rows, logits, ld_logits, stream) -> int:
    return load().rl_loss_projection_logits(handle, hidden, ld_hidden, w_lm, ld_w, rows, logits, ld_logits,
                                            ctypes.c_void_p(stream))


def rl_loss_fused_projection_forward_backward(handle, hidden, ld_hidden, w_lm, ld_w, inputs, dhidden, ld_dhidden,
                                              dw_lm, ld_dw, outputs, stream) -> int:
    return load().rl_loss_fused_projection_forward_backward(handle, hidden, ld_hidden, w_lm, ld_w,
                                                            ctypes.byref(inputs), dhidden, ld_dhidden, dw_lm, ld_dw,
                                                            ctypes.byref(outputs), ctypes.c_void_p(stream))


def rl_gae_advantages(config: rl_gae_config, num_tokens, num_seqs, rewards, values, mask, cu_seqlens, rollout_ids,
                      advantages, returns, workspace, workspace_bytes, device_status, stream) -> int:
    return load().rl_gae_advantages(ctypes.byref(config), num_tokens, num_seqs, rewards, values, mask, cu_seqlens,
                                    rollout_ids, advantages, returns, workspace, workspace_bytes, device_status,
                                    ctypes.c_void_p(stream))


def rl_gae_advantages_withheld(config: rl_gae_config, num_tokens, num_seqs, rewards, values, mask, cu_seqlens,
                               rollout_ids, advantages, returns, workspace, workspace_bytes, device_status, stream,
                               withhold_chunk, wait_limit_s) -> int:
    return load().rl_gae_advantages_withheld(ctypes.byref(config), num_tokens, num_seqs, rewards, values, mask,
                                             cu_seqlens, rollout_ids, advantages, returns, workspace, workspace_bytes,
                                             device_status, ctypes.c_void_p(stream), withhold_chunk, wait_limit_s)


def rl_gae_workspace_bytes(num_tokens: int) -> int:
    return int(load().rl_gae_workspace_bytes(int(num_tokens)))


_GAE_WORKSPACE: dict = {}


def gae_workspace(num_tokens: int, device):
    """A GAE workspace for this device of at least this size, zero-filled when
    allocated and kept between calls (every completed call clears its counters
    and flags again)."""
    import torch
    dev = torch.device(device)
    if dev.index is None:
        dev = torch.device(dev.type, torch.cuda.current_device())
    need = rl_gae_workspace_bytes(num_tokens)
    ws = _GAE_WORKSPACE.get(dev)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
        _GAE_WORKSPACE[dev] = ws
    return ws


def gae(rewards, values, mask, cu_seqlens, gamma: float, lam: float, skip_observations: bool = True,
        rollout_ids=None, returns=None, advantages=None, device_status=None, stream=None, workspace=None):
    """Advantages (and optionally returns) on the GPU; torch CUDA tensors in and out."""
    import torch
    T, S = int(rewards.shape[0]), int(cu_seqlens.shape[0]) - 1
    if advantages is None:
        advantages = torch.empty(T, dtype=torch.float32, device=rewards.device)
    if workspace is None:
        workspace = gae_workspace(T, rewards.device)
    cfg = rl_gae_config(gamma, lam, int(skip_observations), int(rollout_ids is not None))
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    _check(rl_gae_advantages(cfg, T, S, _ptr(rewards), _ptr(values), _ptr(mask), _ptr(cu_seqlens), _ptr(rollout_ids),
                             _ptr(advantages), _ptr(returns), _ptr(workspace), workspace.numel(),
                             _ptr(device_status), stream), "rl_gae_advantages")
    return advantages


def rl_topk_max_k() -> int:
    return int(load().rl_topk_max_k())


def topk(scores, k: int, lengths=None, order: str = "score", out_idx=None, out_val=None, want_values=True,
         device_status=None, stream=None):
    """Row-wise deterministic top-k on the GPU; torch CUDA tensors in and out. Returns (positions, scores)."""
    import torch
    if order not in ("score", "index"):
        raise ValueError("order is 'score' or 'index'")
    rows, ld = int(scores.shape[0]), int(scores.shape[1])
    if scores.stride(1) != 1:
        raise ValueError("scores rows must be contiguous")
    if out_idx is None:
        out_idx = torch.empty((rows, k), dtype=torch.int32, device=scores.device)
    if out_val is None and want_values:
        out_val = torch.empty((rows, k), dtype=torch.float32, device=scores.device)
    cfg = rl_topk_config(k, RL_TOPK_BY_SCORE if order == "score" else RL_TOPK_BY_POSITION)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    _check(load().rl_topk(ctypes.byref(cfg), rows, _ptr(scores), int(scores.stride(0)), _ptr(lengths), _ptr(out_idx),
                          _ptr(out_val), int(out_idx.stride(0)), _ptr(device_status), ctypes.c_void_p(stream)),
           "rl_topk")
    return out_idx, out_val


def rl_loss_version() -> int:
    return int(load().rl_loss_version())


# ------------------------------------------------------------------ torch-facing wrapper

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class RlLoss:
    """One handle: fixed vocabulary, group size, hyper-parameters and capacity."""

    def __init__(self, vocab_size: int, group_size: int, max_tokens: int, max_seqs: int, logits_dtype: int,
                 eps_low: float = 0.2, eps_high: float = 0.28, beta: float = 2.0, adv_eps: float = 1e-6,
                 adv_mode: int = RL_ADV_GROUP_REWARDS, std_unbiased: bool = False, pop_indicator: bool = False,
                 objective: int = RL_OBJ_GRPO_ICEPOP, loss_norm: int = RL_NORM_PER_RESPONSE, dis_stopgrad: bool = True):
        self.config = rl_loss_config(vocab_size, group_size, max_tokens, max_seqs, eps_low, eps_high, beta,
                                     adv_eps, adv_mode, int(std_unbiased), int(pop_indicator), logits_dtype,
                                     objective, loss_norm, int(dis_stopgrad))
        self.handle = rl_loss_create(self.config)

    def close(self):
        if self.handle:
            rl_loss_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward_backward(self, logits, targets, logp_old, logp_infer, mask, cu_seqlens, rewards_or_adv, *,
                         loss, dlogits, loss_f64=None, logp=None, entropy=None, flags=None, seq_adv=None,
                         counts=None, mean_entropy=None, stream=None) -> None:
        """Enqueue one forward+backward on ``stream`` (default: torch's current
        stream). All tensors are caller-owned CUDA tensors."""
        import torch
        T = int(targets.shape[0])
        S = int(cu_seqlens.shape[0]) - 1
        inp = rl_loss_inputs(T, S, int(logits.stride(0)) if logits.dim() == 2 else 0, _ptr(logits), _ptr(targets),
                             _ptr(logp_old), _ptr(logp_infer), _ptr(mask), _ptr(cu_seqlens), _ptr(rewards_or_adv))
        out = rl_loss_outputs(_ptr(loss), _ptr(loss_f64), _ptr(dlogits),
                              int(dlogits.stride(0)) if dlogits.dim() == 2 else 0, _ptr(logp), _ptr(entropy),
                              _ptr(flags), _ptr(seq_adv), _ptr(counts), _ptr(mean_entropy))
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        code = rl_loss_forward_backward(self.handle, inp, out, stream)
        if code == CODES["RL_ERR_CUDA"]:
            raise RlLossError(code, "rl_loss_forward_backward (%s)" % rl_loss_last_cuda_error(self.handle))
        _check(code, "rl_loss_forward_backward")

    def forward_backward_from_host(self, host: dict, device: dict, *, loss, dlogits, num_chunks: int = 8,
                                   loss_f64=None, logp=None, entropy=None, flags=None, seq_adv=None, counts=None,
                                   mean_entropy=None, stream=None) -> None:
        """Enqueue one forward+backward whose inputs start in host memory: ``host`` and ``device``
        map the input names (logits, targets, logp_old, logp_infer, mask, cu_seqlens,
        rewards_or_adv) to pinned CPU tensors and to CUDA tensors of the same shapes that receive
        them. The logits go over in ``num_chunks`` row blocks, each computed as soon as it lands."""
        import torch

        def inputs(d):
            lg = d["logits"]
            return rl_loss_inputs(int(d["targets"].shape[0]), int(d["cu_seqlens"].shape[0]) - 1,
                                  int(lg.stride(0)) if lg.dim() == 2 else 0, _ptr(lg), _ptr(d["targets"]),
                                  _ptr(d["logp_old"]), _ptr(d["logp_infer"]), _ptr(d["mask"]), _ptr(d["cu_seqlens"]),
                                  _ptr(d["rewards_or_adv"]))
        out = rl_loss_outputs(_ptr(loss), _ptr(loss_f64), _ptr(dlogits),
                              int(dlogits.stride(0)) if dlogits.dim() == 2 else 0, _ptr(logp), _ptr(entropy),
                              _ptr(flags), _ptr(seq_adv), _ptr(counts), _ptr(mean_entropy))
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        self._raise(rl_loss_forward_backward_from_host(self.handle, inputs(host), inputs(device), out, num_chunks,
                                                       stream), "rl_loss_forward_backward_from_host")

    def _raise(self, code: int, what: str):
        if code == CODES["RL_ERR_CUDA"]:
            raise RlLossError(code, "%s (%s)" % (what, rl_loss_last_cuda_error(self.handle)))
        _check(code, what)

    def projection_setup(self, hidden_dim: int, chunk_tokens: int) -> None:
        rl_loss_projection_setup(self.handle, hidden_dim, chunk_tokens)

    def projection_logits(self, hidden, w_lm, rows: int, logits, stream=None) -> None:
        """logits[:rows] (fp32) = hidden[:rows] @ w_lm^T on the tensor cores."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        self._raise(rl_loss_projection_logits(self.handle, _ptr(hidden), hidden.stride(0), _ptr(w_lm), w_lm.stride(0),
                                              rows, _ptr(logits), logits.stride(0), stream),
                    "rl_loss_projection_logits")

    def fused_projection_forward_backward(self, hidden, w_lm, targets, logp_old, logp_infer, mask, cu_seqlens,
                                          rewards_or_adv, *, loss, dhidden, dw_lm, loss_f64=None, logp=None,
                                          entropy=None, flags=None, seq_adv=None, counts=None, mean_entropy=None,
                                          stream=None) -> None:
        import torch
        T = int(targets.shape[0])
        S = int(cu_seqlens.shape[0]) - 1
        inp = rl_loss_inputs(T, S, 0, None, _ptr(targets), _ptr(logp_old), _ptr(logp_infer), _ptr(mask),
                             _ptr(cu_seqlens), _ptr(rewards_or_adv))
        out = rl_loss_outputs(_ptr(loss), _ptr(loss_f64), None, 0, _ptr(logp), _ptr(entropy), _ptr(flags),
                              _ptr(seq_adv), _ptr(counts), _ptr(mean_entropy))
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        self._raise(rl_loss_fused_projection_forward_backward(
            self.handle, _ptr(hidden), hidden.stride(0), _ptr(w_lm), w_lm.stride(0), inp, _ptr(dhidden),
            dhidden.stride(0), _ptr(dw_lm), dw_lm.stride(0), out, stream), "rl_loss_fused_projection_forward_backward")

    def device_status(self, stream=None) -> int:
        import torch
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        return rl_loss_get_device_status(self.handle, stream)

    def profile_start(self, max_calls: int):
        rl_loss_profile_start(self.handle, max_calls)

    def profile_read(self) -> dict:
        return rl_loss_profile_read(self.handle)

    def launch_count(self) -> int:
        return rl_loss_launch_count(self.handle)


def status_bits_to_names(bits: int) -> list[str]:
    return [STATUS_NAMES[c] for c in sorted(STATUS_NAMES) if c and bits & (1 << c)]


# ------------------------------------------------------------------ batch helpers

def handle_for_batch(batch, max_tokens: int | None = None, max_seqs: int | None = None, **overrides) -> RlLoss:
    """A handle configured for a ``synthetic.Batch`` (capacity = the batch's size)."""
    kw = dict(eps_low=batch.eps_low, eps_high=batch.eps_high, beta=batch.beta, adv_eps=batch.adv_eps,
              adv_mode=batch.adv_mode, objective=batch.objective, loss_norm=batch.loss_norm)
    kw.update(overrides)
    return RlLoss(batch.vocab, batch.group, max(1, max_tokens or batch.num_tokens), max_seqs or batch.num_seqs,
                  RL_BF16 if batch.dtype == "bf16" else RL_F32, **kw)


def alloc_outputs(batch, in_place: bool = False, ld: int | None = None) -> dict:
    """Caller-owned output tensors for one call on ``batch`` (on its device)."""
    import torch
    dev = batch.logits.device
    T, S = batch.num_tokens, batch.num_seqs
    if in_place:
        dlogits = batch.logits
    else:
        ld = ld or batch.logits.stride(0)
        dlogits = torch.empty((T, ld), dtype=batch.logits.dtype, device=dev)
    return dict(loss=torch.empty(1, dtype=torch.float32, device=dev),
                loss_f64=torch.empty(1, dtype=torch.float64, device=dev), dlogits=dlogits,
                logp=torch.empty(T, dtype=torch.float32, device=dev),
                entropy=torch.empty(T, dtype=torch.float32, device=dev),
                flags=torch.empty(T, dtype=torch.uint8, device=dev),
                seq_adv=torch.empty(S, dtype=torch.float32, device=dev),
                counts=torch.empty(4, dtype=torch.int32, device=dev),
                mean_entropy=torch.empty(1, dtype=torch.float32, device=dev))


def run_batch(rl: RlLoss, batch, outputs: dict, stream=None) -> dict:
    """One forward+backward of ``batch`` into ``outputs`` (asynchronous)."""
    adv = batch.token_adv if (batch.adv_mode >= RL_ADV_PER_TOKEN) else batch.rewards_or_adv
    rl.forward_backward(batch.logits, batch.targets, batch.logp_old, batch.logp_infer, batch.mask,
                        batch.cu_seqlens, adv, stream=stream, **outputs)
    return outputs


INPUT_NAMES = ("logits", "targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv")


def batch_inputs(batch) -> dict:
    """The input tensors of ``batch`` by name (the advantage array the batch's mode reads)."""
    adv = batch.token_adv if (batch.adv_mode >= RL_ADV_PER_TOKEN) else batch.rewards_or_adv
    return {n: (adv if n == "rewards_or_adv" else getattr(batch, n)) for n in INPUT_NAMES}


def run_batch_from_host(rl: RlLoss, host: dict, device: dict, outputs: dict, num_chunks: int = 8,
                        stream=None) -> dict:
    """One forward+backward from pinned host inputs ``host`` into the device buffers ``device``."""
    rl.forward_backward_from_host(host, device, num_chunks=num_chunks, stream=stream, **outputs)
    return outputs


def projection_handle(pb, max_tokens: int | None = None, **overrides) -> RlLoss:
    """A bf16 handle with the fused projection path set up for a ``synthetic.ProjBatch``."""
    rl = handle_for_batch(pb.batch, max_tokens=max_tokens, **overrides)
    rl.projection_setup(pb.hidden_dim, pb.chunk)
    return rl


def alloc_projection_outputs(pb) -> dict:
    import torch
    b = pb.batch
    out = alloc_outputs(b, ld=8)
    del out["dlogits"]
    dev = pb.hidden.device
    out["dhidden"] = torch.empty_like(pb.hidden)
    out["dw_lm"] = torch.empty((pb.w.shape[0], pb.w.shape[1]), dtype=torch.float32, device=dev)
    return out


def run_projection(rl: RlLoss, pb, outputs: dict, stream=None) -> dict:
    b = pb.batch
    adv = b.token_adv if (b.adv_mode >= RL_ADV_PER_TOKEN) else b.rewards_or_adv
    rl.fused_projection_forward_backward(pb.hidden, pb.w, b.targets, b.logp_old, b.logp_infer, b.mask, b.cu_seqlens,
                                         adv, stream=stream, **outputs)
    return outputs
