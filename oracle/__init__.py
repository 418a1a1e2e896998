"""fp64 CPU oracle for the GRPO + IcePop token-level policy loss.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module. It
shares no code with the CUDA library and never imports it. The arithmetic lives
in ``rl_loss_oracle.c`` (plain double-precision C, OpenMP over rows); this file
compiles it, loads it with ctypes and composes its three steps:

1. ``seq_prep``: |y_i|, the advantage A_i and the weight w_i = 1/(S |y_i|)
   ("GLM-5: from Vibe Coding to Agentic Engineering", section 3.2, the
   definitions under Eq. (1)).
2. ``rows``: per-token log-prob, entropy, flags, objective term, dL/dlogp and
   optionally the full dL/dlogits row, for any list of rows.
3. ``loss``: L = -sum_i w_i sum_t tok_obj_t (Eq. (1)).

Every function in the C file is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rl_loss_oracle.c")
_LIB_PATH = os.path.join(_HERE, "librl_loss_oracle.so")

F32, BF16, F64 = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
             "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double
    lib.oracle_seq_prep.argtypes = [i64, i64, P, P, P, i32, f32, i32, i32, P, P, P]
    lib.oracle_seq_prep.restype = i32
    lib.oracle_rows.argtypes = [i64, P, i64, i64, i32, P, P, P, P, P, i64, P, P, P, f32, f32, f32, i32,
                                i32, i32, P, P, P, P, P, P, P, P]
    lib.oracle_rows.restype = i32
    lib.oracle_loss.argtypes = [i64, P, P, P]
    lib.oracle_loss.restype = f64
    lib.oracle_pop_in_bounds.argtypes = [f32, f32, f32]
    lib.oracle_pop_in_bounds.restype = i32
    lib.oracle_clip_active.argtypes = [f32, f32, f64, f32, f32]
    lib.oracle_clip_active.restype = i32
    lib.oracle_clip_active_vec.argtypes = [i64, P, P, P, f32, f32, P]
    lib.oracle_clip_active_vec.restype = None
    for name in ("oracle_ln_beta_f32", "oracle_clip_hi_f32", "oracle_clip_lo_f32"):
        getattr(lib, name).argtypes = [f32]
        getattr(lib, name).restype = f32
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class LossParams:
    """Loss hyper-parameters (section 3.2 of the GLM-5 report page: beta = 2,
    eps_low = 0.2, eps_high = 0.28)."""
    group_size: int
    eps_low: float = 0.2
    eps_high: float = 0.28
    beta: float = 2.0
    adv_eps: float = 1e-6
    adv_mode: int = 0          # 0: group-normalised rewards, 1: given per-sequence advantage,
                               # 2: given per-token advantage, 3: teacher log-probs (on-policy distillation)
    std_unbiased: int = 0
    pop_indicator: int = 0     # 0: pop returns rho (printed operator), 1: returns 1
    objective: int = 0         # 0: GRPO + IcePop (Eq. 1), 1: direct double-sided importance sampling
    loss_norm: int = 0         # 0: 1/(S |y_i|) per response (Eq. 1), 1: mean over all generated tokens
    dis_stopgrad: int = 1      # DIS only: 1 = f(r) treated as a constant


def seq_prep(cu_seqlens, mask, rewards_or_adv, p: LossParams):
    """Returns (n_tokens int64 [S], adv f64 [S], w f64 [S])."""
    lib = _load()
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    r = np.ascontiguousarray(rewards_or_adv, dtype=np.float32)
    S = cu.shape[0] - 1
    n = np.zeros(S, np.int64)
    adv = np.zeros(S, np.float64)
    w = np.zeros(S, np.float64)
    if p.adv_mode >= 2:
        r = np.zeros(S, np.float32)  # per-token modes: the [T] array is used by rows()
    rc = lib.oracle_seq_prep(S, p.group_size, _ptr(cu), _ptr(m), _ptr(r), p.adv_mode, p.adv_eps,
                             p.std_unbiased, p.loss_norm, _ptr(n), _ptr(adv), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_seq_prep rejected its arguments")
    return n, adv, w


def rows(row_ids, logits_rows, dtype: int, V: int, targets, logp_old, logp_infer, mask, cu_seqlens, adv, w,
         p: LossParams, want_dz: bool = False, token_adv=None):
    """Per-token results for ``row_ids``; ``logits_rows`` is [len(row_ids), ld]
    (float32, float64, or uint16 holding bf16 bits). ``token_adv`` is the [T]
    array of adv_mode 2 (advantages) or 3 (teacher log-probs). Returns a dict."""
    lib = _load()
    ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    z = np.ascontiguousarray(logits_rows)
    n = ids.shape[0]
    ld = z.shape[1] if z.ndim == 2 else V
    want = {F32: np.float32, BF16: np.uint16, F64: np.float64}[dtype]
    assert z.dtype == want, (z.dtype, want)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    out = {
        "logp": np.zeros(n, np.float64),
        "entropy": np.zeros(n, np.float64),
        "flags": np.zeros(n, np.uint8),
        "tok_obj": np.zeros(n, np.float64),
        "g": np.zeros(n, np.float64),
    }
    dz = np.zeros((n, V), np.float64) if want_dz else None
    tg = np.ascontiguousarray(targets, dtype=np.int32)
    lo = np.ascontiguousarray(logp_old, dtype=np.float32)
    li = np.ascontiguousarray(logp_infer, dtype=np.float32)
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    a = np.ascontiguousarray(adv, dtype=np.float64)
    ww = np.ascontiguousarray(w, dtype=np.float64)
    ta = None if p.adv_mode < 2 else np.ascontiguousarray(token_adv, dtype=np.float32)
    rc = lib.oracle_rows(n, _ptr(ids), V, ld, dtype, _ptr(z), _ptr(tg), _ptr(lo), _ptr(li), _ptr(m),
                         cu.shape[0] - 1, _ptr(cu), _ptr(a), _ptr(ww), p.eps_low, p.eps_high, p.beta,
                         p.pop_indicator, p.objective, p.dis_stopgrad, _ptr(ta if p.adv_mode == 2 else None),
                         _ptr(ta if p.adv_mode == 3 else None), _ptr(out["logp"]), _ptr(out["entropy"]),
                         _ptr(out["flags"]), _ptr(out["tok_obj"]), _ptr(out["g"]), _ptr(dz))
    if rc != 0:
        raise ValueError("oracle_rows rejected its arguments")
    if want_dz:
        out["dz"] = dz
    return out


def loss(cu_seqlens, w, tok_obj) -> float:
    """L = -sum_i w_i sum_{t in i} tok_obj_t, tok_obj indexed by token id."""
    lib = _load()
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    ww = np.ascontiguousarray(w, dtype=np.float64)
    to = np.ascontiguousarray(tok_obj, dtype=np.float64)
    return float(lib.oracle_loss(cu.shape[0] - 1, _ptr(cu), _ptr(ww), _ptr(to)))


def forward_backward(batch: dict, dtype: int, V: int, p: LossParams, want_dz: bool = False,
                     row_block: int = 4096) -> dict:
    """Whole-batch oracle: every row, the loss, and (optionally) all dL/dlogits.

    ``batch`` holds numpy arrays: logits [T, ld], targets, logp_old, logp_infer,
    mask, cu_seqlens, rewards_or_adv. Rows are streamed in blocks.
    """
    cu = batch["cu_seqlens"]
    T = int(cu[-1])
    n, adv, w = seq_prep(cu, batch["mask"], batch["rewards_or_adv"], p)
    parts = []
    for r0 in range(0, T, row_block):
        ids = np.arange(r0, min(T, r0 + row_block), dtype=np.int64)
        parts.append(rows(ids, batch["logits"][r0:r0 + len(ids)], dtype, V, batch["targets"],
                          batch["logp_old"], batch["logp_infer"], batch["mask"], cu, adv, w, p,
                          want_dz=want_dz, token_adv=batch.get("token_adv")))
    if not parts:  # no tokens at all
        parts.append(rows(np.zeros(0, np.int64), np.zeros((0, V), {F32: np.float32, BF16: np.uint16,
                          F64: np.float64}[dtype]), dtype, V, batch["targets"], batch["logp_old"],
                          batch["logp_infer"], batch["mask"], cu, adv, w, p, want_dz=want_dz,
                          token_adv=batch.get("token_adv")))
    out = {k: np.concatenate([o[k] for o in parts]) for k in parts[0]}
    out["loss"] = loss(cu, w, out["tok_obj"])
    out["n_tokens"], out["adv"], out["w"] = n, adv, w
    return out


def pop_in_bounds(logp_old: float, logp_infer: float, beta: float) -> bool:
    return bool(_load().oracle_pop_in_bounds(logp_old, logp_infer, beta))


def clip_active(logp: float, logp_old: float, adv: float, eps_low: float, eps_high: float) -> bool:
    return bool(_load().oracle_clip_active(logp, logp_old, adv, eps_low, eps_high))


def clip_active_vec(logp_f32, logp_old, adv_per_token, eps_low: float, eps_high: float) -> np.ndarray:
    """The clip decision taken from given fp32 log-probs (one per token)."""
    lp = np.ascontiguousarray(logp_f32, dtype=np.float32)
    lo = np.ascontiguousarray(logp_old, dtype=np.float32)
    a = np.ascontiguousarray(adv_per_token, dtype=np.float64)
    out = np.zeros(lp.shape[0], np.uint8)
    _load().oracle_clip_active_vec(lp.shape[0], _ptr(lp), _ptr(lo), _ptr(a), eps_low, eps_high, _ptr(out))
    return out


def thresholds_f32(beta: float, eps_low: float, eps_high: float):
    """(fl32(ln beta), fl32(ln(1 + eps_high)), fl32(ln(1 - eps_low)))."""
    lib = _load()
    return lib.oracle_ln_beta_f32(beta), lib.oracle_clip_hi_f32(eps_high), lib.oracle_clip_lo_f32(eps_low)


# ---------------------------------------------------------------------------- fused projection

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) as float64 (exact: bf16 is the top half of binary32)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def projection_logits(hidden_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """z = h W^T in float64 from bf16 inputs ("GLM-5: from Vibe Coding to
    Agentic Engineering", section 2.4.1: the output projection the chunked path
    computes). A plain library matmul: the products of bf16 values are exact in
    float64."""
    return bf16_bits_to_f64(hidden_bits) @ bf16_bits_to_f64(w_bits).T


def projection_rows(row_ids, hidden_bits, w_bits, targets, logp_old, logp_infer, mask, cu_seqlens, adv, w,
                    p: LossParams, want_dz: bool = False, want_dh: bool = False, w64: np.ndarray | None = None):
    """Per-token results of the loss on projected logits for ``row_ids``;
    with ``want_dh`` also dL/dh_t = sum_v dL/dz_{t,v} W_v for those rows."""
    ids = np.asarray(row_ids, np.int64)
    W = bf16_bits_to_f64(w_bits) if w64 is None else w64
    z = bf16_bits_to_f64(hidden_bits[ids]) @ W.T
    out = rows(ids, np.ascontiguousarray(z), F64, W.shape[0], targets, logp_old, logp_infer, mask, cu_seqlens,
               adv, w, p, want_dz=want_dz or want_dh)
    if want_dh:
        out["dh"] = out["dz"] @ W
    return out


def projection_forward_stats(hidden_bits, w_bits, batch: dict, p: LossParams, row_block: int = 1024,
                             w64: np.ndarray | None = None) -> dict:
    """The forward of the fused path over every row, streamed in blocks of
    ``row_block`` rows so that no [T, V] array is held: per token the log-prob,
    entropy, flags, objective term and dL/dlogp (``g``), and the exact loss of
    Eq. (1) ("GLM-5: from Vibe Coding to Agentic Engineering", section 3.2) on
    the projected logits z = h W^T (section 2.4.1). No dL/dz is formed."""
    cu = batch["cu_seqlens"]
    T = int(cu[-1])
    n, adv, w = seq_prep(cu, batch["mask"], batch["rewards_or_adv"], p)
    W = bf16_bits_to_f64(w_bits) if w64 is None else w64
    keys = ("logp", "entropy", "flags", "tok_obj", "g")
    parts = {k: [] for k in keys}
    for r0 in range(0, T, row_block):
        ids = np.arange(r0, min(T, r0 + row_block), dtype=np.int64)
        z = np.ascontiguousarray(bf16_bits_to_f64(hidden_bits[r0:r0 + len(ids)]) @ W.T)
        o = rows(ids, z, F64, W.shape[0], batch["targets"], batch["logp_old"], batch["logp_infer"], batch["mask"],
                 cu, adv, w, p)
        for k in keys:
            parts[k].append(o[k])
    out = {k: (np.concatenate(v) if v else np.zeros(0)) for k, v in parts.items()}
    out["loss"] = loss(cu, w, out["tok_obj"]) if T else loss(cu, w, np.zeros(0))
    out["n_tokens"], out["adv"], out["w"] = n, adv, w
    return out


def projection_dw_rows(vocab_ids, h: np.ndarray, W: np.ndarray, targets, logp, g, magnitudes: bool = False):
    """Rows ``vocab_ids`` of dL/dW = (dL/dz)^T h for the fused path, from the
    per-token log-probs and dL/dlogp of the forward (``logp``, ``g``) on float64
    h [T, H] and W [V, H]: dL/dz_{t,v} = g_t (1[v = y_t] - exp(z_{t,v} - logZ_t))
    with logZ_t = z_{t,y_t} - logp_t (the chain rule through Eq. (1)'s log-prob,
    section 3.2). Rows with g_t = 0 contribute nothing. With ``magnitudes`` also
    |dL/dz|^T |h| and sqrt((dL/dz)^2^T h^2), the sizes of the product's terms
    (for error bounds)."""
    ids = np.asarray(vocab_ids, np.int64)
    g = np.asarray(g, np.float64)
    live = np.nonzero(g != 0.0)[0]
    hl = h[live]
    y = np.asarray(targets, np.int64)[live]
    zy = np.einsum("th,th->t", hl, W[y])
    logz = zy - np.asarray(logp, np.float64)[live]
    zv = hl @ W[ids].T
    dz = g[live][:, None] * ((y[:, None] == ids[None, :]).astype(np.float64) - np.exp(zv - logz[:, None]))
    if magnitudes:
        return dz.T @ hl, np.abs(dz).T @ np.abs(hl), np.sqrt((dz * dz).T @ (hl * hl))
    return dz.T @ hl


def projection_forward_backward_f64(h: np.ndarray, W: np.ndarray, batch: dict, p: LossParams) -> dict:
    """Whole-batch oracle of the fused path on float64 hidden states h [T, H]
    and LM head W [V, H]: z = h W^T, the loss of Eq. (1) on z, dL/dz, and by the
    chain rule dL/dh = dL/dz W and dL/dW = (dL/dz)^T h."""
    cu = batch["cu_seqlens"]
    T = int(cu[-1])
    n, adv, w = seq_prep(cu, batch["mask"], batch["rewards_or_adv"], p)
    z = np.ascontiguousarray(h[:T] @ W.T)
    out = rows(np.arange(T), z, F64, W.shape[0], batch["targets"], batch["logp_old"], batch["logp_infer"],
               batch["mask"], cu, adv, w, p, want_dz=True)
    out["dh"] = out["dz"] @ W
    out["dW"] = out["dz"].T @ h[:T]
    out["loss"] = loss(cu, w, out["tok_obj"])
    out["n_tokens"], out["adv"], out["w"] = n, adv, w
    return out


def projection_forward_backward(hidden_bits, w_bits, batch: dict, p: LossParams) -> dict:
    """The same on bf16 inputs (bit patterns), widened exactly to float64."""
    return projection_forward_backward_f64(bf16_bits_to_f64(hidden_bits), bf16_bits_to_f64(w_bits), batch, p)


# ---------------------------------------------------------------------------- GAE

def gae(cu_seqlens, rewards, values, mask, gamma: float, lam: float, skip_observations: bool = True,
        rollout_ids=None) -> np.ndarray:
    """Skip-observation GAE per response, optionally with the cross-trajectory
    discount over consecutive responses of one rollout (see oracle_gae)."""
    lib = _load()
    if not hasattr(lib, "_gae_typed"):
        P = ctypes.c_void_p
        lib.oracle_gae.argtypes = [ctypes.c_int64, P, P, P, P, ctypes.c_double, ctypes.c_double, ctypes.c_int32,
                                   P, P]
        lib.oracle_gae.restype = ctypes.c_int32
        lib._gae_typed = True
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    r = np.ascontiguousarray(rewards, dtype=np.float32)
    v = np.ascontiguousarray(values, dtype=np.float32)
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    ro = None if rollout_ids is None else np.ascontiguousarray(rollout_ids, dtype=np.int32)
    out = np.zeros(int(cu[-1]) if cu.size else 0, np.float64)
    rc = lib.oracle_gae(cu.shape[0] - 1, _ptr(cu), _ptr(r), _ptr(v), _ptr(m), gamma, lam, int(skip_observations),
                        _ptr(ro), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_gae rejected its arguments")
    return out
