"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports exactly the functions ``include/rl_loss.h`` declares,
and its structs have the layout the binding marshals."""
import ctypes
import os
import subprocess
import tempfile

import pytest

from rl_post_loss_gb300 import build as nvbuild
from rl_post_loss_gb300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return capi.load()


def test_library_exports_every_declared_function(lib):
    names = capi.header_functions()
    assert "rl_loss_forward_backward" in names and "rl_loss_create" in names
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.check_output(["nm", "-D", "--defined-only", capi.LIB_PATH]).decode()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    api = {n for n in exported if n.startswith(("rl_loss_", "rl_gae_", "rl_topk"))}
    assert api == set(names), (api ^ set(names))


def test_struct_layout_matches_header():
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "rl_loss.h"
#define F(s, f) printf(#s "." #f " %zu\n", offsetof(s, f));
int main(void) {
  printf("rl_loss_config %zu\n", sizeof(rl_loss_config));
  printf("rl_loss_inputs %zu\n", sizeof(rl_loss_inputs));
  printf("rl_loss_outputs %zu\n", sizeof(rl_loss_outputs));
  printf("rl_loss_profile %zu\n", sizeof(rl_loss_profile));
  printf("rl_gae_config %zu\n", sizeof(rl_gae_config));
  F(rl_loss_config, logits_dtype) F(rl_loss_config, adv_eps)
  F(rl_loss_inputs, ld_logits) F(rl_loss_inputs, logits) F(rl_loss_inputs, rewards_or_adv)
  F(rl_loss_outputs, ld_dlogits) F(rl_loss_outputs, mean_entropy) F(rl_loss_outputs, counts)
  F(rl_loss_profile, launches) F(rl_loss_profile, total_ms)
  F(rl_gae_config, skip_observations) F(rl_gae_config, cross_trajectory)
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write(src)
        subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), c, "-o", exe])
        got = dict(line.split() for line in subprocess.check_output([exe]).decode().splitlines())
    sizes = {"rl_loss_config": capi.rl_loss_config, "rl_loss_inputs": capi.rl_loss_inputs,
             "rl_loss_outputs": capi.rl_loss_outputs, "rl_loss_profile": capi.rl_loss_profile,
             "rl_gae_config": capi.rl_gae_config}
    for name, cls in sizes.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
    for key, val in got.items():
        if "." in key:
            s, f = key.split(".")
            assert getattr(sizes[s], f).offset == int(val), key


def test_host_only_entry_points(lib):
    assert capi.rl_loss_version() >= 100
    assert capi.rl_loss_status_string(0) == "ok"
    for code in range(1, 15):
        assert capi.rl_loss_status_string(code) not in ("", "unknown status")
    assert capi.rl_loss_status_string(99) == "unknown status"
    assert set(capi.STATUS_NAMES.values()) >= {"RL_OK", "RL_ERR_SEQLENS"}


def test_null_arguments_are_rejected_without_a_device(lib):
    # these return before touching CUDA
    assert lib.rl_loss_create(None, None) == capi.CODES["RL_ERR_INVALID_ARG"]
    assert lib.rl_loss_forward_backward(None, None, None, None) == capi.CODES["RL_ERR_INVALID_ARG"]
    inp, out = capi.rl_loss_inputs(), capi.rl_loss_outputs()
    for args in ((None, None, None, None, 8, None),
                 (None, ctypes.byref(inp), ctypes.byref(inp), ctypes.byref(out), 8, None)):
        assert lib.rl_loss_forward_backward_from_host(*args) == capi.CODES["RL_ERR_INVALID_ARG"]
    assert lib.rl_loss_destroy(None) == 0
    bad = capi.rl_loss_config(0, 1, 1, 1, 0.2, 0.28, 2.0, 1e-6, 0, 0, 0, 1)
    h = ctypes.c_void_p()
    assert lib.rl_loss_create(ctypes.byref(bad), ctypes.byref(h)) == capi.CODES["RL_ERR_SHAPE"]
    bad = capi.rl_loss_config(8, 1, 1, 1, 0.2, 0.28, 1.0, 1e-6, 0, 0, 0, 1)  # beta must be > 1
    assert lib.rl_loss_create(ctypes.byref(bad), ctypes.byref(h)) == capi.CODES["RL_ERR_INVALID_ARG"]
    bad = capi.rl_loss_config(8, 1, 1, 1, 0.2, 0.28, 2.0, 1e-6, 0, 0, 0, 7)
    assert lib.rl_loss_create(ctypes.byref(bad), ctypes.byref(h)) == capi.CODES["RL_ERR_DTYPE"]


def test_binding_fails_loudly_without_library(tmp_path):
    saved = capi._lib
    capi._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            capi.load(str(tmp_path / "nope.so"))
    finally:
        capi._lib = saved


def test_gae_host_side_argument_checks(lib):
    # every check below returns before any CUDA call; the pointers are never dereferenced
    cfg = capi.rl_gae_config(1.0, 0.95, 1, 0)
    fake = ctypes.c_void_p(0x10000)
    T = 10000
    need = capi.rl_gae_workspace_bytes(T)
    assert need >= 256 + 3 * 32
    args = lambda ws, nbytes: (ctypes.byref(cfg), T, 4, fake, fake, fake, fake, None, fake, None, ws, nbytes, None,
                               None)
    assert lib.rl_gae_advantages(*args(fake, need - 1)) == capi.CODES["RL_ERR_CAPACITY"]
    assert lib.rl_gae_advantages(*args(ctypes.c_void_p(0x10010), need)) == capi.CODES["RL_ERR_ALIGNMENT"]
    assert lib.rl_gae_advantages(*args(None, need)) == capi.CODES["RL_ERR_INVALID_ARG"]
    bad = capi.rl_gae_config(1.5, 0.95, 1, 0)
    assert lib.rl_gae_advantages(ctypes.byref(bad), T, 4, fake, fake, fake, fake, None, fake, None, fake, need, None,
                                 None) == capi.CODES["RL_ERR_INVALID_ARG"]
    cross = capi.rl_gae_config(1.0, 0.95, 1, 1)
    assert lib.rl_gae_advantages(ctypes.byref(cross), T, 4, fake, fake, fake, fake, None, fake, None, fake, need, None,
                                 None) == capi.CODES["RL_ERR_INVALID_ARG"]


def test_topk_host_side_argument_checks(lib):
    fake = ctypes.c_void_p(0x10000)
    ok = capi.rl_topk_config(2048, capi.RL_TOPK_BY_SCORE)
    assert capi.rl_topk_max_k() == 4096
    call = lambda cfg, rows=4, ld=4096, scores=fake, ldo=2048: lib.rl_topk(
        ctypes.byref(cfg), rows, scores, ld, None, fake, None, ldo, None, None)
    assert call(capi.rl_topk_config(0, 0)) == capi.CODES["RL_ERR_UNSUPPORTED"]
    assert call(capi.rl_topk_config(4097, 0)) == capi.CODES["RL_ERR_UNSUPPORTED"]
    assert call(capi.rl_topk_config(16, 7)) == capi.CODES["RL_ERR_INVALID_ARG"]
    assert call(ok, ldo=100) == capi.CODES["RL_ERR_SHAPE"]
    assert call(ok, rows=-1) == capi.CODES["RL_ERR_SHAPE"]
    assert call(ok, ld=4098) == capi.CODES["RL_ERR_ALIGNMENT"]
    assert call(ok, scores=ctypes.c_void_p(0x10004)) == capi.CODES["RL_ERR_ALIGNMENT"]
    assert call(ok, scores=None) == capi.CODES["RL_ERR_INVALID_ARG"]
    assert call(ok, rows=0) == capi.CODES["RL_OK"]
