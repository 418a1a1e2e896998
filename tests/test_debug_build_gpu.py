"""The debug build of the library: every kernel also checks its index
invariants (a token's response range, the row and the target of a gradient
write, the chunk index of a GAE block, the top-k buffer bounds) and raises
RL_ERR_INTERNAL, skipping the access, where one fails. The small-case parity,
edge-case, fused-projection, GAE and top-k tests run against that build in a
child process (RL_LOSS_LIB names it) and must pass unchanged: their status
checks would see any check that fired."""
import os
import subprocess
import sys

import pytest

from rl_post_loss_gb300 import build as nvbuild

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_small_cases_pass_on_the_debug_build():
    lib = nvbuild.build(debug=True)
    env = dict(os.environ, RL_LOSS_LIB=lib)
    files = ["tests/test_parity_gpu.py", "tests/test_projection_gpu.py", "tests/test_gae_gpu.py",
             "tests/test_topk_gpu.py", "tests/test_canaries_gpu.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "gpu and not slow",
                        "-k", "not mid_size"] + files, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout + r.stderr)[-4000:]
    assert " passed" in r.stdout
