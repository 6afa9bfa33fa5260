"""The bounds-checked build: small calls of every kernel family run against
libs4_checked.so, built with -DS4_BOUNDS_CHECK (every global and shared-memory
index of the instrumented kernels compared with its buffer's extent, an index
outside counted and its access skipped, nothing trapped); none may be counted.
The calls run in a child process (tests/bounds_cases.py) that loads the checked
library through S4_LIB, so this process keeps the normal build."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

from structured_state_space_gb300 import build as s4build  # noqa: E402

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_no_index_leaves_its_buffer():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = s4build.build(bounds_check=True)
    env = dict(os.environ, S4_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["calls"] >= 40
    assert out["violations"] == 0, out
