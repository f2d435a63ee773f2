"""The single-role tensor-core prefill (`prefill_tc_kernel`: 128 threads per CTA,
thread = query row, two CTAs per SM). Head_dim 64 always runs it; head_dim 128
runs the warp-specialised kernel unless UQ_PREFILL=tc, which the library reads
once per process. So the prefill and cascade parity tests run a second time in
a child process with it selected, to the same bar as the default kernel."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_prefill_and_cascade_on_single_role_kernel():
    env = dict(os.environ, UQ_PREFILL="tc")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        "tests/test_gpu_prefill.py", "tests/test_gpu_cascade.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-6000:] + r.stderr[-3000:]
    print(r.stdout[-2000:])
