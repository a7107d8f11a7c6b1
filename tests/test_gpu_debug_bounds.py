"""The bounds-checking build (DFA_DEBUG_BOUNDS): the attention kernels check
every global index they compute against its tensor's extent and report a
violation through the status word (DFA_ERR_BOUNDS) instead of making the
access.  This runs the small odd-shape parity cases -- sequences of 1, 2, 63,
65, 129, 513 tokens, grouped-query heads, ragged tiles, block striping, a
chunk pair that sees no key, documents -- once in a child process that loads
that build, and requires them to pass with every status check clean (each
case reads the status word back through dfa_stream_status)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_small_cases_clean_under_bounds_checks():
    env = dict(os.environ, DFA_DEBUG_BOUNDS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_gpu_parity.py"), os.path.join(ROOT, "tests",
                                                                           "test_gpu_docs.py"),
           "-k", "small or block_striped or fully_masked or partitioned or docs"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "error" not in r.stdout.lower().split("passed")[-1], tail
    # the child really ran the bounds-checking build
    assert os.path.exists(os.path.join(ROOT, "long_context_flashattention_gb300",
                                       "libdfa_bounds.so"))
