"""bench.py rejects flag combinations it cannot run, before it touches a GPU."""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("argv", [
    ["--form", "gated"],                                   # a form without a profiling mode
    ["--decode-only", "2", "--form", "gated"],             # decode has the plain and fused forms only
    ["--prefill-only", "--form", "fused"],                 # fused is a decode form
    ["--prefill-only", "--decode-only", "2"],              # one profiling mode at a time
    ["--prologue-only", "--prefill-only"],
])
def test_rejected_combinations(argv):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], capture_output=True, text=True,
                       cwd=ROOT, timeout=120)
    assert r.returncode == 2 and "error:" in r.stderr, (r.returncode, r.stderr[-300:])
