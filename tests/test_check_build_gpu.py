"""The check build (libtkg_check.so, TKG_CHECK=1): every kernel verifies its
internal invariants -- tensor-memory column ranges, ring-slot, accumulator,
tile, group and list indices, TMA x alignment -- and reports a failure as
TKG_ERR_CHECK instead of trapping.  The random, tail-split, list, epilogue and
strided suites run again against it in a subprocess: each of their cases
asserts a clean device status, so any failed invariant fails them, and their
outputs are still compared with the oracle."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_suites_pass_on_the_check_build():
    from dense_block_scaled_gb300 import build
    lib = build.build(check=True)
    env = dict(os.environ, TKG_LIBRARY=lib)
    probe = subprocess.run([sys.executable, "-c", "from dense_block_scaled_gb300 import tkg; print(tkg.load()._name)"],
                           cwd=ROOT, env=env, capture_output=True, text=True)
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libtkg_check.so"), probe.stdout + probe.stderr
    suites = ["tests/test_random_gpu.py", "tests/test_tail_gpu.py", "tests/test_list_gpu.py",
              "tests/test_epilogue_gpu.py", "tests/test_strided_gpu.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *suites],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
