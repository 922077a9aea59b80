"""The debug-checks build: every kernel compiled with S3D8_DEBUG_CHECKS, whose
in-kernel bounds checks (ring slots and stage indexes, tensor-memory column
ranges, global output and partial-sum indexes) record S3D8_ERR_BOUNDS in the
device status word instead of touching memory out of range.  It stands in for a
memory checker: the parity tests on the small case, the odd shapes of every
algorithm and the grouped launches run against that build in a child process
(S3D8_LIBRARY=debug), must pass, and must leave the device status clear (each
test module asserts it on teardown).
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SELECTION = ("tiny or small_exact or tc_tiles or tmem_in_full or tc_unaligned or int32_extremes "
             "or layer_fused or mixed_jobs or zero_activation or plain_entry")


def test_parity_suite_passes_with_bounds_checks_compiled_in():
    env = dict(os.environ, S3D8_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", SELECTION,
                        os.path.join(ROOT, "tests", "test_gpu_parity.py"),
                        os.path.join(ROOT, "tests", "test_gpu_batch.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
