"""The debug build (-DATTN_DEBUG) checks every computed index on the device
and records a failed check in the workspace header instead of accessing
memory.  Small ragged / windowed / GQA cases must run clean (device status 0,
which the binding checks after every call) and still match the oracle."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_index_checks_clean():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_build_cases.py")],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert r.stdout.count("ok ") == 27, r.stdout
