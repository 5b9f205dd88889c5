"""Launch set-up is per device and safe under concurrent first calls.

The library raises each kernel's shared-memory limit and reads the SM count
once per device, under a lock.  A fresh child process makes its first two
calls from two host threads at once (two streams, two different paths) and
checks them bit for bit against the same calls made one after the other.
Only one GPU is available here, so the per-device part is exercised for one
device; the threaded part is exercised in full.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_concurrent_first_calls_match_serial_calls():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    r = subprocess.run([sys.executable, os.path.join("tests", "_threaded_first_calls.py")],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["ok"], line
