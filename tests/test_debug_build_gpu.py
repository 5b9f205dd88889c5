"""The debug build (-DKDA_DEBUG): device-side bounds checks on the two-kernel
path that report KDA_ERR_BOUNDS instead of trapping.

A fresh child process loads the debug library as its only libkda.so.  On a
dense batch, a packed batch and a dense batch in the segmented form it must
match the fp64 oracle with no check firing;
told (through a debug-only hook) that the workspace holds just two chunk
records, its kernels must report KDA_ERR_BOUNDS without touching memory past
that point (the real workspace holds every record, so nothing can go astray
even if a check were missing); and the next normal call must give the same
bits as before.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_checks_fire_and_clean_calls_match():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build, kda
    build.build(debug=True)
    r = subprocess.run([sys.executable, os.path.join("tests", "_debug_build_child.py")],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert "debug build" in res["info"]
    for name in ("dense", "packed", "segmented"):
        c = res[name]
        assert c["rc"] == 0 and c["status"] == kda.KDA_OK, (name, c)
        assert c["err_o"] <= 1e-2 and c["err_s"] <= 1e-2, (name, c)
        assert c["rc_small"] == 0 and c["status_small"] == kda.KDA_ERR_BOUNDS, (name, c)
        assert c["status_after"] == kda.KDA_OK and c["same_after"], (name, c)
