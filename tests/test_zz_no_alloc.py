"""The allocation-free segmented forward (kda_chunk_fwd_seg_static).

It is for callers that may not allocate device memory at all -- an engine
that has reserved every byte of HBM for its own pools, or a host framework
that neither provides a workspace nor permits allocation.  It keeps its
segment scratch in a fixed array inside the library; this test checks that
two calls in a row through the C ABI give the same result as the workspace
entry point (kda_chunk_fwd_seg) on the same inputs.  Collected last so that
a failure here stops a run only after every other test.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_32_gb300 import kda
from kda_inputs import make_inputs, small_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    kda.load()


def _inputs(seed):
    w = small_workload("na", B=2, T=1000, H=3, dk=128, dv=128, seed=seed, s0_std=0.05)
    x = make_inputs(w)
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}


def _rel(a, b):
    a, b = a.float().cpu().numpy(), b.float().cpu().numpy()
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def test_static_scratch_matches_workspace_entry_twice():
    nseg = 3
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((21, 22)):  # two calls in a row, fresh inputs each
        d = _inputs(seed)
        B, T, H = d["B"], d["T"], d["H"]
        out_a = torch.empty_like(d["v"])
        fs_a = torch.empty(B, H, 128, 128, device="cuda")
        rc = kda.kda_chunk_fwd_seg_static(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                          d["init_state"], out_a, fs_a, B, T, H, 128, 128, 1.0,
                                          nseg, None, stream)
        assert rc == 0, kda.status_string(rc)
        out_b = torch.empty_like(d["v"])
        fs_b = torch.empty(B, H, 128, 128, device="cuda")
        rc = kda.kda_chunk_fwd_seg(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                   out_b, fs_b, B, T, H, 128, 128, 1.0, nseg, None, 0, None,
                                   stream)
        assert rc == 0, kda.status_string(rc)
        torch.cuda.synchronize()
        assert _rel(out_a, out_b) <= 1e-2, call
        assert _rel(fs_a, fs_b) <= 1e-2, call


def test_static_scratch_rejects_oversized_batches():
    d = _inputs(23)
    # 32 heads x 8 segments x 192 KiB exceeds the fixed 16 MiB array
    rc = kda.kda_chunk_fwd_seg_static(d["q"], d["k"], d["v"], d["g"], d["beta"], None,
                                      torch.empty_like(d["v"]), None, 1, 10, 32, 128, 128, 1.0,
                                      8, None, torch.cuda.current_stream())
    assert rc == kda.KDA_ERR_WORKSPACE
