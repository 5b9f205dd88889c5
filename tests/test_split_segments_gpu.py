"""The segmented form of the two-kernel path (dense batches of few long
sequences): each sequence is cut into G segments; pass 1 runs segment 0 in
full and summarises segments 1 .. G - 2 (zero-start final state and
cumulative transition, the state update being affine in the entering
state); the entry states follow by composition; pass 2 reruns segments
1 .. G - 1 from them.

Parity against the fp64 oracle (max |gpu - ref| / max |ref| <= 1e-2 on the
output and the final state), and against the plain two-kernel run by the
triangle bound (2e-2): the two take different rounding paths, so they are
not bit-identical.  A workspace below the segmented size must give the
plain run exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_32_gb300 import kda
from kda_inputs import make_inputs, small_workload

pytestmark = pytest.mark.gpu

SPLIT = kda.KDA_ALGO_SPLIT


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    kda.load()
    yield
    kda.kda_debug_split_segments(0)


def rel(a, b):
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / den) if den > 0 else float(np.abs(a).max())


def run(x, segments, ws_bytes=None, final=True):
    """One forward with `segments` forced (-1: none); the workspace the
    path asks for under that setting unless ws_bytes is given."""
    kda.kda_debug_split_segments(segments)
    try:
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
        B, T, H = x["B"], x["T"], x["H"]
        nb = ws_bytes or kda.kda_workspace_bytes(B, T, H, 128, 128, kda.KDA_BF16, 0, SPLIT, 0)
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        out = torch.empty_like(d["v"])
        fs = torch.empty(B, H, 128, 128, device="cuda") if final else None
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                  out, fs, B, T, H, 128, 128, None, kda.KDA_BF16, 0, 1.0, SPLIT,
                                  ws, nb, status, torch.cuda.current_stream())
        assert rc == 0, kda.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        return (out.float().cpu().numpy(), fs.cpu().numpy() if final else None, nb)
    finally:
        kda.kda_debug_split_segments(0)


@pytest.mark.parametrize("B,T,H,G,s0_std,g_mean", [
    (2, 1500, 2, 3, 0.02, 0.0),    # 24 chunks, the last ragged: 8 + 8 + 8
    (1, 645, 3, 3, 0.0, 0.0),      # 11 chunks: 4 + 4 + 3
    (1, 645, 2, 5, 0.03, 0.0),     # five asked, four possible: 3 + 3 + 3 + 2
    (2, 2048, 1, 6, 0.02, 4.0),    # heavy decay (many steps at the floor)
    (1, 1000, 2, 4, 0.02, -200.0), # alpha = 1 exactly (no decay)
])
def test_segments_match_oracle_and_plain_run(B, T, H, G, s0_std, g_mean):
    w = small_workload("segsplit", B=B, T=T, H=H, dk=128, dv=128, s0_std=s0_std,
                       g_mean=g_mean, seed=61)
    x = make_inputs(w)
    o_seg, s_seg, nb_seg = run(x, G)
    o_pl, s_pl, nb_pl = run(x, -1)
    assert nb_seg > nb_pl                      # the segmented form was chosen
    o_ref, s_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"])
    assert rel(o_seg, o_ref) <= 1e-2, rel(o_seg, o_ref)
    assert rel(s_seg, s_ref) <= 1e-2, rel(s_seg, s_ref)
    assert rel(o_seg, o_pl) <= 2e-2 and rel(s_seg, s_pl) <= 2e-2


def test_segments_without_final_state_and_run_to_run_identical():
    w = small_workload("segsplit2", B=1, T=1200, H=2, dk=128, dv=128, s0_std=0.02, seed=62)
    x = make_inputs(w)
    o1, _, _ = run(x, 3, final=False)
    o2, s2, _ = run(x, 3)
    np.testing.assert_array_equal(o1, o2)      # the final state changes nothing else
    o3, s3, _ = run(x, 3)
    np.testing.assert_array_equal(o2, o3)      # deterministic
    np.testing.assert_array_equal(s2, s3)


def test_workspace_below_the_segmented_size_runs_the_plain_form():
    w = small_workload("segsplit3", B=1, T=1000, H=2, dk=128, dv=128, s0_std=0.02, seed=63)
    x = make_inputs(w)
    o_pl, s_pl, nb_pl = run(x, -1)
    # segments asked for, but the workspace only holds the plain form's
    o_small, s_small, _ = run(x, 3, ws_bytes=nb_pl)
    np.testing.assert_array_equal(o_small, o_pl)
    np.testing.assert_array_equal(s_small, s_pl)


def test_segment_state_stall_reports_timeout():
    """The bounded waits of both state passes: the first wait of every state
    CTA runs out, the call reports KDA_ERR_TIMEOUT, and the next normal
    segmented call is bit-identical to a clean one."""
    w = small_workload("segsplit4", B=1, T=1000, H=1, dk=128, dv=128, seed=64)
    x = make_inputs(w)
    clean_o, clean_s, _ = run(x, 3)
    kda.kda_debug_split_segments(3)
    kda.kda_debug_stall_test(2)
    try:
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
        nb = kda.kda_workspace_bytes(1, 1000, 1, 128, 128, kda.KDA_BF16, 0, SPLIT, 0)
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        out = torch.empty_like(d["v"])
        fs = torch.empty(1, 1, 128, 128, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], None, out, fs, 1,
                                  1000, 1, 128, 128, None, kda.KDA_BF16, 0, 1.0, SPLIT, ws, nb,
                                  status, torch.cuda.current_stream())
        assert rc == 0
        torch.cuda.synchronize()
        assert int(status.item()) == kda.KDA_ERR_TIMEOUT
    finally:
        kda.kda_debug_stall_test(0)
        kda.kda_debug_split_segments(0)
    o, s, _ = run(x, 3)
    np.testing.assert_array_equal(o, clean_o)
    np.testing.assert_array_equal(s, clean_s)


def test_segments_update_the_state_in_place():
    """init_state and final_state may be one buffer: segment 0 reads it in
    pass 1, the last segment writes it at the end of pass 2."""
    w = small_workload("segsplit5", B=2, T=1100, H=2, dk=128, dv=128, s0_std=0.03, seed=65)
    x = make_inputs(w)
    o_ref, s_ref = run(x, 3)[:2]
    kda.kda_debug_split_segments(3)
    try:
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
        nb = kda.kda_workspace_bytes(2, 1100, 2, 128, 128, kda.KDA_BF16, 0, SPLIT, 0)
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        out = torch.empty_like(d["v"])
        st = d["init_state"].clone()
        rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], st, out, st, 2,
                                  1100, 2, 128, 128, None, kda.KDA_BF16, 0, 1.0, SPLIT, ws, nb,
                                  None, torch.cuda.current_stream())
        assert rc == 0, kda.status_string(rc)
        torch.cuda.synchronize()
    finally:
        kda.kda_debug_split_segments(0)
    np.testing.assert_array_equal(out.float().cpu().numpy(), o_ref)
    np.testing.assert_array_equal(st.cpu().numpy(), s_ref)
