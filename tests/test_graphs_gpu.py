"""The two-kernel path inside a captured CUDA graph.

A serving loop captures its per-step launches once and replays them.  With
a workspace allocated beforehand the forward enqueues nothing but kernels
and one memset, so it can be captured; the library's own overlapped and
segmented schedules (which order kernels on streams of their own by events)
fall back to the caller's stream while it is being captured.  Each replay
must give the same bits as an eager call on the same inputs, including after
the inputs are rewritten in place between replays.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_32_gb300 import kda
from kda_inputs import make_inputs, small_workload

pytestmark = pytest.mark.gpu

SPLIT = kda.KDA_ALGO_SPLIT
REC = 66048


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    kda.load()
    yield
    kda.kda_debug_split_segments(0)


CASES = {
    # one slice, 12 state chains
    "dense": dict(w=dict(B=2, T=1000, H=3, s0_std=0.02, seed=101), ws_chunks=None, seg=-1),
    # few chains and a workspace of 4 chunks: eagerly the overlapped slice
    # schedule (two library streams), captured one slice after another
    "overlapped": dict(w=dict(B=1, T=1500, H=2, s0_std=0.02, seed=102), ws_chunks=4, seg=-1),
    # three segments: eagerly the last segment's records beside pass 1
    "segmented": dict(w=dict(B=1, T=1500, H=2, s0_std=0.02, seed=103), ws_chunks=None, seg=3),
    "packed": dict(w=dict(B=1, T=577, H=2, varlen=True, lengths=(130, 0, 1, 300, 64, 65, 17),
                          s0_std=0.03, seed=104), ws_chunks=None, seg=-1),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_forward_replays_in_a_cuda_graph(name):
    case = CASES[name]
    w = small_workload("graph_" + name, dk=128, dv=128, **case["w"])
    x = make_inputs(w)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    packed = d["cu_seqlens"] is not None
    N = d["cu_seqlens"].numel() - 1 if packed else x["B"]
    T, H = x["T"], x["H"]
    kda.kda_debug_split_segments(case["seg"])
    try:
        if case["ws_chunks"]:
            carry = (N * H * 128 * 128 * 4 + 255) // 256 * 256
            nb = carry + N * H * REC * case["ws_chunks"]
        else:
            nb = kda.kda_workspace_bytes(N, T, H, 128, 128, kda.KDA_BF16, 0, SPLIT, int(packed))
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        out = torch.empty_like(d["v"])
        fs = torch.empty(N, H, 128, 128, device="cuda")

        def call():
            rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                      d["init_state"], out, fs, N, T, H, 128, 128,
                                      d["cu_seqlens"], kda.KDA_BF16, 0, 1.0, SPLIT, ws, nb,
                                      None, torch.cuda.current_stream())
            assert rc == 0, kda.status_string(rc)

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call()                                   # eager, on a side stream
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        o_eager, s_eager = out.clone(), fs.clone()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        out.zero_()
        fs.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, o_eager) and torch.equal(fs, s_eager)
        # new inputs written in place, then replay against an eager call
        gen = torch.Generator(device="cpu").manual_seed(7)
        for key in ("q", "k", "v"):
            d[key].copy_((d[key].float().cpu() *
                          (1.0 + 0.1 * torch.rand(d[key].shape, generator=gen))).to(d[key].dtype))
        graph.replay()
        torch.cuda.synchronize()
        o_replay, s_replay = out.clone(), fs.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(o_replay, out) and torch.equal(s_replay, fs)
        assert not torch.equal(o_replay, o_eager)
    finally:
        kda.kda_debug_split_segments(0)
