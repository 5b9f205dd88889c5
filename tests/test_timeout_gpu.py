"""The bounded waits of the two-kernel path run out and recover.

Every wait of the tensor-core kernels is bounded; when one gives up, the
kernel records KDA_ERR_TIMEOUT in the device status word, waits (bounded) for
the copies and products it still has in flight, frees its tensor memory and
returns, so the context stays usable.  The test hook kda_debug_stall_test
makes the first wait of the intra-chunk kernel and / or the state kernel wait
on a barrier that nothing ever completes (a 1 ms limit): no fault, no trap,
no hang.  Each case checks that the status reports the timeout and that the
next normal call on the same stream is bit for bit a clean run.
"""
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
    yield
    kda.kda_debug_stall_test(0)


def _run(d, B, T, H, status):
    out = torch.full_like(d["v"], float("nan"))
    fs = torch.full((B, H, 128, 128), float("nan"), device="cuda")
    rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], out,
                              fs, B, T, H, 128, 128, None, kda.KDA_BF16, 0, 1.0,
                              kda.KDA_ALGO_SPLIT, None, 0, status, torch.cuda.current_stream())
    assert rc == 0, kda.status_string(rc)
    torch.cuda.synchronize()
    return out, fs


@pytest.mark.parametrize("flags", [1, 2, 3])
@pytest.mark.parametrize("B,T,H", [(1, 64, 1), (2, 300, 2)])
def test_wait_runs_out_then_next_call_is_clean(flags, B, T, H):
    w = small_workload("to", B=B, T=T, H=H, dk=128, dv=128, seed=61, s0_std=0.05)
    x = make_inputs(w)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_clean, s_clean = _run(d, B, T, H, status)
    assert int(status.item()) == kda.KDA_OK
    try:
        assert kda.kda_debug_stall_test(flags) == kda.KDA_OK
        _run(d, B, T, H, status)
        assert int(status.item()) == kda.KDA_ERR_TIMEOUT
    finally:
        kda.kda_debug_stall_test(0)
    o, s = _run(d, B, T, H, status)
    assert int(status.item()) == kda.KDA_OK
    assert torch.equal(o, o_clean)
    assert torch.equal(s, s_clean)
