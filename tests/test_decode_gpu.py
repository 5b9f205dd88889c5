"""Recurrent decode / speculative-decoding rebuild (kda_decode) against the
oracle, continuing from a state; and equality with the chunked path."""
import numpy as np
import pytest
import torch

import oracle
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


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, 1e-2), (torch.float32, 1e-4)])
@pytest.mark.parametrize("T", [1, 3, 8, 16, 37])
@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 32), (64, 64), (128, 128), (32, 64),
                                   (128, 16)])
def test_decode_matches_oracle(dtype, tol, T, dk, dv):
    # every head size the entry point accepts: dk = 16 leaves two key rows per
    # warp, dv = 16 half of a CTA's 32 value lanes idle
    w = small_workload("dec", B=3, T=T, H=4, dk=dk, dv=dv, dtype=dtype, s0_std=0.5,
                       seed=T * dk + dv)
    x = make_inputs(w)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    st = dev["init_state"].clone()
    out = torch.empty_like(dev["v"])
    dt = kda.KDA_BF16 if dtype == torch.bfloat16 else kda.KDA_F32
    rc = kda.kda_decode(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], st, out, 3, T, 4,
                        dk, dv, dt, 1.0, torch.cuda.current_stream())
    assert rc == 0
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"])
    assert rel(out.float().cpu().numpy(), o_ref) <= tol
    assert rel(st.cpu().numpy(), s_ref) <= tol


def test_decode_continues_a_prefill():
    # prefill 200 tokens with the chunked path, then decode 4 more: equals one run
    w = small_workload("pd", B=2, T=204, H=2, dk=128, dv=128, seed=9, s0_std=0.02)
    x = make_inputs(w)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    st = d["init_state"].clone()
    out1 = torch.empty(2, 200, 2, 128, dtype=torch.bfloat16, device="cuda")
    sl = {k: d[k][:, :200].contiguous() for k in ("q", "k", "v", "g", "beta")}
    assert kda.kda_chunk_fwd(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], st, out1, st, 2, 200,
                             2, 128, 128, None, torch.cuda.current_stream()) == 0
    sl = {k: d[k][:, 200:].contiguous() for k in ("q", "k", "v", "g", "beta")}
    out2 = torch.empty(2, 4, 2, 128, dtype=torch.bfloat16, device="cuda")
    assert kda.kda_decode(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], st, out2, 2, 4, 2, 128,
                          128, kda.KDA_BF16, 1.0, torch.cuda.current_stream()) == 0
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"])
    o = torch.cat([out1, out2], 1).float().cpu().numpy()
    assert rel(o, o_ref) <= 1e-2
    assert rel(st.cpu().numpy(), s_ref) <= 1e-2


def test_decode_zero_tokens_keeps_state():
    st = torch.randn(1, 1, 128, 128, device="cuda")
    before = st.clone()
    assert kda.kda_decode(None, None, None, None, None, st, None, 1, 0, 1, 128, 128,
                          kda.KDA_BF16, 1.0, torch.cuda.current_stream()) == 0
    torch.cuda.synchronize()
    assert torch.equal(st, before)
