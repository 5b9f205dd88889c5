"""Step-by-step parity of the tensor-core path's intra-chunk quantities
(cumulative decay, Gram matrices, (I + A_kk)^-1, W, U) against the oracle's
fp64 chunk mirror, through the kda_debug_intra test hook."""
import numpy as np
import pytest
import torch

from oracle import chunk_mirror
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


@pytest.mark.parametrize("gmode", ["normal", "floor_heavy", "alpha_one"])
def test_intra_steps(gmode):
    T, H, n, h = 150, 2, 0, 1
    w = small_workload("st", B=1, T=T, H=H, dk=128, dv=128, seed=21)
    x = make_inputs(w)
    if gmode == "floor_heavy":
        x["g"] = (torch.randn(x["g"].shape, generator=torch.Generator().manual_seed(1)) + 6.0
                  ).to(torch.bfloat16)
    elif gmode == "alpha_one":
        x["g"] = torch.full_like(x["g"], -200.0)
    nch = (T + 63) // 64
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    buf = {k: torch.zeros(nch, 64, c, device="cuda")
           for k, c in (("gam", 128), ("aqk", 64), ("akk", 64), ("tinv", 64), ("w", 128),
                        ("u", 128))}
    rc = kda.kda_debug_intra(d["q"], d["k"], d["v"], d["g"], d["beta"], 1, T, H, 128, 128, None,
                             n, h, buf["gam"], buf["aqk"], buf["akk"], buf["tinv"], buf["w"],
                             buf["u"], torch.cuda.current_stream())
    assert rc == 0
    torch.cuda.synchronize()
    f64 = lambda t: t[n, :, h].double().numpy()
    _, _, steps = chunk_mirror.forward_unit(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]),
                                            f64(x["beta"]), None, chunk=64, return_steps=True)
    got = {k: v.cpu().numpy() for k, v in buf.items()}
    for c, st in enumerate(steps):
        L = min(64, T - 64 * c)
        gam_ref = np.exp(st["Gam"])
        assert np.abs(got["gam"][c][:L] - gam_ref[:L]).max() <= 1e-5, c
        assert rel(got["aqk"][c][:L, :L], st["Aqk"][:L, :L]) <= 1e-2, c
        assert rel(got["akk"][c][:L, :L], st["Akk"][:L, :L]) <= 1e-2, c
        assert rel(got["tinv"][c][:L, :L], st["T"][:L, :L]) <= 1e-2, c
        assert rel(got["w"][c][:L], st["W"][:L]) <= 2e-2, c
        assert rel(got["u"][c][:L], st["U"][:L]) <= 2e-2, c
