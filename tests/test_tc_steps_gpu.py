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
    kk, vv, bb = f64(x["k"]), f64(x["v"]), f64(x["beta"])
    for c, st in enumerate(steps):
        L = min(64, T - 64 * c)
        gam_ref = np.exp(st["Gam"])
        assert np.abs(got["gam"][c][:L] - gam_ref[:L]).max() <= 1e-5, c
        assert rel(got["aqk"][c][:L, :L], st["Aqk"][:L, :L]) <= 1e-2, c
        assert rel(got["akk"][c][:L, :L], st["Akk"][:L, :L]) <= 1e-2, c
        assert rel(got["tinv"][c][:L, :L], st["T"][:L, :L]) <= 1e-2, c
        # Error bound of W = T X (X = beta K gamma) and U = T X (X = beta V),
        # from the arithmetic, elementwise (relative to the terms of each sum,
        # not to max |W|: cancellation can make an entry far smaller than its
        # terms).  With u = 2^-9 the unit roundoff of bf16:
        #   - both operands of the product are rounded to bf16: 2 u |T| |X|;
        #   - the Gram operands are rounded to bf16, so each entry of A =
        #     beta A_kk is off by about 2 u |A|_abs, where |A|_abs sums the
        #     absolute terms beta_r |k_rj| |k_ij| e^{G_rj - G_ij}; through the
        #     inverse this moves T by about |T| (2 u |A|_abs) |T|;
        #   - rounding T to bf16 and the solve's own tf32 steps: about u |T|.
        # The check allows twice the sum.
        kc = np.zeros((64, 128)); kc[:L] = kk[64 * c:64 * c + L]
        vc = np.zeros((64, 128)); vc[:L] = vv[64 * c:64 * c + L]
        bc = np.zeros(64); bc[:L] = bb[64 * c:64 * c + L]
        u = 2.0 ** -9
        absT = np.abs(st["T"])
        G = st["Gam"]
        dec = np.exp(np.minimum(G[:, None, :] - G[None, :, :], 0.0))      # [r, i, j]
        absA = bc[:, None] * np.einsum("rj,ij,rij->ri", np.abs(kc), np.abs(kc), dec)
        absA = np.tril(absA, -1)
        dT = 2 * u * absT @ absA @ absT + u * absT
        for key, X in (("w", bc[:, None] * kc * gam_ref), ("u", bc[:, None] * vc)):
            aX = np.abs(X)
            bound = 2 * (2 * u * absT @ aX + dT @ aX) + 1e-6 * np.abs(st[key.upper()]).max()
            err = np.abs(got[key][c] - st[key.upper()])
            assert (err[:L] <= bound[:L]).all(), (key, c, float((err / bound)[:L].max()))
