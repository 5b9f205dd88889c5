"""Step-level parity of the two-kernel path's intra-chunk kernel.

The intra kernel writes one record per (sequence, head, chunk): (K dec)^T,
A_qk (masked), [W; Q gamma], T Diag(beta) (all bf16, in the state kernel's
shared-memory operand layouts) and gamma_C (fp32).  This test runs that
kernel alone (kda_split_stage stage 1), decodes the records from the
workspace and compares every piece with the fp64 chunk mirror of the
oracle:
  - elementwise products of the bf16 inputs with decay factors (K dec, Q
    gamma) and gamma_C: relative error per element within 2^-7 (bf16
    rounding of the result, 2^-9, plus the decay factors' own error);
  - A_qk and T Diag(beta): within 1e-2 of their largest entry;
  - W = T (beta K gamma): the elementwise bound derived in
    tests/test_tc_steps_gpu.py (bf16 operands, Gram errors through the
    inverse).
"""
import numpy as np
import pytest
import torch

from oracle import chunk_mirror
from gated_delta_rule_32_gb300 import kda
from kda_inputs import make_inputs, small_workload

pytestmark = pytest.mark.gpu

REC = 66048
U = 2.0 ** -9


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    kda.load()


def k64_off(mn, k):
    return (mn >> 3) * 1024 + (k >> 3) * 128 + (mn & 7) * 16 + (k & 7) * 2


def mn_off(mn, k, lbo):
    return (mn >> 3) * 128 + (k >> 3) * lbo + (k & 7) * 16 + (mn & 7) * 2


def _bf16_at(raw, base, offs):
    """bf16 values at byte offsets `offs` (any shape) after `base`."""
    idx = (base + offs) // 2
    u16 = raw.view(np.uint16)[idx]
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


J, R = np.meshgrid(np.arange(128), np.arange(64), indexing="ij")        # [128][64]
R2, I2 = np.meshgrid(np.arange(64), np.arange(64), indexing="ij")      # [64][64]
M, K = np.meshgrid(np.arange(128), np.arange(128), indexing="ij")      # [128][128]
OFF_KD = k64_off(J, R)          # (K dec)^T [j][r]
OFF_AQ = 16384 + k64_off(R2, I2)
OFF_WQ = 24576 + mn_off(M, K, 2048)
OFF_T = 57344 + k64_off(R2, I2)


@pytest.mark.parametrize("gmode", ["normal", "floor_heavy", "alpha_one"])
def test_intra_kernel_records(gmode):
    B, T, H = 2, 150, 2                       # 3 chunks, the last ragged (22 rows)
    w = small_workload("rec", B=B, T=T, H=H, dk=128, dv=128, seed=81)
    x = make_inputs(w)
    if gmode == "floor_heavy":
        x["g"] = (torch.randn(x["g"].shape, generator=torch.Generator().manual_seed(2)) + 6.0
                  ).to(torch.bfloat16)
    elif gmode == "alpha_one":
        x["g"] = torch.full_like(x["g"], -200.0)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    nch = (T + 63) // 64
    nb = kda.kda_workspace_bytes(B, T, H, 128, 128, kda.KDA_BF16, 0, kda.KDA_ALGO_SPLIT, 0)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["v"])
    rc = kda.kda_split_stage(1, d["q"], d["k"], d["v"], d["g"], d["beta"], None, out, None, B,
                             T, H, 1.0, ws, nb, None, torch.cuda.current_stream())
    assert rc == 0, kda.status_string(rc)
    torch.cuda.synchronize()
    raw = ws.cpu().numpy()
    carry = (B * H * 128 * 128 * 4 + 255) // 256 * 256
    f64 = lambda t, n, h: t[n, :, h].double().numpy()
    for n in range(B):
        for h in range(H):
            q, k, v, g, beta = (f64(x[key], n, h) for key in ("q", "k", "v", "g", "beta"))
            _, _, steps = chunk_mirror.forward_unit(q, k, v, g, beta, None, chunk=64,
                                                    return_steps=True)
            for c, st in enumerate(steps):
                L = min(64, T - 64 * c)
                base = carry + ((n * H + h) * nch + c) * REC
                kc = np.zeros((64, 128)); kc[:L] = k[64 * c:64 * c + L]
                qc = np.zeros((64, 128)); qc[:L] = q[64 * c:64 * c + L]
                bc = np.zeros(64); bc[:L] = beta[64 * c:64 * c + L]
                G = st["Gam"]
                gam = np.exp(G)
                # gamma_C: the decay of the whole chunk (last valid row)
                gc = raw[base + 65536:base + 65536 + 512].view(np.float32).astype(np.float64)
                np.testing.assert_allclose(gc, gam[L - 1], rtol=2 ** -7, atol=1e-30)
                # (K dec)^T and Q gamma, elementwise
                kd = _bf16_at(raw, base, OFF_KD).T                        # [r][j]
                kd_ref = kc * np.exp(G[L - 1] - G)
                assert (np.abs(kd - kd_ref) <= 2 ** -7 * np.abs(kd_ref) + 1e-30).all(), c
                wq = _bf16_at(raw, base, OFF_WQ)                          # [row][j]
                qg_ref = qc * gam
                assert (np.abs(wq[64:] - qg_ref) <= 2 ** -7 * np.abs(qg_ref) + 1e-30).all(), c
                # A_qk (masked) and T Diag(beta)
                aq = _bf16_at(raw, base, OFF_AQ)
                aq_ref = st["Aqk"]
                assert np.abs(aq - aq_ref)[:L, :L].max() <= 1e-2 * np.abs(aq_ref).max(), c
                tb = _bf16_at(raw, base, OFF_T)
                tb_ref = st["T"] * bc[None, :]
                assert np.abs(tb - tb_ref)[:L, :L].max() <= 1e-2 * np.abs(tb_ref).max(), c
                # W (rows 0..63 of [W; Q gamma]) against the derived bound
                absT = np.abs(st["T"])
                dec = np.exp(np.minimum(G[:, None, :] - G[None, :, :], 0.0))
                absA = np.tril(bc[:, None] * np.einsum("rj,ij,rij->ri", np.abs(kc),
                                                        np.abs(kc), dec), -1)
                dT = 2 * U * absT @ absA @ absT + U * absT
                aX = np.abs(bc[:, None] * kc * gam)
                bound = 2 * (2 * U * absT @ aX + dT @ aX) + 1e-6 * np.abs(st["W"]).max()
                err = np.abs(wq[:64] - st["W"])
                assert (err[:L] <= bound[:L]).all(), (c, float((err / bound)[:L].max()))
