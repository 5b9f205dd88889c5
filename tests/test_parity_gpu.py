"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Metric (per tensor): max |gpu - ref| / max |ref|, on the output and on the
final state separately.  Bounds: 1e-2 for BF16 inputs, 1e-4 for fp32.
"""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_32_gb300 as pkg
from gated_delta_rule_32_gb300 import kda
from kda_inputs import WORKLOADS, make_inputs, make_unit, small_workload

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 1e-2, torch.float32: 1e-4}
# AUTO: the two-kernel tensor-core path on dense batches, the fused kernel on
# packed ones; TC: the fused kernel on both
ALGOS = [kda.KDA_ALGO_SIMT, kda.KDA_ALGO_AUTO, kda.KDA_ALGO_TC]


def rel(a, ref):
    den = np.abs(ref).max()
    if den == 0:
        return float(np.abs(a).max())
    return float(np.abs(a - ref).max() / den)


def to_dev(x):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}


def gpu_fwd(x, algo=kda.KDA_ALGO_AUTO, scale=1.0, chunk_size=0, status=None):
    d = to_dev(x)
    out, fs = pkg.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                          d["cu_seqlens"], scale=scale, algo=algo, chunk_size=chunk_size,
                          dev_status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fs.cpu().numpy()


def ref_fwd(x, scale=1.0):
    return oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"],
                      x["cu_seqlens"], scale=scale)


def check(x, dtype, algo=kda.KDA_ALGO_AUTO, scale=1.0):
    o, s = gpu_fwd(x, algo, scale)
    o_ref, s_ref = ref_fwd(x, scale)
    eo, es = rel(o, o_ref), rel(s, s_ref)
    assert eo <= TOL[dtype] and es <= TOL[dtype], (eo, es)
    return eo, es


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    kda.load()


def test_tiny_fp32_workload():
    w = WORKLOADS["tiny_fp32"]
    x = make_inputs(w)
    check(x, torch.float32)


@pytest.mark.parametrize("algo", ALGOS)
def test_h4_t4k_workload(algo):
    w = WORKLOADS["h4_t4k"]
    x = make_inputs(w)
    check(x, torch.bfloat16, algo)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 32), (128, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 15, 17, 64, 130])
def test_small_shapes(dtype, dk, dv, T):
    w = small_workload("s", B=2, T=T, H=3, dk=dk, dv=dv, dtype=dtype, s0_std=0.05, seed=T + dk)
    check(make_inputs(w), dtype, kda.KDA_ALGO_SIMT)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("T", [1, 15, 17, 63, 64, 65, 130, 333])
def test_ragged_d128_bf16(algo, T):
    w = small_workload("r", B=2, T=T, H=2, dk=128, dv=128, s0_std=0.02, seed=100 + T)
    check(make_inputs(w), torch.bfloat16, algo)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_varlen_edge_lengths(algo, dtype):
    if dtype == torch.float32 and algo == kda.KDA_ALGO_TC:
        pytest.skip("the fused tensor-core kernel takes bf16 inputs")
    lens = (1, 15, 16, 17, 63, 64, 65, 130)
    w = small_workload("v", B=1, T=sum(lens), H=2, dk=128, dv=128, dtype=dtype, seed=9,
                       varlen=True, lengths=lens, s0_std=0.03)
    check(make_inputs(w), dtype, algo)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("case", ["all_floor", "alpha_one", "beta_zero", "beta_one"])
def test_degenerate_gates(algo, case):
    w = small_workload("d", B=1, T=200, H=2, dk=128, dv=128, s0_std=0.05, seed=31)
    x = make_inputs(w)
    if case == "all_floor":
        x["g"] = torch.full_like(x["g"], 30.0)
    elif case == "alpha_one":
        x["g"] = torch.full_like(x["g"], -200.0)
    elif case == "beta_zero":
        # beta = 0 leaves only the decay of S0; keep it mild so the exact
        # final state stays far above fp32 underflow
        x["beta"] = torch.zeros_like(x["beta"])
        x["g"] = torch.full_like(x["g"], -4.0)
    else:
        x["beta"] = torch.ones_like(x["beta"])
    check(x, torch.bfloat16, algo)


def test_retrieval_identity_on_gpu():
    # beta = 1 and q = k (unit): o_t = v_t exactly, whatever the history
    w = small_workload("p1", B=1, T=256, H=2, dk=128, dv=128, s0_std=0.05, seed=41)
    x = make_inputs(w)
    x["beta"] = torch.ones_like(x["beta"])
    x["q"] = x["k"].clone()
    o, _ = gpu_fwd(x)
    assert rel(o, x["v"].float().numpy()) <= 1e-2


@pytest.mark.parametrize("algo", ALGOS)
def test_scale(algo):
    w = small_workload("sc", B=1, T=100, H=2, dk=128, dv=128, seed=5)
    check(make_inputs(w), torch.bfloat16, algo, scale=128 ** -0.5)


def test_inplace_state_and_split():
    # init_state aliased with final_state, and a run split in two equals one run
    w = small_workload("ip", B=1, T=300, H=2, dk=128, dv=128, s0_std=0.05, seed=77)
    x = make_inputs(w)
    d = to_dev(x)
    full_o, full_s = pkg.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"])
    st = d["init_state"].clone()
    outs = []
    for t0, t1 in ((0, 77), (77, 300)):
        sl = {k: d[k][:, t0:t1].contiguous() for k in ("q", "k", "v", "g", "beta")}
        out = torch.empty_like(sl["v"])
        rc = kda.kda_chunk_fwd(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], st, out, st,
                               1, t1 - t0, 2, 128, 128, None, torch.cuda.current_stream())
        assert rc == 0
        outs.append(out)
    torch.cuda.synchronize()
    o = torch.cat(outs, 1).float().cpu().numpy()
    assert rel(o, full_o.float().cpu().numpy()) <= 1e-2
    assert rel(st.cpu().numpy(), full_s.cpu().numpy()) <= 1e-2


def test_empty_sequence_passes_state_through():
    w = small_workload("e", B=2, T=0, H=2, dk=64, dv=64, s0_std=0.1, seed=3)
    x = make_inputs(w)
    _, s = gpu_fwd(x)
    np.testing.assert_array_equal(s, x["init_state"].numpy())


def test_bad_seqlens_reported_on_device():
    lens = (10, 20, 30)
    w = small_workload("b", B=1, T=60, H=1, dk=64, dv=64, seed=1, varlen=True, lengths=lens)
    x = make_inputs(w)
    x["cu_seqlens"] = torch.tensor([0, 20, 10, 60], dtype=torch.int32)   # not monotone
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_fwd(x, status=status)
    assert int(status.item()) == kda.KDA_ERR_BAD_SEQLENS
    x["cu_seqlens"] = torch.tensor([0, 20, 40, 50], dtype=torch.int32)   # ends before T
    status.zero_()
    gpu_fwd(x, status=status)
    assert int(status.item()) == kda.KDA_ERR_BAD_SEQLENS


@pytest.mark.parametrize("algo", ALGOS)
def test_deterministic(algo):
    w = small_workload("det", B=2, T=500, H=4, dk=128, dv=128, s0_std=0.02, seed=8)
    x = make_inputs(w)
    a = gpu_fwd(x, algo)
    b = gpu_fwd(x, algo)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_host_buffer_entry():
    w = small_workload("host", B=2, T=190, H=2, dk=128, dv=128, s0_std=0.02, seed=12)
    x = make_inputs(w)
    pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()}
    out = torch.empty(2, 190, 2, 128, dtype=torch.bfloat16).pin_memory()
    fs = torch.empty(2, 2, 128, 128).pin_memory()
    rc = kda.kda_chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"],
                                pin["init_state"], out, fs, 2, 190, 2, 128, 128, None,
                                kda.KDA_BF16, 1.0, None, 0, torch.cuda.current_stream())
    assert rc == 0
    o_ref, s_ref = ref_fwd(x)
    assert rel(out.float().numpy(), o_ref) <= 1e-2
    assert rel(fs.numpy(), s_ref) <= 1e-2


# ---- full-size workloads: sampled (sequence, head) units -------------------

def _sampled_check(name, units, algo=kda.KDA_ALGO_AUTO):
    w = WORKLOADS[name]
    x = make_inputs(w)
    o, s = gpu_fwd(x, algo)
    cu = x["cu_seqlens"]
    worst = (0.0, 0.0)
    for (b, h) in units:
        u = make_unit(w, b, h)
        args = [u[key].to(w.dtype)[None, :, None] for key in ("q", "k", "v", "g")]
        bt = u["beta"].to(w.dtype)[None, :, None]
        if w.varlen:
            s0 = u["s0"][:, None] if w.s0_std > 0 else None
            o_ref, s_ref = oracle.fwd(*args[:3], args[3], bt, s0, cu)
            o_gpu = o[0, :, h]
            s_gpu = s[:, h]
        else:
            s0 = u["s0"][:, None] if w.s0_std > 0 else None
            o_ref, s_ref = oracle.fwd(*args[:3], args[3], bt, s0)
            o_gpu = o[b, :, h]
            s_gpu = s[b, h]
        eo = rel(o_gpu, o_ref[0, :, 0])
        es = rel(s_gpu, s_ref[:, 0] if w.varlen else s_ref[0, 0])
        worst = (max(worst[0], eo), max(worst[1], es))
        assert eo <= 1e-2 and es <= 1e-2, (b, h, eo, es)
    return worst


def test_full_b2_h32_t32k_sampled():
    # the fused kernel at full size (the automatic path's two-kernel form is
    # checked at full size in test_split_gpu.py)
    _sampled_check("b2_h32_t32k", [(0, 0), (1, 31), (0, 17), (1, 5)], algo=kda.KDA_ALGO_TC)


def test_full_varlen_floor_sampled():
    _sampled_check("varlen_floor", [(0, 0), (0, 7), (0, 15)])


def test_full_varlen_floor_hard_sampled():
    _sampled_check("varlen_floor_hard", [(0, 3)])


def test_full_ctx1m_sampled():
    _sampled_check("ctx1m", [(0, 0), (0, 11)])


def test_full_varlen_ctx1m_sampled():
    # 1M tokens packed in 28 sequences: the default workspace holds every
    # chunk column's records (one slice); with 4 GiB of records the same
    # call runs in slices of chunk columns, sequences carrying their state
    # across them, and must give the same bits
    w = WORKLOADS["varlen_ctx1m"]
    N, T, H = w.n_seqs(), w.T, w.H
    assert kda.kda_resolve_path(N, T, H, packed=True) == kda.KDA_ALGO_SPLIT
    g_max = T // 64 + N
    full = kda.kda_workspace_bytes(N, T, H, 128, 128, packed=1)
    assert full >= g_max * H * 66048
    _sampled_check("varlen_ctx1m", [(0, 9)])
    x = make_inputs(w)
    d = to_dev(x)

    def run(nb):
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        out = torch.empty_like(d["v"])
        fs = torch.empty(N, H, 128, 128, device="cuda")
        rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                  out, fs, N, T, H, 128, 128, d["cu_seqlens"], kda.KDA_BF16, 0,
                                  1.0, kda.KDA_ALGO_SPLIT, ws, nb, None,
                                  torch.cuda.current_stream())
        assert rc == 0, kda.status_string(rc)
        del ws
        return out, fs
    o1, s1 = run(full)
    cols = (4 << 30) // (H * 66048)
    assert cols < g_max
    o2, s2 = run(full - (g_max - cols) * H * 66048)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
