"""The two-kernel tensor-core path (KDA_ALGO_SPLIT): every chunk's
state-independent part in one parallel kernel, then the serial state pass.

Parity against the fp64 oracle (max |gpu - ref| / max |ref| <= 1e-2 on the
output and the final state, BF16 inputs), and the slicing contract: a
workspace below the default runs the sequence in more slices, and since the
state crosses a slice boundary in fp32 unchanged, the result is bit-identical
to the one-slice run.
"""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_32_gb300 as pkg
from gated_delta_rule_32_gb300 import kda
from kda_inputs import WORKLOADS, make_inputs, make_unit, small_workload

pytestmark = pytest.mark.gpu

SPLIT = kda.KDA_ALGO_SPLIT
REC = 66048  # bytes of one chunk record


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    kda.load()


def rel(a, b):
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / den) if den > 0 else float(np.abs(a).max())


def min_ws(N, H):
    carry = (N * H * 128 * 128 * 4 + 255) // 256 * 256
    return carry + N * H * REC


def run(x, workspace_bytes=None, final=True, inplace=False, scale=1.0, status=None):
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    B, T, H = x["B"], x["T"], x["H"]
    out = torch.empty_like(d["v"])
    s0 = d["init_state"]
    if inplace:
        fs = s0.clone() if s0 is not None else torch.zeros(B, H, 128, 128, device="cuda")
        s0 = fs
    else:
        fs = torch.empty(B, H, 128, 128, device="cuda") if final else None
    ws, nb = None, 0
    if workspace_bytes is not None:
        nb = workspace_bytes
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], s0, out, fs, B, T, H,
                              128, 128, None, kda.KDA_BF16, 0, scale, SPLIT, ws, nb, status,
                              torch.cuda.current_stream())
    assert rc == 0, kda.status_string(rc)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (fs.cpu().numpy() if fs is not None else None)


def ref(x, scale=1.0):
    return oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"], scale=scale)


@pytest.mark.parametrize("T", [1, 15, 63, 64, 65, 130, 333, 1000])
def test_split_matches_oracle(T):
    w = small_workload("sp", B=2, T=T, H=2, dk=128, dv=128, s0_std=0.03, seed=500 + T)
    x = make_inputs(w)
    o, s = run(x)
    o_ref, s_ref = ref(x)
    assert rel(o, o_ref) <= 1e-2, rel(o, o_ref)
    assert rel(s, s_ref) <= 1e-2, rel(s, s_ref)


def test_split_no_initial_state_and_scale():
    w = small_workload("sp0", B=1, T=450, H=3, dk=128, dv=128, s0_std=0.0, seed=9)
    x = make_inputs(w)
    sc = 128 ** -0.5
    o, s = run(x, scale=sc)
    o_ref, s_ref = ref(x, scale=sc)
    assert rel(o, o_ref) <= 1e-2
    assert rel(s, s_ref) <= 1e-2


@pytest.mark.parametrize("case", ["all_floor", "alpha_one", "beta_zero", "beta_one"])
def test_split_degenerate_gates(case):
    w = small_workload("spd", B=1, T=200, H=2, dk=128, dv=128, s0_std=0.05, seed=31)
    x = make_inputs(w)
    if case == "all_floor":
        x["g"] = torch.full_like(x["g"], 30.0)
    elif case == "alpha_one":
        x["g"] = torch.full_like(x["g"], -200.0)
    elif case == "beta_zero":
        x["beta"] = torch.zeros_like(x["beta"])
        x["g"] = torch.full_like(x["g"], -4.0)
    else:
        x["beta"] = torch.ones_like(x["beta"])
    o, s = run(x)
    o_ref, s_ref = ref(x)
    assert rel(o, o_ref) <= 1e-2
    assert rel(s, s_ref) <= 1e-2


@pytest.mark.parametrize("extra_chunks", [0, 1, 3])
def test_slices_bit_identical(extra_chunks):
    # 11 chunks with a ragged tail; slices of 1 chunk (room for 1 per chain:
    # one slice after another) and, with room for 2 or 4 chunks, slices of 1
    # and 2 chunks on the overlapped schedule (4 chains leave most SMs idle:
    # the next slice's intra kernel runs beside the current state pass, the
    # records alternating between the two halves of the buffer)
    w = small_workload("sl", B=2, T=690, H=2, dk=128, dv=128, s0_std=0.05, seed=21)
    x = make_inputs(w)
    o1, s1 = run(x)
    ws = min_ws(2, 2) + extra_chunks * 2 * 2 * REC
    o2, s2 = run(x, workspace_bytes=ws)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)
    # without a final state the carry lives in the workspace
    o3, s3 = run(x, workspace_bytes=ws, final=False)
    assert s3 is None
    np.testing.assert_array_equal(o1, o3)
    # state updated in place (init_state aliased with final_state)
    o4, s4 = run(x, workspace_bytes=ws, inplace=True)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(s1, s4)


def test_workspace_too_small_is_refused():
    w = small_workload("wsr", B=1, T=128, H=2, dk=128, dv=128, seed=2)
    x = make_inputs(w)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    out = torch.empty_like(d["v"])
    nb = min_ws(1, 2) - 256
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], None, out, None, 1, 128,
                              2, 128, 128, None, kda.KDA_BF16, 0, 1.0, SPLIT, ws, nb, None,
                              torch.cuda.current_stream())
    assert rc == kda.KDA_ERR_WORKSPACE
    # (a packed batch needs at least one chunk column of records:
    # test_split_packed_workspace_below_one_column_is_refused)
    assert kda.kda_resolve_algo(kda.KDA_BF16, 128, 128, 0, SPLIT) == SPLIT
    assert kda.kda_resolve_algo(kda.KDA_F32, 128, 128, 0, SPLIT) == -1
    assert kda.kda_workspace_bytes(2, 32768, 32, 128, 128, algo=SPLIT) >= min_ws(2, 32)


def test_split_deterministic_and_close_to_fused():
    w = small_workload("spf", B=2, T=777, H=3, dk=128, dv=128, s0_std=0.02, seed=8)
    x = make_inputs(w)
    a = run(x)
    b = run(x)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    of, sf = pkg.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                         algo=kda.KDA_ALGO_TC)
    torch.cuda.synchronize()
    # two approximations of the same forward, each within 1e-2 of the oracle
    # (the paths round U at different points): within 2e-2 of each other
    assert rel(a[0], of.float().cpu().numpy()) <= 2e-2
    assert rel(a[1], sf.cpu().numpy()) <= 2e-2


def test_full_b2_h32_t32k_split_sampled():
    # the benchmark's workload at full size; sampled (sequence, head) units
    w = WORKLOADS["b2_h32_t32k"]
    x = make_inputs(w)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    out, fs = pkg.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                          algo=SPLIT)
    torch.cuda.synchronize()
    o, s = out.float().cpu().numpy(), fs.cpu().numpy()
    for (b, h) in [(0, 0), (1, 31), (0, 17)]:
        u = make_unit(w, b, h)
        args = [u[key].to(w.dtype)[None, :, None] for key in ("q", "k", "v", "g")]
        bt = u["beta"].to(w.dtype)[None, :, None]
        s0 = u["s0"][:, None] if w.s0_std > 0 else None
        o_ref, s_ref = oracle.fwd(*args, bt, s0)
        eo, es = rel(o[b, :, h], o_ref[0, :, 0]), rel(s[b, h], s_ref[0, 0])
        assert eo <= 1e-2 and es <= 1e-2, (b, h, eo, es)


# ---- the end-to-end entry: pieces copied in, run and copied out in turn ----

@pytest.mark.parametrize("T,s0_std,final", [(1000, 0.02, True), (640, 0.0, True),
                                            (333, 0.02, False), (65, 0.0, True)])
def test_host_pipeline_matches_device(T, s0_std, final):
    """kda_chunk_fwd_host runs the two-kernel path in pieces of whole chunks
    (inputs of the next piece copied in while the current one runs): the
    result is bit-identical to the one-call device run."""
    w = small_workload("hostpipe", B=2, T=T, H=3, dk=128, dv=128, s0_std=s0_std, seed=31)
    x = make_inputs(w)
    o_dev, s_dev = run(x, final=final)
    pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()}
    out = torch.empty(2, T, 3, 128, dtype=torch.bfloat16).pin_memory()
    fs = torch.empty(2, 3, 128, 128).pin_memory() if final else None
    nb = kda.kda_host_staging_bytes(2, T, 3, 128, 128, kda.KDA_BF16,
                                    int(x["init_state"] is not None), int(final), 0)
    staging = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rc = kda.kda_chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"],
                                pin["init_state"], out, fs, 2, T, 3, 128, 128, None,
                                kda.KDA_BF16, 1.0, staging, nb, torch.cuda.current_stream())
    assert rc == 0, kda.status_string(rc)
    np.testing.assert_array_equal(out.float().numpy(), o_dev)
    if final:
        np.testing.assert_array_equal(fs.numpy(), s_dev)
    o_ref, s_ref = ref(x)
    assert rel(out.float().numpy(), o_ref) <= 1e-2


# ---- packed batches (cu_seqlens): chunk columns of every sequence at once --

def run_packed(x, algo=SPLIT, status=None, workspace=True, ws_bytes=None, final=True,
               inplace=False):
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    N = d["cu_seqlens"].numel() - 1
    T, H = x["T"], x["H"]
    out = torch.empty_like(d["v"])
    s0 = d["init_state"]
    fs = torch.empty(N, H, 128, 128, device="cuda") if final else None
    if inplace:
        fs = s0.clone()
        s0 = fs
    ws, nb = None, 0
    if workspace:
        nb = ws_bytes or kda.kda_workspace_bytes(N, T, H, 128, 128, algo=algo, packed=1)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], s0, out,
                              fs, N, T, H, 128, 128, d["cu_seqlens"], kda.KDA_BF16, 0, 1.0, algo,
                              ws, nb, status, torch.cuda.current_stream())
    assert rc == 0, kda.status_string(rc)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (fs.cpu().numpy() if fs is not None else None)


def packed_min_ws(N, T, H):
    # [carry][chunk offsets][sequence order][chunk table][records of one chunk column]
    def r256(v):
        return (v + 255) // 256 * 256
    g_max = (T + 63) // 64 + N
    return (r256(N * H * 128 * 128 * 4) + r256((N + 1) * 4) + r256(N * 4) + r256(g_max * 8) +
            H * REC)


@pytest.mark.parametrize("extra_cols", [0, 2, 5])
def test_split_packed_slices_bit_identical(extra_cols):
    """A packed batch in slices of 1, 3 and 6 chunk columns (the workspace
    holds that many columns of records): sequences that span slices carry
    their state across them, empty and one-token sequences pass through;
    bit-identical to the one-slice run, with and without a final state and
    with the state updated in place."""
    lens = (130, 0, 1, 300, 64, 0, 65, 17)
    w = small_workload("pks", B=1, T=sum(lens), H=2, dk=128, dv=128, seed=43, varlen=True,
                       lengths=lens, s0_std=0.03)
    x = make_inputs(w)
    o1, s1 = run_packed(x)
    N, T, H = len(lens), sum(lens), 2
    nb = packed_min_ws(N, T, H) + extra_cols * H * REC
    o2, s2 = run_packed(x, ws_bytes=nb)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)
    o3, s3 = run_packed(x, ws_bytes=nb, final=False)
    assert s3 is None
    np.testing.assert_array_equal(o1, o3)
    o4, s4 = run_packed(x, ws_bytes=nb, inplace=True)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(s1, s4)
    o_ref, s_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"],
                              x["cu_seqlens"])
    assert rel(o2, o_ref) <= 1e-2 and rel(s2, s_ref) <= 1e-2


@pytest.mark.parametrize("lens,s0_std,final", [
    ((130, 0, 1, 300, 64, 0, 65, 17), 0.03, True),   # 18 column bound: 6 pieces of 3
    ((1000,), 0.0, True),                            # one sequence across every piece
    ((5, 7, 0, 3, 1, 2), 0.02, False),               # one column per piece, the last empty
])
def test_host_pipeline_packed_matches_device(lens, s0_std, final):
    """kda_chunk_fwd_host on a packed batch runs the two-kernel path in
    pieces of chunk columns (contiguous token rows, copied in while the
    previous piece runs, each copy reaching 64 rows past its piece for the
    tile of a short last chunk): bit-identical to the one-call device run."""
    N, T, H = len(lens), sum(lens), 2
    w = small_workload("hostpk", B=1, T=T, H=H, dk=128, dv=128, seed=47, varlen=True,
                       lengths=lens, s0_std=s0_std)
    x = make_inputs(w)
    o_dev, s_dev = run_packed(x, final=final)
    pin = {k: (v.pin_memory() if torch.is_tensor(v) and k != "cu_seqlens" else v)
           for k, v in x.items()}
    out = torch.empty(1, T, H, 128, dtype=torch.bfloat16).pin_memory()
    fs = torch.empty(N, H, 128, 128).pin_memory() if final else None
    nb = kda.kda_host_staging_bytes(N, T, H, 128, 128, kda.KDA_BF16,
                                    int(x["init_state"] is not None), int(final), 1)
    staging = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rc = kda.kda_chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"],
                                pin["init_state"], out, fs, N, T, H, 128, 128,
                                x["cu_seqlens"], kda.KDA_BF16, 1.0, staging, nb,
                                torch.cuda.current_stream())
    assert rc == 0, kda.status_string(rc)
    np.testing.assert_array_equal(out.float().numpy(), o_dev)
    if final:
        np.testing.assert_array_equal(fs.numpy(), s_dev)


def test_split_packed_many_short_sequences():
    """9 000 sequences of 0 to 3 tokens (more than the 8 192 the state CTAs are
    ordered for, so they run in their own order): every chunk column holds a
    whole short sequence, empty sequences pass their state through."""
    rng = np.random.default_rng(5)
    lens = tuple(int(v) for v in rng.integers(0, 4, size=9000))
    w = small_workload("pkmany", B=1, T=sum(lens), H=1, dk=128, dv=128, seed=46, varlen=True,
                       lengths=lens, s0_std=0.03)
    x = make_inputs(w)
    o, s = run_packed(x)
    o_ref, s_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"],
                              x["cu_seqlens"])
    assert rel(o, o_ref) <= 1e-2 and rel(s, s_ref) <= 1e-2


def test_split_packed_workspace_below_one_column_is_refused():
    lens = (100, 28)
    w = small_workload("pkr", B=1, T=sum(lens), H=2, dk=128, dv=128, seed=44, varlen=True,
                       lengths=lens)
    x = make_inputs(w)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    nb = packed_min_ws(2, sum(lens), 2) - 256
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], None,
                              torch.empty_like(d["v"]), None, 2, sum(lens), 2, 128, 128,
                              d["cu_seqlens"], kda.KDA_BF16, 0, 1.0, SPLIT, ws, nb, None,
                              torch.cuda.current_stream())
    assert rc == kda.KDA_ERR_WORKSPACE


@pytest.mark.parametrize("lens,s0_std", [((100, 64, 0, 1, 257, 130), 0.02),
                                         ((640, 5, 63, 1000), 0.0),
                                         ((1,), 0.03),
                                         ((65, 0, 0, 128), 0.02)])
def test_split_packed_matches_oracle(lens, s0_std):
    """Sequences of every kind of length (empty, one token, partial and
    whole chunks) packed in one batch: parity with the oracle, and agreement
    with the fused kernel.  The two paths round U at different points (T
    Diag(beta) times V here, T times bf16(beta V) there), so they are
    compared by the triangle bound: each within 1e-2 of the oracle, so within
    2e-2 of each other."""
    w = small_workload("pk", B=1, T=sum(lens), H=3, dk=128, dv=128, seed=41, varlen=True,
                       lengths=lens, s0_std=s0_std)
    x = make_inputs(w)
    o, s = run_packed(x)
    o_ref, s_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"],
                              x["cu_seqlens"])
    assert rel(o, o_ref) <= 1e-2
    assert rel(s, s_ref) <= 1e-2
    o2, s2 = run_packed(x)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(s, s2)
    of, sf = run_packed(x, algo=kda.KDA_ALGO_TC, workspace=False)
    assert rel(o, of) <= 2e-2 and rel(s, sf) <= 2e-2


def test_split_packed_bad_seqlens_reported():
    lens = (100, 60, 96)
    w = small_workload("pkb", B=1, T=256, H=2, dk=128, dv=128, seed=5, varlen=True,
                       lengths=lens)
    x = make_inputs(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x["cu_seqlens"] = torch.tensor([0, 100, 60, 256], dtype=torch.int32)  # not monotone
    run_packed(x, status=status)
    assert int(status.item()) == kda.KDA_ERR_BAD_SEQLENS
    status.zero_()
    x["cu_seqlens"] = torch.tensor([0, 100, 160, 250], dtype=torch.int32)  # ends before T
    run_packed(x, status=status)
    assert int(status.item()) == kda.KDA_ERR_BAD_SEQLENS


def test_split_packed_checkpoints():
    """Checkpoints of a packed batch on the two-kernel path equal the states
    the oracle reaches at those positions of each sequence."""
    lens = (200, 384, 64)
    w = small_workload("pkc", B=1, T=sum(lens), H=2, dk=128, dv=128, seed=17, varlen=True,
                       lengths=lens, s0_std=0.02)
    x = make_inputs(w)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    N, T, H = 3, sum(lens), 2
    out = torch.empty_like(d["v"])
    fs = torch.empty(N, H, 128, 128, device="cuda")
    ck = torch.full((N, H, 6, 128, 128), float("nan"), device="cuda")
    assert kda.kda_resolve_path(N, T, H, packed=True) == SPLIT
    rc = kda.kda_chunk_fwd_ckpt(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], out,
                                fs, N, T, H, 128, 128, d["cu_seqlens"], kda.KDA_BF16, 1.0, ck,
                                128, 6, None, torch.cuda.current_stream())
    assert rc == 0, kda.status_string(rc)
    torch.cuda.synchronize()
    ck = ck.cpu().numpy()
    cu = x["cu_seqlens"].tolist()
    for n in range(N):
        for slot in range(6):
            pos = 128 * (slot + 1)
            if pos > lens[n]:
                assert np.isnan(ck[n, :, slot]).all()
                continue
            sl = slice(cu[n], cu[n] + pos)
            s0 = x["init_state"][n:n + 1]
            _, s_ref = oracle.fwd(x["q"][:, sl], x["k"][:, sl], x["v"][:, sl], x["g"][:, sl],
                                  x["beta"][:, sl], s0)
            assert rel(ck[n, :, slot], s_ref[0]) <= 1e-2, (n, slot)


def test_split_packed_first_call_in_a_process(tmp_path):
    """A packed batch as the first two-kernel call of a process (nothing
    before it has prepared the kernels' shared-memory limits)."""
    import subprocess
    import sys
    import os
    code = (
        "import torch, numpy as np\n"
        "from kda_inputs import small_workload, make_inputs\n"
        "import gated_delta_rule_32_gb300 as pkg\n"
        "from gated_delta_rule_32_gb300 import kda\n"
        "kda.load()\n"
        "w = small_workload('pk1', B=1, T=300, H=2, dk=128, dv=128, seed=3, varlen=True,"
        " lengths=(100, 200))\n"
        "x = make_inputs(w, device='cuda')\n"
        "assert kda.kda_resolve_path(2, 300, 2, packed=True) == kda.KDA_ALGO_SPLIT\n"
        "o, s = pkg.forward(x['q'], x['k'], x['v'], x['g'], x['beta'], None, x['cu_seqlens'])\n"
        "torch.cuda.synchronize()\n"
        "assert np.isfinite(o.float().cpu().numpy()).all()\n"
        "print('ok')\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stderr[-2000:]
