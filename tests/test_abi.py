"""The C-ABI library: builds, loads, exports every declared symbol, and
rejects bad host-visible arguments before touching the GPU.  CPU only."""
import ctypes

import pytest

import gated_delta_rule_32_gb300 as pkg
from gated_delta_rule_32_gb300 import kda


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_32_gb300 import build
    build.build()
    return kda.load()


def test_exports_every_declared_symbol(lib):
    names = kda.header_functions()
    assert len(names) >= 9
    raw = ctypes.CDLL(kda.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(lib):
    for code in range(9):
        s = kda.status_string(code)
        assert s.startswith("KDA_")
    assert kda.status_string(99) == "KDA_ERR_UNKNOWN"
    assert "sm_103a" in kda.kda_build_info()


A = 1 << 20   # fake, 16-byte aligned addresses: never dereferenced on the host


def _call(**over):
    args = dict(q=A, k=2 * A, v=3 * A, g_logit=4 * A, beta=5 * A, init_state=None,
                out=6 * A, final_state=None, B=1, T=64, H=1, dk=128, dv=128)
    args.update(over)
    return kda.kda_chunk_fwd_ex(**args)


def test_rejects_null_pointers(lib):
    for name in ("q", "k", "v", "g_logit", "beta", "out"):
        assert _call(**{name: None}) == kda.KDA_ERR_INVALID_ARG


def test_rejects_sizes(lib):
    assert _call(B=0) == kda.KDA_ERR_INVALID_ARG
    assert _call(H=0) == kda.KDA_ERR_INVALID_ARG
    assert _call(T=-1) == kda.KDA_ERR_INVALID_ARG
    assert _call(dk=48) == kda.KDA_ERR_UNSUPPORTED
    assert _call(dv=256) == kda.KDA_ERR_UNSUPPORTED
    assert _call(chunk_size=32) == kda.KDA_ERR_UNSUPPORTED
    assert _call(dtype=7) == kda.KDA_ERR_UNSUPPORTED
    assert _call(algo=9) == kda.KDA_ERR_INVALID_ARG


def test_rejects_misaligned(lib):
    assert _call(q=A + 8) == kda.KDA_ERR_MISALIGNED
    assert _call(out=6 * A + 2) == kda.KDA_ERR_MISALIGNED
    assert _call(beta=5 * A + 1) == kda.KDA_ERR_MISALIGNED
    assert _call(init_state=7 * A + 4) == kda.KDA_ERR_MISALIGNED


def test_rejects_aliasing(lib):
    assert _call(out=A) == kda.KDA_ERR_INVALID_ARG          # out == q
    assert _call(out=3 * A + 64) == kda.KDA_ERR_INVALID_ARG  # out overlaps v
    assert _call(final_state=2 * A) == kda.KDA_ERR_INVALID_ARG


def test_host_entry_rejects_bad_seqlens(lib):
    import numpy as np
    cu = np.array([0, 10, 5, 64], dtype=np.int32)      # decreasing
    rc = kda.kda_chunk_fwd_host(A, 2 * A, 3 * A, 4 * A, 5 * A, None, 6 * A, None, 3, 64, 1,
                                128, 128, cu.ctypes.data)
    assert rc == kda.KDA_ERR_BAD_SEQLENS
    cu = np.array([0, 10, 60], dtype=np.int32)          # does not end at T
    rc = kda.kda_chunk_fwd_host(A, 2 * A, 3 * A, 4 * A, 5 * A, None, 6 * A, None, 2, 64, 1,
                                128, 128, cu.ctypes.data)
    assert rc == kda.KDA_ERR_BAD_SEQLENS


def test_staging_bytes(lib):
    n = kda.kda_host_staging_bytes(2, 100, 3, 128, 64, kda.KDA_BF16, 1, 1, 0)
    qk = 2 * 100 * 3 * 128 * 2
    assert n >= 3 * qk + 2 * 2 * 100 * 3 * 64 * 2 + 2 * 2 * 3 * 128 * 64 * 4


def test_staging_bytes_of_the_pipelined_host_call(lib):
    # dense bf16 at dk = dv = 128 runs the end-to-end call in up to eight
    # pieces of whole chunks: the staging holds the inputs, outputs and
    # states plus the chunk records of one piece (64 of the 512 chunks here)
    def r256(x):
        return (x + 255) // 256 * 256
    B, T, H = 2, 32768, 32
    qk = B * T * H * 128 * 2
    state = B * H * 128 * 128 * 4
    fixed = 3 * r256(qk) + 2 * r256(qk) + r256(B * T * H * 2) + 2 * r256(state) + 256
    piece = r256(state) + B * H * 66048 * 64
    n = kda.kda_host_staging_bytes(B, T, H, 128, 128, kda.KDA_BF16, 1, 1, 0)
    assert n == fixed + r256(piece)
    # a single chunk is not cut: the whole-call workspace
    n1 = kda.kda_host_staging_bytes(B, 64, H, 128, 128, kda.KDA_BF16, 0, 1, 0)
    qk1 = B * 64 * H * 128 * 2
    assert n1 == 5 * r256(qk1) + r256(B * 64 * H * 2) + r256(state) + 256 + \
        r256(kda.kda_workspace_bytes(B, 64, H, 128, 128))



def test_workspace_of_the_segmented_two_kernel_form(lib):
    # with segments forced, a dense batch on the two-kernel path asks for the
    # records of every chunk and three [N][G][H][128][128] fp32 state buffers
    # (entry states, zero-start states, transitions) after the carried state
    def r256(x):
        return (x + 255) // 256 * 256
    N, T, H = 2, 1500, 3
    nchunks = (T + 63) // 64
    carry = r256(N * H * 128 * 128 * 4)
    try:
        assert kda.kda_debug_split_segments(3) == 0
        n3 = kda.kda_workspace_bytes(N, T, H, 128, 128, kda.KDA_BF16, 0, kda.KDA_ALGO_SPLIT, 0)
        assert n3 == carry + N * H * nchunks * 66048 + 3 * r256(N * 3 * H * 128 * 128 * 4)
        # the form a call takes follows the workspace it is given
        assert kda.kda_split_segment_count(N, T, H, n3) == 3
        assert kda.kda_split_segment_count(N, T, H, n3 - 1) == 1
        # five asked for, four possible (every segment holds a chunk: 11 chunks)
        kda.kda_debug_split_segments(5)
        n4 = kda.kda_workspace_bytes(1, 645, 2, 128, 128, kda.KDA_BF16, 0,
                                     kda.KDA_ALGO_SPLIT, 0)
        assert n4 == r256(2 * 128 * 128 * 4) + 2 * 11 * 66048 + 3 * r256(4 * 2 * 128 * 128 * 4)
        # off: the plain sliced form
        kda.kda_debug_split_segments(-1)
        n0 = kda.kda_workspace_bytes(N, T, H, 128, 128, kda.KDA_BF16, 0, kda.KDA_ALGO_SPLIT, 0)
        assert n0 == carry + N * H * nchunks * 66048
    finally:
        kda.kda_debug_split_segments(0)


def test_staging_bytes_of_the_pipelined_packed_host_call(lib):
    # a packed bf16 batch at dk = dv = 128 runs in up to eight pieces of chunk
    # columns (of the bound ceil(T / 64) + N): the staging holds the inputs,
    # outputs, states and offsets plus the packed workspace of one piece
    def r256(x):
        return (x + 255) // 256 * 256
    N, T, H = 28, 1 << 20, 16
    qk = T * H * 128 * 2
    state = N * H * 128 * 128 * 4
    fixed = 5 * r256(qk) + r256(T * H * 2) + 2 * r256(state) + r256((N + 1) * 4) + 256
    g_max = (T + 63) // 64 + N
    per = (g_max + 7) // 8
    piece = r256(state) + r256((N + 1) * 4) + r256(N * 4) + r256(g_max * 8) + per * H * 66048
    n = kda.kda_host_staging_bytes(N, T, H, 128, 128, kda.KDA_BF16, 1, 1, 1)
    assert n == fixed + r256(piece)

def test_package_fails_loudly_without_library(tmp_path):
    saved = kda._lib
    try:
        kda._lib = None
        with pytest.raises(RuntimeError, match="libkda.so not found"):
            kda.load(str(tmp_path / "missing.so"))
    finally:
        kda._lib = saved


def test_split_path_host_checks(lib):
    # workspace sizing of the two-kernel path: carried state + one slice of
    # 66048-byte chunk records per (sequence, head); a packed batch keeps
    # every chunk column (ceil(T / 64) + N of them at most) at once, after
    # its chunk offsets, sequence order and chunk table
    carry = 2 * 32 * 128 * 128 * 4
    nb = kda.kda_workspace_bytes(2, 32768, 32, 128, 128, algo=kda.KDA_ALGO_SPLIT)
    assert nb == carry + 2 * 32 * 512 * 66048
    assert kda.kda_workspace_bytes(2, 100, 1, 128, 128, algo=kda.KDA_ALGO_SPLIT) == \
        2 * 128 * 128 * 4 + 2 * 2 * 66048
    g_max = 32768 // 64 + 2
    assert kda.kda_workspace_bytes(2, 32768, 32, 128, 128, algo=kda.KDA_ALGO_SPLIT,
                                   packed=1) == carry + 256 + 256 + 4352 + 32 * g_max * 66048
    assert g_max * 8 <= 4352
    assert kda.kda_resolve_algo(kda.KDA_BF16, 128, 128, 0, kda.KDA_ALGO_SPLIT) == \
        kda.KDA_ALGO_SPLIT
    assert kda.kda_resolve_algo(kda.KDA_BF16, 64, 128, 0, kda.KDA_ALGO_SPLIT) == -1
    # the stage hook rejects bad arguments before anything is queued
    st = dict(q=A, k=2 * A, v=3 * A, g_logit=4 * A, beta=5 * A, init_state=None, out=6 * A,
              final_state=None, B=1, T=64, H=1, workspace=7 * A, workspace_bytes=1 << 30)
    assert kda.kda_split_stage(3, **st) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_split_stage(1, **dict(st, workspace=None)) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_split_stage(1, **dict(st, q=A + 8)) == kda.KDA_ERR_MISALIGNED
    assert kda.kda_split_stage(2, **dict(st, T=0)) == kda.KDA_ERR_INVALID_ARG


def test_packed_workspace_sizes(lib):
    # [carry][chunk offsets][sequence order][chunk table][records of a slice of
    # chunk columns]
    def r256(x):
        return (x + 255) // 256 * 256
    # (by default the records of every column while they fit in 32 GiB)
    N, T, H = 3, 1 << 20, 16
    g_max = T // 64 + N
    rec_at = r256(N * H * 128 * 128 * 4) + r256((N + 1) * 4) + r256(N * 4) + r256(g_max * 8)
    assert kda.kda_workspace_bytes(N, T, H, 128, 128, packed=1) == rec_at + g_max * H * 66048
    N, T, H = 3, 1 << 21, 16
    g_max = T // 64 + N
    rec_at = r256(N * H * 128 * 128 * 4) + r256((N + 1) * 4) + r256(N * 4) + r256(g_max * 8)
    cols = (32 << 30) // (H * 66048)
    assert cols < g_max
    assert kda.kda_workspace_bytes(N, T, H, 128, 128, packed=1) == rec_at + cols * H * 66048


def test_resolve_path(lib):
    # the automatic path of a bf16 batch at d = 128 is the two-kernel form,
    # fp32 inputs and other head sizes take the CUDA-core path
    rp = kda.kda_resolve_path
    assert rp(2, 32768, 32) == kda.KDA_ALGO_SPLIT
    assert rp(2, 32768, 32, packed=True) == kda.KDA_ALGO_SPLIT
    # a packed batch too long to hold every chunk record at once runs in
    # slices of chunk columns, its default workspace capped at 32 GiB of records
    assert rp(1, 1 << 20, 16, packed=True) == kda.KDA_ALGO_SPLIT
    assert rp(2, 32768, 32, algo=kda.KDA_ALGO_TC) == kda.KDA_ALGO_TC
    assert rp(2, 100, 4, dtype=kda.KDA_F32) == kda.KDA_ALGO_SIMT
    assert rp(2, 100, 4, dk=64) == kda.KDA_ALGO_SIMT
    assert rp(0, 100, 4) == -1
    assert rp(2, 100, 4, dtype=kda.KDA_F32, algo=kda.KDA_ALGO_SPLIT) == -1


def test_allocation_free_entry_has_the_same_argument_rules(lib):
    # kda_chunk_fwd_seg_static refuses exactly what kda_chunk_fwd_seg refuses,
    # before anything is queued (fake addresses, never dereferenced)
    def st(**over):
        a = dict(q=A, k=2 * A, v=3 * A, g_logit=4 * A, beta=5 * A, init_state=None,
                 out=6 * A, final_state=None, B=1, T=256, H=2, dk=128, dv=128, scale=1.0,
                 nseg=2)
        a.update(over)
        return kda.kda_chunk_fwd_seg_static(**a)
    assert st(out=A) == kda.KDA_ERR_INVALID_ARG              # out == q
    assert st(out=3 * A + 64) == kda.KDA_ERR_INVALID_ARG     # out overlaps v
    assert st(final_state=2 * A) == kda.KDA_ERR_INVALID_ARG  # final state over k
    assert st(init_state=6 * A) == kda.KDA_ERR_INVALID_ARG   # initial state under out
    assert st(q=None) == kda.KDA_ERR_INVALID_ARG
    assert st(q=A + 8) == kda.KDA_ERR_MISALIGNED
    assert st(init_state=7 * A + 4) == kda.KDA_ERR_MISALIGNED
    assert st(dk=64) == kda.KDA_ERR_UNSUPPORTED
    assert st(nseg=1) == kda.KDA_ERR_INVALID_ARG
    # past the fixed scratch array: refused before any device work
    assert st(H=32, nseg=8) == kda.KDA_ERR_WORKSPACE


def test_stall_test_hook_flags(lib):
    assert kda.kda_debug_stall_test(4) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_debug_stall_test(-1) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_debug_stall_test(0) == kda.KDA_OK
