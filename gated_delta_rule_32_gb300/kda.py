"""ctypes binding of libkda.so (include/kda.h), argument marshalling only.

The functions keep the C names.  Tensor arguments may be torch tensors
(their data_ptr() is passed) or raw integer addresses; None is NULL.  Every
step of the forward runs in the library's kernels: if the library is not
built, or there is no GPU, calls fail loudly; nothing here computes.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "kda.h")

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_MISALIGNED = 3
KDA_ERR_BAD_SEQLENS = 4
KDA_ERR_TIMEOUT = 5
KDA_ERR_CUDA = 6
KDA_ERR_WORKSPACE = 7
KDA_ERR_BOUNDS = 8
KDA_BF16 = 0
KDA_F32 = 1
KDA_ALGO_AUTO = 0
KDA_ALGO_SIMT = 1
KDA_ALGO_TC = 2
KDA_ALGO_SPLIT = 3

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_SIGS = {
    "kda_status_string": (ctypes.c_char_p, [_i]),
    "kda_build_info": (ctypes.c_char_p, []),
    "kda_resolve_algo": (_i, [_i] * 5),
    "kda_resolve_path": (_i, [_i] * 9),
    "kda_chunk_fwd": (_i, [_vp] * 8 + [_i] * 5 + [_vp, _vp]),
    "kda_chunk_fwd_f32": (_i, [_vp] * 8 + [_i] * 5 + [_vp, _vp]),
    "kda_chunk_fwd_ex": (_i, [_vp] * 8 + [_i] * 5 + [_vp, _i, _i, ctypes.c_float, _i, _vp,
                                                   ctypes.c_size_t, _vp, _vp]),
    "kda_workspace_bytes": (ctypes.c_size_t, [_i] * 9),
    "kda_chunk_fwd_seg": (_i, [_vp] * 8 + [_i] * 5 + [ctypes.c_float, _i, _vp, ctypes.c_size_t,
                                                    _vp, _vp]),
    "kda_seg_workspace_bytes": (ctypes.c_size_t, [_i] * 5),
    "kda_chunk_fwd_seg_static": (_i, [_vp] * 8 + [_i] * 5 + [ctypes.c_float, _i, _vp, _vp]),
    "kda_decode": (_i, [_vp] * 7 + [_i] * 6 + [ctypes.c_float, _vp]),
    "kda_chunk_fwd_ckpt": (_i, [_vp] * 8 + [_i] * 5 + [_vp, _i, ctypes.c_float, _vp, _i, _i,
                                                     _vp, _vp]),
    "kda_chunk_fwd_host": (_i, [_vp] * 8 + [_i] * 5 + [_vp, _i, ctypes.c_float, _vp,
                                                   ctypes.c_size_t, _vp]),
    "kda_host_staging_bytes": (ctypes.c_size_t, [_i] * 9),
    "kda_debug_umma": (_i, [_vp] * 3 + [_i] * 6 + [_vp, _vp]),
    "kda_split_stage": (_i, [_i] + [_vp] * 8 + [_i] * 3 + [ctypes.c_float, _vp, ctypes.c_size_t,
                                                        _vp, _vp]),
    "kda_debug_intra": (_i, [_vp] * 5 + [_i] * 5 + [_vp, _i, _i] + [_vp] * 6 + [_vp]),
    "kda_debug_stall_test": (_i, [_i]),
    "kda_debug_split_segments": (_i, [_i]),
    "kda_split_segment_count": (_i, [_i, _i, _i, ctypes.c_size_t]),
    "kda_segment_summary": (_i, [_vp] * 6 + [_i] * 5 + [_vp, _vp]),
    "kda_summary_floats": (ctypes.c_size_t, [_i] * 4),
    "kda_state_compose": (_i, [_vp, _i, _vp, _vp] + [_i] * 4 + [_vp]),
    "kda_debug_record_capacity": (_i, [ctypes.c_int64]),
}


class KdaError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__("%s failed: %s" % (fn, status_string(code) if _lib else code))


def load(path: str = LIB_PATH):
    """Load libkda.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    "libkda.so not found at %s: build it with "
                    "`python -m gated_delta_rule_32_gb300.build` (needs nvcc)" % path)
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def header_functions(header: str = HEADER):
    """Names of the functions include/kda.h declares."""
    txt = open(header).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(kda_[a-z_0-9]+)\s*\(",
                                 txt, flags=re.M)))


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_string(code: int) -> str:
    return load().kda_status_string(int(code)).decode()


def kda_build_info() -> str:
    return load().kda_build_info().decode()


def kda_resolve_path(N, T, H, dk=128, dv=128, dtype=KDA_BF16, chunk_size=0,
                     algo=KDA_ALGO_AUTO, packed=False) -> int:
    return load().kda_resolve_path(N, T, H, dk, dv, dtype, chunk_size, algo, int(packed))


def kda_resolve_algo(dtype=KDA_BF16, dk=128, dv=128, chunk_size=0, algo=KDA_ALGO_AUTO) -> int:
    return load().kda_resolve_algo(dtype, dk, dv, chunk_size, algo)


def kda_chunk_fwd(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk, dv,
                  cu_seqlens=None, stream=None) -> int:
    return load().kda_chunk_fwd(_p(q), _p(k), _p(v), _p(g_logit), _p(beta), _p(init_state),
                                _p(out), _p(final_state), B, T, H, dk, dv, _p(cu_seqlens),
                                _stream(stream))


def kda_chunk_fwd_f32(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk, dv,
                      cu_seqlens=None, stream=None) -> int:
    return load().kda_chunk_fwd_f32(_p(q), _p(k), _p(v), _p(g_logit), _p(beta),
                                    _p(init_state), _p(out), _p(final_state), B, T, H, dk, dv,
                                    _p(cu_seqlens), _stream(stream))


def kda_chunk_fwd_ex(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk, dv,
                     cu_seqlens=None, dtype=KDA_BF16, chunk_size=0, scale=1.0,
                     algo=KDA_ALGO_AUTO, workspace=None, workspace_bytes=0, dev_status=None,
                     stream=None) -> int:
    return load().kda_chunk_fwd_ex(_p(q), _p(k), _p(v), _p(g_logit), _p(beta), _p(init_state),
                                   _p(out), _p(final_state), B, T, H, dk, dv, _p(cu_seqlens),
                                   dtype, chunk_size, float(scale), algo, _p(workspace),
                                   workspace_bytes, _p(dev_status), _stream(stream))


def kda_chunk_fwd_ckpt(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk, dv,
                       cu_seqlens=None, dtype=KDA_BF16, scale=1.0, checkpoints=None, every=512,
                       max_per_seq=1, dev_status=None, stream=None) -> int:
    return load().kda_chunk_fwd_ckpt(_p(q), _p(k), _p(v), _p(g_logit), _p(beta),
                                     _p(init_state), _p(out), _p(final_state), B, T, H, dk, dv,
                                     _p(cu_seqlens), dtype, float(scale), _p(checkpoints),
                                     every, max_per_seq, _p(dev_status), _stream(stream))


def kda_chunk_fwd_seg(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk, dv,
                      scale=1.0, nseg=1, workspace=None, workspace_bytes=0, dev_status=None,
                      stream=None) -> int:
    return load().kda_chunk_fwd_seg(_p(q), _p(k), _p(v), _p(g_logit), _p(beta), _p(init_state),
                                    _p(out), _p(final_state), B, T, H, dk, dv, float(scale),
                                    nseg, _p(workspace), workspace_bytes, _p(dev_status),
                                    _stream(stream))


def kda_chunk_fwd_seg_static(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk,
                             dv, scale=1.0, nseg=2, dev_status=None, stream=None) -> int:
    return load().kda_chunk_fwd_seg_static(_p(q), _p(k), _p(v), _p(g_logit), _p(beta),
                                           _p(init_state), _p(out), _p(final_state), B, T, H,
                                           dk, dv, float(scale), nseg, _p(dev_status),
                                           _stream(stream))


def kda_seg_workspace_bytes(B, H, nseg, dk=128, dv=128) -> int:
    return load().kda_seg_workspace_bytes(B, H, nseg, dk, dv)


def kda_decode(q, k, v, g_logit, beta, state, out, N, T, H, dk, dv, dtype=KDA_BF16, scale=1.0,
               stream=None) -> int:
    return load().kda_decode(_p(q), _p(k), _p(v), _p(g_logit), _p(beta), _p(state), _p(out), N,
                             T, H, dk, dv, dtype, float(scale), _stream(stream))


def kda_workspace_bytes(N, T, H, dk, dv, dtype=KDA_BF16, chunk_size=0, algo=KDA_ALGO_AUTO,
                        packed=0) -> int:
    return load().kda_workspace_bytes(N, T, H, dk, dv, dtype, chunk_size, algo, int(packed))


def kda_chunk_fwd_host(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk, dv,
                       cu_seqlens=None, dtype=KDA_BF16, scale=1.0, dev_buffer=None,
                       dev_buffer_bytes=0, stream=None) -> int:
    return load().kda_chunk_fwd_host(_p(q), _p(k), _p(v), _p(g_logit), _p(beta),
                                     _p(init_state), _p(out), _p(final_state), B, T, H, dk, dv,
                                     _p(cu_seqlens), dtype, float(scale), _p(dev_buffer),
                                     dev_buffer_bytes, _stream(stream))


def kda_host_staging_bytes(B, T, H, dk, dv, dtype=KDA_BF16, has_init=0, has_final=0,
                           packed=0) -> int:
    return load().kda_host_staging_bytes(B, T, H, dk, dv, dtype, int(has_init),
                                         int(has_final), int(packed))


def kda_debug_intra(q, k, v, g_logit, beta, B, T, H, dk, dv, cu_seqlens, n, h, gam=None,
                    aqk=None, akk=None, tinv=None, w=None, u=None, stream=None) -> int:
    return load().kda_debug_intra(_p(q), _p(k), _p(v), _p(g_logit), _p(beta), B, T, H, dk, dv,
                                  _p(cu_seqlens), n, h, _p(gam), _p(aqk), _p(akk), _p(tinv),
                                  _p(w), _p(u), _stream(stream))


def kda_split_stage(stage, q, k, v, g_logit, beta, init_state, out, final_state, B, T, H,
                    scale=1.0, workspace=None, workspace_bytes=0, dev_status=None,
                    stream=None) -> int:
    return load().kda_split_stage(stage, _p(q), _p(k), _p(v), _p(g_logit), _p(beta),
                                  _p(init_state), _p(out), _p(final_state), B, T, H,
                                  float(scale), _p(workspace), workspace_bytes, _p(dev_status),
                                  _stream(stream))


def kda_debug_umma(A, B, D, M, N, K, a_mode=0, b_mode=0, pack=0, dev_status=None,
                   stream=None) -> int:
    return load().kda_debug_umma(_p(A), _p(B), _p(D), M, N, K, a_mode, b_mode, pack,
                                 _p(dev_status), _stream(stream))


def forward(q, k, v, g_logit, beta, init_state=None, cu_seqlens=None, scale=1.0,
            output_final_state=True, chunk_size=0, algo=KDA_ALGO_AUTO, dev_status=None,
            stream=None):
    """Allocate the outputs and call kda_chunk_fwd_ex on the current stream.

    q, k, g_logit [B,T,H,dk], v [B,T,H,dv], beta [B,T,H] CUDA tensors of one
    dtype (bfloat16 or float32); init_state [N,H,dk,dv] fp32 or None;
    cu_seqlens int32 [N+1] CUDA tensor or None.  Returns (out, final_state).
    The workspace comes from PyTorch's caching allocator (a block it keeps
    and hands out again on the next call), not from the library's own
    stream-ordered allocation.
    """
    import torch
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    dtype = {torch.bfloat16: KDA_BF16, torch.float32: KDA_F32}[q.dtype]
    out = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
    fs = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device) \
        if output_final_state else None
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    nb = kda_workspace_bytes(N, T, H, dk, dv, dtype, chunk_size, algo,
                             int(cu_seqlens is not None))
    ws = torch.empty(nb, dtype=torch.uint8, device=q.device) if nb else None
    if ws is not None and isinstance(stream, torch.cuda.Stream):
        ws.record_stream(stream)  # (freed for reuse only after the work on `stream`)
    rc = kda_chunk_fwd_ex(q, k, v, g_logit, beta, init_state, out, fs, N, T, H, dk, dv,
                          cu_seqlens, dtype, chunk_size, scale, algo, ws, nb, dev_status,
                          stream)
    if rc != KDA_OK:
        raise KdaError("kda_chunk_fwd_ex", rc)
    return out, fs


def kda_debug_stall_test(flags: int) -> int:
    """Test hook: make the two-kernel path's first waits run out (bit 0 intra
    kernel, bit 1 state kernel); 0 restores normal calls."""
    return load().kda_debug_stall_test(int(flags))


def kda_debug_split_segments(segments: int) -> int:
    """Test hook: force that many segments per sequence on the two-kernel
    path for dense batches (> 0), turn segments off (< 0) or restore the
    automatic choice (0)."""
    return load().kda_debug_split_segments(int(segments))


def kda_split_segment_count(N: int, T: int, H: int, workspace_bytes: int) -> int:
    """Segments per sequence the two-kernel path takes for a dense batch with
    this workspace (1: the plain form)."""
    return load().kda_split_segment_count(int(N), int(T), int(H), int(workspace_bytes))


def kda_debug_record_capacity(items: int) -> int:
    """Debug builds: the chunk-record capacity the kernels are told (0 = real)."""
    return load().kda_debug_record_capacity(int(items))


def kda_segment_summary(q, k, v, g_logit, beta, summary, B, T, H, dk=128, dv=128,
                        dev_status=None, stream=None) -> int:
    return load().kda_segment_summary(_p(q), _p(k), _p(v), _p(g_logit), _p(beta),
                                      _p(summary), B, T, H, dk, dv, _p(dev_status),
                                      _stream(stream))


def kda_summary_floats(N, H, dk=128, dv=128) -> int:
    return load().kda_summary_floats(N, H, dk, dv)


def kda_state_compose(summaries, m, init_state, state_out, N, H, dk=128, dv=128,
                      stream=None) -> int:
    return load().kda_state_compose(_p(summaries), m, _p(init_state), _p(state_out), N, H,
                                    dk, dv, _stream(stream))
