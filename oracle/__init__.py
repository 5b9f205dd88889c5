"""fp64 CPU oracle for the KDA chunked forward -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the CPU-baseline leg of the benchmark may
import this package.  The product path (the CUDA library and its binding)
never imports, links or runs anything here, and nothing here imports the
product package.

Contents:
  kda_oracle.c     plain fp64 token loop (the recurrence written out), built
                   with gcc into _build/libkda_oracle.so and driven by
                   ``fwd`` below.
  chunk_mirror.py  the chunkwise-parallel form in numpy fp64, step by step,
                   for the chunked-equals-recurrent pin and per-step
                   comparisons.

Pins (tests/test_oracle_pins.py) tie both to closed forms and invariants that
follow from the pages and from linear algebra; every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

LOG_FLOOR = -5.0


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (IEEE fp64, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_fwd_f64.restype = ctypes.c_int
            lib.kda_oracle_fwd_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_int32), ctypes.c_double,
                                               ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
            lib.kda_oracle_log_decay.restype = ctypes.c_double
            lib.kda_oracle_log_decay.argtypes = [ctypes.c_double]
            lib.kda_oracle_log_decay_vec.restype = None
            lib.kda_oracle_log_decay_vec.argtypes = [dp, dp, ctypes.c_int64]
            _lib = lib
    return _lib


def _f64(x):
    """Upcast a torch tensor or array (already rounded to its storage dtype)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def log_decay(x) -> np.ndarray:
    """a = max(-softplus(x), -5) elementwise, via the C oracle."""
    lib = _load()
    xa = _f64(x)
    out = np.empty_like(xa)
    lib.kda_oracle_log_decay_vec(_ptr(xa), _ptr(out), xa.size)
    return out


def fwd(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale=1.0, nthreads=0,
        return_threads=False):
    """fp64 token-loop forward.

    q, k, g [rows, T, H, dk]; v [rows, T, H, dv]; beta [rows, T, H];
    init_state [nseq, H, dk, dv] or None; cu_seqlens int [nseq+1] or None
    (then rows == 1 and the batch is packed).  Inputs may be torch tensors
    of any dtype (their stored values are upcast exactly) or numpy arrays.
    Returns (out [rows, T, H, dv], final_state [nseq, H, dk, dv]) as fp64
    numpy arrays (and the thread count if return_threads).
    """
    lib = _load()
    qa, ka, va, ga, ba = (_f64(t) for t in (q, k, v, g, beta))
    rows, T, H, dk = qa.shape
    dv = va.shape[-1]
    s0 = _f64(init_state)
    cu = None
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        nseq = cu.size - 1
        if rows != 1:
            raise ValueError("packed batch must have one row")
    else:
        nseq = rows
    out = np.zeros((rows, T, H, dv), dtype=np.float64)
    fs = np.zeros((nseq, H, dk, dv), dtype=np.float64)
    used = ctypes.c_int(0)
    rc = lib.kda_oracle_fwd_f64(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), _ptr(ba), _ptr(s0),
                                _ptr(out), _ptr(fs), nseq, T, H, dk, dv,
                                None if cu is None else cu.ctypes.data_as(
                                    ctypes.POINTER(ctypes.c_int32)),
                                float(scale), int(nthreads), ctypes.byref(used))
    if rc != 0:
        raise RuntimeError("kda_oracle_fwd_f64 failed with %d" % rc)
    if return_threads:
        return out, fs, used.value
    return out, fs


def fwd_unit(q, k, v, g, beta, s0=None, scale=1.0):
    """Single (sequence, head) unit: q,k,g [T,dk], v [T,dv], beta [T], s0 [dk,dv]."""
    qa, ka, va, ga, ba = (_f64(t) for t in (q, k, v, g, beta))
    T, dk = qa.shape
    dv = va.shape[1]
    s0a = None if s0 is None else _f64(s0).reshape(1, 1, dk, dv)
    out, fs = fwd(qa.reshape(1, T, 1, dk), ka.reshape(1, T, 1, dk), va.reshape(1, T, 1, dv),
                  ga.reshape(1, T, 1, dk), ba.reshape(1, T, 1), s0a, scale=scale, nthreads=1)
    return out.reshape(T, dv), fs.reshape(dk, dv)
