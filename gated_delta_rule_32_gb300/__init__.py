"""KDA chunked forward on GB300 (sm_103a): C-ABI library + thin ctypes binding.

The compute path is libkda.so (csrc/): hand-written CUDA kernels behind the
C ABI declared in include/kda.h.  This package only builds and loads it and
marshals arguments (kda.py).  There is no CPU fallback: without the built
library or a GPU, calls raise.
"""
from .kda import (forward, load, status_string, kda_chunk_fwd, kda_chunk_fwd_f32,  # noqa: F401
                  kda_chunk_fwd_ex, kda_chunk_fwd_host, kda_workspace_bytes,
                  kda_host_staging_bytes, kda_debug_intra, kda_build_info, kda_resolve_algo, KdaError,
                  KDA_OK, KDA_BF16, KDA_F32, KDA_ALGO_AUTO, KDA_ALGO_SIMT, KDA_ALGO_TC)

__all__ = ["forward", "load", "status_string", "kda_chunk_fwd", "kda_chunk_fwd_f32",
           "kda_chunk_fwd_ex", "kda_chunk_fwd_host", "kda_workspace_bytes",
           "kda_host_staging_bytes", "kda_debug_intra", "kda_build_info", "KdaError"]
