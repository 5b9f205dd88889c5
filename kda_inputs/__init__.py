"""Seeded synthetic inputs for the KDA chunked forward.

This module holds no part of the method's arithmetic: it only draws random
tensors (torch CPU generators), L2-normalises q and k per (token, head) and
maps the beta logits through a sigmoid, as the workload recipes prescribe.
Both the GPU path's tests/bench and the fp64 oracle take their inputs from
here; neither imports the other.

Layouts (row-major, contiguous):
  q, k, g_logit  [B, T, H, dk]     v  [B, T, H, dv]     beta  [B, T, H]
  init_state     [N, H, dk, dv] fp32 (N = B, or the number of packed
                                      sequences when cu_seqlens is given)
  cu_seqlens     int32 [N + 1]  (packed layout: B == 1, T == cu_seqlens[-1])

Each (batch row b, head h) unit is drawn from its own generator, seeded with
``unit_seed(seed, b, h)``, in the fixed order q, k, v, beta-logit, g-logit,
then (if the workload has one) the initial state of every sequence that
starts in that row.  Any unit can therefore be regenerated on its own, which
lets the oracle recompute a sample of heads of a large workload without
materialising the whole batch.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import os
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "unit_seed", "varlen_lengths", "make_unit", "make_inputs",
           "small_workload"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    chunk: int
    dtype: torch.dtype
    seed: int
    g_mean: float = 0.0
    g_std: float = 1.0
    beta_mean: float = 0.0
    beta_std: float = 1.0
    s0_std: float = 0.0          # 0 -> zero initial state
    varlen: bool = False          # packed batch described by cu_seqlens
    lengths: Optional[tuple] = None  # explicit varlen lengths (else drawn)
    varlen_lo: int = 128
    varlen_hi: int = 4096
    # added to the batch row of every unit's stream: ranks of a multi-GPU
    # run draw rows r*B .. r*B+B-1 of one long batch, so their data differ
    row_offset: int = 0

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def seqlens(self):
        if not self.varlen:
            return None
        if self.lengths is not None:
            return list(self.lengths)
        return varlen_lengths(self.T, self.seed, self.varlen_lo, self.varlen_hi)

    def n_seqs(self) -> int:
        return len(self.seqlens()) if self.varlen else self.B


# The five workloads of the KDA forward, plus the stronger decay-stress variant.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", B=1, T=64, H=1, dk=16, dv=16, chunk=16,
                          dtype=torch.float32, seed=0),
    "h4_t4k": Workload("h4_t4k", B=1, T=4096, H=4, dk=128, dv=128, chunk=64,
                       dtype=torch.bfloat16, seed=1, s0_std=0.02),
    "b2_h32_t32k": Workload("b2_h32_t32k", B=2, T=32768, H=32, dk=128, dv=128, chunk=64,
                            dtype=torch.bfloat16, seed=2),
    "varlen_floor": Workload("varlen_floor", B=1, T=32768, H=16, dk=128, dv=128, chunk=64,
                             dtype=torch.bfloat16, seed=3, g_mean=4.0, beta_mean=2.0,
                             varlen=True),
    "varlen_floor_hard": Workload("varlen_floor_hard", B=1, T=32768, H=16, dk=128, dv=128,
                                  chunk=64, dtype=torch.bfloat16, seed=3, g_mean=6.0,
                                  beta_mean=2.0, varlen=True),
    "ctx1m": Workload("ctx1m", B=1, T=1 << 20, H=16, dk=128, dv=128, chunk=64,
                      dtype=torch.bfloat16, seed=4, g_mean=-1.0),
    # a packed 1M-token batch too long to hold every chunk record at once
    # (slices of chunk columns), with initial states: not one of the five
    # workloads, a check of the sliced packed path at full size
    "varlen_ctx1m": Workload("varlen_ctx1m", B=1, T=1 << 20, H=16, dk=128, dv=128, chunk=64,
                             dtype=torch.bfloat16, seed=5, g_mean=-1.0, s0_std=0.02,
                             varlen=True, varlen_lo=1024, varlen_hi=65536),
}


def small_workload(name: str, **kw) -> Workload:
    """A workload of arbitrary (usually small) size, for parity and edge cases."""
    base = dict(B=1, T=64, H=1, dk=128, dv=128, chunk=64, dtype=torch.bfloat16, seed=0)
    base.update(kw)
    return Workload(name, **base)


_MASK64 = (1 << 64) - 1


def _splitmix64(x: int) -> int:
    """One step of the splitmix64 generator (Steele, Lea and Flood, "Fast
    splittable pseudorandom number generators", OOPSLA 2014): a bijective
    64-bit mix in which every input bit reaches every output bit."""
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & _MASK64
    return x ^ (x >> 31)


def unit_seed(seed: int, b: int, h: int) -> int:
    """Seed of the (batch row b, head h) stream of a workload seeded ``seed``.

    torch's CPU generator keeps only the low 32 bits of a seed, so the three
    numbers are chained through splitmix64 and the result is cut to 32 bits:
    every workload seed, row and head reaches the bits the generator uses.
    """
    x = _splitmix64(seed & _MASK64)
    x = _splitmix64(x ^ (b & _MASK64))
    x = _splitmix64(x ^ (h & _MASK64))
    return x & 0xFFFFFFFF


def varlen_lengths(total: int, seed: int, lo: int = 128, hi: int = 4096) -> list:
    """Sequence lengths in [lo, hi] summing exactly to ``total``.

    While more than ``hi`` tokens remain, draw L uniformly in
    [lo, min(hi, remaining - lo)]; the remainder (then in [lo, hi]) closes
    the list.
    """
    g = torch.Generator().manual_seed(seed)
    out = []
    rem = total
    while rem > hi:
        top = min(hi, rem - lo)
        L = int(torch.randint(lo, top + 1, (1,), generator=g).item())
        out.append(L)
        rem -= L
    out.append(rem)
    return out


def _l2norm_rows(x: torch.Tensor) -> torch.Tensor:
    n = torch.linalg.vector_norm(x, dim=-1, keepdim=True)
    return x / n.clamp_min(1e-30)


def make_unit(w: Workload, b: int, h: int):
    """Tensors of one (batch row, head) unit, fp32, before the dtype cast.

    Returns dict q [T,dk], k [T,dk], v [T,dv], beta [T], g [T,dk] and s0
    [n_seq_in_row, dk, dv] (zeros when the workload has a zero state).
    """
    g = torch.Generator().manual_seed(unit_seed(w.seed, b + w.row_offset, h))
    T = w.T
    q = torch.randn(T, w.dk, generator=g)
    k = torch.randn(T, w.dk, generator=g)
    v = torch.randn(T, w.dv, generator=g)
    bl = torch.randn(T, generator=g) * w.beta_std + w.beta_mean
    gl = torch.randn(T, w.dk, generator=g) * w.g_std + w.g_mean
    nseq = w.n_seqs() if w.varlen else 1
    if w.s0_std > 0:
        s0 = torch.randn(nseq, w.dk, w.dv, generator=g) * w.s0_std
    else:
        s0 = torch.zeros(nseq, w.dk, w.dv)
    return dict(q=_l2norm_rows(q), k=_l2norm_rows(k), v=v, beta=torch.sigmoid(bl), g=gl, s0=s0)


def make_inputs(w: Workload, device="cpu"):
    """Every input of workload ``w`` in its storage dtype.

    Returns dict with q, k, v, g, beta (w.dtype), init_state (fp32 or None),
    cu_seqlens (int32 or None) and the shape arguments.
    """
    B, T, H = w.B, w.T, w.H
    dt = w.dtype
    q = torch.empty(B, T, H, w.dk, dtype=dt)
    k = torch.empty_like(q)
    gt = torch.empty_like(q)
    v = torch.empty(B, T, H, w.dv, dtype=dt)
    beta = torch.empty(B, T, H, dtype=dt)
    N = w.n_seqs()
    s0 = torch.zeros(N, H, w.dk, w.dv) if w.s0_std > 0 else None
    def fill(bh):
        b, h = bh
        u = make_unit(w, b, h)
        q[b, :, h] = u["q"].to(dt)
        k[b, :, h] = u["k"].to(dt)
        v[b, :, h] = u["v"].to(dt)
        beta[b, :, h] = u["beta"].to(dt)
        gt[b, :, h] = u["g"].to(dt)
        if s0 is not None:
            if w.varlen:
                s0[:, h] = u["s0"]
            else:
                s0[b, h] = u["s0"][0]

    units = [(b, h) for b in range(B) for h in range(H)]
    # units write disjoint slices; torch kernels release the GIL
    workers = max(1, min(len(units), os.cpu_count() or 1, 32))
    if workers == 1 or B * T * H < (1 << 16):
        for u in units:
            fill(u)
    else:
        with cf.ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, units))
    cu = None
    if w.varlen:
        lens = w.seqlens()
        cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    out = dict(q=q, k=k, v=v, g=gt, beta=beta, init_state=s0, cu_seqlens=cu,
               B=(N if w.varlen else B), T=T, H=H, dk=w.dk, dv=w.dv, chunk=w.chunk)
    if device != "cpu":
        for key in ("q", "k", "v", "g", "beta", "init_state", "cu_seqlens"):
            if out[key] is not None:
                out[key] = out[key].to(device)
    return out
