"""Context parallelism: the token axis of a batch split across the ranks of a
process group, with one fixed-size all-gather.

Rank r holds tokens [t_r, t_{r+1}) of every sequence of a dense batch (its
shard, [B, T_r, H, d]; shards in rank order).  The state update of a span is
affine in the state entering it, S_out = P S_in + S0, with P the span's
cumulative transition and S0 its final state from a zero start (Kimi K3
architecture, orkas.ai, "The cost is paid in the serving stack"; Towards AI
walkthrough, "Infrastructure co-design").  So each rank

  1. summarises its span: (P_r, S0_r), B * H * (dk * dk + dk * dv) floats
     (the library's kda_segment_summary);
  2. takes part in one all-gather of those fixed-size summaries;
  3. folds the summaries of the ranks before it into its entry state,
     S_in(r) = P_{r-1} S_in(r-1) + S0_{r-1} from the batch's initial state
     (kda_state_compose);
  4. runs its span from that state (kda_chunk_fwd_ex), writing its part of
     the output and the state after its span (the last rank's is the
     sequences' final state).

The exchange is the only step that crosses ranks, and its size does not
depend on the sequence length.  No kernel waits on another rank: the
all-gather is a torch.distributed collective between the ranks' own launches
(NCCL moves device tensors; backends that move host tensors, such as gloo,
get a host copy of the summary).  This module only orders those calls and
marshals tensors; the arithmetic runs in the library's kernels (LibraryOps).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import kda

__all__ = ["LibraryOps", "context_parallel_forward"]


class LibraryOps:
    """The three GPU steps of a rank, through the C ABI of libkda.so."""

    def __init__(self, stream=None):
        self.stream = stream

    def _s(self, t):
        return self.stream if self.stream is not None else torch.cuda.current_stream(t.device)

    def summary(self, q, k, v, g_logit, beta):
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        out = torch.empty(kda.kda_summary_floats(B, H, dk, dv), dtype=torch.float32,
                          device=q.device)
        rc = kda.kda_segment_summary(q, k, v, g_logit, beta, out, B, T, H, dk, dv, None,
                                     self._s(q))
        if rc != 0:
            raise kda.KdaError("kda_segment_summary", rc)
        return out

    def compose(self, summaries, m, init_state, B, H, dk, dv, device):
        out = torch.empty(B, H, dk, dv, dtype=torch.float32, device=device)
        stream = self.stream if self.stream is not None else torch.cuda.current_stream(device)
        rc = kda.kda_state_compose(summaries, m, init_state, out, B, H, dk, dv, stream)
        if rc != 0:
            raise kda.KdaError("kda_state_compose", rc)
        return out

    def forward(self, q, k, v, g_logit, beta, init_state, scale):
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        out = torch.empty_like(v)
        fs = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
        dtype = kda.KDA_BF16 if q.dtype == torch.bfloat16 else kda.KDA_F32
        rc = kda.kda_chunk_fwd_ex(q, k, v, g_logit, beta, init_state, out, fs, B, T, H, dk, dv,
                                  None, dtype, 0, scale, kda.KDA_ALGO_AUTO, None, 0, None,
                                  self._s(q))
        if rc != 0:
            raise kda.KdaError("kda_chunk_fwd_ex", rc)
        return out, fs


def context_parallel_forward(q, k, v, g_logit, beta, init_state=None, scale=1.0, group=None,
                             ops=None):
    """Forward of this rank's shard of a token-split batch.

    q, k, g_logit [B, T_r, H, dk]; v [B, T_r, H, dv]; beta [B, T_r, H]: this
    rank's tokens of every sequence.  init_state: the state entering every
    sequence (the same tensor on every rank) or None.  Returns (out
    [B, T_r, H, dv], the state after this rank's span [B, H, dk, dv]).
    `ops` supplies the three per-rank steps (default: the library's kernels).
    """
    ops = ops if ops is not None else LibraryOps()
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    B, _, H, dk = q.shape
    dv = v.shape[-1]
    summ = ops.summary(q, k, v, g_logit, beta)
    # the one exchange: every rank's fixed-size summary, in rank order
    host = dist.get_backend(group) == "gloo"
    send = summ.cpu() if host and summ.is_cuda else summ
    parts = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(parts, send, group=group)
    before = None
    if rank > 0:
        before = torch.stack(parts[:rank]).to(summ.device)
    s_in = ops.compose(before, rank, init_state, B, H, dk, dv, summ.device)
    return ops.forward(q, k, v, g_logit, beta, s_in, scale)
