"""Ranks of the context-parallel tests (tests/test_cp.py, tests/test_cp_gpu.py).

Each rank joins a gloo process group on 127.0.0.1, takes its shard of a
seeded batch (uneven spans of the token axis, in rank order), runs
gated_delta_rule_32_gb300.cp.context_parallel_forward and saves its output
and the state after its span.  In "oracle" mode the three per-rank steps are
computed by the fp64 oracle (CPU only: this checks the exchange, its order
and the composition); in "gpu" mode by the library's kernels on cuda:0.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402


class OracleOps:
    """The per-rank steps from the fp64 oracle: a span's cumulative transition
    is its final state from the identity with zero values, its zero-start
    state its final state from zero; composition is matrix arithmetic."""

    def summary(self, q, k, v, g, beta):
        import oracle
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        P = np.zeros((B, H, dk, dk))
        S0 = np.zeros((B, H, dk, dv))
        for b in range(B):
            for h in range(H):
                args = (q[b, :, h], k[b, :, h])
                _, P[b, h] = oracle.fwd_unit(*args, np.zeros((T, dk)), g[b, :, h], beta[b, :, h],
                                             np.eye(dk))
                _, S0[b, h] = oracle.fwd_unit(*args, v[b, :, h], g[b, :, h], beta[b, :, h],
                                              None)
        return torch.from_numpy(np.concatenate([P.ravel(), S0.ravel()]))

    def compose(self, summaries, m, init_state, B, H, dk, dv, device):
        S = np.zeros((B, H, dk, dv)) if init_state is None else init_state.double().numpy()
        for j in range(m):
            x = summaries[j].double().numpy()
            P = x[:B * H * dk * dk].reshape(B, H, dk, dk)
            S0 = x[B * H * dk * dk:].reshape(B, H, dk, dv)
            S = np.einsum("bhij,bhjv->bhiv", P, S) + S0
        return torch.from_numpy(S)

    def forward(self, q, k, v, g, beta, init_state, scale):
        import oracle
        o, s = oracle.fwd(q, k, v, g, beta, init_state, scale=scale)
        return torch.from_numpy(o), torch.from_numpy(s)


def shard_bounds(T, world):
    """Uneven spans of [0, T): rank r gets a share proportional to r + 2."""
    w = np.arange(world) + 2.0
    cuts = np.concatenate([[0], np.round(np.cumsum(w) / w.sum() * T)]).astype(int)
    cuts[-1] = T
    return cuts


def run(rank, world, port, mode, outdir, B, T, H, d, seed):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from gated_delta_rule_32_gb300 import cp
        from kda_inputs import make_inputs, small_workload
        dtype = torch.float32 if mode == "oracle" else torch.bfloat16
        w = small_workload("cp", B=B, T=T, H=H, dk=d, dv=d, seed=seed, s0_std=0.05, dtype=dtype)
        x = make_inputs(w)
        cuts = shard_bounds(T, world)
        t0, t1 = int(cuts[rank]), int(cuts[rank + 1])
        sh = {key: x[key][:, t0:t1].contiguous() for key in ("q", "k", "v", "g", "beta")}
        s0 = x["init_state"]
        if mode == "gpu":
            dev = torch.device("cuda", 0)
            torch.cuda.set_device(dev)
            sh = {key: t.to(dev) for key, t in sh.items()}
            s0 = s0.to(dev)
            ops = cp.LibraryOps()
        else:
            sh = {key: t.double() for key, t in sh.items()}
            s0 = s0.double()
            ops = OracleOps()
        out, st = cp.context_parallel_forward(sh["q"], sh["k"], sh["v"], sh["g"], sh["beta"],
                                              s0, group=None, ops=ops)
        if mode == "gpu":
            torch.cuda.synchronize()
        np.savez(os.path.join(outdir, "rank%d.npz" % rank), out=out.float().cpu().double().numpy()
                 if mode == "gpu" else out.numpy(), state=st.cpu().double().numpy(),
                 t0=t0, t1=t1)
    finally:
        dist.destroy_process_group()
