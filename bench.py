#!/usr/bin/env python3
"""Benchmark of the KDA chunked forward on GB300.

One step = one full forward (every (sequence, head) of the workload, all
steps of the chunked path) over one batch of synthetic inputs resident in
HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle as the arm

Multi-GPU (torchrun): every rank runs an independent batch of the same
workload (different seed), no collective on the data path; the time is
the max over ranks and the value counts every rank's tokens (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from kda_inputs import WORKLOADS, make_inputs, make_unit, small_workload  # noqa: E402

METRIC = "KDA chunked-forward tokens/s at H=32,d=128,T=32K; % of BF16 TC roofline"
DEFAULT_WORKLOAD = "b2_h32_t32k"
PROFILES = os.path.join(ROOT, "profiles")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_workload(base, rank: int):
    """Rank r's batch: the same workload, its units drawn as rows r B ..
    r B + B - 1 of one long batch (and seed + 1000 r), so that the ranks run
    independent batches; rank 0 keeps the base workload."""
    import dataclasses
    if not rank:
        return base
    return dataclasses.replace(base, seed=base.seed + 1000 * rank,
                               row_offset=base.row_offset + rank * base.B)


def max_over_ranks(x: float, ws: int, device) -> float:
    """The largest x over the ranks (x itself on one rank)."""
    if ws <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(ws: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's step."""
    return ws * tokens_per_rank / (ms_per_step / 1e3)


def alg_bytes(w, has_init: bool, has_final: bool) -> int:
    """Algorithmic HBM bytes of one forward: every input read once, every
    output written once (bf16 q, k, g, v, beta, out; fp32 states)."""
    esz = 2 if w.dtype == torch.bfloat16 else 4
    th = w.B * w.T * w.H
    per_th = esz * (3 * w.dk + w.dv) + esz + esz * w.dv
    nstate = w.n_seqs() * w.H
    st = 4 * w.dk * w.dv * nstate * (int(has_init) + int(has_final))
    return th * per_th + st


def alg_flops(w) -> float:
    """Algorithmic FLOPs of the chunked form at chunk C (lower-triangular
    parts counted once): Grams 2*C^2/2*dk*2, UT solve C^3/3, W and U
    C^2*(dk+dv), W S, (Q*gam) S and K^T Delta 3*2*C*dk*dv, intra output
    C^2*dv; per chunk, times the number of chunks."""
    C, dk, dv = 64, w.dk, w.dv
    per_chunk = 2 * C * C * dk + C ** 3 / 3 + C * C * (dk + dv) + 6 * C * dk * dv + C * C * dv
    th = w.B * w.T * w.H
    return per_chunk * th / C


# the translation unit of the two-kernel path (less the C header's
# declarations): the source of the kernels the committed DRAM counters
# describe, so that edits elsewhere do not make them stale
SPLIT_SOURCES = ("kda_split.cu", "kda_common.cuh", "sm100.cuh", "kda_tc_util.cuh")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_32_gb300", "csrc")
    for name in SPLIT_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if
    it was taken on the current kernel source; else None."""
    path = os.path.join(PROFILES, "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
    except Exception:
        return None
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        sm = sorted(r[0] for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2])
                          if v.lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": reasons}


def oracle_sample(w, n_units: int, tokens: int, threads: int = 0, min_seconds: float = 0.0):
    """Time the fp64 oracle on the first n_units (row, head) units of the
    workload, first `tokens` tokens each, repeated (inputs drawn once) until
    at least `min_seconds` of oracle time have passed.  Returns (seconds,
    token-heads, threads used), summed over the repetitions."""
    import oracle
    units = [(b, h) for b in range(w.B) for h in range(w.H)][:n_units]
    T = min(tokens, w.T)
    qs, ks, vs, gs, bs, s0s = [], [], [], [], [], []
    for (b, h) in units:
        u = make_unit(w, b, h)
        qs.append(u["q"][:T].to(w.dtype)); ks.append(u["k"][:T].to(w.dtype))
        vs.append(u["v"][:T].to(w.dtype)); gs.append(u["g"][:T].to(w.dtype))
        bs.append(u["beta"][:T].to(w.dtype)); s0s.append(u["s0"][0])
    # the units as heads of one batch row
    q = torch.stack(qs, 1)[None]; k = torch.stack(ks, 1)[None]
    v = torch.stack(vs, 1)[None]; g = torch.stack(gs, 1)[None]
    beta = torch.stack(bs, 1)[None]
    s0 = torch.stack(s0s, 0)[None] if w.s0_std > 0 else None
    cu = None
    if w.varlen:
        cu = [0]
        for L in w.seqlens():
            if cu[-1] + L > T:
                break
            cu.append(cu[-1] + L)
        if cu[-1] < T:
            cu.append(T)
        cu = np.array(cu, dtype=np.int32)
        s0 = None
    dt, reps = 0.0, 0
    while reps == 0 or dt < min_seconds:
        t0 = time.perf_counter()
        _, _, used = oracle.fwd(q, k, v, g, beta, s0, cu, nthreads=threads, return_threads=True)
        dt += time.perf_counter() - t0
        reps += 1
    return dt, reps * len(units) * T, used


def resolve_workload(args):
    """The named workload, optionally resized (--B/--H/--T) for small
    profiling captures; a resized workload carries a '+resized' name."""
    import dataclasses
    w = WORKLOADS[args.workload]
    over = {k: getattr(args, k) for k in ("B", "H", "T") if getattr(args, k)}
    if over:
        w = dataclasses.replace(w, name=w.name + "+resized", **over)
    return w


def run_reference(args):
    ws, rank, _ = dist_env()
    if ws > 1 and rank != 0:
        return 0
    w = resolve_workload(args)
    import oracle
    oracle.build()
    n_units, tokens = args.ref_units, args.ref_tokens
    for _ in range(args.warmup):
        oracle_sample(w, n_units, min(tokens, 1024))
    times = []
    used = 1
    th = 0
    for _ in range(args.steps):
        dt, th, used = oracle_sample(w, n_units, tokens)
        times.append(dt)
    mean = sum(times) / len(times)
    value = th / w.H / mean          # tokens (all heads) per second
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk,
                       "dv": w.dv, "chunk": w.chunk},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used,
                             "kind": "oracle",
                             "sample": "%d (row, head) units x first %d tokens per step"
                                       % (n_units, min(tokens, w.T))},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_ours(args):
    import gated_delta_rule_32_gb300 as pkg
    from gated_delta_rule_32_gb300 import build as kbuild
    from gated_delta_rule_32_gb300 import kda

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        kbuild.build()
    if ws > 1:
        torch.distributed.barrier()
    kda.load()

    base = resolve_workload(args)
    w = rank_workload(base, rank)
    x = make_inputs(w)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
    N, T, H, dk, dv = x["B"], x["T"], x["H"], x["dk"], x["dv"]
    out = torch.empty(w.B, T, H, dv, dtype=w.dtype, device=dev)
    fs = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    dtype = kda.KDA_BF16 if w.dtype == torch.bfloat16 else kda.KDA_F32

    # the workspace the path asks for, allocated once like a serving engine would
    ws_bytes = kda.kda_workspace_bytes(N, T, H, dk, dv, dtype, 0, args.algo, int(w.varlen))
    work = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None

    def step():
        rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                  out, fs, N, T, H, dk, dv, d["cu_seqlens"], dtype, 0, 1.0,
                                  args.algo, work, ws_bytes, None, stream)
        if rc != 0:
            raise RuntimeError("kda_chunk_fwd_ex: " + kda.status_string(rc))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if not args.steps:
        # no count given: enough steps for a timed region of about 1.2 s, so
        # that the clock sampler sees several readings under load
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        est = max(e0.elapsed_time(e1) / 3, 1e-3)
        n = int(min(5000, max(20, 1200.0 / est)))
        if ws > 1:   # every rank times the same count
            t = torch.tensor([n], dtype=torch.int64, device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            n = int(t.item())
        args.steps = n

    # ---- device-timed region: K steps, inputs resident in HBM --------------
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_idx = vis.split(",")[local] if vis else str(local)
    clocks = ClockSampler(smi_idx)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), ws, dev)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    ms_per_step = total_ms / args.steps
    tokens = w.B * w.T
    value = job_value(ws, tokens, ms_per_step)

    # ---- the two kernels of the split path, each timed alone ----------------
    path = kda.kda_resolve_path(N, T, H, dk, dv, dtype, 0, args.algo, w.varlen)
    split = path == kda.KDA_ALGO_SPLIT
    launches_per_step = 1
    split_ms = {}
    segments = 1
    if split:
        rec = 66048  # bytes of one chunk record
        sws = ws_bytes
        carry = (N * H * dk * dv * 4 + 255) // 256 * 256
        nchunks = (T + 63) // 64
        if w.varlen:
            # [carry][chunk offsets][sequence order][chunk table][records of a
            # slice of columns]; the chunk table and the order cost three
            # launches, each slice two more
            g_max = nchunks + N
            rec_at = carry + (((N + 1) * 4 + 255) // 256 + (N * 4 + 255) // 256 +
                              (g_max * 8 + 255) // 256) * 256
            cols = (ws_bytes - rec_at) // (H * rec)
            launches_per_step = 3 + 2 * ((g_max + cols - 1) // cols)
            one_slice = False
        else:
            segments = kda.kda_split_segment_count(N, T, H, ws_bytes)
            slice_chunks = (ws_bytes - carry) // (N * H * rec)
            # the segmented form: the first segments' records, pass 1, the
            # entry states, the last segment's records, pass 2
            launches_per_step = 5 if segments > 1 else \
                2 * ((nchunks + slice_chunks - 1) // slice_chunks)
            one_slice = segments == 1 and slice_chunks >= nchunks
        swork = work

        def stage(sg):
            return kda.kda_split_stage(sg, d["q"], d["k"], d["v"], d["g"], d["beta"],
                                       d["init_state"], out, fs, N, T, H, 1.0, swork, sws,
                                       None, stream)
        if one_slice and stage(1) == 0 and stage(2) == 0:
            n_k = max(3, min(args.steps, 50))
            for sg, name in ((1, "kda_tc_intra_kernel"), (2, "kda_tc_state_kernel")):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(n_k):
                    stage(sg)
                e1.record(stream)
                torch.cuda.synchronize()
                split_ms[name] = e0.elapsed_time(e1) / n_k

    # ---- end to end: host buffers through kda_chunk_fwd_host ---------------
    e2e = None
    if not args.no_e2e:
        pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()}
        hout = torch.empty(w.B, T, H, dv, dtype=w.dtype).pin_memory()
        hfs = torch.empty(N, H, dk, dv, dtype=torch.float32).pin_memory()
        nbytes = kda.kda_host_staging_bytes(w.B if not w.varlen else N, T, H, dk, dv, dtype,
                                            x["init_state"] is not None, 1, w.varlen)
        staging = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def host_step():
            rc = kda.kda_chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"],
                                        pin["init_state"], hout, hfs, N, T, H, dk, dv,
                                        pin["cu_seqlens"], dtype, 1.0, staging, nbytes, stream)
            if rc != 0:
                raise RuntimeError("kda_chunk_fwd_host: " + kda.status_string(rc))
        host_step()
        n_e2e = max(1, min(args.steps, 5))
        if ws > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_step()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, ws, dev)
        h2d = sum(pin[k].numel() * pin[k].element_size()
                  for k in ("q", "k", "v", "g", "beta", "init_state", "cu_seqlens")
                  if pin[k] is not None)
        d2h = hout.numel() * hout.element_size() + hfs.numel() * 4 + 4
        e2e = {"value": job_value(ws, tokens, e2e_s * 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e}

    if ws > 1 and rank != 0:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
        return 0

    hbm_gbs, bf16_tf, peak_src = measured_peaks()
    kname = "kda_tc_fused_kernel" if path == kda.KDA_ALGO_TC else "kda_simt_kernel"
    traffic = None
    kernels = None
    if split:
        # the path is two kernels; the roofline is taken over the pair (one
        # forward), each kernel's own time and traffic listed beside it
        kname = "kda_tc_intra_kernel + kda_tc_state_kernel"
        if segments > 1:
            # the segmented form (two state passes and the entry states):
            # the per-kernel times taken alone would describe the plain form
            kname += " (%d segments per sequence)" % segments
        else:
            tr = [ncu_traffic(k, w.name) for k in ("kda_tc_intra_kernel",
                                                   "kda_tc_state_kernel")]
            traffic = sum(tr) if all(t is not None for t in tr) else None
            tot = sum(split_ms.values()) if split_ms else None
            kernels = {k: {"ms": v, "share": v / tot, "dram_bytes": ncu_traffic(k, w.name)}
                       for k, v in split_ms.items()} if split_ms else None
    else:
        traffic = ncu_traffic(kname, w.name)
    kernel_ms = float(np.mean(launch_ms))
    nbytes = alg_bytes(w, x["init_state"] is not None, True)
    achieved = nbytes / (kernel_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "traffic": traffic, "kernels": kernels,
                "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs, STREAM copy)",
                "kernel": kname, "alg_bytes_per_launch": nbytes,
                "kernel_ms_mean": kernel_ms,
                "tensor": {"alg_flops_per_launch": alg_flops(w),
                           "achieved_tflops": alg_flops(w) / (kernel_ms / 1e3) / 1e12,
                           "peak_tflops": bf16_tf,
                           "frac": alg_flops(w) / (kernel_ms / 1e3) / 1e12 / bf16_tf}}
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and ws == 1:
        dt, th, used = oracle_sample(w, args.cpu_units, args.cpu_tokens,
                                     min_seconds=args.cpu_seconds)
        n_u, n_t = min(args.cpu_units, w.B * w.H), min(args.cpu_tokens, w.T)
        cpu = {"value": th / w.H / dt, "unit": "tokens/s", "cores": used, "kind": "oracle",
               "sample": "%d (row, head) units x first %d tokens (of %d heads x %d tokens), "
                         "repeated %d times (%.1f s of oracle time)"
                         % (n_u, n_t, w.B * w.H, w.T, th // (n_u * n_t), dt),
               "seconds": dt}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": H, "dk": dk, "dv": dv,
                       "chunk": w.chunk, "n_seqs": N, "final_state": True,
                       "init_state": x["init_state"] is not None,
                       "l2": "inputs %.2f GB > 129 MB L2 (no flush needed)"
                             % (nbytes / 1e9) if nbytes > 129e6 else "L2-resident"},
            "clocks": clk, "e2e": e2e, "gpu_launches": args.steps * launches_per_step,
            "roofline": roofline, "cpu_baseline": cpu}
    print(json.dumps(line))
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_decode(args):
    """The decode / rebuild kernel alone (one GPU): T tokens per call for B x H
    states of d = 128, bf16 inputs; one JSON line with tokens/s and the
    fraction of the measured HBM bandwidth its state and input bytes take."""
    from gated_delta_rule_32_gb300 import build as kbuild
    from gated_delta_rule_32_gb300 import kda

    B, H, T = args.B or 64, args.H or 32, args.decode
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda:0")
    kbuild.build()
    kda.load()
    w = small_workload("decode", B=B, T=T, H=H, dk=128, dv=128, s0_std=0.02, seed=9)
    x = make_inputs(w)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
    state = d["init_state"].clone()
    out = torch.empty_like(d["v"])
    stream = torch.cuda.current_stream(dev)

    def step():
        rc = kda.kda_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], state, out, B, T, H, 128,
                            128, kda.KDA_BF16, 1.0, stream)
        if rc != 0:
            raise RuntimeError("kda_decode: " + kda.status_string(rc))
    for _ in range(args.warmup):
        step()
    steps = args.steps or 200
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    nbytes = B * H * 128 * 128 * 4 * 2 + B * T * H * (4 * 128 + 1) * 2 + B * T * H * 128 * 2
    hbm_gbs, _, peak_src = measured_peaks()
    achieved = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({"metric": "KDA decode tokens/s (state in registers, %d tokens per call)" % T,
                      "value": B * T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
                      "steps": steps, "warmup": args.warmup, "ms_per_step": ms,
                      "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": "decode", "B": B, "H": H, "T": T, "dk": 128,
                                 "dv": 128},
                      "gpu_launches": steps,
                      "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs,
                                   "unit": "GB/s", "frac": achieved / hbm_gbs,
                                   "traffic": None, "alg_bytes_per_launch": nbytes,
                                   "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)"}}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (default: as many as fill about 1.2 s)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--algo", type=int, default=0,
                    help="0 auto, 1 CUDA-core, 2 tensor-core fused, 3 tensor-core two-kernel")
    ap.add_argument("--B", type=int, default=0, help="resize (profiling captures only)")
    ap.add_argument("--H", type=int, default=0, help="resize (profiling captures only)")
    ap.add_argument("--T", type=int, default=0, help="resize (profiling captures only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-units", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle time the CPU baseline accumulates")
    ap.add_argument("--cpu-tokens", type=int, default=32768)
    ap.add_argument("--ref-units", type=int, default=16)
    ap.add_argument("--ref-tokens", type=int, default=4096)
    ap.add_argument("--decode", type=int, default=0, metavar="TOKENS",
                    help="instead of the forward: the decode kernel on --B x --H states "
                         "(default 64 x 32, d = 128) for TOKENS tokens per call")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.decode:
        return run_decode(args)
    if args.impl == "reference":
        if not args.steps:
            args.steps = 5
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
