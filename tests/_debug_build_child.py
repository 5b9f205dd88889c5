"""Child process of tests/test_debug_build_gpu.py: loads the KDA_DEBUG build
of libkda.so (device-side bounds checks) as the only library of a fresh
process and prints one JSON line with what it saw."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from gated_delta_rule_32_gb300 import build, kda  # noqa: E402
from kda_inputs import make_inputs, small_workload  # noqa: E402


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def main():
    kda.load(build.LIB_DEBUG)
    res = {"info": kda.kda_build_info()}
    cases = {"dense": small_workload("dbg", B=2, T=300, H=2, seed=71, s0_std=0.05),
             "packed": small_workload("dbgp", B=1, T=461, H=2, seed=72, varlen=True,
                                      lengths=(100, 1, 64, 296)),
             # the segmented form (three segments forced): records of every
             # chunk, two state passes
             "segmented": small_workload("dbgs", B=1, T=1000, H=2, seed=73, s0_std=0.05)}
    for name, w in cases.items():
        kda.kda_debug_split_segments(3 if name == "segmented" else 0)
        x = make_inputs(w)
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
        N, T, H = x["B"], x["T"], x["H"]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")

        def run():
            out = torch.zeros_like(d["v"])
            fs = torch.zeros(N, H, 128, 128, device="cuda")
            rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                      d["init_state"], out, fs, N, T, H, 128, 128,
                                      d["cu_seqlens"], kda.KDA_BF16, 0, 1.0, kda.KDA_ALGO_SPLIT,
                                      None, 0, status, torch.cuda.current_stream())
            torch.cuda.synchronize()
            return rc, int(status.item()), out, fs
        rc, st, out, fs = run()
        o_ref, s_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"],
                                  x["cu_seqlens"])
        res[name] = {"rc": rc, "status": st, "err_o": rel(out.float().cpu().numpy(), o_ref),
                     "err_s": rel(fs.cpu().numpy(), s_ref)}
        # the kernels are told the workspace holds two chunk records: the
        # later items' checks fire (the real workspace holds all of them)
        kda.kda_debug_record_capacity(2)
        try:
            rc2, st2, _, _ = run()
        finally:
            kda.kda_debug_record_capacity(0)
        rc3, st3, out3, fs3 = run()
        res[name].update({"rc_small": rc2, "status_small": st2, "status_after": st3,
                          "same_after": bool(torch.equal(out3, out) and torch.equal(fs3, fs))})
    kda.kda_debug_split_segments(0)
    print(json.dumps(res))


if __name__ == "__main__":
    main()
