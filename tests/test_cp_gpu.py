"""Context parallelism on the GPU: two and three gloo ranks, each its own
process on cuda:0, run their spans of one batch through the library's
kernels (span summary, composition, forward); the exchange is a host-side
all-gather, so no kernel waits on another rank.  The concatenated outputs
and the last rank's final state must match the fp64 oracle's forward of the
whole batch within the bf16 bound."""
import numpy as np
import pytest
import torch

import oracle
from kda_inputs import make_inputs, small_workload
from tests.test_cp import run_ranks

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world,T", [(2, 300), (3, 257)])
def test_context_parallel_on_one_gpu(world, T, tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    B, H, d, seed = 1, 2, 128, 34
    ranks = run_ranks(world, "gpu", tmp_path, B, T, H, d, seed)
    w = small_workload("cp", B=B, T=T, H=H, dk=d, dv=d, seed=seed, s0_std=0.05)
    x = make_inputs(w)
    o_ref, s_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"])
    out = np.concatenate([r["out"] for r in ranks], axis=1)
    assert np.abs(out - o_ref).max() <= 1e-2 * np.abs(o_ref).max()
    s = ranks[-1]["state"]
    assert np.abs(s - s_ref).max() <= 1e-2 * np.abs(s_ref).max()
