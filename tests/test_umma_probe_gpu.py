"""tcgen05 building blocks on the GPU: one tile product D = A * B^T through
the library's probe entry point, for every operand layout the tensor-core
path uses, against a torch fp32 product of the same bf16 values."""
import pytest
import torch

from gated_delta_rule_32_gb300 import kda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    kda.load()


def run(M, N, K, a_mode, b_mode, pack, seed=0):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    D = torch.full((128, N), -1.0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = kda.kda_debug_umma(A.cuda(), B.cuda(), D, M, N, K, a_mode, b_mode, pack, st,
                            torch.cuda.current_stream())
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = A.float() @ B.float().T
    return D.cpu(), ref


@pytest.mark.parametrize("pack", [0, 1])
@pytest.mark.parametrize("a_mode,b_mode", [(0, 0), (0, 1), (1, 0), (1, 1), (2, 0), (2, 1)])
@pytest.mark.parametrize("N,K", [(16, 16), (64, 128), (128, 64), (192, 64), (256, 128)])
def test_tile_product_m128(N, K, a_mode, b_mode, pack):
    D, ref = run(128, N, K, a_mode, b_mode, pack, seed=N + K)
    err = (D - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err


def test_m64_lane_placement():
    N, K = 32, 64
    D, ref = run(64, N, K, 0, 0, 0, seed=3)
    # every row of the 64-row product must appear in exactly one lane
    found = {}
    for lane in range(128):
        row = D[lane]
        if torch.isnan(row).all():
            continue
        for r in range(64):
            if torch.allclose(row, ref[r], rtol=1e-5, atol=1e-4):
                found.setdefault(r, []).append(lane)
    print("M=64 lane of each row:", {r: found.get(r) for r in range(64)})
    assert sorted(found) == list(range(64))
    assert all(len(v) == 1 for v in found.values())


@pytest.mark.parametrize("K", [16, 64, 128])
@pytest.mark.parametrize("a_mode", [0, 1])
def test_tile_product_swizzled_mn_major_b(K, a_mode):
    # B in the layout a 128-byte-swizzled TMA load of a [K rows][64 channels]
    # tile writes (the state kernel's V operand)
    D, ref = run(128, 64, K, a_mode, 2, 0, seed=K + 7)
    err = (D - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err
