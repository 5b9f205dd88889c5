"""The seeded input generator: every workload is drawn from its own seed.

CPU only.  torch's CPU generator keeps only the low 32 bits of a seed, so
the workload seed, batch row and head are mixed into those bits; these tests
check that each of the three changes the draws, and that the five workloads
carry the seeds 0-4 their recipes state.
"""
import dataclasses
import itertools

import torch

from kda_inputs import WORKLOADS, _splitmix64, make_unit, small_workload, unit_seed


def test_splitmix64_published_value():
    # first output of the splitmix64 generator started from state 0
    assert _splitmix64(0) == 0xE220A8397B1DCDAF


def test_workload_seeds_are_the_recipes():
    seeds = {"tiny_fp32": 0, "h4_t4k": 1, "b2_h32_t32k": 2, "varlen_floor": 3, "ctx1m": 4}
    for name, s in seeds.items():
        assert WORKLOADS[name].seed == s, name


def test_unit_seeds_distinct_and_32_bit():
    seen = set()
    for s, b, h in itertools.product(range(6), range(4), range(40)):
        u = unit_seed(s, b, h)
        assert 0 <= u < (1 << 32)
        seen.add(u)
    assert len(seen) == 6 * 4 * 40


def test_generator_keeps_only_low_32_bits():
    # why the mix is needed: seeds that differ only above bit 31 draw alike
    a = torch.randn(4, generator=torch.Generator().manual_seed((2 << 32) + 5))
    b = torch.randn(4, generator=torch.Generator().manual_seed((7 << 32) + 5))
    assert torch.equal(a, b)


def test_different_seeds_draw_different_inputs():
    draws = {}
    for name in ("tiny_fp32", "h4_t4k", "b2_h32_t32k", "varlen_floor", "ctx1m"):
        w = dataclasses.replace(WORKLOADS[name], T=32, dk=16, dv=16, varlen=False)
        u = make_unit(w, 0, 0)
        draws[name] = torch.cat([u["q"].flatten(), u["v"].flatten()])
    names = list(draws)
    for a, b in itertools.combinations(names, 2):
        assert not torch.equal(draws[a], draws[b]), (a, b)


def test_rows_heads_and_ranks_draw_different_inputs():
    w = small_workload("s", B=2, T=16, H=2, dk=16, dv=16, seed=9)
    units = [make_unit(w, b, h)["k"] for b in range(2) for h in range(2)]
    units.append(make_unit(dataclasses.replace(w, row_offset=2), 0, 0)["k"])
    for a, b in itertools.combinations(range(len(units)), 2):
        assert not torch.equal(units[a], units[b]), (a, b)


def test_same_seed_redraws_the_same_inputs():
    w = small_workload("s", B=1, T=16, H=1, dk=16, dv=16, seed=3)
    assert torch.equal(make_unit(w, 0, 0)["g"], make_unit(w, 0, 0)["g"])
