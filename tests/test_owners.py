"""Host checks of the owner assignment (greedy LPT with a byte cap and layer
spreading; DMuon-2 section 3.3 and Appendix B).  No GPU is needed."""
import itertools
import random

import pytest

from newton_schulz_gb300 import binding


@pytest.fixture(autouse=True)
def _lib(lib):
    yield


def _loads(owner, costs, n):
    t = [0.0] * n
    for o, c in zip(owner, costs):
        t[o] += c
    return t


def test_lpt_within_graham_bound_of_the_optimum():
    # tiny instances: brute force over all assignments; LPT's makespan is at
    # most (4/3 - 1/(3N)) of the optimum (Graham 1969)
    rng = random.Random(1)
    for trial in range(40):
        n_units, n = rng.randint(3, 7), rng.randint(2, 3)
        costs = [rng.uniform(0.1, 10.0) for _ in range(n_units)]
        owner = binding.muon_assign_owners(costs, n, eps=1e9)
        lpt = max(_loads(owner, costs, n))
        best = min(max(_loads(a, costs, n)) for a in itertools.product(range(n), repeat=n_units))
        assert lpt <= (4 / 3 - 1 / (3 * n)) * best + 1e-9, (costs, n, lpt, best)


def test_lpt_rule_step_by_step():
    # units sorted by cost; each to the least-loaded rank (lowest index on ties)
    # loads after each unit: [5,0,0] [5,4,0] [5,4,3] [5,4,6] [5,6,6] [7,6,6] [7,7,6]
    costs = [5, 4, 3, 3, 2, 2, 1]
    owner = binding.muon_assign_owners(costs, 3, eps=1e9)
    assert owner == [0, 1, 2, 2, 1, 0, 1]


def test_ties_break_by_elements_then_order():
    owner = binding.muon_assign_owners([1.0, 1.0, 1.0], 3, elems=[5, 9, 5], eps=1e9)
    assert owner == [1, 0, 2]


def test_layer_spreading():
    rng = random.Random(2)
    costs = [rng.uniform(1, 2) for _ in range(12)]
    layers = [i // 4 for i in range(12)]          # 3 layers of 4 units, 4 ranks
    owner = binding.muon_assign_owners(costs, 4, layers=layers, eps=1e9)
    for l in range(3):
        assert sorted(owner[4 * l:4 * l + 4]) == [0, 1, 2, 3]


def test_byte_cap_and_fallback():
    # by time alone rank 1 would take every small unit (160 of 170 bytes);
    # the cap (1.1 x 85) sends the later ones to rank 0
    costs = [9.0, 1.0, 1.0, 1.0, 1.0]
    nbytes = [10, 40, 40, 40, 40]
    owner = binding.muon_assign_owners(costs, 2, nbytes=nbytes, eps=0.1)
    b = [0, 0]
    for o, x in zip(owner, nbytes):
        b[o] += x
    assert owner == [0, 1, 1, 0, 0] and max(b) <= 1.1 * sum(nbytes) / 2
    uncapped = binding.muon_assign_owners(costs, 2, nbytes=nbytes, eps=1e9)
    assert uncapped == [0, 1, 1, 1, 1]
    # infeasible cap: each unit goes to the candidate with the fewest bytes
    owner = binding.muon_assign_owners([1.0, 1.0], 2, nbytes=[100, 100], eps=0.0)
    assert sorted(owner) == [0, 1]


def test_balanced_better_than_round_robin():
    # one heavy unit in every eight: round-robin in parameter order gives all
    # of them to rank 0; LPT spreads them
    costs = ([10.0] + [1.0] * 7) * 4
    owner = binding.muon_assign_owners(costs, 8, eps=1e9)
    lpt = max(_loads(owner, costs, 8))
    rr = max(_loads([i % 8 for i in range(len(costs))], costs, 8))
    mean = sum(costs) / 8
    assert lpt <= 1.3 * mean and rr >= 4 * mean


def test_argument_errors(lib):
    import ctypes
    out = (ctypes.c_int32 * 2)()
    arr = (binding.Unit * 2)(binding.Unit(1.0, 0, 0, -1), binding.Unit(1.0, 0, 0, -1))
    assert lib.muon_assign_owners(arr, 2, 0, 0.1, out) == 1
    assert lib.muon_assign_owners(arr, -1, 2, 0.1, out) == 1
    assert lib.muon_assign_owners(arr, 2, 2, -0.5, out) == 1
    assert lib.muon_assign_owners(None, 2, 2, 0.1, out) == 1
    bad = (binding.Unit * 1)(binding.Unit(float("nan"), 0, 0, -1))
    assert lib.muon_assign_owners(bad, 1, 2, 0.1, out) == 1
    assert lib.muon_assign_owners(arr, 0, 2, 0.1, out) == 0
    assert lib.muon_ns_cost_table(None, 1, None, 3, None, None) == 1
