"""Pins of the oracle's assignment of slices to replicas (oracle.slice_costs,
oracle.partition), against facts that do not come from the oracle itself:

  * the slice loads summed over the four benchmark workloads equal the
    Newton-Schulz flop and optimizer-state byte totals tabulated for them
    (standard count, 5 steps; 14 bytes per bf16 element);
  * Graham's tight example for longest-first scheduling (jobs 3, 3, 2, 2, 2
    on two machines: makespan 7 against the optimum 6, the bound
    4/3 - 1/(3w) reached exactly);
  * on small random instances the makespan lies between the brute-force
    optimum and Graham's bound times it;
  * equal loads are dealt out round robin; one replica takes everything.
"""
import itertools
import math

import numpy as np
import pytest

import oracle

SKINNY_74 = [(24, 10240)] * 74
STACKS_EXPERTS = [(32, 24, 10240)] * 8 + [(64, 1408, 2048)] * 2 + [(64, 2048, 1408)]
DENSE_24L = [(4096, 4096)] * 96 + [(11008, 4096)] * 24 + [(4096, 11008)] * 48
MOE_24L = ([(2048, 2048)] * 4 + [(16, 1408, 2048)] * 2 + [(16, 2048, 1408)]) * 24 + [(24, 10240)] * 74


@pytest.mark.parametrize("shapes,gflop,gbytes", [(SKINNY_74, 8.74, 0.2546), (STACKS_EXPERTS, 20980, 8.63),
                                                 (DENSE_24L, 513334, 68.0), (MOE_24L, 150448, 52.4)],
                         ids=["skinny_74x24x10240", "stacks_experts", "dense_24L", "moe_24L"])
def test_slice_loads_sum_to_the_tabulated_totals(shapes, gflop, gbytes):
    dts = ["bf16"] * len(shapes)
    # a rate of 1e9 per second turns seconds into giga-units; the other rate
    # is made so large that its term never wins the max
    f = math.fsum(oracle.slice_costs(shapes, dts, 5, 1e9, 1e300))
    b = math.fsum(oracle.slice_costs(shapes, dts, 5, 1e300, 1e9))
    assert f == pytest.approx(gflop, rel=6e-4)
    assert b == pytest.approx(gbytes, rel=3e-3)


def test_load_is_the_larger_roofline_term():
    # [24, 10240] at 1.9 PFLOP/s and 6.8 TB/s is bandwidth bound, [4096, 4096]
    # is compute bound; fp32 parameters carry 20 bytes per element
    (skinny,) = oracle.slice_costs([(24, 10240)], ["bf16"], 5, 1.9e15, 6.8e12)
    (dense,) = oracle.slice_costs([(4096, 4096)], ["bf16"], 5, 1.9e15, 6.8e12)
    (f32,) = oracle.slice_costs([(24, 10240)], ["f32"], 5, 1.9e15, 6.8e12)
    assert skinny == 24 * 10240 * 14 / 6.8e12
    assert f32 == 24 * 10240 * 20 / 6.8e12
    assert dense == 5 * 6 * 4096 ** 3 / 1.9e15
    # the transposed shape costs the same; an [E, M, N] tensor gives E equal loads
    assert oracle.slice_costs([(10240, 24)], ["bf16"], 5, 1.9e15, 6.8e12) == [skinny]
    assert oracle.slice_costs([(3, 24, 10240)], ["bf16"], 5, 1.9e15, 6.8e12) == [skinny] * 3


def test_graham_tight_example():
    # loads 3, 3, 2, 2, 2: [1, 3] and [1, 2] bf16 slices at T = 0 and 14 B/s
    costs = oracle.slice_costs([(1, 3), (1, 3), (1, 2), (1, 2), (1, 2)], ["bf16"] * 5, 0, 1.0, 14.0)
    assert costs == [3.0, 3.0, 2.0, 2.0, 2.0]
    owner, load = oracle.partition(costs, 2)
    assert owner == [0, 1, 0, 1, 0]
    assert load == [7.0, 5.0]
    assert max(load) / 6.0 == pytest.approx(4 / 3 - 1 / (3 * 2))


def _brute_force_makespan(costs, world):
    best = math.inf
    for assign in itertools.product(range(world), repeat=len(costs)):
        load = [0.0] * world
        for c, r in zip(costs, assign):
            load[r] += c
        best = min(best, max(load))
    return best


def test_within_graham_bound_of_the_optimum():
    rng = np.random.default_rng(7)
    for _ in range(60):
        world = int(rng.integers(2, 4))
        n = int(rng.integers(1, 9 if world == 2 else 7))
        costs = [float(c) for c in rng.integers(1, 20, size=n)]
        owner, load = oracle.partition(costs, world)
        opt = _brute_force_makespan(costs, world)
        assert opt <= max(load) <= (4 / 3 - 1 / (3 * world)) * opt + 1e-9
        # every slice has one owner and the loads are the owners' sums
        assert sorted(set(owner)) <= list(range(world))
        for r in range(world):
            assert load[r] == pytest.approx(sum(c for c, o in zip(costs, owner) if o == r))


def test_equal_loads_are_dealt_round_robin():
    costs = oracle.slice_costs(SKINNY_74, ["bf16"] * 74, 5, 1.9e15, 6.8e12)
    owner, load = oracle.partition(costs, 8)
    assert owner == [i % 8 for i in range(74)]
    assert load.count(load[0]) == 2 and load.count(load[7]) == 6


def test_one_replica_takes_everything():
    costs = oracle.slice_costs(STACKS_EXPERTS, ["bf16"] * len(STACKS_EXPERTS), 5, 1.9e15, 6.8e12)
    owner, load = oracle.partition(costs, 1)
    assert owner == [0] * 448
    assert load[0] == pytest.approx(math.fsum(costs), rel=1e-12)


def test_largest_first_order_on_the_mixed_workload():
    # the MoE layer set on 8 replicas: the [2048, 2048] slices are the largest, and longest
    # first deals the first eight of them to ranks 0..7 in slice order
    costs = oracle.slice_costs(MOE_24L, ["bf16"] * len(MOE_24L), 5, 1.9e15, 6.8e12)
    owner, load = oracle.partition(costs, 8)
    big = [s for s, c in enumerate(costs) if c == max(costs)]
    assert len(big) == 96
    assert [owner[s] for s in big[:8]] == list(range(8))
    # list scheduling places each slice on the least loaded replica, so the
    # final spread of the loads is at most the largest slice load
    assert max(load) - min(load) <= max(costs)
