"""Owner planner ("MatrixFSDP", section 4.1, Algorithm 1), host only: the
library's assignment is bit-exact against an independent Python restatement
of RoleGreedy, ScopeGreedy and CostAware, and satisfies the invariants of
greedy list scheduling."""
import random

import pytest

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import build as mo_build
from matrix_optimizers_zero_gb300 import workloads


@pytest.fixture(scope="module", autouse=True)
def lib():
    mo_build.build()
    return mo.load_library()


def py_plan(roles, world, strategy, cap=0):
    n = len(roles)

    def assign(order, owner, load):
        for i in order:
            r = min(range(world), key=lambda k: (load[k], k))
            owner[i] = r
            load[r] += roles[i][0]

    def largest_first(idx):
        return sorted(idx, key=lambda i: -roles[i][0])     # stable: ties keep table order

    def role_greedy():
        owner, load = [None] * n, [0] * world
        for b in sorted({r[1] for r in roles}):
            assign(largest_first([i for i in range(n) if roles[i][1] == b]), owner, load)
        return owner, load

    def scope_greedy():
        owner, load = [None] * n, [0] * world
        assign(largest_first(range(n)), owner, load)
        return owner, load

    if strategy == mo.PLAN_ROLE_GREEDY:
        return (*role_greedy(), mo.PLAN_ROLE_GREEDY)
    if strategy == mo.PLAN_SCOPE_GREEDY:
        return (*scope_greedy(), mo.PLAN_SCOPE_GREEDY)
    o_r, l_r = role_greedy()
    o_s, l_s = scope_greedy()
    worst_block = 0
    for b in {r[1] for r in roles}:
        per = [0] * world
        for i in range(n):
            if roles[i][1] == b:
                per[o_s[i]] += roles[i][0]
        worst_block = max(worst_block, max(per))
    if n and (cap <= 0 or worst_block <= cap) and max(l_s) < max(l_r):
        return o_s, l_s, mo.PLAN_SCOPE_GREEDY
    return o_r, l_r, mo.PLAN_ROLE_GREEDY


def role_sets():
    sets = {
        "gpt2l": workloads.owner_roles(workloads.get_workload("gpt2l"), 4),
        "llama8b": workloads.owner_roles(workloads.get_workload("llama8b"), 7),
        "share32b": workloads.owner_roles(workloads.get_workload("share32b"), 7),
    }
    rng = random.Random(3)
    for k in range(4):
        sets[f"random{k}"] = [(rng.choice([0, 1, 7, 64, 64, 1000, 4096, 5000]) * rng.randint(1, 4),
                               rng.randint(0, 5), rng.randint(0, 1)) for _ in range(rng.randint(1, 60))]
    return sets


ROLE_SETS = role_sets()


@pytest.mark.parametrize("name", sorted(ROLE_SETS))
@pytest.mark.parametrize("world", [1, 2, 3, 8, 64])
@pytest.mark.parametrize("strategy", [0, 1, 2])
def test_bit_exact_against_restatement(name, world, strategy):
    roles = ROLE_SETS[name]
    got = mo.mo_plan_owners(roles, world, strategy)
    want = py_plan(roles, world, strategy)
    assert got == (list(want[0]), list(want[1]), want[2])


@pytest.mark.parametrize("name", sorted(ROLE_SETS))
@pytest.mark.parametrize("world", [2, 8, 64])
def test_invariants(name, world):
    roles = ROLE_SETS[name]
    total = sum(r[0] for r in roles)
    for strategy in (0, 1, 2):
        owners, loads, _ = mo.mo_plan_owners(roles, world, strategy)
        assert all(0 <= o < world for o in owners)
        recomputed = [0] * world
        for (numel, _, _), o in zip(roles, owners):
            recomputed[o] += numel
        assert recomputed == loads and sum(loads) == total
        # greedy list scheduling never exceeds the average load by more than one role
        assert max(loads) <= total / world + max(r[0] for r in roles)


def test_cost_aware_cap_and_choice():
    roles = ROLE_SETS["gpt2l"]
    _, l_role, _ = mo.mo_plan_owners(roles, 8, mo.PLAN_ROLE_GREEDY)
    _, l_scope, _ = mo.mo_plan_owners(roles, 8, mo.PLAN_SCOPE_GREEDY)
    _, _, chosen = mo.mo_plan_owners(roles, 8, mo.PLAN_COST_AWARE)
    assert chosen == (mo.PLAN_SCOPE_GREEDY if max(l_scope) < max(l_role) else mo.PLAN_ROLE_GREEDY)
    # a cap below any single role forces RoleGreedy
    _, _, chosen = mo.mo_plan_owners(roles, 8, mo.PLAN_COST_AWARE, block_cap=1)
    assert chosen == mo.PLAN_ROLE_GREEDY


def test_hand_example():
    # one block: 10, 7, 5, 4, 3 over 2 ranks -> largest first to the lightest
    roles = [(5, 0, 0), (10, 0, 0), (3, 0, 1), (7, 0, 0), (4, 0, 0)]
    owners, loads, _ = mo.mo_plan_owners(roles, 2, mo.PLAN_ROLE_GREEDY)
    # 10 -> r0 (10|0), 7 -> r1 (10|7), 5 -> r1 (10|12), 4 -> r0 (14|12), 3 -> r1 (14|15)
    assert owners == [1, 0, 1, 1, 0] and loads == [14, 15]


def test_validation():
    lib = mo.load_library()
    with pytest.raises(mo.MoError):
        mo.mo_plan_owners([(5, 0, 0)], 0)
    with pytest.raises(mo.MoError):
        mo.mo_plan_owners([(5, 0, 0)], 2, strategy=7)
    with pytest.raises(mo.MoError):
        mo.mo_plan_owners([(-1, 0, 0)], 2)
    assert mo.mo_plan_owners([], 4) == ([], [0, 0, 0, 0], mo.PLAN_ROLE_GREEDY)
